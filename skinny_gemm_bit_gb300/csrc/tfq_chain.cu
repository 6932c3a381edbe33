// The whole per-token weight stream of a dense decoder in one persistent kernel
// (Husky page, "Experiments with a full-step megakernel": what pays is loading the
// next stage's weights while the current stage computes).
//
// Stages, in order: for every layer l, (0) RMSNorm + QKV, (1) O + residual (the Q
// part of the QKV output stands in for attention), (2) RMSNorm + gate/up + SwiGLU,
// (3) down + residual; then (4) the final RMSNorm + readout. Every stage is split
// into whole 16-row blocks (all of K), block i going to CTA i mod C; the grid is one
// CTA per SM, launched cooperatively so that every CTA is resident.
//
// One producer warp walks the CTA's blocks of every stage in order and streams
// their tiles into a ring of 32-tile slots with bulk copies: weights never depend
// on activations, so it runs ahead across stage boundaries, bounded only by the
// ring. The eight consumer warps, stage by stage: wait until every CTA has finished
// the previous stage (a per-stage arrival counter in global memory), load the
// stage's activation rows from L2 straight into B-fragment order (normalising
// them when the stage folds an RMSNorm in), run the rounds of the stage (R blocks
// side by side, the consumer warps split evenly over them, one slot per step),
// sum each block's warps,
// apply the epilogue and store, then arrive on the stage's counter.
//
// Every wait is bounded; a wait that gives up records TF_E_TIMEOUT in the status
// word, which every spinning CTA also polls, so the whole grid leaves promptly.
// The last CTA to finish resets the counters, so the workspace is left as found.
#include "tfq_internal.h"
#include "tfq_ptx.cuh"
#include "tfq_qproj.cuh"

namespace tfq {
namespace {

constexpr int kChainWarps = 12;
constexpr int kChainMaxR = 4;  // blocks side by side in a round; divides kChainWarps
static_assert(kChainWarps % kChainMaxR == 0, "every round's blocks get the same number of warps");
constexpr int kChainThreads = (kChainWarps + 1) * 32;
constexpr int kChainBarAll = 15;  // named barrier of the consumer warps; 1, 2 are team barriers

struct StageDesc {
    const uint8_t* w0;
    const uint8_t* w1;
    const uint16_t* x;
    const uint16_t* gamma;
    const uint16_t* res;
    uint16_t* y;
    int64_t ldx, ldr, ldy;
    int N, K, n_rb, groups, mats, R, cg;
};

__device__ __forceinline__ uint16_t* act_ptr(const ChainParams& p, int role, int l)
{
    return p.buf[role] + (int64_t)l * p.lstride[role] + (int64_t)(l & 1) * p.astride[role];
}

__device__ __forceinline__ StageDesc stage_desc(const ChainParams& p, int s)
{
    StageDesc d;
    const int l = s >> 2;
    const int kind = s < 4 * p.L ? (s & 3) : 4;
    const uint16_t* h_in = l == 0 ? p.x : act_ptr(p, 3, l - 1);  // residual stream entering layer l
    const int qkv_n = p.Q + 2 * p.KV;
    d.w1 = nullptr;
    d.gamma = nullptr;
    d.res = nullptr;
    d.ldr = 0;
    d.mats = 1;
    if (kind == 0) {
        d.w0 = p.layer[l].qkv;
        d.x = h_in;
        d.ldx = p.D;
        d.gamma = p.layer[l].attn_norm;
        d.y = act_ptr(p, 0, l);
        d.N = qkv_n;
        d.ldy = qkv_n;
        d.K = p.D;
    } else if (kind == 1) {
        d.w0 = p.layer[l].o;
        d.x = act_ptr(p, 0, l);
        d.ldx = qkv_n;
        d.res = h_in;
        d.ldr = p.D;
        d.y = act_ptr(p, 1, l);
        d.N = p.D;
        d.ldy = p.D;
        d.K = p.Q;
    } else if (kind == 2) {
        d.w0 = p.layer[l].gate;
        d.w1 = p.layer[l].up;
        d.mats = 2;
        d.x = act_ptr(p, 1, l);
        d.ldx = p.D;
        d.gamma = p.layer[l].mlp_norm;
        d.y = act_ptr(p, 2, l);
        d.N = p.F;
        d.ldy = p.F;
        d.K = p.D;
    } else if (kind == 3) {
        d.w0 = p.layer[l].down;
        d.x = act_ptr(p, 2, l);
        d.ldx = p.F;
        d.res = act_ptr(p, 1, l);
        d.ldr = p.D;
        d.y = act_ptr(p, 3, l);
        d.N = p.D;
        d.ldy = p.D;
        d.K = p.F;
    } else {
        d.w0 = p.readout;
        d.x = p.L == 0 ? p.x : act_ptr(p, 3, p.L - 1);
        d.ldx = p.D;
        d.gamma = p.final_norm;
        d.y = p.logits;
        d.N = p.V;
        d.ldy = p.V;
        d.K = p.D;
    }
    d.n_rb = (d.N + kRowsPerBlock - 1) / kRowsPerBlock;
    d.groups = d.K / kGroup;
    // up to kChainMaxR blocks side by side (as many as a CTA has, a power of two)
    const int per_cta = (d.n_rb + p.C - 1) / p.C;
    d.R = 1;
    while (2 * d.R <= per_cta && 2 * d.R <= kChainMaxR)
        d.R *= 2;
    d.cg = kChainSlotTiles / (d.mats * d.R);
    return d;
}

// blocks of the stage owned by CTA c: c, c + C, c + 2C, ...
__device__ __forceinline__ int blocks_of(const StageDesc& d, int c, int C)
{
    return c < d.n_rb ? (d.n_rb - c + C - 1) / C : 0;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* ptr)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Thread 0: wait until every CTA has arrived on counter `s` (bounded; gives up at
// once when another CTA has recorded a failure).
__device__ bool grid_wait(const ChainParams& p, int s, volatile int* flags)
{
    const long long t0 = clock64();
    const long long limit = (long long)(p.limit_ns * 2);
    int polls = 0;
    while (ld_acquire_u32(p.bar + s) < (unsigned)p.C) {
        if ((++polls & 63) == 0) {
            if (*reinterpret_cast<volatile int*>(p.status) != 0) {
                flags[0] = 1;
                return false;
            }
            if (clock64() - t0 > limit) {
                flags[0] = 1;
                atomicCAS(p.status, 0, TF_E_TIMEOUT);
                return false;
            }
        }
    }
    return true;  // the acquire load orders every later read after the arrivals
}

// Thread 0, after the CTA's barrier: release the CTA's stores of stage s and arrive.
__device__ __forceinline__ void grid_arrive(const ChainParams& p, int s)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p.bar + s) : "memory");
}

// Block rb's outputs from one lane's accumulator fragment (rows rb*16 + gi, + 8;
// activation rows 2t, 2t + 1): SwiGLU for gate/up, residual add, bf16 store.
// The residual values of block rb for one lane's fragment (0 where there is none);
// written by other CTAs in earlier stages, so read through L2.
__device__ __forceinline__ void load_residual(const StageDesc& d, int rb, int lane, int M, float (&r)[4])
{
    const int gi = lane >> 2, t = lane & 3;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int n = rb * kRowsPerBlock + gi + 8 * (v >> 1);
        const int m = 2 * t + (v & 1);
        r[v] = (d.res != nullptr && n < d.N && m < M)
                   ? __uint_as_float((uint32_t)__ldcg(d.res + (int64_t)m * d.ldr + n) << 16)
                   : 0.f;
    }
}

// Block rb's outputs from one lane's accumulator fragment (rows rb*16 + gi, + 8;
// activation rows 2t, 2t + 1): SwiGLU for gate/up, residual add, bf16 store.
__device__ __forceinline__ void store_block(const StageDesc& d, int rb, int lane, int M, const float (&a0)[4],
                                            const float (&a1)[4], const float (&res)[4])
{
    const int gi = lane >> 2, t = lane & 3;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int n = rb * kRowsPerBlock + gi + 8 * (v >> 1);
        const int m = 2 * t + (v & 1);
        if (n >= d.N || m >= M)
            continue;
        float val = a0[v];
        if (d.mats == 2)
            val = val / (1.f + expf(-val)) * a1[v];
        if (d.res != nullptr)
            val += res[v];
        reinterpret_cast<__nv_bfloat16*>(d.y)[(int64_t)m * d.ldy + n] = __float2bfloat16_rn(val);
    }
}

// 13 warps: at most 4 per SM sub-partition, whose 16K registers hold 4 x 32 x 128
template <int BITS>
__global__ void __maxnreg__(128) chain_kernel(const __grid_constant__ ChainParams p)
{
    constexpr int TILE = tile_bytes_for(BITS);
    constexpr int SLOT = kChainSlotTiles * TILE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [16]
    uint64_t* empty = full + 16;                          // [16]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + 256);  // [0] abort, [1] its snapshot
    float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    uint8_t* xraw = smem + p.xraw_off;
    uint8_t* ring = smem + p.ring_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int S = 4 * p.L + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kChainWarps);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer
    if (warp == kChainWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int seq = 0, pslot = 0;
            uint32_t pphase = 0;
            bool ok = true;
            for (int s = 0; s < S && ok; ++s) {
                const StageDesc d = stage_desc(p, s);
                const int nb = blocks_of(d, c, p.C);
                const int rounds = (nb + d.R - 1) / d.R, steps = (d.groups + d.cg - 1) / d.cg;
                for (int t = 0; t < rounds && ok; ++t) {
                    const int nv = min(d.R, nb - t * d.R);
                    for (int k = 0; k < steps; ++k, ++seq) {
                        const int slot = pslot;
                        const uint32_t ph = pphase;
                        if (++pslot == p.nst) {
                            pslot = 0;
                            pphase ^= 1u;
                        }
                        if (!wait_or_abort(&empty[slot], ph ^ 1u, flags, p.status, p.limit_ns)) {
                            ok = false;
                            break;
                        }
                        const int cnt = min(d.cg, d.groups - k * d.cg);
                        mbar_arrive_expect_tx(&full[slot], (uint32_t)(nv * d.mats * cnt * TILE));
                        uint8_t* sb = ring + slot * SLOT;
                        for (int r = 0; r < nv; ++r) {
                            const int64_t tile = (int64_t)(c + (t * d.R + r) * p.C) * d.groups + k * d.cg;
                            bulk_g2s(sb + (r * d.cg) * TILE, d.w0 + tile * TILE, (uint32_t)(cnt * TILE), &full[slot],
                                     pol);
                            if (d.mats == 2)
                                bulk_g2s(sb + ((d.R + r) * d.cg) * TILE, d.w1 + tile * TILE, (uint32_t)(cnt * TILE),
                                         &full[slot], pol);
                        }
                    }
                }
            }
            // no copy may still be in flight when the CTA leaves (also after an abort)
            for (int q = max(0, seq - p.nst); q < seq; ++q)
                mbar_wait_bounded(&full[q % p.nst], (q / p.nst) & 1u, p.limit_ns);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int cw = warp, gi = lane >> 2, tq = lane & 3;
    int slot = 0;
    uint32_t phase = 0;
    bool alive = true;
    for (int s = 0; s < S; ++s) {
        const StageDesc d = stage_desc(p, s);
        if (s > 0) {
            // the stage's inputs are the previous stage's outputs, from every CTA; the
            // abort decision is thread 0's snapshot, so every consumer warp takes it alike
            if (threadIdx.x == 0) {
                if (!flags[0])
                    grid_wait(p, s - 1, flags);
                flags[1] = flags[0];
            }
            __syncwarp();
            named_bar_sync(kChainBarAll, kChainWarps * 32);
            if (flags[1])
                break;
        }
        const int nb = blocks_of(d, c, p.C);
        const int KW = kChainWarps / d.R, r_me = cw / KW, kp = cw - r_me * KW;
        // the first round's residual values travel while the activations are staged
        float res0[4];
        load_residual(d, c + r_me * p.C, lane, (kp == 0 && r_me < nb) ? p.M : 0, res0);
        if (nb > 0)  // CTA-uniform
            x_direct_raw<12>(d.x, d.ldx, d.K, d.gamma, p.eps, p.x_rs, xraw, p.M, xsum, red, cw, lane, kChainWarps,
                             kChainBarAll);

        const int rounds = (nb + d.R - 1) / d.R, steps = (d.groups + d.cg - 1) / d.cg;
        for (int t = 0; t < rounds; ++t) {
            const int kb = t * d.R + r_me;
            const bool valid = kb < nb;
            float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
            float bcc0[4] = {0.f, 0.f, 0.f, 0.f}, bcc1[4] = {0.f, 0.f, 0.f, 0.f};  // second chain
            for (int k = 0; k < steps; ++k) {
                const bool ok = alive && wait_or_abort(&full[slot], phase, flags, p.status, p.limit_ns);
                alive = __all_sync(0xffffffffu, ok);
                const int cnt = min(d.cg, d.groups - k * d.cg);
                if (alive && valid) {
                    const uint8_t* sb = ring + slot * SLOT;
                    const uint8_t* t0 = sb + (r_me * d.cg) * TILE;
                    const uint8_t* t1 = sb + ((d.R + r_me) * d.cg) * TILE;
                    int j = kp;
                    // two tiles per iteration into separate accumulators: independent chains
                    for (; j + KW < cnt; j += 2 * KW) {
                        const int g = k * d.cg + j;
                        uint4 xa, xb, ya, yb;
                        x_frag(xraw, p.x_rs, gi, tq, g, p.M, xa, xb);
                        x_frag(xraw, p.x_rs, gi, tq, g + KW, p.M, ya, yb);
                        const float2 xs = *reinterpret_cast<const float2*>(xsum + g * kMaxM + 2 * tq);
                        const float2 ys = *reinterpret_cast<const float2*>(xsum + (g + KW) * kMaxM + 2 * tq);
                        tile_mac<BITS>(t0 + j * TILE, lane, xa, xb, xs, acc0);
                        tile_mac<BITS>(t0 + (j + KW) * TILE, lane, ya, yb, ys, bcc0);
                        if (d.mats == 2) {
                            tile_mac<BITS>(t1 + j * TILE, lane, xa, xb, xs, acc1);
                            tile_mac<BITS>(t1 + (j + KW) * TILE, lane, ya, yb, ys, bcc1);
                        }
                    }
                    if (j < cnt) {
                        const int g = k * d.cg + j;
                        uint4 xa, xb;
                        x_frag(xraw, p.x_rs, gi, tq, g, p.M, xa, xb);
                        const float2 xs = *reinterpret_cast<const float2*>(xsum + g * kMaxM + 2 * tq);
                        tile_mac<BITS>(t0 + j * TILE, lane, xa, xb, xs, acc0);
                        if (d.mats == 2)
                            tile_mac<BITS>(t1 + j * TILE, lane, xa, xb, xs, acc1);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[slot]);
                if (++slot == p.nst) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc0[i] += bcc0[i];
                acc1[i] += bcc1[i];
            }
            // sum the KW warps of the block (team barrier 1 + r_me)
            if (KW > 1) {
                float4* red4 = reinterpret_cast<float4*>(red);
                if (t > 0)
                    named_bar_sync(1 + r_me, KW * 32);  // the previous round's reads are done
                red4[cw * 32 + lane] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
                red4[kChainWarps * 32 + cw * 32 + lane] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
                named_bar_sync(1 + r_me, KW * 32);
                if (kp == 0) {
                    for (int q = 1; q < KW; ++q) {
                        const float4 o0 = red4[(cw + q) * 32 + lane];
                        const float4 o1 = red4[kChainWarps * 32 + (cw + q) * 32 + lane];
                        acc0[0] += o0.x;
                        acc0[1] += o0.y;
                        acc0[2] += o0.z;
                        acc0[3] += o0.w;
                        acc1[0] += o1.x;
                        acc1[1] += o1.y;
                        acc1[2] += o1.z;
                        acc1[3] += o1.w;
                    }
                }
            }
            if (alive && valid && kp == 0) {
                if (t == 0) {
                    store_block(d, c + kb * p.C, lane, p.M, acc0, acc1, res0);
                } else {
                    float rv[4];
                    load_residual(d, c + kb * p.C, lane, p.M, rv);
                    store_block(d, c + kb * p.C, lane, p.M, acc0, acc1, rv);
                }
            }
        }
        // every store of this CTA for stage s is done: arrive (every consumer warp gets
        // here, whatever its own waits returned)
        __syncwarp();
        named_bar_sync(kChainBarAll, kChainWarps * 32);
        if (threadIdx.x == 0 && !flags[0])
            grid_arrive(p, s);
    }
    // the last CTA to finish resets every counter (nobody waits on them any more)
    if (threadIdx.x == 0 && !flags[0]) {
        __threadfence();
        if (atomicAdd(p.bar + S, 1u) == (unsigned)(p.C - 1)) {
            for (int i = 0; i <= S; ++i)
                p.bar[i] = 0u;
            __threadfence();
        }
    }
}

}  // namespace

size_t chain_smem(int bits, int kmax, int* nst, int* x_rs, int* xsum_off, int* red_off, int* xraw_off, int* ring_off)
{
    const size_t slot = (size_t)kChainSlotTiles * tile_bytes_for(bits);
    *xsum_off = 512;
    *red_off = 512 + kChainMaxGroups * kMaxM * 4;                     // 2048
    *xraw_off = *red_off + 2 * kChainWarps * 32 * 16;                 // two float4 per lane and warp
    *x_rs = kmax * 2 + 16;
    *ring_off = (int)((*xraw_off + (size_t)kMaxM * *x_rs + 127) / 128 * 128);
    const size_t budget = 227 * 1024;
    const int n = budget > *ring_off + 2 * slot ? (int)((budget - *ring_off) / slot) : 0;
    *nst = n > 16 ? 16 : n;
    return *ring_off + (size_t)*nst * slot;
}

bool chain_fits(int bits, size_t smem)
{
    const void* fn = bits == 4 ? reinterpret_cast<const void*>(&chain_kernel<4>)
                               : reinterpret_cast<const void*>(&chain_kernel<8>);
    int dev = 0, coop = 0, blocks = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
        return false;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kChainThreads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return blocks >= 1;
}

cudaError_t launch_chain(int bits, const ChainParams& p, size_t smem, cudaStream_t stream)
{
    const void* fn = bits == 4 ? reinterpret_cast<const void*>(&chain_kernel<4>)
                               : reinterpret_cast<const void*>(&chain_kernel<8>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.C);
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (bits == 4)
        return cudaLaunchKernelEx(&cfg, chain_kernel<4>, p);
    return cudaLaunchKernelEx(&cfg, chain_kernel<8>, p);
}

}  // namespace tfq
