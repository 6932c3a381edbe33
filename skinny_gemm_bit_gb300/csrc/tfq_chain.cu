// The per-token weight stream of a dense decoder's layers in one persistent kernel
// (Husky page, "Experiments with a full-step megakernel": what pays is loading the
// next stage's weights while the current stage computes).
//
// Stages, in order: for every layer l, (0) RMSNorm + QKV, (1) O + residual (the Q
// part of the QKV output stands in for attention), (2) RMSNorm + gate/up + SwiGLU,
// (3) down + residual. (The final RMSNorm + readout is its own kernel, launched
// right after this one.) Every stage is split into whole 16-row blocks (all of K);
// the grid is one CTA per SM, launched cooperatively so that every CTA is resident.
//
// One producer warp walks the CTA's blocks of every stage in order and streams
// their tiles into a ring of 32-tile slots with bulk copies: weights never depend
// on activations, so it runs ahead across stage boundaries, bounded only by the
// ring. The twelve consumer warps, stage by stage:
//   - a CTA with no block in the stage arrives on the stage's counter at once and
//     moves on (its weights are already streaming for the next stage it works in);
//   - otherwise thread 0 waits until every CTA has arrived on the counter of the
//     stage that wrote the input (and of the one that wrote the residual), then
//     copies the stage's activation rows (and the RMSNorm weight) into shared
//     memory with one bulk copy per row: on GB300 a bulk copy of a row that other
//     SMs have just written reaches every SM far sooner than the same bytes loaded
//     by the threads;
//   - the RMSNorm statistics of a row come with it: the stages that write the
//     residual stream (O, down) add each row's sum of squares of the values they
//     store into a per-row fixed-point accumulator (integer adds: exact, so the sum
//     does not depend on the order the CTAs arrive in), and the next RMSNorm stage
//     reads it once its input is complete, so the rows are normalised, rounded to
//     bf16 and summed per group in one pass;
//   - the consumers then run the stage's blocks in rounds (R blocks side by side, the
//     warps split evenly over them), sum each block's warps, apply the epilogue
//     (SwiGLU, residual add, bf16 store) and arrive on the stage's counter;
//   - in the QKV stage only the Q blocks feed a later stage (O); the K and V blocks
//     are computed after the CTA has arrived, by CTAs that have no block in O.
//
// Every wait is bounded; a wait that gives up records TF_E_TIMEOUT in the status
// word, which every spinning CTA also polls, so the whole grid leaves promptly.
// The last CTA to finish resets the counters and accumulators, so the workspace is
// left as found.
#include "tfq_internal.h"
#include "tfq_ptx.cuh"
#include "tfq_qproj.cuh"

namespace tfq {
namespace {

constexpr int kChainWarps = 12;
constexpr int kChainMaxR = 4;  // blocks side by side in a round; divides kChainWarps
static_assert(kChainWarps % kChainMaxR == 0, "every round's blocks get the same number of warps");
constexpr int kChainThreads = (kChainWarps + 1) * 32;
constexpr int kChainBarAll = 15;  // named barrier of the consumer warps; 1..4 are team barriers
constexpr int kArriveThread = (kChainWarps - 1) * 32;  // lane 0 of the last consumer warp

// shared-memory offsets below 512 bytes
constexpr int kOffFull = 0;     // full[16]
constexpr int kOffEmpty = 128;  // empty[16]
constexpr int kOffXbar = 256;   // activation copy barrier
constexpr int kOffFlags = 264;  // [0] abort, [1] its snapshot
constexpr int kOffInv = 288;    // inv_rms[8]

struct StageDesc {
    const uint8_t* w0;
    const uint8_t* w1;
    const uint16_t* x;
    const uint16_t* gamma;
    const uint16_t* res;
    uint16_t* y;
    int64_t ldx, ldr, ldy;
    int N, K, n_rb, groups, mats;
    int n_crit;       // blocks [0, n_crit) feed a later stage; the rest are computed after arriving
    int n_next;       // CTAs with a block in the next stage (the deferred blocks go to the others)
    int in_stage;     // stage that wrote x (-1: the step's input)
    int res_stage;    // stage that wrote res (-1: none or the step's input)
    const unsigned long long* ssq_in;  // per-row sums of squares of x (RMSNorm stages after the first), or null
    unsigned long long* ssq_out;       // where this stage adds its outputs' per-row sums of squares, or null
};

// Fixed-point scale of the per-row sums of squares: 2^16 units per 1.0.
constexpr float kSsqScale = 65536.f;

__device__ __forceinline__ uint16_t* act_ptr(const ChainParams& p, int role, int l)
{
    return p.buf[role] + (int64_t)l * p.lstride[role] + (int64_t)(l & 1) * p.astride[role];
}

__device__ __forceinline__ StageDesc stage_desc(const ChainParams& p, int s)
{
    StageDesc d;
    const int l = s >> 2;
    const int kind = s & 3;
    const uint16_t* h_in = l == 0 ? p.x : act_ptr(p, 3, l - 1);  // residual stream entering layer l
    const int h_stage = l == 0 ? -1 : 4 * l - 1;
    const int qkv_n = p.Q + 2 * p.KV;
    d.w1 = nullptr;
    d.gamma = nullptr;
    d.res = nullptr;
    d.ldr = 0;
    d.mats = 1;
    d.res_stage = -1;
    d.in_stage = s - 1;
    d.ssq_in = nullptr;
    d.ssq_out = nullptr;
    if (kind == 0) {
        d.w0 = p.layer[l].qkv;
        d.x = h_in;
        d.in_stage = h_stage;
        d.ldx = p.D;
        d.gamma = p.layer[l].attn_norm;
        d.ssq_in = l > 0 ? p.ssq + (size_t)(2 * l) * kMaxM : nullptr;  // layer 0: from the staged rows
        d.y = act_ptr(p, 0, l);
        d.N = qkv_n;
        d.ldy = qkv_n;
        d.K = p.D;
    } else if (kind == 1) {
        d.w0 = p.layer[l].o;
        d.x = act_ptr(p, 0, l);
        d.ldx = qkv_n;
        d.res = h_in;
        d.res_stage = h_stage;
        d.ldr = p.D;
        d.y = act_ptr(p, 1, l);
        d.ssq_out = p.ssq + (size_t)(2 * l + 1) * kMaxM;
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
        d.ssq_in = p.ssq + (size_t)(2 * l + 1) * kMaxM;
        d.y = act_ptr(p, 2, l);
        d.N = p.F;
        d.ldy = p.F;
        d.K = p.D;
    } else {
        d.w0 = p.layer[l].down;
        d.x = act_ptr(p, 2, l);
        d.ldx = p.F;
        d.res = act_ptr(p, 1, l);
        d.res_stage = s - 2;
        d.ldr = p.D;
        d.y = act_ptr(p, 3, l);
        d.ssq_out = l + 1 < p.L ? p.ssq + (size_t)(2 * (l + 1)) * kMaxM : nullptr;
        d.N = p.D;
        d.ldy = p.D;
        d.K = p.F;
    }
    d.n_rb = (d.N + kRowsPerBlock - 1) / kRowsPerBlock;
    d.groups = d.K / kGroup;
    // the Q blocks of the QKV stage are the only ones a later stage reads (when Q is a
    // whole number of blocks, so that no block mixes Q and K columns)
    d.n_crit = (kind == 0 && p.Q % kRowsPerBlock == 0) ? p.Q / kRowsPerBlock : d.n_rb;
    d.n_next = kind == 0 ? min(p.C, (p.D + kRowsPerBlock - 1) / kRowsPerBlock) : p.C;  // O has D / 16 blocks
    return d;
}

// The blocks of one stage owned by CTA c, as two lists walked in order:
//   critical: c, c + C, ... below n_crit
//   deferred: the K and V blocks, spread over the CTAs that have no block in the next
//             stage (so that computing them after arriving delays no next-stage work)
// and how the CTA's consumer warps walk a list: rounds of R blocks side by side, KW
// warps per block (warp cw in block r_me of the round, k-part kp), `steps` ring slots
// of cg groups per block and round.
struct PartPlan {
    int first, count, stride;
    int R, cg, KW, r_me, kp, rounds, steps;
};
// up to kChainMaxR blocks side by side (a power of two, at most the list's length)
__device__ __forceinline__ int round_width(int count)
{
    int R = 1;
    while (2 * R <= count && 2 * R <= kChainMaxR)
        R *= 2;
    return R;
}
__device__ __forceinline__ PartPlan part_plan(const StageDesc& d, int part, int c, int C, int cw)
{
    PartPlan q;
    if (part == 0) {
        q.first = c;
        q.stride = C;
        q.count = c < d.n_crit ? (d.n_crit - c + C - 1) / C : 0;
    } else {
        const int n = d.n_rb - d.n_crit;
        const int lo = d.n_next < C ? d.n_next : 0, span = C - lo;  // CTAs [lo, C)
        q.first = d.n_crit + (c - lo);
        q.stride = span;
        q.count = (c >= lo && c - lo < n) ? (n - (c - lo) + span - 1) / span : 0;
    }
    q.R = round_width(q.count);
    q.cg = kChainSlotTiles / (d.mats * q.R);
    q.KW = kChainWarps / q.R;
    q.r_me = cw / q.KW;
    q.kp = cw - q.r_me * q.KW;
    q.rounds = (q.count + q.R - 1) / q.R;
    q.steps = (d.groups + q.cg - 1) / q.cg;
    return q;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* ptr)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// Thread 0: wait until every CTA has arrived on counter `s` (bounded; gives up at
// once when another CTA has recorded a failure). s < 0: nothing to wait for.
__device__ bool grid_wait(const ChainParams& p, int s, volatile int* flags)
{
    if (s < 0)
        return true;
    if (ld_acquire_u32(p.bar + s) >= (unsigned)p.C)
        return true;
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

// Orders the reads that follow (bulk copies, which run in the async proxy) after the
// generic-proxy writes of other CTAs that an acquire has made visible.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The residual values of block rb for one lane's fragment, as raw bf16 bits (0 where
// there is none); written by other CTAs in earlier stages, so read through L2. They
// are converted only at the store, so the loads overlap the tile math.
__device__ __forceinline__ void load_residual(const StageDesc& d, int rb, int lane, int M, uint32_t (&r)[4])
{
    const int gi = lane >> 2, t = lane & 3;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int n = rb * kRowsPerBlock + gi + 8 * (v >> 1);
        const int m = 2 * t + (v & 1);
        r[v] = (d.res != nullptr && n < d.N && m < M) ? (uint32_t)__ldcg(d.res + (int64_t)m * d.ldr + n) : 0u;
    }
}

// Block rb's outputs from one lane's accumulator fragment (rows rb*16 + gi, + 8;
// activation rows 2t, 2t + 1): SwiGLU for gate/up, residual add, bf16 store; and,
// when the stage writes the residual stream, each activation row's sum of squares of
// the stored values over the block (the 8 lanes of a column pair summed in a fixed
// order), added to the row's fixed-point accumulator.
__device__ __forceinline__ void store_block(const StageDesc& d, int rb, int lane, int M, const float (&a0)[4],
                                            const float (&a1)[4], const uint32_t (&res)[4])
{
    const int gi = lane >> 2, t = lane & 3;
    float sq[2] = {0.f, 0.f};
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
            val += __uint_as_float(res[v] << 16);
        const __nv_bfloat16 b = __float2bfloat16_rn(val);
        reinterpret_cast<__nv_bfloat16*>(d.y)[(int64_t)m * d.ldy + n] = b;
        const float r = __bfloat162float(b);
        sq[v & 1] = fmaf(r, r, sq[v & 1]);
    }
    if (d.ssq_out != nullptr) {  // warp-uniform
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], o);
            sq[1] += __shfl_xor_sync(0xffffffffu, sq[1], o);
        }
        if (gi == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = 2 * t + h;
                if (m < M) {
                    const unsigned long long fx = (unsigned long long)__float2ll_rn(sq[h] * kSsqScale);
                    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(d.ssq_out + m), "l"(fx) : "memory");
                }
            }
        }
    }
}

// Consumer warps, after the rows have landed: with an RMSNorm, the per-row factor
// inv_rms[m] (already there when the row's sum of squares came with the input,
// have_inv; otherwise computed here first, a warp per row, lanes over the row in a
// fixed order, so a row normalises to the same bits whatever M is), then normalise
// and round to bf16 in place; and the group sums xs[g * 8 + m] of the values used
// (zero for rows >= M). Ends with a barrier.
__device__ void chain_prepare(uint8_t* buf, int x_rs, const uint16_t* gbuf, bool have_inv, int M, int K, float eps,
                              float* xs, float* inv_rms, int cw, int lane)
{
    const int groups = K / kGroup;
    if (gbuf != nullptr && !have_inv) {
        for (int m = cw; m < M; m += kChainWarps) {
            const uint4* row = reinterpret_cast<const uint4*>(buf + m * x_rs);
            float sq[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = lane; i < K / 8; i += 32) {
                const uint4 v = row[i];
                const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float a = bf16lo_f32(vv[q]), b = bf16hi_f32(vv[q]);
                    sq[q] = fmaf(b, b, fmaf(a, a, sq[q]));
                }
            }
            const float ss = warp_sum((sq[0] + sq[1]) + (sq[2] + sq[3]));
            if (lane == 0)
                inv_rms[m] = rsqrtf(ss / (float)K + eps);
        }
        named_bar_sync(kChainBarAll, kChainWarps * 32);
    }
    for (int i = cw * 32 + lane; i < groups * kMaxM; i += kChainWarps * 32)
        if ((i & 7) >= M)
            xs[i] = 0.f;
    // a lane handles one 8-column chunk cc of one (group, row); four per warp
    for (int base = cw * 4; base < groups * M; base += kChainWarps * 4) {
        const int pi = base + (lane >> 3);
        const int cc = lane & 7;
        const int g = pi / M, m = pi - g * M;
        const bool valid = pi < groups * M;
        float part = 0.f;
        if (valid) {
            uint4* chunk = reinterpret_cast<uint4*>(buf + m * x_rs + g * 128) + cc;
            uint4 v = *chunk;
            uint32_t vv[4] = {v.x, v.y, v.z, v.w};
            if (gbuf != nullptr) {
                const uint4 gv = *reinterpret_cast<const uint4*>(gbuf + g * kGroup + cc * 8);
                const uint32_t gg[4] = {gv.x, gv.y, gv.z, gv.w};
                const float inv = inv_rms[m];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    vv[q] = f32x2_to_bf16x2(bf16lo_f32(vv[q]) * inv * bf16lo_f32(gg[q]),
                                            bf16hi_f32(vv[q]) * inv * bf16hi_f32(gg[q]));
                *chunk = make_uint4(vv[0], vv[1], vv[2], vv[3]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                part += bf16lo_f32(vv[q]) + bf16hi_f32(vv[q]);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        if (valid && cc == 0)
            xs[g * kMaxM + m] = part;
    }
    named_bar_sync(kChainBarAll, kChainWarps * 32);
}

// 13 warps: at most 4 per SM sub-partition, whose 16K registers hold 4 x 32 x 128
template <int BITS>
__global__ void __maxnreg__(128) chain_kernel(const __grid_constant__ ChainParams p)
{
    constexpr int TILE = tile_bytes_for(BITS);
    constexpr int SLOT = kChainSlotTiles * TILE;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffFull);    // [16]
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kOffEmpty);  // [16]
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + kOffXbar);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
    float* inv_rms = reinterpret_cast<float*>(smem + kOffInv);
    float* xsum = reinterpret_cast<float*>(smem + p.xsum_off);
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    uint16_t* gbuf = reinterpret_cast<uint16_t*>(smem + p.gamma_off);
    uint8_t* xraw = smem + p.xraw_off;
    uint8_t* ring = smem + p.ring_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int S = 4 * p.L;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kChainWarps);
        }
        mbar_init(xbar, 1);
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
                for (int part = 0; part < 2 && ok; ++part) {
                    const PartPlan q = part_plan(d, part, c, p.C, 0);
                    for (int t = 0; t < q.rounds && ok; ++t) {
                        const int nv = min(q.R, q.count - t * q.R);
                        for (int k = 0; k < q.steps; ++k, ++seq) {
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
                            const int cnt = min(q.cg, d.groups - k * q.cg);
                            mbar_arrive_expect_tx(&full[slot], (uint32_t)(nv * d.mats * cnt * TILE));
                            uint8_t* sb = ring + slot * SLOT;
                            for (int r = 0; r < nv; ++r) {
                                const int64_t tile = (int64_t)(q.first + (t * q.R + r) * q.stride) * d.groups + k * q.cg;
                                bulk_g2s(sb + (r * q.cg) * TILE, d.w0 + tile * TILE, (uint32_t)(cnt * TILE),
                                         &full[slot], pol);
                                if (d.mats == 2)
                                    bulk_g2s(sb + ((q.R + r) * q.cg) * TILE, d.w1 + tile * TILE,
                                             (uint32_t)(cnt * TILE), &full[slot], pol);
                            }
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
    uint32_t phase = 0, xphase = 0;
    int nstaged = 0;
    bool alive = true;
    for (int s = 0; s < S; ++s) {
        const StageDesc d = stage_desc(p, s);
        const PartPlan q0 = part_plan(d, 0, c, p.C, cw), q1 = part_plan(d, 1, c, p.C, cw);
        if (q0.count + q1.count == 0) {  // CTA-uniform: nothing to read or write here
            if (threadIdx.x == kArriveThread && !flags[0])
                grid_arrive(p, s);
            continue;
        }
        // ---- the stage's input: wait for its writers, then one bulk copy per row
        // (and the RMSNorm weight); the row factors of the RMSNorm come with the input
        // after the first layer. The abort decision is thread 0's snapshot, so every
        // consumer warp takes it alike.
        if (threadIdx.x == 0) {
            if (!flags[0] && grid_wait(p, d.res_stage, flags) && grid_wait(p, d.in_stage, flags)) {
                fence_proxy_async_global();
                const uint32_t row_bytes = (uint32_t)d.K * 2;
                mbar_arrive_expect_tx(xbar, row_bytes * p.M + (d.gamma != nullptr ? row_bytes : 0u));
                for (int m = 0; m < p.M; ++m)
                    bulk_g2s_plain(xraw + m * p.x_rs, d.x + (int64_t)m * d.ldx, row_bytes, xbar);
                if (d.gamma != nullptr)
                    bulk_g2s_plain(gbuf, d.gamma, row_bytes, xbar);
                ++nstaged;
                // the rows' RMSNorm factors, read while the rows are on their way (all loads first)
                if (d.ssq_in != nullptr) {
                    unsigned long long v[kMaxM];
#pragma unroll
                    for (int m = 0; m < kMaxM; ++m)
                        v[m] = m < p.M ? __ldcg(d.ssq_in + m) : 0ull;
#pragma unroll
                    for (int m = 0; m < kMaxM; ++m)
                        if (m < p.M)
                            inv_rms[m] = rsqrtf((float)(long long)v[m] * (1.f / kSsqScale) / (float)d.K + p.eps);
                }
            }
            flags[1] = flags[0];
        }
        named_bar_sync(kChainBarAll, kChainWarps * 32);
        if (flags[1])
            break;
        // the first round's residual values travel while the rows are staged
        uint32_t res[4];
        load_residual(d, q0.first + q0.r_me * q0.stride, lane, (q0.kp == 0 && q0.r_me < q0.count) ? p.M : 0, res);
        {
            const bool ok = wait_or_abort(xbar, xphase, flags, p.status, p.limit_ns);
            alive = __all_sync(0xffffffffu, ok) && alive;
        }
        xphase ^= 1u;
        chain_prepare(xraw, p.x_rs, d.gamma != nullptr ? gbuf : nullptr, d.ssq_in != nullptr, p.M, d.K, p.eps, xsum,
                      inv_rms, cw, lane);

        for (int part = 0; part < 2; ++part) {
            const PartPlan& q = part == 0 ? q0 : q1;
            for (int t = 0; t < q.rounds; ++t) {
                const int kb = t * q.R + q.r_me;
                const bool valid = kb < q.count;
                const int rb = q.first + kb * q.stride;
                if (part != 0 || t != 0)
                    load_residual(d, rb, lane, (q.kp == 0 && valid) ? p.M : 0, res);
                float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
                float bcc0[4] = {0.f, 0.f, 0.f, 0.f}, bcc1[4] = {0.f, 0.f, 0.f, 0.f};  // second chain
                for (int k = 0; k < q.steps; ++k) {
                    const bool ok = alive && wait_or_abort(&full[slot], phase, flags, p.status, p.limit_ns);
                    alive = __all_sync(0xffffffffu, ok);
                    const int cnt = min(q.cg, d.groups - k * q.cg);
                    if (alive && valid) {
                        const uint8_t* sb = ring + slot * SLOT;
                        const uint8_t* t0 = sb + (q.r_me * q.cg) * TILE;
                        const uint8_t* t1 = sb + ((q.R + q.r_me) * q.cg) * TILE;
                        int j = q.kp;
                        // two tiles per iteration into separate accumulators: independent chains
                        for (; j + q.KW < cnt; j += 2 * q.KW) {
                            const int g = k * q.cg + j;
                            uint4 xa, xb, ya, yb;
                            x_frag(xraw, p.x_rs, gi, tq, g, p.M, xa, xb);
                            x_frag(xraw, p.x_rs, gi, tq, g + q.KW, p.M, ya, yb);
                            const float2 xs = *reinterpret_cast<const float2*>(xsum + g * kMaxM + 2 * tq);
                            const float2 ys = *reinterpret_cast<const float2*>(xsum + (g + q.KW) * kMaxM + 2 * tq);
                            tile_mac<BITS>(t0 + j * TILE, lane, xa, xb, xs, acc0);
                            tile_mac<BITS>(t0 + (j + q.KW) * TILE, lane, ya, yb, ys, bcc0);
                            if (d.mats == 2) {
                                tile_mac<BITS>(t1 + j * TILE, lane, xa, xb, xs, acc1);
                                tile_mac<BITS>(t1 + (j + q.KW) * TILE, lane, ya, yb, ys, bcc1);
                            }
                        }
                        if (j < cnt) {
                            const int g = k * q.cg + j;
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
                // sum the KW warps of the block (team barrier 1 + r_me); before the first
                // round, the reduction buffer was last read before a CTA-wide barrier
                if (q.KW > 1) {
                    float4* red4 = reinterpret_cast<float4*>(red);
                    if (t > 0)
                        named_bar_sync(1 + q.r_me, q.KW * 32);  // the previous round's reads of red are done
                    red4[cw * 32 + lane] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
                    if (d.mats == 2)
                        red4[kChainWarps * 32 + cw * 32 + lane] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
                    named_bar_sync(1 + q.r_me, q.KW * 32);
                    if (q.kp == 0) {
                        for (int o = 1; o < q.KW; ++o) {
                            const float4 o0 = red4[(cw + o) * 32 + lane];
                            acc0[0] += o0.x;
                            acc0[1] += o0.y;
                            acc0[2] += o0.z;
                            acc0[3] += o0.w;
                            if (d.mats == 2) {
                                const float4 o1 = red4[kChainWarps * 32 + (cw + o) * 32 + lane];
                                acc1[0] += o1.x;
                                acc1[1] += o1.y;
                                acc1[2] += o1.z;
                                acc1[3] += o1.w;
                            }
                        }
                    }
                }
                if (q.kp == 0 && valid && alive)
                    store_block(d, rb, lane, p.M, acc0, acc1, res);
            }
            if (part == 0) {
                // every critical store of this CTA for stage s is issued: arrive (every
                // consumer warp gets here, whatever its own waits returned). The release
                // holds the arriving thread until the CTA's stores are visible, so the last
                // consumer warp arrives, not thread 0, which waits for the next input.
                __syncwarp();
                named_bar_sync(kChainBarAll, kChainWarps * 32);
                if (threadIdx.x == kArriveThread && !flags[0])
                    grid_arrive(p, s);
            }
        }
        // the staged rows and the reduction buffer are reused by the next stage
        __syncwarp();
        named_bar_sync(kChainBarAll, kChainWarps * 32);
    }
    // no activation copy may still be in flight when the CTA leaves (after an abort)
    if (threadIdx.x == 0 && flags[0] && nstaged > 0)
        mbar_wait_bounded(xbar, xphase ^ 1u, p.limit_ns);
    // the last CTA to finish resets every counter and accumulator (nobody reads them any
    // more). The thread that made this CTA's stage arrivals counts it out, so that its
    // last arrival is ordered before the reset.
    if (threadIdx.x == kArriveThread && !flags[0]) {
        __threadfence();
        if (atomicAdd(p.bar + S, 1u) == (unsigned)(p.C - 1)) {
            for (int i = 0; i <= S; ++i)
                p.bar[i] = 0u;
            for (int i = 0; i < 2 * p.L * kMaxM; ++i)
                p.ssq[i] = 0ull;
            __threadfence();
        }
    }
}

}  // namespace

size_t chain_smem(int bits, int kmax, int dmax, int* nst, int* x_rs, int* xsum_off, int* red_off, int* gamma_off,
                  int* xraw_off, int* ring_off)
{
    const size_t slot = (size_t)kChainSlotTiles * tile_bytes_for(bits);
    *xsum_off = 512;
    *red_off = 512 + kChainMaxGroups * kMaxM * 4;                   // 2048
    *gamma_off = *red_off + 2 * kChainWarps * 32 * 16;              // two float4 per lane and warp
    *xraw_off = (int)((*gamma_off + (size_t)dmax * 2 + 127) / 128 * 128);
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
