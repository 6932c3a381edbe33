// Streaming schedule of one large projection (a single matrix, one problem):
// y[m][n] = sum_k xn[m][k] * (s q + b)[n][k], for calls with many more weight bytes
// than one kernel launch hides.
//
// The units (16-row x 64-column tiles) of each K split form a row-block-major
// sequence; the grid is S groups of C / S CTAs, group s taking split s, and each CTA
// an exact 1 / (C / S) share of its split's units (stream-K). A CTA therefore needs
// only its split's slice of the activation rows, staged once.
//
//   producer warp   one lane issues bulk async copies (TMA engine) of the CTA's
//                   tiles, CH at a time, into an NS-deep ring, from the first
//                   instruction on: the weights do not depend on the previous kernel,
//                   so with programmatic dependent launch they stream while that
//                   kernel finishes.
//   compute warps   (W) wait for the previous grid, stage the activation slice
//                   (normalised when an RMSNorm is folded in) with its per-group
//                   sums, then take tiles w, w + W, w + 2W, ... of the share, tile j
//                   into accumulator (j / W) mod 2. When a warp's next tile belongs
//                   to a later row block, it hands its sum for the finished one to
//                   the reducer through a ring of NR shared-memory slots (one float4
//                   per lane and warp), with zero for any row block it had no tile of.
//   reducer warp    sums the W hand-offs of each row block in warp order as soon as
//                   they are complete, and stores the row block (whole and unsplit)
//                   or writes its fp32 partial slot. After the last row block, it
//                   bumps the arrival counters of the partial row blocks together.
//   last contributors  of a row block (arrival count complete) sum its slots in
//                   (split, contributor) order, store, and zero the slots and the
//                   counter; the compute warps and the reducer share these sums.
//
// No CTA-wide barrier after the activation staging; every wait is bounded and an
// expired wait sets TF_E_TIMEOUT and makes the CTA leave (after the producer has
// drained its copies). Results do not depend on M: the split count and the order of
// every sum are fixed by the weights' shape and the SM count alone.
#pragma once

#include "tfq_qproj.cuh"

namespace tfq {

struct StreamSmem {
    static constexpr int kFull = 0;      // full[8]: a ring slot's copies landed
    static constexpr int kEmpty = 64;    // empty[8]: the compute warps are done with a slot
    static constexpr int kRFull = 128;   // rfull[8]: all hand-offs of a row block written
    static constexpr int kREmpty = 192;  // rempty[8]: the reducer has read a hand-off slot
    static constexpr int kFlag = 256;    // [0] abort
    static constexpr int kSsPart = 272;  // RMSNorm: per-warp sums of squares [16]
    static constexpr int kXs = 384;      // per-group activation sums [groups staged][8]
    static constexpr int kMaxRing = 8;
    static constexpr int kMaxRed = 8;
};

constexpr int kStreamBarX = 1;      // named barrier of the compute warps (activation staging)
constexpr int kStreamBarFinal = 2;  // compute warps and reducer, before the last contributors' sums

template <int BITS, int W>
__global__ void __launch_bounds__((W + 2) * 32, W <= 8 ? 2 : 1) qstream_kernel(const __grid_constant__ QProjParams p)
{
    constexpr int TILE = tile_bytes_for(BITS);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + StreamSmem::kFull);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + StreamSmem::kEmpty);
    uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + StreamSmem::kRFull);
    uint64_t* rempty = reinterpret_cast<uint64_t*>(smem + StreamSmem::kREmpty);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + StreamSmem::kFlag);
    float* ss_part = reinterpret_cast<float*>(smem + StreamSmem::kSsPart);
    float* xs = reinterpret_cast<float*>(smem + StreamSmem::kXs);
    uint8_t* xbuf = smem + p.xraw_off;
    float4* red = reinterpret_cast<float4*>(smem + p.red_off);
    uint8_t* ring = smem + p.stage_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = p.nst, CH = p.cg, NR = p.pw;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], W);
        }
        for (int i = 0; i < NR; ++i) {  // one arrival per warp (after its lanes' accesses)
            mbar_init(&rfull[i], W);
            mbar_init(&rempty[i], 1);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // ---- this CTA's share: split s, units [u0, u1) of the split's n_rb * Gs
    const int Cg = p.C / p.S;
    const int s = (int)blockIdx.x / Cg, cl = (int)blockIdx.x - s * Cg;
    const uint32_t Us = (uint32_t)p.n_rb * (uint32_t)p.Gs;
    const int u0 = (int)Part::muldiv(Us, (uint32_t)cl, (uint32_t)Cg);
    const int u1 = (int)Part::muldiv(Us, (uint32_t)cl + 1u, (uint32_t)Cg);
    const int nU = u1 - u0;
    const int nch = (nU + CH - 1) / CH;
    const int rb0 = u0 / p.Gs;
    const int nseg = nU > 0 ? (u1 - 1) / p.Gs - rb0 + 1 : 0;

    // ------------------------------------------------------------ producer
    if (warp == W) {
        if (lane == 0 && nU > 0) {
            const uint64_t pol = policy_evict_first();
            const uint8_t* wbase = p.w0 + (int64_t)s * p.Gs * TILE;
            int k = 0;
            for (; k < nch; ++k) {
                const int slot = k % NS;
                if (!wait_or_abort(&empty[slot], (uint32_t)((k / NS) & 1) ^ 1u, flags, p.status, p.limit_ns))
                    break;
                const int a = u0 + k * CH, cnt = min(CH, u1 - a);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(cnt * TILE));
                uint8_t* dst = ring + (size_t)slot * CH * TILE;
                int rb = a / p.Gs, g = a - rb * p.Gs, left = cnt;
                while (left > 0) {  // one copy per row block piece (contiguous in the packed layout)
                    const int len = min(p.Gs - g, left);
                    bulk_g2s(dst, wbase + ((int64_t)rb * p.groups + g) * TILE, (uint32_t)(len * TILE), &full[slot], pol);
                    dst += len * TILE;
                    left -= len;
                    ++rb;
                    g = 0;
                }
            }
            // no copy may still be in flight when the CTA leaves (also after an abort:
            // copies complete by themselves, so this wait ignores the abort flag)
            for (int q = max(0, k - NS); q < k; ++q)
                mbar_wait_bounded(&full[q % NS], (uint32_t)(q / NS) & 1u, p.limit_ns);
        }
        return;
    }

    Part pt;  // the stream-K partition of one split (every split has the same)
    pt.items = p.n_rb;
    pt.U = Us;
    pt.C = Cg;
    pt.per_p = 0;
    pt.per_ps = 0;
    pt.Gs = p.Gs;
    pt.aligned = false;
    pt.inv_U = 1.f / (float)max(Us, 1u);

    int* lastf = reinterpret_cast<int*>(smem + p.last_off);  // per row block of the CTA: ours to sum
    // a row block goes to a partial slot unless it is unsplit and wholly this CTA's
    auto partial = [&](int rb) { return !(p.S == 1 && pt.contributors((int64_t)rb * p.Gs) == 1); };

    if (warp == W + 1) {
        // ------------------------------------------------------------ reducer
        pdl_wait();  // partial slots, counters and outputs are shared with the previous call
        bool alive = true;
        for (int js = 0; js < nseg; ++js) {
            const int slot = js % NR;
            const bool ok = wait_or_abort(&rfull[slot], (uint32_t)(js / NR) & 1u, flags, p.status, p.limit_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                alive = false;
                break;
            }
            float4 t = red[(slot * W) * 32 + lane];
#pragma unroll
            for (int w = 1; w < W; ++w) {
                const float4 o = red[(slot * W + w) * 32 + lane];
                t.x += o.x;
                t.y += o.y;
                t.z += o.z;
                t.w += o.w;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&rempty[slot]);
            const int rb = rb0 + js;
            if (!partial(rb)) {
                const float a[4] = {t.x, t.y, t.z, t.w};
                store_outputs<false, false>(p, 0, p.M, rb * kRowsPerBlock, lane, a, a);
            } else {
                const int k = min(cl - pt.cta_of((int64_t)rb * p.Gs), p.kmax - 1);  // k < kmax by construction
                __stcg(reinterpret_cast<float4*>(p.partials +
                                                 ((((int64_t)s * p.n_rb + rb) * p.kmax + k) * 32 + lane) * 4),
                       t);
            }
        }
        // ---- arrival counters of the partial row blocks, a lane each
        if (alive) {
            __threadfence();
            __syncwarp();
        }
        for (int js = lane; js < nseg; js += 32) {
            int is_last = 0;
            if (alive && partial(rb0 + js)) {
                const int rb = rb0 + js;
                const int old = atomicAdd(&p.counters[rb], 1);
                is_last = old == p.S * pt.contributors((int64_t)rb * p.Gs) - 1;
            }
            lastf[js] = is_last;
        }
    } else {
    // ------------------------------------------------------------ compute warps
    const int w = warp;
    const int gi = lane >> 2, tq = lane & 3;
    pdl_wait();
    const bool norm = p.gamma != nullptr;  // then S == 1 and the whole row is staged
    // rows M..7 of the buffer read as zero (no per-tile row clamp); x_direct_raw's
    // closing barrier orders these stores before any fragment load
    for (int i = (w * 32 + lane) * 16 + p.M * p.x_rs; i < kMaxM * p.x_rs; i += W * 32 * 16)
        *reinterpret_cast<uint4*>(xbuf + i) = make_uint4(0u, 0u, 0u, 0u);
    x_direct_raw<4>(p.x + (norm ? 0 : (int64_t)s * p.Gs * kGroup), p.ldx, norm ? p.K : p.Gs * kGroup, p.gamma, p.eps,
                    p.x_rs, xbuf, p.M, xs, ss_part, w, lane, W, kStreamBarX);
    if (p.rht != nullptr)  // input Hadamard transform of the staged slice
        x_rht(xbuf, p.x_rs, xs, p.M, norm ? 0 : s * p.Gs, norm ? p.groups : p.Gs, p.rht, w, lane, W, kStreamBarX);

    bool alive = true;
    int cur = 0;  // row block (relative to rb0) the accumulators belong to
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    // hand the accumulators to row block cur, zero to the ones before `upto`
    auto flush_to = [&](int upto) {
        for (; cur < upto; ++cur) {
            const int slot = cur % NR;
            const bool ok =
                alive && wait_or_abort(&rempty[slot], (uint32_t)((cur / NR) & 1) ^ 1u, flags, p.status, p.limit_ns);
            alive = __all_sync(0xffffffffu, ok);
            if (!alive)
                return;
            red[(slot * W + w) * 32 + lane] =
                make_float4(acc0[0] + acc1[0], acc0[1] + acc1[1], acc0[2] + acc1[2], acc0[3] + acc1[3]);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&rfull[slot]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc0[i] = 0.f;
                acc1[i] = 0.f;
            }
        }
    };

    // this warp's next unit: u0 + w, then every W-th
    int rb = (u0 + w) / p.Gs;
    int g = u0 + w - rb * p.Gs;
    const int Gs = p.Gs;
    for (int k = 0; k < nch && alive; ++k) {
        const int slot = k % NS;
        const bool ok = wait_or_abort(&full[slot], (uint32_t)(k / NS) & 1u, flags, p.status, p.limit_ns);
        alive = __all_sync(0xffffffffu, ok);
        if (!alive)
            break;
        const uint8_t* base = ring + (size_t)slot * CH * TILE;
        const int jend = min(CH, nU - k * CH);
        for (int jj = w; jj < jend; jj += 2 * W) {
            // tile A = jj (accumulator 0), tile B = jj + W (accumulator 1)
            if (rb - rb0 != cur) {
                flush_to(rb - rb0);
                if (!alive)
                    break;
            }
            int rbB = rb, gB = g + W;
            while (gB >= Gs) {
                gB -= Gs;
                ++rbB;
            }
            const bool hasB = jj + W < jend;
            uint4 xa, xb;
            x_frag8(xbuf, p.x_rs, lane, g, xa, xb);
            const float2 xsa = *reinterpret_cast<const float2*>(xs + g * kMaxM + 2 * tq);
            if (hasB && rbB == rb) {
                uint4 ya, yb;
                x_frag8(xbuf, p.x_rs, lane, gB, ya, yb);
                const float2 xsb = *reinterpret_cast<const float2*>(xs + gB * kMaxM + 2 * tq);
                tile_mac_chain<BITS>(base + jj * TILE, lane, xa, xb, xsa, acc0);
                tile_mac_chain<BITS>(base + (jj + W) * TILE, lane, ya, yb, xsb, acc1);
            } else {
                tile_mac_chain<BITS>(base + jj * TILE, lane, xa, xb, xsa, acc0);
                if (hasB) {
                    flush_to(rbB - rb0);
                    if (!alive)
                        break;
                    uint4 ya, yb;
                    x_frag8(xbuf, p.x_rs, lane, gB, ya, yb);
                    const float2 xsb = *reinterpret_cast<const float2*>(xs + gB * kMaxM + 2 * tq);
                    tile_mac_chain<BITS>(base + (jj + W) * TILE, lane, ya, yb, xsb, acc1);
                }
            }
            rb = rbB;
            g = gB + W;
            while (g >= Gs) {
                g -= Gs;
                ++rb;
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[slot]);
    }
    if (alive)
        flush_to(nseg);
    }

    // ------------------------------------------------------------ last contributors
    // the row blocks this CTA arrived last on are summed (slots in fixed order),
    // stored and reset by the compute warps and the reducer together; every one of
    // them reaches this barrier exactly once, also after an abort
    named_bar_sync(kStreamBarFinal, (W + 1) * 32);
    for (int js = warp == W + 1 ? W : warp; js < nseg; js += W + 1) {
        if (!lastf[js])
            continue;
        const int rb = rb0 + js;
        __threadfence();
        float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
        sum_partials<false, 8>(p, pt, 0, rb, lane, t0, t1);
        store_outputs<false, false>(p, 0, p.M, rb * kRowsPerBlock, lane, t0, t1);
        if (lane == 0)
            p.counters[rb] = 0;
    }
}

template <int BITS, int W>
cudaError_t launch_qstream_w(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    auto kern = qstream_kernel<BITS, W>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.C, 1, 1);
    cfg.blockDim = dim3((W + 2) * 32, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BITS>
cudaError_t launch_qstream(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    return plan.nw == 8 ? launch_qstream_w<BITS, 8>(plan, p, stream, pdl)
                        : launch_qstream_w<BITS, 16>(plan, p, stream, pdl);
}

}  // namespace tfq
