// The projection of one 16-row block by one CTA, for calls whose every row block fits a
// CTA whole (one K split, at most a few hundred row blocks): the common case of a decoder
// step, where each projection is one dependent stage and its time is latency, not bytes.
//
//   thread 0        issues the row block's weight copy (one bulk copy per matrix: a row
//                   block's groups are contiguous in the packed layout) before the kernel
//                   waits for the previous one (programmatic dependent launch), and every
//                   thread loads its chunks of the RMSNorm gamma: weights never depend on
//                   the previous kernel, so they stream during its tail
//   all NW warps    stage the activation rows straight from L2 into registers (normalised
//                   when an RMSNorm is folded in; rotated when an input Hadamard transform
//                   is), form the per-group sums, then warp w
//                   multiplies groups w, w + NW, ... of the row block (two tiles per
//                   iteration into independent accumulators), the warps' sums are added
//                   in warp order through shared memory, and warp 0 applies the epilogue
//                   (SwiGLU, residual: loaded right after the wait, so its L2 round trip
//                   overlaps the staging and the tiles) and stores.
//
// The same tile math, activation staging and epilogue as the general schedules, without
// their machinery (segment lists, rounds, a weight ring, split-K partial sums): one
// bounded wait on one barrier, three CTA barriers. Shared memory: the row block's tiles,
// the staged rows and the warps' sums.
//
// Included by tfq_qproj.cuh, inside namespace tfq, after the helpers it uses.
#pragma once

constexpr int kBarStage = 1;  // named barrier of the compute warps

// gamma's chunks j 32 + lane (j < 4) for the RMSNorm staging below. gamma is a weight:
// it does not depend on the previous kernel, so this runs before the grid-dependency
// wait and its latency hides behind it.
__device__ __forceinline__ void stage_gamma_prefetch(const uint16_t* gamma, int K, int lane, uint4 (&gv)[4])
{
    const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        gv[j] = j * 32 + lane < K / 8 ? ld_nc_v4_here(g4 + j * 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
}

// The rows x[m][0, K) (m < M, K <= 1024), normalised with the prefetched gamma and
// rounded to bf16 into buf (row stride x_rs), with the per-group sums into xs[g * 8 + m]
// (zero for rows >= M): one warp a row, four chunks a lane, the row's sum of squares a
// warp reduction in an order that does not depend on M (the same arithmetic as the
// other schedules' staging). Ends with a barrier of the NW warps.
template <int NW>
__device__ __forceinline__ void stage_rows_norm(const uint16_t* x, int64_t ldx, int K, const uint4 (&gv)[4], float eps,
                                                int x_rs, uint8_t* buf, int M, float* xs, int warp, int lane)
{
    const int nch = K / 8;
    for (int i = warp * 32 + lane; i < (K / kGroup) * kMaxM; i += NW * 32)
        if ((i & 7) >= M)
            xs[i] = 0.f;
    for (int m = warp; m < M; m += NW) {
        const uint4* x4 = reinterpret_cast<const uint4*>(x + (int64_t)m * ldx);
        uint4 v[4];
        float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = j * 32 + lane < nch ? __ldcg(x4 + j * 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t vv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = bf16lo_f32(vv[q]), b = bf16hi_f32(vv[q]);
                sq[q] = fmaf(b, b, fmaf(a, a, sq[q]));
            }
        }
        const float inv = rsqrtf(warp_sum((sq[0] + sq[1]) + (sq[2] + sq[3])) / (float)K + eps);
        float part[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = j * 32 + lane;
            const uint32_t xv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            const uint32_t gg[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
            uint32_t vv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                vv[q] = f32x2_to_bf16x2(bf16lo_f32(xv[q]) * inv * bf16lo_f32(gg[q]),
                                        bf16hi_f32(xv[q]) * inv * bf16hi_f32(gg[q]));
            float s = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                s += bf16lo_f32(vv[q]) + bf16hi_f32(vv[q]);
            part[j] = s;
            if (c < nch)
                *reinterpret_cast<uint4*>(buf + m * x_rs + c * 16) = make_uint4(vv[0], vv[1], vv[2], vv[3]);
        }
        // the group sums: lane l holds chunks j 32 + l (j < 4) of four groups; a butterfly
        // over the 8 lanes of a group (2 + 1 + 1 shuffles for the four, not 3 each) leaves
        // lanes l and l ^ 1 with the sum for j = 2 bit2(l) + bit1(l), added in the order of
        // x_put_chunk's reduction (the same bits); the even lane stores it
        const bool h4 = (lane & 4) != 0, h2 = (lane & 2) != 0;
        float b[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float r = __shfl_xor_sync(0xffffffffu, h4 ? part[i] : part[i + 2], 4);
            b[i] = (h4 ? part[i + 2] : part[i]) + r;
        }
        const float r2 = __shfl_xor_sync(0xffffffffu, h2 ? b[0] : b[1], 2);
        const float cq = (h2 ? b[1] : b[0]) + r2;
        const float sum = cq + __shfl_xor_sync(0xffffffffu, cq, 1);
        const int jj = (h4 ? 2 : 0) + (h2 ? 1 : 0), cc = jj * 32 + lane;
        if ((lane & 1) == 0 && cc < nch)
            xs[(cc >> 3) * kMaxM + m] = sum;
    }
    named_bar_sync(kBarStage, NW * 32);
}

// NW warps: 8 (two CTAs an SM) or 16 (calls with at most one row block an SM)
template <int BITS, bool DUAL, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 2 : 1) qstage_kernel(const __grid_constant__ QProjParams p)
{
    constexpr int MATS = DUAL ? 2 : 1;
    constexpr int TILE = tile_bytes_for(BITS);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + QSmem::kFullOff);
    float* xsum = reinterpret_cast<float*>(smem + QSmem::kXsumOff);
    float4* red4 = reinterpret_cast<float4*>(smem + p.red_off);  // [MATS][NW][32]
    uint8_t* xraw = smem + p.xraw_off;
    uint8_t* wt = smem + p.stage_off;  // [MATS][groups] tiles

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = lane >> 2, tq = lane & 3;
    const int rb = blockIdx.x;
    const int G = p.groups;

    if (threadIdx.x == 0) {
        mbar_init(wbar, 1);
        fence_mbar_init();
        const uint64_t pol = policy_evict_first();
        const uint32_t bytes = (uint32_t)(G * TILE);
        mbar_arrive_expect_tx(wbar, bytes * MATS);
        bulk_g2s(wt, p.w0 + (int64_t)rb * G * TILE, bytes, wbar, pol);
        if constexpr (DUAL)
            bulk_g2s(wt + (size_t)G * TILE, p.w1 + (int64_t)rb * G * TILE, bytes, wbar, pol);
    }
    pdl_launch_dependents();
    // gamma (a weight) before the wait
    uint4 gpre[4];
    if (p.gamma != nullptr)
        stage_gamma_prefetch(p.gamma, p.K, lane, gpre);
    pdl_wait();

    // warp 0's residual values (it stores the outputs), raw bits: the L2 round trip runs
    // while the rows are staged and the tiles multiplied
    uint32_t res[4] = {0u, 0u, 0u, 0u};
    if (warp == 0 && p.residual != nullptr) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int n = rb * kRowsPerBlock + gi + 8 * (v >> 1);
            const int m = 2 * tq + (v & 1);
            if (n < p.N && m < p.M)
                res[v] = (uint32_t)__ldcg(p.residual + (int64_t)m * p.ldr + n);
        }
    }

    // ---- the activation rows (and their group sums), straight from L2; ends with a barrier
    // that also publishes the barrier initialisation above
    if (p.gamma != nullptr)
        stage_rows_norm<NW>(p.x, p.ldx, p.K, gpre, p.eps, p.x_rs, xraw, p.M, xsum, warp, lane);
    else
        x_direct_raw<4>(p.x, p.ldx, p.K, nullptr, p.eps, p.x_rs, xraw, p.M, xsum, nullptr, warp, lane, NW, kBarStage);
    if (p.rht != nullptr)  // the input Hadamard transform, a pass over the staged rows
        x_rht(xraw, p.x_rs, xsum, p.M, 0, G, p.rht, warp, lane, NW, kBarStage);

    // ---- the row block's tiles
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0u, p.limit_ns));
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    float bcc0[4] = {0.f, 0.f, 0.f, 0.f}, bcc1[4] = {0.f, 0.f, 0.f, 0.f};  // second chain
    if (ok) {
        const uint8_t* t0 = wt;
        const uint8_t* t1 = wt + (size_t)G * TILE;
        int g = warp;
        for (; g + NW < G; g += 2 * NW) {
            uint4 xa, xb, ya, yb;
            x_frag(xraw, p.x_rs, gi, tq, g, p.M, xa, xb);
            x_frag(xraw, p.x_rs, gi, tq, g + NW, p.M, ya, yb);
            const float2 xs = *reinterpret_cast<const float2*>(xsum + g * kMaxM + 2 * tq);
            const float2 ys = *reinterpret_cast<const float2*>(xsum + (g + NW) * kMaxM + 2 * tq);
            tile_mac<BITS>(t0 + g * TILE, lane, xa, xb, xs, acc0);
            tile_mac<BITS>(t0 + (g + NW) * TILE, lane, ya, yb, ys, bcc0);
            if constexpr (DUAL) {
                tile_mac<BITS>(t1 + g * TILE, lane, xa, xb, xs, acc1);
                tile_mac<BITS>(t1 + (g + NW) * TILE, lane, ya, yb, ys, bcc1);
            }
        }
        if (g < G) {
            uint4 xa, xb;
            x_frag(xraw, p.x_rs, gi, tq, g, p.M, xa, xb);
            const float2 xs = *reinterpret_cast<const float2*>(xsum + g * kMaxM + 2 * tq);
            tile_mac<BITS>(t0 + g * TILE, lane, xa, xb, xs, acc0);
            if constexpr (DUAL)
                tile_mac<BITS>(t1 + g * TILE, lane, xa, xb, xs, acc1);
        }
    } else if (lane == 0) {
        atomicCAS(p.status, 0, TF_E_TIMEOUT);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc0[i] += bcc0[i];
        acc1[i] += bcc1[i];
    }
    // ---- the warps' sums, in warp order, by warp 0; then the epilogue
    red4[warp * 32 + lane] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
    if constexpr (DUAL)
        red4[(NW + warp) * 32 + lane] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
    named_bar_sync(kBarStage, NW * 32);
    if (warp == 0) {
#pragma unroll
        for (int q = 1; q < NW; ++q) {
            const float4 o0 = red4[q * 32 + lane];
            acc0[0] += o0.x;
            acc0[1] += o0.y;
            acc0[2] += o0.z;
            acc0[3] += o0.w;
            if constexpr (DUAL) {
                const float4 o1 = red4[(NW + q) * 32 + lane];
                acc1[0] += o1.x;
                acc1[1] += o1.y;
                acc1[2] += o1.z;
                acc1[3] += o1.w;
            }
        }
        if constexpr (BITS == kNvfp4) {  // the matrices' global scales
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc0[i] *= p.wscale0;
                if constexpr (DUAL)
                    acc1[i] *= p.wscale1;
            }
        }
        if (ok) {
            // rows rb*16 + gi (+ 8) of the block, activation rows 2 tq (+ 1): SwiGLU for
            // gate/up, residual add, store
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int n = rb * kRowsPerBlock + gi + 8 * (v >> 1);
                const int m = 2 * tq + (v & 1);
                if (n >= p.N || m >= p.M)
                    continue;
                float val = acc0[v];
                if constexpr (DUAL)
                    val = val / (1.f + expf(-val)) * acc1[v];
                if (p.residual != nullptr)
                    val += __uint_as_float(res[v] << 16);
                const int64_t idx = (int64_t)m * p.ldy + n;
                if (p.y_f32)
                    static_cast<float*>(p.y)[idx] = val;
                else
                    static_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(val);
            }
        }
    }
    // a wait that gave up: no copy may still be in flight when the CTA leaves
    if (!ok && threadIdx.x == 0)
        mbar_wait_bounded(wbar, 0u, p.limit_ns);
}

template <int BITS, bool DUAL, int NW>
cudaError_t launch_qstage_w(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    auto kern = qstage_kernel<BITS, DUAL, NW>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.C, 1, 1);
    cfg.blockDim = dim3(NW * 32, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BITS, bool DUAL>
cudaError_t launch_qstage(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    return plan.nw == 16 ? launch_qstage_w<BITS, DUAL, 16>(plan, p, stream, pdl)
                         : launch_qstage_w<BITS, DUAL, 8>(plan, p, stream, pdl);
}
