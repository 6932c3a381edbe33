// MoE routing and combine kernels, and the bounded-wait self-test kernel.
//
// Routing (uzu page, "Internals 1" table, mlp row: MixtureOfExperts with a
// routing function; "radix top-k" is among its kernels): per row, the top_k
// experts by fp32 logit, descending, equal logits to the lower index; weights
// are the softmax of the selected logits (computed in double, stored fp32).
// The router then buckets the (row, slot) pairs by expert so that every
// selected expert's weights are streamed once with all of its rows as MMA
// columns, and writes the inverse map used by the deterministic combine.
#include "tfq_internal.h"
#include "tfq_ptx.cuh"

namespace tfq {
namespace {

constexpr int kRouteThreads = 1024;

__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const float* __restrict__ logits, int M, int E,
                                                                  int top_k, int32_t* __restrict__ idx_out,
                                                                  float* __restrict__ w_out, MoeMeta* meta)
{
    __shared__ int32_t sel[kMaxM * 8];
    __shared__ int32_t cnt[1024];
    __shared__ int32_t warp_tot[32];

    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- top-k per row: k rounds of a warp arg-max over the not-yet-taken experts
    if (warp < M) {
        const float* l = logits + (int64_t)warp * E;
        uint32_t taken = 0;  // bit i: expert lane + 32 i taken (E <= 1024)
        float vals[32];
        const int per = (E + 31) / 32;
        for (int i = 0; i < per; ++i) {
            const int e = lane + 32 * i;
            vals[i] = e < E ? __ldcg(l + e) : 0.f;
        }
        float top = 0.f, mine = 0.f;  // the largest selected logit; lane j: the j-th one
        for (int j = 0; j < top_k; ++j) {
            float bv = 0.f;
            int be = -1;
            for (int i = 0; i < per; ++i) {
                const int e = lane + 32 * i;
                if (e >= E || ((taken >> i) & 1u))
                    continue;
                if (be < 0 || vals[i] > bv) {  // ascending e: strict '>' keeps the lower index
                    bv = vals[i];
                    be = e;
                }
            }
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane)
                taken |= 1u << (be >> 5);
            if (j == 0)
                top = bv;
            if (lane == j)
                mine = bv;
            if (lane == 0)
                sel[warp * 8 + j] = be;
        }
        // softmax over the selected logits: lane j takes exp(l_j - l_0) <= 1 (the k
        // exponentials run side by side; 2 ulp each), every lane adds them in ascending j
        // with Knuth's TwoSum, so the denominator is exact to about 2^-48 as the pair
        // (s, c), and lane j divides its own: w = e / s * (1 - c / s)
        const float ex = lane < top_k ? expf(mine - top) : 0.f;
        float s_hi = 0.f, s_lo = 0.f;
        for (int j = 0; j < top_k; ++j) {
            const float a = __shfl_sync(0xffffffffu, ex, j);
            const float t = s_hi + a;
            const float bp = t - s_hi;
            s_lo += (s_hi - (t - bp)) + (a - bp);
            s_hi = t;
        }
        __syncwarp();
        if (lane < top_k) {
            const float q = ex / s_hi;
            const float w = fmaf(-q, s_lo / s_hi, q);
            idx_out[warp * top_k + lane] = sel[warp * 8 + lane];
            w_out[warp * top_k + lane] = w;
            meta->w[warp * 8 + lane] = w;
        }
    }
    __syncthreads();

    // ---- bucket (row, slot) pairs by expert; active experts get slots in ascending expert order
    for (int e = threadIdx.x; e < 1024; e += blockDim.x) {
        int c = 0;
        if (e < E)
            for (int q = 0; q < M * 8; ++q)
                c += ((q & 7) < top_k && (q >> 3) < M && sel[q] == e) ? 1 : 0;
        cnt[e] = c;
    }
    __syncthreads();
    // exclusive prefix count of active experts: one ballot per warp of 32 experts
    const int e = threadIdx.x;  // blockDim == 1024 covers every expert index
    const bool act = cnt[e] > 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, act);
    if (lane == 0)
        warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = __popc(bal & ((1u << lane) - 1u));
    for (int w = 0; w < warp; ++w)
        before += warp_tot[w];
    if (threadIdx.x == 1023) {
        int tot = 0;
        for (int w = 0; w < 32; ++w)
            tot += warp_tot[w];
        meta->n_active = tot;
    }
    if (act) {
        MoeSlot& s = meta->slot[before];
        s.expert = e;
        int c = 0;
        for (int m = 0; m < M; ++m)
            for (int j = 0; j < top_k; ++j)
                if (sel[m * 8 + j] == e) {
                    s.rows[c] = m;
                    s.js[c] = j;
                    meta->inv[m * 8 + j] = before * 8 + c;
                    ++c;
                }
        for (int c2 = c; c2 < kMaxM; ++c2) {
            s.rows[c2] = 0;
            s.js[c2] = 0;
        }
        s.count = c;
    }
}

// y[m][n] = sum_j w[m][j] * o[inv[m][j]][n], j ascending (fixed order).
__global__ void moe_combine_kernel(const MoeMeta* __restrict__ meta, const float* __restrict__ o, int top_k, int H,
                                   uint16_t* __restrict__ y)
{
    pdl_wait();
    pdl_launch_dependents();
    const int m = blockIdx.y;
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= H)
        return;
    float acc = 0.f;
    for (int j = 0; j < top_k; ++j) {
        const int src = __ldcg(&meta->inv[m * 8 + j]);
        const float w = __ldcg(&meta->w[m * 8 + j]);
        acc = fmaf(w, __ldcg(o + (int64_t)src * H + n), acc);
    }
    reinterpret_cast<__nv_bfloat16*>(y)[(int64_t)m * H + n] = __float2bfloat16_rn(acc);
}

// A barrier that nothing ever arrives on, waited on with a wall-time bound.
__global__ void timeout_probe_kernel(int* status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = mbar_try_wait(&bar, 0);
        if (!ok) {
            const uint64_t t0 = globaltimer_ns();
            while (!(ok = mbar_try_wait(&bar, 0)))
                if (globaltimer_ns() - t0 > limit_ns)
                    break;
        }
        if (!ok)
            atomicCAS(status, 0, TF_E_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_moe_route(const float* logits, int M, int E, int top_k, int32_t* idx, float* w, MoeMeta* meta,
                             cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(kRouteThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, moe_route_kernel, logits, M, E, top_k, idx, w, meta);
}

cudaError_t launch_moe_combine(const MoeMeta* meta, const float* o, int M, int top_k, int H, uint16_t* y,
                               cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((H + 255) / 256), (unsigned)M, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_combine_kernel, meta, o, top_k, H, y);
}

cudaError_t launch_timeout_probe(int* status, uint64_t limit_ns, cudaStream_t stream)
{
    timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace tfq
