// MoE routing and combine kernels, and the bounded-wait self-test kernel.
//
// Routing (uzu page, "Internals 1" table, mlp row: MixtureOfExperts with a
// routing function; "radix top-k" is among its kernels): per row, the top_k
// experts by fp32 logit, descending, equal logits to the lower index; weights
// are the softmax of the selected logits (fp32 with a compensated sum).
// The router then buckets the (row, slot) pairs by expert so that every
// selected expert's weights are streamed once with all of its rows as MMA
// columns, and writes the inverse map used by the deterministic combine.
#include "tfq_internal.h"
#include "tfq_ptx.cuh"

namespace tfq {
namespace {

constexpr int kRouteThreads = 256;

// Order-preserving unsigned key of an fp32 logit (-0 as +0): a > b iff key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One CTA. PER = logits per lane (E <= 32 PER), so a row's logits sit in registers.
template <int PER>
__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const float* __restrict__ logits, int M, int E,
                                                                  int top_k, int32_t* __restrict__ idx_out,
                                                                  float* __restrict__ w_out, MoeMeta* meta)
{
    __shared__ int32_t sel[kMaxM * 8];  // (row, j) -> expert, -1 when unused
    __shared__ uint8_t act[1024];       // expert selected by some row
    __shared__ int32_t slot_of[1024];   // active expert -> its slot
    __shared__ int32_t warp_tot[kRouteThreads / 32];

    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 1024; i += kRouteThreads)
        act[i] = 0;
    if (threadIdx.x < kMaxM * 8)
        sel[threadIdx.x] = -1;
    __syncthreads();

    // ---- top-k per row (warp m): k rounds of a warp arg-max over the experts not yet
    // taken: each lane proposes its largest logit (lowest expert on ties), one warp max
    // of the order keys finds the value, one warp min the lowest expert holding it
    for (int m = warp; m < M; m += kRouteThreads / 32) {
        const float* l = logits + (int64_t)m * E;
        uint32_t keys[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int e = lane + 32 * i;
            keys[i] = e < E ? order_key(__ldcg(l + e)) : 0u;
        }
        uint32_t taken = 0;  // bit i: expert lane + 32 i taken
        float top = 0.f, mine = 0.f;  // the largest selected logit; lane j: the j-th one
        for (int j = 0; j < top_k; ++j) {
            uint32_t bk = 0;
            int bi = -1;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (bi < 0 || keys[i] > bk)) {  // ascending i keeps the lower
                    bk = keys[i];
                    bi = i;
                }
            }
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t be = __reduce_min_sync(0xffffffffu, bi >= 0 && bk == kmax ? (uint32_t)(lane + 32 * bi)
                                                                                       : 0xffffffffu);
            if ((int)(be & 31u) == lane)
                taken |= 1u << (be >> 5);
            const float v = key_value(kmax);
            if (j == 0)
                top = v;
            if (lane == j)
                mine = v;
            if (lane == 0) {
                sel[m * 8 + j] = (int)be;
                act[be] = 1;
            }
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
            idx_out[m * top_k + lane] = sel[m * 8 + lane];
            w_out[m * top_k + lane] = w;
            meta->w[m * 8 + lane] = w;
        }
    }
    __syncthreads();

    // ---- active experts get slots in ascending expert order: thread t owns experts
    // 4t .. 4t + 3; exclusive prefix of their counts over the CTA
    const int e0 = threadIdx.x * 4;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        cnt += act[e0 + i];
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    int before = incl - cnt;
    for (int w = 0; w < warp; ++w)
        before += warp_tot[w];
    if (threadIdx.x == kRouteThreads - 1)
        meta->n_active = before + cnt;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (act[e0 + i])
            slot_of[e0 + i] = before++;
    __syncthreads();

    // ---- one thread per (row, j) pair: its rank among the earlier pairs of the same
    // expert is its column in the expert's slot, so each slot lists its rows in
    // ascending (row, j) order; the first pair of an expert fills the slot's header
    const int q = threadIdx.x;
    if (q < M * 8 && sel[q] >= 0) {
        const int e = sel[q];
        int c = 0, total = 0;
        for (int q2 = 0; q2 < M * 8; ++q2) {
            const int same = sel[q2] == e;
            total += same;
            if (q2 < q)
                c += same;
        }
        const int slot = slot_of[e];
        MoeSlot& s = meta->slot[slot];
        s.rows[c] = q >> 3;
        s.js[c] = q & 7;
        meta->inv[q] = slot * 8 + c;
        if (c == 0) {
            s.expert = e;
            s.count = total;
            for (int c2 = total; c2 < kMaxM; ++c2) {
                s.rows[c2] = 0;
                s.js[c2] = 0;
            }
        }
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
    if (E <= 32)
        return cudaLaunchKernelEx(&cfg, moe_route_kernel<1>, logits, M, E, top_k, idx, w, meta);
    if (E <= 128)
        return cudaLaunchKernelEx(&cfg, moe_route_kernel<4>, logits, M, E, top_k, idx, w, meta);
    if (E <= 256)
        return cudaLaunchKernelEx(&cfg, moe_route_kernel<8>, logits, M, E, top_k, idx, w, meta);
    return cudaLaunchKernelEx(&cfg, moe_route_kernel<32>, logits, M, E, top_k, idx, w, meta);
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
