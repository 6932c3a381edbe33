// Microbenchmark (not part of libtfq.so): the 4-bit affine tile math on the 5th-generation
// tensor cores (tcgen05.mma, accumulators and the A operand in tensor memory), on weights
// resident in shared memory, reported as 16 x 64 tiles per microsecond per SM so that it
// compares directly with tile_math_mma_fma.cu. Build and run on a GB300:
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/tile_math_tcgen05 \
//        skinny_gemm_bit_gb300/csrc/microbench/tile_math_tcgen05.cu && /tmp/tile_math_tcgen05
//
// A CTA holds a 128-row x 512-column block of codes (8 groups of 64 columns, each row's
// (scale, bias) per group) and eight activation rows, and loops over the groups:
//   worker warps 0-3   thread r (row r) unpacks its 64 codes of group g into bf16 (128 + q)
//                      pairs, one LOP3 a pair, and writes them to tensor memory with one
//                      tcgen05.st (32 columns: the A operand of the group's four MMAs);
//                      then the group epilogue of group g - 2: tcgen05.ld of its row's 8
//                      accumulator columns and acc[m] += s D[m] + (b - 128 s) sum_x[m]
//   warp 4, lane 0     four tcgen05.mma kind::f16 per group (M = 128 rows, N = 16: the 8
//                      activation rows and 8 zero rows, K = 16 each) into the group's
//                      accumulator columns, A from tensor memory, B (the activations, no
//                      swizzle, K-major 8 x 16-byte core matrices) from shared memory
//                      through a matrix descriptor; tcgen05.commit to the group's mbarrier
// A is double-buffered (2 x 32 columns), the accumulators a ring of 4 groups (4 x 16
// columns): 128 tensor-memory columns a CTA, so four CTAs fit an SM. A first launch of one
// CTA checks the sums of one pass against a double-precision host reference; every wait
// is bounded and a wait that gives up sets an error flag that the host reports.
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cmath>
#include <vector>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e_)); exit(1);} } while (0)

constexpr int G = 8, ROWS = 128, NC = 16;
constexpr int kCodesB = G * ROWS * 32;      // 32 KB of codes
constexpr int kSbB = G * ROWS * 4;          // (scale, bias) bf16 pairs
constexpr int kBmatB = G * 4 * 512;         // B: 4 MMAs a group, 4 core matrices each
constexpr int kXsB = G * 8 * 4;
constexpr int kOffCodes = 0, kOffSb = kOffCodes + kCodesB, kOffB = kOffSb + kSbB, kOffXs = kOffB + kBmatB,
              kOffBar = kOffXs + kXsB, kSmem = kOffBar + 128;
constexpr uint32_t kCols = 128, kAcol = 0, kDcol = 64;
constexpr long long kLimit = 40000000;  // cycles a wait may take (~20 ms)

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) { asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* b) { asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory"); }
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t par) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(su32(b)), "r"(par) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t par, volatile int* err) {
    if (mbar_try(b, par)) return true;
    const long long t0 = clock64();
    while (!mbar_try(b, par)) {
        if (*err) return false;
        if (clock64() - t0 > kLimit) { *err = 1; return false; }
    }
    return true;
}
__device__ __forceinline__ uint32_t nib2(uint32_t w) {
    uint32_t d; asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u)); return d;
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&a)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),
                    "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15]),
                    "r"(a[16]), "r"(a[17]), "r"(a[18]), "r"(a[19]), "r"(a[20]), "r"(a[21]), "r"(a[22]), "r"(a[23]),
                    "r"(a[24]), "r"(a[25]), "r"(a[26]), "r"(a[27]), "r"(a[28]), "r"(a[29]), "r"(a[30]), "r"(a[31])
                 : "memory");
}
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&d)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr) : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    for (int i = 0; i < 8; ++i) d[i] = __uint_as_float(r[i]);
}
// shared-memory matrix descriptor: no swizzle, K-major core matrices of 8 rows x 16 bytes;
// lbo = byte step between core matrices along K, sbo = along N
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// instruction descriptor, kind::f16: D f32, A bf16, B bf16, both K-major, N = 16, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NC >> 3) << 17) | ((uint32_t)(ROWS >> 4) << 24);

__global__ void __launch_bounds__(160, 2) tc_kernel(const uint8_t* __restrict__ gsrc, int reps, float* out,
                                                     long long* cyc, int* err_out, int lbo, int sbo)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + kOffBar);  // [2]
    uint64_t* done = a_full + 2;                                     // [4]
    uint32_t* taddr_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 64);
    volatile int* err = reinterpret_cast<volatile int*>(smem + kOffBar + 68);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < (kOffBar) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = reinterpret_cast<const uint4*>(gsrc)[i];
    if (threadIdx.x == 0) {
        mbar_init(&a_full[0], 4); mbar_init(&a_full[1], 4);
        for (int i = 0; i < 4; ++i) mbar_init(&done[i], 1);
        *err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(taddr_slot)), "r"(kCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *taddr_slot;
    const int NG = reps * G;
    const long long t0 = clock64();
    if (warp < 4) {
        const int row = warp * 32 + lane;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float* xs = reinterpret_cast<const float*>(smem + kOffXs);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int g = 0; g <= NG + 1; ++g) {
            // A(g) may be written once MMA(g - 2) has read A((g - 2) & 1): then also the epilogue of g - 2
            if (g >= 2 && !mbar_wait(&done[(g - 2) & 3], ((g - 2) >> 2) & 1, err)) break;
            tc_fence_after();
            if (g < NG) {
                const int gg = g % G, s = g & 1;
                const uint4* cp = reinterpret_cast<const uint4*>(smem + kOffCodes + (gg * ROWS + row) * 32);
                const uint4 c0 = cp[0], c1 = cp[1];
                const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint32_t a[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    a[4 * j + 0] = nib2(w[j]);
                    a[4 * j + 1] = nib2(w[j] >> 4);
                    a[4 * j + 2] = nib2(w[j] >> 8);
                    a[4 * j + 3] = nib2(w[j] >> 12);
                }
                tc_st32(tbase + lane_base + kAcol + 32 * s, a);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[s]);
            }
            if (g >= 2) {  // epilogue of group g - 2 (its MMA completed: waited above)
                const int h = g - 2, hg = h % G;
                float d[8];
                tc_ld8(tbase + lane_base + kDcol + 16 * (h & 3), d);
                const uint32_t sbv = *reinterpret_cast<const uint32_t*>(smem + kOffSb + (hg * ROWS + row) * 4);
                const float sc = __uint_as_float(sbv << 16), bi = __uint_as_float(sbv & 0xFFFF0000u);
                const float cc = fmaf(-128.f, sc, bi);
                const float4 x0 = *reinterpret_cast<const float4*>(xs + hg * 8);
                const float4 x1 = *reinterpret_cast<const float4*>(xs + hg * 8 + 4);
                const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int m = 0; m < 8; ++m) acc[m] = fmaf(sc, d[m], fmaf(cc, xv[m], acc[m]));
            }
        }
        for (int m = 0; m < 8; ++m) out[((size_t)blockIdx.x * ROWS + row) * 8 + m] = acc[m];
    } else if (warp == 4 && lane == 0) {
        const uint32_t bbase = su32(smem + kOffB);
        for (int g = 0; g < NG; ++g) {
            const int gg = g % G, s = g & 1;
            if (!mbar_wait(&a_full[s], (g >> 1) & 1, err)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc(bbase + (gg * 4 + kk) * 512, (uint32_t)lbo, (uint32_t)sbo);
                const uint32_t dt = tbase + kDcol + 16 * (g & 3), at = tbase + kAcol + 32 * s + 8 * kk;
                asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                             " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                             :: "r"(dt), "r"(at), "l"(bd), "r"(kIdesc), "r"(kk) : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(&done[g & 3])) : "memory");
        }
    }
    const long long t1 = clock64();
    tc_fence_before();
    __syncthreads();
    // every MMA has completed (the workers waited for the last group's barrier) unless a wait gave up
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kCols) : "memory");
    }
    if (threadIdx.x == 0) {
        cyc[blockIdx.x] = t1 - t0;
        if (*err) atomicExch(err_out, 1);
    }
}

static uint16_t f2bf(float f) { uint32_t u; memcpy(&u, &f, 4); u += 0x7FFFu + ((u >> 16) & 1u); return (uint16_t)(u >> 16); }
static float bf2f(uint16_t h) { uint32_t u = (uint32_t)h << 16; float f; memcpy(&f, &u, 4); return f; }

int main()
{
    CK(cudaSetDevice(0));
    cudaDeviceProp prop; CK(cudaGetDeviceProperties(&prop, 0));
    const int sms = prop.multiProcessorCount;
    srand(1234);
    // host image of the shared-memory block
    std::vector<uint8_t> img(kOffBar, 0);
    std::vector<uint8_t> q((size_t)ROWS * G * 64);
    for (auto& v : q) v = (uint8_t)(rand() & 15);
    std::vector<float> x(8 * G * 64);
    for (auto& v : x) v = bf2f(f2bf((float)((rand() % 2001) - 1000) / 500.f));
    std::vector<float> sc(G * ROWS), bi(G * ROWS);
    for (int i = 0; i < G * ROWS; ++i) { sc[i] = bf2f(f2bf(0.001f * (1 + rand() % 50))); bi[i] = bf2f(f2bf(-0.01f * (rand() % 20))); }
    // codes: row r, group g, word j (8 nibbles): nibble at bit 4t = k 8j + 2t, at bit 4t + 16 = k 8j + 2t + 1
    for (int g = 0; g < G; ++g)
        for (int r = 0; r < ROWS; ++r)
            for (int j = 0; j < 8; ++j) {
                uint32_t w = 0;
                for (int t = 0; t < 4; ++t) {
                    w |= (uint32_t)q[((size_t)r * G + g) * 64 + 8 * j + 2 * t] << (4 * t);
                    w |= (uint32_t)q[((size_t)r * G + g) * 64 + 8 * j + 2 * t + 1] << (4 * t + 16);
                }
                memcpy(&img[kOffCodes + (g * ROWS + r) * 32 + 4 * j], &w, 4);
            }
    for (int g = 0; g < G; ++g)
        for (int r = 0; r < ROWS; ++r) {
            uint32_t v = (uint32_t)f2bf(sc[g * ROWS + r]) | ((uint32_t)f2bf(bi[g * ROWS + r]) << 16);
            memcpy(&img[kOffSb + (g * ROWS + r) * 4], &v, 4);
        }
    // B: [g][kk][kb][nb][8 rows][8 bf16]; row n = nb 8 + r (activation row, zero for n >= 8), k = g 64 + kk 16 + kb 8 + e
    for (int g = 0; g < G; ++g)
        for (int kk = 0; kk < 4; ++kk)
            for (int kb = 0; kb < 2; ++kb)
                for (int nb = 0; nb < 2; ++nb)
                    for (int r = 0; r < 8; ++r)
                        for (int e = 0; e < 8; ++e) {
                            const int n = nb * 8 + r, k = g * 64 + kk * 16 + kb * 8 + e;
                            const uint16_t v = n < 8 ? f2bf(x[n * G * 64 + k]) : 0;
                            memcpy(&img[kOffB + (((g * 4 + kk) * 2 + kb) * 2 + nb) * 128 + r * 16 + e * 2], &v, 2);
                        }
    for (int g = 0; g < G; ++g)
        for (int m = 0; m < 8; ++m) {
            float s = 0.f;
            for (int k = 0; k < 64; ++k) s += x[m * G * 64 + g * 64 + k];
            memcpy(&img[kOffXs + (g * 8 + m) * 4], &s, 4);
        }
    // reference for one pass over the 16 groups
    std::vector<double> ref((size_t)ROWS * 8);
    for (int r = 0; r < ROWS; ++r)
        for (int m = 0; m < 8; ++m) {
            double a = 0;
            for (int g = 0; g < G; ++g) {
                float xsum; memcpy(&xsum, &img[kOffXs + (g * 8 + m) * 4], 4);
                double dsum = 0;
                for (int k = 0; k < 64; ++k) dsum += (128.0 + q[((size_t)r * G + g) * 64 + k]) * x[m * G * 64 + g * 64 + k];
                const double s = sc[g * ROWS + r], b = bi[g * ROWS + r];
                a += s * dsum + (b - 128.0 * s) * xsum;
            }
            ref[r * 8 + m] = a;
        }
    uint8_t* dsrc; float* dout; long long* dcyc; int* derr;
    CK(cudaMalloc(&dsrc, img.size()));
    CK(cudaMemcpy(dsrc, img.data(), img.size(), cudaMemcpyHostToDevice));
    const int maxC = 4 * sms;
    CK(cudaMalloc(&dout, (size_t)maxC * ROWS * 8 * 4));
    CK(cudaMalloc(&dcyc, maxC * 8));
    CK(cudaMalloc(&derr, 4));
    CK(cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
    const int lbo = 256, sbo = 128;  // core-matrix steps along K and along N of the B layout below
    // correctness: one CTA, one pass
    CK(cudaMemset(derr, 0, 4));
    tc_kernel<<<1, 160, kSmem>>>(dsrc, 1, dout, dcyc, derr, lbo, sbo);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    int herr = 0; CK(cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost));
    std::vector<float> got((size_t)ROWS * 8);
    CK(cudaMemcpy(got.data(), dout, got.size() * 4, cudaMemcpyDeviceToHost));
    double maxdiff = 0, maxabs = 0;
    for (size_t i = 0; i < got.size(); ++i) {
        maxabs = fmax(maxabs, fabs(ref[i]));
        maxdiff = fmax(maxdiff, fabs(got[i] - ref[i]));
    }
    printf("one pass, one CTA: wait error %d, max |got - ref| %.3g (max |ref| %.3g) -> %s\n", herr, maxdiff, maxabs,
           (herr == 0 && maxdiff <= 1e-4 * maxabs + 1e-3) ? "MATCH" : "MISMATCH");
    if (herr || maxdiff > 1e-4 * maxabs + 1e-3) return 1;
    // throughput: one or two CTAs an SM
    cudaEvent_t e0, e1; CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
    for (int per = 1; per <= 4; ++per) {
        const int C = per * sms, reps = 4000;
        tc_kernel<<<C, 160, kSmem>>>(dsrc, 20, dout, dcyc, derr, lbo, sbo);
        CK(cudaDeviceSynchronize());
        CK(cudaEventRecord(e0));
        tc_kernel<<<C, 160, kSmem>>>(dsrc, reps, dout, dcyc, derr, lbo, sbo);
        CK(cudaEventRecord(e1));
        CK(cudaEventSynchronize(e1));
        float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
        CK(cudaMemcpy(&herr, derr, 4, cudaMemcpyDeviceToHost));
        const double tiles = (double)C * reps * G * (ROWS / 16);
        printf("tcgen05 %d CTA/SM: %.2f tiles/us/SM (%.0f GB/s of 4-bit weights GPU-wide)  wait error %d\n", per,
               tiles / (ms * 1e3) / sms, tiles * 576.0 / (ms * 1e-3) / 1e9, herr);
    }
    return 0;
}
