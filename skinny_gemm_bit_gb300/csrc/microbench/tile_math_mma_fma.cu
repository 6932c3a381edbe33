// Microbenchmark (not part of libtfq.so): the 16 x 64 4-bit affine tile math alone, on tiles
// resident in shared memory, per SM, for the forms the kernels could use:
//   mma_bf16  mma.sync m16n8k16 on bf16 (128 + q) codes, the light and stage kernels' form
//   mma_f16   the same on fp16 (1024 + q, 1024 + 16 q) codes, the warp workers' form
//   fma_m1    CUDA-core fp32 FMAs at one activation row: each lane converts its 32 codes
//             to fp32 exactly (2^23 + q - 2^23), multiplies and sums, and the 4 lanes of a
//             row pair reduce by shuffles
//   fma_m8    the same for eight activation rows (eight FMAs a code)
// All use the kernels' packed tile (lane l: 16 bytes = its A fragments of the 4 k blocks;
// 64 bytes of (scale, bias) pairs) and a group epilogue, and report tiles per microsecond
// per SM. The sums are not checked (the kernels' parity tests cover the arithmetic): this
// measures the instruction stream. Build and run on a GB300:
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -o /tmp/tile_math_mma_fma \
//        skinny_gemm_bit_gb300/csrc/microbench/tile_math_mma_fma.cu && /tmp/tile_math_mma_fma
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s at %d: %s\n", #x, __LINE__, cudaGetErrorString(e_)); exit(1);} } while (0)

constexpr int kTile = 576, kTiles = 64;  // 36 KB of tiles in shared memory
constexpr int kWarps = 8;

__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d; asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c)); return d;
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3]) : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3]) : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t nib2_bf16(uint32_t w) { return lop3(w, 0x000F000Fu, 0x43004300u); }
__device__ __forceinline__ uint32_t nib2_f16(uint32_t w) { return lop3(w, 0x000F000Fu, 0x64006400u); }
__device__ __forceinline__ uint32_t nib2_f16_x16(uint32_t w) { return lop3(w, 0x00F000F0u, 0x64006400u); }
__device__ __forceinline__ float lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }
// exact code -> fp32: 2^23 + q, minus 2^23
__device__ __forceinline__ float codef(uint32_t w, int sh) { return __uint_as_float(0x4B000000u | ((w >> sh) & 0xFu)) - 8388608.f; }

template <int V>
__global__ void __launch_bounds__(kWarps * 32) kern(const uint8_t* __restrict__ tiles_g, const float* __restrict__ xg,
                                                    int iters, float* out, long long* cyc)
{
    __shared__ __align__(16) uint8_t tiles[kTiles * kTile];
    __shared__ __align__(16) float xs[8 * 64];      // 8 activation rows x 64 columns (fp32, for the FMA paths)
    __shared__ __align__(16) uint32_t xb[8 * 32];   // the same as bf16 / fp16 pairs (B fragments)
    for (int i = threadIdx.x; i < kTiles * kTile / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(tiles)[i] = reinterpret_cast<const uint4*>(tiles_g)[i];
    for (int i = threadIdx.x; i < 8 * 64; i += blockDim.x) xs[i] = xg[i];
    for (int i = threadIdx.x; i < 8 * 32; i += blockDim.x) {
        const float a = xg[2 * i], b = xg[2 * i + 1];
        if (V == 1) { __half2 h = __floats2half2_rn(a, b); xb[i] = *reinterpret_cast<uint32_t*>(&h); }
        else { __nv_bfloat162 h = __floats2bfloat162_rn(a, b); xb[i] = *reinterpret_cast<uint32_t*>(&h); }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gi = lane >> 2, tq = lane & 3;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // B fragments of the group (k-block kb: x rows n = gi, k = 2 tq + {0,1} and + 8)
    uint32_t b0[4], b1[4];
    for (int kb = 0; kb < 4; ++kb) {
        b0[kb] = xb[gi * 32 + kb * 8 + tq];
        b1[kb] = xb[gi * 32 + kb * 8 + 4 + tq];
    }
    const float2 xsum = make_float2(1.f, 2.f);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
        const uint8_t* tile = tiles + ((it * kWarps + warp) % kTiles) * kTile;
        const uint4 wv = *reinterpret_cast<const uint4*>(tile + lane * 16);
        const uint2 sb = *reinterpret_cast<const uint2*>(tile + 512 + (lane >> 2) * 8);
        const float s_lo = lo(sb.x), s_hi = hi(sb.x), b_lo = lo(sb.y), b_hi = hi(sb.y);
        const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
        if (V == 0 || V == 1) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                if (V == 0)
                    mma_bf16(d, nib2_bf16(w[kb]), nib2_bf16(w[kb] >> 4), nib2_bf16(w[kb] >> 8), nib2_bf16(w[kb] >> 12), b0[kb], b1[kb]);
                else
                    mma_f16(d, nib2_f16(w[kb]), nib2_f16_x16(w[kb]), nib2_f16(w[kb] >> 8), nib2_f16_x16(w[kb] >> 8), b0[kb], b1[kb]);
            }
            const float off = V == 0 ? 128.f : 1024.f;
            const float c_lo = fmaf(-off, s_lo, b_lo), c_hi = fmaf(V == 0 ? -128.f : -64.f, s_hi, b_hi);
            const float s_h = V == 0 ? s_hi : s_hi * 0.0625f;
            acc[0] = fmaf(s_lo, d[0], fmaf(c_lo, xsum.x, acc[0]));
            acc[1] = fmaf(s_lo, d[1], fmaf(c_lo, xsum.y, acc[1]));
            acc[2] = fmaf(s_h, d[2], fmaf(c_hi, xsum.x, acc[2]));
            acc[3] = fmaf(s_h, d[3], fmaf(c_hi, xsum.y, acc[3]));
        } else {
            // the lane's codes: rows gi (registers' low halves... here: nibbles 0-3 of each byte pair)
            // and gi + 8, columns 2 tq + {0, 1} + 8 j of every k block: 16 columns, 2 rows
            constexpr int MR = V == 2 ? 1 : 8;
            float dr0[MR], dr1[MR];
#pragma unroll
            for (int m = 0; m < MR; ++m) { dr0[m] = 0.f; dr1[m] = 0.f; }
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {  // register r: row gi + 8 (r & 1), cols 2 tq + 8 (r >> 1) + {0, 1}
                    const int col = kb * 16 + 2 * tq + 8 * (r >> 1);
                    const float q0 = codef(w[kb], 4 * r), q1 = codef(w[kb], 4 * r + 16);
#pragma unroll
                    for (int m = 0; m < MR; ++m) {
                        const float2 xv = *reinterpret_cast<const float2*>(&xs[m * 64 + col]);
                        float& dd = (r & 1) ? dr1[m] : dr0[m];
                        dd = fmaf(q0, xv.x, fmaf(q1, xv.y, dd));
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MR; ++m) {
                // the 4 lanes of a row pair hold disjoint columns: reduce over tq
                float a = dr0[m], b = dr1[m];
                a += __shfl_xor_sync(0xffffffffu, a, 1); a += __shfl_xor_sync(0xffffffffu, a, 2);
                b += __shfl_xor_sync(0xffffffffu, b, 1); b += __shfl_xor_sync(0xffffffffu, b, 2);
                acc[m] = fmaf(s_lo, a, fmaf(b_lo, xsum.x, acc[m]));
                acc[(m + 4) & 7] = fmaf(s_hi, b, fmaf(b_hi, xsum.y, acc[(m + 4) & 7]));
            }
        }
    }
    const long long t1 = clock64();
    float s = 0.f;
    for (int i = 0; i < 8; ++i) s += acc[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

int main() {
    CK(cudaSetDevice(0));
    cudaDeviceProp prop; CK(cudaGetDeviceProperties(&prop, 0));
    const int sms = prop.multiProcessorCount;
    uint8_t* tiles; float* x; float* out; long long* cyc;
    CK(cudaMalloc(&tiles, kTiles * kTile));
    CK(cudaMalloc(&x, 8 * 64 * 4));
    CK(cudaMalloc(&out, sms * 4 * kWarps * 32 * 4));
    CK(cudaMalloc(&cyc, sms * 4 * 8));
    uint8_t* ht = (uint8_t*)malloc(kTiles * kTile);
    for (int i = 0; i < kTiles * kTile; ++i) ht[i] = (uint8_t)(i * 2654435761u >> 24);
    for (int t = 0; t < kTiles; ++t)  // (scale, bias) bytes as small bf16 values
        for (int j = 0; j < 16; ++j) { uint16_t v = 0x3C00 + (j & 7); memcpy(ht + t * kTile + 512 + 4 * j, &v, 2); memcpy(ht + t * kTile + 514 + 4 * j, &v, 2); }
    CK(cudaMemcpy(tiles, ht, kTiles * kTile, cudaMemcpyHostToDevice));
    float hx[512]; for (int i = 0; i < 512; ++i) hx[i] = (float)((i * 37) % 17 - 8) * 0.125f;
    CK(cudaMemcpy(x, hx, sizeof hx, cudaMemcpyHostToDevice));
    const char* names[4] = {"mma_bf16 (M<=8)", "mma_f16 (M<=8)", "fma_fp32 M=1", "fma_fp32 M=8"};
    cudaEvent_t e0, e1; CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
    const int iters = 4096;
    for (int blocksPerSM : {1, 2}) {
        for (int v = 0; v < 4; ++v) {
            const int grid = sms * blocksPerSM;
            float best = 1e30f;
            for (int rep = 0; rep < 3; ++rep) {
                CK(cudaEventRecord(e0));
                if (v == 0) kern<0><<<grid, kWarps * 32>>>(tiles, x, iters, out, cyc);
                if (v == 1) kern<1><<<grid, kWarps * 32>>>(tiles, x, iters, out, cyc);
                if (v == 2) kern<2><<<grid, kWarps * 32>>>(tiles, x, iters, out, cyc);
                if (v == 3) kern<3><<<grid, kWarps * 32>>>(tiles, x, iters, out, cyc);
                CK(cudaEventRecord(e1)); CK(cudaEventSynchronize(e1)); CK(cudaGetLastError());
                float ms; CK(cudaEventElapsedTime(&ms, e0, e1)); if (ms < best) best = ms;
            }
            const double tiles_total = (double)grid * kWarps * iters;
            const double per_sm_per_us = tiles_total / sms / (best * 1e3);
            // bytes equivalent: 576 B per tile -> GB/s per SM and for the whole GPU
            printf("%d CTA/SM x %d warps  %-16s %8.2f tiles/us/SM  = %7.1f GB/s/SM  (%.0f GB/s GPU-wide)\n", blocksPerSM, kWarps,
                   names[v], per_sm_per_us, per_sm_per_us * 576e-3, per_sm_per_us * 576e-3 * sms);
        }
    }
    return 0;
}
