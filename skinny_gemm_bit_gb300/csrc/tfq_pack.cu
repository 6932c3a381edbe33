// Repacking of MLX affine quantised weights into the projection kernel's tile order.
//
// A tile is 16 output rows x 64 input columns (one quantisation group). Its code
// bytes are laid out so that lane l of a warp loads, with one 16-byte (4-bit) or
// two 16-byte (8-bit) shared-memory loads, exactly the A fragments it needs for
// the four m16n8k16 MMAs that cover the 64 columns; the scales and biases of the
// 16 rows follow as 8 pairs (row i, row i+8), which is what a lane's accumulator
// fragment needs. Rows past N are zero (code 0, scale 0, bias 0).
//
// MMA A-fragment (row-major 16x16, bf16): register r of lane l = (gi = l/4, t = l%4)
// holds rows gi + 8*(r&1) and columns 2t + 8*(r>>1) + {0, 1}.
//
// 4-bit: word kb of lane l holds the 8 codes of k-block kb; code p of the word
//   (bits 4p..4p+3) is row gi + 8*(p&1), column 2t + (p>>2) + 8*((p>>1)&1), so
//   that ((w >> 4r) & 0x000F000F) yields register r as two codes.
// 8-bit: words 2kb + jp of lane l; byte bp is row gi + 8*(bp&1), column
//   2t + 8*jp + (bp>>1). The low nibbles of a word give registers 2jp, 2jp+1 of
//   the "low" fragment, the high nibbles the same registers of the "high" one.
//
// NVFP4 (E2M1 codes, one E4M3 scale per 16 columns): byte r of word kb of lane l is
//   register r of k-block kb as two codes, the even column in the low nibble (the
//   order in which one cvt.rn.f16x2.e2m1x2 turns a byte into a register); the 64
//   scale bytes follow as 8 groups of 8, group gi = {row gi, row gi + 8} for k-blocks
//   0..3 in turn, so one 16-bit half converts to the (row gi, row gi + 8) pair.
#include <cuda_bf16.h>

#include "tfq_internal.h"
#include "tfq_ptx.cuh"

namespace tfq {
namespace {

__device__ __forceinline__ uint32_t code_at(const uint32_t* wq_row, int64_t k, int bits)
{
    const int per = 32 / bits;
    const uint32_t word = wq_row[k / per];
    return (word >> (bits * (int)(k % per))) & ((1u << bits) - 1u);
}

__global__ void pack_kernel(const uint32_t* __restrict__ wq, const uint16_t* __restrict__ sc,
                            const uint16_t* __restrict__ bi, int64_t batch, int64_t N, int64_t K, int bits,
                            uint8_t* __restrict__ packed, PackHeader hdr)
{
    const int64_t G = K / kGroup;
    const int64_t n_rb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
    const int tile_words = tile_bytes_for(bits) / 4;
    const int q_words = tile_q_bytes_for(bits) / 4;
    const int64_t words_per_row = K * bits / 32;
    const int64_t total = batch * n_rb * G * tile_words;
    uint32_t* out = reinterpret_cast<uint32_t*>(packed + TF_PACK_HEADER_BYTES);

    if (blockIdx.x == 0 && threadIdx.x == 0)
        *reinterpret_cast<PackHeader*>(packed) = hdr;

    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int wi = (int)(idx % tile_words);
        const int64_t tile = idx / tile_words;
        const int64_t g = tile % G;
        const int64_t rb = (tile / G) % n_rb;
        const int64_t b = tile / (G * n_rb);
        const uint32_t* wq_b = wq + b * N * words_per_row;
        uint32_t word = 0;
        if (wi < q_words) {
            if (bits == 4) {
                const int lane = wi >> 2, kb = wi & 3, gi = lane >> 2, t = lane & 3;
                for (int p = 0; p < 8; ++p) {
                    const int64_t row = rb * kRowsPerBlock + gi + 8 * (p & 1);
                    const int64_t k = g * kGroup + kb * 16 + 2 * t + (p >> 2) + 8 * ((p >> 1) & 1);
                    if (row < N)
                        word |= code_at(wq_b + row * words_per_row, k, 4) << (4 * p);
                }
            } else {
                const int lane = wi >> 3, kb = (wi >> 1) & 3, jp = wi & 1, gi = lane >> 2, t = lane & 3;
                for (int bp = 0; bp < 4; ++bp) {
                    const int64_t row = rb * kRowsPerBlock + gi + 8 * (bp & 1);
                    const int64_t k = g * kGroup + kb * 16 + 2 * t + 8 * jp + (bp >> 1);
                    if (row < N)
                        word |= code_at(wq_b + row * words_per_row, k, 8) << (8 * bp);
                }
            }
        } else {
            const int j = wi - q_words;     // 0..15
            const int gi = j >> 1;
            const uint16_t* src = (j & 1) ? bi : sc;
            const int64_t row_lo = rb * kRowsPerBlock + gi, row_hi = row_lo + 8;
            const uint32_t lo = row_lo < N ? src[(b * N + row_lo) * G + g] : 0u;
            const uint32_t hi = row_hi < N ? src[(b * N + row_hi) * G + g] : 0u;
            word = lo | (hi << 16);
        }
        out[idx] = word;
    }
}

// Locate element (row rr of its 16-row block, column kk of its 64-column group)
// inside a tile: returns the word index and the bit shift of its code.
__device__ __forceinline__ void locate(int rr, int kk, int bits, int& word, int& shift)
{
    const int kb = kk >> 4, c = kk & 15, half = c & 1, t = (c & 7) >> 1, gi = rr & 7;
    const int lane = gi * 4 + t;
    if (bits == 4) {
        const int p = (rr >> 3) + 2 * (c >> 3) + 4 * half;
        word = lane * 4 + kb;
        shift = 4 * p;
    } else {
        const int jp = c >> 3;
        const int bp = (rr >> 3) | (half << 1);
        word = lane * 8 + kb * 2 + jp;
        shift = 8 * bp;
    }
}

__global__ void unpack_codes_kernel(const uint8_t* __restrict__ packed, int64_t batch, int64_t N, int64_t K,
                                    int bits, uint32_t* __restrict__ wq)
{
    const int64_t G = K / kGroup;
    const int64_t n_rb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
    const int per = 32 / bits;
    const int64_t words_per_row = K / per;
    const int64_t total = batch * N * words_per_row;
    const int tile_words = tile_bytes_for(bits) / 4;
    const uint32_t* tiles = reinterpret_cast<const uint32_t*>(packed + TF_PACK_HEADER_BYTES);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = idx % words_per_row;
        const int64_t row = (idx / words_per_row) % N;
        const int64_t b = idx / (words_per_row * N);
        uint32_t out = 0;
        for (int i = 0; i < per; ++i) {
            const int64_t k = j * per + i;
            int w, sh;
            locate((int)(row % kRowsPerBlock), (int)(k % kGroup), bits, w, sh);
            const int64_t tile = (b * n_rb + row / kRowsPerBlock) * G + k / kGroup;
            const uint32_t code = (tiles[tile * tile_words + w] >> sh) & ((1u << bits) - 1u);
            out |= code << (bits * i);
        }
        wq[idx] = out;
    }
}

__global__ void unpack_scales_kernel(const uint8_t* __restrict__ packed, int64_t batch, int64_t N, int64_t K,
                                     int bits, uint16_t* __restrict__ sc, uint16_t* __restrict__ bi)
{
    const int64_t G = K / kGroup;
    const int64_t n_rb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t total = batch * N * G;
    const int tile_words = tile_bytes_for(bits) / 4;
    const int q_words = tile_q_bytes_for(bits) / 4;
    const uint32_t* tiles = reinterpret_cast<const uint32_t*>(packed + TF_PACK_HEADER_BYTES);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = idx % G;
        const int64_t row = (idx / G) % N;
        const int64_t b = idx / (G * N);
        const int rr = (int)(row % kRowsPerBlock);
        const int64_t tile = (b * n_rb + row / kRowsPerBlock) * G + g;
        const uint32_t* tw = tiles + tile * tile_words + q_words;
        const int sh = (rr >> 3) * 16;
        sc[idx] = (uint16_t)(tw[2 * (rr & 7)] >> sh);
        bi[idx] = (uint16_t)(tw[2 * (rr & 7) + 1] >> sh);
    }
}

// Rows of a packed matrix (batch 0) dequantised to bf16: x[m][k] = bf16(s q + b) of
// row ids[m], column k, rounded to nearest even (s q + b is exact in fp32 whenever
// |b| / |s| < 2^15, so the rounding is that of the exact value). NVFP4 (bits ==
// kNvfp4): bf16(gscale * (e4m3 scale * e2m1 code)), the inner product exact in fp32, so
// the fp32 value is the exact product rounded once. An id outside [0, N) records
// TF_E_INVALID_ARG in *status and gives a zero row.
__global__ void embed_rows_kernel(const uint8_t* __restrict__ packed, int64_t N, int64_t K, int bits, float gscale,
                                  const int32_t* __restrict__ ids, int64_t M, uint16_t* __restrict__ x, int64_t ldx,
                                  int* status)
{
    const int64_t G = K / kGroup;
    const int tile_words = tile_bytes_for(bits) / 4;
    const int q_words = tile_q_bytes_for(bits) / 4;
    const uint32_t* tiles = reinterpret_cast<const uint32_t*>(packed + TF_PACK_HEADER_BYTES);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < M * K;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = idx / K, k = idx - m * K;
        const int64_t row = __ldg(ids + m);
        float v = 0.f;
        if (row < 0 || row >= N) {
            if (k == 0)
                atomicCAS(status, 0, TF_E_INVALID_ARG);
        } else if (bits == kNvfp4) {
            const int rr = (int)(row % kRowsPerBlock), c = (int)(k % kGroup), cc = c & 15, kb = c >> 4;
            const uint8_t* tb = reinterpret_cast<const uint8_t*>(tiles) +
                                ((row / kRowsPerBlock) * G + k / kGroup) * (int64_t)tile_bytes_for(kNvfp4);
            const int lane = (rr & 7) * 4 + ((cc & 7) >> 1), r = (rr >> 3) + 2 * (cc >> 3);
            uint32_t q2, u1, u2, u3;  // the byte's two codes as an fp16 pair, even column low
            e2m1x8_to_f16x2(__ldg(tb + lane * 16 + kb * 4 + r), q2, u1, u2, u3);
            const uint32_t s2 = e4m3x2_to_f16x2(__ldg(tb + tile_q_bytes_for(kNvfp4) + (rr & 7) * 8 + 2 * kb + (rr >> 3)));
            const __half2 qh = *reinterpret_cast<const __half2*>(&q2), sh = *reinterpret_cast<const __half2*>(&s2);
            const float q = (cc & 1) ? __high2float(qh) : __low2float(qh);
            v = gscale * (__low2float(sh) * q);
        } else {
            const int rr = (int)(row % kRowsPerBlock);
            int w, sh;
            locate(rr, (int)(k % kGroup), bits, w, sh);
            const uint32_t* tw = tiles + ((row / kRowsPerBlock) * G + k / kGroup) * tile_words;
            const uint32_t q = (__ldg(tw + w) >> sh) & ((1u << bits) - 1u);
            const int shs = (rr >> 3) * 16;
            const float sc = __uint_as_float(((__ldg(tw + q_words + 2 * (rr & 7)) >> shs) & 0xFFFFu) << 16);
            const float bi = __uint_as_float(((__ldg(tw + q_words + 2 * (rr & 7) + 1) >> shs) & 0xFFFFu) << 16);
            v = fmaf(sc, (float)q, bi);
        }
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        x[m * ldx + k] = *reinterpret_cast<const uint16_t*>(&h);
    }
}

__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int64_t N,
                                  int64_t K, uint8_t* __restrict__ packed, PackHeader hdr, bool write_header)
{
    const int64_t G = K / kGroup;
    const int64_t n_rb = (N + kRowsPerBlock - 1) / kRowsPerBlock;
    constexpr int tile_words = tile_bytes_for(kNvfp4) / 4, q_words = tile_q_bytes_for(kNvfp4) / 4;
    const int64_t total = n_rb * G * tile_words;
    uint32_t* out = reinterpret_cast<uint32_t*>(packed + TF_PACK_HEADER_BYTES);
    if (write_header && blockIdx.x == 0 && threadIdx.x == 0)
        *reinterpret_cast<PackHeader*>(packed) = hdr;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int wi = (int)(idx % tile_words);
        const int64_t tile = idx / tile_words;
        const int64_t g = tile % G, rb = tile / G;
        uint32_t word = 0;
        if (wi < q_words) {
            const int lane = wi >> 2, kb = wi & 3, gi = lane >> 2, t = lane & 3;
            for (int r = 0; r < 4; ++r) {
                const int64_t row = rb * kRowsPerBlock + gi + 8 * (r & 1);
                const int64_t col = g * kGroup + kb * 16 + 2 * t + 8 * (r >> 1);  // even
                if (row < N)
                    word |= (uint32_t)codes[row * (K / 2) + col / 2] << (8 * r);
            }
        } else {
            const int j = wi - q_words, gi = j >> 1;
            for (int b = 0; b < 4; ++b) {
                const int kb = 2 * (j & 1) + (b >> 1);
                const int64_t row = rb * kRowsPerBlock + gi + 8 * (b & 1);
                if (row < N)
                    word |= (uint32_t)scales[row * (K / 16) + g * 4 + kb] << (8 * b);
            }
        }
        out[idx] = word;
    }
}

// Inverse of pack_nvfp4_kernel: one thread per code byte, then per scale byte.
__global__ void unpack_nvfp4_kernel(const uint8_t* __restrict__ packed, int64_t N, int64_t K,
                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales)
{
    const int64_t G = K / kGroup;
    constexpr int tile_b = tile_bytes_for(kNvfp4), q_b = tile_q_bytes_for(kNvfp4);
    const uint8_t* tiles = packed + TF_PACK_HEADER_BYTES;
    const int64_t n_codes = N * (K / 2), total = n_codes + N * (K / 16);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        if (idx < n_codes) {
            const int64_t row = idx / (K / 2), col = 2 * (idx % (K / 2));
            const int rr = (int)(row % kRowsPerBlock), c = (int)(col % kGroup), cc = c & 15;
            const int lane = (rr & 7) * 4 + ((cc & 7) >> 1), r = (rr >> 3) + 2 * (cc >> 3);
            const uint8_t* tb = tiles + ((row / kRowsPerBlock) * G + col / kGroup) * tile_b;
            codes[idx] = tb[lane * 16 + (c >> 4) * 4 + r];
        } else {
            const int64_t i = idx - n_codes, row = i / (K / 16), sj = i % (K / 16);
            const int rr = (int)(row % kRowsPerBlock), kb = (int)(sj % 4);
            const uint8_t* tb = tiles + ((row / kRowsPerBlock) * G + sj / 4) * tile_b;
            scales[i] = tb[q_b + (rr & 7) * 8 + 2 * kb + (rr >> 3)];
        }
    }
}

int grid_for(int64_t total, int threads)
{
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 65535LL * 32)
        blocks = 65535LL * 32;
    return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_pack(const uint32_t* wq, const uint16_t* s, const uint16_t* b, int64_t batch, int64_t N,
                        int64_t K, int bits, uint8_t* packed, cudaStream_t stream)
{
    PackHeader h{};
    h.magic = TF_QWEIGHT_MAGIC;
    h.version = TF_PACK_VERSION;
    h.bits = bits;
    h.group = kGroup;
    h.code = TF_CODE_AFFINE;
    h.global_scale = 1.f;
    h.batch = batch;
    h.N = N;
    h.K = K;
    h.n_pad = (N + kRowsPerBlock - 1) / kRowsPerBlock * kRowsPerBlock;
    h.tile_bytes = tile_bytes_for(bits);
    h.matrix_bytes = h.n_pad / kRowsPerBlock * (K / kGroup) * h.tile_bytes;
    const int64_t total = batch * (h.n_pad / kRowsPerBlock) * (K / kGroup) * (tile_bytes_for(bits) / 4);
    pack_kernel<<<grid_for(total, 256), 256, 0, stream>>>(wq, s, b, batch, N, K, bits, packed, h);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* packed, int64_t batch, int64_t N, int64_t K, int bits, uint32_t* wq,
                          uint16_t* s, uint16_t* b, cudaStream_t stream)
{
    const int64_t words = batch * N * (K * bits / 32);
    unpack_codes_kernel<<<grid_for(words, 256), 256, 0, stream>>>(packed, batch, N, K, bits, wq);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int64_t groups = batch * N * (K / kGroup);
    unpack_scales_kernel<<<grid_for(groups, 256), 256, 0, stream>>>(packed, batch, N, K, bits, s, b);
    return cudaGetLastError();
}

// The per-matrix fp32 scales of a packed NVFP4 buffer, after its matrices: from a device
// array (src != nullptr) or, for one matrix, the value given.
__global__ void nvfp4_scale_table_kernel(float* __restrict__ table, const float* __restrict__ src, float value,
                                         int64_t batch)
{
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < batch; e += (int64_t)gridDim.x * blockDim.x)
        table[e] = src != nullptr ? src[e] : value;
}

cudaError_t launch_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, const float* gscales, int64_t batch,
                              int64_t N, int64_t K, uint8_t* packed, const PackHeader& hdr, cudaStream_t stream)
{
    const int64_t total = (hdr.n_pad / kRowsPerBlock) * (K / kGroup) * (tile_bytes_for(kNvfp4) / 4);
    for (int64_t e = 0; e < batch; ++e) {
        pack_nvfp4_kernel<<<grid_for(total, 256), 256, 0, stream>>>(codes + e * N * (K / 2), scales + e * N * (K / 16),
                                                                    N, K, packed + e * hdr.matrix_bytes, hdr, e == 0);
        const cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess)
            return err;
    }
    float* table = reinterpret_cast<float*>(packed + TF_PACK_HEADER_BYTES + batch * hdr.matrix_bytes);
    nvfp4_scale_table_kernel<<<grid_for(batch, 128), 128, 0, stream>>>(table, gscales, hdr.global_scale, batch);
    return cudaGetLastError();
}

cudaError_t launch_unpack_nvfp4(const uint8_t* packed, int64_t N, int64_t K, uint8_t* codes, uint8_t* scales,
                                cudaStream_t stream)
{
    const int64_t total = N * (K / 2) + N * (K / 16);
    unpack_nvfp4_kernel<<<grid_for(total, 256), 256, 0, stream>>>(packed, N, K, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_embed_rows(const uint8_t* packed, int64_t N, int64_t K, int bits, float gscale, const int32_t* ids,
                              int64_t M, uint16_t* x, int64_t ldx, int* status, cudaStream_t stream)
{
    embed_rows_kernel<<<grid_for(M * K, 256), 256, 0, stream>>>(packed, N, K, bits, gscale, ids, M, x, ldx, status);
    return cudaGetLastError();
}

}  // namespace tfq
