// The quantised projection kernel: y[m][n] = sum_k xn[m][k] * (s q + b)[n][k].
//
// Work is a linear sequence of 16-row x 64-column tiles ("units"), ordered by
// problem (an MoE expert slot; one problem otherwise), K split, 16-row block,
// group. The grid is persistent (at most one CTA per SM); each CTA takes one
// contiguous range of it, either whole row blocks ("aligned", when that balances
// within about 10 %) or an exact 1/C share of the units ("stream-K", cutting row
// blocks anywhere). A CTA lists its segments (maximal runs inside one row block)
// once, then walks them in rounds: R teams of KW warps, one segment per team.
//
//   producer warp   one lane streams the range's tiles (contiguous per row block
//                   in the packed layout) into an nst-deep ring of shared-memory
//                   stages with bulk async copies (TMA engine) completing on
//                   mbarriers. It starts before the kernel waits on the previous
//                   grid (programmatic dependent launch), so the weight stream
//                   overlaps the previous kernel's tail, and it never stops
//                   between rounds.
//   consumer warps  (16) copy the activation rows of the current (problem,
//                   split) into shared memory with bulk copies, normalise and
//                   round them to bf16 when an RMSNorm is folded in, form the
//                   per-group sums of the rounded values and lay each group out
//                   in MMA B-fragment order. The KW warps of a team split the
//                   groups of their segment. Per 16x64 tile: one 16-byte (4-bit) load gives a
//                   lane its A fragments for four m16n8k16 MMAs; codes become
//                   bf16 (128 + q) pairs with one LOP3 each; the group epilogue
//                   folds scale and bias back in:
//                      y += s * sum_k x (128 + q) + (b - 128 s) * sum_k x
//                   which equals sum_k x (s q + b).
//   reduction       the warps of a team are summed through shared memory in fixed
//                   order. A segment that is a whole row block of an unsplit
//                   problem is stored directly; any other contributes an fp32
//                   partial to a workspace slot, and once the CTA has finished
//                   its range the last contributor of each row block (a counter
//                   per row block) sums the slots in (split, contributor) order,
//                   zeroes them and its counter again, and stores: deterministic,
//                   no float atomics, and the workspace is left as it was found.
//
// Every wait is bounded in wall time; a wait that runs out records TF_E_TIMEOUT
// in the status word and the CTA leaves after draining its own copies.
#pragma once

#include "tfq_internal.h"
#include "tfq_ptx.cuh"

namespace tfq {

struct QSmem {
    static constexpr int kFullOff = 0;    // full[8]
    static constexpr int kEmptyOff = 64;  // empty[8]
    static constexpr int kXbarOff = 128;  // activation copy barrier
    static constexpr int kFlagOff = 144;  // [0] abort
    static constexpr int kInvOff = 160;   // inv_rms[8]
    static constexpr int kRowOff = 192;   // activation row of each column [8]
    static constexpr int kSlotOff = 256;  // MoE: per problem {expert, count} [kMaxSlots] then rows [kMaxSlots][8]
    static constexpr int kSlotBytes = kMaxSlots * 8 + kMaxSlots * kMaxM * 4;
    static constexpr int kXsumOff = kSlotOff + kSlotBytes;  // xsum[Gs][8] fp32, then the offsets in the params
};

// Bounded by the SM cycle counter (cheap to read, unlike the global timer);
// limit_ns is converted at 2 cycles per ns, which over-estimates the wall time
// only at clocks below 2 GHz.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int* status, uint64_t limit_ns)
{
    if (mbar_test_wait(bar, parity))  // the common case: already complete, no suspension
        return true;
    const long long t0 = clock64();
    const long long limit = (long long)(limit_ns * 2);
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicCAS(status, 0, TF_E_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One 16x64 tile of affine codes against the B fragments (xa, xb) and group sums (xs)
// of its group.
template <int BITS>
__device__ __forceinline__ void tile_mac_affine(const uint8_t* tile, int lane, const uint4& xa, const uint4& xb,
                                                const float2& xs, float (&acc)[4])
{
    constexpr int QB = tile_q_bytes_for(BITS);
    const uint2 sb = *reinterpret_cast<const uint2*>(tile + QB + (lane >> 2) * 8);
    const float s_lo = bf16lo_f32(sb.x), s_hi = bf16hi_f32(sb.x);
    const float b_lo = bf16lo_f32(sb.y), b_hi = bf16hi_f32(sb.y);
    if constexpr (BITS == 4) {
        const uint4 wv = *reinterpret_cast<const uint4*>(tile + lane * 16);
        // two independent accumulation chains (k blocks 0, 2 and 1, 3) halve the
        // dependent MMA latency of a tile
        float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16_16816(d, nib2_bf16(wv.x), nib2_bf16(wv.x >> 4), nib2_bf16(wv.x >> 8), nib2_bf16(wv.x >> 12),
                       xa.x, xa.y);
        mma_bf16_16816(e, nib2_bf16(wv.y), nib2_bf16(wv.y >> 4), nib2_bf16(wv.y >> 8), nib2_bf16(wv.y >> 12),
                       xa.z, xa.w);
        mma_bf16_16816(d, nib2_bf16(wv.z), nib2_bf16(wv.z >> 4), nib2_bf16(wv.z >> 8), nib2_bf16(wv.z >> 12),
                       xb.x, xb.y);
        mma_bf16_16816(e, nib2_bf16(wv.w), nib2_bf16(wv.w >> 4), nib2_bf16(wv.w >> 8), nib2_bf16(wv.w >> 12),
                       xb.z, xb.w);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d[i] += e[i];
        // sum_k x (s q + b) = s * sum_k x (128 + q) + (b - 128 s) * sum_k x
        const float c_lo = fmaf(-128.f, s_lo, b_lo), c_hi = fmaf(-128.f, s_hi, b_hi);
        acc[0] = fmaf(s_lo, d[0], fmaf(c_lo, xs.x, acc[0]));
        acc[1] = fmaf(s_lo, d[1], fmaf(c_lo, xs.y, acc[1]));
        acc[2] = fmaf(s_hi, d[2], fmaf(c_hi, xs.x, acc[2]));
        acc[3] = fmaf(s_hi, d[3], fmaf(c_hi, xs.y, acc[3]));
    } else {
        // 8-bit code q = 16 hi + lo: two nibble MMAs per k block.
        const uint4 w01 = *reinterpret_cast<const uint4*>(tile + lane * 32);
        const uint4 w23 = *reinterpret_cast<const uint4*>(tile + lane * 32 + 16);
        float dl[4] = {0.f, 0.f, 0.f, 0.f}, dh[4] = {0.f, 0.f, 0.f, 0.f};
#define TFQ_KB8(w0, w1, b0, b1)                                                                             \
    mma_bf16_16816(dl, nib2_bf16(w0), nib2_bf16((w0) >> 8), nib2_bf16(w1), nib2_bf16((w1) >> 8), b0, b1); \
    mma_bf16_16816(dh, nib2_bf16((w0) >> 4), nib2_bf16((w0) >> 12), nib2_bf16((w1) >> 4), nib2_bf16((w1) >> 12), b0, b1);
        TFQ_KB8(w01.x, w01.y, xa.x, xa.y)
        TFQ_KB8(w01.z, w01.w, xa.z, xa.w)
        TFQ_KB8(w23.x, w23.y, xb.x, xb.y)
        TFQ_KB8(w23.z, w23.w, xb.z, xb.w)
#undef TFQ_KB8
        // sum_k x (s q + b) = s * (sum x (128+lo) + 16 sum x (128+hi)) + (b - 2176 s) * sum x
        const float c_lo = fmaf(-2176.f, s_lo, b_lo), c_hi = fmaf(-2176.f, s_hi, b_hi);
        acc[0] = fmaf(s_lo, fmaf(16.f, dh[0], dl[0]), fmaf(c_lo, xs.x, acc[0]));
        acc[1] = fmaf(s_lo, fmaf(16.f, dh[1], dl[1]), fmaf(c_lo, xs.y, acc[1]));
        acc[2] = fmaf(s_hi, fmaf(16.f, dh[2], dl[2]), fmaf(c_hi, xs.x, acc[2]));
        acc[3] = fmaf(s_hi, fmaf(16.f, dh[3], dl[3]), fmaf(c_hi, xs.y, acc[3]));
    }
}

// tile_mac with one accumulation chain for 4-bit codes (the caller keeps two tiles
// in flight, which hides the MMA latency); 8-bit codes as tile_mac.
template <int BITS>
__device__ __forceinline__ void tile_mac_chain(const uint8_t* tile, int lane, const uint4& xa, const uint4& xb,
                                               const float2& xs, float (&acc)[4])
{
    if constexpr (BITS == 4) {
        const uint2 sb = *reinterpret_cast<const uint2*>(tile + tile_q_bytes_for(4) + (lane >> 2) * 8);
        const uint4 wv = *reinterpret_cast<const uint4*>(tile + lane * 16);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16_16816(d, nib2_bf16(wv.x), nib2_bf16(wv.x >> 4), nib2_bf16(wv.x >> 8), nib2_bf16(wv.x >> 12),
                       xa.x, xa.y);
        mma_bf16_16816(d, nib2_bf16(wv.y), nib2_bf16(wv.y >> 4), nib2_bf16(wv.y >> 8), nib2_bf16(wv.y >> 12),
                       xa.z, xa.w);
        mma_bf16_16816(d, nib2_bf16(wv.z), nib2_bf16(wv.z >> 4), nib2_bf16(wv.z >> 8), nib2_bf16(wv.z >> 12),
                       xb.x, xb.y);
        mma_bf16_16816(d, nib2_bf16(wv.w), nib2_bf16(wv.w >> 4), nib2_bf16(wv.w >> 8), nib2_bf16(wv.w >> 12),
                       xb.z, xb.w);
        const float s_lo = bf16lo_f32(sb.x), s_hi = bf16hi_f32(sb.x);
        const float c_lo = fmaf(-128.f, s_lo, bf16lo_f32(sb.y)), c_hi = fmaf(-128.f, s_hi, bf16hi_f32(sb.y));
        acc[0] = fmaf(s_lo, d[0], fmaf(c_lo, xs.x, acc[0]));
        acc[1] = fmaf(s_lo, d[1], fmaf(c_lo, xs.y, acc[1]));
        acc[2] = fmaf(s_hi, d[2], fmaf(c_hi, xs.x, acc[2]));
        acc[3] = fmaf(s_hi, d[3], fmaf(c_hi, xs.y, acc[3]));
    } else {
        tile_mac_affine<BITS>(tile, lane, xa, xb, xs, acc);
    }
}

// The tile math on fp16 activations (B fragments converted from bf16 after staging).
//   4-bit: A registers 0 and 2 (rows gi) hold 1024 + q and registers 1 and 3 (rows
//   gi + 8) hold 1024 + 16 q (one LOP3 each, no shift), so
//      sum_k x (s q + b) = s D + (b - 1024 s) sum x          (rows gi)
//                        = (s / 16) D + (b - 64 s) sum x     (rows gi + 8)
//   8-bit: q = 16 hi + lo, and the low- and high-nibble MMAs of a k block share one
//   accumulator: D = sum x (1024 + lo) + sum x (1024 + 16 hi) = sum x q + 2048 sum x.
template <int BITS>
__device__ __forceinline__ void tile_mac_f16(const uint8_t* tile, int lane, const uint4& xa, const uint4& xb,
                                             const float2& xs, float (&acc)[4])
{
    constexpr int QB = tile_q_bytes_for(BITS);
    const uint2 sb = *reinterpret_cast<const uint2*>(tile + QB + (lane >> 2) * 8);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (BITS == 4) {
        const uint4 wv = *reinterpret_cast<const uint4*>(tile + lane * 16);
        mma_f16_16816(d, nib2_f16(wv.x), nib2_f16_x16(wv.x), nib2_f16(wv.x >> 8), nib2_f16_x16(wv.x >> 8), xa.x, xa.y);
        mma_f16_16816(d, nib2_f16(wv.y), nib2_f16_x16(wv.y), nib2_f16(wv.y >> 8), nib2_f16_x16(wv.y >> 8), xa.z, xa.w);
        mma_f16_16816(d, nib2_f16(wv.z), nib2_f16_x16(wv.z), nib2_f16(wv.z >> 8), nib2_f16_x16(wv.z >> 8), xb.x, xb.y);
        mma_f16_16816(d, nib2_f16(wv.w), nib2_f16_x16(wv.w), nib2_f16(wv.w >> 8), nib2_f16_x16(wv.w >> 8), xb.z, xb.w);
        const float s_lo = bf16lo_f32(sb.x), s_hi = bf16hi_f32(sb.x);
        const float c_lo = fmaf(-1024.f, s_lo, bf16lo_f32(sb.y)), c_hi = fmaf(-64.f, s_hi, bf16hi_f32(sb.y));
        const float s_hi16 = s_hi * 0.0625f;
        acc[0] = fmaf(s_lo, d[0], fmaf(c_lo, xs.x, acc[0]));
        acc[1] = fmaf(s_lo, d[1], fmaf(c_lo, xs.y, acc[1]));
        acc[2] = fmaf(s_hi16, d[2], fmaf(c_hi, xs.x, acc[2]));
        acc[3] = fmaf(s_hi16, d[3], fmaf(c_hi, xs.y, acc[3]));
    } else {
        const uint4 w01 = *reinterpret_cast<const uint4*>(tile + lane * 32);
        const uint4 w23 = *reinterpret_cast<const uint4*>(tile + lane * 32 + 16);
#define TFQ_KB8H(w0, w1, b0, b1)                                                                               \
    mma_f16_16816(d, nib2_f16(w0), nib2_f16((w0) >> 8), nib2_f16(w1), nib2_f16((w1) >> 8), b0, b1);            \
    mma_f16_16816(d, nib2_f16_x16(w0), nib2_f16_x16((w0) >> 8), nib2_f16_x16(w1), nib2_f16_x16((w1) >> 8), b0, b1);
        TFQ_KB8H(w01.x, w01.y, xa.x, xa.y)
        TFQ_KB8H(w01.z, w01.w, xa.z, xa.w)
        TFQ_KB8H(w23.x, w23.y, xb.x, xb.y)
        TFQ_KB8H(w23.z, w23.w, xb.z, xb.w)
#undef TFQ_KB8H
        const float s_lo = bf16lo_f32(sb.x), s_hi = bf16hi_f32(sb.x);
        const float c_lo = fmaf(-2048.f, s_lo, bf16lo_f32(sb.y)), c_hi = fmaf(-2048.f, s_hi, bf16hi_f32(sb.y));
        acc[0] = fmaf(s_lo, d[0], fmaf(c_lo, xs.x, acc[0]));
        acc[1] = fmaf(s_lo, d[1], fmaf(c_lo, xs.y, acc[1]));
        acc[2] = fmaf(s_hi, d[2], fmaf(c_hi, xs.x, acc[2]));
        acc[3] = fmaf(s_hi, d[3], fmaf(c_hi, xs.y, acc[3]));
    }
}

// The tile math of an NVFP4 tile. Each A register (two E2M1 codes of one row) becomes
// an fp16 pair and is multiplied by the row's E4M3 block scale, also converted to
// fp16: a 2-bit times a 4-bit significand is exact in fp16 (|w| <= 6 * 448, nonzero
// |w| >= 2^-10), so the MMA accumulates the weights themselves and there is no group
// epilogue; the matrix's global scale multiplies the finished sums. With bf16
// activations (F16 false) the exact fp16 weights are converted, again exactly, to bf16.
template <bool F16>
__device__ __forceinline__ void tile_mac_nvfp4(const uint8_t* tile, int lane, const uint4& xa, const uint4& xb,
                                               float (&acc)[4])
{
    const uint4 wv = *reinterpret_cast<const uint4*>(tile + lane * 16);
    const uint2 sv = *reinterpret_cast<const uint2*>(tile + tile_q_bytes_for(kNvfp4) + (lane >> 2) * 8);
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint32_t sp[4] = {e4m3x2_to_f16x2(sv.x), e4m3x2_to_f16x2(sv.x >> 16), e4m3x2_to_f16x2(sv.y),
                            e4m3x2_to_f16x2(sv.y >> 16)};
    const uint32_t b0[4] = {xa.x, xa.z, xb.x, xb.z}, b1[4] = {xa.y, xa.w, xb.y, xb.w};
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        uint32_t a0, a1, a2, a3;  // registers r: rows gi + 8 (r & 1), columns 2 t + 8 (r >> 1) + {0, 1}
        e2m1x8_to_f16x2(w[kb], a0, a1, a2, a3);
        a0 = hmul2_lo(a0, sp[kb]);
        a1 = hmul2_hi(a1, sp[kb]);
        a2 = hmul2_lo(a2, sp[kb]);
        a3 = hmul2_hi(a3, sp[kb]);
        if constexpr (F16)
            mma_f16_16816(acc, a0, a1, a2, a3, b0[kb], b1[kb]);
        else
            mma_bf16_16816(acc, f16x2_to_bf16x2(a0), f16x2_to_bf16x2(a1), f16x2_to_bf16x2(a2), f16x2_to_bf16x2(a3),
                           b0[kb], b1[kb]);
    }
}

// One tile on bf16 activations, any code (the lock-step team schedules).
template <int BITS>
__device__ __forceinline__ void tile_mac(const uint8_t* tile, int lane, const uint4& xa, const uint4& xb,
                                         const float2& xs, float (&acc)[4])
{
    if constexpr (BITS == kNvfp4)
        tile_mac_nvfp4<false>(tile, lane, xa, xb, acc);
    else
        tile_mac_affine<BITS>(tile, lane, xa, xb, xs, acc);
}

template <int BITS, bool F16>
__device__ __forceinline__ void tile_mac_x(const uint8_t* tile, int lane, const uint4& xa, const uint4& xb,
                                           const float2& xs, float (&acc)[4])
{
    if constexpr (BITS == kNvfp4)
        tile_mac_nvfp4<F16>(tile, lane, xa, xb, acc);
    else if constexpr (F16)
        tile_mac_f16<BITS>(tile, lane, xa, xb, xs, acc);
    else
        tile_mac_chain<BITS>(tile, lane, xa, xb, xs, acc);
}

// ---------------------------------------------------------------- activation staging
//
// A staged activation buffer holds rows rows[0..Mrows) of x, columns
// [xg0 * 64, (xg0 + xgc) * 64), in natural (row-major) order with row stride
// p.x_rs bytes = columns * 2 + 16: the 16-byte pieces of the 8 rows at one column
// then fall in 8 different bank groups, so the ldmatrix that builds the MMA's B
// fragments (8 rows x 16 bytes per matrix) is conflict-free.

// Input randomized Hadamard transform of one 64-column group held by 8 lanes (lane &
// 7 = chunk cc, columns 8 cc .. 8 cc + 7; every lane of the warp must call it): the
// signs byte's bit i negates column 8 cc + i, then the Sylvester-ordered 64-point
// Walsh-Hadamard transform as H8 over the columns inside a lane (three butterfly
// stages) and H8 over the chunks across the 8 lanes (three shuffle stages), scaled by
// 1/8: H64[8 c + i][8 c' + i'] = (-1)^(popcount(c & c') + popcount(i & i')).
__device__ __forceinline__ void rht_group(float (&v)[8], uint32_t sign_bits, int lane)
{
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if ((sign_bits >> i) & 1u)
            v[i] = -v[i];
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (!(i & h)) {
                const float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    const int cc = lane & 7;
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, v[i], h);
            v[i] = (cc & h) ? o - v[i] : v[i] + o;
        }
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] *= 0.125f;
}

// bf16 pairs <-> 8 floats
__device__ __forceinline__ void unpack8(const uint32_t (&vv)[4], float (&v)[8])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[2 * q] = bf16lo_f32(vv[q]);
        v[2 * q + 1] = bf16hi_f32(vv[q]);
    }
}

__device__ __forceinline__ void pack8(const float (&v)[8], uint32_t (&vv)[4])
{
#pragma unroll
    for (int q = 0; q < 4; ++q)
        vv[q] = f32x2_to_bf16x2(v[2 * q], v[2 * q + 1]);
}

// One thread: copy the rows into the buffer (and, with an RMSNorm, gamma into
// gbuf); completion on `bar`.
__device__ __forceinline__ void x_issue(const QProjParams& p, uint8_t* buf, uint8_t* gbuf, const int* rows, int Mrows,
                                        int64_t xbase, int xg0, int xgc, uint64_t* bar)
{
    const bool norm = p.gamma != nullptr;
    mbar_arrive_expect_tx(bar, (uint32_t)(Mrows * xgc * 128 + (norm ? p.K * 2 : 0)));
    for (int m = 0; m < Mrows; ++m)
        bulk_g2s_plain(buf + m * p.x_rs, p.x + xbase + (int64_t)rows[m] * p.ldx + (int64_t)xg0 * kGroup,
                       (uint32_t)(xgc * 128), bar);
    if (norm)
        bulk_g2s_plain(gbuf, p.gamma, (uint32_t)(p.K * 2), bar);
}

// Consumer warps (nwarps of them, named barrier bar_id): after the copy has landed,
// RMSNorm statistics when gamma is set (the whole row is staged then), then for the
// groups [g_lo, g_lo + ng) of the problem (staged from group xg0): normalise and
// round to bf16 in place (with an RMSNorm), and group sums of the values used into
// xs[(g - g_lo) * 8 + m] (zero for rows >= Mrows).
__device__ __forceinline__ void x_prepare(const QProjParams& p, uint8_t* buf, const uint8_t* gbuf, int Mrows, int xg0,
                                          int g_lo, int ng, float* xs, float* inv_rms, int cw, int lane, int nwarps,
                                          int bar_id)
{
    const bool norm = p.gamma != nullptr;
    if (norm) {
        for (int m = cw; m < Mrows; m += nwarps) {
            const uint4* row = reinterpret_cast<const uint4*>(buf + m * p.x_rs);
            float sq[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i = lane; i < p.K / 8; i += 32) {
                const uint4 v = row[i];
                const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float a = bf16lo_f32(vv[q]), b = bf16hi_f32(vv[q]);
                    sq[q] = fmaf(b, b, fmaf(a, a, sq[q]));
                }
            }
            float ss = warp_sum((sq[0] + sq[1]) + (sq[2] + sq[3]));
            if (lane == 0)
                inv_rms[m] = rsqrtf(ss / (float)p.K + p.eps);
        }
        named_bar_sync(bar_id, nwarps * 32);
    }
    // group sums of the rows that are not there are zero
    for (int i = cw * 32 + lane; i < ng * kMaxM; i += nwarps * 32)
        if ((i & 7) >= Mrows)
            xs[i] = 0.f;
    // a lane handles one 8-column chunk cc of one (group, live row)
    for (int base = cw * 4; base < ng * Mrows; base += nwarps * 4) {
        const int pi = base + (lane >> 3);
        const int cc = lane & 7;
        const int gl = pi / Mrows, m = pi - gl * Mrows;
        const bool valid = pi < ng * Mrows;
        float part = 0.f;
        if (valid) {
            uint4* chunk = reinterpret_cast<uint4*>(buf + m * p.x_rs + (g_lo - xg0 + gl) * 128) + cc;
            uint4 v = *chunk;
            uint32_t vv[4] = {v.x, v.y, v.z, v.w};
            if (norm) {
                const uint4 gv = *reinterpret_cast<const uint4*>(gbuf + ((g_lo + gl) * kGroup + cc * 8) * 2);
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
            xs[gl * kMaxM + m] = part;
    }
    named_bar_sync(bar_id, nwarps * 32);
}

// Activations of an unsplit call staged straight from global memory (where the
// previous kernel left them, so loads bypass L1) through registers: every 8-column
// chunk c of row m is (normalised, rounded and) summed over its group by the 8 lanes
// that hold the group, and stored at buf + m * x_rs + c * 16; group sums go to
// xs[g * 8 + m] (zero for rows >= Mrows). With an RMSNorm a warp owns a row (K <= 1024: four chunks a lane), so
// the row's sum of squares is a warp reduction; without one, (row, chunk) items
// are spread over all consumer threads, four loads in flight per thread.
__device__ __forceinline__ void x_put_chunk(uint8_t* buf, int x_rs, float* xs, int m, int c, bool valid,
                                            const uint32_t (&vv)[4])
{
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        part += bf16lo_f32(vv[q]) + bf16hi_f32(vv[q]);
    part += __shfl_xor_sync(0xffffffffu, part, 4);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    if (!valid)
        return;
    *reinterpret_cast<uint4*>(buf + m * x_rs + c * 16) = make_uint4(vv[0], vv[1], vv[2], vv[3]);
    if ((c & 7) == 0)
        xs[(c >> 3) * kMaxM + m] = part;
}

// The rows x[m][0, K) (m < Mrows, row stride ldx) of an unsplit call; gamma != NULL
// folds the RMSNorm in (K <= 1024); fragments at buf (row stride x_rs).
// NB: loads a thread keeps in flight at once on the path without an RMSNorm (rounded
// up to whole sets of kMaxM rows).
template <int NB = 4>
__device__ __forceinline__ void x_direct_raw(const uint16_t* x, int64_t ldx, int K, const uint16_t* gamma, float eps,
                                             int x_rs, uint8_t* buf, int Mrows, float* xs, float* ss_part, int cw,
                                             int lane, int nwarps, int bar_id)
{
    const int groups = K / kGroup;
    const int nch = groups * 8;  // 8-column chunks per row
    for (int i = cw * 32 + lane; i < groups * kMaxM; i += nwarps * 32)
        if ((i & 7) >= Mrows)
            xs[i] = 0.f;
    if (gamma != nullptr) {
        // one warp a row, four chunks a lane (K <= 1024): the row's sum of squares is a
        // warp reduction in an order that does not depend on how many rows are staged,
        // so a row normalises to the same bits alone or in a block of eight
        const int nch_row = nch;
        const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
        for (int m = cw; m < Mrows; m += nwarps) {
            const uint4* x4 = reinterpret_cast<const uint4*>(x + (int64_t)m * ldx);
            uint4 v[4], gv[4];
            float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = j * 32 + lane;
                const bool ok = c < nch_row;
                v[j] = ok ? __ldcg(x4 + c) : make_uint4(0u, 0u, 0u, 0u);
                gv[j] = ok ? __ldg(g4 + c) : make_uint4(0u, 0u, 0u, 0u);
            }
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
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j * 32 >= nch_row)  // warp-uniform
                    break;
                const int c = j * 32 + lane;
                const uint32_t xv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                const uint32_t gg[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
                uint32_t vv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    vv[q] = f32x2_to_bf16x2(bf16lo_f32(xv[q]) * inv * bf16lo_f32(gg[q]),
                                            bf16hi_f32(xv[q]) * inv * bf16hi_f32(gg[q]));
                x_put_chunk(buf, x_rs, xs, m, c, c < nch_row, vv);
            }
        }
    } else {
        // thread t takes chunks c = t, t + T, ... of every row: NB loads in flight
        const int T = nwarps * 32;
        for (int c_base = 0; c_base < nch; c_base += T * ((NB + kMaxM - 1) / kMaxM)) {
#pragma unroll
            for (int jc = 0; jc < (NB + kMaxM - 1) / kMaxM; ++jc) {
                const int c_w = c_base + jc * T + cw * 32;  // warp-uniform
                if (c_w >= nch)
                    break;
                const int c = c_w + lane;
                uint4 v[kMaxM];
#pragma unroll
                for (int m = 0; m < kMaxM; ++m)
                    v[m] = (m < Mrows && c < nch)
                               ? __ldcg(reinterpret_cast<const uint4*>(x + (int64_t)m * ldx) + c)
                               : make_uint4(0u, 0u, 0u, 0u);
                if (Mrows == 1) {  // uniform
                    const uint32_t vv[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
                    x_put_chunk(buf, x_rs, xs, 0, c, c < nch, vv);
                } else {
                    // each row's partial sums of the chunk, then a butterfly over the 8 lanes
                    // of the group (4 + 2 + 1 shuffles for all 8 rows, not 3 per row) leaves
                    // lane l with row (l & 7)'s group sum, added in the same order as the
                    // per-row reduction of x_put_chunk (so the sums are the same bits)
                    float a[kMaxM];
#pragma unroll
                    for (int m = 0; m < kMaxM; ++m) {
                        const uint32_t vv[4] = {v[m].x, v[m].y, v[m].z, v[m].w};
                        float part = 0.f;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            part += bf16lo_f32(vv[q]) + bf16hi_f32(vv[q]);
                        a[m] = part;
                        if (m < Mrows && c < nch)
                            *reinterpret_cast<uint4*>(buf + m * x_rs + c * 16) = v[m];
                    }
                    const bool h4 = (lane & 4) != 0, h2 = (lane & 2) != 0, h1 = (lane & 1) != 0;
                    float b[4], d2[2];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float r = __shfl_xor_sync(0xffffffffu, h4 ? a[i] : a[i + 4], 4);
                        b[i] = (h4 ? a[i + 4] : a[i]) + r;
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float r = __shfl_xor_sync(0xffffffffu, h2 ? b[i] : b[i + 2], 2);
                        d2[i] = (h2 ? b[i + 2] : b[i]) + r;
                    }
                    const float r = __shfl_xor_sync(0xffffffffu, h1 ? d2[0] : d2[1], 1);
                    const float sum = (h1 ? d2[1] : d2[0]) + r;  // group sum of row lane & 7
                    if (c < nch && (lane & 7) < Mrows)
                        xs[(c >> 3) * kMaxM + (lane & 7)] = sum;
                }
            }
        }
    }
    named_bar_sync(bar_id, nwarps * 32);
}

__device__ __forceinline__ void x_direct(const QProjParams& p, uint8_t* buf, int Mrows, float* xs, float* ss_part,
                                         int cw, int lane, int nwarps, int bar_id)
{
    x_direct_raw<4>(p.x, p.ldx, p.K, p.gamma, p.eps, p.x_rs, buf, Mrows, xs, ss_part, cw, lane, nwarps, bar_id);
}

// Input Hadamard transform of a staged buffer, in place: groups [0, ng) of rows
// [0, Mrows) (the buffer's group gl is group g_abs0 + gl of K), then their group sums
// again; 8 lanes a (group, row), four a warp at a time. Runs between the staging and
// the tile loop, so the staging code carries none of it; ends with a barrier.
__device__ __forceinline__ void x_rht(uint8_t* buf, int x_rs, float* xs, int Mrows, int g_abs0, int ng,
                                     const uint8_t* rht, int cw, int lane, int nwarps, int bar_id)
{
    const int cc = lane & 7;
    for (int base = cw * 4; base < ng * Mrows; base += nwarps * 4) {
        const int pi = base + (lane >> 3);
        const bool valid = pi < ng * Mrows;
        const int gl = valid ? pi / Mrows : 0, m = valid ? pi - gl * Mrows : 0;
        uint4* chunk = reinterpret_cast<uint4*>(buf + m * x_rs + gl * 128) + cc;
        uint32_t vv[4] = {0u, 0u, 0u, 0u};
        if (valid) {
            const uint4 v = *chunk;
            vv[0] = v.x;
            vv[1] = v.y;
            vv[2] = v.z;
            vv[3] = v.w;
        }
        float f[8];
        unpack8(vv, f);
        rht_group(f, valid ? __ldg(rht + (g_abs0 + gl) * 8 + cc) : 0u, lane);
        pack8(f, vv);
        float part = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            part += bf16lo_f32(vv[q]) + bf16hi_f32(vv[q]);
        part += __shfl_xor_sync(0xffffffffu, part, 4);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        if (valid) {
            *chunk = make_uint4(vv[0], vv[1], vv[2], vv[3]);
            if (cc == 0)
                xs[gl * kMaxM + m] = part;
        }
    }
    named_bar_sync(bar_id, nwarps * 32);
}

// The B fragments (xa: k blocks 0, 1; xb: k blocks 2, 3) of group g_rel of a buffer,
// by two ldmatrix of four 8x8 matrices each (warp-wide: every lane must call it):
// lane l gives the address of row l % 8 of matrix l / 8 (columns 8 (l / 8) .. + 7 of
// the half group), and receives in register i the pair (row l / 4, columns 2 (l % 4),
// +1) of matrix i, which is its B-fragment word. Only rows < mrows are staged (and
// addressed: the others point at row 0); their fragments read as zero.
__device__ __forceinline__ void x_frag(const uint8_t* buf, int x_rs, int gi, int tq, int g_rel, int mrows, uint4& xa,
                                       uint4& xb)
{
    const int lane = gi * 4 + tq;
    const int r = (lane & 7) < mrows ? (lane & 7) : 0;
    const uint32_t a = smem_u32(buf + r * x_rs + g_rel * 128 + (lane >> 3) * 16);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(xa.x), "=r"(xa.y), "=r"(xa.z), "=r"(xa.w)
                 : "r"(a));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(xb.x), "=r"(xb.y), "=r"(xb.z), "=r"(xb.w)
                 : "r"(a + 64));
    if (gi >= mrows) {
        xa = make_uint4(0u, 0u, 0u, 0u);
        xb = xa;
    }
}

// B fragments of group g_rel of a buffer whose 8 rows are all staged (rows >= M
// zero-filled): the same two ldmatrix as x_frag, without the row clamp.
__device__ __forceinline__ void x_frag8_row(const uint8_t* xrow, int lane, int g_rel, uint4& xa, uint4& xb)
{
    const uint32_t a = smem_u32(xrow + g_rel * 128 + (lane >> 3) * 16);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(xa.x), "=r"(xa.y), "=r"(xa.z), "=r"(xa.w)
                 : "r"(a));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(xb.x), "=r"(xb.y), "=r"(xb.z), "=r"(xb.w)
                 : "r"(a + 64));
}

__device__ __forceinline__ void x_frag8(const uint8_t* buf, int x_rs, int lane, int g_rel, uint4& xa, uint4& xb)
{
    x_frag8_row(buf + (lane & 7) * x_rs, lane, g_rel, xa, xb);
}

// True when some bf16 value in rows [0, rows) of a staged buffer (cols columns) has
// |v| >= 2^e_lim or is not finite. 2^16: an fp16 copy would not hold it exactly; 2^12
// for 4-bit codes, whose fp16 offset of 1024 code units (against 128 in bf16) would
// otherwise cost more in the cancellation s D - 1024 s sum x than the bf16 path.
template <int e_lim>
__device__ __forceinline__ bool x_beyond_f16(const uint8_t* buf, int x_rs, int rows, int cols, int t, int nt)
{
    constexpr uint32_t kLim = (127u + e_lim) << 7;  // bf16 exponent field of 2^e_lim
    const int per_row = cols / 8;  // 16-byte chunks
    bool big = false;
    for (int i = t; i < rows * per_row; i += nt) {
        const int m = i / per_row, c = i - m * per_row;
        const uint4 v = *reinterpret_cast<const uint4*>(buf + m * x_rs + c * 16);
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            big |= (vv[q] & 0x7F80u) >= kLim || ((vv[q] >> 16) & 0x7F80u) >= kLim;
    }
    return big;
}

// Rows [0, rows) of a staged buffer from bf16 to fp16 in place.
__device__ __forceinline__ void x_to_f16(uint8_t* buf, int x_rs, int rows, int cols, int t, int nt)
{
    const int per_row = cols / 8;
    for (int i = t; i < rows * per_row; i += nt) {
        const int m = i / per_row, c = i - m * per_row;
        uint4* ptr = reinterpret_cast<uint4*>(buf + m * x_rs + c * 16);
        const uint4 v = *ptr;
        *ptr = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
    }
}

// Final values of one lane's accumulator fragment (rows row0 + gi, row0 + gi + 8;
// columns 2t, 2t + 1) -> outputs.
template <bool DUAL, bool MOE>
__device__ __forceinline__ void store_outputs(const QProjParams& p, int prob, int Mrows, int row0, int lane,
                                              const float (&a0)[4], const float (&a1)[4])
{
    const int gi = lane >> 2, t = lane & 3;
    const int64_t ybase = MOE ? (int64_t)prob * p.y_slot_stride : 0;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int n = row0 + gi + 8 * (v >> 1);
        const int m = 2 * t + (v & 1);
        if (n >= p.N || m >= Mrows)
            continue;
        float val;
        if constexpr (DUAL) {
            const float g = a0[v];
            val = g / (1.f + expf(-g)) * a1[v];
        } else {
            val = a0[v];
        }
        if (!MOE && p.residual != nullptr)  // written by an earlier kernel: read through L2, not L1
            val += __uint_as_float((uint32_t)__ldcg(p.residual + (int64_t)m * p.ldr + n) << 16);
        const int64_t idx = ybase + (int64_t)m * p.ldy + n;
        if (p.y_f32)
            static_cast<float*>(p.y)[idx] = val;
        else
            static_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(val);
    }
}

// Static partition of the unit sequence over the CTAs.
//   aligned  : CTA c takes whole (problem, split, row-block) items [I c / C, I (c+1) / C)
//   stream-K : CTA c takes units [U c / C, U (c+1) / C), cutting row blocks anywhere
struct Part {
    int64_t items, U;
    int C;       // CTAs with work: min(grid, items or U)
    int per_p;   // units per problem = n_rb * groups
    int per_ps;  // units per (problem, split) = n_rb * Gs
    int Gs;
    bool aligned;
    // floor(a c / C) for 0 <= c <= C <= 2^16 in 32-bit arithmetic
    __device__ __forceinline__ static uint32_t muldiv(uint32_t a, uint32_t c, uint32_t C)
    {
        const uint32_t q = a / C, r = a - q * C;
        return q * c + r * c / C;
    }
    __device__ __forceinline__ int64_t start(int c) const
    {
        return aligned ? (int64_t)muldiv((uint32_t)items, (uint32_t)c, (uint32_t)C) * Gs
                       : (int64_t)muldiv((uint32_t)U, (uint32_t)c, (uint32_t)C);
    }
    float inv_U;  // 1 / U, for the quotient estimate below
    // floor(((u + 1) C - 1) / U): the quotient is at most C, so a float estimate is within
    // one of it; two integer comparisons make it exact
    __device__ __forceinline__ int cta_of(int64_t u) const
    {
        const int64_t n = (u + 1) * C - 1;
        int q = (int)((float)n * inv_U);
        if ((int64_t)(q + 1) * U <= n)
            ++q;
        else if ((int64_t)q * U > n)
            --q;
        return q;
    }
    // CTAs contributing to the row block starting at unit f (stream-K only)
    __device__ __forceinline__ int contributors(int64_t f) const { return cta_of(f + Gs - 1) - cta_of(f) + 1; }
};

// Sum of the fp32 partial slots of row block rb of problem prob, in (split,
// contributor) order, zeroing every slot read (the workspace is left as it was
// found). Loads are issued B slots at a time before any is used, so the L2 round
// trips overlap.
template <bool DUAL, int B = 4>
__device__ __forceinline__ void sum_partials(const QProjParams& p, const Part& pt, int prob, int rb, int lane,
                                             float (&t0)[4], float (&t1)[4])
{
    constexpr int VALS = DUAL ? 8 : 4;
    auto kc_of = [&](int s2) {
        return pt.aligned ? 1
                          : min(pt.contributors((int64_t)prob * pt.per_p + (int64_t)s2 * pt.per_ps + (int64_t)rb * p.Gs),
                                p.kmax);
    };
    int s2 = 0, kq = 0, kc = kc_of(0);
    while (s2 < p.S) {
        float4* src[B];
        bool valid[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            valid[j] = s2 < p.S;
            src[j] = nullptr;
            if (valid[j]) {
                src[j] = reinterpret_cast<float4*>(
                    p.partials + (((((int64_t)prob * p.S + s2) * p.n_rb + rb) * p.kmax + kq) * 32 + lane) * VALS);
                if (++kq == kc) {
                    kq = 0;
                    if (++s2 < p.S)
                        kc = kc_of(s2);
                }
            }
        }
        float4 a[B], b[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (valid[j]) {
                a[j] = __ldcg(src[j]);
                if constexpr (DUAL)
                    b[j] = __ldcg(src[j] + 1);
            }
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            if (valid[j]) {
                __stcg(src[j], make_float4(0.f, 0.f, 0.f, 0.f));
                t0[0] += a[j].x;
                t0[1] += a[j].y;
                t0[2] += a[j].z;
                t0[3] += a[j].w;
                if constexpr (DUAL) {
                    __stcg(src[j] + 1, make_float4(0.f, 0.f, 0.f, 0.f));
                    t1[0] += b[j].x;
                    t1[1] += b[j].y;
                    t1[2] += b[j].z;
                    t1[3] += b[j].w;
                }
            }
        }
    }
}

constexpr int kBarConsumers = 15;  // named barrier of all consumer warps; 1..8 are team barriers

// Light teams (NWT = 8) run two CTAs per SM (and leave room for the next kernel's).
template <int BITS, bool DUAL, bool MOE, int KW, int NWT>
__global__ void __launch_bounds__((NWT + 1) * 32, NWT == 8 ? 2 : 1) qproj_kernel(const __grid_constant__ QProjParams p)
{
    constexpr int R = NWT / KW;
    constexpr int MATS = DUAL ? 2 : 1;
    constexpr int TILE = tile_bytes_for(BITS);
    constexpr int VALS = DUAL ? 8 : 4;
    constexpr int NCT = NWT * 32;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + QSmem::kFullOff);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + QSmem::kEmptyOff);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + QSmem::kXbarOff);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + QSmem::kFlagOff);  // [0] abort [1] snapshot
    int* counts = reinterpret_cast<int*>(smem + QSmem::kFlagOff + 8);                // [0] segments [1] rounds
    float* inv_rms = reinterpret_cast<float*>(smem + QSmem::kInvOff);
    int* rowsel = reinterpret_cast<int*>(smem + QSmem::kRowOff);
    int2* slot_ec = reinterpret_cast<int2*>(smem + QSmem::kSlotOff);                   // {expert, count}
    int* slot_rows = reinterpret_cast<int*>(smem + QSmem::kSlotOff + kMaxSlots * 8);  // [slot][8]
    float* xsum = reinterpret_cast<float*>(smem + QSmem::kXsumOff);
    float* red = reinterpret_cast<float*>(smem + p.red_off);
    int4* segs = reinterpret_cast<int4*>(smem + p.seg_off);      // {problem, split, row block, g0 << 16 | len}
    int2* rounds = reinterpret_cast<int2*>(smem + p.round_off);  // {first segment, longest segment}
    int* lastf = reinterpret_cast<int*>(smem + p.last_off);      // per segment: this CTA sums the row block
    uint8_t* xraw = smem + p.xraw_off;
    uint8_t* stages = smem + p.stage_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const int stage_bytes = MATS * R * p.cg * TILE;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NWT);
        }
        mbar_init(xbar, 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (!MOE)
        pdl_launch_dependents();

    int P = p.P;
    if constexpr (MOE) {
        // the routing table comes from the previous kernel, or from an earlier one that had
        // completed before this launch could start (meta_ready: the gate/up launch waited for
        // it before it let its dependents start, so the down launch reads it at once and
        // streams its experts' weights while gate/up finishes)
        if (!p.meta_ready)
            pdl_wait();
        pdl_launch_dependents();
        P = __ldcg(&p.meta->n_active);
        for (int i = threadIdx.x; i < P; i += blockDim.x) {
            slot_ec[i] = make_int2(__ldcg(&p.meta->slot[i].expert), __ldcg(&p.meta->slot[i].count));
            for (int j = 0; j < kMaxM; ++j)
                slot_rows[i * kMaxM + j] = p.gather ? __ldcg(&p.meta->slot[i].rows[j]) : j;
        }
    }
    Part pt;
    pt.per_p = p.n_rb * p.groups;
    pt.per_ps = p.n_rb * p.Gs;
    pt.Gs = p.Gs;
    pt.aligned = p.aligned != 0;
    pt.items = (int64_t)P * p.S * p.n_rb;
    pt.U = pt.items * p.Gs;
    pt.inv_U = 1.f / (float)max(pt.U, (int64_t)1);
    pt.C = (int)min((int64_t)p.C, max(pt.aligned ? pt.items : pt.U, (int64_t)1));
    int64_t u0 = 0, u1 = 0;
    if (c < pt.C) {  // CTAs past the work (fewer MoE slots active than planned for) stay idle
        if (pt.aligned && pt.C == pt.items) {  // one item per CTA: no division
            u0 = (int64_t)c * p.Gs;
            u1 = u0 + p.Gs;
        } else {
            u0 = pt.start(c);
            u1 = pt.start(c + 1);
        }
    }

    // ---- this CTA's segments (maximal runs inside one (problem, split, row block)) and
    // rounds (up to R consecutive segments of one (problem, split)), built by warp 0 with
    // a lane per segment and read by every warp
    if (warp == 0) {
        int nseg = 0, nround = 0;
        if (u0 < u1 && pt.items == p.n_rb && pt.aligned && pt.C == pt.items) {  // row block c, whole
            nseg = 1;
            nround = 1;
            if (lane == 0) {
                segs[0] = make_int4(0, 0, c, p.Gs);
                rounds[0] = make_int2(0, p.Gs);
            }
        } else if (u0 < u1) {
            const int Gs = p.Gs, a0 = (int)u0, a1 = (int)u1;  // units fit in 30 bits (checked on the host)
            const int b0 = a0 / Gs;                            // (problem, split, row block) flattened
            nseg = (a1 - 1) / Gs - b0 + 1;
            if (nseg > p.segmax) {  // the host sizes the list; never expected
                nseg = 0;
                if (lane == 0) {
                    flags[0] = 1;
                    atomicCAS(p.status, 0, TF_E_INTERNAL);
                }
            }
            for (int i0 = 0; i0 < nseg; i0 += 32) {
                const int i = i0 + lane;
                bool starts = false;
                if (i < nseg) {
                    const int idx = b0 + i;
                    const int key = idx / p.n_rb, rb = idx - key * p.n_rb;
                    const int pp = key / p.S, ss = key - pp * p.S;
                    const int lo = max(a0, idx * Gs), hi = min(a1, (idx + 1) * Gs);
                    segs[i] = make_int4(pp, ss, rb, ((lo - idx * Gs) << 16) | (hi - lo));
                    // a round starts every R segments of the CTA's run of one (problem, split)
                    starts = (idx - max(key * p.n_rb, b0)) % R == 0;
                }
                const unsigned bal = __ballot_sync(0xffffffffu, starts);
                if (starts)
                    rounds[nround + __popc(bal & ((1u << lane) - 1u))].x = i;
                nround += __popc(bal);
            }
            __syncwarp();
            for (int t = lane; t < nround; t += 32) {  // longest segment of each round
                const int e = t + 1 < nround ? rounds[t + 1].x : nseg;
                int m = 0;
                for (int i = rounds[t].x; i < e; ++i)
                    m = max(m, segs[i].w & 0xFFFF);
                rounds[t].y = m;
            }
        }
        __syncwarp();
        if (lane == 0) {
            rounds[nround].x = nseg;
            counts[0] = nseg;
            counts[1] = flags[0] ? 0 : nround;
        }
    }
    __syncthreads();
    const int nseg = counts[0], nround = counts[1];

    // ------------------------------------------------------------ producer
    if (warp == NWT) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int st_global = 0;
            bool ok = true;
            for (int t = 0; t < nround && ok; ++t) {
                const int i0 = rounds[t].x, n = rounds[t + 1].x - i0, maxlen = rounds[t].y;
                const int4 first = segs[i0];
                const int64_t mbase = MOE ? (int64_t)slot_ec[first.x].x * p.matrix_bytes : 0;
                for (int g = 0; g < maxlen; g += p.cg, ++st_global) {
                    const int s = st_global % p.nst;
                    const uint32_t ph = (st_global / p.nst) & 1u;
                    if (!wait_or_abort(&empty[s], ph ^ 1u, flags, p.status, p.limit_ns)) {
                        ok = false;
                        break;
                    }
                    uint32_t bytes = 0;
                    for (int r = 0; r < n; ++r)
                        bytes += (uint32_t)max(0, min(p.cg, (segs[i0 + r].w & 0xFFFF) - g)) * TILE;
                    mbar_arrive_expect_tx(&full[s], bytes * MATS);
                    uint8_t* sbase = stages + s * stage_bytes;
                    for (int r = 0; r < n; ++r) {
                        const int4 e = segs[i0 + r];
                        const int cnt = min(p.cg, (e.w & 0xFFFF) - g);
                        if (cnt <= 0)
                            continue;
                        const int64_t tile = (int64_t)e.z * p.groups + e.y * p.Gs + (e.w >> 16) + g;
#pragma unroll
                        for (int mat = 0; mat < MATS; ++mat) {
                            const uint8_t* src = (mat ? p.w1 : p.w0) + mbase + tile * TILE;
                            bulk_g2s(sbase + (mat * R + r) * p.cg * TILE, src, (uint32_t)(cnt * TILE), &full[s], pol);
                        }
                    }
                }
            }
            // no copy may still be in flight when the CTA leaves (also after an abort:
            // copies complete by themselves, so this wait ignores the abort flag)
            for (int q = max(0, st_global - p.nst); q < st_global; ++q)
                mbar_wait_bounded(&full[q % p.nst], (q / p.nst) & 1u, p.limit_ns);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int cw = warp;
    const int r_me = cw / KW, kp = cw % KW;
    const int gi = lane >> 2, tq = lane & 3;
    if (!MOE || p.meta_ready)  // the activations come from the previous kernel
        pdl_wait();
    const bool norm = p.gamma != nullptr;
    bool alive = true;
    int cur_p = -1, cur_s = -1, Mrows = p.M, xphase = 0, nstaged = 0, st_global = 0;

    for (int t = 0; t < nround; ++t) {
        const int i0 = rounds[t].x, n = rounds[t + 1].x - i0, maxlen = rounds[t].y;
        const int4 first = segs[i0];

        if (first.x != cur_p || first.y != cur_s) {
            // ---- stage the activation rows of (problem, split): the whole row when an
            // RMSNorm is folded in (its statistics need every column), else the split's groups
            named_bar_sync(kBarConsumers, NCT);  // everyone is done with the previous rows
            if (MOE)
                Mrows = slot_ec[first.x].y;
            if (!MOE && p.x_direct) {  // unsplit plain rows: no bulk copy, no wait
                x_direct(p, xraw, Mrows, xsum, red, cw, lane, NWT, kBarConsumers);
                if (!MOE && p.rht != nullptr)
                    x_rht(xraw, p.x_rs, xsum, Mrows, 0, p.groups, p.rht, cw, lane, NWT, kBarConsumers);
            } else {
                if (threadIdx.x < kMaxM)
                    rowsel[threadIdx.x] = MOE ? slot_rows[first.x * kMaxM + threadIdx.x] : (int)threadIdx.x;
                const int xg0 = norm ? 0 : first.y * p.Gs;
                const int xgc = norm ? p.groups : p.Gs;
                if (cw == 0) {
                    __syncwarp();
                    if (lane == 0 && !flags[0])
                        x_issue(p, xraw, smem + p.gamma_off, rowsel, Mrows,
                                MOE && !p.gather ? (int64_t)first.x * p.x_slot_stride : 0, xg0, xgc, xbar);
                }
                bool ok = alive && wait_or_abort(xbar, (uint32_t)xphase, flags, p.status, p.limit_ns);
                xphase ^= 1;
                ++nstaged;
                alive = __all_sync(0xffffffffu, ok);
                x_prepare(p, xraw, smem + p.gamma_off, Mrows, xg0, first.y * p.Gs, p.Gs, xsum, inv_rms, cw, lane, NWT,
                          kBarConsumers);
                if (!MOE && p.rht != nullptr)  // the split's groups, where the buffer holds them
                    x_rht(xraw + (first.y * p.Gs - xg0) * 128, p.x_rs, xsum, Mrows, first.y * p.Gs, p.Gs, p.rht, cw,
                          lane, NWT, kBarConsumers);
            }
            cur_p = first.x;
            cur_s = first.y;
        }

        // ---- this team's segment of the round
        int rb = 0, gs = 0, len = 0;
        if (r_me < n) {
            const int4 e = segs[i0 + r_me];
            rb = e.z;
            gs = e.w >> 16;
            len = e.w & 0xFFFF;
        }
        const int xoff = norm ? first.y * p.Gs : 0;  // first group of the split inside the staged rows
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        float bcc0[4] = {0.f, 0.f, 0.f, 0.f}, bcc1[4] = {0.f, 0.f, 0.f, 0.f};  // second chain
        for (int g = 0; g < maxlen; g += p.cg, ++st_global) {
            const int s = st_global % p.nst;
            const uint32_t ph = (st_global / p.nst) & 1u;
            bool ok = alive && wait_or_abort(&full[s], ph, flags, p.status, p.limit_ns);
            alive = __all_sync(0xffffffffu, ok);
            const int cnt = alive ? min(p.cg, len - g) : 0;
            const uint8_t* sbase = stages + s * stage_bytes;
            const uint8_t* t0 = sbase + (r_me * p.cg) * TILE;
            const uint8_t* t1 = sbase + ((R + r_me) * p.cg) * TILE;
            int j = kp;
            // a single matrix takes two tiles per iteration into separate accumulators (gate
            // and up are two independent chains already)
            for (; !DUAL && j + KW < cnt; j += 2 * KW) {
                const int gl = gs + g + j;  // group within the split
                uint4 xa, xb, ya, yb;
                x_frag(xraw, p.x_rs, gi, tq, xoff + gl, Mrows, xa, xb);
                x_frag(xraw, p.x_rs, gi, tq, xoff + gl + KW, Mrows, ya, yb);
                const float2 xs = *reinterpret_cast<const float2*>(xsum + gl * kMaxM + 2 * tq);
                const float2 ys = *reinterpret_cast<const float2*>(xsum + (gl + KW) * kMaxM + 2 * tq);
                tile_mac<BITS>(t0 + j * TILE, lane, xa, xb, xs, acc0);
                tile_mac<BITS>(t0 + (j + KW) * TILE, lane, ya, yb, ys, bcc0);
                if constexpr (DUAL) {
                    tile_mac<BITS>(t1 + j * TILE, lane, xa, xb, xs, acc1);
                    tile_mac<BITS>(t1 + (j + KW) * TILE, lane, ya, yb, ys, bcc1);
                }
            }
            for (; j < cnt; j += KW) {
                const int gl = gs + g + j;
                uint4 xa, xb;
                x_frag(xraw, p.x_rs, gi, tq, xoff + gl, Mrows, xa, xb);
                const float2 xs = *reinterpret_cast<const float2*>(xsum + gl * kMaxM + 2 * tq);
                tile_mac<BITS>(t0 + j * TILE, lane, xa, xb, xs, acc0);
                if constexpr (DUAL)
                    tile_mac<BITS>(t1 + j * TILE, lane, xa, xb, xs, acc1);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
        }

#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc0[i] += bcc0[i];
            acc1[i] += bcc1[i];
        }
        // ---- sum the KW warps of the team (team barrier: ids 1..R)
        if constexpr (KW > 1) {
            if (t > 0)
                named_bar_sync(1 + r_me, KW * 32);  // the previous round's reads of red are done
            // one float4 per lane and matrix, the lanes of a warp side by side (no bank conflicts)
            float4* red4 = reinterpret_cast<float4*>(red);
            red4[cw * 32 + lane] = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
            if constexpr (DUAL)
                red4[NWT * 32 + cw * 32 + lane] = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
            named_bar_sync(1 + r_me, KW * 32);
            if (kp == 0) {
                const float4* red4 = reinterpret_cast<const float4*>(red);
                for (int q = 1; q < KW; ++q) {
                    const float4 o0 = red4[(cw + q) * 32 + lane];
                    acc0[0] += o0.x;
                    acc0[1] += o0.y;
                    acc0[2] += o0.z;
                    acc0[3] += o0.w;
                    if constexpr (DUAL) {
                        const float4 o1 = red4[NWT * 32 + (cw + q) * 32 + lane];
                        acc1[0] += o1.x;
                        acc1[1] += o1.y;
                        acc1[2] += o1.z;
                        acc1[3] += o1.w;
                    }
                }
            }
        }

        if constexpr (BITS == kNvfp4) {  // the matrices' global scales (an MoE problem's: its expert's)
            float sc0 = p.wscale0, sc1 = p.wscale1;
            if constexpr (MOE) {
                const int e = slot_ec[first.x].x;
                sc0 = __ldg(p.wscales0 + e);
                if constexpr (DUAL)
                    sc1 = __ldg(p.wscales1 + e);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc0[i] *= sc0;
                if constexpr (DUAL)
                    acc1[i] *= sc1;
            }
        }

        // ---- whole row block of an unsplit problem: store; else an fp32 partial
        if (alive && kp == 0 && r_me < n) {
            const int Mr = MOE ? slot_ec[first.x].y : p.M;
            if (p.S == 1 && len == p.groups) {
                store_outputs<DUAL, MOE>(p, first.x, Mr, rb * kRowsPerBlock, lane, acc0, acc1);
            } else {
                int k = 0;
                if (!pt.aligned) {
                    const int64_t f = (int64_t)first.x * pt.per_p + (int64_t)first.y * pt.per_ps + (int64_t)rb * p.Gs;
                    k = min(c - pt.cta_of(f), p.kmax - 1);  // k < kmax by construction
                }
                float4* dst = reinterpret_cast<float4*>(
                    p.partials +
                    (((((int64_t)first.x * p.S + first.y) * p.n_rb + rb) * p.kmax + k) * 32 + lane) * VALS);
                __stcg(dst, make_float4(acc0[0], acc0[1], acc0[2], acc0[3]));
                if constexpr (DUAL)
                    __stcg(dst + 1, make_float4(acc1[0], acc1[1], acc1[2], acc1[3]));
            }
        }
    }

    if (p.S == 1 && pt.aligned) {  // every segment was a whole row block, stored above
        if (flags[0] && cw == 0 && lane == 0 && nstaged > 0)
            mbar_wait_bounded(xbar, (uint32_t)(xphase ^ 1), p.limit_ns);  // no copy left in flight
        return;
    }
    // abort is decided once for the whole CTA: every consumer warp reads one snapshot
    named_bar_sync(kBarConsumers, NCT);
    if (threadIdx.x == 0)
        flags[1] = flags[0];
    named_bar_sync(kBarConsumers, NCT);
    if (flags[1]) {
        // a bounded wait gave up (the status word says so); no activation copy may
        // be left in flight when the CTA leaves
        if (cw == 0 && lane == 0 && nstaged > 0)
            mbar_wait_bounded(xbar, (uint32_t)(xphase ^ 1), p.limit_ns);
        return;
    }

    // ------------------------------------------------------------ last contributor of a row block sums it
    auto is_partial = [&](const int4& e) { return !(p.S == 1 && (e.w & 0xFFFF) == p.groups); };
    bool any = false;
    for (int i = 0; i < nseg; ++i)
        any |= is_partial(segs[i]);
    if (!any)
        return;
    __threadfence();
    named_bar_sync(kBarConsumers, NCT);
    for (int i = threadIdx.x; i < nseg; i += NCT) {
        const int4 e = segs[i];
        int last = 0;
        if (is_partial(e)) {
            int expected = p.S;
            if (!pt.aligned) {
                expected = 0;
                for (int s2 = 0; s2 < p.S; ++s2)
                    expected += pt.contributors((int64_t)e.x * pt.per_p + (int64_t)s2 * pt.per_ps + (int64_t)e.z * p.Gs);
            }
            const int old = atomicAdd(&p.counters[(int64_t)e.x * p.n_rb + e.z], 1);
            last = old == expected - 1;
        }
        lastf[i] = last;
    }
    named_bar_sync(kBarConsumers, NCT);
    for (int i = cw; i < nseg; i += NWT) {
        if (!lastf[i])
            continue;
        const int4 e = segs[i];
        __threadfence();
        float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
        sum_partials<DUAL>(p, pt, e.x, e.z, lane, t0, t1);
        const int Mr = MOE ? slot_ec[e.x].y : p.M;
        store_outputs<DUAL, MOE>(p, e.x, Mr, e.z * kRowsPerBlock, lane, t0, t1);
        if (lane == 0)
            p.counters[(int64_t)e.x * p.n_rb + e.z] = 0;
    }
}

// One chunk of a warp worker: cnt tiles of one row block (and, for gate + up, the
// matching tiles of the second matrix T tiles further), groups g0.. of the staged
// buffer (xrow: the lane's activation row, lane & 7, or the zero row past M), group
// sums from xs0; a single matrix takes two tiles per iteration into separate
// accumulators (gate and up are two independent chains already).
template <int BITS, bool DUAL, bool F16>
__device__ __forceinline__ void warp_chunk(const uint8_t* sb, const uint8_t* xrow, const float* xs, int lane, int tq,
                                           int g0, int xs0, int cnt, int T, float (&acc0)[4], float (&acc1)[4])
{
    constexpr int TILE = tile_bytes_for(BITS);
    int j = 0;
    for (; !DUAL && j + 1 < cnt; j += 2) {
        uint4 xa, xbv, ya, ybv;
        x_frag8_row(xrow, lane, g0 + j, xa, xbv);
        x_frag8_row(xrow, lane, g0 + j + 1, ya, ybv);
        const float2 xsv = *reinterpret_cast<const float2*>(xs + (xs0 + j) * kMaxM + 2 * tq);
        const float2 ysv = *reinterpret_cast<const float2*>(xs + (xs0 + j + 1) * kMaxM + 2 * tq);
        tile_mac_x<BITS, F16>(sb + j * TILE, lane, xa, xbv, xsv, acc0);
        tile_mac_x<BITS, F16>(sb + (j + 1) * TILE, lane, ya, ybv, ysv, acc1);
    }
    for (; j < cnt; ++j) {
        uint4 xa, xbv;
        x_frag8_row(xrow, lane, g0 + j, xa, xbv);
        const float2 xsv = *reinterpret_cast<const float2*>(xs + (xs0 + j) * kMaxM + 2 * tq);
        tile_mac_x<BITS, F16>(sb + j * TILE, lane, xa, xbv, xsv, acc0);
        if constexpr (DUAL)
            tile_mac_x<BITS, F16>(sb + (T + j) * TILE, lane, xa, xbv, xsv, acc1);
    }
}

// ---------------------------------------------------------------- warp mode
//
// For bandwidth-bound calls. The C x nw consumer warps of the grid are "workers";
// worker v takes either whole (problem, split, row block) items [I v / W, I (v+1) / W)
// or an exact stream-K share [U v / W, U (v+1) / W) of the units (W = C nw). A worker
// walks its range row block by row block in chunks of T tiles; every chunk is one
// bulk copy (two for gate + up) into one of the worker's own SW ring slots, issued
// by lane w of the producer warp, so the workers of a CTA never wait for each other
// (a slot is only ever waited on by its owner, at most one phase ahead). A
// segment that is a whole row block of an unsplit problem is stored directly;
// boundary segments become fp32 partials: when its range is done, a worker counts
// each of its row blocks with one acquire-release add, and the worker whose add
// completes a count sums that row block's slots (no CTA barrier on the way).
template <int BITS, bool DUAL, bool MOE>
__global__ void __launch_bounds__(kThreads, 1) qproj_warp_kernel(const __grid_constant__ QProjParams p)
{
    constexpr int MATS = DUAL ? 2 : 1;
    constexpr int TILE = tile_bytes_for(BITS);
    constexpr int VALS = DUAL ? 8 : 4;
    const int NW = p.nw;                 // active consumer warps
    const int T = p.cg;                  // tiles per chunk
    const int SW = p.nst;                // ring slots per worker
    const int slot_bytes = MATS * T * TILE;

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + QSmem::kXbarOff);  // [2]
    volatile int* flags = reinterpret_cast<volatile int*>(smem + QSmem::kFlagOff);
    float* inv0 = reinterpret_cast<float*>(smem + QSmem::kInvOff);
    int* rows0 = reinterpret_cast<int*>(smem + QSmem::kRowOff);
    int2* slot_ec = reinterpret_cast<int2*>(smem + QSmem::kSlotOff);
    int* slot_rows = reinterpret_cast<int*>(smem + QSmem::kSlotOff + kMaxSlots * 8);
    float* xs0 = reinterpret_cast<float*>(smem + QSmem::kXsumOff);
    float* xs1 = reinterpret_cast<float*>(smem + p.xsum1_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.red_off);  // [NW * SW]
    uint64_t* empty = full + NW * SW;
    float* inv1 = reinterpret_cast<float*>(smem + p.round_off);
    int* rows1 = reinterpret_cast<int*>(smem + p.round_off + 32);
    int4* pending = reinterpret_cast<int4*>(smem + p.seg_off);         // [NW][pw] {problem, row block, split, k}
    uint8_t* xb0 = smem + p.xraw_off;
    uint8_t* xb1 = smem + p.xraw1_off;
    uint8_t* ring = smem + p.stage_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const bool norm = p.gamma != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NW * SW; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        flags[0] = 0;
        flags[2] = 0;  // a staged value has no exact fp16 copy
        fence_mbar_init();
    }
    __syncthreads();
    if constexpr (!MOE)
        pdl_launch_dependents();

    int P = p.P;
    if constexpr (MOE) {
        // as in the team kernel: wait for the routing table unless it was complete before
        // this launch could start, and let dependents start only once it is known complete
        if (!p.meta_ready)
            pdl_wait();
        pdl_launch_dependents();
        P = __ldcg(&p.meta->n_active);
        for (int i = threadIdx.x; i < P; i += blockDim.x) {
            slot_ec[i] = make_int2(__ldcg(&p.meta->slot[i].expert), __ldcg(&p.meta->slot[i].count));
            for (int j = 0; j < kMaxM; ++j)
                slot_rows[i * kMaxM + j] = p.gather ? __ldcg(&p.meta->slot[i].rows[j]) : j;
        }
        __syncthreads();
    }
    Part pt;
    pt.per_p = p.n_rb * p.groups;
    pt.per_ps = p.n_rb * p.Gs;
    pt.Gs = p.Gs;
    pt.aligned = p.aligned != 0;
    pt.items = (int64_t)P * p.S * p.n_rb;
    pt.U = pt.items * p.Gs;
    pt.inv_U = 1.f / (float)max(pt.U, (int64_t)1);
    // stream-K workers take at least half a row block's units each (fewer workers for
    // small problems), which bounds the contributors of a row block
    const int64_t wcap = pt.aligned ? pt.items : pt.U / max(1, p.Gs / 2);
    const int W = (int)min((int64_t)p.C * NW, max(wcap, (int64_t)1));
    pt.C = W;  // the partition is over workers
    auto wrange = [&](int v, int64_t& a, int64_t& b) {
        if (v < W) {
            a = pt.start(v);
            b = pt.start(v + 1);
        } else {
            a = b = 0;
        }
    };
    // runs (problem, split) of this CTA: at most two (the host sizes work so)
    const int64_t ca = pt.start(min(c * NW, W)), cb = pt.start(min(c * NW + NW, W));
    const int run0 = ca < cb ? (int)(ca / pt.per_ps) : 0;  // = problem * S + split
    const int run1 = ca < cb ? (int)((cb - 1) / pt.per_ps) : 0;
    const bool two = !norm && run1 != run0;
    if (run1 > run0 + 1) {  // never expected: every thread sees it and the CTA leaves untouched
        if (threadIdx.x == 0)
            atomicCAS(p.status, 0, TF_E_INTERNAL);
        return;
    }

    // walk helper: unit u -> (problem, split, row block, group in split)
    auto decomp = [&](int64_t u, int& pp, int& ss, int& rb, int& gl) {
        const int uu = (int)u;
        pp = uu / pt.per_p;
        int rem = uu - pp * pt.per_p;
        ss = rem / pt.per_ps;
        rem -= ss * pt.per_ps;
        rb = rem / p.Gs;
        gl = rem - rb * p.Gs;
    };

    // ------------------------------------------------------------ producer: lane w feeds worker w
    if (warp == kConsumerWarps) {
        if (lane < NW && !flags[0]) {
            const uint64_t pol = policy_evict_first();
            int64_t u, u1;
            wrange(c * NW + lane, u, u1);
            int k = 0;
            bool ok = true;
            if (u < u1) {
                int pp, ss, rb, gl;
                decomp(u, pp, ss, rb, gl);
                while (u < u1 && ok) {
                    const int len = (int)min((int64_t)(p.Gs - gl), u1 - u);
                    const int64_t mbase = MOE ? (int64_t)slot_ec[pp].x * p.matrix_bytes : 0;
                    const int64_t tile0 = (int64_t)rb * p.groups + ss * p.Gs + gl;
                    for (int g = 0; g < len; g += T, ++k) {
                        const int cnt = min(T, len - g);
                        const int s = lane * SW + k % SW;
                        if (!wait_or_abort(&empty[s], ((k / SW) & 1u) ^ 1u, flags, p.status, p.limit_ns)) {
                            ok = false;
                            break;
                        }
                        // a worker's second chunk is requested once its first has landed: every
                        // CTA requests its whole ring at the start, and without this the first
                        // chunks land only when that burst has drained (readout M=1: 20.8 ->
                        // 19.9 us)
                        if (k == 1 && !wait_or_abort(&full[lane * SW], 0u, flags, p.status, p.limit_ns)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], (uint32_t)(MATS * cnt * TILE));
#pragma unroll
                        for (int mat = 0; mat < MATS; ++mat)
                            bulk_g2s(ring + s * slot_bytes + mat * T * TILE,
                                     (mat ? p.w1 : p.w0) + mbase + (tile0 + g) * TILE, (uint32_t)(cnt * TILE), &full[s],
                                     pol);
                    }
                    u += len;
                    gl = 0;
                    if (++rb == p.n_rb) {
                        rb = 0;
                        if (++ss == p.S) {
                            ss = 0;
                            ++pp;
                        }
                    }
                }
            }
            // no copy may still be in flight when the CTA leaves (also after an abort)
            for (int q = max(0, k - SW); q < k; ++q)
                mbar_wait_bounded(&full[lane * SW + q % SW], (q / SW) & 1u, p.limit_ns);
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int cw = warp;
    const int gi = lane >> 2, tq = lane & 3;
    if (!MOE || p.meta_ready)  // the activations come from the previous kernel
        pdl_wait();

    // stage the activations of the CTA's runs (once)
    const int S = p.S;
    int M0 = p.M, M1 = p.M;
    if (MOE) {
        M0 = slot_ec[run0 / S].y;
        M1 = slot_ec[run1 / S].y;
    }
    if (threadIdx.x < kMaxM) {
        rows0[threadIdx.x] = MOE ? slot_rows[(run0 / S) * kMaxM + threadIdx.x] : (int)threadIdx.x;
        rows1[threadIdx.x] = MOE ? slot_rows[(run1 / S) * kMaxM + threadIdx.x] : (int)threadIdx.x;
    }
    const int xg0_0 = norm ? 0 : (run0 % S) * p.Gs, xg0_1 = (run1 % S) * p.Gs;
    const int xgc = norm ? p.groups : p.Gs;
    bool alive = ca < cb && !flags[0];
    // row M of each activation buffer (allocated when M < 8) is a zero row that the
    // fragment loads of rows M..7 read (no per-tile row clamp); the bulk copies write
    // only rows below M, and x_prepare's closing barrier orders these stores before
    // any fragment load
    if (M0 < kMaxM)
        for (int i = (cw * 32 + lane) * 16; i < p.x_rs; i += kConsumerWarps * 32 * 16)
            *reinterpret_cast<uint4*>(xb0 + M0 * p.x_rs + i) = make_uint4(0u, 0u, 0u, 0u);
    if (two && M1 < kMaxM)
        for (int i = (cw * 32 + lane) * 16; i < p.x_rs; i += kConsumerWarps * 32 * 16)
            *reinterpret_cast<uint4*>(xb1 + M1 * p.x_rs + i) = make_uint4(0u, 0u, 0u, 0u);
    if (cw == 0) {
        __syncwarp();
        if (lane == 0 && alive) {
            x_issue(p, xb0, smem + p.gamma_off, rows0, M0, MOE && !p.gather ? (int64_t)(run0 / S) * p.x_slot_stride : 0,
                    xg0_0, xgc, &xbar[0]);
            if (two)
                x_issue(p, xb1, nullptr, rows1, M1, MOE && !p.gather ? (int64_t)(run1 / S) * p.x_slot_stride : 0, xg0_1,
                        xgc, &xbar[1]);
        }
    }
    if (alive) {
        bool ok = wait_or_abort(&xbar[0], 0, flags, p.status, p.limit_ns);
        if (two)
            ok = ok && wait_or_abort(&xbar[1], 0, flags, p.status, p.limit_ns);
        alive = __all_sync(0xffffffffu, ok);
    }
    x_prepare(p, xb0, smem + p.gamma_off, M0, xg0_0, norm ? 0 : xg0_0, norm ? p.groups : p.Gs, xs0, inv0, cw, lane,
              kConsumerWarps, kBarConsumers);
    if (two)
        x_prepare(p, xb1, nullptr, M1, xg0_1, xg0_1, p.Gs, xs1, inv1, cw, lane, kConsumerWarps, kBarConsumers);
    if (!MOE && p.rht != nullptr) {  // input Hadamard transform of the staged rows
        x_rht(xb0, p.x_rs, xs0, M0, norm ? 0 : xg0_0, norm ? p.groups : p.Gs, p.rht, cw, lane, kConsumerWarps,
              kBarConsumers);
        if (two)
            x_rht(xb1, p.x_rs, xs1, M1, xg0_1, p.Gs, p.rht, cw, lane, kConsumerWarps, kBarConsumers);
    }
    // fp16 activations when every staged value converts exactly and, for 4-bit affine
    // codes, |x| < 4096 (the group sums above are of the same values): the codes then
    // unpack with fewer instructions. The decision is the CTA's, from one snapshot.
    {
        constexpr int kLimExp = BITS == 4 ? 12 : 16;
        const int t = cw * 32 + lane, nt = kConsumerWarps * 32;
        bool big = x_beyond_f16<kLimExp>(xb0, p.x_rs, M0, xgc * kGroup, t, nt);
        if (two)
            big |= x_beyond_f16<kLimExp>(xb1, p.x_rs, M1, xgc * kGroup, t, nt);
        if (big)
            flags[2] = 1;
        named_bar_sync(kBarConsumers, kConsumerWarps * 32);
    }
    const bool f16 = flags[2] == 0;
    if (f16) {
        const int t = cw * 32 + lane, nt = kConsumerWarps * 32;
        x_to_f16(xb0, p.x_rs, M0, xgc * kGroup, t, nt);
        if (two)
            x_to_f16(xb1, p.x_rs, M1, xgc * kGroup, t, nt);
        named_bar_sync(kBarConsumers, kConsumerWarps * 32);
    }

    if (cw < NW && alive) {
        int64_t u, u1;
        wrange(c * NW + cw, u, u1);
        const int v = c * NW + cw;
        int k = 0, np = 0;
        if (u < u1) {
            int pp, ss, rb, gl;
            decomp(u, pp, ss, rb, gl);
            while (u < u1 && alive) {
                const int len = (int)min((int64_t)(p.Gs - gl), u1 - u);
                const bool b1 = two && (pp * S + ss) == run1;
                const uint8_t* xrow = (b1 ? xb1 : xb0) + min(lane & 7, b1 ? M1 : M0) * p.x_rs;
                const float* xs = b1 ? xs1 : xs0;
                const int Mr = MOE ? slot_ec[pp].y : p.M;
                const int grel0 = norm ? ss * p.Gs + gl : gl;  // group of the buffer at the segment start
                float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
                for (int g = 0; g < len; g += T, ++k) {
                    const int cnt = min(T, len - g);
                    const int s = cw * SW + k % SW;
                    bool ok = wait_or_abort(&full[s], (k / SW) & 1u, flags, p.status, p.limit_ns);
                    if (!__all_sync(0xffffffffu, ok)) {
                        alive = false;
                        break;
                    }
                    const uint8_t* sb = ring + s * slot_bytes;
                    const int xs0 = norm ? ss * p.Gs + gl + g : gl + g;  // group sums of the chunk start
                    if (f16)
                        warp_chunk<BITS, DUAL, true>(sb, xrow, xs, lane, tq, grel0 + g, xs0, cnt, T, acc0, acc1);
                    else
                        warp_chunk<BITS, DUAL, false>(sb, xrow, xs, lane, tq, grel0 + g, xs0, cnt, T, acc0, acc1);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&empty[s]);
                }
                if (!alive)
                    break;
                if constexpr (!DUAL) {  // the second chain of a single matrix
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc0[i] += acc1[i];
                        acc1[i] = 0.f;
                    }
                }
                if constexpr (BITS == kNvfp4) {  // the matrices' global scales (an MoE problem's: its expert's)
                    float sc0 = p.wscale0, sc1 = p.wscale1;
                    if constexpr (MOE) {
                        const int e = slot_ec[pp].x;
                        sc0 = __ldg(p.wscales0 + e);
                        if constexpr (DUAL)
                            sc1 = __ldg(p.wscales1 + e);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc0[i] *= sc0;
                        if constexpr (DUAL)
                            acc1[i] *= sc1;
                    }
                }
                if (S == 1 && len == p.groups) {
                    store_outputs<DUAL, MOE>(p, pp, Mr, rb * kRowsPerBlock, lane, acc0, acc1);
                } else if (np < p.pw) {
                    int kk = 0;
                    if (!pt.aligned) {
                        const int64_t f = (int64_t)pp * pt.per_p + (int64_t)ss * pt.per_ps + (int64_t)rb * p.Gs;
                        kk = min(v - pt.cta_of(f), p.kmax - 1);  // k < kmax by construction
                    }
                    float4* dst = reinterpret_cast<float4*>(
                        p.partials + (((((int64_t)pp * S + ss) * p.n_rb + rb) * p.kmax + kk) * 32 + lane) * VALS);
                    __stcg(dst, make_float4(acc0[0], acc0[1], acc0[2], acc0[3]));
                    if constexpr (DUAL)
                        __stcg(dst + 1, make_float4(acc1[0], acc1[1], acc1[2], acc1[3]));
                    if (lane == 0)
                        pending[cw * p.pw + np] = make_int4(pp, rb, 0, 0);
                    ++np;
                } else {  // the host sizes the list; never expected
                    if (lane == 0) {
                        flags[0] = 1;
                        atomicCAS(p.status, 0, TF_E_INTERNAL);
                    }
                    alive = false;
                    break;
                }
                u += len;
                gl = 0;
                if (++rb == p.n_rb) {
                    rb = 0;
                    if (++ss == S) {
                        ss = 0;
                        ++pp;
                    }
                }
            }
        }
        // publish the worker's partial slots: one acquire-release count per row block
        // (after the warp barrier, so every lane's slot stores are covered); the worker
        // whose count completes a row block sums its slots in fixed order and stores it
        if (alive && np > 0) {
            __syncwarp();
            for (int j0 = 0; j0 < np; j0 += 32) {
                const int j = j0 + lane;
                bool last = false;
                int4 e = make_int4(0, 0, 0, 0);
                if (j < np) {
                    e = pending[cw * p.pw + j];
                    int expected = S;
                    if (!pt.aligned) {
                        expected = 0;
                        for (int s2 = 0; s2 < S; ++s2)
                            expected += pt.contributors((int64_t)e.x * pt.per_p + (int64_t)s2 * pt.per_ps +
                                                        (int64_t)e.y * p.Gs);
                    }
                    const unsigned old = atom_add_acq_rel_gpu(
                        reinterpret_cast<unsigned*>(&p.counters[(int64_t)e.x * p.n_rb + e.y]), 1u);
                    last = old == (unsigned)(expected - 1);
                }
                unsigned mask = __ballot_sync(0xffffffffu, last);
                while (mask) {
                    const int src = __ffs(mask) - 1;
                    mask &= mask - 1;
                    const int px = __shfl_sync(0xffffffffu, e.x, src), ry = __shfl_sync(0xffffffffu, e.y, src);
                    __syncwarp();
                    float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
                    sum_partials<DUAL>(p, pt, px, ry, lane, t0, t1);
                    const int Mr = MOE ? slot_ec[px].y : p.M;
                    store_outputs<DUAL, MOE>(p, px, Mr, ry * kRowsPerBlock, lane, t0, t1);
                    if (lane == 0)
                        p.counters[(int64_t)px * p.n_rb + ry] = 0;
                }
            }
        }
    }

    // abort is decided once for the whole CTA
    named_bar_sync(kBarConsumers, kConsumerWarps * 32);
    if (threadIdx.x == 0)
        flags[1] = flags[0];
    named_bar_sync(kBarConsumers, kConsumerWarps * 32);
    if (flags[1]) {
        if (cw == 0 && lane == 0 && ca < cb) {  // no activation copy may be left in flight
            mbar_wait_bounded(&xbar[0], 0, p.limit_ns);
            if (two)
                mbar_wait_bounded(&xbar[1], 0, p.limit_ns);
        }
        return;
    }
}

#include "tfq_stage.cuh"

template <int BITS, bool DUAL, bool MOE>
cudaError_t launch_qproj_warp(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    auto kern = qproj_warp_kernel<BITS, DUAL, MOE>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.C, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BITS, bool DUAL, bool MOE, int KW, int NWT>
cudaError_t launch_qproj_kw(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    auto kern = qproj_kernel<BITS, DUAL, MOE, KW, NWT>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.C, 1, 1);
    cfg.blockDim = dim3((NWT + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BITS, bool DUAL, bool MOE>
cudaError_t launch_qproj_t(const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl)
{
    if constexpr (!MOE) {
        if (plan.mode == 3)
            return launch_qstage<BITS, DUAL>(plan, p, stream, pdl);
    }
    if (plan.mode == 1)
        return launch_qproj_warp<BITS, DUAL, MOE>(plan, p, stream, pdl);
    if (plan.nw == 8) {  // light teams: one item per CTA, several CTAs per SM
        switch (plan.KW) {
        case 1: return launch_qproj_kw<BITS, DUAL, MOE, 1, 8>(plan, p, stream, pdl);
        case 2: return launch_qproj_kw<BITS, DUAL, MOE, 2, 8>(plan, p, stream, pdl);
        case 4: return launch_qproj_kw<BITS, DUAL, MOE, 4, 8>(plan, p, stream, pdl);
        case 8: return launch_qproj_kw<BITS, DUAL, MOE, 8, 8>(plan, p, stream, pdl);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (plan.KW) {
    case 1: return launch_qproj_kw<BITS, DUAL, MOE, 1, 16>(plan, p, stream, pdl);
    case 2: return launch_qproj_kw<BITS, DUAL, MOE, 2, 16>(plan, p, stream, pdl);
    case 4: return launch_qproj_kw<BITS, DUAL, MOE, 4, 16>(plan, p, stream, pdl);
    case 8: return launch_qproj_kw<BITS, DUAL, MOE, 8, 16>(plan, p, stream, pdl);
    case 16: return launch_qproj_kw<BITS, DUAL, MOE, 16, 16>(plan, p, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tfq
