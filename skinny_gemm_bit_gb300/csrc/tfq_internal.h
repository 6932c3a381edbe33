// Internal definitions shared by the CUDA translation units of libtfq.so.
#pragma once

#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>

#include "tfq.h"

namespace tfq {

constexpr int kGroup = 64;
constexpr int kRowsPerBlock = 16;             // rows of one tile (MMA M dimension)
constexpr int kMaxM = 8;                      // activation rows (MMA N dimension)
constexpr int kConsumerWarps = 16;            // compute warps per CTA (plus one producer warp)
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kMaxSlots = 64;                 // MoE: distinct experts per call (M * top_k <= 64)
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// The kernels' BITS template argument: 4 or 8 for MLX affine codes of that width,
// kNvfp4 for NVFP4 (E2M1 codes, an E4M3 scale per 16 columns; 576-byte tiles).
constexpr int kNvfp4 = -4;

__host__ __device__ constexpr int tile_bytes_for(int bits) { return bits == 8 ? 1088 : 576; }
__host__ __device__ constexpr int tile_q_bytes_for(int bits) { return bits == 8 ? 1024 : 512; }

// Device header written at the start of every packed buffer.
struct PackHeader {
    uint32_t magic, version;
    int32_t bits, group;
    int32_t code;
    float global_scale;
    int64_t batch, N, K, n_pad, tile_bytes, matrix_bytes;
    uint8_t reserved[TF_PACK_HEADER_BYTES - 9 * 8];
};
static_assert(sizeof(PackHeader) == TF_PACK_HEADER_BYTES, "header size");

// MoE routing table, written by the router kernel into the workspace.
struct MoeSlot {
    int32_t expert;
    int32_t count;           // rows routed to this expert (1..8)
    int32_t rows[kMaxM];     // activation row of each column
    int32_t js[kMaxM];       // top-k slot of each column
};
struct MoeMeta {
    int32_t n_active;
    int32_t pad[15];
    MoeSlot slot[kMaxSlots];
    int32_t inv[kMaxM * 8];  // (m, j) -> slot * 8 + column
    float w[kMaxM * 8];      // routing weight of (m, j)
};

// Everything the projection kernel needs; passed by value as a grid constant.
struct QProjParams {
    const uint8_t* w0;       // first tile of matrix 0 (gate, or the only matrix)
    const uint8_t* w1;       // first tile of matrix 1 (up), dual mode
    int64_t matrix_bytes;    // expert stride (MoE)
    int n_rb;                // 16-row blocks per matrix
    int groups;              // K / 64
    int S;                   // K splits (S divides groups)
    int Gs;                  // groups per split
    int N;                   // valid output rows
    int K;
    const uint16_t* x;
    int64_t ldx;
    int M;                   // activation rows (non-MoE)
    int64_t x_slot_stride;   // MoE, gather == 0: x offset of a problem (elements)
    int gather;              // MoE: x row of column j is meta->slot[p].rows[j]
    const uint16_t* gamma;   // RMSNorm weight or nullptr
    float eps;
    const uint16_t* residual;
    int64_t ldr;
    void* y;
    int64_t ldy;
    int y_f32;
    int64_t y_slot_stride;   // MoE: y offset of a problem (elements)
    const MoeMeta* meta;     // MoE routing table or nullptr
    int meta_ready;          // MoE: the table was complete before this launch could start (it is
                             // read before the wait for the previous kernel, which wrote x)
    int P;                   // problems (1 unless MoE, whose count comes from meta)
    int C;                   // CTAs in the persistent grid
    int aligned;             // 1: CTAs take whole row blocks; 0: stream-K shares of the units
    int kmax;                // partial slots per (problem, split, row block)
    int cg;                  // groups per pipeline stage
    int nst;                 // pipeline stages
    int segmax;              // capacity of a CTA's segment list
    float* partials;
    int* counters;
    int* status;             // device status word
    uint64_t limit_ns;       // bound of every wait
    int red_off, seg_off, round_off, last_off, xraw_off, x_rs, stage_off;  // shared-memory layout (bytes)
    // warp mode: active consumer warps, pending capacity per warp, second activation buffer
    int nw, pw, xsum1_off, xraw1_off;
    int gamma_off;  // staged RMSNorm weight (K bf16)
    int x_direct;   // activations loaded straight into registers (unsplit calls), not by bulk copy
    const uint8_t* rht;  // input Hadamard transform signs (K bits, LSB first, set = -1) or nullptr
    float wscale0, wscale1;  // NVFP4: global scale of matrix 0 / 1 (unused by affine codes)
    // NVFP4 MoE: the fp32 scale of every expert of matrix 0 / 1, indexed by expert
    const float* wscales0;
    const float* wscales1;
};

struct Plan {
    int mode;  // 0: teams in lock-step (latency-bound calls), 1: warp workers, 2: streaming (one large matrix),
               // 3: one CTA per whole row block (the stage kernel)
    int KW, R, S, Gs, cg, nst, C, aligned, kmax, segmax, slots;
    int red_off, seg_off, round_off, last_off, xraw_off, x_rs, stage_off;
    int nw, pw, xsum1_off, xraw1_off, gamma_off;
    int x_direct;
    size_t smem;
    size_t ws_partials;      // bytes
    size_t ws_counters;      // bytes
};

// ---------------------------------------------------------------- decoder-step megakernel

constexpr int kChainMaxLayers = 48;   // layer table carried in the kernel parameters
constexpr int kChainMaxGroups = 48;   // K up to 3072 per stage
constexpr int kChainSlotTiles = 32;   // tiles per ring slot

struct ChainLayerW {
    const uint8_t *qkv, *o, *gate, *up, *down;  // packed tiles (past the header)
    const uint16_t *attn_norm, *mlp_norm;
};

struct ChainParams {
    int L, M, D, F, Q, KV;
    float eps;
    int C;                                         // CTAs (all co-resident)
    int nst, x_rs, xsum_off, red_off, gamma_off, xraw_off, ring_off;  // shared-memory layout
    uint64_t limit_ns;
    const uint16_t* x;                             // residual stream entering layer 0, [M][D]
    // activation buffers by role (0 qkv, 1 h1, 2 a, 3 h): layer l uses
    // buf[r] + l * lstride[r] + (l & 1) * astride[r] (elements)
    uint16_t* buf[4];
    int64_t lstride[4], astride[4];
    unsigned* bar;                                 // [4 L + 1] stage arrival counters (zero, left zero)
    unsigned long long* ssq;                       // [2 L][8] per-row sums of squares, fixed point (zero, left zero)
    int* status;
    ChainLayerW layer[kChainMaxLayers];
};

// tfq_chain.cu
cudaError_t launch_chain(int bits, const ChainParams& p, size_t smem, cudaStream_t stream);
bool chain_fits(int bits, size_t smem);  // cooperative launch possible, one CTA per SM fits
// kmax: the largest K of a stage (staged rows); dmax: d_model (the staged RMSNorm weight)
size_t chain_smem(int bits, int kmax, int dmax, int* nst, int* x_rs, int* xsum_off, int* red_off, int* gamma_off,
                  int* xraw_off, int* ring_off);

// host helpers (tfq_api.cu)
void set_error(const char* fmt, ...);
int device_sms();
// k_full: K when the activation rows are staged whole (RMSNorm prologue), else 0;
// rows: activation rows to allocate shared memory for (8 for MoE).
Plan plan_qproj(int n_rb, int groups, int mats, int bits, int slots, int k_full, int rows);

// Error reporting and descriptor validation shared by the entry points (tfq_api.cu).
int report_error(int status, const char* fmt, ...);
int validate_desc(const tf_qweight* w, const char* name);
// The current device's fixed scratch array of tf_qlinear_run_noalloc (tfq_noalloc.cu).
int noalloc_scratch(void** out, size_t* bytes);
// tf_qlinear_run with the caller's entry-point name in its error messages
int qlinear_run_named(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint16_t* rms_gamma,
                      float rms_eps, const uint16_t* residual, void* y, int y_dtype, void* ws, size_t ws_bytes,
                      unsigned flags, void* stream, const char* name);

// launchers (tfq_qproj_b*_*.cu, one instantiation unit per bit width and matrix count)
cudaError_t launch_qproj_b4_single(bool moe, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_qproj_b4_dual(bool moe, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_qproj_b8_single(bool moe, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_qproj_b8_dual(bool moe, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl);

uint64_t tune_fingerprint();  // the calling thread's tuning overrides, hashed
cudaError_t launch_qproj_nvfp4(bool dual, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_qproj_nvfp4_moe(bool dual, const Plan& plan, const QProjParams& p, cudaStream_t stream, bool pdl);

inline cudaError_t launch_qproj(int bits, bool dual, bool moe, const Plan& plan, const QProjParams& p,
                                cudaStream_t stream, bool pdl)
{
    if (bits == kNvfp4)
        return moe ? launch_qproj_nvfp4_moe(dual, plan, p, stream, pdl) : launch_qproj_nvfp4(dual, plan, p, stream, pdl);
    if (bits == 4)
        return dual ? launch_qproj_b4_dual(moe, plan, p, stream, pdl) : launch_qproj_b4_single(moe, plan, p, stream, pdl);
    return dual ? launch_qproj_b8_dual(moe, plan, p, stream, pdl) : launch_qproj_b8_single(moe, plan, p, stream, pdl);
}

// pack kernels (tfq_pack.cu)
cudaError_t launch_pack(const uint32_t* wq, const uint16_t* s, const uint16_t* b, int64_t batch, int64_t N,
                        int64_t K, int bits, uint8_t* packed, cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t* packed, int64_t batch, int64_t N, int64_t K, int bits, uint32_t* wq,
                          uint16_t* s, uint16_t* b, cudaStream_t stream);
// batch matrices [batch][N][K/2] codes, [batch][N][K/16] scales; their fp32 scales from the
// device array gscales [batch], or hdr.global_scale when gscales is null (batch 1)
cudaError_t launch_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, const float* gscales, int64_t batch,
                              int64_t N, int64_t K, uint8_t* packed, const PackHeader& hdr, cudaStream_t stream);
cudaError_t launch_unpack_nvfp4(const uint8_t* packed, int64_t N, int64_t K, uint8_t* codes, uint8_t* scales,
                                cudaStream_t stream);

// MoE helpers (tfq_moe.cu)
cudaError_t launch_moe_route(const float* logits, int M, int E, int top_k, int32_t* idx, float* w, MoeMeta* meta,
                             cudaStream_t stream, bool pdl);
cudaError_t launch_moe_combine(const MoeMeta* meta, const float* o, int M, int top_k, int H, uint16_t* y,
                               cudaStream_t stream);
cudaError_t launch_timeout_probe(int* status, uint64_t limit_ns, cudaStream_t stream);
// bits: the kernels' BITS value (kNvfp4 for NVFP4, whose matrix scale is gscale)
cudaError_t launch_embed_rows(const uint8_t* packed, int64_t N, int64_t K, int bits, float gscale, const int32_t* ids,
                              int64_t M, uint16_t* x, int64_t ldx, int* status, cudaStream_t stream);
// The kernels' BITS value of a descriptor's weight code.
inline int desc_kernel_bits(const tf_qweight* w) { return w->code == TF_CODE_NVFP4 ? kNvfp4 : w->bits; }
// Bytes of the per-matrix fp32 scale table after the matrices of an NVFP4 pack.
inline size_t nvfp4_scale_table_bytes(int64_t batch) { return ((size_t)batch * 4 + 15) / 16 * 16; }

}  // namespace tfq
