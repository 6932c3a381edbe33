/*
 * tfq.h -- C ABI of libtfq.so: 4/8-bit group-quantised decode projections on
 * NVIDIA GB300 (sm_103a).
 *
 * What is computed (all entry points):
 *
 *   y[m][n] = sum_k x[m][k] * w[n][k],   w[n][k] = scale[n][k/64] * q[n][k] + bias[n][k/64]
 *
 * over MLX affine group-quantised weights (code TF_CODE_AFFINE): q in [0, 2^bits), one bf16 scale and
 * one bf16 bias per 64 consecutive K elements, q packed 32/bits values per
 * uint32 along K (uzu page, "Internals 1: models are assembled from
 * configuration", weight_matrix row: MLX 4/8-bit originals consumed as-is;
 * TensorFold page, box smoke-test table, "info" row: "4-bit group 64"). M is 1
 * (decode) to 8 (an 8-row speculative verify block; Husky page, "Limits of
 * plain writing and how editing is accelerated": 8-token blocks are verified at
 * about 1.5x the cost of one token).
 *
 * A second weight code, TF_CODE_NVFP4 (tf_qlinear_pack_nvfp4), holds
 *   w[n][k] = global_scale * e4m3(block_scale[n][k/16]) * e2m1(q[n][k])
 * with 4-bit E2M1 codes, one E4M3 scale per 16 consecutive K elements and one
 * fp32 scale per matrix (TensorFold page, "qualified" model table: NVFP4
 * checkpoints; the pages give no layout, the format read here is NVIDIA's
 * published NVFP4, weights only: activations stay bf16). tf_qlinear_run,
 * tf_qlinear_run_rht, tf_qlinear_run_noalloc, tf_qmlp_gateup_run,
 * tf_qmoe_run (experts packed by tf_qlinear_pack_nvfp4_experts, one fp32 scale per
 * expert), tf_decode_step_run (every matrix of the decoder in the one code; not the
 * single-kernel step of TF_TUNE_CHAIN = 2), tf_embed_rows and tf_generate_greedy
 * accept it.
 *
 * Conventions shared by every call:
 *   - Pointers named x, y, h, logits, residual, gamma, ws, packed and the
 *     wq/scales/biases inputs of the packer are DEVICE pointers owned by the
 *     caller. tf_qweight / tf_decoder_desc structs are HOST memory, read during
 *     the call only.
 *   - bf16 values are passed as uint16_t bit patterns. Activation matrices are
 *     row-major with the stated leading dimension (elements).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on it: they enqueue kernels and return. They never
 *     allocate, synchronise or print, so a sequence of calls can be captured
 *     into a CUDA graph. Exceptions (they synchronise): tf_qweight_check,
 *     tf_workspace_status, tf_generate_greedy (a host-driven loop).
 *   - Workspaces: each run entry point has a *_workspace_bytes query. The
 *     workspace must be zero-filled once before its first use (every call
 *     leaves it in the state it found it); one workspace must not be used by
 *     two calls that may run concurrently.
 *   - Return value: TF_OK or a TF_E_* status. Host-side validation happens
 *     before anything is enqueued; on error nothing is enqueued.
 *     tf_last_error() gives a message for the calling thread's last error.
 *     Device-side failures (a bounded wait that ran out) are recorded in the
 *     workspace and read with tf_workspace_status.
 */
#ifndef TFQ_H
#define TFQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TF_OK 0
#define TF_E_INVALID_ARG 1        /* null pointer, bad size, bad dtype, misaligned pointer */
#define TF_E_UNSUPPORTED_SHAPE 2  /* shape outside what the kernels implement (e.g. M > 8) */
#define TF_E_WORKSPACE_TOO_SMALL 3
#define TF_E_BAD_PACK 4           /* descriptor / packed header mismatch, stale pack */
#define TF_E_CUDA 5               /* a CUDA runtime call failed; see tf_last_error */
#define TF_E_TIMEOUT 6            /* a bounded device-side wait gave up */
#define TF_E_INTERNAL 7           /* a launch-plan invariant failed on the device (a library bug;
                                     recorded in the status word like TF_E_TIMEOUT) */

#define TF_DTYPE_BF16 0
#define TF_DTYPE_F32 1

/* run flags */
#define TF_RUN_PDL 1u  /* the caller asserts that the kernel enqueued just before
                          this call on `stream` does not write this call's
                          weights or RMSNorm gamma: the first kernel may then be
                          launched with programmatic dependent launch and read
                          them while that kernel finishes. */

#define TF_QWEIGHT_MAGIC 0x31515446u /* "TFQ1" */
#define TF_PACK_VERSION 2u

/* weight codes */
#define TF_CODE_AFFINE 0 /* MLX affine: w = scale * q + bias, bits 4 or 8, group 64 */
#define TF_CODE_NVFP4 1  /* NVFP4: w = global * e4m3 scale * e2m1 q, bits 4, group 16 */
#define TF_PACK_HEADER_BYTES 256

/* Host-side descriptor of a packed weight buffer, filled by tf_qlinear_pack. */
typedef struct tf_qweight {
    uint32_t magic;        /* TF_QWEIGHT_MAGIC once filled by tf_qlinear_pack */
    uint32_t version;      /* TF_PACK_VERSION */
    int32_t bits;          /* 4 or 8 (NVFP4: 4) */
    int32_t group;         /* 64 (NVFP4: 16, the K elements sharing one block scale) */
    int32_t code;          /* TF_CODE_AFFINE or TF_CODE_NVFP4 */
    float global_scale;    /* NVFP4: the matrix's fp32 scale; 1 for TF_CODE_AFFINE */
    int64_t batch;         /* number of matrices (experts); 1 for a plain projection */
    int64_t N;             /* output rows per matrix */
    int64_t K;             /* input columns per matrix */
    int64_t n_pad;         /* N rounded up to a multiple of 16 */
    int64_t tile_bytes;    /* bytes of one 16-row x 64-column tile (576 for 4-bit and NVFP4, 1088 for 8-bit) */
    int64_t matrix_bytes;  /* bytes of one packed matrix (tiles only) */
    const void* data;      /* device pointer: start of the packed buffer (header first) */
} tf_qweight;

/* ---------------------------------------------------------------- status */

/* Name of a status code ("TF_OK", "TF_E_INVALID_ARG", ...). Never NULL. */
const char* tf_status_str(int status);
/* Message describing the calling thread's most recent error ("" if none). */
const char* tf_last_error(void);
/* Library version (major*10000 + minor*100 + patch). */
int tf_version(void);

/* ---------------------------------------------------------------- packing */

/*
 * Bytes of the packed buffer for `batch` matrices of N x K at `bits` with
 * `group` (bits 4 with group 16: the NVFP4 code, whose buffer ends with a table of
 * one fp32 scale per matrix). Returns 0 for an unsupported combination (not 4/64,
 * 8/64 or 4/16, K not a multiple of 64, N < 1, batch < 1).
 */
size_t tf_qlinear_packed_bytes(int64_t batch, int64_t N, int64_t K, int bits, int group);

/*
 * Repack MLX-layout weights into the kernels' tile order (Husky page, "Four
 * implementation elements of MSI": 4-bit weights are stored in the order the
 * kernel reads them, so that nothing is converted at load time).
 *   wq      uint32 [batch][N][K*bits/32]; element j of a word in bits [bits*j, bits*j+bits)
 *   scales  bf16   [batch][N][K/group]
 *   biases  bf16   [batch][N][K/group]
 *   packed  output, `packed_bytes` >= tf_qlinear_packed_bytes(...), 16-byte aligned
 *   desc    output host descriptor; desc->data = packed
 * Requirements: bits in {4, 8}, group == 64, K % 64 == 0, N >= 1, batch >= 1.
 * The kernel reads the inputs and writes `packed` on `stream`; the inputs may be
 * freed once the stream has passed this point.
 */
int tf_qlinear_pack(const uint32_t* wq, const uint16_t* scales, const uint16_t* biases,
                    int64_t batch, int64_t N, int64_t K, int bits, int group,
                    void* packed, size_t packed_bytes, tf_qweight* desc, void* stream);

/*
 * Repack NVFP4 weights into the kernels' tile order (a 16 x 64 tile is 512 bytes
 * of codes and 64 bytes of block scales, the size of an MLX 4-bit tile).
 *   codes         uint8 [N][K/2]: two E2M1 codes a byte along K, the even column in
 *                 bits 0-3 (bit 3 sign, bits 2-1 exponent with bias 1, bit 0 mantissa)
 *   block_scales  uint8 [N][K/16]: E4M3 (bit 7 sign, bits 6-3 exponent with bias 7,
 *                 bits 2-0 mantissa, S.1111.111 NaN) for columns 16 j .. 16 j + 15
 *   global_scale  fp32 scale of the whole matrix (finite)
 *   packed        output, `packed_bytes` >= tf_qlinear_packed_bytes(1, N, K, 4, 16),
 *                 16-byte aligned
 *   desc          output host descriptor (code TF_CODE_NVFP4, bits 4, group 16, batch 1)
 * Requirements: K % 64 == 0, N >= 1. Asynchronous on `stream` as tf_qlinear_pack.
 */
int tf_qlinear_pack_nvfp4(const uint8_t* codes, const uint8_t* block_scales, float global_scale,
                          int64_t N, int64_t K, void* packed, size_t packed_bytes, tf_qweight* desc,
                          void* stream);

/*
 * tf_qlinear_pack_nvfp4 for a stack of E expert matrices of one MoE layer (the
 * TensorFold page's NVFP4 checkpoints hold one scale per matrix):
 *   codes          uint8 [E][N][K/2], block_scales uint8 [E][N][K/16] (as above)
 *   global_scales  device fp32 [E]: the scale of each expert's matrix (read during the call)
 *   packed         output, `packed_bytes` >= tf_qlinear_packed_bytes(E, N, K, 4, 16)
 *   desc           output (batch E); desc->global_scale is 1 and unused: each matrix's
 *                  scale is the packed buffer's table entry
 * For tf_qmoe_run (gate, up: [E][I][H]; down: [E][H][I]). Asynchronous on `stream`.
 */
int tf_qlinear_pack_nvfp4_experts(const uint8_t* codes, const uint8_t* block_scales, const float* global_scales,
                                  int64_t E, int64_t N, int64_t K, void* packed, size_t packed_bytes,
                                  tf_qweight* desc, void* stream);

/*
 * Inverse of tf_qlinear_pack: write the MLX-layout arrays back out of a packed
 * buffer (same shapes as the packer's inputs). Used to prove the packing is a
 * lossless permutation. For NVFP4 weights: the codes go to `wq` (the bytes of
 * uint8 [batch][N][K/2]), the block scales to `scales` (the bytes of uint8
 * [batch][N][K/16]), and `biases`, when not NULL, receives the per-matrix fp32
 * scales (the bytes of fp32 [batch]).
 */
int tf_qlinear_unpack_debug(const tf_qweight* w, uint32_t* wq, uint16_t* scales, uint16_t* biases,
                            void* stream);

/*
 * Read the header at w->data back to the host and compare it with the
 * descriptor (magic, version, shape). Synchronises `stream`. TF_E_BAD_PACK on
 * mismatch.
 */
int tf_qweight_check(const tf_qweight* w, void* stream);

/* ---------------------------------------------------------------- projections */

/*
 * y[m][n] = residual[m][n] + sum_k xn[m][k] * w[n][k] for m < M, n < N, where
 * xn = x, or, when rms_gamma != NULL, the RMSNorm prologue
 * xn[m][k] = x[m][k] / sqrt(mean_k(x[m][k]^2) + rms_eps) * gamma[k], rounded to
 * bf16 (Husky page, "Four implementation elements of MSI": the preceding
 * normalisation is merged into each projection kernel).
 *   w          packed weights (batch must be 1)
 *   x          bf16 [M][ldx], ldx >= K, ldx a multiple of 8, 16-byte aligned
 *   M          1..8
 *   rms_gamma  bf16 [K] or NULL, 16-byte aligned (whole rows are staged on chip: K up to ~6000)
 *   residual   bf16 [M][ldr] or NULL (ldr = N when given: residual is [M][N])
 *   y          [M][N] of y_dtype (TF_DTYPE_BF16: round to nearest even; TF_DTYPE_F32)
 *   ws         workspace of tf_qlinear_workspace_bytes(w, M) bytes
 */
size_t tf_qlinear_workspace_bytes(const tf_qweight* w, int64_t M);
int tf_qlinear_run(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M,
                   const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual,
                   void* y, int y_dtype, void* ws, size_t ws_bytes, unsigned flags, void* stream);

/*
 * tf_qlinear_run with an input randomized Hadamard transform folded into the
 * activation staging (uzu page, "Internals 1: models are assembled from
 * configuration", linear row of the table: an input-side RHT block that spreads
 * quantisation error). The pages give no block size or layout; here
 *   xr[m][64 g + i] = (1/8) sum_j H[i][j] d[64 g + j] xn[m][64 g + j],
 *   H[i][j] = (-1)^popcount(i & j)   (the Sylvester-ordered 64-point
 *                                     Walsh-Hadamard matrix, one per group)
 * and y[m][n] = residual[m][n] + sum_k xr[m][k] * w[n][k]: w holds weights
 * quantised in the rotated basis, xn is x or its RMSNorm as in tf_qlinear_run
 * (normalisation first), and xr is rounded to bf16 once.
 *   rht_signs  device uint8 [K / 8]: bit (k % 8) of byte k / 8 set means d[k] = -1
 *              (must not be NULL; read during the call only)
 *   Other arguments, the workspace query and the errors: as tf_qlinear_run.
 */
int tf_qlinear_run_rht(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M, const uint8_t* rht_signs,
                       const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual, void* y, int y_dtype,
                       void* ws, size_t ws_bytes, unsigned flags, void* stream);

/*
 * tf_qlinear_run without a workspace argument: the same projection, the same
 * kernels and the same results, with the split-K scratch (status word, arrival
 * counters, fp32 partial slots) taken from one fixed 4 MiB device array inside
 * the library (one per device) instead of caller memory. The pages have no
 * counterpart; it exists for callers that cannot allocate device memory where
 * they make the call: code running inside an allocator or memory-pool callback,
 * a path that has reserved all of its memory up front and must never reach an
 * allocator, or a host without access to a device allocator. This call itself
 * allocates nothing.
 *   Arguments: as tf_qlinear_run, minus ws / ws_bytes.
 *   Limit: shapes whose tf_qlinear_workspace_bytes exceeds 4 MiB are refused
 *          with TF_E_WORKSPACE_TOO_SMALL (nothing enqueued); every shape whose
 *          K splits need at most that much is served (e.g. K=12800, N=2560).
 *   First call on a device: looks up the array's device address
 *          (cudaGetSymbolAddress, with that device current), which may load the
 *          library's device code; make that first call before any stream
 *          capture begins.
 *   Sharing: every call on a device uses the same array. The array starts at
 *          zero and each call leaves it at zero, so it needs no clearing; but two
 *          calls that may run at the same time on one device (different streams,
 *          or host threads) race on it and must not overlap. A device-side wait
 *          that gives up records TF_E_TIMEOUT in the array and may leave its
 *          split-K counters and slots dirty, so that later calls would be wrong:
 *          tf_qlinear_noalloc_status reports such a failure and clears the array.
 *   Device reset: the array's address is cached per device for the life of the
 *          process; after cudaDeviceReset (or any teardown of the primary context)
 *          the cached address is stale, so this call must not be used afterwards.
 */
int tf_qlinear_run_noalloc(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M,
                           const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual,
                           void* y, int y_dtype, unsigned flags, void* stream);

/*
 * The status word of tf_qlinear_run_noalloc's fixed array on the current device:
 * TF_OK, or the status a device-side failure recorded there (TF_E_TIMEOUT,
 * TF_E_INTERNAL). After a failure the whole array (status word, arrival counters,
 * partial slots) is set back to zero, so the next call starts clean. Synchronises
 * `stream` (the array lives on the current device); allocates nothing. Must not
 * overlap a tf_qlinear_run_noalloc call on the same device.
 */
int tf_qlinear_noalloc_status(void* stream);

/*
 * Gate and up together with a SwiGLU epilogue (Husky page, "Four
 * implementation elements of MSI": gate and up projections are processed
 * together; the preceding normalisation is merged in):
 *   h[m][n] = silu(g[m][n]) * u[m][n],  g = xn . gate^T,  u = xn . up^T,
 *   silu(g) = g / (1 + exp(-g)); xn as in tf_qlinear_run.
 *   gate, up   packed, same N and K, batch 1
 *   h          bf16 [M][N]
 */
size_t tf_qmlp_gateup_workspace_bytes(const tf_qweight* gate, const tf_qweight* up, int64_t M);
int tf_qmlp_gateup_run(const tf_qweight* gate, const tf_qweight* up, const uint16_t* x, int64_t ldx,
                       int64_t M, const uint16_t* rms_gamma, float rms_eps, uint16_t* h,
                       void* ws, size_t ws_bytes, unsigned flags, void* stream);

/*
 * Mixture-of-experts layer with per-row expert gathering (uzu page,
 * "Internals 1" table, mlp row: MixtureOfExperts with a routing function):
 *   idx[m][0..top_k) = the top_k experts by router logit (descending; equal
 *                      logits: lower expert index first)
 *   w[m][j]          = softmax over the top_k selected logits
 *   y[m]             = sum_j w[m][j] * down_e(silu(gate_e x[m]) * up_e x[m]),  e = idx[m][j]
 * Every selected expert's weights are read once per call, however many rows
 * chose it; the weighted sum runs in slot order j (deterministic).
 *   gate, up       packed, batch = E experts of [I][H]
 *   down           packed, batch = E experts of [H][I]
 *                  (all three in one weight code: MLX affine 4/8-bit from tf_qlinear_pack,
 *                  or NVFP4 from tf_qlinear_pack_nvfp4_experts, each expert's matrix
 *                  scaled by its own fp32 scale)
 *   router_logits  fp32 [M][E]
 *   x              bf16 [M][H] (row stride H)
 *   y              bf16 [M][H]
 *   topk_idx       int32 [M][top_k] out
 *   topk_w         fp32  [M][top_k] out
 * Limits: 1 <= M <= 8, 1 <= top_k <= 8, E <= 1024.
 */
size_t tf_qmoe_workspace_bytes(const tf_qweight* gate, const tf_qweight* up, const tf_qweight* down,
                               int64_t M, int top_k);
int tf_qmoe_run(const tf_qweight* gate, const tf_qweight* up, const tf_qweight* down,
                const float* router_logits, int64_t M, int top_k, const uint16_t* x, uint16_t* y,
                int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes, unsigned flags,
                void* stream);

/* ---------------------------------------------------------------- decoder step */

/* One decoder layer's projections; gammas are bf16 [d_model] device pointers. */
typedef struct tf_decoder_layer {
    tf_qweight qkv;             /* [q_dim + 2*kv_dim][d_model] : q | k | v */
    tf_qweight o;               /* [d_model][q_dim] */
    tf_qweight gate;            /* [d_ff][d_model] */
    tf_qweight up;              /* [d_ff][d_model] */
    tf_qweight down;            /* [d_model][d_ff] */
    const uint16_t* attn_norm;  /* RMSNorm gamma ahead of qkv */
    const uint16_t* mlp_norm;   /* RMSNorm gamma ahead of gate/up */
} tf_decoder_layer;

typedef struct tf_decoder_desc {
    int32_t n_layers;
    int64_t d_model, d_ff, q_dim, kv_dim, vocab;
    float eps;                        /* RMSNorm epsilon */
    const tf_decoder_layer* layers;   /* HOST array [n_layers] */
    const uint16_t* final_norm;       /* bf16 [d_model] */
    tf_qweight readout;               /* [vocab][d_model] (tied embedding) */
} tf_decoder_desc;

/*
 * The per-token weight stream of a dense decoder, attention excluded (Husky
 * page, "Four implementation elements of MSI": a layer is four consecutive
 * kernels; "Experiments with a full-step megakernel": what pays is overlapping
 * the next stage's weight loads with the current stage). Per layer, in order:
 *   qkv = rmsnorm(h, attn_norm) . Wqkv^T            [M][q_dim + 2 kv_dim]
 *   h1  = h + qkv[:, :q_dim] . Wo^T                  (q stands in for the attention output)
 *   a   = silu(rmsnorm(h1, mlp_norm) . Wg^T) * (rmsnorm(h1, mlp_norm) . Wu^T)
 *   h   = h1 + a . Wd^T
 * then logits = rmsnorm(h, final_norm) . Wreadout^T. Each projection is one kernel,
 * chained on `stream` with programmatic dependent launch (every kernel streams its
 * weights while the previous one finishes); tf_tune_set(TF_TUNE_CHAIN, 2) runs the
 * whole step as one persistent cooperative kernel instead.
 *   x        bf16 [M][d_model], the residual stream entering layer 0
 *   logits   bf16 [M][vocab]
 *   debug    NULL, or bf16 scratch of tf_decode_step_debug_elems(d, M) elements
 *            that receives every intermediate: per layer [qkv | h1 | a | h]
 *            blocks of M x (q_dim+2kv_dim), M x d_model, M x d_ff, M x d_model.
 */
size_t tf_decode_step_workspace_bytes(const tf_decoder_desc* d, int64_t M);
size_t tf_decode_step_debug_elems(const tf_decoder_desc* d, int64_t M);
int tf_decode_step_run(const tf_decoder_desc* d, const uint16_t* x, int64_t M, uint16_t* logits,
                       void* ws, size_t ws_bytes, uint16_t* debug, unsigned flags, void* stream);

/* ---------------------------------------------------------------- verify block */

/*
 * Greedy decoding with an M = 8 verify block (Husky page, the passage before "Flash
 * draft model and candidate selection": when the last tokens just generated also
 * occur in the prompt, the 7 tokens that followed them there are proposed; one
 * step verifies the block, the matching drafts are kept, and the text is the one
 * plain decoding gives). The pages fix no n-gram length or choice among several
 * occurrences; here the longest suffix of at most max_ngram tokens is tried first,
 * and its first occurrence in the prompt with a token after it is used.
 */

/*
 * idx[m] = the lowest index n of the largest value of row m of the bf16 array
 * v[M][ld] over n < N (-0 equals +0; NaN is never chosen unless the row holds
 * nothing else). v device, idx device int32 [M]; 1 <= M <= 65535, N < 2^31.
 */
int tf_argmax_rows(const uint16_t* v, int64_t ld, int64_t M, int64_t N, int32_t* idx, void* stream);

/*
 * x[m][k] = bf16(s q + b) of row ids[m] of a packed matrix (batch 1), k < K:
 * the dequantised row, rounded to nearest even (exact whenever |b| / |s| < 2^15).
 * NVFP4: bf16(global_scale * (e4m3 scale * e2m1 code)), the fp32 product of the
 * exact code-scale product and the matrix scale, rounded to nearest even.
 * ids device int32 [M], x device bf16 [M][K]. ws: 256 zeroed, 256-aligned bytes; an
 * id outside [0, N) records TF_E_INVALID_ARG there (tf_workspace_status) and gives
 * a zero row. Used as the token embedding of a tied readout.
 */
int tf_embed_rows(const tf_qweight* w, const int32_t* ids, int64_t M, uint16_t* x, void* ws, size_t ws_bytes,
                  void* stream);

/*
 * The draft of one step (host only, no GPU): for ng = min(max_ngram, tail_len)
 * down to 1, the first occurrence prompt[p, p + ng) of the tail's last ng tokens
 * with p + ng < prompt_len; the draft is prompt[p + ng, p + ng + cnt), cnt =
 * min(max_draft, prompt_len - p - ng). Returns cnt (0: no occurrence), -1 on bad
 * arguments. prompt, tail, draft: host int32.
 */
int64_t tf_draft_prompt_lookup(const int32_t* prompt, int64_t prompt_len, const int32_t* tail, int64_t tail_len,
                               int max_ngram, int max_draft, int32_t* draft);

/*
 * Greedy generation with the decoder step (tf_decode_step_run) and the tied readout
 * as token embedding: each step embeds the block [last token, draft...] (1 + cnt <=
 * 8 rows, cnt = tf_draft_prompt_lookup(prompt, ..., max_draft) capped by the tokens
 * still wanted), runs one decoder step at M = 1 + cnt, takes the per-row argmax,
 * keeps the drafts that match the predictions in order and appends the prediction
 * after the last kept one. max_draft = 0 is plain one-token decoding; any max_draft
 * gives the same tokens (a row's logits do not depend on the rows beside it).
 *   prompt      host int32 [prompt_len], tokens in [0, vocab), prompt_len >= 1
 *   max_new     tokens to generate; out host int32 [max_new]
 *   max_draft   0..7; max_ngram 1..64
 *   n_out       host: tokens written (= max_new); n_steps, n_accepted (host, may be
 *               NULL): decoder steps run, drafts kept
 *   ws          tf_generate_workspace_bytes(d) bytes, 256-aligned, zeroed once
 * Synchronises `stream` once per step (the predictions decide the next block).
 * The device part of a step (embed, decoder step, argmax) is captured as a CUDA
 * graph the first time a (decoder, ws, block length) is seen on the calling thread
 * and replayed after that; the thread keeps up to 16 such graphs and one capture
 * stream per device until the CUDA context is destroyed. A step whose graph cannot
 * be captured or launched is launched directly.
 */
size_t tf_generate_workspace_bytes(const tf_decoder_desc* d);
int tf_generate_greedy(const tf_decoder_desc* d, const int32_t* prompt, int64_t prompt_len, int64_t max_new,
                       int max_draft, int max_ngram, int32_t* out, int64_t* n_out, int64_t* n_steps,
                       int64_t* n_accepted, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- diagnostics */

/*
 * Read the device status word of a workspace (offset 0): TF_OK, or the status
 * of a device-side failure (TF_E_TIMEOUT) recorded by a call that used it,
 * which is then cleared. Synchronises `stream`.
 */
int tf_workspace_status(void* ws, void* stream);

/*
 * Run one kernel whose bounded wait on a shared-memory barrier is never
 * satisfied, with a limit of `limit_ns` nanoseconds, so that the timeout path
 * can be exercised without hanging the GPU. Records TF_E_TIMEOUT in `ws` (read
 * it with tf_workspace_status). `ws` needs 256 bytes; ws = NULL targets the
 * status word of tf_qlinear_run_noalloc's fixed array on the current device
 * (read it with tf_qlinear_noalloc_status).
 */
int tf_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream);

/*
 * Tuning override for the launch planner: key is one of TF_TUNE_*; value < 0
 * restores the planner's own choice. The setting belongs to the calling host
 * thread: it changes the plans of that thread's later calls only, never another
 * thread's. A workspace sized by a *_workspace_bytes query under one setting may
 * be too small for a call made under another (the call then returns
 * TF_E_WORKSPACE_TOO_SMALL): query and run under the same setting.
 */
#define TF_TUNE_ROWBLOCKS 0   /* 16-row blocks processed side by side per round (1, 2, 4, 8, 16) */
#define TF_TUNE_SPLITK 1      /* K splits (must divide K / 64) */
#define TF_TUNE_STAGE_GROUPS 2 /* 64-column groups per pipeline stage */
#define TF_TUNE_STAGES 3      /* pipeline depth (ring slots per worker in warp mode) */
#define TF_TUNE_WARPS 4       /* warp mode: consumer warps per CTA (1..16); streaming: 8 or 16 */
#define TF_TUNE_MODE 5        /* 1: lock-step teams, 2: warp workers, 3: light teams (one item per CTA),
                                 4: light teams with bulk-copied (not register-loaded) activations,
                                 5: streaming CTAs (one matrix; RMSNorm only for K <= 1024) */
#define TF_TUNE_CHAIN 6       /* tf_decode_step_run: 2 = the whole step as one persistent kernel
                                 (TF_E_UNSUPPORTED_SHAPE where it cannot run); otherwise one kernel
                                 per projection, chained with programmatic dependent launch */
int tf_tune_set(int key, int value);

#ifdef __cplusplus
}
#endif

#endif /* TFQ_H */
