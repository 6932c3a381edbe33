// Greedy decoding with a verify block (Husky page, "Flash draft model and candidate
// selection" and the prompt-lookup passage before it: when the last tokens just
// generated also occur in the prompt, the tokens that followed them there are
// proposed, a block of up to 8 tokens is verified in one step, the matching drafts
// are kept, and the text is the one plain decoding gives).
//
//   tf_argmax_rows          per-row argmax of bf16 logits (device)
//   tf_embed_rows           rows of a packed matrix dequantised to bf16 (device; the
//                           tied readout serves as the token embedding)
//   tf_draft_prompt_lookup  the draft of one step (host only)
//   tf_generate_greedy      the loop: embed the block, one decoder step at M = block
//                           length, argmax, accept the matching drafts (host-driven,
//                           synchronises once per step). The device part of a step
//                           (embed, ~115 projection launches, argmax) is replayed from a
//                           CUDA graph kept per thread for the decoder, workspace and
//                           block length, so a step costs one launch on the host.
#include <algorithm>
#include <cstring>
#include <vector>

#include "tfq_internal.h"

namespace tfq {
namespace {

constexpr int kArgmaxThreads = 1024;
constexpr int kMaxDraft = kMaxM - 1;  // the block is the current token plus the drafts

// ---- step graphs: the embed, decoder-step and argmax launches of one block length,
// captured once and replayed. Keyed by everything the launches bake in: the decoder's
// descriptors (shapes and pointers), the workspace, the block length, the device and the
// tuning overrides. A small per-thread cache; the oldest entry is replaced (its
// executable destroyed). Entries are never freed at thread exit: the CUDA context may
// already be gone then, and its teardown releases them.
struct StepGraph {
    uint64_t key;
    cudaGraphExec_t exec;
};
constexpr int kStepGraphs = 16;
thread_local StepGraph g_step_graphs[kStepGraphs] = {};
thread_local int g_step_graph_next = 0;
thread_local cudaStream_t g_capture_stream[64] = {};

uint64_t fnv_bytes(uint64_t h, const void* p, size_t n)
{
    const unsigned char* b = static_cast<const unsigned char*>(p);
    for (size_t i = 0; i < n; ++i) {
        h ^= b[i];
        h *= 1099511628211ull;
    }
    return h;
}

uint64_t step_graph_key(const tf_decoder_desc* d, const void* ws, size_t ws_bytes, int64_t M, int dev)
{
    uint64_t h = fnv_bytes(1469598103934665603ull, d, sizeof *d);
    h = fnv_bytes(h, d->layers, sizeof(tf_decoder_layer) * (size_t)d->n_layers);
    h = fnv_bytes(h, &ws, sizeof ws);
    h = fnv_bytes(h, &ws_bytes, sizeof ws_bytes);
    h = fnv_bytes(h, &M, sizeof M);
    h = fnv_bytes(h, &dev, sizeof dev);
    const uint64_t t = tune_fingerprint();
    return fnv_bytes(h, &t, sizeof t);
}

// Order-preserving key of a bf16 value (-0 as +0, NaN below every number).
__device__ __forceinline__ uint32_t bf16_order_key(uint32_t h)
{
    if ((h & 0x7F80u) == 0x7F80u && (h & 0x7Fu) != 0u)
        return 0u;
    if ((h & 0x7FFFu) == 0u)
        h = 0u;
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}

// out[m] = the lowest index of the largest value of row m (NaN never chosen unless
// the row holds nothing else). One CTA per row.
__global__ void __launch_bounds__(kArgmaxThreads) argmax_rows_kernel(const uint16_t* __restrict__ v, int64_t ld,
                                                                     int64_t N, int32_t* __restrict__ out)
{
    __shared__ unsigned long long best[kArgmaxThreads / 32];
    const uint16_t* row = v + blockIdx.x * ld;
    // (key << 32) | (2^32 - 1 - index): the largest is the largest value, then the lowest index
    unsigned long long b = 0ull;
    for (int64_t n = threadIdx.x; n < N; n += blockDim.x) {
        const unsigned long long c =
            ((unsigned long long)bf16_order_key(__ldg(row + n)) << 32) | (0xFFFFFFFFull - (unsigned long long)n);
        b = c > b ? c : b;
    }
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long c = __shfl_xor_sync(0xffffffffu, b, o);
        b = c > b ? c : b;
    }
    if ((threadIdx.x & 31) == 0)
        best[threadIdx.x >> 5] = b;
    __syncthreads();
    if (threadIdx.x < 32) {
        b = threadIdx.x < blockDim.x / 32 ? best[threadIdx.x] : 0ull;
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long c = __shfl_xor_sync(0xffffffffu, b, o);
            b = c > b ? c : b;
        }
        if (threadIdx.x == 0)
            out[blockIdx.x] = (int32_t)(0xFFFFFFFFull - (b & 0xFFFFFFFFull));
    }
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace of the generation loop: [pred int32 x 8 | status int32] [ids int32 x 8]
// [x bf16 8 x d_model] [logits bf16 8 x vocab] [decoder step workspace].
struct GenLayout {
    size_t pred, ids, x, logits, step, step_bytes, total;
};

GenLayout gen_layout(const tf_decoder_desc* d)
{
    GenLayout L{};
    L.pred = 0;
    L.ids = 256;
    L.x = 512;
    L.logits = L.x + align_up((size_t)kMaxM * d->d_model * 2, 256);
    L.step = L.logits + align_up((size_t)kMaxM * d->vocab * 2, 256);
    L.step_bytes = tf_decode_step_workspace_bytes(d, kMaxM);
    L.total = L.step_bytes == 0 ? 0 : L.step + L.step_bytes;
    return L;
}

void forget_step_graph(cudaGraphExec_t exec)
{
    for (StepGraph& g : g_step_graphs)
        if (g.exec == exec) {
            g.exec = nullptr;
            g.key = 0;
        }
}

// The cached graph of one step for (decoder, workspace, M), captured on first use on this
// thread's capture stream; nullptr when it cannot be had (the capture or the
// instantiation failed: the caller then launches the step directly, after the error
// state those calls left has been cleared).
template <class Enqueue>
cudaGraphExec_t step_graph(const tf_decoder_desc* d, const void* ws, size_t ws_bytes, int64_t M, Enqueue&& enqueue)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    const uint64_t key = step_graph_key(d, ws, ws_bytes, M, dev);
    for (const StepGraph& g : g_step_graphs)
        if (g.exec != nullptr && g.key == key)
            return g.exec;
    if (g_capture_stream[dev] == nullptr &&
        cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess) {
        g_capture_stream[dev] = nullptr;
        cudaGetLastError();
        return nullptr;
    }
    cudaStream_t cs = g_capture_stream[dev];
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        g_capture_stream[dev] = nullptr;  // made again next time (the old one may be from a gone context)
        return nullptr;
    }
    const int rc = enqueue(cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(cs, &graph);
    cudaGraphExec_t exec = nullptr;
    if (rc == TF_OK && ce == cudaSuccess && graph != nullptr && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
        exec = nullptr;
    if (graph != nullptr)
        cudaGraphDestroy(graph);
    cudaGetLastError();
    if (exec == nullptr)
        return nullptr;
    StepGraph& slot = g_step_graphs[g_step_graph_next];
    g_step_graph_next = (g_step_graph_next + 1) % kStepGraphs;
    if (slot.exec != nullptr)
        cudaGraphExecDestroy(slot.exec);
    slot.key = key;
    slot.exec = exec;
    return exec;
}

}  // namespace
}  // namespace tfq

using namespace tfq;

extern "C" {

int tf_argmax_rows(const uint16_t* v, int64_t ld, int64_t M, int64_t N, int32_t* idx, void* stream)
{
    if (v == nullptr || idx == nullptr)
        return report_error(TF_E_INVALID_ARG, "tf_argmax_rows: NULL pointer");
    if (M < 1 || M > 65535 || N < 1 || N > INT32_MAX || ld < N)
        return report_error(TF_E_UNSUPPORTED_SHAPE, "tf_argmax_rows: need 1 <= M <= 65535, 1 <= N < 2^31, ld >= N");
    argmax_rows_kernel<<<(unsigned)M, kArgmaxThreads, 0, static_cast<cudaStream_t>(stream)>>>(v, ld, N, idx);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TF_OK : report_error(TF_E_CUDA, "tf_argmax_rows: %s", cudaGetErrorString(e));
}

int tf_embed_rows(const tf_qweight* w, const int32_t* ids, int64_t M, uint16_t* x, void* ws, size_t ws_bytes,
                  void* stream)
{
    int rc = validate_desc(w, "tf_embed_rows");
    if (rc)
        return rc;
    if (ids == nullptr || x == nullptr || ws == nullptr)
        return report_error(TF_E_INVALID_ARG, "tf_embed_rows: NULL pointer");
    if (w->batch != 1 || M < 1 || M > INT32_MAX / w->K)
        return report_error(TF_E_UNSUPPORTED_SHAPE, "tf_embed_rows: batch must be 1 and 1 <= M");
    if (ws_bytes < 256 || reinterpret_cast<uintptr_t>(ws) % 256 != 0)
        return report_error(TF_E_WORKSPACE_TOO_SMALL, "tf_embed_rows: workspace of 256 aligned bytes needed");
    const cudaError_t e = launch_embed_rows(static_cast<const uint8_t*>(w->data), w->N, w->K, desc_kernel_bits(w),
                                            w->global_scale, ids, M, x, w->K, static_cast<int*>(ws),
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TF_OK : report_error(TF_E_CUDA, "tf_embed_rows: %s", cudaGetErrorString(e));
}

int64_t tf_draft_prompt_lookup(const int32_t* prompt, int64_t prompt_len, const int32_t* tail, int64_t tail_len,
                               int max_ngram, int max_draft, int32_t* draft)
{
    if (prompt_len < 0 || tail_len < 0 || max_ngram < 1 || max_draft < 0 || (prompt_len > 0 && !prompt) ||
        (tail_len > 0 && !tail) || (max_draft > 0 && !draft))
        return -1;
    // longest suffix of the tail first; its first occurrence in the prompt that has a
    // token after it; the tokens that follow it there are the draft
    for (int64_t ng = std::min<int64_t>(max_ngram, tail_len); ng >= 1; --ng) {
        const int32_t* suffix = tail + tail_len - ng;
        for (int64_t p = 0; p + ng < prompt_len; ++p) {
            if (std::memcmp(prompt + p, suffix, (size_t)ng * sizeof(int32_t)) != 0)
                continue;
            const int64_t cnt = std::min<int64_t>(max_draft, prompt_len - (p + ng));
            std::memcpy(draft, prompt + p + ng, (size_t)cnt * sizeof(int32_t));
            return cnt;
        }
    }
    return 0;
}

size_t tf_generate_workspace_bytes(const tf_decoder_desc* d)
{
    if (d == nullptr)
        return 0;
    return gen_layout(d).total;
}

int tf_generate_greedy(const tf_decoder_desc* d, const int32_t* prompt, int64_t prompt_len, int64_t max_new,
                       int max_draft, int max_ngram, int32_t* out, int64_t* n_out, int64_t* n_steps,
                       int64_t* n_accepted, void* ws, size_t ws_bytes, void* stream)
{
    if (d == nullptr || prompt == nullptr || prompt_len < 1 || max_new < 0 || (max_new > 0 && out == nullptr) ||
        n_out == nullptr || ws == nullptr)
        return report_error(TF_E_INVALID_ARG, "tf_generate_greedy: NULL pointer or empty prompt");
    if (max_draft < 0 || max_draft > kMaxDraft || max_ngram < 1 || max_ngram > 64)
        return report_error(TF_E_UNSUPPORTED_SHAPE, "tf_generate_greedy: need 0 <= max_draft <= %d, 1 <= max_ngram <= 64",
                            kMaxDraft);
    const GenLayout L = gen_layout(d);
    if (L.total == 0)
        return TF_E_INVALID_ARG;  // the decoder step's query has set the message
    if (ws_bytes < L.total || reinterpret_cast<uintptr_t>(ws) % 256 != 0)
        return report_error(TF_E_WORKSPACE_TOO_SMALL, "tf_generate_greedy: workspace has %zu bytes, needs %zu (256-aligned)",
                            ws_bytes, L.total);
    for (int64_t i = 0; i < prompt_len; ++i)
        if (prompt[i] < 0 || prompt[i] >= d->vocab)
            return report_error(TF_E_INVALID_ARG, "tf_generate_greedy: prompt token %lld = %d outside [0, %lld)",
                                (long long)i, prompt[i], (long long)d->vocab);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    int32_t* pred = reinterpret_cast<int32_t*>(wsb + L.pred);
    int* status = reinterpret_cast<int*>(wsb + L.pred + kMaxM * 4);
    int32_t* ids = reinterpret_cast<int32_t*>(wsb + L.ids);
    uint16_t* x = reinterpret_cast<uint16_t*>(wsb + L.x);
    uint16_t* logits = reinterpret_cast<uint16_t*>(wsb + L.logits);
    const tf_qweight& E = d->readout;  // tied: the readout rows are the token embeddings

    std::vector<int32_t> seq(prompt, prompt + prompt_len);
    seq.reserve((size_t)(prompt_len + max_new));
    int64_t produced = 0, steps = 0, accepted = 0;
    int32_t block[kMaxM], draft[kMaxDraft], host[kMaxM + 1];
    auto cuda_err = [&](cudaError_t e, const char* what) {
        return report_error(TF_E_CUDA, "tf_generate_greedy: %s: %s", what, cudaGetErrorString(e));
    };
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
    if (e != cudaSuccess)
        return cuda_err(e, "status reset");
    while (produced < max_new) {
        // drafts: never more than the tokens still wanted after the step's own
        int64_t k = 0;
        const int64_t want = std::min<int64_t>(max_draft, max_new - produced - 1);
        if (want > 0) {
            const int64_t tl = std::min<int64_t>((int64_t)seq.size(), max_ngram);
            k = tf_draft_prompt_lookup(prompt, prompt_len, seq.data() + seq.size() - tl, tl, max_ngram, (int)want, draft);
            k = std::max<int64_t>(k, 0);
        }
        const int64_t M = k + 1;
        block[0] = seq.back();
        for (int64_t i = 0; i < k; ++i)
            block[i + 1] = draft[i];
        if ((e = cudaMemcpyAsync(ids, block, (size_t)M * sizeof(int32_t), cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return cuda_err(e, "ids to device");
        // the device part of the step: embed, decoder step, argmax
        auto enqueue = [&](cudaStream_t q) -> int {
            cudaError_t le = launch_embed_rows(static_cast<const uint8_t*>(E.data), E.N, E.K, desc_kernel_bits(&E),
                                               E.global_scale, ids, M, x, E.K, status, q);
            if (le != cudaSuccess)
                return cuda_err(le, "embed");
            const int r = tf_decode_step_run(d, x, M, logits, wsb + L.step, L.step_bytes, nullptr, 0, q);
            if (r)
                return r;
            argmax_rows_kernel<<<(unsigned)M, kArgmaxThreads, 0, q>>>(logits, d->vocab, d->vocab, pred);
            le = cudaGetLastError();
            return le == cudaSuccess ? TF_OK : cuda_err(le, "argmax");
        };
        cudaGraphExec_t exec = step_graph(d, ws, ws_bytes, M, enqueue);
        if (exec != nullptr && cudaGraphLaunch(exec, s) != cudaSuccess) {
            // a cached executable that no longer launches (the context it was made in is
            // gone): forget it and launch the step directly
            cudaGetLastError();
            forget_step_graph(exec);
            exec = nullptr;
        }
        if (exec == nullptr)
            if (int rc = enqueue(s))
                return rc;
        if ((e = cudaMemcpyAsync(host, pred, (kMaxM + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
            return cuda_err(e, "predictions to host");
        if ((e = cudaStreamSynchronize(s)) != cudaSuccess)
            return cuda_err(e, "synchronise");
        if (host[kMaxM] != 0)
            return report_error(host[kMaxM], "tf_generate_greedy: a device step recorded %s",
                                tf_status_str(host[kMaxM]));
        // accept the drafts the model predicts, then the model's own next token
        int64_t a = 0;
        while (a < k && host[a] == draft[a])
            ++a;
        for (int64_t i = 0; i <= a && produced < max_new; ++i) {
            const int32_t t = i < a ? draft[i] : host[a];
            seq.push_back(t);
            out[produced++] = t;
        }
        ++steps;
        accepted += a;
    }
    // the decoder steps' own device status (a bounded wait that gave up)
    const int st = tf_workspace_status(wsb + L.step, stream);
    if (st != TF_OK)
        return report_error(st, "tf_generate_greedy: a decoder step recorded %s", tf_status_str(st));
    *n_out = produced;
    if (n_steps)
        *n_steps = steps;
    if (n_accepted)
        *n_accepted = accepted;
    return TF_OK;
}

}  // extern "C"
