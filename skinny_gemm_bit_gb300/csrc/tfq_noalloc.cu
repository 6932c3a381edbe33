// tf_qlinear_run_noalloc: the projection of tf_qlinear_run without a
// caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory where they make the
// call -- code running inside an allocator or memory-pool callback (allocating
// there re-enters the allocator), a latency-critical path that has reserved all
// of its memory up front and must never reach cudaMalloc or a caching allocator,
// or a foreign-language host that can call a C function but has no handle on a
// device allocator. For them, the split-K / stream-K scratch of the projection
// lives in one fixed, file-scope device array of kNoAllocScratchBytes per device,
// shared by every call of this entry point.
//
// The array is zero when the module is loaded, and every projection leaves its
// scratch as it found it (split-K counters and partial slots are re-zeroed by the
// CTA that consumes them), so it needs no clearing between calls. Its address is
// looked up once per device, with that device current, on the first call there.
// A device-side failure (a bounded wait that ran out) leaves its status in the
// array's first word and may leave counters or partial slots dirty:
// tf_qlinear_noalloc_status reports it and puts the array back to zero.
#include <atomic>
#include <mutex>

#include "tfq_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

// Status word (first 256 bytes), split-K arrival counters and fp32 partial slots
// of tf_qlinear_run, in the layout that call gives its workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_lookup_mu;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// The device address of g_noalloc_scratch on the current device (looked up on
// the first call there, then cached).
int scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return tfq::report_error(TF_E_CUDA, "tf_qlinear_run_noalloc: cudaGetDevice failed: %s",
                                 cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return tfq::report_error(TF_E_UNSUPPORTED_SHAPE, "tf_qlinear_run_noalloc: device %d beyond the %d supported",
                                 dev, kMaxDevices);
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(g_lookup_mu);
        p = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (p == nullptr) {
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr)
                return tfq::report_error(TF_E_CUDA,
                                         "tf_qlinear_run_noalloc: cudaGetSymbolAddress of the scratch array "
                                         "failed on device %d: %s",
                                         dev, cudaGetErrorString(e));
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return TF_OK;
}

}  // namespace

namespace tfq {
// The current device's fixed array (for the diagnostics in tfq_api.cu).
int noalloc_scratch(void** out, size_t* bytes)
{
    *bytes = kNoAllocScratchBytes;
    return scratch_address(out);
}
}  // namespace tfq

extern "C" int tf_qlinear_run_noalloc(const tf_qweight* w, const uint16_t* x, int64_t ldx, int64_t M,
                                      const uint16_t* rms_gamma, float rms_eps, const uint16_t* residual, void* y,
                                      int y_dtype, unsigned flags, void* stream)
{
    // the size check needs only the descriptor: nothing is looked up or enqueued
    // for a shape the fixed array cannot serve
    int rc = tfq::validate_desc(w, "tf_qlinear_run_noalloc");
    if (rc)
        return rc;
    if (M < 1 || M > tfq::kMaxM)
        return tfq::report_error(TF_E_UNSUPPORTED_SHAPE, "tf_qlinear_run_noalloc: M must be in [1, 8] (got %lld)",
                                 (long long)M);
    const size_t need = tf_qlinear_workspace_bytes(w, M);
    if (need == 0)
        return TF_E_INVALID_ARG;  // the query has set the message
    if (need > kNoAllocScratchBytes)
        return tfq::report_error(TF_E_WORKSPACE_TOO_SMALL,
                                 "tf_qlinear_run_noalloc: this shape (N=%lld, K=%lld) needs %zu bytes of scratch, "
                                 "more than the fixed %zu; call tf_qlinear_run with a workspace instead",
                                 (long long)w->N, (long long)w->K, need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)))
        return rc;
    return tfq::qlinear_run_named(w, x, ldx, M, rms_gamma, rms_eps, residual, y, y_dtype, scratch,
                                  kNoAllocScratchBytes, flags, stream, "tf_qlinear_run_noalloc");
}

extern "C" int tf_qlinear_noalloc_status(void* stream)
{
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc)
        return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, scratch, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && st != 0) {
        // the failed call may have left arrival counters and partial slots behind
        e = cudaMemsetAsync(scratch, 0, kNoAllocScratchBytes, s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess)
        return tfq::report_error(TF_E_CUDA, "tf_qlinear_noalloc_status: %s", cudaGetErrorString(e));
    if (st != 0)
        tfq::report_error(st, "tf_qlinear_noalloc_status: a device-side failure was recorded in the fixed array "
                              "(now cleared)");
    return st;
}
