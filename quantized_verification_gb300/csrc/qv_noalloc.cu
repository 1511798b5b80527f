// qv_noalloc.cu -- qv_w8a8_linear for callers that cannot allocate device
// memory (see include/qv.h). The split-K workspace of the streaming GEMM is a
// static device array compiled into the library; this file owns the array,
// looks up its device address once per device, clears the part a call uses and
// hands it to qv_w8a8_linear as the workspace.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "qv.h"
#include "qv_internal.h"

namespace qv {
qv_status report_error(qv_status st, const char* msg);
}

namespace {

// The scratch buffer. In host code `g_noalloc_scratch` names a host-side
// stand-in, not device memory: only the address from cudaGetSymbolAddress may
// be handed to a kernel.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QV_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch buffer, per (device, context): a context
// that is destroyed and created again (cudaDeviceReset, or the primary
// context released and retained anew) loads the module again, and the
// address may change, so the lookup is repeated whenever the current
// context differs from the one the cached address came from.
struct ScratchEntry {
    int dev = -1;
    CUcontext ctx = nullptr;
    void* ptr = nullptr;
};
constexpr int kMaxEntries = 64;
ScratchEntry g_entries[kMaxEntries];
std::mutex g_scratch_mu;
using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
PFN_ctxGetCurrent g_ctx_get_current = nullptr;

qv_status fail_cuda(const char* what, cudaError_t e) {
    char msg[200];
    snprintf(msg, sizeof msg, "qv_w8a8_linear_noalloc: %s: %s", what, cudaGetErrorString(e));
    return qv::report_error(QV_ERR_CUDA, msg);
}

// Device address of the scratch buffer for the current device and context
// (looked up with that device current, once per context).
qv_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0) return fail_cuda("no usable current device", e);
    // make the device's primary context current (it is created if need be;
    // nothing is allocated)
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return fail_cuda("context set-up failed", e);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_ctx_get_current) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return qv::report_error(QV_ERR_CUDA, "qv_w8a8_linear_noalloc: cuCtxGetCurrent is not available");
        g_ctx_get_current = reinterpret_cast<PFN_ctxGetCurrent>(fn);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx)
        return qv::report_error(QV_ERR_CUDA, "qv_w8a8_linear_noalloc: no current context");
    ScratchEntry* slot = nullptr;
    for (int i = 0; i < kMaxEntries; ++i) {
        if (g_entries[i].dev == dev) { slot = &g_entries[i]; break; }
        if (!slot && g_entries[i].dev < 0) slot = &g_entries[i];
    }
    if (!slot) return qv::report_error(QV_ERR_CUDA, "qv_w8a8_linear_noalloc: too many devices");
    if (slot->dev != dev || slot->ctx != ctx || !slot->ptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return fail_cuda("cudaGetSymbolAddress failed", e);
        slot->dev = dev;
        slot->ctx = ctx;
        slot->ptr = p;
    }
    *out = slot->ptr;
    return QV_OK;
}

}  // namespace

extern "C" qv_status qv_w8a8_linear_noalloc(const int8_t* xq, const float* sx, int M, int K,
                                            const int8_t* wq, const float* sw, int N, void* y,
                                            qv_dtype y_dtype, int32_t* acc_debug,
                                            cudaStream_t stream) {
    const size_t need = qv_workspace_bytes(QV_OP_LINEAR, M, K, N);
    if (need == 0)   // invalid shape: let the regular entry point describe it
        return qv_w8a8_linear(xq, sx, M, K, wq, sw, N, y, y_dtype, acc_debug, nullptr, 0, stream);
    if (need > QV_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "qv_w8a8_linear_noalloc: M=%d N=%d needs %zu bytes of scratch, the built-in buffer "
                 "holds %u; use qv_w8a8_linear with a workspace",
                 M, N, need, (unsigned)QV_NOALLOC_SCRATCH_BYTES);
        return qv::report_error(QV_ERR_UNSUPPORTED, msg);
    }
    void* scratch = nullptr;
    qv_status st = scratch_address(&scratch);
    if (st != QV_OK) return st;
    // The GEMM needs a zero-filled workspace. A call that completes leaves
    // its part zeroed, but one that gave up on a wait limit (qv_device_error)
    // can leave partial sums behind, and the caller has no way to clear this
    // buffer: so every call clears what it uses, in stream order, first.
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, stream);
    if (e != cudaSuccess) return fail_cuda("clearing the scratch failed", e);
    return qv_w8a8_linear(xq, sx, M, K, wq, sw, N, y, y_dtype, acc_debug, scratch,
                          QV_NOALLOC_SCRATCH_BYTES, stream);
}
