// qv_noalloc.cu -- qv_w8a8_linear for callers that cannot allocate device
// memory (see include/qv.h). The split-K workspace of the streaming GEMM is a
// static device array compiled into the library; this file owns the array,
// looks up its device address once per device, clears the part a call uses and
// hands it to qv_w8a8_linear as the workspace.

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

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch buffer on the current device (looked up once
// per device, with that device current).
qv_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return qv::report_error(QV_ERR_CUDA, "qv_w8a8_linear_noalloc: no usable current device");
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            char msg[160];
            snprintf(msg, sizeof msg, "qv_w8a8_linear_noalloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            return qv::report_error(QV_ERR_CUDA, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
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
    // The GEMM needs a zero-filled workspace; clear what this call uses.
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, stream);
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof msg, "qv_w8a8_linear_noalloc: clearing the scratch failed: %s",
                 cudaGetErrorString(e));
        return qv::report_error(QV_ERR_CUDA, msg);
    }
    return qv_w8a8_linear(xq, sx, M, K, wq, sw, N, y, y_dtype, acc_debug, scratch,
                          QV_NOALLOC_SCRATCH_BYTES, stream);
}
