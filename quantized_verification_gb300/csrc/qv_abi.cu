// qv_abi.cu -- the C ABI of libqv (declared in include/qv.h): argument
// validation, TMA descriptor encoding and dispatch to the kernels. Every
// check happens before anything is enqueued, so a rejected call leaves all
// outputs untouched.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <atomic>
#include <mutex>

#include "qv.h"
#include "qv_internal.h"

namespace {

thread_local char g_last_error[512] = "";

qv_status fail(qv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

qv_status ok() {
    g_last_error[0] = '\0';
    return QV_OK;
}

qv_status cuda_fail(cudaError_t e, const char* what) {
    return fail(QV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Every buffer a kernel touches must be device (or managed) memory of the
// current device: a host pointer handed to a kernel would fault the GPU.
qv_status check_dev(const void* p, const char* name) {
    if (!p) return QV_OK;   // optional buffers; required ones are checked for null first
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(QV_ERR_INVALID_ARG, "%s: not a CUDA allocation (%s)", name, cudaGetErrorName(e));
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fail(QV_ERR_INVALID_ARG, "%s: not device memory", name);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || at.device != dev)
        return fail(QV_ERR_INVALID_ARG, "%s: memory of device %d, current device is %d", name, at.device, dev);
    return QV_OK;
}

#define QV_CHECK_DEV(p)                                   \
    do {                                                  \
        qv_status st_ = check_dev((p), #p);               \
        if (st_ != QV_OK) return st_;                     \
    } while (0)

// ------------------------------------------------------------------ device info
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {0};
std::mutex g_mu;

int sms_of_current_device(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices && g_sms[dev] > 0) return g_sms[dev];
    int n = 0;
    *err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (*err != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) g_sms[dev] = n;
    return n;
}

// ------------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

qv_status get_encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return QV_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(QV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return QV_OK;
}

// Row-major [rows][inner] matrix with a 128-byte swizzled box of
// box_inner x box_rows elements; out-of-range elements read as zero.
qv_status encode_2d(CUtensorMap* map, CUtensorMapDataType dt, size_t elem_bytes, const void* base,
                    uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
    qv_status st = get_encoder();
    if (st != QV_OK) return st;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return QV_OK;
}

// A [B][Lmax][Hkv][D] bf16 key or value cache as a 4-D tensor map (D, Hkv,
// Lmax, B) with a box of 64 values x 1 head x box_pos positions x 1 sequence
// and the 128-byte swizzle; positions past Lmax read as zero.
qv_status encode_kv_cache(CUtensorMap* map, const void* base, int B, int Lmax, int Hkv, int D, unsigned box_pos) {
    qv_status st = get_encoder();
    if (st != QV_OK) return st;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)Lmax, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2, (cuuint64_t)Lmax * Hkv * D * 2};
    const cuuint32_t box[4] = {64, 1, box_pos, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QV_ERR_CUDA, "cuTensorMapEncodeTiled (KV cache) failed (CUresult %d)", (int)r);
    return QV_OK;
}

// W8A8 streaming GEMM kernel by padded token count. Up to 16 tokens the
// int8 (8) or f16 (16) mma.sync kernel keeps pace with HBM; from 32 tokens
// mma.sync is latency- or compute-bound and the tcgen05 kernel (exact f16
// widening, TMEM accumulators), whose per-tile cost hardly grows with the
// token count, is faster (measured on GB300 at 32 tokens: gate|up 33.8 vs
// 36.8 us, LM head 166 vs 195 us, qkv level). Packed int4 weights always use
// the streaming kernel.
cudaError_t launch_w8a8(const qv::W8A8Launch& L, int sms, cudaStream_t s) {
    if (L.w4 && L.MP > qv::kMaxMPerLaunchW4) return cudaErrorInvalidValue;
    if (!L.w4 && L.MP >= 32) return qv::launch_w8a8_tc(L, sms, s);
    return qv::launch_w8a8_stream(L, sms, s);
}

// Padded token count of a W8A8 launch of mc <= kMaxMPerLaunch rows (and of
// a BF16 launch of mc <= kMaxMPerLaunchBf16 rows).
int mp_for(int mc) {
    const int p = qv::pad_tokens(mc);
    return p <= 8 ? 8 : p <= 16 ? 16 : p <= 32 ? 32 : p <= 64 ? 64 : 80;
}

qv_status check_k(int K) {
    if (K < 16 || K % 16 != 0 || K > QV_MAX_K)
        return fail(QV_ERR_INVALID_ARG, "K=%d must be a positive multiple of 16 and <= %d", K, QV_MAX_K);
    return QV_OK;
}

qv_status check_gemm_common(const void* xq, const void* sx, int M, int K, const void* wq,
                            const void* sw, int N, const void* ws, size_t ws_bytes, qv_op op) {
    if (!xq || !sx || !wq || !sw) return fail(QV_ERR_INVALID_ARG, "null input pointer");
    if (M < 1 || M > QV_MAX_M) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, %d]", M, QV_MAX_M);
    if (N < 1) return fail(QV_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    qv_status st = check_k(K);
    if (st != QV_OK) return st;
    if (!aligned(xq, 16) || !aligned(wq, 16)) return fail(QV_ERR_INVALID_ARG, "xq and wq must be 16-byte aligned");
    if (!aligned(sx, 4) || !aligned(sw, 4)) return fail(QV_ERR_INVALID_ARG, "sx and sw must be 4-byte aligned");
    const size_t need = qv_workspace_bytes(op, M, K, N);
    if (!ws) return fail(QV_ERR_WORKSPACE, "workspace is null (%zu bytes needed)", need);
    if (!aligned(ws, 16)) return fail(QV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (ws_bytes < need) return fail(QV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, need);
    QV_CHECK_DEV(xq);
    QV_CHECK_DEV(sx);
    QV_CHECK_DEV(wq);
    QV_CHECK_DEV(sw);
    QV_CHECK_DEV(ws);
    return QV_OK;
}

size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

// Offset of the materialised codes in a *_ACT workspace: after the
// streaming-GEMM part, 256-byte aligned.
size_t act_codes_offset(bool lm, int M, int K, int N) {
    const int mp = mp_for(M < qv::kMaxMPerLaunch ? M : qv::kMaxMPerLaunch);
    return (qv::ws_layout(mp, N, lm).total + 255) & ~size_t(255);
}

// One streaming GEMM call (W8A8 or W4A8) over all token rows: the weight
// tensor map once, then one launch per slice. Rows beyond kMaxMPerLaunch
// (kMaxMPerLaunchW4 for packed int4 weights) are split into the fewest
// slices of that size, of equal row counts rounded up to 8 (128 rows run as
// two 64-row launches, measured faster than 80 + 48).
struct GemmCall {
    bool w4;
    qv::Epi epi;
    const int8_t* xq;
    const float* sx;
    int M, K;
    const void* wq;
    const float* sw;
    int N;
    uint8_t* y;            // Linear / SwiGLU output, row pitch y_row_bytes
    size_t y_row_bytes;
    int y_bf16;
    int32_t* acc_debug;
    int32_t* tokens;       // LmHead
    float* max_logit;
    void* ws;
};

qv_status run_gemm(const GemmCall& c, const char* what, cudaStream_t stream) {
    cudaError_t e;
    const int sms = sms_of_current_device(&e);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    qv::W8A8Launch L = {};
    qv_status st;
    const uint64_t w_inner = c.w4 ? (uint64_t)c.K / 2 : (uint64_t)c.K;   // weight bytes per row
    if ((st = encode_2d(&L.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, c.wq, w_inner, (uint64_t)c.N,
                        qv::kTileKBytes, qv::kTileN)) != QV_OK)
        return st;
    const int cap = c.w4 ? qv::kMaxMPerLaunchW4 : qv::kMaxMPerLaunch;
    const int nslices = (c.M + cap - 1) / cap;
    const int step = qv::pad_tokens((c.M + nslices - 1) / nslices);   // <= cap
    for (int m0 = 0; m0 < c.M; m0 += step) {
        const int mc = c.M - m0 < step ? c.M - m0 : step;
        L.M = mc; L.N = c.N; L.K = c.K; L.MP = mp_for(mc);
        if ((st = encode_2d(&L.tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, c.xq + (size_t)m0 * c.K,
                            (uint64_t)c.K, (uint64_t)mc, qv::kTileKBytes, (uint32_t)L.MP)) != QV_OK)
            return st;
        L.sx = c.sx + m0; L.sw = c.sw;
        L.y = c.y ? c.y + (size_t)m0 * c.y_row_bytes : nullptr;
        L.y_bf16 = c.y_bf16;
        L.acc_debug = c.acc_debug ? c.acc_debug + (size_t)m0 * c.N : nullptr;
        L.tokens = c.tokens ? c.tokens + m0 : nullptr;
        L.max_logit = c.max_logit ? c.max_logit + m0 : nullptr;
        L.ws = c.ws;
        L.epi = c.epi;
        L.w4 = c.w4 ? 1 : 0;
        e = launch_w8a8(L, sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, what);
    }
    return ok();
}

qv_status check_k_w4(int K) {
    if (K < 32 || K % 32 != 0 || K > QV_MAX_K)
        return fail(QV_ERR_INVALID_ARG, "K=%d must be a positive multiple of 32 and <= %d for int4 weights", K,
                    QV_MAX_K);
    return QV_OK;
}

}  // namespace

namespace qv {
// Lets other translation units of the library report through qv_last_error().
qv_status report_error(qv_status st, const char* msg) { return fail(st, "%s", msg); }

std::atomic<unsigned long long> g_debug_slot_wait_ns{0};
std::atomic<int> g_debug_drop_partials{0};
std::atomic<int> g_debug_hold_attention{0};
unsigned long long debug_slot_wait_ns() {
    const unsigned long long v = g_debug_slot_wait_ns.load();
    return v ? v : kWaitLimitNs;
}
bool debug_take_drop_partials() {
    int n = g_debug_drop_partials.load();
    while (n > 0 && !g_debug_drop_partials.compare_exchange_weak(n, n - 1)) {
    }
    return n > 0;
}
bool debug_take_hold_attention() {
    int n = g_debug_hold_attention.load();
    while (n > 0 && !g_debug_hold_attention.compare_exchange_weak(n, n - 1)) {
    }
    return n > 0;
}
}  // namespace qv

extern "C" {

const char* qv_last_error(void) { return g_last_error; }

int qv_num_sms(void) {
    cudaError_t e;
    const int n = sms_of_current_device(&e);
    return e == cudaSuccess ? n : 0;
}

size_t qv_workspace_bytes(qv_op op, int M, int K, int N) {
    if (op == QV_OP_SPEC_SAMPLE)
        return (M >= 1 && M <= 65535 && N >= 1 && N <= (1 << 24)) ? qv::spec_workspace_bytes(M, N) : 0;
    if (M < 1 || M > QV_MAX_M || N < 1 || K < 16 || K % 16 != 0 || K > QV_MAX_K) return 0;
    const int mp = mp_for(M < qv::kMaxMPerLaunch ? M : qv::kMaxMPerLaunch);
    switch (op) {
        case QV_OP_LINEAR: return qv::ws_layout(mp, N, false).total;
        case QV_OP_LM_HEAD: return qv::ws_layout(mp, N, true).total;
        case QV_OP_BF16_LINEAR:
            return qv::ws_layout(mp_for(M < qv::kMaxMPerLaunchBf16 ? M : qv::kMaxMPerLaunchBf16), N, false).total;
        case QV_OP_VERIFY_STACK:
            if (M > qv::kMaxStackM) return 0;
            return qv::stack_ws_bytes(mp, M, N, K);
        case QV_OP_SPEC_SAMPLE:
            return 0;   // handled above
        case QV_OP_LINEAR_ACT:
        case QV_OP_LM_HEAD_ACT: {
            const size_t off = act_codes_offset(op == QV_OP_LM_HEAD_ACT, M, K, N);
            return off + al16((size_t)M * K) + al16((size_t)M * 4);
        }
    }
    return 0;
}

qv_status qv_quantize_act(const void* x, qv_dtype x_dtype, int M, int K, const float* act_mul,
                          int8_t* xq, float* sx, cudaStream_t stream) {
    if (!x || !xq || !sx) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (x_dtype != QV_F32 && x_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "x_dtype must be QV_F32 or QV_BF16");
    if (M < 1 || M > 65535) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, 65535]", M);
    qv_status st = check_k(K);
    if (st != QV_OK) return st;
    if (!aligned(x, 16) || !aligned(xq, 16)) return fail(QV_ERR_INVALID_ARG, "x and xq must be 16-byte aligned");
    if (!aligned(sx, 4) || (act_mul && !aligned(act_mul, 4))) return fail(QV_ERR_INVALID_ARG, "sx/act_mul must be 4-byte aligned");
    QV_CHECK_DEV(x);
    QV_CHECK_DEV(act_mul);
    QV_CHECK_DEV(xq);
    QV_CHECK_DEV(sx);
    cudaError_t e = qv::launch_quantize_rows(x, x_dtype == QV_BF16, M, K, act_mul, xq, sx, true, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_quantize_act launch");
    return ok();
}

qv_status qv_quantize_weight(const void* w, qv_dtype w_dtype, int N, int K, int8_t* wq, float* sw,
                             cudaStream_t stream) {
    if (!w || !wq || !sw) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (w_dtype != QV_F32 && w_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "w_dtype must be QV_F32 or QV_BF16");
    if (N < 1 || N > 0x7FFFFFFF) return fail(QV_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    qv_status st = check_k(K);
    if (st != QV_OK) return st;
    if (!aligned(w, 16) || !aligned(wq, 16)) return fail(QV_ERR_INVALID_ARG, "w and wq must be 16-byte aligned");
    if (!aligned(sw, 4)) return fail(QV_ERR_INVALID_ARG, "sw must be 4-byte aligned");
    QV_CHECK_DEV(w);
    QV_CHECK_DEV(wq);
    QV_CHECK_DEV(sw);
    cudaError_t e = qv::launch_quantize_rows(w, w_dtype == QV_BF16, N, K, nullptr, wq, sw, false, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_quantize_weight launch");
    return ok();
}

qv_status qv_w8a8_linear(const int8_t* xq, const float* sx, int M, int K, const int8_t* wq,
                         const float* sw, int N, void* y, qv_dtype y_dtype, int32_t* acc_debug,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    qv_status st = check_gemm_common(xq, sx, M, K, wq, sw, N, workspace, workspace_bytes, QV_OP_LINEAR);
    if (st != QV_OK) return st;
    if (!y) return fail(QV_ERR_INVALID_ARG, "y is null");
    if (y_dtype != QV_F32 && y_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "y_dtype must be QV_F32 or QV_BF16");
    if (!aligned(y, y_dtype == QV_F32 ? 4 : 2) || (acc_debug && !aligned(acc_debug, 4)))
        return fail(QV_ERR_INVALID_ARG, "y/acc_debug misaligned");
    QV_CHECK_DEV(y);
    QV_CHECK_DEV(acc_debug);
    const size_t ybytes = y_dtype == QV_F32 ? 4 : 2;
    const GemmCall c = {false, qv::Epi::Linear, xq, sx, M, K, wq, sw, N, static_cast<uint8_t*>(y),
                        (size_t)N * ybytes, y_dtype == QV_BF16, acc_debug, nullptr, nullptr, workspace};
    return run_gemm(c, "qv_w8a8_linear launch", stream);
}

qv_status qv_w8a8_swiglu(const int8_t* xq, const float* sx, int M, int K, const int8_t* wq_gu,
                         const float* sw_gu, int F, float* a, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    if (F < 64 || F % 64 != 0) return fail(QV_ERR_INVALID_ARG, "F=%d must be a positive multiple of 64", F);
    qv_status st = check_gemm_common(xq, sx, M, K, wq_gu, sw_gu, 2 * F, workspace, workspace_bytes, QV_OP_LINEAR);
    if (st != QV_OK) return st;
    if (!a) return fail(QV_ERR_INVALID_ARG, "a is null");
    if (!aligned(a, 4)) return fail(QV_ERR_INVALID_ARG, "a misaligned");
    QV_CHECK_DEV(a);
    const GemmCall c = {false, qv::Epi::SwiGLU, xq, sx, M, K, wq_gu, sw_gu, 2 * F,
                        reinterpret_cast<uint8_t*>(a), (size_t)F * 4, 0, nullptr, nullptr, nullptr, workspace};
    return run_gemm(c, "qv_w8a8_swiglu launch", stream);
}

qv_status qv_lm_head_argmax(const int8_t* xq, const float* sx, int M, int K, const int8_t* wq,
                            const float* sw, int V, int32_t* tokens, float* max_logit,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    qv_status st = check_gemm_common(xq, sx, M, K, wq, sw, V, workspace, workspace_bytes, QV_OP_LM_HEAD);
    if (st != QV_OK) return st;
    if (!tokens) return fail(QV_ERR_INVALID_ARG, "tokens is null");
    if (!aligned(tokens, 4) || (max_logit && !aligned(max_logit, 4)))
        return fail(QV_ERR_INVALID_ARG, "tokens/max_logit misaligned");
    QV_CHECK_DEV(tokens);
    QV_CHECK_DEV(max_logit);
    const GemmCall c = {false, qv::Epi::LmHead, xq, sx, M, K, wq, sw, V, nullptr, 0, 0, nullptr,
                        tokens, max_logit, workspace};
    return run_gemm(c, "qv_lm_head_argmax launch", stream);
}

qv_status qv_quantize_weight_w4(const void* w, qv_dtype w_dtype, int N, int K, uint8_t* wq4, float* sw,
                                cudaStream_t stream) {
    if (!w || !wq4 || !sw) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (w_dtype != QV_F32 && w_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "w_dtype must be QV_F32 or QV_BF16");
    if (N < 1) return fail(QV_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    qv_status st = check_k_w4(K);
    if (st != QV_OK) return st;
    if (!aligned(w, 16) || !aligned(wq4, 16)) return fail(QV_ERR_INVALID_ARG, "w and wq4 must be 16-byte aligned");
    if (!aligned(sw, 4)) return fail(QV_ERR_INVALID_ARG, "sw must be 4-byte aligned");
    QV_CHECK_DEV(w);
    QV_CHECK_DEV(wq4);
    QV_CHECK_DEV(sw);
    cudaError_t e = qv::launch_quantize_weight_w4(w, w_dtype == QV_BF16, N, K, wq4, sw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_quantize_weight_w4 launch");
    return ok();
}

qv_status qv_w4a8_linear(const int8_t* xq, const float* sx, int M, int K, const uint8_t* wq4,
                         const float* sw, int N, void* y, qv_dtype y_dtype, int32_t* acc_debug,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    qv_status st = check_k_w4(K);
    if (st != QV_OK) return st;
    if ((st = check_gemm_common(xq, sx, M, K, wq4, sw, N, workspace, workspace_bytes, QV_OP_LINEAR)) != QV_OK)
        return st;
    if (!y) return fail(QV_ERR_INVALID_ARG, "y is null");
    if (y_dtype != QV_F32 && y_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "y_dtype must be QV_F32 or QV_BF16");
    if (!aligned(y, y_dtype == QV_F32 ? 4 : 2) || (acc_debug && !aligned(acc_debug, 4)))
        return fail(QV_ERR_INVALID_ARG, "y/acc_debug misaligned");
    QV_CHECK_DEV(y);
    QV_CHECK_DEV(acc_debug);
    const size_t ybytes = y_dtype == QV_F32 ? 4 : 2;
    const GemmCall c = {true, qv::Epi::Linear, xq, sx, M, K, wq4, sw, N, static_cast<uint8_t*>(y),
                        (size_t)N * ybytes, y_dtype == QV_BF16, acc_debug, nullptr, nullptr, workspace};
    return run_gemm(c, "qv_w4a8_linear launch", stream);
}

qv_status qv_w4a8_swiglu(const int8_t* xq, const float* sx, int M, int K, const uint8_t* wq4_gu,
                         const float* sw_gu, int F, float* a, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    if (F < 64 || F % 64 != 0) return fail(QV_ERR_INVALID_ARG, "F=%d must be a positive multiple of 64", F);
    qv_status st = check_k_w4(K);
    if (st != QV_OK) return st;
    if ((st = check_gemm_common(xq, sx, M, K, wq4_gu, sw_gu, 2 * F, workspace, workspace_bytes, QV_OP_LINEAR)) != QV_OK)
        return st;
    if (!a) return fail(QV_ERR_INVALID_ARG, "a is null");
    if (!aligned(a, 4)) return fail(QV_ERR_INVALID_ARG, "a misaligned");
    QV_CHECK_DEV(a);
    const GemmCall c = {true, qv::Epi::SwiGLU, xq, sx, M, K, wq4_gu, sw_gu, 2 * F,
                        reinterpret_cast<uint8_t*>(a), (size_t)F * 4, 0, nullptr, nullptr, nullptr, workspace};
    return run_gemm(c, "qv_w4a8_swiglu launch", stream);
}

qv_status qv_w4a8_lm_head_argmax(const int8_t* xq, const float* sx, int M, int K, const uint8_t* wq4,
                                 const float* sw, int V, int32_t* tokens, float* max_logit,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    qv_status st = check_k_w4(K);
    if (st != QV_OK) return st;
    if ((st = check_gemm_common(xq, sx, M, K, wq4, sw, V, workspace, workspace_bytes, QV_OP_LM_HEAD)) != QV_OK)
        return st;
    if (!tokens) return fail(QV_ERR_INVALID_ARG, "tokens is null");
    if (!aligned(tokens, 4) || (max_logit && !aligned(max_logit, 4)))
        return fail(QV_ERR_INVALID_ARG, "tokens/max_logit misaligned");
    QV_CHECK_DEV(tokens);
    QV_CHECK_DEV(max_logit);
    const GemmCall c = {true, qv::Epi::LmHead, xq, sx, M, K, wq4, sw, V, nullptr, 0, 0, nullptr,
                        tokens, max_logit, workspace};
    return run_gemm(c, "qv_w4a8_lm_head_argmax launch", stream);
}

namespace {
// Shared body of qv_w8a8_linear_act / qv_lm_head_argmax_act.
qv_status linear_act(bool lm, const void* x, qv_dtype x_dtype, const float* act_mul, int M, int K,
                     const int8_t* wq, const float* sw, int N, void* y, qv_dtype y_dtype,
                     int32_t* tokens, float* max_logit, void* workspace, size_t workspace_bytes,
                     cudaStream_t stream) {
    if (!x || !wq || !sw) return fail(QV_ERR_INVALID_ARG, "null input pointer");
    if (x_dtype != QV_F32 && x_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "x_dtype must be QV_F32 or QV_BF16");
    if (M < 1 || M > QV_MAX_M) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, %d]", M, QV_MAX_M);
    if (N < 1) return fail(QV_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    qv_status st = check_k(K);
    if (st != QV_OK) return st;
    if (!aligned(x, 16) || !aligned(wq, 16) || (act_mul && !aligned(act_mul, 16)))
        return fail(QV_ERR_INVALID_ARG, "x, wq and act_mul must be 16-byte aligned");
    if (!aligned(sw, 4)) return fail(QV_ERR_INVALID_ARG, "sw must be 4-byte aligned");
    if (lm) {
        if (!tokens) return fail(QV_ERR_INVALID_ARG, "tokens is null");
        if (!aligned(tokens, 4) || (max_logit && !aligned(max_logit, 4)))
            return fail(QV_ERR_INVALID_ARG, "tokens/max_logit misaligned");
    } else {
        if (!y) return fail(QV_ERR_INVALID_ARG, "y is null");
        if (y_dtype != QV_F32 && y_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "y_dtype must be QV_F32 or QV_BF16");
        if (!aligned(y, y_dtype == QV_F32 ? 4 : 2)) return fail(QV_ERR_INVALID_ARG, "y misaligned");
    }
    const qv_op op = lm ? QV_OP_LM_HEAD_ACT : QV_OP_LINEAR_ACT;
    const size_t need = qv_workspace_bytes(op, M, K, N);
    if (!workspace) return fail(QV_ERR_WORKSPACE, "workspace is null (%zu bytes needed)", need);
    if (!aligned(workspace, 16)) return fail(QV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (workspace_bytes < need) return fail(QV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    QV_CHECK_DEV(x);
    QV_CHECK_DEV(act_mul);
    QV_CHECK_DEV(wq);
    QV_CHECK_DEV(sw);
    QV_CHECK_DEV(workspace);
    QV_CHECK_DEV(y);
    QV_CHECK_DEV(tokens);
    QV_CHECK_DEV(max_logit);
    // The codes and token scales go to the workspace (qv_quantize_act's
    // kernel), then the GEMM streams the weights against them.
    cudaError_t e;
    // The codes sit at the end of the caller's buffer, 256-byte aligned, so a
    // buffer shared by calls of different shapes keeps every call's GEMM part
    // (which must stay zero-filled) clear of any call's codes.
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    const size_t codes = al16((size_t)M * K) + al16((size_t)M * 4);
    const size_t off = (workspace_bytes - codes) & ~size_t(255);
    int8_t* xq = reinterpret_cast<int8_t*>(wsb + off);
    float* sx = reinterpret_cast<float*>(wsb + off + al16((size_t)M * K));
    e = qv::launch_quantize_rows(x, x_dtype == QV_BF16, M, K, act_mul, xq, sx, true, stream);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantization launch");
    if (lm)
        return qv_lm_head_argmax(xq, sx, M, K, wq, sw, N, tokens, max_logit, workspace, off, stream);
    return qv_w8a8_linear(xq, sx, M, K, wq, sw, N, y, y_dtype, nullptr, workspace, off, stream);
}
}  // namespace

qv_status qv_w8a8_linear_act(const void* x, qv_dtype x_dtype, const float* act_mul, int M, int K,
                             const int8_t* wq, const float* sw, int N, void* y, qv_dtype y_dtype,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return linear_act(false, x, x_dtype, act_mul, M, K, wq, sw, N, y, y_dtype, nullptr, nullptr,
                      workspace, workspace_bytes, stream);
}

qv_status qv_lm_head_argmax_act(const void* x, qv_dtype x_dtype, const float* act_mul, int M, int K,
                                const int8_t* wq, const float* sw, int V, int32_t* tokens,
                                float* max_logit, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
    return linear_act(true, x, x_dtype, act_mul, M, K, wq, sw, V, nullptr, QV_F32, tokens, max_logit,
                      workspace, workspace_bytes, stream);
}

qv_status qv_rmsnorm_quant(uint16_t* h, const uint16_t* delta, const uint16_t* gamma, float eps,
                           const float* act_mul, int M, int H, int8_t* xq, float* sx, uint16_t* x_out,
                           cudaStream_t stream) {
    if (!h || !gamma || !xq || !sx) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (M < 1 || M > 65535) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, 65535]", M);
    if (H < 16 || H > 16384 || H % 16 != 0)
        return fail(QV_ERR_INVALID_ARG, "H=%d must be a multiple of 16 in [16, 16384]", H);
    if (!(eps >= 0.0f) || eps > 3.0e38f) return fail(QV_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (!aligned(h, 16) || (delta && !aligned(delta, 16)) || !aligned(gamma, 16) || !aligned(xq, 16) ||
        (act_mul && !aligned(act_mul, 16)) || (x_out && !aligned(x_out, 16)) || !aligned(sx, 4))
        return fail(QV_ERR_INVALID_ARG, "h, delta, gamma, xq, act_mul, x_out must be 16-byte aligned");
    QV_CHECK_DEV(h);
    QV_CHECK_DEV(delta);
    QV_CHECK_DEV(gamma);
    QV_CHECK_DEV(act_mul);
    QV_CHECK_DEV(xq);
    QV_CHECK_DEV(sx);
    QV_CHECK_DEV(x_out);
    cudaError_t e = qv::launch_residual_rmsnorm_quant(h, delta, gamma, eps, act_mul, M, H, xq, sx, x_out, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_rmsnorm_quant launch");
    return ok();
}

qv_status qv_swiglu_quant(const float* gate_up, int M, int F, int8_t* xq, float* sx, cudaStream_t stream) {
    if (!gate_up || !xq || !sx) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (M < 1 || M > 65535) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, 65535]", M);
    if (F < 16 || F > 32768 || F % 16 != 0)
        return fail(QV_ERR_INVALID_ARG, "F=%d must be a multiple of 16 in [16, 32768]", F);
    if (!aligned(gate_up, 16) || !aligned(xq, 16) || !aligned(sx, 4))
        return fail(QV_ERR_INVALID_ARG, "gate_up and xq must be 16-byte aligned");
    QV_CHECK_DEV(gate_up);
    QV_CHECK_DEV(xq);
    QV_CHECK_DEV(sx);
    cudaError_t e = qv::launch_swiglu_quant(gate_up, M, F, xq, sx, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_swiglu_quant launch");
    return ok();
}

qv_status qv_tree_accept(const int32_t* verify_tokens, const int32_t* draft, const int32_t* parent, int B, int N,
                         int32_t* accept_len, int32_t* out_tokens, int32_t* best_node, cudaStream_t stream) {
    if (!verify_tokens || !draft || !parent || !accept_len || !out_tokens) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (B < 1 || B > 65535) return fail(QV_ERR_INVALID_ARG, "B=%d outside [1, 65535]", B);
    if (N < 1 || N > 1024) return fail(QV_ERR_INVALID_ARG, "N=%d outside [1, 1024]", N);
    if (!aligned(verify_tokens, 4) || !aligned(draft, 4) || !aligned(parent, 4) || !aligned(accept_len, 4) ||
        !aligned(out_tokens, 4) || (best_node && !aligned(best_node, 4)))
        return fail(QV_ERR_INVALID_ARG, "int32 buffers must be 4-byte aligned");
    QV_CHECK_DEV(verify_tokens);
    QV_CHECK_DEV(draft);
    QV_CHECK_DEV(parent);
    QV_CHECK_DEV(accept_len);
    QV_CHECK_DEV(out_tokens);
    QV_CHECK_DEV(best_node);
    cudaError_t e = qv::launch_tree_accept(verify_tokens, draft, parent, B, N, accept_len, out_tokens, best_node,
                                           stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_tree_accept launch");
    return ok();
}

qv_status qv_spec_sample(const float* logits, const int32_t* draft, const float* draft_probs, int B,
                         int gamma, int V, float temperature, uint64_t seed, int32_t* accept_len,
                         int32_t* out_tokens, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!logits || !accept_len || !out_tokens) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (B < 1) return fail(QV_ERR_INVALID_ARG, "B=%d must be >= 1", B);
    if (gamma < 0 || gamma > 1023) return fail(QV_ERR_INVALID_ARG, "gamma=%d outside [0, 1023]", gamma);
    if (gamma > 0 && (!draft || !draft_probs)) return fail(QV_ERR_INVALID_ARG, "draft / draft_probs null with gamma > 0");
    if (V < 1 || V > (1 << 24)) return fail(QV_ERR_INVALID_ARG, "V=%d outside [1, 2^24]", V);
    if (!(temperature > 0.0f) || temperature > 3.0e38f)
        return fail(QV_ERR_INVALID_ARG, "temperature must be finite and > 0");
    if ((long long)B * (gamma + 1) > 65535) return fail(QV_ERR_INVALID_ARG, "B*(gamma+1) must be <= 65535");
    if (!aligned(logits, 4) || (draft && !aligned(draft, 4)) || (draft_probs && !aligned(draft_probs, 4)) ||
        !aligned(accept_len, 4) || !aligned(out_tokens, 4))
        return fail(QV_ERR_INVALID_ARG, "buffers must be 4-byte aligned");
    const int M = B * (gamma + 1);
    const size_t need = qv_workspace_bytes(QV_OP_SPEC_SAMPLE, M, 16, V);
    if (!workspace) return fail(QV_ERR_WORKSPACE, "workspace is null (%zu bytes needed)", need);
    if (!aligned(workspace, 16)) return fail(QV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (workspace_bytes < need) return fail(QV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    QV_CHECK_DEV(logits);
    QV_CHECK_DEV(draft);
    QV_CHECK_DEV(draft_probs);
    QV_CHECK_DEV(accept_len);
    QV_CHECK_DEV(out_tokens);
    QV_CHECK_DEV(workspace);
    cudaError_t e = qv::launch_spec_sample(logits, gamma > 0 ? draft : nullptr, gamma > 0 ? draft_probs : nullptr,
                                           B, gamma, V, temperature, seed, accept_len, out_tokens, workspace,
                                           stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_spec_sample launch");
    return ok();
}

namespace {
qv_status check_attention_shape(int B, int T, int Hq, int Hkv, int D, int Lmax) {
    if (B < 1 || B > 65535) return fail(QV_ERR_INVALID_ARG, "B=%d outside [1, 65535]", B);
    if (T < 1) return fail(QV_ERR_INVALID_ARG, "T=%d must be >= 1", T);
    if (Hkv < 1 || Hkv > 65535 || Hq < Hkv || Hq % Hkv != 0)
        return fail(QV_ERR_INVALID_ARG, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
    if ((long long)T * (Hq / Hkv) > 32) return fail(QV_ERR_INVALID_ARG, "T * Hq / Hkv must be <= 32");
    if (D != 64 && D != 128) return fail(QV_ERR_INVALID_ARG, "D=%d must be 64 or 128", D);
    if (Lmax < 0 || Lmax > (1 << 24)) return fail(QV_ERR_INVALID_ARG, "Lmax=%d outside [0, 2^24]", Lmax);
    return QV_OK;
}
}  // namespace

size_t qv_attention_workspace_bytes(int B, int T, int Hq, int Hkv, int D, int Lmax) {
    if (check_attention_shape(B, T, Hq, Hkv, D, Lmax) != QV_OK) return 0;
    return qv::attention_workspace_bytes(B, T, Hq, Hkv, D, Lmax);
}

qv_status qv_attention_verify(const uint16_t* qkv, const uint16_t* k_cache, const uint16_t* v_cache,
                              const int32_t* cache_len, int B, int T, int Hq, int Hkv, int D, int Lmax,
                              float scale, float* out, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    qv_status st = check_attention_shape(B, T, Hq, Hkv, D, Lmax);
    if (st != QV_OK) return st;
    if (!qkv || !cache_len || !out) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (Lmax > 0 && (!k_cache || !v_cache)) return fail(QV_ERR_INVALID_ARG, "k_cache / v_cache null with Lmax > 0");
    if (!(scale > 0.0f) || scale > 3.0e38f) return fail(QV_ERR_INVALID_ARG, "scale must be finite and > 0");
    if (!aligned(qkv, 16) || (k_cache && !aligned(k_cache, 16)) || (v_cache && !aligned(v_cache, 16)) ||
        !aligned(cache_len, 4) || !aligned(out, 4))
        return fail(QV_ERR_INVALID_ARG, "qkv and the caches must be 16-byte aligned");
    (void)workspace;          // the kernel needs none (partials stay in distributed shared memory)
    (void)workspace_bytes;
    QV_CHECK_DEV(qkv);
    QV_CHECK_DEV(k_cache);
    QV_CHECK_DEV(v_cache);
    QV_CHECK_DEV(cache_len);
    QV_CHECK_DEV(out);
    qv::KvMaps maps;
    if (Lmax > 0) {
        st = encode_kv_cache(&maps.k64, k_cache, B, Lmax, Hkv, D, 64);
        if (st == QV_OK) st = encode_kv_cache(&maps.v64, v_cache, B, Lmax, Hkv, D, 64);
        if (st == QV_OK) st = encode_kv_cache(&maps.k16, k_cache, B, Lmax, Hkv, D, 16);
        if (st == QV_OK) st = encode_kv_cache(&maps.v16, v_cache, B, Lmax, Hkv, D, 16);
        if (st != QV_OK) return st;
    }
    const int hold = qv::debug_take_hold_attention() ? 1 : 0;
    cudaError_t e = qv::launch_attention_verify(qkv, Lmax > 0 ? &maps : nullptr, cache_len, B, T, Hq, Hkv, D, Lmax,
                                                scale, out, hold, qv::debug_slot_wait_ns(), stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_attention_verify launch");
    return ok();
}

qv_status qv_logit_fidelity(const float* ref_logits, const float* logits, int M, int V, float* kl,
                            int32_t* top1_ref, int32_t* top1, cudaStream_t stream) {
    if (!ref_logits || !logits || !kl || !top1_ref || !top1) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (M < 1 || M > 65535) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, 65535]", M);
    if (V < 1 || V > (1 << 24)) return fail(QV_ERR_INVALID_ARG, "V=%d outside [1, 2^24]", V);
    if (!aligned(ref_logits, 4) || !aligned(logits, 4) || !aligned(kl, 4) || !aligned(top1_ref, 4) ||
        !aligned(top1, 4))
        return fail(QV_ERR_INVALID_ARG, "buffers must be 4-byte aligned");
    QV_CHECK_DEV(ref_logits);
    QV_CHECK_DEV(logits);
    QV_CHECK_DEV(kl);
    QV_CHECK_DEV(top1_ref);
    QV_CHECK_DEV(top1);
    cudaError_t e = qv::launch_logit_fidelity(ref_logits, logits, M, V, kl, top1_ref, top1, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_logit_fidelity launch");
    return ok();
}

qv_status qv_accept(const int32_t* verify_tokens, const int32_t* draft, int B, int gamma,
                    int32_t* accept_len, int32_t* out_tokens, cudaStream_t stream) {
    if (!verify_tokens || !accept_len || !out_tokens) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (B < 1) return fail(QV_ERR_INVALID_ARG, "B=%d must be >= 1", B);
    if (gamma < 0 || gamma > 1023) return fail(QV_ERR_INVALID_ARG, "gamma=%d outside [0, 1023]", gamma);
    if (gamma > 0 && !draft) return fail(QV_ERR_INVALID_ARG, "draft is null with gamma > 0");
    if (!aligned(verify_tokens, 4) || !aligned(accept_len, 4) || !aligned(out_tokens, 4) ||
        (draft && !aligned(draft, 4)))
        return fail(QV_ERR_INVALID_ARG, "int32 buffers must be 4-byte aligned");
    QV_CHECK_DEV(verify_tokens);
    QV_CHECK_DEV(draft);
    QV_CHECK_DEV(accept_len);
    QV_CHECK_DEV(out_tokens);
    cudaError_t e = qv::launch_accept(verify_tokens, draft, B, gamma, accept_len, out_tokens, stream);
    if (e != cudaSuccess) return cuda_fail(e, "qv_accept launch");
    return ok();
}

qv_status qv_bf16_linear(const uint16_t* x, int M, int K, const uint16_t* w, int N, float* y,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!x || !w || !y) return fail(QV_ERR_INVALID_ARG, "null pointer");
    if (M < 1 || M > QV_MAX_M) return fail(QV_ERR_INVALID_ARG, "M=%d outside [1, %d]", M, QV_MAX_M);
    if (N < 1) return fail(QV_ERR_INVALID_ARG, "N=%d must be >= 1", N);
    qv_status st = check_k(K);
    if (st != QV_OK) return st;
    if (!aligned(x, 16) || !aligned(w, 16)) return fail(QV_ERR_INVALID_ARG, "x and w must be 16-byte aligned");
    if (!aligned(y, 4)) return fail(QV_ERR_INVALID_ARG, "y must be 4-byte aligned");
    const size_t need = qv_workspace_bytes(QV_OP_BF16_LINEAR, M, K, N);
    if (!workspace) return fail(QV_ERR_WORKSPACE, "workspace is null (%zu bytes needed)", need);
    if (!aligned(workspace, 16)) return fail(QV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (workspace_bytes < need) return fail(QV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    QV_CHECK_DEV(x);
    QV_CHECK_DEV(w);
    QV_CHECK_DEV(y);
    QV_CHECK_DEV(workspace);
    cudaError_t e;
    const int sms = sms_of_current_device(&e);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    qv::Bf16Launch L = {};
    if ((st = encode_2d(&L.tmap_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, (uint64_t)K, (uint64_t)N,
                        qv::kTileKBytes / 2, qv::kTileN)) != QV_OK)
        return st;
    for (int m0 = 0; m0 < M; m0 += qv::kMaxMPerLaunchBf16) {
        const int mc = M - m0 < qv::kMaxMPerLaunchBf16 ? M - m0 : qv::kMaxMPerLaunchBf16;
        L.M = mc; L.N = N; L.K = K; L.MP = mp_for(mc);
        if ((st = encode_2d(&L.tmap_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x + (size_t)m0 * K,
                            (uint64_t)K, (uint64_t)mc, qv::kTileKBytes / 2, (uint32_t)L.MP)) != QV_OK)
            return st;
        L.y = y + (size_t)m0 * N;
        L.ws = workspace;
        e = qv::launch_bf16_stream(L, sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "qv_bf16_linear launch");
    }
    return ok();
}

qv_status qv_verify_stack(const qv_linear_desc* linears, int n_linears, const qv_linear_desc* lm_head,
                          int M, qv_dtype x_dtype, const int32_t* draft, int B, int gamma,
                          int32_t* tokens, float* max_logit, int32_t* accept_len, int32_t* out_tokens,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (n_linears < 0 || (n_linears > 0 && !linears)) return fail(QV_ERR_INVALID_ARG, "bad linears array");
    if (n_linears == 0 && !lm_head) return fail(QV_ERR_INVALID_ARG, "nothing to run");
    if (M < 1 || M > qv::kMaxStackM)
        return fail(QV_ERR_UNSUPPORTED, "M=%d outside [1, %d] for the stack kernel", M, qv::kMaxStackM);
    if (x_dtype != QV_F32 && x_dtype != QV_BF16) return fail(QV_ERR_INVALID_ARG, "x_dtype must be QV_F32 or QV_BF16");
    int n_max = 0, k_max = 0;
    auto check_desc = [&](const qv_linear_desc& d, int idx, bool lm) -> qv_status {
        if (!d.x || !d.wq || !d.sw) return fail(QV_ERR_INVALID_ARG, "phase %d: null x/wq/sw", idx);
        if (d.N < 1) return fail(QV_ERR_INVALID_ARG, "phase %d: N=%d", idx, d.N);
        qv_status st = check_k(d.K);
        if (st != QV_OK) return st;
        if (!aligned(d.x, 16) || !aligned(d.wq, 16) || (d.act_mul && !aligned(d.act_mul, 16)))
            return fail(QV_ERR_INVALID_ARG, "phase %d: x, wq and act_mul must be 16-byte aligned", idx);
        if (!aligned(d.sw, 4) || (!lm && d.y && !aligned(d.y, 4)))
            return fail(QV_ERR_INVALID_ARG, "phase %d: misaligned sw/y", idx);
        if ((st = check_dev(d.x, "x")) != QV_OK || (st = check_dev(d.wq, "wq")) != QV_OK ||
            (st = check_dev(d.sw, "sw")) != QV_OK || (st = check_dev(d.act_mul, "act_mul")) != QV_OK ||
            (!lm && (st = check_dev(d.y, "y")) != QV_OK))
            return st;
        if (d.N > n_max) n_max = d.N;
        if (d.K > k_max) k_max = d.K;
        return QV_OK;
    };
    for (int i = 0; i < n_linears; ++i) {
        qv_status st = check_desc(linears[i], i, false);
        if (st != QV_OK) return st;
    }
    if (lm_head) {
        qv_status st = check_desc(*lm_head, n_linears, true);
        if (st != QV_OK) return st;
        if (!tokens || !aligned(tokens, 4) || (max_logit && !aligned(max_logit, 4)))
            return fail(QV_ERR_INVALID_ARG, "tokens required (4-byte aligned) with an LM head");
        QV_CHECK_DEV(tokens);
        QV_CHECK_DEV(max_logit);
        if (accept_len || out_tokens) {
            if (!accept_len || !out_tokens) return fail(QV_ERR_INVALID_ARG, "accept_len and out_tokens go together");
            if (B < 1 || gamma < 0 || (long long)B * (gamma + 1) != M)
                return fail(QV_ERR_INVALID_ARG, "B*(gamma+1) must equal M (B=%d gamma=%d M=%d)", B, gamma, M);
            if (gamma > 0 && !draft) return fail(QV_ERR_INVALID_ARG, "draft is null with gamma > 0");
            if (!aligned(accept_len, 4) || !aligned(out_tokens, 4) || (draft && !aligned(draft, 4)))
                return fail(QV_ERR_INVALID_ARG, "int32 buffers must be 4-byte aligned");
            QV_CHECK_DEV(accept_len);
            QV_CHECK_DEV(out_tokens);
            QV_CHECK_DEV(draft);
        }
    } else if (tokens || accept_len || out_tokens) {
        return fail(QV_ERR_INVALID_ARG, "tokens/acceptance outputs need an LM head");
    }
    const size_t need = qv_workspace_bytes(QV_OP_VERIFY_STACK, M, k_max, n_max);
    if (!workspace) return fail(QV_ERR_WORKSPACE, "workspace is null (%zu bytes needed)", need);
    if (!aligned(workspace, 16)) return fail(QV_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    if (workspace_bytes < need) return fail(QV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    QV_CHECK_DEV(workspace);

    cudaError_t e;
    const int sms = sms_of_current_device(&e);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    static thread_local qv::StackLaunchPhase ph[qv::kMaxStackPhases];
    const int total = n_linears + (lm_head ? 1 : 0);
    const int mp = mp_for(M);
    CUtensorMap tmap_x;
    {
        const int8_t* xq = static_cast<const int8_t*>(workspace) + qv::stack_xq_offset(mp, n_max);
        qv_status st = encode_2d(&tmap_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xq, (uint64_t)k_max,
                                 (uint64_t)M, qv::kTileKBytes, (uint32_t)mp);
        if (st != QV_OK) return st;
    }
    for (int first = 0; first < total; first += qv::kMaxStackPhases) {
        const int count = total - first < qv::kMaxStackPhases ? total - first : qv::kMaxStackPhases;
        for (int j = 0; j < count; ++j) {
            const int idx = first + j;
            const qv_linear_desc& d = idx < n_linears ? linears[idx] : *lm_head;
            qv_status st = encode_2d(&ph[j].tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, d.wq, (uint64_t)d.K,
                                     (uint64_t)d.N, qv::kTileKBytes, qv::kTileN);
            if (st != QV_OK) return st;
            ph[j].x = d.x; ph[j].act_mul = d.act_mul; ph[j].sw = d.sw;
            ph[j].y = idx < n_linears ? d.y : nullptr;
            ph[j].K = d.K; ph[j].N = d.N;
        }
        qv::StackLaunch L = {};
        L.phases = ph; L.n_phases = count;
        L.lm_last = lm_head && first + count == total;
        L.M = M; L.MP = mp; L.x_bf16 = x_dtype == QV_BF16;
        L.B = B; L.gamma = gamma; L.draft = draft;
        L.tokens = tokens; L.max_logit = max_logit;
        L.accept_len = accept_len; L.out_tokens = out_tokens;
        L.ws = workspace; L.n_max = n_max; L.kmax = k_max; L.tmap_x = tmap_x;
        e = qv::launch_verify_stack(L, sms, stream);
        if (e != cudaSuccess) return cuda_fail(e, "qv_verify_stack launch");
    }
    return ok();
}

void qv_debug_set_slot_wait_ns(unsigned long long ns) { qv::g_debug_slot_wait_ns.store(ns); }

void qv_debug_drop_partials(int n) { qv::g_debug_drop_partials.store(n > 0 ? n : 0); }

void qv_debug_hold_attention_loads(int n) { qv::g_debug_hold_attention.store(n > 0 ? n : 0); }

qv_status qv_device_error(unsigned int* code) {
    if (!code) return fail(QV_ERR_INVALID_ARG, "code is null");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned tc = 0, at = 0;
    e = qv::read_and_clear_stream_gemm_error(code);
    if (e == cudaSuccess) e = qv::read_and_clear_tc_gemm_error(&tc);
    if (e == cudaSuccess) e = qv::read_and_clear_attn_error(&at);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    *code |= tc | at;
    return ok();
}

}  // extern "C"
