// qv_internal.h -- host-side interfaces between the C ABI (qv_abi.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace qv {

// Upper bound on any wait inside a kernel, in nanoseconds of %globaltimer.
// A wait that runs out sets a bit in the device error word and the kernel
// finishes without waiting again.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Streaming-GEMM tile: BN output channels x BK bytes of the reduction axis.
constexpr int kTileN = 128;
constexpr int kTileKBytes = 128;

// Largest padded token count one W8A8 GEMM launch handles (the tcgen05
// kernel takes 64 or 80 token columns); larger M is processed in slices of
// this many rows. The BF16 comparator's launches take up to 64.
constexpr int kMaxMPerLaunch = 80;
constexpr int kMaxMPerLaunchBf16 = 64;

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
inline int pad_tokens(int m) { return ((m + 7) / 8) * 8; }

// Most CTAs of one streaming-GEMM launch (one per SM, at most this many);
// the workspace holds one split-K slot per CTA.
constexpr int kMaxStreamCtas = 160;
inline int stream_grid(long long tiles, int num_sms) {
    long long g = tiles < num_sms ? tiles : num_sms;
    return (int)(g < kMaxStreamCtas ? g : kMaxStreamCtas);
}

// Workspace layout of one GEMM call (all offsets in bytes, 16-byte aligned).
// Streaming kernels (stack = false): [slots: kMaxStreamCtas x 128 x MP
// 8-byte words][keys: MP 8-byte words][done counter]. Persistent stack
// (stack = true): [acc: Npad*MP 4-byte words][tile counters: NT words]
// [keys][done].
struct WsLayout {
    size_t slots = 0, acc = 0, counters = 0, keys = 0, done = 0, total = 0;
};
WsLayout ws_layout(int mp, int n, bool lm_head, bool stack = false);

// Linear: y = dequant(acc). LmHead: greedy argmax over y. SwiGLU: the
// gate|up weight rows interleaved by 64 (tile t holds gate rows 64t..64t+63,
// then up rows 64t..64t+63) and a = silu(y_gate) * y_up written as [M][N/2].
enum class Epi : int { Linear = 0, LmHead = 1, SwiGLU = 2 };

struct W8A8Launch {
    CUtensorMap tmap_w;       // int8 [N rows][K], box {128, 128}, 128B swizzle
    CUtensorMap tmap_x;       // int8 [M rows][K], box {128, MP}, 128B swizzle
    int M, N, K, MP;
    const float* sx;
    const float* sw;
    void* y;                  // Linear: [M*N] fp32 or bf16
    int y_bf16;
    int32_t* acc_debug;       // Linear: [M*N] or null
    int32_t* tokens;          // LmHead: [M]
    float* max_logit;         // LmHead: [M] or null
    void* ws;
    Epi epi;
    int w4;                   // 1: packed int4 weights [N rows][K/2 bytes] (streaming kernel only)
};

struct Bf16Launch {
    CUtensorMap tmap_w;       // bf16 [N rows][K], box {64, 128}, 128B swizzle
    CUtensorMap tmap_x;       // bf16 [M rows][K], box {64, MP}, 128B swizzle
    int M, N, K, MP;
    float* y;                 // [M*N] fp32
    void* ws;
};

// Phases (linears + the LM head) one persistent verify-stack launch holds;
// longer stacks are split into several launches.
constexpr int kMaxStackPhases = 150;
// Largest token count of the persistent verify-stack kernel.
constexpr int kMaxStackM = 16;

struct StackLaunchPhase {
    CUtensorMap tmap_w;
    const void* x;
    const float* act_mul;
    const float* sw;
    float* y;
    int K, N;
};

struct StackLaunch {
    const StackLaunchPhase* phases;
    int n_phases;
    bool lm_last;
    int M, MP;
    bool x_bf16;
    int B, gamma;
    const int32_t* draft;
    int32_t* tokens;
    float* max_logit;
    int32_t* accept_len;
    int32_t* out_tokens;
    void* ws;
    int n_max;                // largest N of the phases (workspace layout)
    int kmax;                 // largest K of the phases (row stride of the codes)
    CUtensorMap tmap_x;       // int8 codes [M rows][kmax] in the workspace, box {128, MP}
};

// Workspace bytes of qv_verify_stack and the offset of its int8 code buffer.
size_t stack_ws_bytes(int mp, int M, int n_max, int kmax);
size_t stack_xq_offset(int mp, int n_max);

// Test hooks (qv_debug_set_slot_wait_ns, qv_debug_drop_partials in qv.h),
// read when a streaming W8A8 / W4A8 launch is enqueued.
unsigned long long debug_slot_wait_ns();
bool debug_take_drop_partials();
bool debug_take_hold_attention();

cudaError_t launch_w8a8_stream(const W8A8Launch& a, int num_sms, cudaStream_t s);
cudaError_t launch_w8a8_tc(const W8A8Launch& a, int num_sms, cudaStream_t s);

// Largest dynamic shared memory of one CTA on sm_103a (227 KB).
constexpr size_t kMaxDynSmem = 232448;
// Dynamic shared memory that keeps a second CTA of the same kernel off an SM
// (an SM has 228 KB, each CTA also takes 1 KB of reserved shared memory).
constexpr size_t kMinSmemOneCtaPerSm = 118 * 1024;
cudaError_t launch_verify_stack(const StackLaunch& a, int num_sms, cudaStream_t s);
cudaError_t launch_bf16_stream(const Bf16Launch& a, int num_sms, cudaStream_t s);
// Greedy tree verification (k_tree.cu), N <= 1024 nodes per tree.
cudaError_t launch_tree_accept(const int32_t* t, const int32_t* d, const int32_t* par, int B, int N,
                               int32_t* len, int32_t* out, int32_t* node, cudaStream_t s);

// int4 weight quantization for the W4A8 verifier (k_w4.cu): [N][K] fp32 or
// bf16 -> packed [N][K/2] bytes + [N] scales.
cudaError_t launch_quantize_weight_w4(const void* w, bool bf16, int N, int K, uint8_t* wq4, float* sw,
                                      cudaStream_t s);
// Packed int4 weights go through the streaming kernel only: at most 32 token
// rows per launch.
constexpr int kMaxMPerLaunchW4 = 32;

// Attention over a short KV cache (k_attn.cu): one cluster launch, no workspace.
// The key and value caches as 4-D tensor maps (dims D, Hkv, Lmax, B; bf16,
// 128-byte swizzle) with boxes of 64 values x 1 head x 64 positions x 1
// sequence (k64, v64) and x 16 positions (k16, v16); NULL when Lmax == 0.
struct KvMaps {
    CUtensorMap k64, v64, k16, v16;
};
size_t attention_workspace_bytes(int B, int T, int Hq, int Hkv, int D, int Lmax);
// hold_loads, wait_ns: test hook (qv_debug_hold_attention_loads) and the
// stage-wait limit (0: kWaitLimitNs).
cudaError_t launch_attention_verify(const uint16_t* qkv, const KvMaps* maps, const int32_t* len, int B, int T, int Hq,
                                    int Hkv, int D, int Lmax, float scale, float* out, int hold_loads,
                                    unsigned long long wait_ns, cudaStream_t s);
cudaError_t read_and_clear_attn_error(unsigned* code);

// Logit-fidelity diagnostic (k_fidelity.cu): per row KL(softmax(a) ||
// softmax(b)) and both top-1 indices.
cudaError_t launch_logit_fidelity(const float* a, const float* b, int M, int V, float* kl, int32_t* top_a,
                                  int32_t* top_b, cudaStream_t s);

// Speculative sampling at T > 0 (k_spec.cu): per-chunk maxima and sums, row
// statistics and the decisions for M rows of V tokens (every call rewrites
// all of it, so the workspace needs no initialisation).
size_t spec_workspace_bytes(int M, int V);
cudaError_t launch_spec_sample(const float* logits, const int32_t* draft, const float* q, int B, int gamma,
                               int V, float T, uint64_t seed, int32_t* accept_len, int32_t* out_tokens,
                               void* ws, cudaStream_t s);

// The layer's fused non-linear steps (k_layer.cu).
cudaError_t launch_residual_rmsnorm_quant(uint16_t* h, const uint16_t* delta, const uint16_t* gamma, float eps,
                                          const float* mul, int M, int H, int8_t* xq, float* sx,
                                          uint16_t* x_out, cudaStream_t s);
cudaError_t launch_swiglu_quant(const float* gate_up, int M, int F, int8_t* xq, float* sx, cudaStream_t s);

cudaError_t launch_quantize_rows(const void* x, bool bf16, int rows, int K,
                                 const float* mul, int8_t* q, float* scale,
                                 bool early_dependents, cudaStream_t s);
cudaError_t launch_accept(const int32_t* t, const int32_t* d, int B, int gamma,
                          int32_t* len, int32_t* out, cudaStream_t s);
cudaError_t read_and_clear_stream_gemm_error(unsigned* code);
cudaError_t read_and_clear_tc_gemm_error(unsigned* code);

}  // namespace qv
