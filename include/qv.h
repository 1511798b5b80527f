/*
 * qv.h -- C ABI of libqv, the GB300 (sm_103a) W8A8 quantized verify pass.
 *
 * The method: "Quasar: Quantized Self-Speculative Acceleration for Rapid
 * Inference via Memory-Efficient Verification". The verify pass of
 * speculative decoding runs on a W8A8 copy of the target model: activations
 * are quantized per token to symmetric int8, multiplied by per-output-channel
 * symmetric int8 weights with exact int32 accumulation, dequantized back to
 * high precision, and the greedy verifier tokens decide how many draft tokens
 * are accepted. Passages are cited by the summary page (site and language)
 * and its section.
 *
 * Conventions shared by every entry point
 *   - All pointers except `stream` are DEVICE pointers of the current device
 *     (device or managed memory; checked with cudaPointerGetAttributes, a
 *     host pointer is rejected with QV_ERR_INVALID_ARG).
 *     The caller allocates and owns every buffer, including workspaces;
 *     libqv allocates no device memory and never synchronizes the device.
 *   - Every call only enqueues work on `stream` (NULL = legacy default
 *     stream) and returns immediately.
 *   - Matrices are row-major and densely packed: element (r, c) of an
 *     R x C matrix is at r*C + c.
 *   - Arguments are validated on the host before anything is enqueued. A call
 *     that returns a status other than QV_OK has enqueued nothing and left
 *     every output untouched; qv_last_error() then describes the problem.
 *     QV_ERR_CUDA reports a failed launch (the CUDA error is in the message).
 *   - int8 and bf16 buffers must be 16-byte aligned; fp32 and int32 buffers
 *     4-byte aligned. K must be a positive multiple of 16 and at most
 *     QV_MAX_K, the largest K for which every int32 sum of K products of
 *     codes in [-127, 127] is exact.
 *   - Kernels of this library may begin before the previous kernel on the
 *     same stream has finished (programmatic dependent launch). Before that
 *     wait completes they read only weight codes (`wq`); everything else is
 *     read after all earlier work on the stream is complete and visible.
 *     Weight codes therefore must not be written by a kernel that is still
 *     running when the call is enqueued; qv_quantize_weight never lets its
 *     successor start early, so quantize-then-use on one stream is safe.
 *   - Results are deterministic: every call returns identical bits for
 *     identical inputs. The fp32 results of the bf16 comparator, of
 *     attention and of the logit-fidelity diagnostic also depend on how the
 *     work is split (the SM count, the cluster size), so they are repeatable
 *     on one GPU model, not across.
 */
#ifndef QV_H
#define QV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define QV_API __attribute__((visibility("default")))
#else
#define QV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QV_OK = 0,
    QV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size        */
    QV_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels handle    */
    QV_ERR_WORKSPACE = 3,     /* workspace missing or too small           */
    QV_ERR_CUDA = 4           /* a CUDA call failed                        */
} qv_status;

typedef enum { QV_F32 = 0, QV_BF16 = 1 } qv_dtype;

typedef enum {
    QV_OP_LINEAR = 0,         /* qv_w8a8_linear                            */
    QV_OP_LM_HEAD = 1,        /* qv_lm_head_argmax (N = vocabulary size V) */
    QV_OP_BF16_LINEAR = 2,    /* qv_bf16_linear                            */
    QV_OP_VERIFY_STACK = 3,   /* qv_verify_stack (K, N = largest K, N / V) */
    QV_OP_LINEAR_ACT = 4,     /* qv_w8a8_linear_act                        */
    QV_OP_LM_HEAD_ACT = 5,    /* qv_lm_head_argmax_act (N = V)             */
    QV_OP_SPEC_SAMPLE = 6     /* qv_spec_sample (M = B*(gamma+1), N = V; K ignored) */
} qv_op;

/* floor((2^31 - 1) / 127^2): the int32 accumulation stays exact up to here. */
#define QV_MAX_K 133144
/* Largest number of verify tokens (rows of activations) per call. */
#define QV_MAX_M 256

/*
 * qv_quantize_act -- a1: dynamic per-token symmetric int8 activation
 * quantization, with an optional smoothing multiply.
 *
 *   Quasar, gist.science/ja summary, section 2.2 "Enhanced SmoothQuant",
 *   item 3: the BF16 input activation is scaled by the per-channel smoothing
 *   factor and converted to INT8 online; item 1 gives the smoothing identity
 *   Y = (W diag(s)^-1)(diag(s) X). gist.science/de summary, section 2
 *   "Methodik", "Online-Prozess". Per-token granularity and the rounding rule
 *   are this library's reading of the summaries (they give neither).
 *
 * For every row m < M (one token):
 *   x'[k]  = fl32(x[m][k] * act_mul[k])      (x'[k] = x[m][k] if act_mul NULL)
 *   amax   = max_k |x'[k]|
 *   sx[m]  = fl32(amax / 127)                (IEEE division)
 *   xq[m][k] = clamp(round_half_even(fl32(x'[k] / sx[m])), -127, 127),
 *              or 0 for every k when sx[m] == 0.
 *
 *   x       [M*K] fp32 or bf16 (x_dtype), 16-byte aligned
 *   act_mul [K] fp32 multipliers already in "multiply" form, or NULL
 *   xq      [M*K] int8 out, 16-byte aligned
 *   sx      [M] fp32 out
 *   1 <= M <= 65535 (rows are independent; M is not bounded by QV_MAX_M here).
 * Non-finite inputs are outside the contract.
 */
QV_API qv_status qv_quantize_act(const void* x, qv_dtype x_dtype, int M, int K,
                          const float* act_mul, int8_t* xq, float* sx,
                          cudaStream_t stream);

/*
 * qv_w8a8_linear -- a2: int8 x int8 GEMM with exact int32 accumulation and a
 * fused dequantization epilogue.
 *
 *   Quasar, gist.science/ja summary, section 2.2 item 3: INT8 GEMM,
 *   accumulation in INT32, dequantization to high precision before the
 *   non-linear layers; gist.science/fr summary, section 2 "Pipeline
 *   Technique" (INT8 tensor cores, results dequantized).
 *
 *   acc[m][n] = sum_k xq[m][k] * wq[n][k]            (exact integer)
 *   y[m][n]   = fl32( fl32((float)acc[m][n]) * fl32(sx[m] * sw[n]) )
 *               stored as fp32, or rounded to bf16 (nearest even) when
 *               y_dtype == QV_BF16.
 *
 *   xq  [M*K] int8, sx [M] fp32      -- from qv_quantize_act
 *   wq  [N*K] int8, sw [N] fp32      -- from qv_quantize_weight (row n =
 *                                       output channel n, K contiguous)
 *   y   [M*N] fp32 or bf16 out
 *   acc_debug [M*N] int32 out, or NULL: the exact accumulators
 *   workspace: at least qv_workspace_bytes(QV_OP_LINEAR, M, K, N) bytes,
 *     16-byte aligned, ZERO-FILLED before its first use. Every call leaves
 *     it zero-filled again when its work completes, so one workspace can be
 *     reused by any sequence of stream-ordered calls. Calls that run
 *     concurrently (different streams) need separate workspaces.
 *     Recovery: a call that gives up on a wait limit (qv_device_error then
 *     reports QV_DEVICE_ERR_SLOT_WAIT) has undefined outputs and may leave
 *     partial sums in its workspace; zero-fill the workspace again before
 *     the next call that uses it.
 *   1 <= M <= QV_MAX_M, N >= 1. Codes of -128 are accepted; the sums are
 *   exact whenever they fit int32, which codes in [-127, 127] guarantee.
 *   Co-residency: the kernel runs at most one CTA per SM (no more CTAs than
 *   SMs), and where a channel tile's K range is split between CTAs, the CTA
 *   holding the tile's first K block waits at the end for the others'
 *   partial sums. It therefore expects all of its CTAs to run at the same
 *   time: if a kernel on another stream (or another process under MPS)
 *   holds SMs for longer than the wait limit (about one second), the call
 *   gives up with QV_DEVICE_ERR_SLOT_WAIT instead of waiting forever.
 */
QV_API qv_status qv_w8a8_linear(const int8_t* xq, const float* sx, int M, int K,
                         const int8_t* wq, const float* sw, int N,
                         void* y, qv_dtype y_dtype, int32_t* acc_debug,
                         void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * qv_lm_head_argmax -- a3: the W8A8 LM head fused with the greedy argmax.
 *
 *   The logits stay in high precision for the acceptance test:
 *   gist.science/it summary, section 2 item 3 ("Campionamento di Rifiuto
 *   Lossless"); greedy decoding (T=0), gist.science/ja summary, section 4.
 *
 *   y[m][v]     = the qv_w8a8_linear value for N = V (never stored)
 *   tokens[m]   = the smallest v with y[m][v] == max_v' y[m][v']
 *   max_logit[m]= that maximum (optional)
 * Ties go to the lowest index; -0 and +0 compare equal. NaN is outside the
 * contract.
 *
 *   wq [V*K] int8, sw [V] fp32, tokens [M] int32 out, max_logit [M] or NULL
 *   workspace: qv_workspace_bytes(QV_OP_LM_HEAD, M, K, V) bytes, same
 *   zero-fill contract as qv_w8a8_linear.
 *   1 <= M <= QV_MAX_M, 1 <= V.
 */
QV_API qv_status qv_lm_head_argmax(const int8_t* xq, const float* sx, int M, int K,
                            const int8_t* wq, const float* sw, int V,
                            int32_t* tokens, float* max_logit,
                            void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * qv_w8a8_linear_act -- a1 + a2 in one call: per-token quantization of the
 * activations (qv_quantize_act) followed by the W8A8 linear (qv_w8a8_linear),
 * with the same kernels, so y is bit-identical to the two calls.
 *
 *   Quasar, gist.science/ja summary, section 2.2 items 2-3: BF16
 *   activations scaled by the smoothing factor, converted to INT8 online,
 *   INT8 GEMM with INT32 accumulation, dequantized to high precision.
 *
 *   x [M*K] fp32 or bf16 (x_dtype), 16-byte aligned; act_mul [K] fp32 or
 *   NULL, 16-byte aligned; wq, sw, y, y_dtype as qv_w8a8_linear.
 *   workspace: at least qv_workspace_bytes(QV_OP_LINEAR_ACT, M, K, N)
 *   bytes, 16-byte aligned, ZERO-FILLED before its first use. Its start is
 *   the qv_w8a8_linear workspace (left zero-filled, as there); the int8 codes
 *   and token scales are written to its last M*K + 4*M bytes (each rounded
 *   up to 16, placed at a 256-byte boundary). A buffer shared by several
 *   stream-ordered *_ACT calls of different shapes must therefore hold the
 *   largest GEMM part (qv_workspace_bytes of QV_OP_LINEAR / QV_OP_LM_HEAD,
 *   rounded up to 256) plus the largest code part.
 *   1 <= M <= QV_MAX_M, N >= 1. Two kernels are enqueued (quantization,
 *   then the streaming GEMM, which starts loading weights while the first
 *   one runs). A single kernel doing both was measured slower on GB300:
 *   every CTA needs the whole-row scales, so it would repeat the amax pass.
 */
QV_API qv_status qv_w8a8_linear_act(const void* x, qv_dtype x_dtype, const float* act_mul,
                                    int M, int K, const int8_t* wq, const float* sw, int N,
                                    void* y, qv_dtype y_dtype,
                                    void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream);

/*
 * qv_lm_head_argmax_act -- a1 + a3 in one call: qv_quantize_act of the
 * final hidden state followed by qv_lm_head_argmax, bit-identical to the two
 * calls (same fusion rule and workspace contract as qv_w8a8_linear_act,
 * workspace qv_workspace_bytes(QV_OP_LM_HEAD_ACT, M, K, V)).
 */
QV_API qv_status qv_lm_head_argmax_act(const void* x, qv_dtype x_dtype, const float* act_mul,
                                       int M, int K, const int8_t* wq, const float* sw, int V,
                                       int32_t* tokens, float* max_logit,
                                       void* workspace, size_t workspace_bytes,
                                       cudaStream_t stream);

/*
 * qv_w8a8_swiglu -- the gate|up projection of a layer's MLP with SiLU(gate) *
 * up fused into its epilogue (a2 with a SwiGLU epilogue).
 *
 *   gist.science/ja summary, section 2.2 item 3 (INT8 GEMM, INT32
 *   accumulation, dequantization to high precision before the non-linear
 *   layer, here applied in the same kernel).
 *
 *   wq_gu [2F][K] int8, sw_gu [2F]: the gate and up weight rows interleaved
 *     by 64: rows 128t .. 128t+63 are gate rows 64t .. 64t+63 and rows
 *     128t+64 .. 128t+127 the up rows 64t .. 64t+63 (so one 128-channel tile
 *     holds both operands of 64 features). F % 64 == 0.
 *   y_g, y_u = the qv_w8a8_linear outputs (fp32) of the gate and up rows
 *   a [M][F] fp32 out: a[m][f] = fl32(silu(y_g[m][f]) * y_u[m][f]), silu as
 *     in qv_swiglu_quant.
 *   xq, sx, M, K, workspace: as qv_w8a8_linear (workspace:
 *     qv_workspace_bytes(QV_OP_LINEAR, M, K, 2F)).
 */
QV_API qv_status qv_w8a8_swiglu(const int8_t* xq, const float* sx, int M, int K,
                                const int8_t* wq_gu, const float* sw_gu, int F, float* a,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * qv_rmsnorm_quant -- the residual add and RMSNorm in front of a layer's
 * linears, fused with the a1 quantization of their input (one row per token).
 *
 *   gist.science/ja summary, section 2.2 item 3: the GEMM's result returns to
 *   high precision before the non-linear layers, and the next linear's BF16
 *   input is converted to INT8 online. The layer itself (a Qwen3-shaped
 *   decoder with a bf16 residual stream) is this library's reading; the
 *   summaries do not spell it out.
 *
 *   if delta:  h[m][k] = rne_bf16(fl32(h[m][k] + delta[m][k]))   (written back)
 *   ss   = sum_k h[m][k]^2 in binary64;  var = fl32(ss / H)
 *   rstd = fl32(1 / fl32(sqrt(fl32(var + eps))))
 *   x[m][k] = rne_bf16(fl32(gamma[k] * rne_bf16(fl32(h[m][k] * rstd))))
 *   xq, sx = the qv_quantize_act codes and scale of x (times act_mul if given)
 *
 *   h      [M*H] bf16, in/out (updated only when delta is given), 16-byte aligned
 *   delta  [M*H] bf16 (a linear's bf16 output) or NULL, 16-byte aligned
 *   gamma  [H] bf16 norm weights, 16-byte aligned; act_mul [H] fp32 or NULL
 *   xq     [M*H] int8 out, sx [M] fp32 out; x_out [M*H] bf16 out or NULL (x)
 *   1 <= M <= 65535, 16 <= H <= 16384, H % 16 == 0, eps >= 0 finite.
 * The kernel adds the exact binary32 squares in float-float (about 48 bits),
 * which matches the binary64 sum to about 2^-47 relative: var is the same
 * unless ss / H lies that close to a binary32 rounding boundary. Non-finite
 * inputs are outside the contract.
 */
QV_API qv_status qv_rmsnorm_quant(uint16_t* h, const uint16_t* delta, const uint16_t* gamma,
                                  float eps, const float* act_mul, int M, int H,
                                  int8_t* xq, float* sx, uint16_t* x_out, cudaStream_t stream);

/*
 * qv_swiglu_quant -- SiLU(gate) * up on the gate|up linear's output, fused
 * with the a1 quantization of the down projection's input.
 *
 *   gist.science/ja summary, section 2.2 item 3 (non-linear layers in high
 *   precision after dequantization, INT8 input for the next linear).
 *
 *   gate_up [M][2F] fp32: gate in columns [0, F), up in [F, 2F)
 *   a[m][k] = fl32(fl32(g * sigma(g)) * up[m][k]), g = gate[m][k],
 *   sigma(v) = fl32(1 / fl32(1 + E(-v))), E the library's binary32 exp:
 *     v > 88 -> +inf, v < -87 -> 0, else k = rne(fl(v * 1.44269504)),
 *     r = fl(fl(v - fl(k * 0.693145751953125)) - fl(k * 1.4286068e-6)),
 *     E = fl(p(r) * 2^k) with p the degree-7 Taylor polynomial of e^r by
 *     Horner (coefficients fl(1/n!)); within 2 ulp of e^v.
 *   xq [M*F] int8, sx [M] fp32 = the per-token quantization of a.
 *   gate_up 16-byte aligned; 1 <= M <= 65535, 16 <= F <= 32768, F % 16 == 0.
 */
QV_API qv_status qv_swiglu_quant(const float* gate_up, int M, int F, int8_t* xq, float* sx,
                                 cudaStream_t stream);

/*
 * qv_tree_accept -- greedy (T = 0) verification of a draft tree.
 *
 *   Tree-structured verification is the extension the summaries name for
 *   the drafts (gist.science/de and gist.science/ja summaries, section 5);
 *   along each root path the rule is qv_accept's.
 *
 * Tree b has N nodes, stored at [b*N + i]: node 0 is the root (the last
 * accepted position); node i >= 1 has parent[i] (valid when in [0, i)) and
 * drafted token draft[i] (draft[0] and parent[0] are ignored);
 * verify_tokens[i] is the verifier's greedy token after node i's root path
 * (e.g. qv_lm_head_argmax over the M = B*N tree rows with a tree attention
 * mask). Node i is accepted when every node j != 0 on its root path has a
 * valid parent p and draft[j] == verify_tokens[p].
 *   best = the accepted node of largest depth, the lowest index among them
 *   accept_len[b] = depth(best) + 1                       (in [1, N])
 *   out_tokens[b*N + 0 .. depth-1] = the drafted tokens on the root -> best
 *   path, out_tokens[b*N + depth] = verify_tokens[best], then -1
 *   best_node[b] = best (or NULL)
 * Token ids are compared as raw int32. 1 <= B <= 65535, 1 <= N <= 1024.
 */
QV_API qv_status qv_tree_accept(const int32_t* verify_tokens, const int32_t* draft, const int32_t* parent,
                                int B, int N, int32_t* accept_len, int32_t* out_tokens, int32_t* best_node,
                                cudaStream_t stream);

/*
 * qv_spec_sample -- acceptance at temperature T > 0: lossless rejection
 * sampling (speculative sampling) over the verifier's logits.
 *
 *   gist.science/it summary, section 2 item 3 ("Campionamento di Rifiuto
 *   Lossless"): the verifier's logits stay precise so that the target
 *   distribution is kept. The rule is the textbook one: keep draft d_j with
 *   probability min(1, p_j(d_j) / q_j(d_j)); at the first rejection draw from
 *   the normalized max(0, p_j - q_j); with every draft kept, draw the bonus
 *   token from p_gamma. Emitted tokens are distributed as sampling from p.
 *
 *   logits      [B*(gamma+1)][V] fp32 (e.g. qv_w8a8_linear of the LM head);
 *               row b*(gamma+1)+j follows prefix position j
 *   draft       [B*gamma] int32 drafted tokens (drawn from draft_probs)
 *   draft_probs [B*gamma][V] fp32 draft probabilities q (values clamped to
 *               [0, 1]; need not sum to 1)
 *   temperature > 0; p_j = softmax(logits_j / temperature)
 *   seed        selects the uniforms (same seed, same inputs: same outputs)
 *   accept_len  [B] out, in [1, gamma+1]; out_tokens [B*(gamma+1)] out: the
 *               kept drafts, the replacement or bonus token, then -1
 *   workspace   qv_workspace_bytes(QV_OP_SPEC_SAMPLE, B*(gamma+1), 16, V)
 *               bytes, 16-byte aligned (per-chunk maxima and sums, row
 *               statistics; no zero-fill needed)
 * Arithmetic (so that every decision is exact and reproducible): with E the
 * library's binary32 exp (qv_swiglu_quant), m = max_v z_v,
 * w_v = floor(E(fl32(fl32(z_v - m) / T)) * 2^24), Z = sum w_v,
 * c_v = floor(fl32(q_v * 2^24)), Q = sum c_v; keep d iff
 * u * Z * c_d < w_d * Q * 2^24 (128-bit integers); replacement weights
 * max(0, w_v * Q - c_v * Z), or w when all are 0; a draw from weights x is
 * the smallest v whose prefix sum exceeds floor(u' * sum(x) / 2^24). u, u'
 * are the top 24 bits of SplitMix64 draws 2*row and 2*row + 1 of the seed
 * (counter-based: mix(seed + (n+1) * 0x9E3779B97F4A7C15)).
 * Draft tokens outside [0, V) are never kept. B >= 1, 0 <= gamma <= 1023,
 * 1 <= V <= 16777216, logits and draft_probs 4-byte aligned.
 */
QV_API qv_status qv_spec_sample(const float* logits, const int32_t* draft, const float* draft_probs,
                                int B, int gamma, int V, float temperature, uint64_t seed,
                                int32_t* accept_len, int32_t* out_tokens,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * qv_accept -- a4: greedy acceptance of the longest matching draft prefix
 * plus one verifier token.
 *
 *   gist.science/fr summary, lay explanation: a wrong draft token is
 *   rejected and generation continues from the verifier's token; at least
 *   one token is produced per step (acceptance length L ~ 1.03 for a nearly
 *   useless verifier, gist.science/ja summary, section 4). At T = 0 the
 *   rejection-sampling rule of gist.science/it summary, section 2 item 3
 *   reduces to exact matching against the argmax.
 *
 * Sequence b has gamma+1 verify rows: verify_tokens[b*(gamma+1) + j] is the
 * verifier's token after prefix position j (j = 0 is the last accepted
 * token); draft[b*gamma + j] is the (j+1)-th drafted token.
 *   k = the largest i <= gamma with draft[b][j] == verify[b][j] for all j < i
 *   accept_len[b]       = k + 1                       (in [1, gamma+1])
 *   out_tokens[b][j]    = verify[b][j] for j <= k, else -1
 * Token ids are compared as raw int32. B >= 1, 0 <= gamma <= 1023;
 * draft may be NULL when gamma == 0.
 */
QV_API qv_status qv_accept(const int32_t* verify_tokens, const int32_t* draft,
                    int B, int gamma, int32_t* accept_len,
                    int32_t* out_tokens, cudaStream_t stream);

/*
 * qv_quantize_weight -- a0 (setup, not on the timed path): per-output-channel
 * symmetric int8 weight quantization. Same rule as qv_quantize_act with one
 * row per output channel and no smoothing multiply:
 *   sw[n] = fl32(amax_n / 127), wq[n][k] = clamp(rne(fl32(w[n][k] / sw[n])))
 *   Quasar, gist.science/ja summary, section 2.2 item 2 (weights quantized
 *   to INT8 offline); gist.science/it summary, section 2 "Preparazione
 *   Offline".
 *   w [N*K] fp32 or bf16, wq [N*K] int8 out, sw [N] fp32 out; 1 <= N.
 * The kernel it launches lets no successor start before it has finished.
 */
QV_API qv_status qv_quantize_weight(const void* w, qv_dtype w_dtype, int N, int K,
                             int8_t* wq, float* sw, cudaStream_t stream);

/*
 * qv_attention_verify -- attention over a short KV cache for the verify
 * tokens: the attention between the qkv and o projections of the decoder
 * layer that the verify pass runs (the non-GEMM computation stays in high
 * precision: Quasar, gist.science/ja summary, section 2.2 item 3). The
 * summaries do not spell attention out; this is causal grouped-query
 * scaled dot-product attention.
 *   qkv       [B*T][(Hq + 2 Hkv) * D] bf16 device, 16-byte aligned: the qkv
 *             projection's rows (token-major, sequence-contiguous: row
 *             b*T + j), Hq query heads, then Hkv key heads, then Hkv value
 *             heads, D values each (no positional rotation is applied here)
 *   k_cache, v_cache [B][Lmax][Hkv][D] bf16 device, 16-byte aligned (may be
 *             NULL when Lmax == 0); cache_len [B] int32 device, each in
 *             [0, Lmax] (values outside are clamped)
 *   out       [B*T][Hq * D] fp32 device: for token j of sequence b and query
 *             head h (key/value head h / (Hq/Hkv)), the softmax over the
 *             cache_len[b] cached positions and the step's tokens 0..j of
 *             scale * q . k, applied to the values
 *   T * Hq/Hkv <= 32, D in {64, 128}, 1 <= B <= 65535, 0 <= Lmax <= 2^24
 *   workspace, workspace_bytes: not used (may be NULL / 0); kept so that
 *             callers sized by qv_attention_workspace_bytes keep working
 *             (it returns 16 for a valid shape, 0 for an invalid one)
 * One launch of 8-CTA thread-block clusters, one cluster per (sequence,
 * key/value head): the CTAs split the key positions, load the caches with
 * TMA, score them and form P V on the bf16 tensor cores (fp32
 * accumulation; P is split into two bf16 parts) with an online softmax, and
 * merge their partials through distributed shared memory. Cache positions
 * at and past cache_len[b] are never read (they may hold anything). Each
 * CTA asks for about 195 KB of shared memory and a cluster needs 8 such SMs
 * at once: where the device cannot place one (e.g. a small MPS partition)
 * the call returns QV_ERR_CUDA. A wait inside the kernel that runs out
 * sets QV_DEVICE_ERR_FULL_WAIT (qv_device_error).
 * The outputs are within about 1e-5 of max |v| of the binary64 definition.
 */
QV_API size_t qv_attention_workspace_bytes(int B, int T, int Hq, int Hkv, int D, int Lmax);
QV_API qv_status qv_attention_verify(const uint16_t* qkv, const uint16_t* k_cache, const uint16_t* v_cache,
                                     const int32_t* cache_len, int B, int T, int Hq, int Hkv, int D,
                                     int Lmax, float scale, float* out, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream);

/*
 * qv_logit_fidelity -- diagnostic: how far the quantized verifier's output
 * distribution is from a reference verifier's, per row.
 *   The Quasar summaries report negligible KL divergence between the
 *   full-precision and the quantized verifier's logit distributions
 *   (gist.science/fr summary, contributions item 3; shd-paper.top summary,
 *   method details, core idea).
 *   ref_logits, logits [M*V] fp32 device, row-major (e.g. the BF16
 *   verifier's and the W8A8 verifier's logits of the same tokens);
 *   kl [M] fp32 out = KL(p || q) in nats, p = softmax(ref row),
 *   q = softmax(row); top1_ref, top1 [M] int32 out = the first index of
 *   each row's maximum (top-1 agreement = equality).
 *   Computed as log1p(E_p[expm1(d - c)]) with d = logits - ref_logits and
 *   c = E_p[d] (binary32 terms, sums of about 48 bits): relative error about
 *   1e-3 of KL or better for KL down to 1e-8. Logits must be finite with
 *   |d - c| < 80. 1 <= M <= 65535, 1 <= V <= 2^24.
 *   One launch of M thread-block clusters of 16 CTAs (a non-portable
 *   cluster size: the GPU must fit 16 co-resident CTAs of 1024 threads in
 *   one GPC, which GB300 does; QV_ERR_CUDA otherwise), up to about 200 KB
 *   of shared memory per CTA; no workspace.
 */
QV_API qv_status qv_logit_fidelity(const float* ref_logits, const float* logits, int M, int V,
                                   float* kl, int32_t* top1_ref, int32_t* top1, cudaStream_t stream);

/*
 * W4A8 -- the lower-bit verifier: int4 weights against the int8 activation
 * codes of qv_quantize_act.
 *   Lower bit widths (4-bit, 2-bit) for the verifier are the next step the
 *   Quasar summaries name (gist.science/it, gist.science/de and
 *   gist.science/ja summaries, section 5); INT4 is among the widths the
 *   authors tried (shd-paper.top summary, method details, key design).
 *   The pages give no int4 format; the one here keeps a2's exact integer
 *   accumulation and dequantization unchanged.
 *
 * qv_quantize_weight_w4 (setup): per-output-channel symmetric int4,
 *   sw[n] = fl32(amax_n / 7), q = clamp(rne(fl32(w[n][k] / sw[n])), -7, 7),
 *   q = 0 for a row whose scale is 0. Packed two codes per byte:
 *   wq4[n*K/2 + j] = (q[n][2j] & 0xF) | (q[n][2j+1] & 0xF) << 4 (4-bit two's
 *   complement; -8 is never produced).
 *   w [N*K] fp32 or bf16 (16-byte aligned), wq4 [N*K/2] bytes out (16-byte
 *   aligned), sw [N] fp32 out; K a multiple of 32 in [32, QV_MAX_K].
 *
 * qv_w4a8_linear, qv_w4a8_swiglu, qv_w4a8_lm_head_argmax: qv_w8a8_linear,
 *   qv_w8a8_swiglu and qv_lm_head_argmax with packed int4 weights in place
 *   of int8 ones; every other argument, the results, the workspace (sized by
 *   qv_workspace_bytes with QV_OP_LINEAR / QV_OP_LM_HEAD, left zero-filled)
 *   and the errors are theirs. acc[m][n] = sum_k xq[m][k] * q[n][k] exactly
 *   (|acc| <= 127 * 7 * K), y = fl32(fl32((float)acc) * fl32(sx[m]*sw[n])).
 *   K must be a multiple of 32 (QV_ERR_INVALID_ARG otherwise). For
 *   qv_w4a8_swiglu the 2F packed rows are interleaved like qv_w8a8_swiglu's.
 *   Up to 32 token rows run per launch; more rows take several launches.
 */
QV_API qv_status qv_quantize_weight_w4(const void* w, qv_dtype w_dtype, int N, int K,
                                       uint8_t* wq4, float* sw, cudaStream_t stream);
QV_API qv_status qv_w4a8_linear(const int8_t* xq, const float* sx, int M, int K,
                                const uint8_t* wq4, const float* sw, int N,
                                void* y, qv_dtype y_dtype, int32_t* acc_debug,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);
QV_API qv_status qv_w4a8_swiglu(const int8_t* xq, const float* sx, int M, int K,
                                const uint8_t* wq4_gu, const float* sw_gu, int F, float* a,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);
QV_API qv_status qv_w4a8_lm_head_argmax(const int8_t* xq, const float* sx, int M, int K,
                                        const uint8_t* wq4, const float* sw, int V,
                                        int32_t* tokens, float* max_logit,
                                        void* workspace, size_t workspace_bytes,
                                        cudaStream_t stream);

/*
 * qv_bf16_linear -- the high-precision verifier being replaced, as a traffic
 * comparator: y = x w^T with bf16 operands and fp32 accumulation.
 *   The verify pass "in full precision (BF16)" whose weight traffic the
 *   method halves: gist.science/ja summary, sections 2.1 and 2.3;
 *   gist.science/de summary, section 3 item 4 (T_verify ~ M*2B/BW versus
 *   M*1B/BW).
 *   x [M*K] bf16, w [N*K] bf16, y [M*N] fp32 out.
 *   workspace: qv_workspace_bytes(QV_OP_BF16_LINEAR, M, K, N) bytes, same
 *   zero-fill contract as qv_w8a8_linear. The fp32 partial sums of one
 *   output (one per CTA its K range is split over) are added in K order; the
 *   split depends only on the shape and the SM count, so repeated calls on
 *   one GPU give identical results.
 *   1 <= M <= QV_MAX_M.
 */
QV_API qv_status qv_bf16_linear(const uint16_t* x, int M, int K, const uint16_t* w,
                         int N, float* y, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * qv_verify_stack -- one whole verify pass in a single persistent launch:
 * a sequence of quantize -> W8A8 linear phases (a1 + a2 per phase), then
 * optionally the LM head with the greedy argmax (a3) and the acceptance (a4).
 * It computes exactly what the per-op calls compute, in the same order, with
 * bit-identical results: phase i equals qv_quantize_act(linears[i].x) followed
 * by qv_w8a8_linear, the LM head equals qv_quantize_act + qv_lm_head_argmax,
 * the acceptance equals qv_accept.
 *   Quasar, gist.science/ja summary, section 2.2 item 3 (online quantize,
 *   INT8 GEMM, dequantize, for every linear of the verifier's forward pass);
 *   gist.science/it summary, section 2 item 3 (acceptance on the dequantized
 *   logits).
 * Phase i+1 starts only after every output of phase i is written (a
 * device-wide barrier), as if its input depended on them; weight codes of
 * later phases are streamed while earlier phases compute, since they never
 * depend on activations.
 *
 *   linears   host array of n_linears descriptors (read during the call only);
 *             each: x [M*K] (x_dtype, 16-byte aligned), act_mul [K] or NULL
 *             (16-byte aligned), wq [N*K] int8, sw [N], y [M*N] fp32 or NULL
 *             (output not stored).
 *   lm_head   host descriptor of the LM head (N = V; its y is ignored), or
 *             NULL to run the linears only.
 *   tokens [M], max_logit [M] or NULL: as qv_lm_head_argmax (required with
 *             lm_head).
 *   accept_len [B], out_tokens [B*(gamma+1)]: as qv_accept, or both NULL to
 *             skip acceptance; then B*(gamma+1) must equal M and draft
 *             [B*gamma] must be given when gamma > 0.
 *   workspace: qv_workspace_bytes(QV_OP_VERIFY_STACK, M, K_max, N_max) bytes
 *             with K_max the largest K and N_max the largest N (or V),
 *             zero-filled before first use; every call leaves its counters
 *             and partial sums zero-filled (its int8 code area is scratch).
 *   1 <= M <= 16. The kernel keeps one CTA resident on every SM (cooperative
 *   launch); at most 150 phases (linears + LM head) run per launch and longer
 *   stacks are split into consecutive launches on the stream.
 */
typedef struct {
    const void* x;          /* [M*K] input activations, x_dtype of the call */
    const float* act_mul;   /* [K] smoothing multipliers, or NULL           */
    const int8_t* wq;       /* [N*K] int8 weight codes                       */
    const float* sw;        /* [N] fp32 weight scales                        */
    float* y;               /* [M*N] fp32 dequantized output, or NULL        */
    int K, N;
} qv_linear_desc;

QV_API qv_status qv_verify_stack(const qv_linear_desc* linears, int n_linears,
                                 const qv_linear_desc* lm_head, int M, qv_dtype x_dtype,
                                 const int32_t* draft, int B, int gamma,
                                 int32_t* tokens, float* max_logit,
                                 int32_t* accept_len, int32_t* out_tokens,
                                 void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* Workspace bytes an op needs for the given shape (N = V for the LM head);
 * 0 for an invalid shape. Host function, enqueues nothing. */
QV_API size_t qv_workspace_bytes(qv_op op, int M, int K, int N);

/* Message for the last non-OK status returned on the calling thread
 * (thread-local; "" if none). Host function. */
QV_API const char* qv_last_error(void);

/*
 * qv_device_error -- reads and clears the library's device-side error word.
 * Kernels never trap: a wait inside a kernel that exceeds its time limit
 * (about one second) sets a bit here and the kernel returns early with
 * undefined outputs. 0 means no such event since the last read.
 * Synchronizes the current device. Host function.
 */
#define QV_DEVICE_ERR_FULL_WAIT  1u   /* a consumer waited too long for a tile    */
#define QV_DEVICE_ERR_EMPTY_WAIT 2u   /* the producer waited too long for a slot  */
#define QV_DEVICE_ERR_DRAIN_WAIT 4u   /* copies still in flight at the kernel end */
#define QV_DEVICE_ERR_GRID_WAIT  8u   /* a grid barrier of qv_verify_stack        */
#define QV_DEVICE_ERR_TC_WAIT    16u  /* the tensor-core pipeline (large M)       */
#define QV_DEVICE_ERR_SLOT_WAIT  32u  /* a split-K head waited for partial sums   */
QV_API qv_status qv_device_error(unsigned int* code);

/*
 * Test hooks. They let a test make a bounded in-kernel wait run out, without
 * faulting or hanging the GPU, and check the error reporting and the
 * recovery rule above; production code leaves them alone. Host functions;
 * they affect calls enqueued (or captured) after them, on every thread.
 *   qv_debug_set_slot_wait_ns(ns): limit, in ns of %globaltimer, of the
 *     split-K head's wait for partial sums in the streaming kernels of
 *     qv_w8a8_linear / qv_w8a8_swiglu / qv_lm_head_argmax and the W4A8 calls
 *     (up to 32 token rows per launch); 0 restores the default (1 s).
 *   qv_debug_drop_partials(n): the next n such launches publish no split-K
 *     partial sums, so every split tile's head waits out its limit, sets
 *     QV_DEVICE_ERR_SLOT_WAIT and finishes with incomplete sums.
 *   qv_debug_hold_attention_loads(n): the next n qv_attention_verify calls
 *     request none of their key/value stages, so every stage wait runs out
 *     (after the qv_debug_set_slot_wait_ns limit, else 1 s), sets
 *     QV_DEVICE_ERR_FULL_WAIT and the outputs are undefined; no copy is left
 *     in flight, and later calls are unaffected.
 */
QV_API void qv_debug_set_slot_wait_ns(unsigned long long ns);
QV_API void qv_debug_drop_partials(int n);
QV_API void qv_debug_hold_attention_loads(int n);

/* Number of SMs the kernels size their grids for on the current device
 * (queried once per device). Host function. */
QV_API int qv_num_sms(void);

/* Bytes of the library's built-in scratch buffer (see qv_w8a8_linear_noalloc). */
#define QV_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * qv_w8a8_linear_noalloc -- qv_w8a8_linear for callers that cannot allocate
 * device memory. The paper has no counterpart: this is a deployment aid.
 *
 * Who needs it: code that runs where cudaMalloc is off limits -- a plugin or
 * callback handed only the input and output buffers of a host framework, code
 * running under a memory budget owned by someone else, or a caller that must
 * not allocate between steps -- and therefore cannot provide the zero-filled
 * workspace qv_w8a8_linear asks for.
 *
 * Same arguments and same results (bit for bit) as qv_w8a8_linear, minus the
 * workspace: the split-K partial sums live in a buffer of
 * QV_NOALLOC_SCRATCH_BYTES compiled into the library (a static device array;
 * every GPU that loads the library holds it until the process exits). The
 * call itself allocates nothing.
 *   - The first call on a device looks up the buffer's device address for
 *     that device (once); make that first call before any stream capture.
 *   - Shapes whose workspace, qv_workspace_bytes(QV_OP_LINEAR, M, K, N), is
 *     larger than the buffer are rejected with QV_ERR_UNSUPPORTED. With the
 *     present workspace layout (split-K slots of at most 13.1 MB, at M > 64)
 *     every shape that qv_w8a8_linear accepts fits.
 *   - The address is looked up again when the current context of the device
 *     changes (after cudaDeviceReset the module, and the buffer, are loaded
 *     anew).
 *   - Each call clears the part of the buffer it uses (cudaMemsetAsync on
 *     `stream`, 1.3 MB for up to 8 token rows, 13.1 MB above 64) before its
 *     kernel runs: a completed call leaves that part zeroed, but a call that
 *     gave up on a wait limit (qv_device_error reports it) may leave partial
 *     sums behind, and the caller has no other way to clear the buffer.
 *   - All calls on a device share the one buffer: calls whose GPU work
 *     overlaps (different streams, no ordering between them) race on it and
 *     give wrong results. Order them on one stream, or use qv_w8a8_linear
 *     with a workspace per stream.
 */
QV_API qv_status qv_w8a8_linear_noalloc(const int8_t* xq, const float* sx, int M, int K,
                                        const int8_t* wq, const float* sw, int N,
                                        void* y, qv_dtype y_dtype, int32_t* acc_debug,
                                        cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QV_H */
