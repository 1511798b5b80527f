/*
 * qv_oracle.c -- plain, slow CPU oracle for the W8A8 quantized verify pass.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * CPU-baseline leg of the benchmark load this library. The product path (the
 * CUDA library under quantized_verification_gb300/csrc) never links, loads or
 * calls it, and this file includes nothing from there.
 *
 * What it computes, and where the pages say so
 * (all pages summarise "Quasar: Quantized Self-Speculative Acceleration for
 * Rapid Inference via Memory-Efficient Verification"; pages are named by
 * site and language):
 *
 *   a0  per-output-channel symmetric int8 weight quantization
 *       -- gist.science/ja summary, section 2.2 "Enhanced SmoothQuant",
 *          item 2 (offline preparation: weights quantized to INT8);
 *          gist.science/it summary, section 2 "Pipeline di Esecuzione".
 *   a1  dynamic per-token symmetric int8 activation quantization, after an
 *       optional per-input-channel smoothing multiply
 *       -- gist.science/ja summary, section 2.2 item 3 (online inference:
 *          scale the BF16 input by the smoothing factor, convert to INT8);
 *          gist.science/de summary, section 2 "Methodik", "Online-Prozess";
 *          the smoothing identity Y = (W diag(s)^-1)(diag(s) X) of the
 *          gist.science/ja summary, section 2.2 item 1.
 *   a2  INT8 GEMM with exact INT32 accumulation, then dequantization back to
 *       high precision before any non-linear layer
 *       -- gist.science/ja summary, section 2.2 item 3;
 *          gist.science/fr summary, section 2 "Pipeline Technique".
 *   a3  greedy (T=0) verify token = argmax over the dequantized vocabulary
 *       logits, which stay in high precision for the acceptance test
 *       -- gist.science/it summary, section 2 item 3 ("Campionamento di
 *          Rifiuto Lossless"); greedy setting, gist.science/ja summary,
 *          section 4 "main results".
 *   f1  the non-linear steps between the quantized linears of one decoder
 *       layer, run in high precision after dequantization (residual add,
 *       RMSNorm, SiLU(gate) * up), each followed by the a1 quantization of
 *       the next linear's input
 *       -- gist.science/ja summary, section 2.2 item 3 (dequantize back to
 *          high precision before the non-linear layers);
 *          gist.science/fr summary, section 2 "Pipeline Technique".
 *   f2  lossless rejection sampling at temperature T > 0: draft token d_j is
 *       kept with probability min(1, p_j(d_j) / q_j(d_j)); at the first
 *       rejection a token is drawn from the normalized max(0, p_j - q_j); when
 *       every draft is kept, the bonus token is drawn from p_gamma
 *       -- gist.science/it summary, section 2 item 3 ("Campionamento di
 *          Rifiuto Lossless": the verifier's logits stay precise so that
 *          the target distribution is kept).
 *   f3  tree verification at T = 0: the drafts form a tree; the verifier's
 *       greedy tokens are computed for every node at once, and the deepest
 *       root path whose every drafted token equals the verifier's token after
 *       its parent is accepted, plus the verifier's token after its last node
 *       -- tree-structured verification named as an extension by the
 *          summaries (gist.science/de and gist.science/ja summaries,
 *          section 5); the acceptance rule is a4's applied along each path.
 *   f1' attention over a short KV cache: for each verify token, grouped-query
 *       scaled dot-product attention over the sequence's cached keys and
 *       values and the step's own new ones up to and including itself
 *       (causal) -- the decoder layer that the verify pass runs between the
 *       quantized linears (gist.science/ja summary, section 2.2 item 3:
 *       high-precision computation outside the INT8 GEMMs); the summaries
 *       do not spell attention out, so this is the textbook form.
 *   f3' logit fidelity (diagnostic): KL(p || q) between the softmax of a
 *       reference verifier's logits (p) and of the quantized verifier's (q),
 *       and whether their top-1 tokens agree -- the summaries report that
 *       quantization keeps the logit distribution (negligible KL divergence;
 *       gist.science/fr summary, contributions item 3) and that the
 *       quantized verifier keeps a high logit-distribution similarity
 *       (shd-paper.top summary, method details, core idea).
 *   f4  a lower-bit verifier, W4A8: int4 weights against the a1 int8
 *       activations, accumulated exactly in integers and dequantized as in a2
 *       -- lower bit widths (4-bit, 2-bit) named as the next step by the
 *          summaries (gist.science/it, gist.science/de and gist.science/ja
 *          summaries, section 5), INT4 among the bit widths the authors
 *          tried (shd-paper.top summary, method details, key design).
 *   a4  acceptance: the longest draft prefix equal to the verifier's tokens,
 *       plus one token from the verifier (so at least one token per step)
 *       -- gist.science/fr summary, lay explanation (a wrong guess is
 *          rejected and generation restarts from there); acceptance length
 *          L >= 1 implied by L ~ 1.03 for the pruned verifier,
 *          gist.science/ja summary, section 4.
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes of the repository):
 *   - scale s = fl32(amax / 127) by IEEE division; q = rne(fl32(x / s)),
 *     i.e. division by s, then round-half-to-even, then clamp to [-127, 127];
 *     -128 is never produced.
 *   - a row whose scale is 0 (all zeros, or amax/127 underflows) gets q = 0
 *     and s = 0.
 *   - smoothing: x' = fl32(x * c[k]) before amax; c == NULL is the identity.
 *   - dequant: y = fl32( fl32((float)acc) * fl32(sx * sw) ), every operation
 *     rounded to nearest-even, no fused multiply-add.
 *   - argmax ties go to the lowest index; -0 compares equal to +0.
 *   - f1 (the layer is not spelled out by the summaries; the readings follow
 *     the Qwen3-shaped decoder layer of the workloads, with a bf16 residual
 *     stream):
 *       residual add  h = rne_bf16(h + d), d the bf16 output of a linear;
 *       RMSNorm       ss = sum of h_k^2 in binary64 (every bf16 square is
 *                     exact there), var = fl32(ss / H),
 *                     rstd = fl32(1 / fl32(sqrt(fl32(var + eps)))),
 *                     x_k = rne_bf16(g_k * rne_bf16(fl32(h_k * rstd)));
 *       SwiGLU        a_k = fl32(fl32(gate_k * sigma(gate_k)) * up_k) on the
 *                     fp32 gate|up outputs, sigma(v) = fl32(1 / fl32(1 + E(-v)))
 *                     with E the exp defined at qvo_exp (Cody-Waite reduction
 *                     and a Taylor polynomial, written out so that the GPU side
 *                     can evaluate the identical binary32 operations);
 *     then the a1 quantization of x (bf16) or a (fp32).
 *   - f2 (the summaries name the rule, not its arithmetic): probabilities
 *     become integer weights so that every sum over the vocabulary is exact:
 *       p: m = max_v z_v, w_v = floor(E(fl32(fl32(z_v - m) / T)) * 2^24),
 *          Z = sum w_v;     q: c_v = floor(fl32(clamp(q_v, 0, 1) * 2^24)),
 *          Q = sum c_v;
 *       keep d iff u * (w_d / Z) / (c_d / Q) ... i.e. u24 * Z * c_d <
 *       w_d * Q * 2^24 (128-bit integers), u24 the top 24 bits of one draw;
 *       the replacement at the first rejection k: weights
 *       r_v = max(0, w_v * Q - c_v * Z) (128-bit), or w when R = sum r = 0;
 *       the bonus (no rejection): weights w of row gamma; a draw from
 *       weights x with total X is the smallest v whose prefix sum exceeds
 *       floor(u24' * X / 2^24), u24' from a second draw.
 *     Draws: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 *     pseudorandom number generators", 2014) used as a counter-based
 *     generator: draw n of seed s is mix(s + (n + 1) * 0x9E3779B97F4A7C15);
 *     n = 2 * row + purpose (0: keep test, 1: sample), row = b * (gamma + 1) + j.
 *   - f4 (no int4 format is given): per-output-channel symmetric int4, the
 *     a0 rule with 7 in place of 127: s = fl32(amax / 7),
 *     q = clamp(rne(fl32(w / s)), -7, 7), q = 0 when s = 0; two codes per
 *     byte, code k even in the low nibble and k + 1 in the high nibble, each
 *     a 4-bit two's complement (so -8 is never produced); the integer sums
 *     and the dequantization are a2's.
 *   - acceptance: row j of sequence b holds the verifier token t[b][j] that
 *     follows prefix position j; draft d[b][j] is accepted iff it equals
 *     t[b][j] and all earlier drafts were accepted; the verifier token at the
 *     first mismatch (or after the last draft) is always emitted.
 *
 * Floating point: every fp32 operation is a single IEEE binary32 operation
 * in round-to-nearest-even. The library must be compiled with
 * -ffp-contract=off and without -ffast-math (the build script does so).
 * These choices are also the ones that decide integers (quantized codes,
 * argmax), so they are taken in fp32, the precision the GPU path uses.
 * The unquantized comparator reference (qvo_linear_f64) is fp64.
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32                                                        */
/* ------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of a binary32 pattern: widening is exact. */
float qvo_bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Narrow binary32 to bf16 rounding to nearest, ties to even, on the 16
 * discarded bits. NaN inputs are outside the contract. */
uint16_t qvo_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

void qvo_bf16_to_f32_array(const uint16_t* h, float* f, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) f[i] = qvo_bf16_to_f32(h[i]);
}

void qvo_f32_to_bf16_array(const float* f, uint16_t* h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = qvo_f32_to_bf16_rne(f[i]);
}

/* ------------------------------------------------------------------ */
/* a0 / a1: symmetric per-row int8 quantization                         */
/* ------------------------------------------------------------------ */

/* Round a binary32 value to the nearest integer, ties to even. Written out
 * with floor so that it does not depend on the FPU rounding mode. */
static float round_half_even(float v)
{
    float f = floorf(v);
    float diff = v - f;            /* exact: v and f are within one unit */
    if (diff > 0.5f) return f + 1.0f;
    if (diff < 0.5f) return f;
    /* exact tie: pick the even neighbour */
    return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

/*
 * Quantize `rows` rows of length K, one scale per row.
 *   x    : rows*K binary32 values, row-major
 *   mul  : K per-column multipliers (smoothing), or NULL for the identity
 *   q    : rows*K int8 codes out
 *   s    : rows scales out
 * The same routine serves weights (one row per output channel, mul = NULL)
 * and activations (one row per token).
 */
void qvo_quantize_rows_f32(const float* x, int64_t rows, int64_t K,
                           const float* mul, int8_t* q, float* s)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * K;
        /* amax over the (optionally smoothed) row */
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = mul ? xr[k] * mul[k] : xr[k];
            float a = fabsf(v);
            if (a > amax) amax = a;
        }
        float scale = amax / 127.0f;
        s[r] = scale;
        for (int64_t k = 0; k < K; ++k) {
            if (scale == 0.0f) { q[r * K + k] = 0; continue; }
            float v = mul ? xr[k] * mul[k] : xr[k];
            float t = round_half_even(v / scale);
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            q[r * K + k] = (int8_t)t;
        }
    }
}

/* Same as above for bf16 input: each element is widened exactly first. */
void qvo_quantize_rows_bf16(const uint16_t* x, int64_t rows, int64_t K,
                            const float* mul, int8_t* q, float* s)
{
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = qvo_bf16_to_f32(x[r * K + k]);
            if (mul) v = v * mul[k];
            float a = fabsf(v);
            if (a > amax) amax = a;
        }
        float scale = amax / 127.0f;
        s[r] = scale;
        for (int64_t k = 0; k < K; ++k) {
            if (scale == 0.0f) { q[r * K + k] = 0; continue; }
            float v = qvo_bf16_to_f32(x[r * K + k]);
            if (mul) v = v * mul[k];
            float t = round_half_even(v / scale);
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            q[r * K + k] = (int8_t)t;
        }
    }
}

/* ------------------------------------------------------------------ */
/* a2: int8 x int8 -> exact integer sums, then dequantization            */
/* ------------------------------------------------------------------ */

/*
 * acc[m][n] = sum_k xq[m][k] * wq[n][k], the exact integer sum.
 * Summed in int64; returns the number of sums that do not fit int32 (0 for
 * every K the library accepts), and stores the low 32 bits regardless.
 */
int64_t qvo_int8_matmul(const int8_t* xq, const int8_t* wq,
                        int64_t M, int64_t N, int64_t K, int32_t* acc)
{
    int64_t overflow = 0;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t sum = 0;
            const int8_t* a = xq + m * K;
            const int8_t* b = wq + n * K;
            for (int64_t k = 0; k < K; ++k)
                sum += (int64_t)a[k] * (int64_t)b[k];
            if (sum > INT32_MAX || sum < INT32_MIN) ++overflow;
            acc[m * N + n] = (int32_t)sum;
        }
    }
    return overflow;
}

/* y = fl32( fl32((float)acc) * fl32(sx[m] * sw[n]) ). */
float qvo_dequant_one(int32_t acc, float sx, float sw)
{
    float a = (float)acc;          /* int -> float, round to nearest even */
    float scale = sx * sw;
    return a * scale;
}

void qvo_dequant(const int32_t* acc, const float* sx, const float* sw,
                 int64_t M, int64_t N, float* y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            y[m * N + n] = qvo_dequant_one(acc[m * N + n], sx[m], sw[n]);
}

/* ------------------------------------------------------------------ */
/* a3: greedy argmax over each row                                      */
/* ------------------------------------------------------------------ */

/* tok[m] = lowest index of the maximum of y[m][:]; maxv[m] that maximum.
 * Comparison is the plain float '>' so -0 == +0 and the first index wins. */
void qvo_argmax_rows(const float* y, int64_t M, int64_t N,
                     int32_t* tok, float* maxv)
{
    for (int64_t m = 0; m < M; ++m) {
        int64_t best = 0;
        float bv = y[m * N];
        for (int64_t n = 1; n < N; ++n) {
            if (y[m * N + n] > bv) { bv = y[m * N + n]; best = n; }
        }
        tok[m] = (int32_t)best;
        if (maxv) maxv[m] = bv;
    }
}

/* LM head: logits are formed one at a time with the a2 arithmetic and
 * reduced on the fly, never stored. Same result as dequant + argmax. */
void qvo_lm_head_argmax(const int8_t* xq, const float* sx,
                        const int8_t* wq, const float* sw,
                        int64_t M, int64_t V, int64_t K,
                        int32_t* tok, float* maxv)
{
    for (int64_t m = 0; m < M; ++m) {
        int64_t best = -1;
        float bv = 0.0f;
        for (int64_t v = 0; v < V; ++v) {
            int64_t sum = 0;
            for (int64_t k = 0; k < K; ++k)
                sum += (int64_t)xq[m * K + k] * (int64_t)wq[v * K + k];
            float y = qvo_dequant_one((int32_t)sum, sx[m], sw[v]);
            if (best < 0 || y > bv) { bv = y; best = v; }
        }
        tok[m] = (int32_t)best;
        if (maxv) maxv[m] = bv;
    }
}

/* ------------------------------------------------------------------ */
/* a4: greedy acceptance                                                 */
/* ------------------------------------------------------------------ */

/*
 * t   : B*(gamma+1) verifier tokens; row j of sequence b is t[b*(gamma+1)+j]
 * d   : B*gamma draft tokens; d[b*gamma+j] is the (j+1)-th drafted token
 * len : B accepted lengths, in [1, gamma+1]
 * out : B*(gamma+1) emitted tokens, t[b][0..len-1], then -1
 */
void qvo_accept(const int32_t* t, const int32_t* d, int64_t B, int64_t gamma,
                int32_t* len, int32_t* out)
{
    int64_t G = gamma + 1;
    for (int64_t b = 0; b < B; ++b) {
        int64_t k = 0;
        while (k < gamma && d[b * gamma + k] == t[b * G + k]) ++k;
        len[b] = (int32_t)(k + 1);
        for (int64_t j = 0; j < G; ++j)
            out[b * G + j] = (j <= k) ? t[b * G + j] : -1;
    }
}

/* ------------------------------------------------------------------ */
/* Unquantized reference for the BF16-weight comparator                 */
/* ------------------------------------------------------------------ */

/* y[m][n] = sum_k x[m][k] * w[n][k] in binary64 (inputs are binary32, which
 * holds every bf16 value exactly). */
void qvo_linear_f64(const float* x, const float* w, int64_t M, int64_t N,
                    int64_t K, double* y)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k)
                sum += (double)x[m * K + k] * (double)w[n * K + k];
            y[m * N + n] = sum;
        }
}

/* ------------------------------------------------------------------ */
/* f1: the non-linear steps between the quantized linears of a layer    */
/* ------------------------------------------------------------------ */

/*
 * exp(x) in binary32 by Cody and Waite's additive range reduction and a
 * Taylor polynomial (W. J. Cody, W. Waite, "Software Manual for the
 * Elementary Functions", 1980), each step one binary32 operation in
 * round-to-nearest-even:
 *   x > 88        -> +inf;   x < -87 -> 0
 *   k = rne(fl(x * LOG2E))                     (an integer, |k| <= 127)
 *   r = fl(fl(x - fl(k * LN2_HI)) - fl(k * LN2_LO)),   |r| <= ~0.347
 *   p = 1 + r(1 + r(c2 + r(c3 + r(c4 + r(c5 + r(c6 + r c7))))))  (Horner,
 *       c_n = fl(1 / n!), one multiply and one add per step)
 *   E = fl(p * 2^k)                            (2^k built from its exponent bits)
 * LN2_HI = 0.693145751953125 has 16 significant bits, so k * LN2_HI is exact;
 * LN2_LO = fl(ln 2 - LN2_HI). The degree-7 truncation is below 6e-9 relative
 * on |r| <= ln 2 / 2.
 */
static const float QVO_LOG2E = 1.44269504088896341f;
static const float QVO_LN2_HI = 0.693145751953125f;
static const float QVO_LN2_LO = 1.42860682030941723212e-6f;

float qvo_exp(float x)
{
    if (x > 88.0f) return INFINITY;
    if (x < -87.0f) return 0.0f;
    float k = round_half_even(x * QVO_LOG2E);
    float r = x - k * QVO_LN2_HI;
    r = r - k * QVO_LN2_LO;
    const float c[8] = {1.0f, 1.0f, 0.5f, 1.0f / 6.0f, 1.0f / 24.0f, 1.0f / 120.0f,
                        1.0f / 720.0f, 1.0f / 5040.0f};
    float p = c[7];
    for (int n = 6; n >= 0; --n) {
        p = p * r;
        p = p + c[n];
    }
    union { uint32_t u; float f; } two_k;
    two_k.u = (uint32_t)((int32_t)k + 127) << 23;
    return p * two_k.f;
}

/* sigma(v) = fl32(1 / fl32(1 + E(-v))), silu(v) = fl32(v * sigma(v)). */
float qvo_silu(float v)
{
    float e = qvo_exp(-v);
    float den = 1.0f + e;
    float sig = 1.0f / den;
    return v * sig;
}

/*
 * SwiGLU then a1: gu is M rows of 2F fp32 values, gate in columns [0, F),
 * up in [F, 2F) (the concatenated gate|up linear's output).
 *   a_k = fl32(silu(gate_k) * up_k); q, s = the per-row quantization of a.
 */
void qvo_swiglu_quant(const float* gu, int64_t M, int64_t F, int8_t* q, float* s)
{
    float* a = (float*)malloc((size_t)F * sizeof(float));
    for (int64_t m = 0; m < M; ++m) {
        const float* row = gu + m * 2 * F;
        for (int64_t k = 0; k < F; ++k) a[k] = qvo_silu(row[k]) * row[F + k];
        qvo_quantize_rows_f32(a, 1, F, NULL, q + m * F, s + m);
    }
    free(a);
}

/*
 * Residual add, RMSNorm, then a1. h: M rows of H bf16 values, updated in
 * place when d (M x H bf16, the delta) is given; g: H bf16 norm weights;
 * mul: the a1 smoothing multipliers or NULL.
 *   h_k   = rne_bf16(fl32(h_k + d_k))
 *   ss    = sum_k h_k^2 in binary64, var = fl32(ss / H)
 *   rstd  = fl32(1 / fl32(sqrt(fl32(var + eps))))
 *   x_k   = rne_bf16(fl32(g_k * rne_bf16(fl32(h_k * rstd))))
 *   q, s  = the per-row quantization of x (bf16), after mul.
 * x_out (M x H bf16) receives x when not NULL.
 */
void qvo_residual_rmsnorm_quant(uint16_t* h, const uint16_t* d, const uint16_t* g, float eps,
                                const float* mul, int64_t M, int64_t H, int8_t* q, float* s,
                                uint16_t* x_out)
{
    uint16_t* x = (uint16_t*)malloc((size_t)H * sizeof(uint16_t));
    for (int64_t m = 0; m < M; ++m) {
        uint16_t* hr = h + m * H;
        if (d) {
            for (int64_t k = 0; k < H; ++k)
                hr[k] = qvo_f32_to_bf16_rne(qvo_bf16_to_f32(hr[k]) + qvo_bf16_to_f32(d[m * H + k]));
        }
        double ss = 0.0;
        for (int64_t k = 0; k < H; ++k) {
            double v = (double)qvo_bf16_to_f32(hr[k]);
            ss += v * v;
        }
        float var = (float)(ss / (double)H);
        float t = var + eps;
        float sq = sqrtf(t);
        float rstd = 1.0f / sq;
        for (int64_t k = 0; k < H; ++k) {
            float u = qvo_bf16_to_f32(qvo_f32_to_bf16_rne(qvo_bf16_to_f32(hr[k]) * rstd));
            x[k] = qvo_f32_to_bf16_rne(qvo_bf16_to_f32(g[k]) * u);
        }
        if (x_out) memcpy(x_out + m * H, x, (size_t)H * sizeof(uint16_t));
        qvo_quantize_rows_bf16(x, 1, H, mul, q + m * H, s + m);
    }
    free(x);
}

/* ------------------------------------------------------------------ */
/* f2: lossless rejection sampling at T > 0                             */
/* ------------------------------------------------------------------ */

typedef unsigned __int128 u128;

/* SplitMix64 output n of the sequence seeded with s (counter-based form). */
uint64_t qvo_splitmix64(uint64_t s, uint64_t n)
{
    uint64_t z = s + (n + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Integer weight floor(x * 2^24) of a value x in [0, 1] (clamped). */
static uint32_t weight24(float x)
{
    if (!(x > 0.0f)) return 0u;
    if (x >= 1.0f) return 1u << 24;
    return (uint32_t)(x * 16777216.0f);     /* exact product, truncated */
}

/* p weights of one logits row: w_v = floor(E((z_v - m) / T) * 2^24). */
static uint64_t p_weights(const float* z, int64_t V, float T, uint32_t* w)
{
    float m = z[0];
    for (int64_t v = 1; v < V; ++v)
        if (z[v] > m) m = z[v];
    uint64_t Z = 0;
    for (int64_t v = 0; v < V; ++v) {
        float t = (z[v] - m) / T;
        w[v] = weight24(qvo_exp(t));
        Z += w[v];
    }
    return Z;
}

/* Smallest v whose prefix sum of x exceeds floor(u24 * X / 2^24). */
static int32_t draw_u64(const uint64_t* x, int64_t V, uint64_t X, uint32_t u24)
{
    u128 target = ((u128)u24 * (u128)X) >> 24;
    u128 acc = 0;
    for (int64_t v = 0; v < V; ++v) {
        acc += x[v];
        if (acc > target) return (int32_t)v;
    }
    return (int32_t)(V - 1);
}
static int32_t draw_u128(const u128* x, int64_t V, u128 X, uint32_t u24)
{
    /* floor(u24 * X / 2^24) without overflow: X < 2^106 here */
    u128 target = (X >> 24) * u24 + (((X & 0xFFFFFFull) * u24) >> 24);
    u128 acc = 0;
    for (int64_t v = 0; v < V; ++v) {
        acc += x[v];
        if (acc > target) return (int32_t)v;
    }
    return (int32_t)(V - 1);
}

/* The draw of qvo_spec_sample from integer weights x (total X), exported
 * for the tests. */
int32_t qvo_draw_index(const uint64_t* x, int64_t V, uint64_t X, uint32_t u24)
{
    return draw_u64(x, V, X, u24);
}

/*
 * Speculative sampling for B sequences of gamma drafts.
 *   z   : M = B*(gamma+1) rows of V fp32 verifier logits (row b*(gamma+1)+j
 *         follows prefix position j)
 *   d   : B*gamma draft tokens; q: B*gamma rows of V draft probabilities
 *   len : B accepted lengths (kept drafts + 1); out: B*(gamma+1) tokens,
 *         the kept drafts, then the replacement or bonus token, then -1
 */
void qvo_spec_sample(const float* z, const int32_t* d, const float* q, int64_t B, int64_t gamma,
                     int64_t V, float T, uint64_t seed, int32_t* len, int32_t* out)
{
    int64_t G = gamma + 1;
    uint32_t* w = (uint32_t*)malloc((size_t)V * sizeof(uint32_t));
    uint32_t* c = (uint32_t*)malloc((size_t)V * sizeof(uint32_t));
    uint64_t* x64 = (uint64_t*)malloc((size_t)V * sizeof(uint64_t));
    u128* x128 = (u128*)malloc((size_t)V * sizeof(u128));
    for (int64_t b = 0; b < B; ++b) {
        int64_t k = 0;
        int32_t tok = -1;
        for (; k < gamma; ++k) {
            int64_t row = b * G + k;
            uint64_t Z = p_weights(z + row * V, V, T, w);
            uint64_t Q = 0;
            for (int64_t v = 0; v < V; ++v) { c[v] = weight24(q[(b * gamma + k) * V + v]); Q += c[v]; }
            int32_t dk = d[b * gamma + k];
            uint32_t u24 = (uint32_t)(qvo_splitmix64(seed, (uint64_t)(2 * row)) >> 40);
            u128 lhs = (u128)u24 * (u128)Z * (u128)c[dk];
            u128 rhs = ((u128)w[dk] * (u128)Q) << 24;
            if (lhs < rhs) continue;                         /* kept */
            /* rejected: draw from max(0, w*Q - c*Z), or from w if that is all 0 */
            u128 R = 0;
            for (int64_t v = 0; v < V; ++v) {
                u128 a1 = (u128)w[v] * Q, a2 = (u128)c[v] * Z;
                x128[v] = a1 > a2 ? a1 - a2 : 0;
                R += x128[v];
            }
            uint32_t u2 = (uint32_t)(qvo_splitmix64(seed, (uint64_t)(2 * row + 1)) >> 40);
            if (R > 0) {
                tok = draw_u128(x128, V, R, u2);
            } else {
                for (int64_t v = 0; v < V; ++v) x64[v] = w[v];
                tok = draw_u64(x64, V, Z, u2);
            }
            break;
        }
        if (k == gamma) {                                    /* every draft kept: the bonus */
            int64_t row = b * G + gamma;
            uint64_t Z = p_weights(z + row * V, V, T, w);
            for (int64_t v = 0; v < V; ++v) x64[v] = w[v];
            uint32_t u2 = (uint32_t)(qvo_splitmix64(seed, (uint64_t)(2 * row + 1)) >> 40);
            tok = draw_u64(x64, V, Z, u2);
        }
        len[b] = (int32_t)(k + 1);
        for (int64_t j = 0; j < G; ++j)
            out[b * G + j] = j < k ? d[b * gamma + j] : (j == k ? tok : -1);
    }
    free(w); free(c); free(x64); free(x128);
}

/* ------------------------------------------------------------------ */
/* f3: tree verification at T = 0                                      */
/* ------------------------------------------------------------------ */

/*
 * B trees of N nodes. Node 0 of tree b is its root (the last accepted
 * position); node i >= 1 has parent par[b*N+i] (valid when in [0, i)) and
 * drafted token d[b*N+i]; t[b*N+i] is the verifier's greedy token after the
 * root path of node i.
 *   accepted(0) = true; accepted(i) = par in [0, i) and accepted(par) and
 *   d[i] == t[par]; depth(0) = 0, depth(i) = depth(par) + 1.
 *   best = the accepted node of largest depth, the lowest index among them.
 *   len[b] = depth(best) + 1; out[b][0 .. depth-1] = the drafted tokens on
 *   the path root -> best (root excluded), out[b][depth] = t[best], then -1
 *   (out has N entries per tree); node[b] = best.
 */
void qvo_tree_accept(const int32_t* t, const int32_t* d, const int32_t* par, int64_t B, int64_t N,
                     int32_t* len, int32_t* out, int32_t* node)
{
    int32_t* depth = (int32_t*)malloc((size_t)N * sizeof(int32_t));
    uint8_t* acc = (uint8_t*)malloc((size_t)N);
    for (int64_t b = 0; b < B; ++b) {
        const int32_t* tb = t + b * N;
        const int32_t* db = d + b * N;
        const int32_t* pb = par + b * N;
        acc[0] = 1;
        depth[0] = 0;
        int64_t best = 0;
        for (int64_t i = 1; i < N; ++i) {
            int32_t p = pb[i];
            acc[i] = (p >= 0 && p < i && acc[p] && db[i] == tb[p]) ? 1 : 0;
            depth[i] = (p >= 0 && p < i) ? depth[p] + 1 : 0;
            if (acc[i] && depth[i] > depth[best]) best = i;
        }
        int32_t D = depth[best];
        len[b] = D + 1;
        for (int64_t j = 0; j < N; ++j) out[b * N + j] = -1;
        out[b * N + D] = tb[best];
        int64_t i = best;
        for (int32_t k = D - 1; k >= 0; --k) {
            out[b * N + k] = db[i];
            i = pb[i];
        }
        if (node) node[b] = (int32_t)best;
    }
    free(depth);
    free(acc);
}

/* ------------------------------------------------------------------ */
/* f4: W4A8, int4 weights                                               */
/* ------------------------------------------------------------------ */

/* Per-row symmetric int4 quantization of weights: the a0 rule with the
 * code range [-7, 7]. x is rows*K binary32 values (bf16 callers widen
 * first); q gets one code per int8. */
void qvo_quantize_rows_w4_f32(const float* x, int64_t rows, int64_t K, int8_t* q, float* s)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float* xr = x + r * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(xr[k]);
            if (a > amax) amax = a;
        }
        float scale = amax / 7.0f;
        s[r] = scale;
        for (int64_t k = 0; k < K; ++k) {
            if (scale == 0.0f) { q[r * K + k] = 0; continue; }
            float t = round_half_even(xr[k] / scale);
            if (t > 7.0f) t = 7.0f;
            if (t < -7.0f) t = -7.0f;
            q[r * K + k] = (int8_t)t;
        }
    }
}

/* Two codes per byte: byte j of a row holds code 2j in bits 0-3 and code
 * 2j+1 in bits 4-7, each as 4-bit two's complement. K is even. */
void qvo_pack_w4(const int8_t* q, int64_t rows, int64_t K, uint8_t* packed)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < K / 2; ++j) {
            unsigned lo = (unsigned)(uint8_t)q[r * K + 2 * j] & 0xFu;
            unsigned hi = (unsigned)(uint8_t)q[r * K + 2 * j + 1] & 0xFu;
            packed[r * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
}

static int8_t nibble_value(unsigned n)
{
    return (int8_t)(n >= 8u ? (int)n - 16 : (int)n);
}

void qvo_unpack_w4(const uint8_t* packed, int64_t rows, int64_t K, int8_t* q)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < K / 2; ++j) {
            unsigned byte = packed[r * (K / 2) + j];
            q[r * K + 2 * j] = nibble_value(byte & 0xFu);
            q[r * K + 2 * j + 1] = nibble_value(byte >> 4);
        }
}

/* ------------------------------------------------------------------ */
/* f3': logit fidelity, in binary64                                     */
/* ------------------------------------------------------------------ */

/* For each row m: p = softmax(a[m]), q = softmax(b[m]) (natural base),
 * kl[m] = sum_v p_v (log p_v - log q_v), written out as the definition with
 * log p_v = a_v - max a - log sum exp(a - max a) (likewise q), in binary64;
 * ta[m], tb[m] = the first index of the maximum of a[m], b[m]. */
void qvo_logit_fidelity(const float* a, const float* b, int64_t M, int64_t V,
                        double* kl, int32_t* ta, int32_t* tb)
{
    for (int64_t m = 0; m < M; ++m) {
        const float* ar = a + m * V;
        const float* br = b + m * V;
        int64_t ia = 0, ib = 0;
        for (int64_t v = 1; v < V; ++v) {
            if (ar[v] > ar[ia]) ia = v;
            if (br[v] > br[ib]) ib = v;
        }
        const double ma = ar[ia], mb = br[ib];
        double za = 0.0, zb = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            za += exp((double)ar[v] - ma);
            zb += exp((double)br[v] - mb);
        }
        const double lza = log(za), lzb = log(zb);
        double s = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            const double lp = (double)ar[v] - ma - lza;
            const double lq = (double)br[v] - mb - lzb;
            s += exp(lp) * (lp - lq);
        }
        kl[m] = s;
        ta[m] = (int32_t)ia;
        tb[m] = (int32_t)ib;
    }
}

/* ------------------------------------------------------------------ */
/* f1': attention over a short KV cache, in binary64                     */
/* ------------------------------------------------------------------ */

/*
 * B sequences, each with T = gamma + 1 verify tokens. qkv holds, per token
 * row m = b*T + j, the bf16 outputs of the qkv projection: Hq query heads,
 * then Hkv key heads, then Hkv value heads, D values each (row stride
 * (Hq + 2 Hkv) D). kc, vc: bf16 caches [B][Lmax][Hkv][D]; len[b] cached
 * positions of sequence b. Query head h uses key/value head h / (Hq/Hkv).
 * Token j of sequence b attends to the len[b] cached positions and to the
 * step's tokens 0..j:
 *   s_i = scale * sum_d q[d] k_i[d],  w_i = e^(s_i - max s) / sum e^(...),
 *   out[m][h*D + d] = sum_i w_i v_i[d]     (binary64 throughout).
 */
void qvo_attention_verify(const uint16_t* qkv, const uint16_t* kc, const uint16_t* vc,
                          const int32_t* len, int64_t B, int64_t T, int64_t Hq, int64_t Hkv,
                          int64_t D, int64_t Lmax, double scale, double* out)
{
    const int64_t G = Hq / Hkv, W = (Hq + 2 * Hkv) * D;
    double* s = (double*)malloc((size_t)(Lmax + T) * sizeof(double));
    for (int64_t b = 0; b < B; ++b) {
        const int64_t L = len[b];
        for (int64_t j = 0; j < T; ++j) {
            const uint16_t* row = qkv + (b * T + j) * W;
            for (int64_t h = 0; h < Hq; ++h) {
                const int64_t kh = h / G;
                const uint16_t* q = row + h * D;
                const int64_t n = L + j + 1;
                double mx = -INFINITY;
                for (int64_t i = 0; i < n; ++i) {
                    const uint16_t* k = i < L ? kc + ((b * Lmax + i) * Hkv + kh) * D
                                              : qkv + (b * T + (i - L)) * W + (Hq + kh) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += (double)qvo_bf16_to_f32(q[d]) * (double)qvo_bf16_to_f32(k[d]);
                    s[i] = scale * dot;
                    if (s[i] > mx) mx = s[i];
                }
                double z = 0.0;
                for (int64_t i = 0; i < n; ++i) {
                    s[i] = exp(s[i] - mx);
                    z += s[i];
                }
                for (int64_t d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < n; ++i) {
                        const uint16_t* v = i < L ? vc + ((b * Lmax + i) * Hkv + kh) * D
                                                  : qkv + (b * T + (i - L)) * W + (Hq + Hkv + kh) * D;
                        acc += s[i] * (double)qvo_bf16_to_f32(v[d]);
                    }
                    out[(b * T + j) * Hq * D + h * D + d] = acc / z;
                }
            }
        }
    }
    free(s);
}
