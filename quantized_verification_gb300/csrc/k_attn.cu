// k_attn.cu -- attention over a short KV cache for the verify tokens.
//
//   The decoder layer that the verify pass runs between the quantized
//   linears (Quasar, gist.science/ja summary, section 2.2 item 3: the
//   non-GEMM computation stays in high precision). The summaries do not
//   spell attention out; this is causal grouped-query scaled dot-product
//   attention: token j of a sequence attends to the sequence's cached
//   positions and to the step's tokens 0..j; query head h reads key/value
//   head h / (Hq / Hkv).
//
// Inputs are the qkv projection's bf16 output rows (Hq query heads, then Hkv
// key heads, then Hkv value heads, D values each) and bf16 caches
// [B][Lmax][Hkv][D]. Split-KV in two kernels:
//   attn_chunk_kernel    one CTA per (128-key chunk, key/value head,
//                        sequence) for all R = T * G query rows of that head
//                        group: scores, the chunk's row max and sum of
//                        e^(s - max), and the unnormalised sum of e^(s - max) v;
//   attn_combine_kernel  one CTA per (head, sequence): merges the chunks
//                        (log-sum-exp) and writes fp32 outputs [token][Hq*D].
// Scores and sums are binary32 on CUDA cores: R <= 32 rows against a
// 128-key chunk is too small a contraction for the tensor cores to pay.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kAttnChunk = 128;            // keys per chunk CTA
constexpr int kAttnThreads = 256;          // 2 row groups x 128 keys (or dims)
constexpr int kAttnMaxRows = 32;           // R = T * G
constexpr int kAttnRowsPerGroup = kAttnMaxRows / 2;

struct AttnArgs {
    const uint16_t* qkv;     // [B*T][(Hq + 2 Hkv) * D] bf16
    const uint16_t* kc;      // [B][Lmax][Hkv][D] bf16
    const uint16_t* vc;
    const int32_t* len;      // [B]
    int T, Hq, Hkv, D, Lmax, nsplit;
    float scale;
    float* part;             // [B][Hkv][nsplit][R][D + 2]: o (D values), max, sum
    float* out;              // [B*T][Hq*D]
};

__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ int seq_len(const AttnArgs& a, int b) {
    const int L = a.len[b];
    return L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);          // out-of-range lengths are clamped
}

// Pointer to key (kv = 0) or value (kv = 1) row i of sequence b, head kh.
__device__ __forceinline__ const uint16_t* kv_row(const AttnArgs& a, int b, int L, int i, int kh, int kv) {
    if (i < L) return (kv ? a.vc : a.kc) + (((size_t)b * a.Lmax + i) * a.Hkv + kh) * a.D;
    const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * a.D;
    return a.qkv + ((size_t)b * a.T + (i - L)) * W + (size_t)(a.Hq + kv * a.Hkv + kh) * a.D;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_chunk_kernel(const AttnArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    extern __shared__ float4 attn_smem[];
    const int G = a.Hq / a.Hkv, R = a.T * G;
    float* qs = reinterpret_cast<float*>(attn_smem);         // [R][D]
    float* ps = qs + kAttnMaxRows * D;                       // [R][kAttnChunk]
    float* st = ps + kAttnMaxRows * kAttnChunk;              // max [R], sum [R]
    const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int L = seq_len(a, b), S = L + a.T;
    const int s0 = split * kAttnChunk;
    const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * D;
    float* part = a.part + ((((size_t)b * a.Hkv + kh) * a.nsplit + split) * R) * (D + 2);
    if (s0 >= S) {                                           // no key here: an empty partial
        for (int r = tid; r < R; r += kAttnThreads) {
            part[(size_t)r * (D + 2) + D] = -__uint_as_float(0x7F800000u);
            part[(size_t)r * (D + 2) + D + 1] = 0.f;
        }
        return;
    }
    // query rows r = j * G + g of heads kh * G + g
    for (int e = tid; e < R * D; e += kAttnThreads) {
        const int r = e / D, d = e - r * D, j = r / G, h = kh * G + (r - j * G);
        qs[e] = bf16f(a.qkv[((size_t)b * a.T + j) * W + (size_t)h * D + d]);
    }
    __syncthreads();

    // scores: thread (key t % 128, row group t / 128)
    {
        const int kl = tid % kAttnChunk, rg = tid / kAttnChunk, s = s0 + kl;
        const int r0 = rg * kAttnRowsPerGroup;
        float acc[kAttnRowsPerGroup];
#pragma unroll
        for (int q = 0; q < kAttnRowsPerGroup; ++q) acc[q] = 0.f;
        if (s < S) {
            const uint16_t* kp = kv_row(a, b, L, s, kh, 0);
#pragma unroll 1
            for (int d0 = 0; d0 < D; d0 += 8) {
                const uint4 raw = *reinterpret_cast<const uint4*>(kp + d0);
                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
                float kv8[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kv8[2 * i] = __uint_as_float(w4[i] << 16);
                    kv8[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u);
                }
#pragma unroll
                for (int q = 0; q < kAttnRowsPerGroup; ++q) {
                    if (r0 + q < R) {
                        const float4 qa = *reinterpret_cast<const float4*>(qs + (r0 + q) * D + d0);
                        const float4 qb = *reinterpret_cast<const float4*>(qs + (r0 + q) * D + d0 + 4);
                        acc[q] += qa.x * kv8[0] + qa.y * kv8[1] + qa.z * kv8[2] + qa.w * kv8[3] +
                                  qb.x * kv8[4] + qb.y * kv8[5] + qb.z * kv8[6] + qb.w * kv8[7];
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kAttnRowsPerGroup; ++q) {
            const int r = r0 + q;
            if (r < R) {
                const int j = r / G;
                const bool vis = s < S && s < L + j + 1;              // causal
                ps[r * kAttnChunk + kl] = vis ? acc[q] * a.scale : -__uint_as_float(0x7F800000u);
            }
        }
    }
    __syncthreads();

    // row statistics over the chunk: one warp per row
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r < R; r += kAttnThreads / 32) {
            float v[kAttnChunk / 32];
            float m = -__uint_as_float(0x7F800000u);
#pragma unroll
            for (int i = 0; i < kAttnChunk / 32; ++i) {
                v[i] = ps[r * kAttnChunk + lane + 32 * i];
                m = fmaxf(m, v[i]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            float l = 0.f;
#pragma unroll
            for (int i = 0; i < kAttnChunk / 32; ++i) {
                const float p = m == -__uint_as_float(0x7F800000u) ? 0.f : expf(v[i] - m);
                ps[r * kAttnChunk + lane + 32 * i] = p;
                l += p;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) {
                st[r] = m;
                st[kAttnMaxRows + r] = l;
            }
        }
    }
    __syncthreads();

    // unnormalised p . v: thread (dim t % 128, row group t / 128), D <= 128
    {
        const int d = tid % kAttnChunk, rg = tid / kAttnChunk, r0 = rg * kAttnRowsPerGroup;
        if (d < D) {
            float acc[kAttnRowsPerGroup];
#pragma unroll
            for (int q = 0; q < kAttnRowsPerGroup; ++q) acc[q] = 0.f;
            const int n = min(kAttnChunk, S - s0);
#pragma unroll 1
            for (int i0 = 0; i0 < n; i0 += 4) {
                float vv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) vv[u] = i0 + u < n ? bf16f(kv_row(a, b, L, s0 + i0 + u, kh, 1)[d]) : 0.f;
#pragma unroll
                for (int q = 0; q < kAttnRowsPerGroup; ++q) {
                    if (r0 + q < R) {
                        const float4 p = *reinterpret_cast<const float4*>(ps + (r0 + q) * kAttnChunk + i0);
                        acc[q] += p.x * vv[0] + p.y * vv[1] + p.z * vv[2] + p.w * vv[3];
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kAttnRowsPerGroup; ++q)
                if (r0 + q < R) part[(size_t)(r0 + q) * (D + 2) + d] = acc[q];
        }
        for (int r = tid; r < R; r += kAttnThreads) {
            part[(size_t)r * (D + 2) + D] = st[r];
            part[(size_t)r * (D + 2) + D + 1] = st[kAttnMaxRows + r];
        }
    }
}

// One CTA per (key/value head, sequence): for each of its R rows, merge the
// chunks: out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c.
template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const AttnArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    const int kh = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int G = a.Hq / a.Hkv, R = a.T * G;
    const int L = seq_len(a, b), S = L + a.T;
    const int n = (S + kAttnChunk - 1) / kAttnChunk;
    const float* base = a.part + (((size_t)b * a.Hkv + kh) * a.nsplit) * R * (D + 2);
    for (int r = 0; r < R; ++r) {
        float M = -__uint_as_float(0x7F800000u);
        for (int c = 0; c < n; ++c) M = fmaxf(M, base[((size_t)c * R + r) * (D + 2) + D]);
        float num = 0.f, den = 0.f;
        for (int c = 0; c < n; ++c) {
            const float* pr = base + ((size_t)c * R + r) * (D + 2);
            const float m = pr[D];
            if (m == -__uint_as_float(0x7F800000u)) continue;        // no visible key in this chunk
            const float w = expf(m - M);
            num += w * pr[d];
            den += w * pr[D + 1];
        }
        const int j = r / G, h = kh * G + (r - j * G);
        a.out[((size_t)b * a.T + j) * (size_t)a.Hq * D + (size_t)h * D + d] = num / den;
    }
}

template <class K>
cudaError_t launch_attn(K kernel, dim3 grid, int threads, size_t smem, const AttnArgs& args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

template <int D>
size_t attn_smem() {
    return (size_t)(kAttnMaxRows * D + kAttnMaxRows * kAttnChunk + 2 * kAttnMaxRows) * sizeof(float);
}

}  // namespace

int attention_splits(int Lmax, int T) { return (Lmax + T + kAttnChunk - 1) / kAttnChunk; }

size_t attention_workspace_bytes(int B, int T, int Hq, int Hkv, int D, int Lmax) {
    const size_t R = (size_t)T * (Hq / Hkv);
    return (size_t)B * Hkv * attention_splits(Lmax, T) * R * (D + 2) * sizeof(float);
}

cudaError_t launch_attention_verify(const uint16_t* qkv, const uint16_t* kc, const uint16_t* vc, const int32_t* len,
                                    int B, int T, int Hq, int Hkv, int D, int Lmax, float scale, float* out,
                                    void* ws, cudaStream_t s) {
    AttnArgs a;
    a.qkv = qkv; a.kc = kc; a.vc = vc; a.len = len;
    a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.Lmax = Lmax;
    a.nsplit = attention_splits(Lmax, T);
    a.scale = scale;
    a.part = static_cast<float*>(ws);
    a.out = out;
    const dim3 g1(a.nsplit, Hkv, B), g2(Hkv, B);
    // at most 33 KB of shared memory: no opt-in above the default 48 KB needed
    static_assert(kAttnMaxRows * 128 + kAttnMaxRows * kAttnChunk + 2 * kAttnMaxRows <= 48 * 1024 / 4, "smem");
    cudaError_t e;
    if (D == 128) {
        if ((e = launch_attn(attn_chunk_kernel<128>, g1, kAttnThreads, attn_smem<128>(), a, s)) != cudaSuccess) return e;
        return launch_attn(attn_combine_kernel<128>, g2, 128, 0, a, s);
    }
    if ((e = launch_attn(attn_chunk_kernel<64>, g1, kAttnThreads, attn_smem<64>(), a, s)) != cudaSuccess) return e;
    return launch_attn(attn_combine_kernel<64>, g2, 64, 0, a, s);
}

}  // namespace qv
