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
//   attn_chunk_kernel    one CTA per (64-key chunk, key/value head,
//                        sequence) for all R = T * G query rows of that head
//                        group: the chunk's keys are staged in shared memory
//                        with coalesced 16-byte loads (rows padded by 16
//                        bytes so that 16-byte reads of consecutive keys hit
//                        distinct banks), scores, the chunk's row max and
//                        sum of e^(s - max); then its values, staged in the
//                        same buffer, and the unnormalised sum of
//                        e^(s - max) v;
//   attn_combine_kernel  one CTA per (query row, key/value head, sequence):
//                        merges the chunks (log-sum-exp) and writes the fp32
//                        outputs [token][Hq*D].
// Scores and sums are binary32 on CUDA cores: R <= 32 rows against a
// 64-key chunk is too small a contraction for the tensor cores to pay, and
// the step reads each key and value once.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kAttnChunk = 64;             // keys per chunk CTA
constexpr int kAttnThreads = 256;
constexpr int kAttnMaxRows = 32;           // R = T * G

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

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ int seq_len(const AttnArgs& a, int b) {
    const int L = a.len[b];
    return L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);          // out-of-range lengths are clamped
}

// Key (kv = 0) or value (kv = 1) row i of sequence b, head kh.
__device__ __forceinline__ const uint16_t* kv_row(const AttnArgs& a, int b, int L, int i, int kh, int kv) {
    if (i < L) return (kv ? a.vc : a.kc) + (((size_t)b * a.Lmax + i) * a.Hkv + kh) * a.D;
    const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * a.D;
    return a.qkv + ((size_t)b * a.T + (i - L)) * W + (size_t)(a.Hq + kv * a.Hkv + kh) * a.D;
}

// Stage the chunk's n key or value rows into shared memory rows of D + 8
// bf16 (zeros past n).
template <int D>
__device__ __forceinline__ void stage_rows(const AttnArgs& a, int b, int L, int s0, int n, int kh, int kv,
                                           uint16_t* buf) {
    constexpr int P = D / 8;                                 // 16-byte pieces per row
    for (int e = threadIdx.x; e < kAttnChunk * P; e += kAttnThreads) {
        const int r = e / P, c = e - r * P;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < n) v = *reinterpret_cast<const uint4*>(kv_row(a, b, L, s0 + r, kh, kv) + c * 8);
        *reinterpret_cast<uint4*>(buf + r * (D + 8) + c * 8) = v;
    }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_chunk_kernel(const AttnArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    extern __shared__ float4 attn_smem[];
    const int G = a.Hq / a.Hkv, R = a.T * G;
    float* qs = reinterpret_cast<float*>(attn_smem);         // [32][D]
    float* ps = qs + kAttnMaxRows * D;                       // [32][64]
    float* st = ps + kAttnMaxRows * kAttnChunk;              // max [32], sum [32]
    uint16_t* kv = reinterpret_cast<uint16_t*>(st + 2 * kAttnMaxRows);   // [64][D + 8]
    const int split = blockIdx.x, kh = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int L = seq_len(a, b), S = L + a.T;
    const int s0 = split * kAttnChunk;
    float* part = a.part + ((((size_t)b * a.Hkv + kh) * a.nsplit + split) * R) * (D + 2);
    if (s0 >= S) {                                           // no key here: an empty partial
        for (int r = tid; r < R; r += kAttnThreads) {
            part[(size_t)r * (D + 2) + D] = -__uint_as_float(0x7F800000u);
            part[(size_t)r * (D + 2) + D + 1] = 0.f;
        }
        return;
    }
    const int n = min(kAttnChunk, S - s0);
    // query rows r = j * G + g of heads kh * G + g, 8 values per load
    {
        const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * D;
        for (int e = tid; e < R * (D / 8); e += kAttnThreads) {
            const int r = e / (D / 8), c = e - r * (D / 8), j = r / G, h = kh * G + (r - j * G);
            const uint4 v = *reinterpret_cast<const uint4*>(a.qkv + ((size_t)b * a.T + j) * W + (size_t)h * D + c * 8);
            float4* q = reinterpret_cast<float4*>(qs + r * D + c * 8);
            q[0] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
            q[1] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
        }
    }
    stage_rows<D>(a, b, L, s0, n, kh, 0, kv);
    __syncthreads();

    // scores: thread (key t % 64, group of 8 rows t / 64)
    {
        const int kl = tid % kAttnChunk, r0 = (tid / kAttnChunk) * 8, s = s0 + kl;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.f;
        if (kl < n && r0 < R) {
            const uint16_t* kr = kv + kl * (D + 8);
#pragma unroll 4
            for (int d0 = 0; d0 < D; d0 += 8) {
                const uint4 w = *reinterpret_cast<const uint4*>(kr + d0);
                const float k0 = bf16lo(w.x), k1 = bf16hi(w.x), k2 = bf16lo(w.y), k3 = bf16hi(w.y);
                const float k4 = bf16lo(w.z), k5 = bf16hi(w.z), k6 = bf16lo(w.w), k7 = bf16hi(w.w);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 qa = *reinterpret_cast<const float4*>(qs + (r0 + q) * D + d0);
                    const float4 qb = *reinterpret_cast<const float4*>(qs + (r0 + q) * D + d0 + 4);
                    acc[q] += qa.x * k0 + qa.y * k1 + qa.z * k2 + qa.w * k3 +
                              qb.x * k4 + qb.y * k5 + qb.z * k6 + qb.w * k7;
                }
            }
        }
        if (r0 < R) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int r = r0 + q;
                if (r < R) {
                    const bool vis = kl < n && s < L + r / G + 1;      // causal
                    ps[r * kAttnChunk + kl] = vis ? acc[q] * a.scale : -__uint_as_float(0x7F800000u);
                }
            }
        }
    }
    __syncthreads();

    // the chunk's values replace its keys; row statistics meanwhile
    stage_rows<D>(a, b, L, s0, n, kh, 1, kv);
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r < R; r += kAttnThreads / 32) {
            const float v0 = ps[r * kAttnChunk + lane], v1 = ps[r * kAttnChunk + lane + 32];
            float m = fmaxf(v0, v1);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            const bool none = m == -__uint_as_float(0x7F800000u);
            const float p0 = none ? 0.f : expf(v0 - m), p1 = none ? 0.f : expf(v1 - m);
            ps[r * kAttnChunk + lane] = p0;
            ps[r * kAttnChunk + lane + 32] = p1;
            float l = p0 + p1;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (lane == 0) {
                st[r] = m;
                st[kAttnMaxRows + r] = l;
            }
        }
    }
    __syncthreads();

    // unnormalised p . v: thread (dim t % D, group of rows t / D)
    {
        constexpr int RG = kAttnThreads / D;                 // row groups: 2 (D = 128) or 4 (D = 64)
        constexpr int RPG = kAttnMaxRows / RG;               // rows per group
        const int d = tid % D, r0 = (tid / D) * RPG;
        if (r0 < R) {
            float acc[RPG];
#pragma unroll
            for (int q = 0; q < RPG; ++q) acc[q] = 0.f;
#pragma unroll 2
            for (int i0 = 0; i0 < kAttnChunk; i0 += 4) {
                const float v0 = __uint_as_float((uint32_t)kv[(i0 + 0) * (D + 8) + d] << 16);
                const float v1 = __uint_as_float((uint32_t)kv[(i0 + 1) * (D + 8) + d] << 16);
                const float v2 = __uint_as_float((uint32_t)kv[(i0 + 2) * (D + 8) + d] << 16);
                const float v3 = __uint_as_float((uint32_t)kv[(i0 + 3) * (D + 8) + d] << 16);
#pragma unroll
                for (int q = 0; q < RPG; ++q) {
                    if (r0 + q < R) {
                        const float4 p = *reinterpret_cast<const float4*>(ps + (r0 + q) * kAttnChunk + i0);
                        acc[q] += p.x * v0 + p.y * v1 + p.z * v2 + p.w * v3;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < RPG; ++q)
                if (r0 + q < R) part[(size_t)(r0 + q) * (D + 2) + d] = acc[q];
        }
        for (int r = tid; r < R; r += kAttnThreads) {
            part[(size_t)r * (D + 2) + D] = st[r];
            part[(size_t)r * (D + 2) + D + 1] = st[kAttnMaxRows + r];
        }
    }
}

// One CTA per (query row, key/value head, sequence):
// out = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c over the chunks.
template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const AttnArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    const int r = blockIdx.x, kh = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
    const int G = a.Hq / a.Hkv, R = a.T * G;
    const int L = seq_len(a, b), S = L + a.T;
    const int n = (S + kAttnChunk - 1) / kAttnChunk;
    const float* base = a.part + (((size_t)b * a.Hkv + kh) * a.nsplit) * R * (D + 2) + (size_t)r * (D + 2);
    const size_t cs = (size_t)R * (D + 2);                    // chunk stride
    float M = -__uint_as_float(0x7F800000u);
#pragma unroll 8
    for (int c = 0; c < n; ++c) M = fmaxf(M, base[c * cs + D]);
    float num = 0.f, den = 0.f;
#pragma unroll 8
    for (int c = 0; c < n; ++c) {
        const float m = base[c * cs + D];
        const float w = m == -__uint_as_float(0x7F800000u) ? 0.f : expf(m - M);   // a chunk with no visible key
        num += w * base[c * cs + d];
        den += w * base[c * cs + D + 1];
    }
    const int j = r / G, h = kh * G + (r - j * G);
    a.out[((size_t)b * a.T + j) * (size_t)a.Hq * D + (size_t)h * D + d] = num / den;
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
constexpr size_t attn_smem() {
    return (size_t)(kAttnMaxRows * D + kAttnMaxRows * kAttnChunk + 2 * kAttnMaxRows) * sizeof(float) +
           (size_t)kAttnChunk * (D + 8) * sizeof(uint16_t);
}
static_assert(attn_smem<128>() <= 48 * 1024, "no shared-memory opt-in needed");

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
    const int R = T * (Hq / Hkv);
    const dim3 g1(a.nsplit, Hkv, B), g2(R, Hkv, B);
    cudaError_t e;
    if (D == 128) {
        if ((e = launch_attn(attn_chunk_kernel<128>, g1, kAttnThreads, attn_smem<128>(), a, s)) != cudaSuccess) return e;
        return launch_attn(attn_combine_kernel<128>, g2, 128, 0, a, s);
    }
    if ((e = launch_attn(attn_chunk_kernel<64>, g1, kAttnThreads, attn_smem<64>(), a, s)) != cudaSuccess) return e;
    return launch_attn(attn_combine_kernel<64>, g2, 64, 0, a, s);
}

}  // namespace qv
