// k_spec.cu -- lossless rejection sampling at temperature T > 0 (speculative
// sampling) over the verifier's dequantized logits.
//
//   Quasar, gist.science/it summary, section 2 item 3 ("Campionamento di
//   Rifiuto Lossless"): the verifier's logits stay precise so that the
//   accept/reject step keeps the target distribution.
//
// Rule, per sequence b with drafts d_0 .. d_{gamma-1} drawn from q_0 ..:
// keep d_j with probability min(1, p_j(d_j) / q_j(d_j)); at the first
// rejection draw the replacement from the normalized max(0, p_j - q_j); when
// every draft is kept draw the bonus token from p_gamma. Probabilities are
// integer weights so that every sum over the vocabulary is exact:
//   p_j: m = max_v z_v, w_v = floor(E(fl32(fl32(z_v - m) / T)) * 2^24),
//        Z = sum_v w_v (E: the layer's exp, layer_exp);
//   q_j: c_v = floor(fl32(clamp(q_v, 0, 1) * 2^24)), Q = sum_v c_v;
//   keep d iff u24 * Z * c_d < w_d * Q * 2^24 (128-bit integers);
//   replacement weights r_v = max(0, w_v * Q - c_v * Z) (w if they are all 0);
//   a draw from weights x (total X) is the smallest v whose prefix sum
//   exceeds floor(u24' * X / 2^24).
// Uniforms: the top 24 bits of SplitMix64 draw n = 2 * row + purpose of the
// caller's seed (counter-based: mix(seed + (n + 1) * 0x9E3779B97F4A7C15),
// G. Steele, D. Lea, C. Flood, 2014), row = b * (gamma + 1) + j, purpose 0
// for the keep test and 1 for the draw.
//
// spec_row_stats_kernel: one CTA per verify row: m, Z, and for draft rows Q,
// w_d, c_d (max and integer sums do not depend on the order, so the loads are
// coalesced). spec_decide_draw_kernel: one CTA per sequence: the keep tests,
// then one pass over the chosen row's weights in contiguous per-thread
// chunks, an exact scan of the chunk totals and a rescan of the chunk that
// holds the target.

#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

using u128 = unsigned __int128;

constexpr int kSpecThreads = 1024;

struct RowStats {
    float m;            // row max
    uint32_t w_d;       // p weight of the draft token (draft rows)
    unsigned long long Z, Q;
    uint32_t c_d;       // q weight of the draft token (draft rows)
    uint32_t pad;
};
static_assert(sizeof(RowStats) == 32, "32-byte row statistics");

__device__ __forceinline__ uint64_t splitmix64(uint64_t s, uint64_t n) {
    uint64_t z = s + (n + 1) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t weight24(float x) {
    if (!(x > 0.0f)) return 0u;
    if (x >= 1.0f) return 1u << 24;
    return (uint32_t)__fmul_rn(x, 16777216.0f);     // exact product, truncated
}

__device__ __forceinline__ uint32_t p_weight(float z, float m, float T) {
    return weight24(layer_exp(__fdiv_rn(__fsub_rn(z, m), T)));
}

__device__ __forceinline__ float block_max_f(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kSpecThreads / 32; ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    return m;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long s = 0;
#pragma unroll
    for (int w = 0; w < kSpecThreads / 32; ++w) s += red[w];
    __syncthreads();
    return s;
}

__global__ void __launch_bounds__(kSpecThreads)
spec_row_stats_kernel(const float* __restrict__ z, const int32_t* __restrict__ draft,
                      const float* __restrict__ q, int gamma, int V, float T, RowStats* __restrict__ stats) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ float red_f[kSpecThreads / 32];
    __shared__ unsigned long long red_u[kSpecThreads / 32];
    const int row = blockIdx.x, tid = threadIdx.x;
    const int G = gamma + 1;
    const int b = row / G, j = row - b * G;
    const bool is_draft = j < gamma;
    const float* zr = z + (size_t)row * V;
    const float* qr = is_draft ? q + ((size_t)b * gamma + j) * V : nullptr;

    float m = -__uint_as_float(0x7F800000u);
    for (int v = tid; v < V; v += kSpecThreads) m = fmaxf(m, zr[v]);
    m = block_max_f(m, red_f);

    unsigned long long Z = 0, Q = 0;
    for (int v = tid; v < V; v += kSpecThreads) {
        Z += p_weight(zr[v], m, T);
        if (is_draft) Q += weight24(qr[v]);
    }
    Z = block_sum_u64(Z, red_u);
    if (is_draft) Q = block_sum_u64(Q, red_u);
    if (tid == 0) {
        RowStats st;
        st.m = m;
        st.Z = Z;
        st.Q = Q;
        st.w_d = 0;
        st.c_d = 0;
        st.pad = 0;
        if (is_draft) {
            const int d = draft[b * gamma + j];
            if (d >= 0 && d < V) {               // a token outside the vocabulary is never kept
                st.w_d = p_weight(zr[d], m, T);
                st.c_d = weight24(qr[d]);
            }
        }
        stats[row] = st;
    }
}

// Residual or bonus weight of token v of row (zr, qr) under the row's stats.
__device__ __forceinline__ u128 draw_weight(const float* zr, const float* qr, int v, float m, float T,
                                            bool residual, uint64_t Z, uint64_t Q) {
    const uint32_t w = p_weight(zr[v], m, T);
    if (!residual) return (u128)w;
    const u128 a1 = (u128)w * Q, a2 = (u128)weight24(qr[v]) * Z;
    return a1 > a2 ? a1 - a2 : (u128)0;
}

__global__ void __launch_bounds__(kSpecThreads)
spec_decide_draw_kernel(const float* __restrict__ z, const int32_t* __restrict__ draft,
                        const float* __restrict__ q, int gamma, int V, float T, uint64_t seed,
                        const RowStats* __restrict__ stats, int32_t* __restrict__ accept_len,
                        int32_t* __restrict__ out_tokens) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ u128 part[kSpecThreads];
    __shared__ int k_s;
    __shared__ int residual_s;
    __shared__ int token_s;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int G = gamma + 1;

    if (tid == 0) {
        int k = 0;
        for (; k < gamma; ++k) {
            const RowStats st = stats[b * G + k];
            const uint32_t u24 = (uint32_t)(splitmix64(seed, 2ull * (uint64_t)(b * G + k)) >> 40);
            const u128 lhs = (u128)u24 * (u128)st.Z * (u128)st.c_d;
            const u128 rhs = ((u128)st.w_d * (u128)st.Q) << 24;
            if (!(lhs < rhs)) break;
        }
        k_s = k;
        residual_s = k < gamma ? 1 : 0;
        token_s = -1;
    }
    __syncthreads();
    const int k = k_s;
    const int row = b * G + k;
    const RowStats st = stats[row];
    const float* zr = z + (size_t)row * V;
    const float* qr = k < gamma ? q + ((size_t)b * gamma + k) * V : nullptr;
    const int C = (V + kSpecThreads - 1) / kSpecThreads;        // contiguous chunk per thread
    const int v0 = tid * C, v1 = min(V, v0 + C);
    const uint32_t u2 = (uint32_t)(splitmix64(seed, 2ull * (uint64_t)row + 1) >> 40);

    // a second round (bonus weights w) only when every residual weight is 0
    for (int pass = 0; pass < 2; ++pass) {
        const bool residual = residual_s != 0;
        u128 s = 0;
        for (int v = v0; v < v1; ++v) s += draw_weight(zr, qr, v, st.m, T, residual, st.Z, st.Q);
        part[tid] = s;
        __syncthreads();
        // exclusive scan of the chunk totals: warp 0, 32 entries per lane
        if (tid < 32) {
            u128 acc = 0;
            for (int i = 0; i < kSpecThreads / 32; ++i) acc += part[tid * (kSpecThreads / 32) + i];
            u128 incl = acc;
            for (int off = 1; off < 32; off <<= 1) {            // inclusive scan of the lane totals
                const uint64_t lo = (uint64_t)incl, hi = (uint64_t)(incl >> 64);
                const uint64_t plo = __shfl_up_sync(0xffffffffu, lo, off);
                const uint64_t phi = __shfl_up_sync(0xffffffffu, hi, off);
                if (tid >= off) incl += ((u128)phi << 64) | plo;
            }
            u128 run = incl - acc;                                // exclusive start of this lane's block
            for (int i = 0; i < kSpecThreads / 32; ++i) {
                const u128 t = part[tid * (kSpecThreads / 32) + i];
                part[tid * (kSpecThreads / 32) + i] = run;
                run += t;
            }
        }
        __syncthreads();
        const u128 start = part[tid];
        __syncthreads();
        if (tid == kSpecThreads - 1) part[0] = start + s;        // the total: last start + last chunk
        __syncthreads();
        const u128 total = part[0];
        if (total == 0 && residual) {                             // p == q: draw from p instead
            __syncthreads();
            if (tid == 0) residual_s = 0;
            __syncthreads();
            continue;
        }
        // floor(u2 * total / 2^24) without overflow (total < 2^106)
        const u128 target = (total >> 24) * u2 + (((total & 0xFFFFFFull) * u2) >> 24);
        if (s > 0 && start <= target && target < start + s) {
            u128 acc = start;
            for (int v = v0; v < v1; ++v) {
                acc += draw_weight(zr, qr, v, st.m, T, residual, st.Z, st.Q);
                if (acc > target) {
                    token_s = v;
                    break;
                }
            }
        }
        __syncthreads();
        break;
    }
    if (tid == 0) {
        int tok = token_s;
        if (tok < 0) tok = V - 1;        // unreachable with a positive total
        accept_len[b] = k + 1;
        for (int j = 0; j < G; ++j)
            out_tokens[b * G + j] = j < k ? draft[b * gamma + j] : (j == k ? tok : -1);
    }
}

cudaError_t launch_pdl(const void* kernel, int grid, void** args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSpecThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace

size_t spec_workspace_bytes(int M) { return (size_t)M * sizeof(RowStats); }

cudaError_t launch_spec_sample(const float* logits, const int32_t* draft, const float* q, int B, int gamma,
                               int V, float T, uint64_t seed, int32_t* accept_len, int32_t* out_tokens,
                               void* ws, cudaStream_t s) {
    RowStats* stats = static_cast<RowStats*>(ws);
    const int M = B * (gamma + 1);
    void* a1[] = {&logits, &draft, &q, &gamma, &V, &T, &stats};
    cudaError_t e = launch_pdl(reinterpret_cast<const void*>(spec_row_stats_kernel), M, a1, s);
    if (e != cudaSuccess) return e;
    const RowStats* cstats = stats;
    void* a2[] = {&logits, &draft, &q, &gamma, &V, &T, &seed, &cstats, &accept_len, &out_tokens};
    return launch_pdl(reinterpret_cast<const void*>(spec_decide_draw_kernel), B, a2, s);
}

}  // namespace qv
