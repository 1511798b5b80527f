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
// Every row is cut into S chunks of kSpecChunk tokens, one CTA per (chunk,
// row), so that the per-token exp runs on all SMs. Each kernel writes every
// value it leaves in the workspace (no atomics, nothing to clear):
//   spec_max_kernel     chunk maxima of the logits;
//   spec_sums_kernel    row max m from the chunk maxima, chunk sums of w and c;
//   spec_decide_kernel  per sequence: Z, Q, w_d, c_d of every row from the
//                       chunk sums, then the keep tests (one thread);
//   spec_chunk_kernel   chunk sums of the chosen row's replacement weights;
//   spec_draw_kernel    exact scan of the chunk sums, then an exact scan
//                       inside the chunk that holds the target.
// Integer sums are exact in any order and the max does not depend on it, so
// the split changes no result.

#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

using u128 = unsigned __int128;

constexpr int kSpecChunk = 2048;    // tokens per (chunk, row) CTA
constexpr int kSpecThreads = 256;   // threads of the per-chunk kernels
constexpr int kDrawThreads = 1024;  // threads of the draw kernel (two tokens each)
static_assert(kSpecChunk == 2 * kDrawThreads, "the draw kernel scans one chunk, two tokens a thread");

struct RowStats {
    float m;            // row max of the logits
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

// Replacement (residual) or bonus weight of token v.
__device__ __forceinline__ u128 draw_weight(const float* zr, const float* qr, int v, float m, float T,
                                            bool residual, uint64_t Z, uint64_t Q) {
    const uint32_t w = p_weight(zr[v], m, T);
    if (!residual) return (u128)w;
    const u128 a1 = (u128)w * Q, a2 = (u128)weight24(qr[v]) * Z;
    return a1 > a2 ? a1 - a2 : (u128)0;
}

__device__ __forceinline__ u128 shfl_up_u128(u128 v, int off) {
    const uint64_t lo = __shfl_up_sync(0xffffffffu, (uint64_t)v, off);
    const uint64_t hi = __shfl_up_sync(0xffffffffu, (uint64_t)(v >> 64), off);
    return ((u128)hi << 64) | lo;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Exclusive prefix of one u128 per thread over the block (NT threads, all of
// them call it); *total gets the block's sum. sm: NT / 32 + 1 entries.
template <int NT>
__device__ __forceinline__ u128 block_exclusive_scan(u128 v, u128* sm, u128* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    u128 incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const u128 o = shfl_up_u128(incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) sm[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const u128 w = lane < NT / 32 ? sm[lane] : (u128)0;
        u128 wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const u128 o = shfl_up_u128(wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < NT / 32) sm[lane] = wi - w;           // exclusive start of each warp
        if (lane == NT / 32 - 1) sm[NT / 32] = wi;       // block total
    }
    __syncthreads();
    const u128 r = sm[warp] + (incl - v);
    *total = sm[NT / 32];
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_max_f(float v, float* red) {
    v = warp_max_f(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kSpecThreads / 32; ++w) m = fmaxf(m, red[w]);
    __syncthreads();
    return m;
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, unsigned long long* red) {
    v = warp_sum_u64(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long s = 0;
#pragma unroll
    for (int w = 0; w < kSpecThreads / 32; ++w) s += red[w];
    __syncthreads();
    return s;
}

struct SpecArgs {
    const float* z;           // [M][V] logits
    const int32_t* draft;     // [B][gamma]
    const float* q;           // [B][gamma][V]
    int gamma, V, S;          // S chunks per row
    float T;
    uint64_t seed;
    float* mc;                // [M][S] chunk maxima
    unsigned long long* zc;   // [M][S] chunk sums of w
    unsigned long long* qc;   // [M][S] chunk sums of c (draft rows)
    RowStats* stats;          // [M]
    u128* xc;                 // [B][S] chunk sums of the chosen row's draw weights
    int* dec;                 // [B] kept drafts
    int32_t* accept_len;
    int32_t* out_tokens;
};

__global__ void __launch_bounds__(kSpecThreads) spec_max_kernel(const SpecArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ float red[kSpecThreads / 32];
    const int row = blockIdx.y, s = blockIdx.x;
    const int v0 = s * kSpecChunk, v1 = min(a.V, v0 + kSpecChunk);
    const float* zr = a.z + (size_t)row * a.V;
    float m = -__uint_as_float(0x7F800000u);
    for (int v = v0 + threadIdx.x; v < v1; v += kSpecThreads) m = fmaxf(m, zr[v]);
    m = block_max_f(m, red);
    if (threadIdx.x == 0) a.mc[(size_t)row * a.S + s] = m;
}

__global__ void __launch_bounds__(kSpecThreads) spec_sums_kernel(const SpecArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ float red_f[kSpecThreads / 32];
    __shared__ unsigned long long red_u[kSpecThreads / 32];
    const int row = blockIdx.y, s = blockIdx.x;
    const int v0 = s * kSpecChunk, v1 = min(a.V, v0 + kSpecChunk);
    const int G = a.gamma + 1, b = row / G, j = row - b * G;
    const bool is_draft = j < a.gamma;
    const float* zr = a.z + (size_t)row * a.V;
    const float* qr = is_draft ? a.q + ((size_t)b * a.gamma + j) * a.V : nullptr;
    float m = -__uint_as_float(0x7F800000u);
    for (int e = threadIdx.x; e < a.S; e += kSpecThreads) m = fmaxf(m, a.mc[(size_t)row * a.S + e]);
    m = block_max_f(m, red_f);
    unsigned long long Zs = 0, Qs = 0;
    for (int v = v0 + threadIdx.x; v < v1; v += kSpecThreads) {
        Zs += p_weight(zr[v], m, a.T);
        if (is_draft) Qs += weight24(qr[v]);
    }
    Zs = block_sum_u64(Zs, red_u);
    if (is_draft) Qs = block_sum_u64(Qs, red_u);
    if (threadIdx.x == 0) {
        a.zc[(size_t)row * a.S + s] = Zs;
        a.qc[(size_t)row * a.S + s] = Qs;
    }
}

// One CTA per sequence: warp w gathers the statistics of rows w, w + 8, ...
__global__ void __launch_bounds__(kSpecThreads) spec_decide_kernel(const SpecArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    const int b = blockIdx.x, G = a.gamma + 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int j = warp; j < G; j += kSpecThreads / 32) {
        const int row = b * G + j;
        float m = -__uint_as_float(0x7F800000u);
        unsigned long long Z = 0, Q = 0;
        for (int e = lane; e < a.S; e += 32) {
            m = fmaxf(m, a.mc[(size_t)row * a.S + e]);
            Z += a.zc[(size_t)row * a.S + e];
            Q += a.qc[(size_t)row * a.S + e];
        }
        m = warp_max_f(m);
        Z = warp_sum_u64(Z);
        Q = warp_sum_u64(Q);
        if (lane == 0) {
            RowStats st{m, 0u, Z, Q, 0u, 0u};
            if (j < a.gamma) {
                const int d = a.draft[b * a.gamma + j];
                if (d >= 0 && d < a.V) {             // a token outside the vocabulary is never kept
                    st.w_d = p_weight(a.z[(size_t)row * a.V + d], m, a.T);
                    st.c_d = weight24(a.q[((size_t)b * a.gamma + j) * a.V + d]);
                }
            }
            a.stats[row] = st;
        }
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    int k = 0;
    for (; k < a.gamma; ++k) {
        const RowStats st = a.stats[b * G + k];
        const uint32_t u24 = (uint32_t)(splitmix64(a.seed, 2ull * (uint64_t)(b * G + k)) >> 40);
        const u128 lhs = (u128)u24 * (u128)st.Z * (u128)st.c_d;
        const u128 rhs = ((u128)st.w_d * (u128)st.Q) << 24;
        if (!(lhs < rhs)) break;
    }
    a.dec[b] = k;
}

__global__ void __launch_bounds__(kSpecThreads) spec_chunk_kernel(const SpecArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ u128 sm[kSpecThreads / 32 + 1];
    const int b = blockIdx.y, s = blockIdx.x, G = a.gamma + 1;
    const int k = a.dec[b], row = b * G + k;
    if (k == a.gamma) {                              // bonus draw: the chunk sums of w are known
        if (threadIdx.x == 0) a.xc[(size_t)b * a.S + s] = (u128)a.zc[(size_t)row * a.S + s];
        return;
    }
    const RowStats st = a.stats[row];
    const float* zr = a.z + (size_t)row * a.V;
    const float* qr = a.q + ((size_t)b * a.gamma + k) * a.V;
    const int v0 = s * kSpecChunk, v1 = min(a.V, v0 + kSpecChunk);
    u128 x = 0;
    for (int v = v0 + threadIdx.x; v < v1; v += kSpecThreads)
        x += draw_weight(zr, qr, v, st.m, a.T, true, st.Z, st.Q);
    u128 total;
    block_exclusive_scan<kSpecThreads>(x, sm, &total);
    if (threadIdx.x == 0) a.xc[(size_t)b * a.S + s] = total;
}

__global__ void __launch_bounds__(kDrawThreads) spec_draw_kernel(const SpecArgs a) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ u128 sm[kDrawThreads / 32 + 1];
    __shared__ u128 base_s;
    __shared__ int chunk_s, token_s;
    const int b = blockIdx.x, tid = threadIdx.x, G = a.gamma + 1;
    const int k = a.dec[b], row = b * G + k;
    const RowStats st = a.stats[row];
    const float* zr = a.z + (size_t)row * a.V;
    const float* qr = k < a.gamma ? a.q + ((size_t)b * a.gamma + k) * a.V : nullptr;
    const uint32_t u2 = (uint32_t)(splitmix64(a.seed, 2ull * (uint64_t)row + 1) >> 40);
    const int E = (a.S + kDrawThreads - 1) / kDrawThreads;     // chunk sums per thread
    const int e0 = min(a.S, tid * E), e1 = min(a.S, e0 + E);
    if (tid == 0) { chunk_s = -1; token_s = -1; base_s = 0; }

    // replacement weights; when they are all zero (p == q on the integer
    // grid) the draw falls back to p itself
    bool residual = k < a.gamma;
    u128 mine, start, total;
    for (;;) {
        mine = 0;
        for (int e = e0; e < e1; ++e) mine += residual ? a.xc[(size_t)b * a.S + e] : (u128)a.zc[(size_t)row * a.S + e];
        start = block_exclusive_scan<kDrawThreads>(mine, sm, &total);
        if (total == 0 && residual) { residual = false; continue; }
        break;
    }
    // floor(u2 * total / 2^24), split so that nothing overflows
    const u128 target = (total >> 24) * u2 + (((total & 0xFFFFFFull) * u2) >> 24);
    if (mine > 0 && start <= target && target < start + mine) {
        u128 acc = start;
        for (int e = e0; e < e1; ++e) {
            const u128 c = residual ? a.xc[(size_t)b * a.S + e] : (u128)a.zc[(size_t)row * a.S + e];
            if (acc + c > target) { chunk_s = e; base_s = acc; break; }
            acc += c;
        }
    }
    __syncthreads();
    const int cs = chunk_s;
    const u128 base = base_s;
    // the owning chunk: two tokens a thread, exact scan, first prefix above the target
    const int v0 = max(cs, 0) * kSpecChunk + 2 * tid;
    const int vend = cs < 0 ? 0 : min(a.V, cs * kSpecChunk + kSpecChunk);   // no chunk: read nothing
    const u128 x0 = v0 < vend ? draw_weight(zr, qr, v0, st.m, a.T, residual, st.Z, st.Q) : (u128)0;
    const u128 x1 = v0 + 1 < vend ? draw_weight(zr, qr, v0 + 1, st.m, a.T, residual, st.Z, st.Q) : (u128)0;
    u128 chunk_total;
    const u128 pre = base + block_exclusive_scan<kDrawThreads>(x0 + x1, sm, &chunk_total);
    if (x0 > 0 && pre <= target && target < pre + x0) token_s = v0;
    else if (x1 > 0 && pre + x0 <= target && target < pre + x0 + x1) token_s = v0 + 1;
    __syncthreads();
    if (tid == 0) {
        int tok = token_s;
        if (tok < 0) tok = a.V - 1;                  // unreachable: the total is positive
        a.accept_len[b] = k + 1;
        for (int j = 0; j < G; ++j)
            a.out_tokens[b * G + j] = j < k ? a.draft[b * a.gamma + j] : (j == k ? tok : -1);
    }
}

cudaError_t launch_spec(const void* kernel, dim3 grid, int threads, const SpecArgs& args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* kargs[] = {const_cast<SpecArgs*>(&args)};
    return cudaLaunchKernelExC(&cfg, kernel, kargs);
}

int spec_chunks(int V) { return (V + kSpecChunk - 1) / kSpecChunk; }

size_t al256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

size_t spec_workspace_bytes(int M, int V) {
    const size_t S = (size_t)spec_chunks(V), m = (size_t)M;
    return al256(m * S * 4) + 2 * al256(m * S * 8) + al256(m * sizeof(RowStats)) + al256(m * S * 16) +
           al256(m * 4);
}

cudaError_t launch_spec_sample(const float* logits, const int32_t* draft, const float* q, int B, int gamma,
                               int V, float T, uint64_t seed, int32_t* accept_len, int32_t* out_tokens,
                               void* ws, cudaStream_t s) {
    const int M = B * (gamma + 1);
    const int S = spec_chunks(V);
    uint8_t* p = static_cast<uint8_t*>(ws);
    SpecArgs a;
    a.z = logits; a.draft = draft; a.q = q;
    a.gamma = gamma; a.V = V; a.S = S; a.T = T; a.seed = seed;
    a.mc = reinterpret_cast<float*>(p);
    p += al256((size_t)M * S * 4);
    a.zc = reinterpret_cast<unsigned long long*>(p);
    p += al256((size_t)M * S * 8);
    a.qc = reinterpret_cast<unsigned long long*>(p);
    p += al256((size_t)M * S * 8);
    a.stats = reinterpret_cast<RowStats*>(p);
    p += al256((size_t)M * sizeof(RowStats));
    a.xc = reinterpret_cast<u128*>(p);
    p += al256((size_t)M * S * 16);
    a.dec = reinterpret_cast<int*>(p);
    a.accept_len = accept_len; a.out_tokens = out_tokens;
    cudaError_t e;
    if ((e = launch_spec(reinterpret_cast<const void*>(spec_max_kernel), dim3(S, M), kSpecThreads, a, s)) != cudaSuccess) return e;
    if ((e = launch_spec(reinterpret_cast<const void*>(spec_sums_kernel), dim3(S, M), kSpecThreads, a, s)) != cudaSuccess) return e;
    if ((e = launch_spec(reinterpret_cast<const void*>(spec_decide_kernel), dim3(B), kSpecThreads, a, s)) != cudaSuccess) return e;
    if ((e = launch_spec(reinterpret_cast<const void*>(spec_chunk_kernel), dim3(S, B), kSpecThreads, a, s)) != cudaSuccess) return e;
    return launch_spec(reinterpret_cast<const void*>(spec_draw_kernel), dim3(B), kDrawThreads, a, s);
}

}  // namespace qv
