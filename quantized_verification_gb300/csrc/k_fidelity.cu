// k_fidelity.cu -- logit-fidelity diagnostic: KL(p || q) between the softmax
// of a reference verifier's logits (p) and of the quantized verifier's (q),
// and both top-1 tokens.
//
//   The Quasar summaries report that quantizing the verifier keeps the logit
//   distribution (negligible KL divergence: gist.science/fr summary,
//   contributions item 3; high logit-distribution similarity: shd-paper.top
//   summary, method details, core idea). This kernel measures that on given logits.
//
// One CTA per row, three passes over the row:
//   1. the maxima of a and b with their lowest indices (64-bit keys,
//      order-preserving value bits above the complemented index);
//   2. Z = sum e^(a_v - max a) and the p-mean of d_v = b_v - a_v,
//      c = sum e^(a_v - max a) d_v / Z;
//   3. KL = log1p(sum e^(a_v - max a) expm1(d_v - c) / Z) - (E_p[d] - c).
// Pass 3 is the identity KL(p || q) = log E_p[e^(d - c)] - E_p[d - c], true
// for any c; with c the binary32 rounding of E_p[d] the last term is that
// rounding's residual (binary64), which cancels its first-order effect on
// the first. Nothing subtracts two large numbers, so KL values far below the
// size of the logits keep their relative accuracy. Per-thread sums are
// binary32, the block's sums binary64.

#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kFidThreads = 1024;

__device__ __forceinline__ unsigned long long fid_key(float f, int v) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)v);
}
__device__ __forceinline__ float fid_val(unsigned long long k) {
    const uint32_t o = (uint32_t)(k >> 32);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ int fid_idx(unsigned long long k) { return (int)(0xFFFFFFFFu - (uint32_t)k); }

template <class T, class Op>
__device__ __forceinline__ T block_reduce(T v, T* sm, Op op) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
    __syncthreads();
    T r = sm[0];
#pragma unroll
    for (int w = 1; w < kFidThreads / 32; ++w) r = op(r, sm[w]);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kFidThreads) logit_fidelity_kernel(const float* __restrict__ a,
                                                                      const float* __restrict__ b, int V,
                                                                      float* __restrict__ kl,
                                                                      int32_t* __restrict__ top_a,
                                                                      int32_t* __restrict__ top_b) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ unsigned long long sk[kFidThreads / 32];
    __shared__ double sd[kFidThreads / 32];
    const size_t row = blockIdx.x;
    const float* ar = a + row * (size_t)V;
    const float* br = b + row * (size_t)V;
    unsigned long long ka = 0, kb = 0;
    for (int v = threadIdx.x; v < V; v += kFidThreads) {
        const unsigned long long x = fid_key(ar[v], v), y = fid_key(br[v], v);
        ka = x > ka ? x : ka;
        kb = y > kb ? y : kb;
    }
    auto umax = [](unsigned long long x, unsigned long long y) { return x > y ? x : y; };
    ka = block_reduce(ka, sk, umax);
    kb = block_reduce(kb, sk, umax);
    const float ma = fid_val(ka);
    float z = 0.f, s1 = 0.f;
    for (int v = threadIdx.x; v < V; v += kFidThreads) {
        const float e = expf(ar[v] - ma);
        z += e;
        s1 += e * (br[v] - ar[v]);
    }
    auto dsum = [](double x, double y) { return x + y; };
    const double Z = block_reduce((double)z, sd, dsum);
    const double S1 = block_reduce((double)s1, sd, dsum);
    const float c = (float)(S1 / Z);
    float s2 = 0.f;
    for (int v = threadIdx.x; v < V; v += kFidThreads) {
        const float e = expf(ar[v] - ma);
        s2 += e * expm1f((br[v] - ar[v]) - c);
    }
    const double S2 = block_reduce((double)s2, sd, dsum);
    if (threadIdx.x == 0) {
        kl[row] = (float)(log1p(S2 / Z) - (S1 / Z - (double)c));
        top_a[row] = fid_idx(ka);
        top_b[row] = fid_idx(kb);
    }
}

}  // namespace

cudaError_t launch_logit_fidelity(const float* a, const float* b, int M, int V, float* kl, int32_t* top_a,
                                  int32_t* top_b, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(kFidThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, logit_fidelity_kernel, a, b, V, kl, top_a, top_b);
}

}  // namespace qv
