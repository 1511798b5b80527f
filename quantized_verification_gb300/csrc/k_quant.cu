// k_quant.cu -- per-row symmetric int8 quantization (a1 activations, one row
// per token; a0 weights, one row per output channel).
//
//   Quasar, gist.science/ja summary, section 2.2 "Enhanced SmoothQuant",
//   items 2-3: weights quantized to INT8 offline; BF16 activations scaled by
//   the smoothing factor and converted to INT8 online.
//
// One CTA of 512 threads per row. Rows of up to 512 x 4 16-byte vectors
// (16384 bf16 / 8192 fp32 elements) are read once into registers with all
// loads in flight together; longer rows are read twice (amax pass, code
// pass). amax = max |x * c| is reduced with warp shuffles and one
// shared-memory step. Every floating point step is a single IEEE operation
// in round-to-nearest-even:
//   s = fl(amax / 127), q = clamp(rne(fl(x' / s)), -127, 127), q = 0 if s == 0,
// where the quotient's rounding is decided from fl(x' * fl(1 / s)) unless
// that product lies within 2^-20 of a half-integer (then from the quotient
// itself; quant_code in qv_ptx.cuh gives the error bound).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kQuantThreads = 512;
constexpr int kQuantRegVecs = 4;   // 16-byte vectors per thread kept in registers

template <bool BF16>
struct Vec;
template <>
struct Vec<true> {       // 8 bf16 per 16-byte load
    static constexpr int E = 8;
    static __device__ __forceinline__ void unpack(const uint4& r, float (&e)[8]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            e[2 * j] = __uint_as_float(w[j] << 16);
            e[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
};
template <>
struct Vec<false> {      // 4 fp32 per 16-byte load
    static constexpr int E = 4;
    static __device__ __forceinline__ void unpack(const uint4& r, float (&e)[4]) {
        e[0] = __uint_as_float(r.x);
        e[1] = __uint_as_float(r.y);
        e[2] = __uint_as_float(r.z);
        e[3] = __uint_as_float(r.w);
    }
};

// x' = fl(x * c) for the E elements of vector v (c = 1 without multipliers).
template <int E>
__device__ __forceinline__ void apply_mul(float (&e)[E], const float* __restrict__ mul, int v) {
    if (mul) {
#pragma unroll
        for (int j = 0; j < E; ++j) e[j] = __fmul_rn(e[j], __ldg(mul + v * E + j));
    }
}

template <int E>
__device__ __forceinline__ void store_codes(int8_t* qr, int v, const float (&e)[E], float s, float r) {
    uint32_t packed[E / 4];
#pragma unroll
    for (int w = 0; w < E / 4; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            word |= (uint32_t)(uint8_t)(int8_t)quant_code(e[4 * w + j], s, r) << (8 * j);
        packed[w] = word;
    }
    if constexpr (E == 8)
        *reinterpret_cast<uint2*>(qr + v * 8) = make_uint2(packed[0], packed[1]);
    else
        *reinterpret_cast<uint32_t*>(qr + v * 4) = packed[0];
}

template <bool BF16>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rows_kernel(const uint8_t* __restrict__ x, int K, const float* __restrict__ mul,
                     int8_t* __restrict__ q, float* __restrict__ scale, int early_dependents) {
    using V = Vec<BF16>;
    constexpr int E = V::E;
    if (early_dependents) allow_dependent_launch();

    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    const int nvec = K / E;
    const bool in_regs = nvec <= kQuantThreads * kQuantRegVecs;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * K * (BF16 ? 2 : 4));
    // Bring the row (and the multipliers) into L2 while the preceding kernel
    // finishes. A prefetch returns nothing to the SM, and L2 is the point of
    // coherence, so it cannot observe data older than the dependency wait.
    if (in_regs) {
        for (int v = tid * 8; v < nvec; v += kQuantThreads * 8) {   // one 128-byte line per 8 vectors
            asm volatile("prefetch.global.L2 [%0];" :: "l"(xr + v));
            if (mul) {   // 8 vectors of multipliers span 8 * E * 4 bytes: one or two lines
                asm volatile("prefetch.global.L2 [%0];" :: "l"(mul + (size_t)v * E));
                if (E == 8) asm volatile("prefetch.global.L2 [%0];" :: "l"(mul + (size_t)v * E + 32));
            }
        }
    }
    grid_dependency_wait();

    uint4 rv[kQuantRegVecs];
    float amax = 0.f;
    if (in_regs) {
#pragma unroll
        for (int u = 0; u < kQuantRegVecs; ++u) {
            const int v = tid + u * kQuantThreads;
            rv[u] = v < nvec ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQuantRegVecs; ++u) {
            const int v = tid + u * kQuantThreads;
            if (v < nvec) {
                float e[E];
                V::unpack(rv[u], e);
                apply_mul<E>(e, mul, v);
#pragma unroll
                for (int j = 0; j < E; ++j) amax = fmaxf(amax, fabsf(e[j]));
            }
        }
    } else {
        for (int v = tid; v < nvec; v += kQuantThreads) {
            float e[E];
            V::unpack(__ldg(xr + v), e);
            apply_mul<E>(e, mul, v);
#pragma unroll
            for (int j = 0; j < E; ++j) amax = fmaxf(amax, fabsf(e[j]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __shared__ float warp_max[kQuantThreads / 32];
    if ((tid & 31) == 0) warp_max[tid >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float r = __frcp_rn(s);
    if (tid == 0) scale[row] = s;

    int8_t* qr = q + (size_t)row * K;
    if (in_regs) {
#pragma unroll
        for (int u = 0; u < kQuantRegVecs; ++u) {
            const int v = tid + u * kQuantThreads;
            if (v < nvec) {
                float e[E];
                V::unpack(rv[u], e);
                apply_mul<E>(e, mul, v);
                store_codes<E>(qr, v, e, s, r);
            }
        }
    } else {
        for (int v = tid; v < nvec; v += kQuantThreads) {
            float e[E];
            V::unpack(__ldg(xr + v), e);
            apply_mul<E>(e, mul, v);
            store_codes<E>(qr, v, e, s, r);
        }
    }
}

}  // namespace

cudaError_t launch_quantize_rows(const void* x, bool bf16, int rows, int K, const float* mul,
                                 int8_t* q, float* scale, bool early_dependents, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows);
    cfg.blockDim = dim3(kQuantThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const int early = early_dependents ? 1 : 0;
    if (bf16) return cudaLaunchKernelEx(&cfg, quantize_rows_kernel<true>, xb, K, mul, q, scale, early);
    return cudaLaunchKernelEx(&cfg, quantize_rows_kernel<false>, xb, K, mul, q, scale, early);
}

}  // namespace qv
