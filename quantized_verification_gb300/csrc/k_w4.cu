// k_w4.cu -- int4 weight quantization for the W4A8 verifier (a setup step,
// like qv_quantize_weight).
//
//   Lower-bit verifiers (4-bit, 2-bit) are the next step the Quasar
//   summaries name (gist.science/it, gist.science/de and gist.science/ja
//   summaries, section 5); INT4 is among the bit widths the authors tried
//   (shd-paper.top summary, method details, key design). No format is given; the rule here
//   is the int8 one with the code range [-7, 7]:
//     s = fl32(amax / 7), q = clamp(rne(fl32(w / s)), -7, 7), q = 0 when
//     s = 0; byte j of a row holds code 2j in bits 0-3 and code 2j+1 in bits
//     4-7, 4-bit two's complement.
// One CTA per output channel: an exact block max, then every thread packs
// pairs of codes.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kW4Threads = 256;

template <bool BF16>
__device__ __forceinline__ float load_w(const void* w, size_t i) {
    if constexpr (BF16) {
        const uint16_t h = static_cast<const uint16_t*>(w)[i];
        return __uint_as_float((uint32_t)h << 16);          // exact widening
    } else {
        return static_cast<const float*>(w)[i];
    }
}

__device__ __forceinline__ uint32_t code4(float v, float s) {
    if (s == 0.0f) return 0u;
    int q = __float2int_rn(__fdiv_rn(v, s));               // IEEE division, ties to even
    q = q > 7 ? 7 : (q < -7 ? -7 : q);
    return (uint32_t)q & 0xFu;
}

template <bool BF16>
__global__ void __launch_bounds__(kW4Threads) quantize_weight_w4_kernel(const void* __restrict__ w, int K,
                                                                         uint8_t* __restrict__ wq4,
                                                                         float* __restrict__ sw) {
    __shared__ float red[kW4Threads / 32];
    const size_t row = blockIdx.x;
    const size_t base = row * (size_t)K;
    float amax = 0.0f;
    for (int k = threadIdx.x; k < K; k += kW4Threads) amax = fmaxf(amax, fabsf(load_w<BF16>(w, base + k)));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < kW4Threads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(amax, 7.0f);
    if (threadIdx.x == 0) sw[row] = s;
    uint8_t* out = wq4 + row * (size_t)(K / 2);
    for (int j = threadIdx.x; j < K / 2; j += kW4Threads) {
        const uint32_t lo = code4(load_w<BF16>(w, base + 2 * j), s);
        const uint32_t hi = code4(load_w<BF16>(w, base + 2 * j + 1), s);
        out[j] = (uint8_t)(lo | (hi << 4));
    }
}

}  // namespace

cudaError_t launch_quantize_weight_w4(const void* w, bool bf16, int N, int K, uint8_t* wq4, float* sw,
                                      cudaStream_t s) {
    if (bf16)
        quantize_weight_w4_kernel<true><<<N, kW4Threads, 0, s>>>(w, K, wq4, sw);
    else
        quantize_weight_w4_kernel<false><<<N, kW4Threads, 0, s>>>(w, K, wq4, sw);
    return cudaGetLastError();
}

}  // namespace qv
