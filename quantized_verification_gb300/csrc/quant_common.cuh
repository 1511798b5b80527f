// quant_common.cuh -- symmetric int8 quantization of one row by the threads
// of a CTA (the activation- and weight-quantization kernel's body), written
// against a caller-supplied barrier so that any group of threads can run it.
//
//   Quasar, gist.science/ja summary, section 2.2 "Enhanced SmoothQuant",
//   items 2-3: BF16 activations scaled by the smoothing factor and converted
//   to INT8 online, one scale per token.
//
// amax = max |x * c| (c = 1 without multipliers), s = fl(amax / 127),
// q = quant_code(x * c, s, fl(1 / s)) (qv_ptx.cuh). Every floating point step
// is a single IEEE operation in round-to-nearest-even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_ptx.cuh"

namespace qv {
namespace {

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
    // fast rule for every element, the IEEE quotient only where some element
    // of the vector lies near a half-integer (rare)
    int c[E];
    unsigned near_mask = 0;
#pragma unroll
    for (int j = 0; j < E; ++j) {
        bool nb;
        c[j] = quant_code_fast(e[j], r, nb);
        near_mask |= (unsigned)nb << j;
    }
    if (s == 0.f) {
#pragma unroll
        for (int j = 0; j < E; ++j) c[j] = 0;
    } else if (near_mask) {
#pragma unroll
        for (int j = 0; j < E; ++j)
            if ((near_mask >> j) & 1u) c[j] = quant_code_exact(e[j], s);
    }
    uint32_t packed[E / 4];
#pragma unroll
    for (int w = 0; w < E / 4; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) word |= (uint32_t)(uint8_t)(int8_t)c[4 * w + j] << (8 * j);
        packed[w] = word;
    }
    if constexpr (E == 8)
        *reinterpret_cast<uint2*>(qr + v * 8) = make_uint2(packed[0], packed[1]);
    else
        *reinterpret_cast<uint32_t*>(qr + v * 4) = packed[0];
}

// Quantize one row of nvec 16-byte vectors (xr) into qr, by threads t in
// [0, NT) of the CTA, which all call it; `sync` is a barrier over exactly
// those threads and red holds NT / 32 floats of shared memory. Rows of up to
// NT * REGV vectors are read once into registers with all loads in flight;
// longer rows are read twice (amax pass, code pass). Returns s to every
// thread. `red` may be reused once the call returns.
template <bool BF16, int NT, int REGV, class Sync>
__device__ __forceinline__ float quantize_row(const uint4* __restrict__ xr, int nvec,
                                              const float* __restrict__ mul, int8_t* __restrict__ qr,
                                              int t, float* red, Sync sync, int slice = -1) {
    using V = Vec<BF16>;
    constexpr int E = V::E;
    const bool in_regs = nvec <= NT * REGV;
    uint4 rv[REGV];
    float amax = 0.f;
    if (in_regs) {
#pragma unroll
        for (int u = 0; u < REGV; ++u) {
            const int v = t + u * NT;
            rv[u] = v < nvec ? __ldg(xr + v) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < REGV; ++u) {
            const int v = t + u * NT;
            if (v < nvec) {
                float e[E];
                V::unpack(rv[u], e);
                apply_mul<E>(e, mul, v);
#pragma unroll
                for (int j = 0; j < E; ++j) amax = fmaxf(amax, fabsf(e[j]));
            }
        }
    } else {
        for (int v = t; v < nvec; v += NT) {
            float e[E];
            V::unpack(__ldg(xr + v), e);
            apply_mul<E>(e, mul, v);
#pragma unroll
            for (int j = 0; j < E; ++j) amax = fmaxf(amax, fabsf(e[j]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((t & 31) == 0) red[t >> 5] = amax;
    sync();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) amax = fmaxf(amax, red[w]);
    const float s = __fdiv_rn(amax, 127.0f);
    const float r = __frcp_rn(s);
    if (in_regs) {
#pragma unroll
        for (int u = 0; u < REGV; ++u) {
            const int v = t + u * NT;
            if (v < nvec && (slice < 0 || u == slice)) {
                float e[E];
                V::unpack(rv[u], e);
                apply_mul<E>(e, mul, v);
                store_codes<E>(qr, v, e, s, r);
            }
        }
    } else if (slice >= 0) {
        const int v = slice * NT + t;
        if (v < nvec) {
            float e[E];
            V::unpack(__ldg(xr + v), e);
            apply_mul<E>(e, mul, v);
            store_codes<E>(qr, v, e, s, r);
        }
    } else {
        for (int v = t; v < nvec; v += NT) {
            float e[E];
            V::unpack(__ldg(xr + v), e);
            apply_mul<E>(e, mul, v);
            store_codes<E>(qr, v, e, s, r);
        }
    }
    return s;
}

// Bring a row (and the multipliers) into L2 ahead of a grid dependency wait,
// by threads t in [0, NT). A prefetch returns nothing to the SM, and L2 is
// the point of coherence, so the reads after the wait still see current data.
template <bool BF16, int NT>
__device__ __forceinline__ void prefetch_row_l2(const uint4* xr, int nvec, const float* mul, int t) {
    constexpr int E = Vec<BF16>::E;
    for (int v = t * 8; v < nvec; v += NT * 8) {   // one 128-byte line per 8 vectors
        asm volatile("prefetch.global.L2 [%0];" :: "l"(xr + v));
        if (mul) {   // 8 vectors of multipliers span 8 * E * 4 bytes: one or two lines
            asm volatile("prefetch.global.L2 [%0];" :: "l"(mul + (size_t)v * E));
            if (E == 8) asm volatile("prefetch.global.L2 [%0];" :: "l"(mul + (size_t)v * E + 32));
        }
    }
}

}  // namespace
}  // namespace qv
