// k_layer.cu -- the non-linear steps between the quantized linears of one
// decoder layer, each fused with the per-token int8 quantization of the next
// linear's input.
//
//   Quasar, gist.science/ja summary, section 2.2 item 3: the INT8 GEMM's
//   result is dequantized back to high precision before the non-linear
//   layers, and the next linear's BF16 input is quantized online;
//   gist.science/fr summary, section 2 "Pipeline Technique".
//
// The layer follows the Qwen3-shaped decoder of the workloads with a bf16
// residual stream (the summaries do not spell it out):
//   residual_rmsnorm_quant  h = rne_bf16(h + d) (d: a linear's bf16 output),
//                           ss = sum h_k^2 in binary64, var = fl32(ss / H),
//                           rstd = fl32(1 / fl32(sqrt(fl32(var + eps)))),
//                           x_k = rne_bf16(g_k * rne_bf16(fl32(h_k * rstd))),
//                           then codes and the token scale of x (times the
//                           optional smoothing multipliers);
//   swiglu_quant            a_k = fl32(fl32(gate_k * sigma(gate_k)) * up_k) on
//                           the fp32 gate|up output, sigma(v) =
//                           fl32(1 / fl32(1 + E(-v))), then codes and scale.
// E is exp by Cody and Waite's range reduction and a degree-7 Taylor
// polynomial (layer_exp); every step is one binary32 operation in
// round-to-nearest-even (explicit _rn intrinsics, never contracted), so the
// results are determined by the definition alone. The sum of squares is the
// one place where the kernel takes another route: it adds the (exact)
// binary32 squares in float-float, which agrees with the definition's
// binary64 sum (index order) to about 2^-37 relative; var = fl32(ss / H) is
// the same unless ss / H lies that close to a binary32 rounding boundary, and
// there (about one row in 2000) one thread recomputes the definition's sum.
//
// One CTA of 512 threads per row; the row is held in registers (H up to
// 16384, F up to 32768).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kLayerThreads = 512;
constexpr int kNormVecs = 4;     // 8-bf16 vectors per thread: H <= 16384
constexpr int kGluVecs = 16;     // 4-float vectors per thread: F <= 32768

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float round_bf16(float f) { return __uint_as_float(bf16_bits(f) << 16); }

// Block-wide max of non-negative floats (all kLayerThreads threads call it).
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kLayerThreads / 32; ++w) m = fmaxf(m, red[w]);
    __syncthreads();   // red is reused
    return m;
}

// Float-float (hi, lo) sums built from Knuth's error-free TwoSum: hi + lo
// carries about 48 significant bits. Explicit _rn operations: a contracted
// or reassociated step would lose the error term.
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, float b) {
    const float t = __fadd_rn(a.hi, b);
    const float bv = __fsub_rn(t, a.hi);
    const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(t, bv)), __fsub_rn(b, bv));
    return FF{t, __fadd_rn(a.lo, err)};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    FF r = ff_add(a, b.hi);
    r.lo = __fadd_rn(r.lo, b.lo);
    return r;
}

// sum_k h_k^2 of a row: every square of a bf16 value is exact in binary32;
// the squares are added in float-float and the block's total returned, to
// every thread, as the binary64 value hi + lo. It agrees with a binary64 sum
// in any order to about 2^-47 relative.
__device__ __forceinline__ double block_sum_squares(FF v, FF* red, double* total) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        FF o;
        o.hi = __shfl_xor_sync(0xffffffffu, v.hi, off);
        o.lo = __shfl_xor_sync(0xffffffffu, v.lo, off);
        v = ff_add(v, o);
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        FF w = threadIdx.x < kLayerThreads / 32 ? red[threadIdx.x] : FF{0.0f, 0.0f};
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
            FF o;
            o.hi = __shfl_xor_sync(0xffffffffu, w.hi, off);
            o.lo = __shfl_xor_sync(0xffffffffu, w.lo, off);
            w = ff_add(w, o);
        }
        if (threadIdx.x == 0) *total = __dadd_rn((double)w.hi, (double)w.lo);
    }
    __syncthreads();
    return *total;
}

// Whether a non-negative binary64 value q lies within 2^-36 q of a point
// where rounding to binary32 changes (the midpoint between two neighbouring
// binary32 values). Error bounds for ss: the sequential binary64 sum of the
// definition is within (H - 1) 2^-53 ss <= 2^-39 ss of the exact sum for
// H <= 16384; the float-float sum is within about 2^-38 ss of it (per-thread
// lo parts gather at most n^2 2^-48 with n <= 32 terms, the tree merges add
// less); q is then rounded once more to binary64. 2^-36 covers all three.
__device__ __forceinline__ bool near_binary32_midpoint(double q) {
    if (!(q > 0.0)) return false;
    const float f = __double2float_rn(q);
    const uint32_t b = __float_as_uint(f);
    if (b >= 0x7F7FFFFFu) return false;                  // FLT_MAX or infinity: not a workload value
    if (b == 0u) return true;                            // below half the least subnormal
    const double fd = (double)f;
    const double up = (double)__uint_as_float(b + 1u);
    const double dn = (double)__uint_as_float(b - 1u);
    const double mid_up = __dadd_rn(fd, __dmul_rn(__dsub_rn(up, fd), 0.5));
    const double mid_dn = __dadd_rn(fd, __dmul_rn(__dsub_rn(dn, fd), 0.5));
    const double d = fmin(fabs(__dsub_rn(q, mid_up)), fabs(__dsub_rn(q, mid_dn)));
    return d <= __dmul_rn(q, 0x1p-36);
}

// The definition's sum of squares of a bf16 row: binary64, index order (one
// thread; the rare exact path of the RMSNorm).
__device__ __noinline__ double sum_squares_in_order(const uint4* hr, int nvec) {
    double s = 0.0;
    for (int v = 0; v < nvec; ++v) {
        const uint4 w4 = hr[v];
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const double a = (double)bf16_lo(w[j]), b = (double)bf16_hi(w[j]);
            s = __dadd_rn(s, __dmul_rn(a, a));
            s = __dadd_rn(s, __dmul_rn(b, b));
        }
    }
    return s;
}

__device__ __forceinline__ uint32_t pack_codes4(float a, float b, float c, float d, float s, float r) {
    // the fast rule for all four, the IEEE quotient only near a half-integer
    const float e[4] = {a, b, c, d};
    int q[4];
    unsigned near_mask = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        bool nb;
        q[j] = quant_code_fast(e[j], r, nb);
        near_mask |= (unsigned)nb << j;
    }
    if (s == 0.f) {
        return 0u;
    } else if (near_mask) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if ((near_mask >> j) & 1u) q[j] = quant_code_exact(e[j], s);
    }
    return (uint32_t)(uint8_t)(int8_t)q[0] | ((uint32_t)(uint8_t)(int8_t)q[1] << 8) |
           ((uint32_t)(uint8_t)(int8_t)q[2] << 16) | ((uint32_t)(uint8_t)(int8_t)q[3] << 24);
}

__global__ void __launch_bounds__(kLayerThreads)
residual_rmsnorm_quant_kernel(uint16_t* __restrict__ h, const uint16_t* __restrict__ delta,
                              const uint16_t* __restrict__ gamma, float eps, const float* __restrict__ mul,
                              int H, int8_t* __restrict__ xq, float* __restrict__ sx,
                              uint16_t* __restrict__ x_out) {
    const int row = blockIdx.x, tid = threadIdx.x;
    const int nvec = H / 8;
    uint4* hr = reinterpret_cast<uint4*>(h + (size_t)row * H);
    const uint4* dr = delta ? reinterpret_cast<const uint4*>(delta + (size_t)row * H) : nullptr;
    for (int v = tid * 8; v < nvec; v += kLayerThreads * 8) {     // one 128-byte line per 8 vectors
        asm volatile("prefetch.global.L2 [%0];" :: "l"(hr + v));
        if (dr) asm volatile("prefetch.global.L2 [%0];" :: "l"(dr + v));
    }
    grid_dependency_wait();
    allow_dependent_launch();   // the next GEMM starts after the previous kernel (as in k_quant.cu)
    __shared__ FF red_ff[kLayerThreads / 32];
    __shared__ float red_f[kLayerThreads / 32];
    __shared__ double ss_total;
    __shared__ float rstd_s;

    uint4 hv[kNormVecs], gv[kNormVecs];
    FF ss{0.0f, 0.0f};
#pragma unroll
    for (int u = 0; u < kNormVecs; ++u) {
        const int v = tid + u * kLayerThreads;
        hv[u] = make_uint4(0u, 0u, 0u, 0u);
        gv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (v < nvec) {
            // the norm weights travel with the row: their latency hides behind the reduction
            gv[u] = reinterpret_cast<const uint4*>(gamma)[v];
            hv[u] = hr[v];
            if (dr) {
                const uint4 dv = dr[v];
                uint32_t* w = reinterpret_cast<uint32_t*>(&hv[u]);
                const uint32_t* dw = reinterpret_cast<const uint32_t*>(&dv);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t lo = bf16_bits(__fadd_rn(bf16_lo(w[j]), bf16_lo(dw[j])));
                    const uint32_t hi = bf16_bits(__fadd_rn(bf16_hi(w[j]), bf16_hi(dw[j])));
                    w[j] = lo | (hi << 16);
                }
                hr[v] = hv[u];
            }
            const uint32_t* w = reinterpret_cast<const uint32_t*>(&hv[u]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
                ss = ff_add(ss, __fmul_rn(a, a));     // exact: 8-bit significands
                ss = ff_add(ss, __fmul_rn(b, b));
            }
        }
    }
    const double sum = block_sum_squares(ss, red_ff, &ss_total);
    if (tid == 0) {
        // ss / H; for H = 2^k that is the exact scaling by 2^-k (bits of the
        // binary64 power of two: exponent field 1023 - k), no division
        double q;
        if ((H & (H - 1)) == 0)
            q = __dmul_rn(sum, __longlong_as_double((long long)(1023 - (__ffs(H) - 1)) << 52));
        else
            q = __ddiv_rn(sum, (double)H);
        if (near_binary32_midpoint(q)) q = __ddiv_rn(sum_squares_in_order(hr, nvec), (double)H);
        const float var = __double2float_rn(q);
        rstd_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
    }
    __syncthreads();
    const float rstd = rstd_s;

    // x = rne_bf16(g * rne_bf16(h * rstd)), then the optional multipliers
    float xv[kNormVecs][8];
    float amax = 0.0f;
#pragma unroll
    for (int u = 0; u < kNormVecs; ++u) {
        const int v = tid + u * kLayerThreads;
#pragma unroll
        for (int j = 0; j < 8; ++j) xv[u][j] = 0.0f;
        if (v < nvec) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(&hv[u]);
            const uint32_t* gw = reinterpret_cast<const uint32_t*>(&gv[u]);
            uint32_t xb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float lo = round_bf16(__fmul_rn(bf16_lo(gw[j]), round_bf16(__fmul_rn(bf16_lo(w[j]), rstd))));
                const float hi = round_bf16(__fmul_rn(bf16_hi(gw[j]), round_bf16(__fmul_rn(bf16_hi(w[j]), rstd))));
                xb[j] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
                xv[u][2 * j] = lo;
                xv[u][2 * j + 1] = hi;
            }
            if (x_out) reinterpret_cast<uint4*>(x_out + (size_t)row * H)[v] = make_uint4(xb[0], xb[1], xb[2], xb[3]);
            if (mul) {
#pragma unroll
                for (int j = 0; j < 8; ++j) xv[u][j] = __fmul_rn(xv[u][j], __ldg(mul + v * 8 + j));
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(xv[u][j]));
        }
    }
    amax = block_max(amax, red_f);
    const float s = __fdiv_rn(amax, 127.0f);
    const float r = __frcp_rn(s);
    if (tid == 0) sx[row] = s;
    int8_t* qr = xq + (size_t)row * H;
#pragma unroll
    for (int u = 0; u < kNormVecs; ++u) {
        const int v = tid + u * kLayerThreads;
        if (v < nvec)
            *reinterpret_cast<uint2*>(qr + v * 8) =
                make_uint2(pack_codes4(xv[u][0], xv[u][1], xv[u][2], xv[u][3], s, r),
                           pack_codes4(xv[u][4], xv[u][5], xv[u][6], xv[u][7], s, r));
    }
}

__global__ void __launch_bounds__(kLayerThreads)
swiglu_quant_kernel(const float* __restrict__ gate_up, int F, int8_t* __restrict__ xq, float* __restrict__ sx) {
    const int row = blockIdx.x, tid = threadIdx.x;
    const int nvec = F / 4;
    const float4* gr = reinterpret_cast<const float4*>(gate_up + (size_t)row * 2 * F);
    const float4* ur = gr + nvec;
    for (int v = tid * 8; v < nvec; v += kLayerThreads * 8) {     // one 128-byte line per 8 vectors
        asm volatile("prefetch.global.L2 [%0];" :: "l"(gr + v));
        asm volatile("prefetch.global.L2 [%0];" :: "l"(ur + v));
    }
    grid_dependency_wait();
    allow_dependent_launch();   // the next GEMM starts after the previous kernel (as in k_quant.cu)
    __shared__ float red_f[kLayerThreads / 32];

    float4 av[kGluVecs];
    float amax = 0.0f;
#pragma unroll
    for (int u = 0; u < kGluVecs; ++u) {
        const int v = tid + u * kLayerThreads;
        av[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (v < nvec) {
            const float4 g = gr[v], up = ur[v];
            av[u] = make_float4(__fmul_rn(silu(g.x), up.x), __fmul_rn(silu(g.y), up.y),
                                __fmul_rn(silu(g.z), up.z), __fmul_rn(silu(g.w), up.w));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(av[u].x), fabsf(av[u].y)), fmaxf(fabsf(av[u].z), fabsf(av[u].w))));
        }
    }
    amax = block_max(amax, red_f);
    const float s = __fdiv_rn(amax, 127.0f);
    const float r = __frcp_rn(s);
    if (tid == 0) sx[row] = s;
    int8_t* qr = xq + (size_t)row * F;
#pragma unroll
    for (int u = 0; u < kGluVecs; ++u) {
        const int v = tid + u * kLayerThreads;
        if (v < nvec)
            *reinterpret_cast<uint32_t*>(qr + v * 4) = pack_codes4(av[u].x, av[u].y, av[u].z, av[u].w, s, r);
    }
}

cudaError_t launch_pdl(const void* kernel, int rows, void** args, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(rows);
    cfg.blockDim = dim3(kLayerThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace

cudaError_t launch_residual_rmsnorm_quant(uint16_t* h, const uint16_t* delta, const uint16_t* gamma, float eps,
                                          const float* mul, int M, int H, int8_t* xq, float* sx,
                                          uint16_t* x_out, cudaStream_t s) {
    void* args[] = {&h, &delta, &gamma, &eps, &mul, &H, &xq, &sx, &x_out};
    return launch_pdl(reinterpret_cast<const void*>(residual_rmsnorm_quant_kernel), M, args, s);
}

cudaError_t launch_swiglu_quant(const float* gate_up, int M, int F, int8_t* xq, float* sx, cudaStream_t s) {
    void* args[] = {&gate_up, &F, &xq, &sx};
    return launch_pdl(reinterpret_cast<const void*>(swiglu_quant_kernel), M, args, s);
}

}  // namespace qv
