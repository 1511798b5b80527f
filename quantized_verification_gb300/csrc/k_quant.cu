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
#include "quant_common.cuh"

namespace qv {
namespace {

constexpr int kQuantThreads = 512;
constexpr int kQuantRegVecs = 4;   // 16-byte vectors per thread kept in registers

template <bool BF16>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rows_kernel(const uint8_t* __restrict__ x, int K, const float* __restrict__ mul,
                     int8_t* __restrict__ q, float* __restrict__ scale, int early_dependents) {
    if (early_dependents) allow_dependent_launch();
    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    const int nvec = K / Vec<BF16>::E;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * K * (BF16 ? 2 : 4));
    // Bring the row into L2 while the preceding kernel finishes.
    if (nvec <= kQuantThreads * kQuantRegVecs) prefetch_row_l2<BF16, kQuantThreads>(xr, nvec, mul, tid);
    grid_dependency_wait();
    __shared__ float warp_max[kQuantThreads / 32];
    const float s = quantize_row<BF16, kQuantThreads, kQuantRegVecs>(xr, nvec, mul, q + (size_t)row * K, tid,
                                                                     warp_max, [] { __syncthreads(); });
    if (tid == 0) scale[row] = s;
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
