// k_quant.cu -- per-row symmetric int8 quantization (a1 activations, one row
// per token; a0 weights, one row per output channel).
//
//   Quasar, gist.science/ja summary, section 2.2 "Enhanced SmoothQuant",
//   items 2-3: weights quantized to INT8 offline; BF16 activations scaled by
//   the smoothing factor and converted to INT8 online.
//
// CTAs of 512 threads. A weight row takes one CTA. An activation row takes
// S = ceil(K / (8 * 512)) CTAs (bf16; K / (4 * 512) for fp32): each reads the
// whole row for amax (every CTA of the row finds the same value) and writes
// the codes of its own slice of 512 16-byte vectors; CTA 0 writes the scale.
// Rows of up to 512 x 4 16-byte vectors (16384 bf16 / 8192 fp32 elements)
// are read once into registers with all loads in flight together; longer
// rows are read twice (amax pass, code pass). amax = max |x * c| is reduced
// with warp shuffles and one shared-memory step. Every floating point step
// is a single IEEE operation in round-to-nearest-even:
//   s = fl(amax / 127), q = clamp(rne(fl(x' / s)), -127, 127), q = 0 if s == 0,
// where the quotient's rounding is decided from fl(x' * fl(1 / s)) unless
// that product lies within 2^-20 of a half-integer (then from the quotient
// itself; quant_code_fast in qv_ptx.cuh gives the error bound).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"
#include "quant_common.cuh"

namespace qv {
namespace {

// Weight rows (setup): one 512-thread CTA per row.
constexpr int kQuantThreads = 512;
constexpr int kQuantRegVecs = 4;   // 16-byte vectors per thread kept in registers
// Activation rows: S = ceil(nvec / 512) CTAs of 512 threads per row, so the
// code work of a long row (K = 12288: three CTAs) runs on several SMs.
// (Smaller CTAs fit beside a resident GEMM CTA but measured slower: their
// loads share the SM with that CTA's weight-ring fill.)
constexpr int kActThreads = 512;
constexpr int kActRegVecs = 4;

// blockIdx.x = row * S + j. With S > 1, CTA j of a row computes the whole
// row's amax (identical in every CTA of the row) and writes the codes of
// vectors [j * NT, (j + 1) * NT) only; CTA 0 writes the scale.
template <bool BF16, int NT, int REGV>
__global__ void __launch_bounds__(NT)
quantize_rows_kernel(const uint8_t* __restrict__ x, int K, const float* __restrict__ mul,
                     int8_t* __restrict__ q, float* __restrict__ scale, int early_dependents, int S) {
    const int row = blockIdx.x / S;
    const int j = blockIdx.x - row * S;
    const int tid = threadIdx.x;
    const int nvec = K / Vec<BF16>::E;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)row * K * (BF16 ? 2 : 4));
    // Bring the row into L2 while the preceding kernel finishes.
    if (nvec <= NT * REGV) {
        if (S > 1) {
            if (j * NT < nvec)
                prefetch_row_l2<BF16, NT>(xr + j * NT, min(NT, nvec - j * NT), mul ? mul + (size_t)j * NT * Vec<BF16>::E : nullptr, tid);
        } else {
            prefetch_row_l2<BF16, NT>(xr, nvec, mul, tid);
        }
    }
    grid_dependency_wait();
    // The GEMM that reads these codes may launch now, not earlier: its CTAs
    // then take SMs and request their first weight tiles only once the
    // preceding kernel has finished, instead of taking HBM from that kernel's
    // last CTAs (the 5-token step measured 0.5 % faster, two GB300s; with the
    // trigger at the start, or with 6 or more early tiles, it was slower).
    if (early_dependents) allow_dependent_launch();
    __shared__ float warp_max[NT / 32];
    const float s = quantize_row<BF16, NT, REGV>(xr, nvec, mul, q + (size_t)row * K, tid, warp_max,
                                                 [] { __syncthreads(); }, S > 1 ? j : -1);
    if (tid == 0 && j == 0) scale[row] = s;
}

}  // namespace

cudaError_t launch_quantize_rows(const void* x, bool bf16, int rows, int K, const float* mul,
                                 int8_t* q, float* scale, bool early_dependents, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    const int early = early_dependents ? 1 : 0;
    if (early_dependents) {
        // activations: the row's code work spread over S CTAs
        const int nvec = K / (bf16 ? 8 : 4);
        const int S = (nvec + kActThreads - 1) / kActThreads;
        cfg.gridDim = dim3(rows * S);
        cfg.blockDim = dim3(kActThreads);
        if (bf16) return cudaLaunchKernelEx(&cfg, quantize_rows_kernel<true, kActThreads, kActRegVecs>, xb, K, mul, q, scale, early, S);
        return cudaLaunchKernelEx(&cfg, quantize_rows_kernel<false, kActThreads, kActRegVecs>, xb, K, mul, q, scale, early, S);
    }
    cfg.gridDim = dim3(rows);
    cfg.blockDim = dim3(kQuantThreads);
    if (bf16) return cudaLaunchKernelEx(&cfg, quantize_rows_kernel<true, kQuantThreads, kQuantRegVecs>, xb, K, mul, q, scale, early, 1);
    return cudaLaunchKernelEx(&cfg, quantize_rows_kernel<false, kQuantThreads, kQuantRegVecs>, xb, K, mul, q, scale, early, 1);
}

}  // namespace qv
