// k_accept.cu -- a4: greedy acceptance of the longest matching draft prefix
// plus the verifier's token at the first mismatch (the "bonus" token).
//
//   Quasar, gist.science/fr summary, lay explanation (a wrong draft token is
//   rejected and generation resumes from the verifier's token); at least one
//   token per step (L ~ 1.03 for a nearly useless verifier, gist.science/ja
//   summary, section 4); at T = 0 the lossless rejection-sampling test of
//   gist.science/it summary, section 2 item 3 is exact matching.
//
// One thread per sequence: the work is a handful of integer compares per
// sequence, so the kernel is bound by launch latency, not by the GPU.

#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kAcceptThreads = 128;

__global__ void __launch_bounds__(kAcceptThreads)
accept_kernel(const int32_t* __restrict__ t, const int32_t* __restrict__ d, int B, int gamma,
              int32_t* __restrict__ len, int32_t* __restrict__ out) {
    allow_dependent_launch();
    grid_dependency_wait();
    const int b = blockIdx.x * kAcceptThreads + threadIdx.x;
    if (b >= B) return;
    const int G = gamma + 1;
    const int32_t* tb = t + (size_t)b * G;
    const int32_t* db = d + (size_t)b * gamma;
    int k = 0;
    while (k < gamma && db[k] == tb[k]) ++k;
    len[b] = k + 1;
    int32_t* ob = out + (size_t)b * G;
    for (int j = 0; j < G; ++j) ob[j] = j <= k ? tb[j] : -1;
}

}  // namespace

cudaError_t launch_accept(const int32_t* t, const int32_t* d, int B, int gamma, int32_t* len,
                          int32_t* out, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((B + kAcceptThreads - 1) / kAcceptThreads);
    cfg.blockDim = dim3(kAcceptThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_kernel, t, d, B, gamma, len, out);
}

}  // namespace qv
