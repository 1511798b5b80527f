// k_tree.cu -- greedy (T = 0) verification of a draft tree.
//
//   Tree-structured verification is the extension the summaries name for
//   the drafts (gist.science/de and gist.science/ja summaries, section 5);
//   along each root path the rule is the linear acceptance of
//   gist.science/fr summary, lay explanation.
//
// Tree b has N nodes; node 0 is the root (the last accepted position); node
// i >= 1 has parent par[i] (valid when in [0, i)) and drafted token d[i];
// t[i] is the verifier's greedy token after node i's root path. Node i is
// accepted when every node j on its path (j != 0) has a valid parent p and
// d[j] == t[p]. The result is the accepted node of largest depth (lowest
// index among them): len = depth + 1, out = the drafted tokens on its path,
// then t[best], then -1.
//
// One CTA per tree, one thread per node: each thread walks up its own path
// (parents strictly decrease, so the walk ends); a block-wide max of the key
// depth * 2^16 + (65535 - i) picks the best node.

#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int kTreeThreads = 1024;

__global__ void __launch_bounds__(kTreeThreads)
tree_accept_kernel(const int32_t* __restrict__ t, const int32_t* __restrict__ d, const int32_t* __restrict__ par,
                   int N, int32_t* __restrict__ len, int32_t* __restrict__ out, int32_t* __restrict__ node) {
    allow_dependent_launch();
    grid_dependency_wait();
    __shared__ unsigned red[kTreeThreads / 32];
    const int b = blockIdx.x, i = threadIdx.x;
    const int32_t* tb = t + (size_t)b * N;
    const int32_t* db = d + (size_t)b * N;
    const int32_t* pb = par + (size_t)b * N;

    unsigned key = 0;
    if (i < N) {
        bool ok = true;
        int depth = 0, j = i;
        while (j != 0) {
            const int p = pb[j];
            if (p < 0 || p >= j) { ok = false; break; }
            if (db[j] != tb[p]) { ok = false; break; }
            ++depth;
            j = p;
        }
        if (ok) key = ((unsigned)depth << 16) | (0xFFFFu - (unsigned)i);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
    if ((i & 31) == 0) red[i >> 5] = key;
    __syncthreads();
    if (i == 0) {
        unsigned k = red[0];
        for (int w = 1; w < kTreeThreads / 32; ++w) k = max(k, red[w]);
        const int best = (int)(0xFFFFu - (k & 0xFFFFu));
        const int D = (int)(k >> 16);
        len[b] = D + 1;
        int32_t* ob = out + (size_t)b * N;
        for (int j = D + 1; j < N; ++j) ob[j] = -1;
        ob[D] = tb[best];
        int j = best;
        for (int s = D - 1; s >= 0; --s) {
            ob[s] = db[j];
            j = pb[j];
        }
        if (node) node[b] = best;
    }
}

}  // namespace

cudaError_t launch_tree_accept(const int32_t* t, const int32_t* d, const int32_t* par, int B, int N,
                               int32_t* len, int32_t* out, int32_t* node, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(kTreeThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tree_accept_kernel, t, d, par, N, len, out, node);
}

}  // namespace qv
