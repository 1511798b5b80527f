// k_fidelity.cu -- logit-fidelity diagnostic: KL(p || q) between the softmax
// of a reference verifier's logits (p) and of the quantized verifier's (q),
// and both top-1 tokens.
//
//   The Quasar summaries report that quantizing the verifier keeps the logit
//   distribution (negligible KL divergence: gist.science/fr summary,
//   contributions item 3; high logit-distribution similarity: shd-paper.top
//   summary, method details, core idea). This kernel measures that on given logits.
//
// A thread-block cluster of kFidCluster CTAs per row; CTA r owns the r-th
// contiguous slice of the row (a multiple of 4 entries long, read as float4
// when the row is 16-byte aligned, and kept in shared memory after the first
// pass when it fits). Three passes over the slice, each closed by a
// cluster-wide combine through distributed shared memory:
//   1. the maxima of a and b;
//   2. Z = sum e^(a_v - max a), the p-mean of d_v = b_v - a_v,
//      c = sum e^(a_v - max a) d_v / Z, and the lowest index holding each
//      maximum (the top-1 tokens; +0 and -0 compare equal);
//   3. KL = log1p(sum e^(a_v - max a) expm1(d_v - c) / Z) - (E_p[d] - c).
// Pass 3 is the identity KL(p || q) = log E_p[e^(d - c)] - E_p[d - c], true
// for any c; with c the binary32 rounding of E_p[d] the last term is that
// rounding's residual (binary64), which cancels its first-order effect on
// the first. Nothing subtracts two large numbers, so KL values far below the
// size of the logits keep their relative accuracy. Per-thread sums are
// binary32; the CTA sums are pairs of binary32 numbers (about 48 bits,
// turned into binary64), and the cluster adds them in binary64, in rank
// order, in one thread.

#include <cuda_runtime.h>
#include <cooperative_groups.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

namespace cg = cooperative_groups;

constexpr int kFidThreads = 1024;
constexpr int kFidCluster = 16;                  // CTAs per row (a non-portable cluster size)
constexpr size_t kFidCacheBytes = 200 * 1024;    // the largest slice kept in shared memory (a and b)
constexpr int kNoIndex = 0x7FFFFFFF;

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// The CTA's reduction of two values by a commutative op: butterfly shuffles
// within each warp, then warp 0 over the 32 warp results; valid (and the
// same) in every lane of warp 0.
template <class T, class Op>
__device__ __forceinline__ void warp0_reduce2(T& x, T& y, T* sm /* [2][32] */, Op op) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        x = op(x, __shfl_xor_sync(0xffffffffu, x, off));
        y = op(y, __shfl_xor_sync(0xffffffffu, y, off));
    }
    if (lane == 0) {
        sm[warp] = x;
        sm[32 + warp] = y;
    }
    __syncthreads();
    if (warp == 0) {
        x = sm[lane];
        y = sm[32 + lane];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            x = op(x, __shfl_xor_sync(0xffffffffu, x, off));
            y = op(y, __shfl_xor_sync(0xffffffffu, y, off));
        }
    }
}

// A sum carried as an unevaluated pair hi + lo of binary32 numbers
// (|lo| <= half an ulp of hi, about 48 significant bits). f2_add adds two
// pairs: Knuth's TwoSum gives the exact rounding error of hi_a + hi_b, the
// low parts are added to it, and Dekker's Fast2Sum renormalises. Every step
// is symmetric in its operands, so both lanes of a butterfly shuffle get the
// same pair. Binary32 arithmetic only: binary64 is slow on this GPU.
struct F2 {
    float hi, lo;
};
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    const float e = (a.hi - (s - bb)) + (b.hi - bb);
    const float l = e + (a.lo + b.lo);
    const float h = s + l;
    return {h, l - (h - s)};
}
__device__ __forceinline__ F2 f2_warp_sum(F2 v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v = f2_add(v, F2{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)});
    return v;
}

// The CTA's sums of NV binary32 per-thread values as binary64 numbers, the
// same in every lane of warp 0 (the only warp where the result is valid):
// butterfly trees of pairs within each warp, then over the 32 warp sums.
template <int NV>
__device__ __forceinline__ void warp0_sum(const float (&v)[NV], double (&out)[NV], float2* sm /* [NV][32] */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const F2 t = f2_warp_sum(F2{v[i], 0.f});
        if (lane == 0) sm[i * 32 + warp] = make_float2(t.hi, t.lo);
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const float2 w = sm[i * 32 + lane];
            const F2 t = f2_warp_sum(F2{w.x, w.y});
            out[i] = (double)t.hi + (double)t.lo;
        }
    }
}

// Visits the entries of [lo, hi) this thread owns: fv(v, x, y) on the
// float4-loaded part (the first 4*n4 entries), ft(v, x, y) on the scalar
// rest. Src 0 reads the row; Src 1 reads it and keeps this thread's float4s
// in shared memory (sa, sb); Src 2 reads them back from there and stores
// what fv leaves in x and y in their place; Src 3 only reads them back. A
// thread only ever reads back what it stored itself.
template <int Src, class FV, class FT>
__device__ __forceinline__ void for_slice(const float* __restrict__ ar, const float* __restrict__ br,
                                          float4* sa, float4* sb, int lo, int n4, int hi, FV&& fv, FT&& ft) {
    const float4* a4 = reinterpret_cast<const float4*>(ar + lo);
    const float4* b4 = reinterpret_cast<const float4*>(br + lo);
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kFidThreads) {
        float4 x, y;
        if (Src >= 2) {
            x = sa[i];
            y = sb[i];
        } else {
            x = a4[i];
            y = b4[i];
            if (Src == 1) {
                sa[i] = x;
                sb[i] = y;
            }
        }
        const int v = lo + 4 * i;
        fv(v, x.x, y.x);
        fv(v + 1, x.y, y.y);
        fv(v + 2, x.z, y.z);
        fv(v + 3, x.w, y.w);
        if (Src == 2) {
            sa[i] = x;
            sb[i] = y;
        }
    }
    for (int v = lo + 4 * n4 + (int)threadIdx.x; v < hi; v += kFidThreads) {
        float x = ar[v], y = br[v];
        ft(v, x, y);
    }
}

__global__ void __launch_bounds__(kFidThreads) logit_fidelity_kernel(const float* __restrict__ a,
                                                                      const float* __restrict__ b, int V,
                                                                      float* __restrict__ kl,
                                                                      int32_t* __restrict__ top_a,
                                                                      int32_t* __restrict__ top_b, int cap4) {
    extern __shared__ float4 fid_cache[];    // [2][cap4]: this CTA's slice of a, then of b
    __shared__ float sm_f[2 * 32];
    __shared__ int sm_i[2 * 32];
    __shared__ float2 sm_f2[2 * 32];
    // written by every CTA of the row, each into its own rank's entry
    __shared__ float c_ma[kFidCluster], c_mb[kFidCluster];
    __shared__ int c_ia[kFidCluster], c_ib[kFidCluster];
    __shared__ double c_z[kFidCluster], c_s1[kFidCluster], c_s2[kFidCluster];
    __shared__ float s_c;
    cg::cluster_group cluster = cg::this_cluster();
    cluster_arrive_relaxed();    // waited for before the first store into another CTA
    allow_dependent_launch();
    grid_dependency_wait();

    const int rank = (int)cluster.block_rank();
    const size_t row = blockIdx.x / kFidCluster;
    const float* ar = a + row * (size_t)V;
    const float* br = b + row * (size_t)V;
    const int per = (((V + kFidCluster - 1) / kFidCluster) + 3) & ~3;
    const int lo = min(V, rank * per), hi = min(V, lo + per);
    const bool vec = ((reinterpret_cast<uintptr_t>(ar) | reinterpret_cast<uintptr_t>(br)) & 15u) == 0;
    const int n4 = vec ? (hi - lo) >> 2 : 0;
    // Passes 2 and 3 read the slice from shared memory; pass 2 leaves
    // e_v = e^(a_v - max a) and d_v there for pass 3.
    const bool cached = n4 > 0 && n4 <= cap4;
    float4* sa = fid_cache;
    float4* sb = fid_cache + cap4;
    auto fmax_op = [](float x, float y) { return fmaxf(x, y); };
    auto imin_op = [](int x, int y) { return min(x, y); };

    // ---- 1. the maxima, pushed to every CTA of the row
    const float NEG_INF = -__uint_as_float(0x7F800000u);
    float ma = NEG_INF, mb = NEG_INF;
    auto maxima = [&](int, float& x, float& y) {
        ma = fmaxf(ma, x);
        mb = fmaxf(mb, y);
    };
    if (cached)
        for_slice<1>(ar, br, sa, sb, lo, n4, hi, maxima, maxima);
    else
        for_slice<0>(ar, br, sa, sb, lo, n4, hi, maxima, maxima);
    warp0_reduce2(ma, mb, sm_f, fmax_op);
    cluster_wait();              // every CTA of the cluster has started
    if (threadIdx.x < kFidCluster) {
        *cluster.map_shared_rank(c_ma + rank, (unsigned)threadIdx.x) = ma;
        *cluster.map_shared_rank(c_mb + rank, (unsigned)threadIdx.x) = mb;
    }
    cluster.sync();
    ma = c_ma[0];
    mb = c_mb[0];
#pragma unroll
    for (int r = 1; r < kFidCluster; ++r) {
        ma = fmaxf(ma, c_ma[r]);
        mb = fmaxf(mb, c_mb[r]);
    }

    // ---- 2. Z, E_p[d] and the first index of each maximum; warp 0 pushes
    // this CTA's results, then thread 0 combines the row's in rank order
    float z = 0.f, s1 = 0.f;
    int ia = kNoIndex, ib = kNoIndex;
    auto moments = [&](int v, float& x, float& y) {
        if (x == ma) ia = min(ia, v);
        if (y == mb) ib = min(ib, v);
        const float e = expf(x - ma), d = y - x;
        z += e;
        s1 += e * d;
        x = e;
        y = d;
    };
    if (cached)
        for_slice<2>(ar, br, sa, sb, lo, n4, hi, moments, moments);
    else
        for_slice<0>(ar, br, sa, sb, lo, n4, hi, moments, moments);
    double zs[2];
    warp0_sum<2>({z, s1}, zs, sm_f2);
    warp0_reduce2(ia, ib, sm_i, imin_op);
    if (threadIdx.x < kFidCluster) {
        *cluster.map_shared_rank(c_z + rank, (unsigned)threadIdx.x) = zs[0];
        *cluster.map_shared_rank(c_s1 + rank, (unsigned)threadIdx.x) = zs[1];
        *cluster.map_shared_rank(c_ia + rank, (unsigned)threadIdx.x) = ia;
        *cluster.map_shared_rank(c_ib + rank, (unsigned)threadIdx.x) = ib;
    }
    cluster.sync();
    double Z = 0.0, S1 = 0.0;
    if (threadIdx.x == 0) {
        for (int r = 0; r < kFidCluster; ++r) {
            Z += c_z[r];
            S1 += c_s1[r];
            ia = min(ia, c_ia[r]);
            ib = min(ib, c_ib[r]);
        }
        s_c = (float)(S1 / Z);
    }
    __syncthreads();
    const float c = s_c;

    // ---- 3. E_p[expm1(d - c)], combined in CTA 0 of the cluster
    float s2 = 0.f;
    auto excess = [&](int, float& x, float& y) { s2 += expf(x - ma) * expm1f((y - x) - c); };
    auto excess_kept = [&](int, float& e, float& d) { s2 += e * expm1f(d - c); };
    if (cached)
        for_slice<3>(ar, br, sa, sb, lo, n4, hi, excess_kept, excess);
    else
        for_slice<0>(ar, br, sa, sb, lo, n4, hi, excess, excess);
    double s2s[1];
    warp0_sum<1>({s2}, s2s, sm_f2);
    if (threadIdx.x == 0) *cluster.map_shared_rank(c_s2 + rank, 0u) = s2s[0];
    cluster.sync();              // the last cross-CTA access: every push into CTA 0 has landed
    if (rank == 0 && threadIdx.x == 0) {
        double S2 = 0.0;
        for (int r = 0; r < kFidCluster; ++r) S2 += c_s2[r];
        kl[row] = (float)(log1p(S2 / Z) - (S1 / Z - (double)c));
        top_a[row] = ia;
        top_b[row] = ib;
    }
}

}  // namespace

cudaError_t launch_logit_fidelity(const float* a, const float* b, int M, int V, float* kl, int32_t* top_a,
                                  int32_t* top_b, cudaStream_t s) {
    // Keep each CTA's slice in shared memory when it fits (the Qwen3
    // vocabulary: 9496 entries of a and of b, 76 KB); else every pass reads
    // the row again (from L2 at the step's sizes).
    const int per = (((V + kFidCluster - 1) / kFidCluster) + 3) & ~3;
    int cap4 = per / 4;
    size_t smem = (size_t)cap4 * 2 * sizeof(float4);
    if (smem > kFidCacheBytes) {
        cap4 = 0;
        smem = 0;
    }
    cudaError_t e =
        cudaFuncSetAttribute(logit_fidelity_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(logit_fidelity_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)M * kFidCluster);
    cfg.blockDim = dim3(kFidThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kFidCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, logit_fidelity_kernel, a, b, V, kl, top_a, top_b, cap4);
}

}  // namespace qv
