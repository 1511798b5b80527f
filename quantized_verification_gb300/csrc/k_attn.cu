// k_attn.cu -- attention over a short KV cache for the verify tokens.
//
//   The decoder layer that the verify pass runs between the quantized
//   linears (Quasar, gist.science/ja summary, section 2.2 item 3: the
//   non-GEMM computation stays in high precision). The summaries do not
//   spell attention out; this is causal grouped-query scaled dot-product
//   attention: token j of a sequence attends to the sequence's cached
//   positions and to the step's tokens 0..j; query head h reads key/value
//   head h / (Hq / Hkv).
//
// Inputs are the qkv projection's bf16 output rows (Hq query heads, then Hkv
// key heads, then Hkv value heads, D values each) and bf16 caches
// [B][Lmax][Hkv][D]. One launch; a thread-block cluster of C = 8 CTAs
// per (sequence, key/value head) covers the R = T * G query rows of that
// head group (G = Hq / Hkv):
//   - the S = len + T key positions are cut into C equal ranges,
//     one per CTA; a CTA streams its range in sub-chunks of kSub keys
//     through a two-stage cp.async ring (keys and values together, 16-byte
//     pieces, rows padded by 16 bytes so that ldmatrix rows fall on distinct
//     banks);
//   - scores Q K^T on the bf16 tensor cores (mma.sync m16n8k16, fp32
//     accumulation: the bf16 products are exact, the sum is a binary32 sum),
//     scaled and masked (causal, and key positions past S);
//   - online softmax per row: running max m, running sum l, running output
//     o rescaled by e^(m_old - m_new) at each sub-chunk;
//   - P V on the tensor cores with P split into two bf16 parts,
//     P = hi + mid + r with |r| <= 2^-18 P, so the product's error is below
//     2^-18 max|v| (values are bf16, exact);
//   - the cluster's partials (m, l, o per row) are exchanged through
//     distributed shared memory: CTA k merges dims [k D / C, (k + 1) D / C)
//     of every row as sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c and
//     writes the fp32 outputs [token][Hq * D].
// No workspace: nothing leaves the SMs but the outputs.

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace cg = cooperative_groups;

namespace qv {
namespace {

// CTAs per (sequence, key/value head). (16-CTA clusters of 225 KB CTAs with
// 160-key sub-chunks measured slower on GB300: 24 us per layer at 2048 cached
// positions against 19.5, and 21 against 9 at 512.)
constexpr int kAttnCluster = 8;
constexpr int kSub = 128;                  // keys per sub-chunk (8 groups of 16)
constexpr int kAttnThreads = 256;          // 8 warps
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnMaxRows = 32;           // R = T * G, two m16 tiles

struct AttnArgs {
    const uint16_t* qkv;     // [B*T][(Hq + 2 Hkv) * D] bf16
    const uint16_t* kc;      // [B][Lmax][Hkv][D] bf16
    const uint16_t* vc;
    const int32_t* len;      // [B]
    int T, Hq, Hkv, Lmax;
    float scale;
    float* out;              // [B*T][Hq*D]
};

template <int D>
struct AttnLayout {
    static constexpr int RS = D + 8;                 // bf16 row stride of Q, K, V
    static constexpr int SS = kSub + 4;              // fp32 row stride of the scores
    static constexpr int PS = kSub + 8;              // bf16 row stride of P
    static constexpr int Q = 0;
    static constexpr int K = Q + kAttnMaxRows * RS * 2;
    static constexpr int V = K + 2 * kSub * RS * 2;
    static constexpr int S = V + 2 * kSub * RS * 2;
    static constexpr int PH = S + kAttnMaxRows * SS * 4;
    static constexpr int PM = PH + kAttnMaxRows * PS * 2;
    static constexpr int M = PM + kAttnMaxRows * PS * 2;       // running max [32]
    static constexpr int L = M + kAttnMaxRows * 4;             // running sum [32]
    static constexpr int F = L + kAttnMaxRows * 4;             // rescale of this sub-chunk [32]
    static constexpr int Bytes = F + kAttnMaxRows * 4;
    // the partial output [32][D] fp32 for the cluster merge reuses stage 0 of K
    static_assert(kAttnMaxRows * D * 4 <= kSub * RS * 2, "partial output fits a key stage");
    static_assert(kSub % 32 == 0, "whole warps of keys per row");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ int seq_len(const AttnArgs& a, int b) {
    const int L = a.len[b];
    return L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);          // out-of-range lengths are clamped
}

// Key (kv = 0) or value (kv = 1) row at key position i of sequence b, head kh:
// the cache below L, the step's own qkv rows from L on.
template <int D>
__device__ __forceinline__ const uint16_t* kv_row(const AttnArgs& a, int b, int L, int i, int kh, int kv) {
    if (i < L) return (kv ? a.vc : a.kc) + (((size_t)b * a.Lmax + i) * a.Hkv + kh) * D;
    const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * D;
    return a.qkv + ((size_t)b * a.T + (i - L)) * W + (size_t)(a.Hq + kv * a.Hkv + kh) * D;
}

// Issue the cp.async copies of the keys and values at positions
// [p0, p0 + kSub) into stage st (zero rows at and past p_end).
template <int D>
__device__ __forceinline__ void stage_kv(const AttnArgs& a, uint32_t sbase, int b, int L, int kh, int p0,
                                         int p_end, int st) {
    using Ly = AttnLayout<D>;
    constexpr int P = D / 8;                                 // 16-byte pieces per row
    for (int e = threadIdx.x; e < 2 * kSub * P; e += kAttnThreads) {
        const int kv = e / (kSub * P), rem = e - kv * kSub * P;
        const int r = rem / P, c = rem - r * P;
        const int pos = p0 + r;
        const bool valid = pos < p_end;
        const uint16_t* src = valid ? kv_row<D>(a, b, L, pos, kh, kv) + c * 8 : a.qkv;
        const uint32_t dst = sbase + (uint32_t)((kv ? Ly::V : Ly::K) + ((st * kSub + r) * Ly::RS + c * 8) * 2);
        cp_async16(dst, src, valid);
    }
}

template <int D, int C>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_cluster_kernel(const AttnArgs a) {
    using Ly = AttnLayout<D>;
    constexpr int DPW = D / kAttnWarps;                      // output dims per warp (16 or 8)
    constexpr int NTO = DPW / 8;                             // n8 tiles of the output per warp
    extern __shared__ __align__(16) uint8_t attn_smem[];
    cg::cluster_group cluster = cg::this_cluster();
    allow_dependent_launch();
    grid_dependency_wait();

    const int rank = (int)cluster.block_rank();
    const int kh = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int G = a.Hq / a.Hkv, R = a.T * G;
    const int L = seq_len(a, b), S = L + a.T;
    const int per = ((S + C - 1) / C + 15) & ~15;            // key positions per CTA
    const int p_begin = rank * per, p_end = min(S, p_begin + per);
    const int nsub = p_begin < p_end ? (p_end - p_begin + kSub - 1) / kSub : 0;
    const uint32_t sbase = smem_u32(attn_smem);
    float* s_sc = reinterpret_cast<float*>(attn_smem + Ly::S);
    uint16_t* s_ph = reinterpret_cast<uint16_t*>(attn_smem + Ly::PH);
    uint16_t* s_pm = reinterpret_cast<uint16_t*>(attn_smem + Ly::PM);
    float* s_m = reinterpret_cast<float*>(attn_smem + Ly::M);
    float* s_l = reinterpret_cast<float*>(attn_smem + Ly::L);
    float* s_f = reinterpret_cast<float*>(attn_smem + Ly::F);
    const float NEG_INF = -__uint_as_float(0x7F800000u);

    // query rows r = j * G + g' of heads kh * G + g' (rows R..31 zero)
    {
        const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * D;
        for (int e = tid; e < kAttnMaxRows * (D / 8); e += kAttnThreads) {
            const int r = e / (D / 8), c = e - r * (D / 8);
            const bool valid = r < R;
            const int j = valid ? r / G : 0, h = kh * G + (valid ? r - j * G : 0);
            cp_async16(sbase + (uint32_t)(Ly::Q + (r * Ly::RS + c * 8) * 2),
                       a.qkv + ((size_t)b * a.T + j) * W + (size_t)h * D + c * 8, valid);
        }
    }
    if (nsub > 0) stage_kv<D>(a, sbase, b, L, kh, p_begin, p_end, 0);
    cp_async_commit();
    if (nsub > 1) stage_kv<D>(a, sbase, b, L, kh, p_begin + kSub, p_end, 1);
    cp_async_commit();
    if (tid < kAttnMaxRows) {
        s_m[tid] = NEG_INF;
        s_l[tid] = 0.f;
    }

    float o[2][NTO][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTO; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;

    const int mi = lane >> 3, ri = lane & 7;                 // ldmatrix: matrix and row of this lane
    for (int sc = 0; sc < nsub; ++sc) {
        const int st = sc & 1;
        const int p0 = p_begin + sc * kSub;
        cp_async_wait<1>();
        __syncthreads();

        // ---- scores: warp w covers the 16-key groups w, w + 8, ... of the sub-chunk, all 32 rows
        for (int grp = warp; grp < kSub / 16; grp += kAttnWarps) {
            float acc[2][2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
            const int n0 = 16 * grp;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t qa[2][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
                    ldmatrix_x4(sbase + (uint32_t)(Ly::Q + ((mt * 16 + (mi & 1) * 8 + ri) * Ly::RS +
                                                            kk * 16 + (mi >> 1) * 8) * 2),
                                qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3]);
                uint32_t kb0, kb1, kb2, kb3;
                ldmatrix_x4(sbase + (uint32_t)(Ly::K + ((st * kSub + n0 + (mi >> 1) * 8 + ri) * Ly::RS +
                                                        kk * 16 + (mi & 1) * 8) * 2),
                            kb0, kb1, kb2, kb3);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma_bf16_16816(acc[mt][0], qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3], kb0, kb1);
                    mma_bf16_16816(acc[mt][1], qa[mt][0], qa[mt][1], qa[mt][2], qa[mt][3], kb2, kb3);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int r = mt * 16 + g + 8 * hh;
                        const int kl = n0 + nt * 8 + 2 * t4;
                        float2 v;
                        // causal, and inside this CTA's key range (the staged rows past it are zeros)
                        const int lim = min(L + (r < R ? r / G : 0) + 1, p_end);
                        v.x = (r < R && p0 + kl < lim) ? acc[mt][nt][2 * hh] * a.scale : NEG_INF;
                        v.y = (r < R && p0 + kl + 1 < lim) ? acc[mt][nt][2 * hh + 1] * a.scale : NEG_INF;
                        *reinterpret_cast<float2*>(s_sc + r * Ly::SS + kl) = v;
                    }
        }
        __syncthreads();

        // ---- online softmax: warp w takes rows w, w + 8, w + 16, w + 24
        for (int r = warp; r < kAttnMaxRows; r += kAttnWarps) {
            float sv[kSub / 32];
            float mx = NEG_INF;
#pragma unroll
            for (int q = 0; q < kSub / 32; ++q) {
                sv[q] = s_sc[r * Ly::SS + lane + 32 * q];
                mx = fmaxf(mx, sv[q]);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_old = s_m[r];
            const float m_new = fmaxf(m_old, mx);
            const bool none = m_new == NEG_INF;                  // no visible key yet
            float lsum = 0.f;
#pragma unroll
            for (int q = 0; q < kSub / 32; ++q) {
                const float p = none ? 0.f : expf(sv[q] - m_new);
                lsum += p;
                const __nv_bfloat16 hi = __float2bfloat16_rn(p);
                const __nv_bfloat16 mid = __float2bfloat16_rn(p - __bfloat162float(hi));
                s_ph[r * Ly::PS + lane + 32 * q] = __bfloat16_as_ushort(hi);
                s_pm[r * Ly::PS + lane + 32 * q] = __bfloat16_as_ushort(mid);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
            if (lane == 0) {
                const float f = none ? 1.f : expf(m_old - m_new);   // e^(-inf) = 0 on the first keys
                s_f[r] = f;
                s_m[r] = m_new;
                s_l[r] = s_l[r] * f + lsum;
            }
        }
        __syncthreads();

        // ---- o = o * f + P V: warp w covers dims [DPW w, DPW w + DPW), all 32 rows
        {
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const float f0 = s_f[mt * 16 + g], f1 = s_f[mt * 16 + g + 8];
#pragma unroll
                for (int nt = 0; nt < NTO; ++nt) {
                    o[mt][nt][0] *= f0;
                    o[mt][nt][1] *= f0;
                    o[mt][nt][2] *= f1;
                    o[mt][nt][3] *= f1;
                }
            }
            const int d0 = DPW * warp;
#pragma unroll
            for (int ks = 0; ks < kSub / 16; ++ks) {
                uint32_t vb[NTO][2];
                if constexpr (NTO == 2) {
                    ldmatrix_x4_trans(sbase + (uint32_t)(Ly::V + ((st * kSub + ks * 16 + (mi & 1) * 8 + ri) * Ly::RS +
                                                                  d0 + (mi >> 1) * 8) * 2),
                                      vb[0][0], vb[0][1], vb[1][0], vb[1][1]);
                } else {
                    ldmatrix_x2_trans(sbase + (uint32_t)(Ly::V + ((st * kSub + ks * 16 + (mi & 1) * 8 + ri) * Ly::RS +
                                                                  d0) * 2),
                                      vb[0][0], vb[0][1]);
                }
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const int base = part ? Ly::PM : Ly::PH;
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        uint32_t pa0, pa1, pa2, pa3;
                        ldmatrix_x4(sbase + (uint32_t)(base + ((mt * 16 + (mi & 1) * 8 + ri) * Ly::PS +
                                                               ks * 16 + (mi >> 1) * 8) * 2),
                                    pa0, pa1, pa2, pa3);
#pragma unroll
                        for (int nt = 0; nt < NTO; ++nt)
                            mma_bf16_16816(o[mt][nt], pa0, pa1, pa2, pa3, vb[nt][0], vb[nt][1]);
                    }
                }
            }
        }
        __syncthreads();                                     // stage st and P are free again
        if (sc + 2 < nsub) stage_kv<D>(a, sbase, b, L, kh, p0 + 2 * kSub, p_end, st);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- this CTA's partial output, then the cluster merge
    float* s_o = reinterpret_cast<float*>(attn_smem + Ly::K);   // [32][D]
    {
        const int d0 = DPW * warp;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTO; ++nt) {
                const int col = d0 + nt * 8 + 2 * t4;
                *reinterpret_cast<float2*>(s_o + (mt * 16 + g) * D + col) = make_float2(o[mt][nt][0], o[mt][nt][1]);
                *reinterpret_cast<float2*>(s_o + (mt * 16 + g + 8) * D + col) = make_float2(o[mt][nt][2], o[mt][nt][3]);
            }
    }
    cluster.sync();
    {
        constexpr int DC = D / C;                            // dims merged by this CTA
        const int dc0 = rank * DC;
        for (int e = tid; e < R * DC; e += kAttnThreads) {
            const int r = e / DC, d = dc0 + (e - r * DC);
            float mc[C];
            float M = NEG_INF;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                mc[c] = *cluster.map_shared_rank(s_m + r, c);
                M = fmaxf(M, mc[c]);
            }
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const float w = mc[c] == NEG_INF ? 0.f : expf(mc[c] - M);   // a CTA with no visible key
                num += w * *cluster.map_shared_rank(s_o + r * D + d, c);
                den += w * *cluster.map_shared_rank(s_l + r, c);
            }
            const int j = r / G, h = kh * G + (r - j * G);
            a.out[((size_t)b * a.T + j) * (size_t)a.Hq * D + (size_t)h * D + d] = num / den;
        }
    }
    cluster.sync();                                          // no CTA leaves while others read its memory
}

template <int D, int C>
cudaError_t launch_cluster(const AttnArgs& args, int B, cudaStream_t s) {
    using Ly = AttnLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Ly::Bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, args.Hkv, B);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = Ly::Bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<D, C>, args);
}

static_assert(AttnLayout<128>::Bytes <= (int)kMaxDynSmem, "shared memory budget");

}  // namespace

size_t attention_workspace_bytes(int, int, int, int, int, int) { return 16; }

cudaError_t launch_attention_verify(const uint16_t* qkv, const uint16_t* kc, const uint16_t* vc, const int32_t* len,
                                    int B, int T, int Hq, int Hkv, int D, int Lmax, float scale, float* out,
                                    void*, cudaStream_t s) {
    AttnArgs a;
    a.qkv = qkv; a.kc = kc; a.vc = vc; a.len = len;
    a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.Lmax = Lmax;
    a.scale = scale;
    a.out = out;
    return D == 128 ? launch_cluster<128, kAttnCluster>(a, B, s) : launch_cluster<64, kAttnCluster>(a, B, s);
}

}  // namespace qv
