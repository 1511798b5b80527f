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
//   - the S = len + T key positions are cut into C equal ranges of whole
//     16-key blocks, one range per CTA;
//   - the range streams through a 5-stage ring of 64-key stages with 4-D
//     TMA loads of the caches (a 64-position box per tensor and 64 values
//     for a stage wholly below len, else one 16-position box per block;
//     128-byte swizzle), keys and values of a stage on one mbarrier; two
//     warps request the first two stages, the rest of the ring follows once
//     those have landed, and the last of a stage's warps to finish with it (a
//     shared counter) issues its refill, so no warp is set aside for copies.
//     Positions at and past len are not the cache's: the warp that owns such
//     a block overwrites those rows with the step's own key/value rows (or
//     zeros past S) before it reads them, and blocks wholly past len load
//     nothing;
//   - warp 4 h + q takes block q of the stages of parity h (a range of one
//     stage is shared: its blocks' P V is split by dims over all 8 warps)
//     and keeps its own online softmax for all R rows in registers
//     (FlashAttention-2 style, no block barrier inside the loop). Keys are
//     the M dimension of the bf16 tensor
//     core products (mma.sync m16n8k16, fp32 accumulation) and query rows
//     the N dimension, in n8 tiles (R = 20 takes 24 rows, not 32):
//     S^T = K Q^T (the bf16 products are exact, the sum is a binary32 sum),
//     scaled to base-2 units (2^(s log2 e) = e^s) and masked (causal, and
//     key positions past the CTA's range); running max m, running sum l and
//     output o^T rescaled by 2^(m_old - m_new) per block; o^T += V^T P^T
//     with P split into two bf16 parts, P = hi + mid + r with
//     |r| <= 2^-18 P, so the product's error is below 2^-18 max|v| (values
//     are bf16, exact). The score fragments, transposed in registers
//     (movmatrix), are the B operand of V^T P^T: P never leaves registers;
//   - the 8 warps' partials merge in shared memory into the CTA's (m, l, o)
//     and go out as pushes: CTA k owns dims [k D / C, (k + 1) D / C) and
//     receives every CTA's rows of those dims and (m, l) in its shared
//     memory (distributed shared-memory stores, one cluster barrier); it
//     merges them as sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c and
//     writes the fp32 outputs [token][Hq * D].
// No workspace: nothing leaves the SMs but the outputs.

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace cg = cooperative_groups;

namespace qv {

__device__ unsigned int g_attn_error;

namespace {

// CTAs per (sequence, key/value head). (16-CTA clusters measured slower on
// GB300 with the earlier cp.async design: 24 us per layer at 2048 cached
// positions against 19.5.)
constexpr int kAttnCluster = 8;
constexpr int kSub = 64;                   // key positions per stage: 4 blocks of 16
constexpr int kBlk = 16;                   // key positions per warp block (one k16 of P V)
constexpr int kStages = 5;                 // 17 blocks of a 2048-position range in flight at once
constexpr int kAttnWarps = 8;              // (255 registers a thread: a warp's o is 128 of them)
constexpr int kGroupWarps = kSub / kBlk;   // warps per stage (4)
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kAttnMaxRows = 32;           // R = T * G, at most four n8 tiles
constexpr float kLog2e = 1.4426950408889634f;   // scores are carried in base-2 units: 2^(s log2 e) = e^s
static_assert(kAttnWarps == 2 * kGroupWarps, "two warp groups take alternate stages");

struct AttnArgs {
    const uint16_t* qkv;     // [B*T][(Hq + 2 Hkv) * D] bf16
    const int32_t* len;      // [B]
    int T, Hq, Hkv, Lmax;
    int has_cache;           // 0: Lmax == 0, no tensor maps
    float scale;
    float* out;              // [B*T][Hq*D]
    int hold_loads;          // test hook: request no stage, so every stage wait runs out
    unsigned long long wait_ns;   // limit of a stage wait (kWaitLimitNs by default)
};

template <int D>
struct AttnLayout {
    static constexpr int H = D / 64;                       // 128-byte halves of a row
    static constexpr int Box = kSub * 128;                 // 64 rows x 128 B, filled by 16-row boxes
    static constexpr int StageBytes = 2 * H * Box;         // keys (H boxes), then values (H boxes)
    static constexpr int RS = D + 8;                       // bf16 row stride of Q (padded)
    static constexpr int Q = kStages * StageBytes;         // stages first: 1024-byte aligned boxes
    static constexpr int DC = D / kAttnCluster;            // dims merged (and written) by each CTA
    static constexpr int RV = Q + kAttnMaxRows * RS * 2;   // received o slices [C][DC][32] fp32
    static constexpr int RM = RV + kAttnCluster * kAttnMaxRows * DC * 4;   // received m [C][32]
    static constexpr int RL = RM + kAttnCluster * kAttnMaxRows * 4;        // received l [C][32]
    static constexpr int WM = RL + kAttnCluster * kAttnMaxRows * 4;        // per-warp running max [8][32]
    static constexpr int WL = WM + kAttnWarps * kAttnMaxRows * 4;   // per-warp running sum [8][32]
    static constexpr int M = WL + kAttnWarps * kAttnMaxRows * 4;    // the CTA's m [32]
    static constexpr int CW = M + kAttnMaxRows * 4;        // cluster weights [32][C] and the denominator
    static constexpr int Bar = CW + kAttnMaxRows * (kAttnCluster + 1) * 4;
    static constexpr int Cnt = Bar + kStages * 8;          // warps done with each stage
    static constexpr int Flag = Cnt + kStages * 4;         // abort word of the bounded waits
    static constexpr int Bytes = Flag + 16;
    static constexpr int Alloc = Bytes + 1024;             // slack to align the base to 1024 B
    // the warps' partial outputs [8][32][D] fp32 reuse the (drained) stages
    static_assert(kAttnWarps * kAttnMaxRows * D * 4 <= kStages * StageBytes, "partials fit the stages");
    static_assert(Bar % 8 == 0 && RV % 16 == 0, "mbarrier and vector alignment");
    static_assert(DC % 4 == 0, "whole float4 slices");
};

// Byte offset of 16-byte chunk c (of D / 8) of row r (0..63) of tensor kv
// (0 keys, 1 values) in a stage: the TMA 128-byte swizzle puts chunk cc of a
// 128-byte row at cc ^ (r mod 8) (boxes are 1024-byte aligned).
template <int D>
__device__ __forceinline__ uint32_t kv_off(int kv, int r, int c) {
    using Ly = AttnLayout<D>;
    const int h = c >> 3, cc = c & 7;
    return (uint32_t)((kv * Ly::H + h) * Ly::Box + r * 128 + ((cc ^ (r & 7)) << 4));
}

// 4-D tiled load of the box at (x, head, position, sequence) into shared
// memory; completion is signalled on `bar` as transaction bytes. x * 2 bytes
// is a multiple of 16 (x is 0 or 64).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int hd, int pos, int seq,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(hd), "r"(pos), "r"(seq),
           "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Transpose of the 8x8 b16 matrix whose row lane / 4, columns 2 (lane % 4)
// and 2 (lane % 4) + 1 this lane holds (the mma.sync fragment layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// mbar_wait_bounded with a limit given at run time.
__device__ __forceinline__ bool stage_wait(uint64_t* bar, unsigned parity, volatile int* abort,
                                           unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort = 1;
            return false;
        }
    }
}

// Generic-proxy writes to shared memory before a later TMA write to it.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ int seq_len(const AttnArgs& a, int b) {
    const int L = a.len[b];
    return L < 0 ? 0 : (L > a.Lmax ? a.Lmax : L);          // out-of-range lengths are clamped
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// p = hi + mid (+ a remainder below 2^-18 p): the two bf16 parts of a pair.
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t& hi, uint32_t& mid) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(p0), h1 = __float2bfloat16_rn(p1);
    hi = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
    mid = pack_bf16(p0 - __bfloat162float(h0), p1 - __bfloat162float(h1));
}

// Issue the TMA loads of sub-chunk sj (stage sj mod kStages). A stage whose
// four blocks all start below L loads as one 64-position box per tensor and
// 64 values; otherwise each block that starts below L loads as 16-position
// boxes (a block wholly at or past L holds no cache rows). With no such
// block the stage's phase completes without copies.
template <int D>
__device__ __forceinline__ void issue_stage(uint32_t sbase, uint64_t* full, const KvMaps& tm, int has_cache, int sj,
                                            int nblk, int p_begin, int L, int kh, int b, uint64_t pol, int hold) {
    using Ly = AttnLayout<D>;
    if (hold) return;                                        // test hook: the stage never completes
    const int s = sj % kStages;
    int nb = 0;
#pragma unroll
    for (int q = 0; q < kGroupWarps; ++q) {
        const int j = sj * kGroupWarps + q;
        nb += (has_cache && j < nblk && p_begin + j * kBlk < L) ? 1 : 0;
    }
    if (nb == 0) {
        mbar_arrive(&full[s]);
        return;
    }
    mbar_arrive_expect_tx(&full[s], (unsigned)(nb * 2 * Ly::H * kBlk * 128));
    const uint32_t st = sbase + (uint32_t)(s * Ly::StageBytes);
    if (nb == kGroupWarps) {
        const int p0 = p_begin + sj * kSub;
#pragma unroll
        for (int h = 0; h < Ly::H; ++h) {
            tma_load_4d(st + (uint32_t)(h * Ly::Box), &tm.k64, 64 * h, kh, p0, b, &full[s], pol);
            tma_load_4d(st + (uint32_t)((Ly::H + h) * Ly::Box), &tm.v64, 64 * h, kh, p0, b, &full[s], pol);
        }
        return;
    }
#pragma unroll
    for (int q = 0; q < kGroupWarps; ++q) {
        const int j = sj * kGroupWarps + q, kp0 = p_begin + j * kBlk;
        if (!(has_cache && j < nblk && kp0 < L)) continue;
#pragma unroll
        for (int h = 0; h < Ly::H; ++h) {
            tma_load_4d(st + (uint32_t)(h * Ly::Box + q * kBlk * 128), &tm.k16, 64 * h, kh, kp0, b, &full[s], pol);
            tma_load_4d(st + (uint32_t)((Ly::H + h) * Ly::Box + q * kBlk * 128), &tm.v16, 64 * h, kh, kp0, b,
                        &full[s], pol);
        }
    }
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

template <int D, int C, int NR>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_cluster_kernel(const __grid_constant__ KvMaps tm, const AttnArgs a) {
    using Ly = AttnLayout<D>;
    constexpr int CH = D / 8;                                // 16-byte chunks of a row
    extern __shared__ uint8_t attn_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(attn_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int kh = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Ly::Bar);
    int* cnt = reinterpret_cast<int*>(smem + Ly::Cnt);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + Ly::Flag);
    float* s_part = reinterpret_cast<float*>(smem);         // [8][D][32], after the stages drain
    float* s_rv = reinterpret_cast<float*>(smem + Ly::RV);
    float* s_rm = reinterpret_cast<float*>(smem + Ly::RM);
    float* s_rl = reinterpret_cast<float*>(smem + Ly::RL);
    float* s_wm = reinterpret_cast<float*>(smem + Ly::WM);
    float* s_wl = reinterpret_cast<float*>(smem + Ly::WL);
    float* s_m = reinterpret_cast<float*>(smem + Ly::M);
    float* s_cw = reinterpret_cast<float*>(smem + Ly::CW);
    const float NEG_INF = -__uint_as_float(0x7F800000u);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            cnt[s] = 0;
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    cluster_arrive_relaxed();       // waited for before the first store into another CTA
    allow_dependent_launch();
    grid_dependency_wait();

    const int G = a.Hq / a.Hkv, R = a.T * G;
    const int L = seq_len(a, b), S = L + a.T;
    const int per = ((S + C - 1) / C + kBlk - 1) / kBlk * kBlk;   // key positions per CTA
    const int p_begin = rank * per, p_end = min(S, p_begin + per);
    const int nblk = p_begin < p_end ? (p_end - p_begin + kBlk - 1) / kBlk : 0;
    const int nsub = (nblk + kGroupWarps - 1) / kGroupWarps;

    const uint64_t pol = policy_evict_first();
    {
        const size_t W = (size_t)(a.Hq + 2 * a.Hkv) * D;
        // query rows r = j * G + g' of heads kh * G + g' (rows R..31 zero),
        // requested before the stages so that they do not queue behind them
        for (int e = tid; e < kAttnMaxRows * CH; e += kAttnThreads) {
            const int r = e / CH, c = e - r * CH;
            const bool valid = r < R;
            const int j = valid ? r / G : 0, h = kh * G + (valid ? r - j * G : 0);
            cp_async16(sbase + (uint32_t)(Ly::Q + (r * Ly::RS + c * 8) * 2),
                       a.qkv + ((size_t)b * a.T + j) * W + (size_t)h * D + c * 8, valid);
        }
        // sub-chunks 0 and 1 now (one warp each), the rest of the ring once 0
        // and 1 have landed, so that the first stages do not share HBM with it
        if (lane == 0 && warp < 2 && warp < nsub) {
            if (a.has_cache) {
                prefetch_tensormap(&tm.k64);
                prefetch_tensormap(&tm.v64);
            }
            issue_stage<D>(sbase, full, tm, a.has_cache, warp, nblk, p_begin, L, kh, b, pol, a.hold_loads);
        }
        cp_async_wait_all();
        __syncthreads();

        const int grp = warp / kGroupWarps, q = warp - grp * kGroupWarps;
        const int mi = lane >> 3, ri = lane & 7;             // ldmatrix: matrix and row of this lane
        const float sl2 = a.scale * kLog2e;                  // scores in base-2 units
        // o^T: dims 16 dm + g (+8) x rows 8 nt + 2 t4 (+1)
        float o[D / 16][NR][4];
        float m_run[NR][2], l_run[NR][2];                    // rows 8 nt + 2 t4 + e
        int lim[NR][2];                                      // visible key positions: [0, lim)
#pragma unroll
        for (int nt = 0; nt < NR; ++nt) {
#pragma unroll
            for (int dm = 0; dm < D / 16; ++dm)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[dm][nt][e] = 0.f;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 8 * nt + 2 * t4 + e;
                m_run[nt][e] = NEG_INF;
                l_run[nt][e] = 0.f;
                lim[nt][e] = r < R ? min(L + r / G + 1, p_end) : INT_MIN;
            }
        }
        bool first = true;                                   // o is still zero

        // Rows at and past len of block kp0 (stage rows r0..r0+15): the step's
        // key/value rows, zeros past S; threads t0, t0 + step, ... share the work.
        auto own_rows = [&](uint32_t st, int r0, int kp0, int t0, int step) {
            for (int e = t0; e < 2 * kBlk * CH; e += step) {
                const int kv = e / (kBlk * CH), rem = e - kv * (kBlk * CH);
                const int r = rem / CH, c = rem - r * CH;
                const int pos = kp0 + r;
                if (pos < L) continue;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (pos < S)
                    v = *reinterpret_cast<const uint4*>(a.qkv + ((size_t)b * a.T + (pos - L)) * W +
                                                        (size_t)(a.Hq + kv * a.Hkv + kh) * D + c * 8);
                sts_v4_u32(st + kv_off<D>(kv, r0 + r, c), v.x, v.y, v.z, v.w);
            }
        };
        // One 16-key block (stage rows r0.., first position kp0) into this
        // warp's softmax state; P V only for the dim tiles [dm0, dm1), and the
        // block's probabilities added to l only if add_l (a block shared by
        // several warps counts once in l and once per dim).
        auto block = [&](uint32_t st, int r0, int kp0, int dm0, int dm1, bool add_l) {
            // ---- S^T = K Q^T: the block's 16 keys (M) x the rows (N, NR tiles of 8)
            float acc[NR][4];
#pragma unroll
            for (int nt = 0; nt < NR; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t ka0, ka1, ka2, ka3;                 // keys (mi & 1) * 8.., dims chunk kk * 2 + (mi >> 1)
                ldmatrix_x4(st + kv_off<D>(0, r0 + (mi & 1) * 8 + ri, kk * 2 + (mi >> 1)), ka0, ka1, ka2, ka3);
#pragma unroll
                for (int nt = 0; nt < NR; ++nt) {
                    uint32_t qb0, qb1;                       // rows 8 nt.., dims kk * 16 + (0 | 8)
                    ldmatrix_x2(sbase + (uint32_t)(Ly::Q + ((8 * nt + ri) * Ly::RS + kk * 16 + (mi & 1) * 8) * 2),
                                qb0, qb1);
                    mma_bf16_16816(acc[nt], ka0, ka1, ka2, ka3, qb0, qb1);
                }
            }

            // ---- online softmax per row (base 2); P^T pairs transposed into the B operand of P V
            uint32_t bh[NR][2], bm[NR][2];
            float f[NR][2];
#pragma unroll
            for (int nt = 0; nt < NR; ++nt) {
                float p[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    // keys g and g + 8 of row 8 nt + 2 t4 + e
                    const float s0 = kp0 + g < lim[nt][e] ? acc[nt][e] * sl2 : NEG_INF;
                    const float s1 = kp0 + g + 8 < lim[nt][e] ? acc[nt][2 + e] * sl2 : NEG_INF;
                    float mx = fmaxf(s0, s1);
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float m_old = m_run[nt][e];
                    const float m_new = fmaxf(m_old, mx);
                    const bool none = m_new == NEG_INF;          // no visible key yet
                    f[nt][e] = none ? 1.f : exp2f(m_old - m_new);   // 2^(-inf) = 0 on the first keys
                    p[e] = none ? 0.f : exp2f(s0 - m_new);
                    p[2 + e] = none ? 0.f : exp2f(s1 - m_new);
                    m_run[nt][e] = m_new;
                    l_run[nt][e] = l_run[nt][e] * f[nt][e] + (add_l ? p[e] + p[2 + e] : 0.f);
                }
                uint32_t h01, m01, h23, m23;             // (key g | g + 8; rows 2 t4, 2 t4 + 1)
                split_pair(p[0], p[1], h01, m01);
                split_pair(p[2], p[3], h23, m23);
                bh[nt][0] = movmatrix_trans(h01);        // (row g; keys 2 t4, 2 t4 + 1)
                bh[nt][1] = movmatrix_trans(h23);        // (row g; keys 8 + 2 t4, 9 + 2 t4)
                bm[nt][0] = movmatrix_trans(m01);
                bm[nt][1] = movmatrix_trans(m23);
            }
            // rescale o unless every factor is 1 (or o is still zero)
            bool ones = true;
#pragma unroll
            for (int nt = 0; nt < NR; ++nt) ones = ones && f[nt][0] == 1.f && f[nt][1] == 1.f;
            if (!first && !__all_sync(0xffffffffu, ones)) {
#pragma unroll
                for (int dm = 0; dm < D / 16; ++dm)
#pragma unroll
                    for (int nt = 0; nt < NR; ++nt) {
                        o[dm][nt][0] *= f[nt][0];
                        o[dm][nt][1] *= f[nt][1];
                        o[dm][nt][2] *= f[nt][0];
                        o[dm][nt][3] *= f[nt][1];
                    }
            }
            first = false;

            // ---- o^T += V^T P^T: dims (M, 16 per tile) x rows (N) over the block's 16 keys
#pragma unroll
            for (int dm = 0; dm < D / 16; ++dm) {
                if (dm < dm0 || dm >= dm1) continue;
                uint32_t va0, va1, va2, va3;                 // keys (mi >> 1) * 8.., dims chunk dm * 2 + (mi & 1)
                ldmatrix_x4_trans(st + kv_off<D>(1, r0 + (mi >> 1) * 8 + ri, dm * 2 + (mi & 1)), va0, va1, va2, va3);
#pragma unroll
                for (int nt = 0; nt < NR; ++nt) {
                    mma_bf16_16816(o[dm][nt], va0, va1, va2, va3, bh[nt][0], bh[nt][1]);
                    mma_bf16_16816(o[dm][nt], va0, va1, va2, va3, bm[nt][0], bm[nt][1]);
                }
            }
        };

        // A range of one stage (at most 4 blocks) would leave warp group 1
        // idle: all 8 warps share its blocks instead (each block's scores and
        // softmax in each of its warps, its P V split by dims among them).
        // (Sharing the last of an odd number of stages measured slower at 2048
        // and 8192 cached positions: there the last stage waits for its data.)
        const bool shared_last = nsub == 1;
        const int nsub_own = shared_last ? nsub - 1 : nsub;
        for (int sj = grp; sj < nsub_own; sj += 2) {
            const int s = sj % kStages;
            if (!stage_wait(&full[s], (unsigned)((sj / kStages) & 1), abort, a.wait_ns)) {
                atomicOr(&g_attn_error, kErrFullWait);
                break;
            }
            if (sj < 2 && q == 0 && lane == 0)               // the rest of the first fill
                for (int x = sj + 2; x < kStages && x < nsub; x += 2)
                    issue_stage<D>(sbase, full, tm, a.has_cache, x, nblk, p_begin, L, kh, b, pol, a.hold_loads);
            const int j = sj * kGroupWarps + q;              // this warp's block of the stage
            if (j < nblk) {
                const uint32_t st = sbase + (uint32_t)(s * Ly::StageBytes);
                const int kp0 = p_begin + j * kBlk;          // its first key position
                const bool fix = kp0 + kBlk > L;
                if (fix) {
                    own_rows(st, q * kBlk, kp0, lane, 32);
                    __syncwarp();
                }
                block(st, q * kBlk, kp0, 0, D / 16, true);
                if (fix) fence_proxy_async_shared();         // before the stage's next TMA write
            }
            __syncwarp();
            // the last of the stage's warps refills it with sub-chunk sj + kStages
            // (the counter only grows: use u of the stage ends at 4 (u + 1) arrivals)
            if (lane == 0 && atomicAdd(&cnt[s], 1) == kGroupWarps * (sj / kStages + 1) - 1) {
                if (sj + kStages < nsub)
                    issue_stage<D>(sbase, full, tm, a.has_cache, sj + kStages, nblk, p_begin, L, kh, b, pol, a.hold_loads);
            }
        }
        if (shared_last) {
            // never refilled (it is the last), so no release count is kept
            const int sj = nsub - 1, s = sj % kStages;
            const bool ok = stage_wait(&full[s], (unsigned)((sj / kStages) & 1), abort, a.wait_ns);
            if (!ok) atomicOr(&g_attn_error, kErrFullWait);
            const uint32_t st = sbase + (uint32_t)(s * Ly::StageBytes);
            const int nb = nblk - sj * kGroupWarps;          // 1..4 blocks
            const int nbp = nb == 3 ? 4 : nb;                // warps split evenly: 8, 4 or 2 per block
            const int wpb = kAttnWarps / nbp;
            const int ns = wpb < D / 16 ? wpb : D / 16;      // dim slices per block
            const int qb = warp % nbp, sl = warp / nbp;
            if (ok) {
                for (int qq = 0; qq < nb; ++qq) {
                    const int kp0 = p_begin + (sj * kGroupWarps + qq) * kBlk;
                    if (kp0 + kBlk > L) own_rows(st, qq * kBlk, kp0, tid, kAttnThreads);   // rows at or past len
                }
            }
            __syncthreads();
            const int j = sj * kGroupWarps + qb;
            if (ok && j < nblk && sl < ns) {
                const int tps = (D / 16) / ns;               // dim tiles per slice
                block(st, qb * kBlk, p_begin + j * kBlk, sl * tps, sl * tps + tps, sl == 0);
            }
        }

        // this warp's running sums over the 8 lanes of a row, then its (m, l) per row
#pragma unroll
        for (int nt = 0; nt < NR; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = l_run[nt][e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                if (g == 0) {
                    const int r = 8 * nt + 2 * t4 + e;
                    s_wm[warp * kAttnMaxRows + r] = m_run[nt][e];
                    s_wl[warp * kAttnMaxRows + r] = l;
                }
            }
        // every stage this CTA loaded has been waited for: the ring may be reused
        __syncthreads();
        // this warp's o^T, scaled by 2^(m_w - M) for the CTA's row maxima M, into
        // [warp][D][32] (rows XOR-swizzled by dim: 2 wavefronts a store)
        float wt[NR][2];
#pragma unroll
        for (int nt = 0; nt < NR; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = 8 * nt + 2 * t4 + e;
                float M = NEG_INF;
#pragma unroll
                for (int c = 0; c < kAttnWarps; ++c) M = fmaxf(M, s_wm[c * kAttnMaxRows + r]);
                wt[nt][e] = m_run[nt][e] == NEG_INF ? 0.f : exp2f(m_run[nt][e] - M);   // no visible key: 0
                if (warp == 0 && g == 0) s_m[r] = M;
            }
#pragma unroll
        for (int dm = 0; dm < D / 16; ++dm)
#pragma unroll
            for (int nt = 0; nt < NR; ++nt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int d = 16 * dm + g + 8 * hh;
                    const int rw = (8 * nt + 2 * t4) ^ ((d & 7) << 2);
                    *reinterpret_cast<float2*>(s_part + (warp * D + d) * kAttnMaxRows + rw) =
                        make_float2(o[dm][nt][2 * hh] * wt[nt][0], o[dm][nt][2 * hh + 1] * wt[nt][1]);
                }
    }
    __syncthreads();
    cluster_wait();                                          // every CTA of the cluster has started
    constexpr int DC = Ly::DC;
    // ---- this CTA's (m, l, o), pushed to the cluster: the o rows of CTA k's
    // dims go into CTA k's receive buffer, (m, l) to all
    if (tid < R) {
        const float m = s_m[tid];
        float l = 0.f;
#pragma unroll
        for (int c = 0; c < kAttnWarps; ++c) {
            const float mw = s_wm[c * kAttnMaxRows + tid];
            l += (mw == NEG_INF ? 0.f : exp2f(mw - m)) * s_wl[c * kAttnMaxRows + tid];
        }
#pragma unroll
        for (int k = 0; k < C; ++k) {
            *cluster.map_shared_rank(s_rm + rank * kAttnMaxRows + tid, k) = m;
            *cluster.map_shared_rank(s_rl + rank * kAttnMaxRows + tid, k) = l;
        }
    }
    {
        const int R4 = (R + 3) / 4;                          // groups of 4 rows
        for (int e = tid; e < D * R4; e += kAttnThreads) {
            const int d = e / R4, r = 4 * (e - d * R4);
            const int rw = r ^ ((d & 7) << 2);               // the four rows stay together
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kAttnWarps; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(s_part + (c * D + d) * kAttnMaxRows + rw);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int k = d / DC;
            *reinterpret_cast<float4*>(cluster.map_shared_rank(s_rv + (rank * DC + (d - k * DC)) * kAttnMaxRows + r, k)) =
                acc;
        }
    }
    cluster.sync();                                          // every push has landed

    // ---- the cluster merge of this CTA's dims [rank DC, (rank + 1) DC) from its receive buffer
    if (tid < R) {
        float M = NEG_INF;
#pragma unroll
        for (int c = 0; c < C; ++c) M = fmaxf(M, s_rm[c * kAttnMaxRows + tid]);
        float den = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const float mc = s_rm[c * kAttnMaxRows + tid];
            const float w = mc == NEG_INF ? 0.f : exp2f(mc - M);  // a CTA with no visible key
            s_cw[tid * (C + 1) + c] = w;
            den += w * s_rl[c * kAttnMaxRows + tid];
        }
        s_cw[tid * (C + 1) + C] = den;
    }
    __syncthreads();
    for (int e = tid; e < R * DC; e += kAttnThreads) {
        const int dl = e / R, r = e - dl * R;
        float num = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) num += s_cw[r * (C + 1) + c] * s_rv[(c * DC + dl) * kAttnMaxRows + r];
        const int j = r / G, h = kh * G + (r - j * G);
        a.out[((size_t)b * a.T + j) * (size_t)a.Hq * D + (size_t)h * D + rank * DC + dl] = num / s_cw[r * (C + 1) + C];
    }
    // nothing reads another CTA's memory after the cluster barrier: no second one
}

template <int D, int C, int NR>
cudaError_t launch_cluster(const KvMaps& tm, const AttnArgs& args, int B, cudaStream_t s) {
    using Ly = AttnLayout<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<D, C, NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Ly::Alloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, args.Hkv, B);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = Ly::Alloc;
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
    return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<D, C, NR>, tm, args);
}

static_assert(AttnLayout<128>::Alloc <= (int)kMaxDynSmem, "shared memory budget");

}  // namespace

size_t attention_workspace_bytes(int, int, int, int, int, int) { return 16; }

cudaError_t launch_attention_verify(const uint16_t* qkv, const KvMaps* maps, const int32_t* len, int B, int T, int Hq,
                                    int Hkv, int D, int Lmax, float scale, float* out, int hold_loads,
                                    unsigned long long wait_ns, cudaStream_t s) {
    AttnArgs a;
    a.hold_loads = hold_loads;
    a.wait_ns = wait_ns ? wait_ns : kWaitLimitNs;
    a.qkv = qkv; a.len = len;
    a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.Lmax = Lmax;
    a.has_cache = maps ? 1 : 0;
    a.scale = scale;
    a.out = out;
    KvMaps none;
    memset(&none, 0, sizeof(none));
    const KvMaps& tm = maps ? *maps : none;
    const int nr = (T * (Hq / Hkv) + 7) / 8;                 // n8 tiles of query rows
#define QV_ATTN_CASE(DV, NRV) \
    if (D == DV && nr == NRV) return launch_cluster<DV, kAttnCluster, NRV>(tm, a, B, s);
    QV_ATTN_CASE(128, 1) QV_ATTN_CASE(128, 2) QV_ATTN_CASE(128, 3) QV_ATTN_CASE(128, 4)
    QV_ATTN_CASE(64, 1) QV_ATTN_CASE(64, 2) QV_ATTN_CASE(64, 3) QV_ATTN_CASE(64, 4)
#undef QV_ATTN_CASE
    return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_attn_error(unsigned* code) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_attn_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(unsigned));
}

}  // namespace qv
