// stream_common.cuh -- pieces shared by the weight-streaming GEMM kernels of
// libqv (the mma.sync kernels and the tcgen05 kernel): tile geometry, the TMA
// producer of the shared-memory ring, the W8A8 kernel parameters and the
// split-K / LM-head segment epilogue. Included by the kernel translation
// units; everything here has internal linkage.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"

namespace qv {
namespace {

constexpr int BN = kTileN;            // output channels per tile
constexpr int BKB = kTileKBytes;      // bytes of K per tile (one 128-byte row)
constexpr int kMaxConsumerWarps = 8;
constexpr int kWTileBytes = BN * BKB;             // 16 KB

template <int CW>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(CW * 32) : "memory");
}

// Order-preserving map of a float to uint32 (larger float -> larger key);
// -0 is folded onto +0 first.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unordered_bits(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
        v = o > v ? o : v;
    }
    return v;
}

// Weight tiles a producer requests before its grid dependency wait. Behind
// the activation quantization (which lets the GEMM launch once the previous
// GEMM has finished) they load during the quantization; 4 and 5 measured
// best on the 5-token step, 6 and 7 slower (the full ring fill takes HBM
// from the quantization's own reads and the previous kernel's last stores).
constexpr int kPreWaitTiles = 5;

// Producer: stream tiles [a, b) into the ring. The first kPreWaitTiles weight
// tiles are requested before the grid dependency wait. With tx == null
// only weight tiles travel (tx_bytes must then count the weight tile alone).
// Each weight tile travels with XB activation boxes: box j of tile kt starts
// at element (kt * XB + j) * kx_elems_per_tile of K (XB = 2 when a weight
// tile's 128 bytes hold 256 int4 codes of K).
template <int Stages, int XB = 1, class SM>
__device__ __forceinline__ void produce(unsigned* err, SM& sm, const CUtensorMap* tw, const CUtensorMap* tx,
                                        int a, int b, int KT, int kx_elems_per_tile,
                                        unsigned tx_bytes) {
    prefetch_tensormap(tw);
    if (tx) prefetch_tensormap(tx);
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const int n = b - a;
    const int pre0 = Stages < kPreWaitTiles ? Stages : kPreWaitTiles;
    const int pre = n < pre0 ? n : pre0;
    for (int j = 0; j < pre; ++j) {
        const int tile = a + j, nt = tile / KT, kt = tile - nt * KT;
        mbar_arrive_expect_tx(&sm.full[j], tx_bytes);
        tma_load_2d(sm.w_tile(j), tw, kt * kx_elems_per_tile, nt * BN, &sm.full[j], pol_w);
    }
    grid_dependency_wait();
    if (tx) {
        for (int j = 0; j < pre; ++j) {
            const int tile = a + j, kt = tile % KT;
#pragma unroll
            for (int xb = 0; xb < XB; ++xb)
                tma_load_2d(sm.x_box(j, xb), tx, (kt * XB + xb) * kx_elems_per_tile, 0, &sm.full[j], pol_x);
        }
    }
    int issued = pre;
    int s = pre % Stages;
    int round = pre / Stages;
    for (int j = pre; j < n; ++j) {
        if (!mbar_wait_bounded_sleep(&sm.empty[s], (round - 1) & 1, sm.abort, 64)) {
            atomicOr(err, kErrEmptyWait);
            break;
        }
        const int tile = a + j, nt = tile / KT, kt = tile - nt * KT;
        mbar_arrive_expect_tx(&sm.full[s], tx_bytes);
        tma_load_2d(sm.w_tile(s), tw, kt * kx_elems_per_tile, nt * BN, &sm.full[s], pol_w);
        if (tx) {
#pragma unroll
            for (int xb = 0; xb < XB; ++xb)
                tma_load_2d(sm.x_box(s, xb), tx, (kt * XB + xb) * kx_elems_per_tile, 0, &sm.full[s], pol_x);
        }
        ++issued;
        if (++s == Stages) { s = 0; ++round; }
    }
    // Do not leave the CTA while copies into its shared memory are in flight.
    const int first = issued > Stages ? issued - Stages : 0;
    for (int j = first; j < issued; ++j) {
        const int st = j % Stages, par = (j / Stages) & 1;
        if (mbar_try_wait(&sm.full[st], par)) continue;
        unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&sm.full[st], par)) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                atomicOr(err, kErrDrainWait);
                return;
            }
        }
    }
}

struct W8A8Params {
    int M, N, K, KT, NT;
    long long T;
    const float* sx;
    const float* sw;
    void* y;
    int y_bf16;
    int32_t* acc_debug;
    int32_t* tokens;
    float* max_logit;
    unsigned long long* slots;   // split-K partials: one BN x MP slot per CTA
    unsigned long long* keys;
    unsigned* done;
    unsigned long long slot_wait_ns;   // limit of the split-K head's wait (kWaitLimitNs by default)
    int drop_partials;                 // test hook: publish no split-K partial sums
};

// ---------------------------------------------------------------------------
// Split-K combination through per-CTA slots of tagged words.
//
// A channel tile whose K range is split over CTAs has exactly one segment
// that starts at K-tile 0: the head, which is the last segment of the CTA
// that holds it (that CTA's range ends inside the tile). Every other segment
// of the tile is the first segment of a later CTA. Those CTAs publish their
// partial sums into their own slot as 64-bit words (1 << 32 | 32-bit value):
// an aligned 64-bit access is single-copy atomic, so a reader that sees the
// tag also sees the value, and publishing needs no fence and no counter. The
// head's CTA adds the slots of the CTAs after it whose ranges start inside
// the tile (read with relaxed loads; words still untagged are re-read
// together until they are tagged, with a time limit), zeroes them and
// finishes the tile. The wait is one-way
// (a CTA waits only on CTAs with a higher index, which publish before they
// wait on anything) and every CTA of the grid is resident before a later
// kernel can take an SM (each CTA allows dependent launches only once it
// runs), so it always ends.
//
// Slot layout: slot c = slots + c * BN * MP words, word [token m][row r].
// ---------------------------------------------------------------------------
constexpr unsigned long long kSlotTag = 1ull << 32;

__device__ __forceinline__ void st_relaxed_v2_u64(unsigned long long* p, unsigned long long a,
                                                  unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" :: "l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ld_relaxed_v2_u64(const unsigned long long* p, unsigned long long& a,
                                                  unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Publish this CTA's staged partial sums (stg[row * SM::SP + token], 32-bit
// words; SP is the staging row stride, MP plus a padding that keeps the
// per-row accesses of a warp on distinct banks) into its slot. The caller synchronises the consumers afterwards
// before stg is written again.
template <int MP, int CW, class SM>
__device__ __forceinline__ void publish_partial(SM& sm, unsigned long long* slots, int M, int tid) {
    constexpr int CT = CW * 32;
    constexpr int SP = SM::SP;
    unsigned long long* slot = slots + (size_t)blockIdx.x * (BN * MP);
    const uint32_t* stg = reinterpret_cast<const uint32_t*>(sm.stg);
    for (int q = tid; q < M * (BN / 2); q += CT) {
        const int m = q / (BN / 2), r = 2 * (q - m * (BN / 2));
        st_relaxed_v2_u64(slot + m * BN + r, kSlotTag | stg[r * SP + m], kSlotTag | stg[(r + 1) * SP + m]);
    }
}

// With this CTA's stream-K range ending at tile index b (exclusive), one
// past the last CTA whose range starts inside the channel tile of tile b-1:
// CTA c starts at floor(c*T/G), so that is the first c with c*T >= E*G,
// E = the end of that channel tile. Computed once, before the grid
// dependency wait.
__device__ __forceinline__ int split_contributors_end(long long T, int KT, int b) {
    const long long G = gridDim.x;
    const long long E = (long long)((b - 1) / KT + 1) * KT;
    const long long c2 = (E * G + T - 1) / T;
    return (int)(c2 < G ? c2 : G);
}

// Head segment of a split tile: add the partials of CTAs blockIdx.x+1 ..
// c2-1 (whose ranges start inside the tile; in CTA order, i.e. in K order)
// onto stg, zeroing their slots. Integer sums (FLOAT = false) or fp32 sums.
// The caller synchronises the consumers before and after.
template <int MP, int CW, bool FLOAT, class SM>
__device__ __forceinline__ void gather_partials(SM& sm, unsigned long long* slots, int M, int c2, int tid,
                                                unsigned* err, unsigned long long limit_ns = kWaitLimitNs) {
    constexpr int CT = CW * 32;
    // Pairs of words per thread and contributor slots per batch in flight:
    // every round of loads is one L2 round trip, so with many token rows
    // each thread keeps more pairs in flight (a split tile has few
    // contributors then); QP * CB stays 16 to bound the registers.
    constexpr int QP = MP >= 64 ? 8 : MP >= 32 ? 4 : 2;
    constexpr int CB = 16 / QP;
    constexpr int SP = SM::SP;
    const int c1 = blockIdx.x + 1;
    uint32_t* stg = reinterpret_cast<uint32_t*>(sm.stg);
    const int pairs = M * (BN / 2);
    for (int q0 = tid; q0 < pairs; q0 += QP * CT) {
        int off[QP];
        uint32_t s[QP][2];
#pragma unroll
        for (int u = 0; u < QP; ++u) {
            const int q = q0 + u * CT;
            const int m = q / (BN / 2), r = 2 * (q - m * (BN / 2));
            off[u] = m * BN + r;
            if (q < pairs) {
                s[u][0] = stg[r * SP + m];
                s[u][1] = stg[(r + 1) * SP + m];
            }
        }
        for (int c = c1; c < c2; c += CB) {
            unsigned long long w[CB][QP][2];
#pragma unroll
            for (int j = 0; j < CB; ++j)
#pragma unroll
                for (int u = 0; u < QP; ++u)
                    if (c + j < c2 && q0 + u * CT < pairs)
                        ld_relaxed_v2_u64(slots + (size_t)(c + j) * (BN * MP) + off[u], w[j][u][0], w[j][u][1]);
            // Words still untagged: re-read all of them together (one round
            // trip per polling round), up to the time limit.
            unsigned long long t0 = 0;
            while (true) {
                bool pending = false;
#pragma unroll
                for (int j = 0; j < CB; ++j)
#pragma unroll
                    for (int u = 0; u < QP; ++u)
                        if (c + j < c2 && q0 + u * CT < pairs && !((w[j][u][0] & w[j][u][1]) >> 32))
                            pending = true;
                if (!pending) break;
                if (t0 == 0) {
                    t0 = global_timer_ns();
                } else if (global_timer_ns() - t0 > limit_ns) {
                    atomicOr(err, kErrSlotWait);
                    break;
                }
                __nanosleep(20);
#pragma unroll
                for (int j = 0; j < CB; ++j)
#pragma unroll
                    for (int u = 0; u < QP; ++u)
                        if (c + j < c2 && q0 + u * CT < pairs && !((w[j][u][0] & w[j][u][1]) >> 32))
                            ld_relaxed_v2_u64(slots + (size_t)(c + j) * (BN * MP) + off[u], w[j][u][0],
                                              w[j][u][1]);
            }
#pragma unroll
            for (int j = 0; j < CB; ++j)
#pragma unroll
                for (int u = 0; u < QP; ++u)
                    if (c + j < c2 && q0 + u * CT < pairs) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t v = (uint32_t)w[j][u][h];
                            s[u][h] = FLOAT ? __float_as_uint(__uint_as_float(s[u][h]) + __uint_as_float(v))
                                            : s[u][h] + v;
                        }
                        st_relaxed_v2_u64(slots + (size_t)(c + j) * (BN * MP) + off[u], 0ull, 0ull);
                    }
        }
#pragma unroll
        for (int u = 0; u < QP; ++u) {
            const int q = q0 + u * CT;
            if (q < pairs) {
                const int m = q / (BN / 2), r = 2 * (q - m * (BN / 2));
                stg[r * SP + m] = s[u][0];
                stg[(r + 1) * SP + m] = s[u][1];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Epilogue of the W8A8 streaming kernels, run by the CW consumer warps
// (thread index tid in [0, 32*CW)).
//
// The LM head finishes a tile by folding each token's best (logit, index)
// key into a global atomicMax word and counts finished tiles per CTA; one
// counter add per CTA at the end decides which CTA decodes the keys (the
// last one), then zeroes them.
//
// Linear: y = fl(fl(acc) * fl(sx * sw)) per element. LM head key:
// (order-preserving bits of y) << 32 | (0xFFFFFFFF - v), so the largest key
// is the largest logit and, among equal logits, the lowest index.
// ---------------------------------------------------------------------------
struct EpiState {
    int c2 = 0;               // split_contributors_end of the CTA's range
    float swn = 0.f;          // channel scale of this thread's row in the current tile
                              // (SwiGLU: of gate row tid % 64)
    float swn_up = 0.f;       // SwiGLU: the scale of up row tid % 64 + 64
    unsigned tiles_done = 0;  // LM head: channel tiles this CTA finished
};

// At the start of a segment of channel tile nt: load the channel scale the
// finish needs, so that its latency hides behind the segment's MMAs.
template <int EPI>
__device__ __forceinline__ void segment_start(EpiState& st, const W8A8Params& p, int nt, int tid) {
    if (EPI == (int)Epi::SwiGLU) {
        const int n = nt * BN + (tid & (BN / 2 - 1));          // gate row; its up row is n + 64
        st.swn = n < p.N ? __ldg(&p.sw[n]) : 0.f;
        st.swn_up = n + BN / 2 < p.N ? __ldg(&p.sw[n + BN / 2]) : 0.f;
        return;
    }
    const int n = nt * BN + (tid & (BN - 1));
    st.swn = n < p.N ? __ldg(&p.sw[n]) : 0.f;
}

// Finish channel tile nt from its complete int32 sums in sm.stg.
template <int MP, int CW, int EPI, class SM>
__device__ __forceinline__ void finish_tile(SM& sm, const W8A8Params& p, int nt, int tid, EpiState& st) {
    constexpr int SP = SM::SP;
    const int warp = tid >> 5, lane = tid & 31;
    const float swn = st.swn;
    if (EPI == (int)Epi::Linear) {
        // TH threads per channel (all CW warps: with two per channel even 5
        // tokens finish measurably sooner), thread h taking tokens h, h + TH, ...
        constexpr int TH = (CW * 32 >= 2 * BN) ? 2 : 1;
        const int rr = tid & (BN - 1), h = tid / BN;
        const int nn = nt * BN + rr;
        if (h < TH && nn < p.N) {
#pragma unroll 4
            for (int m = h; m < MP; m += TH) {
                if (m < p.M) {
                    const int32_t am = sm.stg[rr * SP + m];
                    if (p.acc_debug) p.acc_debug[(size_t)m * p.N + nn] = am;
                    const float yv = __fmul_rn(__int2float_rn(am), __fmul_rn(sm.sx[m], swn));
                    if (p.y_bf16)
                        reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)m * p.N + nn] = __float2bfloat16_rn(yv);
                    else
                        reinterpret_cast<float*>(p.y)[(size_t)m * p.N + nn] = yv;
                }
            }
        }
    } else if (EPI == (int)Epi::SwiGLU) {
        // rows r and r + 64 of the tile: gate and up of feature f; the
        // CW * 32 / 64 threads of a feature take tokens h, h + TH, ...
        constexpr int TH = CW * 32 / (BN / 2);
        const int r = tid & (BN / 2 - 1), h = tid / (BN / 2);
        const int f = nt * (BN / 2) + r;
        if (h < TH && 2 * f < p.N) {
            float* a = reinterpret_cast<float*>(p.y);
            const int F = p.N / 2;
#pragma unroll 4
            for (int m = h; m < MP; m += TH) {
                if (m < p.M) {
                    const float sxm = sm.sx[m];
                    const float yg = __fmul_rn(__int2float_rn(sm.stg[r * SP + m]), __fmul_rn(sxm, swn));
                    const float yu = __fmul_rn(__int2float_rn(sm.stg[(r + BN / 2) * SP + m]),
                                               __fmul_rn(sxm, st.swn_up));
                    a[(size_t)m * F + f] = __fmul_rn(silu(yg), yu);
                }
            }
        }
    } else {
        // TH threads per channel as in the linear epilogue: warp w covers
        // channels 32 * (w % 4) .. +31 of the tile and tokens m = w / 4 mod TH.
        // A token's best key over the warp's channels is the largest
        // order-preserving logit bits, then the largest 0xFFFFFFFF - n among
        // the lanes holding them (the lowest index), each one warp reduction.
        constexpr int TH = (CW * 32 >= 2 * BN) ? 2 : 1;
        const int rr = tid & (BN - 1), h = tid / BN;
        const int nn = nt * BN + rr;
        const bool ok = nn < p.N;
        if (h < TH) {
#pragma unroll 4
            for (int m = h; m < MP; m += TH) {
                if (m < p.M) {
                    unsigned o = 0u, k2 = 0u;
                    if (ok) {
                        const float yv = __fmul_rn(__int2float_rn(sm.stg[rr * SP + m]), __fmul_rn(sm.sx[m], swn));
                        o = ordered_bits(yv);
                        k2 = 0xFFFFFFFFu - (unsigned)nn;
                    }
                    const unsigned om = __reduce_max_sync(0xffffffffu, o);
                    const unsigned km = __reduce_max_sync(0xffffffffu, o == om ? k2 : 0u);
                    if (lane == 0) sm.red[warp * MP + m] = ((unsigned long long)om << 32) | km;
                }
            }
        }
        consumer_sync<CW>();
        if (tid < p.M) {
            const int w0 = (tid % TH) * (BN / 32);
            unsigned long long k = sm.red[w0 * MP + tid];
#pragma unroll
            for (int w = 1; w < BN / 32; ++w) {
                const unsigned long long o = sm.red[(w0 + w) * MP + tid];
                k = o > k ? o : k;
            }
            atomicMax(&p.keys[tid], k);
        }
        ++st.tiles_done;
    }
}

// End of a segment: the channel tile nt's sums over K-tiles [seg_begin,
// seg_begin + seg_len) (tile indices) are staged in sm.stg[row * SM::SP + token]
// and the consumers have synchronised.
template <int MP, int CW, int EPI, class SM>
__device__ __forceinline__ void segment_end(SM& sm, const W8A8Params& p, int nt, int seg_begin, int seg_len,
                                            int tid, EpiState& st, unsigned* err) {
    if (seg_len != p.KT) {
        if (seg_begin != nt * p.KT) {                 // not the head: publish
            if (!p.drop_partials) publish_partial<MP, CW>(sm, p.slots, p.M, tid);
            consumer_sync<CW>();
            return;
        }
        gather_partials<MP, CW, false>(sm, p.slots, p.M, st.c2, tid, err, p.slot_wait_ns);
        consumer_sync<CW>();
    }
    finish_tile<MP, CW, EPI>(sm, p, nt, tid, st);
    consumer_sync<CW>();   // staging buffer and reduction slots are reused
}

// After the CTA's last segment: the LM head's decode.
template <int MP, int CW, int EPI, class SM>
__device__ __forceinline__ void range_end(SM& sm, const W8A8Params& p, int tid, EpiState& st) {
    if (EPI == (int)Epi::LmHead && st.tiles_done > 0) {
        if (tid == 0) {
            __threadfence();
            const unsigned prev = atomicAdd(p.done, st.tiles_done);
            const bool last = prev + st.tiles_done == (unsigned)p.NT;
            if (last) __threadfence();
            *sm.flag = last ? 2 : 0;
        }
        consumer_sync<CW>();
        if (*sm.flag == 2) {
            if (tid < p.M) {
                const unsigned long long k = __ldcg(&p.keys[tid]);
                __stcg(&p.keys[tid], 0ull);
                p.tokens[tid] = (int32_t)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull));
                if (p.max_logit) p.max_logit[tid] = unordered_bits((unsigned)(k >> 32));
            }
            if (tid == 0) __stcg(p.done, 0u);
        }
    }
}

}  // namespace
}  // namespace qv
