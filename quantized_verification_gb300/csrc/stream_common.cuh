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

// Producer: stream tiles [a, b) into the ring. Weight tiles of the first
// ring fill are requested before the grid dependency wait. With tx == null
// only weight tiles travel (tx_bytes must then count the weight tile alone).
template <int Stages, class SM>
__device__ __forceinline__ void produce(unsigned* err, SM& sm, const CUtensorMap* tw, const CUtensorMap* tx,
                                        int a, int b, int KT, int kx_elems_per_tile,
                                        unsigned tx_bytes) {
    prefetch_tensormap(tw);
    if (tx) prefetch_tensormap(tx);
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const int n = b - a;
    const int pre = n < Stages ? n : Stages;
    for (int j = 0; j < pre; ++j) {
        const int tile = a + j, nt = tile / KT, kt = tile - nt * KT;
        mbar_arrive_expect_tx(&sm.full[j], tx_bytes);
        tma_load_2d(sm.w_tile(j), tw, kt * kx_elems_per_tile, nt * BN, &sm.full[j], pol_w);
    }
    grid_dependency_wait();
    if (tx) {
        for (int j = 0; j < pre; ++j) {
            const int tile = a + j, kt = tile % KT;
            tma_load_2d(sm.x_tile(j), tx, kt * kx_elems_per_tile, 0, &sm.full[j], pol_x);
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
        if (tx) tma_load_2d(sm.x_tile(s), tx, kt * kx_elems_per_tile, 0, &sm.full[s], pol_x);
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
    int32_t* ws_acc;
    unsigned* ws_cnt;
    unsigned long long* keys;
    unsigned* done;
};

// ---------------------------------------------------------------------------
// Epilogue of the W8A8 streaming kernels, run by the CW consumer warps
// (thread index tid in [0, 32*CW)).
//
// A channel tile whose K range is split over CTAs is combined with int32
// atomic adds into the workspace (exact, so order does not matter); the CTA
// whose contribution completes the tile (the one that brings the tile's
// counter to KT) finishes it, reading the sums and zeroing them, so the
// workspace is left zeroed. Only thread 0 fences, after the CTA barrier that
// orders the other threads' adds before it (and, on the finishing side,
// before the barrier that releases the reads).
//
// A CTA's stream-K range starts with at most one partial segment that is not
// its last; that segment's counter result is not needed until the range
// ends, so the CTA keeps streaming and finishes the tile (if its add was the
// last) after its final segment. The LM head finishes a tile by folding
// each token's best (logit, index) key into a global atomicMax word and
// counts finished tiles per CTA; one counter add per CTA at the end decides
// which CTA decodes the keys (the last one), then zeroes them.
//
// Linear: y = fl(fl(acc) * fl(sx * sw)) per element. LM head key:
// (order-preserving bits of y) << 32 | (0xFFFFFFFF - v), so the largest key
// is the largest logit and, among equal logits, the lowest index.
// ---------------------------------------------------------------------------
struct EpiState {
    int def_nt = -1;          // channel tile of the deferred partial contribution
    int def_len = 0;
    unsigned def_prev = 0;    // thread 0: tile counter before that contribution
    unsigned tiles_done = 0;  // LM head: channel tiles this CTA finished
};

// Finish channel tile nt from sm.stg (from_ws = false) or from the workspace.
template <int MP, int CW, int EPI, class SM>
__device__ __forceinline__ void finish_tile(SM& sm, const W8A8Params& p, int nt, bool from_ws, int tid,
                                            EpiState& st) {
    const int warp = tid >> 5, lane = tid & 31;
    int32_t* gacc = p.ws_acc + (size_t)nt * BN * MP;
    // the first BN consumer threads (warps 0..3) own one output channel each
    const int r = tid;
    const int n = nt * BN + r;
    const bool valid = r < BN && n < p.N;
    int32_t acc[MP];
#pragma unroll
    for (int m = 0; m < MP; ++m) acc[m] = 0;
    if (valid) {
#pragma unroll
        for (int m = 0; m < MP; ++m)
            if (m < p.M) acc[m] = from_ws ? __ldcg(&gacc[r * MP + m]) : sm.stg[r * MP + m];
        if (from_ws) {
#pragma unroll
            for (int m = 0; m < MP; ++m)
                if (m < p.M) __stcg(&gacc[r * MP + m], 0);
        }
    }
    const float swn = valid ? p.sw[n] : 0.f;
    if (EPI == (int)Epi::Linear) {
        if (valid) {
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                if (m < p.M) {
                    if (p.acc_debug) p.acc_debug[(size_t)m * p.N + n] = acc[m];
                    const float yv = __fmul_rn(__int2float_rn(acc[m]), __fmul_rn(sm.sx[m], swn));
                    if (p.y_bf16)
                        reinterpret_cast<__nv_bfloat16*>(p.y)[(size_t)m * p.N + n] = __float2bfloat16_rn(yv);
                    else
                        reinterpret_cast<float*>(p.y)[(size_t)m * p.N + n] = yv;
                }
            }
        }
    } else {
        if (r < BN) {
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                if (m < p.M) {
                    unsigned long long key = 0ull;
                    if (valid) {
                        const float yv = __fmul_rn(__int2float_rn(acc[m]), __fmul_rn(sm.sx[m], swn));
                        key = ((unsigned long long)ordered_bits(yv) << 32) |
                              (unsigned long long)(0xFFFFFFFFu - (unsigned)n);
                    }
                    key = warp_max_u64(key);
                    if (lane == 0) sm.red[warp * MP + m] = key;
                }
            }
        }
        consumer_sync<CW>();
        if (tid < p.M) {
            unsigned long long k = sm.red[tid];
#pragma unroll
            for (int w = 1; w < BN / 32; ++w) {
                const unsigned long long o = sm.red[w * MP + tid];
                k = o > k ? o : k;
            }
            atomicMax(&p.keys[tid], k);
        }
        ++st.tiles_done;
    }
    if (from_ws && tid == 0) __stcg(&p.ws_cnt[nt], 0u);
}

// End of a segment (the channel tile nt's sums over seg_len of its K-tiles
// are staged in sm.stg[row * MP + token] and the consumers have synchronised);
// last_seg: this is the CTA's final segment.
template <int MP, int CW, int EPI, class SM>
__device__ __forceinline__ void segment_end(SM& sm, const W8A8Params& p, int nt, int seg_len,
                                            bool last_seg, int tid, EpiState& st) {
    constexpr int CT = CW * 32;
    if (seg_len == p.KT) {
        finish_tile<MP, CW, EPI>(sm, p, nt, false, tid, st);
        consumer_sync<CW>();   // staging buffer and reduction slots are reused
        return;
    }
    int32_t* gacc = p.ws_acc + (size_t)nt * BN * MP;
    for (int e = tid; e < BN * MP; e += CT) {
        const int r = e / MP, m = e - (e / MP) * MP;
        if (m < p.M && nt * BN + r < p.N) atomicAdd(&gacc[e], sm.stg[e]);
    }
    consumer_sync<CW>();
    unsigned prev = 0;
    if (tid == 0) {
        __threadfence();
        prev = atomicAdd(&p.ws_cnt[nt], (unsigned)seg_len);
    }
    if (!last_seg) {
        st.def_nt = nt;
        st.def_len = seg_len;
        if (tid == 0) st.def_prev = prev;   // read only when the range ends
        return;
    }
    if (tid == 0) {
        const bool fin = prev + (unsigned)seg_len == (unsigned)p.KT;
        if (fin) __threadfence();
        *sm.flag = fin ? 1 : 0;
    }
    consumer_sync<CW>();
    if (*sm.flag) finish_tile<MP, CW, EPI>(sm, p, nt, true, tid, st);
    consumer_sync<CW>();
}

// After the CTA's last segment: the deferred tile, then the LM head's decode.
template <int MP, int CW, int EPI, class SM>
__device__ __forceinline__ void range_end(SM& sm, const W8A8Params& p, int tid, EpiState& st) {
    if (st.def_nt >= 0) {
        if (tid == 0) {
            const bool fin = st.def_prev + (unsigned)st.def_len == (unsigned)p.KT;
            if (fin) __threadfence();
            *sm.flag = fin ? 1 : 0;
        }
        consumer_sync<CW>();
        if (*sm.flag) finish_tile<MP, CW, EPI>(sm, p, st.def_nt, true, tid, st);
        consumer_sync<CW>();
    }
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
