// k_tc_gemm.cu -- the W8A8 weight-streaming GEMM on the fifth-generation
// tensor cores (tcgen05): y = dequant(xq . wq^T) (qv_w8a8_linear) and the LM
// head fused with the greedy argmax (qv_lm_head_argmax).
//   Quasar, gist.science/ja summary, section 2.2 item 3 (INT8 GEMM with INT32
//   accumulation, dequantization to high precision); gist.science/it summary,
//   section 2 item 3 (logits kept precise for the acceptance test).
//
// sm_103a has no integer kind for tcgen05.mma, so the int8 codes are widened
// exactly to binary16 and multiplied with kind::f16 into an f32 accumulator
// in tensor memory. Every product is an integer of magnitude <= 2^14 and one
// tile sums 128 of them (|sum| <= 2^21 < 2^24), so every partial sum is an
// exact binary32 integer; each tile's accumulator is read back, converted to
// int32 and added in registers, which makes the result the exact int32 dot
// product whatever the order of the tensor core's additions.
//
// Work split: the same stream-K order as the mma.sync kernels (tiles of 128
// output channels x 128 bytes of K, channel-tile major; each CTA one
// contiguous equal range), the same TMA producer and ring, and the same
// split-K / argmax epilogue. Per CTA (one per SM):
//  - warp 9, one thread: TMA producer (weights before the grid-dependency
//    wait, activation codes after it);
//  - warps 0-7, "converters": thread (warp w, lane l) owns output channel
//    32 * (w % 4) + l of the tile and half w / 4 of its 128 K bytes. It widens
//    its 64 weight bytes to 32 f16x2 words and stores them in its TMEM lane
//    (the MMA's A operand, channel = lane, K along the columns); together
//    the converters widen the MP x 128 activation codes into a shared-memory
//    f16 buffer in the 128-byte-swizzled K-major layout (the B operand);
//  - warp 8, one thread: issues the tile's eight M=128 x N x K=16 MMAs into a
//    TMEM accumulator and commits them to an mbarrier;
//  - the MMAs of up to eight consecutive tiles of a channel tile (K = 1024:
//    |sum| <= 1024 * 128^2 = 2^24, still exact in fp32) accumulate into one of
//    two TMEM accumulators; the converters read a group's accumulator back
//    (thread = channel, its half of the token columns) while they widen the
//    next group, convert to int32 and add it to the channel tile's running
//    sums, kept in the epilogue's shared-memory staging buffer, which the
//    common epilogue reads at the end of the channel tile's K range.
// A and B rotate through four slots (two at 80 tokens), so widening of the
// next tiles overlaps the MMAs of tile i.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "qv_internal.h"
#include "qv_ptx.cuh"
#include "stream_common.cuh"

namespace qv {

__device__ unsigned int g_tc_gemm_error;

namespace {

constexpr int kTcConv = 8;          // converter warps 0..7
constexpr int kTcMmaWarp = 8;       // MMA issue and TMEM allocation
constexpr int kTcProdWarp = 9;      // TMA producer
constexpr int kTcThreads = 10 * 32;
constexpr int kTcACols = 64;        // TMEM columns of one A slot (128 f16 of K per lane)
constexpr int kTcGroup = 8;         // tiles accumulated in TMEM before a readout

template <int MP>
struct TcCfg {
    static constexpr int NM = MP < 16 ? 16 : MP;          // MMA N: tokens padded to 16
    static constexpr int MPH = NM / 2;                    // accumulator columns per converter thread
    // A / B operand slots (four, two at 80 tokens for shared memory; two
    // were measured as fast as four at 64 tokens)
    static constexpr int R = MP > 64 ? 2 : 4;
    static constexpr int XBytes = MP * BKB;
    static constexpr int XSlot = ((XBytes + 1023) / 1024) * 1024;
    static constexpr int StageBytes = kWTileBytes + XSlot;
    static constexpr int BSlot = 2 * NM * 128;            // two 64-element K blocks of f16 rows
    static constexpr int Stages = MP <= 16 ? 8 : MP == 32 ? 7 : 5;
    // staging [channel][token] with an odd row stride: a warp's 32 channels
    // of one token fall on 32 distinct banks (a stride of MP = 64 words put
    // them all on one bank: 32-way conflicts in every staging access)
    static constexpr int SP = MP + 1;
    static constexpr int StgWords = BN * SP;
    static constexpr int DCol0 = R * kTcACols;            // first accumulator column
    static constexpr int TmemCols = 512;
    static constexpr int SmemBytes = 1024 + Stages * StageBytes + R * BSlot + StgWords * 4 +
                                     (2 * Stages + 2 * R + 2) * 8 + kMaxConsumerWarps * MP * 8 +
                                     MP * 4 + 64;
    static_assert(DCol0 + 2 * NM <= TmemCols, "TMEM budget");
    static_assert(SmemBytes <= 232448, "shared memory budget");
    static_assert(NM % 16 == 0 && NM <= 256, "MMA N");
    static_assert(MPH % 8 == 0 && (MPH <= 32 || MPH == 40), "accumulator readout widths");
};

template <int MP>
struct TcSmem {
    using C = TcCfg<MP>;
    static constexpr int SP = C::SP;
    uint8_t* stages;           // Stages x (W tile | X tile), 1024-aligned
    uint8_t* bring;            // R x BSlot f16 activation operands
    int32_t* stg;              // BN x MP staged sums
    uint64_t* full;
    uint64_t* empty;
    uint64_t* aready;          // converters -> MMA: A and B of a slot written
    uint64_t* mdone;           // MMA -> converters: slot's MMAs complete (A, B reusable)
    uint64_t* dfull;           // MMA -> converters: a group's accumulator complete (2)
    unsigned long long* red;   // kMaxConsumerWarps x MP (LM head)
    float* sx;                 // MP
    volatile int* abort;
    volatile int* flag;
    uint32_t* tmem_base;

    __device__ __forceinline__ explicit TcSmem(uint8_t* raw) {
        uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023);
        uint8_t* p = reinterpret_cast<uint8_t*>(base);
        stages = p;
        p += C::Stages * C::StageBytes;
        bring = p;
        p += C::R * C::BSlot;
        stg = reinterpret_cast<int32_t*>(p);
        p += C::StgWords * 4;
        full = reinterpret_cast<uint64_t*>(p);
        p += C::Stages * 8;
        empty = reinterpret_cast<uint64_t*>(p);
        p += C::Stages * 8;
        aready = reinterpret_cast<uint64_t*>(p);
        p += C::R * 8;
        mdone = reinterpret_cast<uint64_t*>(p);
        p += C::R * 8;
        dfull = reinterpret_cast<uint64_t*>(p);
        p += 2 * 8;
        red = reinterpret_cast<unsigned long long*>(p);
        p += kMaxConsumerWarps * MP * 8;
        sx = reinterpret_cast<float*>(p);
        p += MP * 4;
        abort = reinterpret_cast<volatile int*>(p);
        flag = reinterpret_cast<volatile int*>(p + 4);
        tmem_base = reinterpret_cast<uint32_t*>(p + 8);
    }
    __device__ __forceinline__ uint8_t* w_tile(int s) { return stages + s * C::StageBytes; }
    __device__ __forceinline__ uint8_t* x_tile(int s) { return stages + s * C::StageBytes + kWTileBytes; }
    __device__ __forceinline__ uint8_t* x_box(int s, int j) { return x_tile(s) + j * MP * BKB; }
    __device__ __forceinline__ uint8_t* b_slot(int j) { return bring + j * C::BSlot; }
};

// Hot-loop waits of this kernel (a non-suspending test_wait loop was
// measured no faster).
__device__ __forceinline__ bool tc_wait(uint64_t* bar, unsigned parity, volatile int* abort) {
    return mbar_wait_bounded(bar, parity, abort);
}

// Wait for an mbarrier phase for at most kWaitLimitNs, whatever the abort
// flag says (used before releasing tensor memory an MMA may still write).
__device__ __forceinline__ bool mbar_wait_timed(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    return true;
}

template <int MP, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
w8a8_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
               const __grid_constant__ CUtensorMap tmap_x, const W8A8Params p) {
    using C = TcCfg<MP>;
    constexpr int NM = C::NM, MPH = C::MPH, Stages = C::Stages, R = C::R;
    extern __shared__ uint8_t smem_raw[];
    TcSmem<MP> sm(smem_raw);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const long long G = gridDim.x;
    const int a = (int)((long long)blockIdx.x * p.T / G);
    const int b = (int)((long long)(blockIdx.x + 1) * p.T / G);
    const int n = b - a;

    if (tid == 0) {
        for (int s = 0; s < Stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kTcConv);
        }
        for (int j = 0; j < R; ++j) {
            mbar_init(&sm.aready[j], kTcConv);
            mbar_init(&sm.mdone[j], 1);
        }
        mbar_init(&sm.dfull[0], 1);
        mbar_init(&sm.dfull[1], 1);
        *sm.abort = 0;
        fence_barrier_init();
    }
    // Zero the activation operand slots once: rows MP..NM-1 (token padding of
    // the MMA's N) are never written again and must hold finite values.
    for (int e = tid; e < R * C::BSlot / 16; e += kTcThreads)
        reinterpret_cast<uint4*>(sm.bring)[e] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == kTcMmaWarp) {
        tmem_alloc(sm.tmem_base, C::TmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_base;
    allow_dependent_launch();

    if (warp == kTcProdWarp) {
        if (lane == 0)
            produce<Stages>(&g_tc_gemm_error, sm, &tmap_w, &tmap_x, a, b, p.KT, BKB,
                            (unsigned)(kWTileBytes + C::XBytes));
        return;
    }

    if (warp == kTcMmaWarp) {
        // ---------------- MMA issue ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, NM);
            int gq = -1, pos = kTcGroup;
            int kt = a % p.KT;                   // K-tile index of tile a + c
            for (int c = 0; c < n; ++c) {
                const int j = c % R;
                if (c == 0 || kt == 0 || pos == kTcGroup) { ++gq; pos = 0; }
                if (!mbar_wait_bounded_sleep(&sm.aready[j], (unsigned)(c / R) & 1u, sm.abort, 32))
                    atomicOr(&g_tc_gemm_error, kErrTcWait);
                tc_fence_after();
                const uint32_t a_t = tmem + (uint32_t)(j * kTcACols);
                const uint32_t d_t = tmem + (uint32_t)(C::DCol0 + (gq & 1) * NM);
                const uint32_t b_s = smem_u32(sm.b_slot(j));
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    umma_f16_ta(d_t, a_t + (uint32_t)(8 * t),
                                sw128_kmajor_desc(b_s + (uint32_t)((t >> 2) * NM * 128 + 32 * (t & 3))),
                                idesc, (pos > 0 || t > 0) ? 1u : 0u);
                umma_commit(&sm.mdone[j]);
                ++pos;
                if (++kt == p.KT) kt = 0;
                if (c + 1 == n || kt == 0 || pos == kTcGroup) umma_commit(&sm.dfull[gq & 1]);
            }
            // Tensor memory stays allocated until the last MMA has completed.
            if (n > 0 && !mbar_wait_timed(&sm.mdone[(n - 1) % R], (unsigned)((n - 1) / R) & 1u))
                atomicOr(&g_tc_gemm_error, kErrTcWait);
        }
        __syncwarp();
        named_bar_sync(2, (kTcConv + 1) * 32);
        tc_fence_after();
        tmem_dealloc(tmem, C::TmemCols);
        return;
    }

    // ---------------- converters (warps 0..7) ----------------
    const int qd = warp & 3;                 // TMEM lane quarter of this warp
    const int h = warp >> 2;                 // K half (widening) and token half (readout)
    const int row = 32 * qd + lane;          // output channel within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
    EpiState est;
    est.c2 = split_contributors_end(p.T, p.KT, b);
    grid_dependency_wait();
    if (tid < MP) sm.sx[tid] = tid < p.M ? p.sx[tid] : 0.f;
    consumer_sync<kTcConv>();
    const bool has_tokens = h * MPH < p.M;  // warp-uniform

    // The channel tile's running int32 sums live in this thread's part of the
    // staging buffer (row `row`, tokens h * MPH .. +MPH-1; the odd row stride
    // keeps a warp's accesses on distinct banks), which the epilogue reads.
    int32_t* accs = sm.stg + row * C::SP + h * MPH;
    // Group g's accumulator (buffer g & 1) completes on dfull[g & 1], the
    // (g >> 1)-th phase of that barrier.
    auto read_group = [&](int g) {
        if (!tc_wait(&sm.dfull[g & 1], (unsigned)(g >> 1) & 1u, sm.abort))
            atomicOr(&g_tc_gemm_error, kErrTcWait);
        tc_fence_after();
        if (has_tokens) {
            const uint32_t col = lane_base + (uint32_t)(C::DCol0 + (g & 1) * NM + h * MPH);
            constexpr int V0 = MPH > 32 ? 32 : MPH;   // columns in a first load, the rest (8) in a second
            uint32_t v[V0], v2[8];
            tmem_ld<V0>(col, v);
            if constexpr (MPH > 32) tmem_ld<8>(col + 32, v2);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < V0; ++m)
                if (h * MPH + m < MP) accs[m] += __float2int_rn(__uint_as_float(v[m]));
            if constexpr (MPH > 32) {
#pragma unroll
                for (int m = 0; m < 8; ++m) accs[32 + m] += __float2int_rn(__uint_as_float(v2[m]));
            }
        }
    };
    int gq = -1, pos = kTcGroup;             // group of the current tile, position in it
    int rq = 0;                              // next group to read out

    // Shared-memory words of one tile held in registers: this thread's 64
    // weight bytes and its share of the activation codes. Within a segment,
    // tile c + 1's words are loaded (its stage waited for first) once tile
    // c's A operand is stored, so their latency overlaps the B widening and
    // the hand-off of tile c.
    constexpr int XI = (MP * 8 + kTcConv * 32 - 1) / (kTcConv * 32);   // activation items per thread
    auto load_tile = [&](int c, uint4 (&w)[4], uint4 (&x)[XI]) {
        const int s = c % Stages;
        if (!tc_wait(&sm.full[s], (unsigned)(c / Stages) & 1u, sm.abort))
            atomicOr(&g_tc_gemm_error, kErrFullWait);
        const uint8_t* wrow = sm.w_tile(s) + row * BKB;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            w[u] = *reinterpret_cast<const uint4*>(wrow + (((4 * h + u) ^ (row & 7)) << 4));
#pragma unroll
        for (int q = 0; q < XI; ++q) {
            const int e = tid + q * kTcConv * 32;
            const int xr = e >> 3, xc = e & 7;
            x[q] = e < MP * 8 ? *reinterpret_cast<const uint4*>(sm.x_tile(s) + xr * BKB + ((xc ^ (xr & 7)) << 4))
                              : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    int i = a;
    while (i < b) {
        const int nt = i / p.KT;
        const int seg_begin = i;
        const int seg_end = min(b, (nt + 1) * p.KT);
        segment_start<EPI>(est, p, nt, tid);
#pragma unroll
        for (int m = 0; m < MPH; ++m)
            if (h * MPH + m < MP) accs[m] = 0;

        for (; i < seg_end; ++i) {
            const int c = i - a;
            const int s = c % Stages, j = c % R;
            if (i == seg_begin || pos == kTcGroup) { ++gq; pos = 0; }
            uint4 wv[4], xv[XI];
            load_tile(c, wv, xv);
            // Slot j is free once the MMAs of tile c - R have completed.
            if (c >= R && !tc_wait(&sm.mdone[j], (unsigned)((c - R) / R) & 1u, sm.abort))
                atomicOr(&g_tc_gemm_error, kErrTcWait);
            // The previous group of this channel tile is read at the third
            // tile of the current group (two tiles after its last MMAs were
            // released, so they are normally complete); its buffer is written
            // again by the next group, so a group start reads anything older.
            if (pos == 0)
                while (rq < gq - 1) read_group(rq++);
            else if (pos == 2)
                while (rq < gq) read_group(rq++);
            ++pos;

            // A: 32 f16x2 words into this thread's TMEM lane.
            uint32_t av[32];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                widen_i8x4_f16(wv[u].x, av[8 * u + 0], av[8 * u + 1]);
                widen_i8x4_f16(wv[u].y, av[8 * u + 2], av[8 * u + 3]);
                widen_i8x4_f16(wv[u].z, av[8 * u + 4], av[8 * u + 5]);
                widen_i8x4_f16(wv[u].w, av[8 * u + 6], av[8 * u + 7]);
            }
            tmem_st_x32(lane_base + (uint32_t)(j * kTcACols + 32 * h), av);

            // B: the MP x 128 activation codes -> f16, 128-byte swizzled K-major.
            uint8_t* bs = sm.b_slot(j);
#pragma unroll
            for (int q = 0; q < XI; ++q) {
                const int e = tid + q * kTcConv * 32;
                if (e < MP * 8) {
                    const int xr = e >> 3, xc = e & 7;
                    uint4 lo, hi;
                    widen_i8x4_f16(xv[q].x, lo.x, lo.y);
                    widen_i8x4_f16(xv[q].y, lo.z, lo.w);
                    widen_i8x4_f16(xv[q].z, hi.x, hi.y);
                    widen_i8x4_f16(xv[q].w, hi.z, hi.w);
                    uint8_t* brow = bs + (xc >> 2) * NM * 128 + xr * 128;
                    const int c0 = 2 * (xc & 3);
                    *reinterpret_cast<uint4*>(brow + ((c0 ^ (xr & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4*>(brow + (((c0 + 1) ^ (xr & 7)) << 4)) = hi;
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.empty[s]);
                mbar_arrive(&sm.aready[j]);
            }

        }
        // Segment end: read the remaining accumulators of this channel tile
        // (the sums are then complete in the staging buffer).
        while (rq <= gq) read_group(rq++);
        consumer_sync<kTcConv>();
        segment_end<MP, kTcConv, EPI>(sm, p, nt, seg_begin, seg_end - seg_begin, tid, est, &g_tc_gemm_error);
    }
    range_end<MP, kTcConv, EPI>(sm, p, tid, est);
    tc_fence_before();
    named_bar_sync(2, (kTcConv + 1) * 32);
}

// Grid of the tcgen05 kernel: the fewest tiles per CTA s >= T / SMs that
// divide the K-tiles of a channel tile, so that every CTA's range is one
// segment of one channel tile, as long as that keeps at least 60 % of the
// SMs busy (80 % at 32 tokens, where qkv on 96 CTAs measured 15.7 against
// 14.7 us); otherwise one CTA per SM. With many tokens a split channel tile
// moves MP x 128 partial sums per contributor, and a range that straddles two
// channel tiles pays two segment ends: on the Qwen3-8B shapes at 64 tokens
// this took o from 20.2 to 16.2 us (128 CTAs of 8 tiles), qkv from 19.9 to
// 18.3 (96 x 16) and down from 29.9 to 27.0 (128 x 24). Ranges of whole
// channel tiles (gate|up on 96 CTAs: 50.2 against 40.3 us) and a 50 % floor
// (the Qwen3-32B shapes on 80 CTAs) measured slower.
int tc_grid(long long T, int KT, int MP, int num_sms) {
    const int g0 = stream_grid(T, num_sms);
    const long long floor10 = MP <= 32 ? 8 : 6;   // tenths of the SMs
    for (long long sz = (T + num_sms - 1) / num_sms; sz <= KT; ++sz) {
        if (KT % sz != 0) continue;
        const long long g = T / sz;
        return (10 * g >= floor10 * num_sms && g <= g0) ? (int)g : g0;
    }
    return g0;
}

template <class P, class... Args>
cudaError_t launch_tc(void (*kern)(Args...), int grid, int smem, cudaStream_t s,
                      const CUtensorMap& tw, const CUtensorMap& tx, const P& params) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tw, tx, params);
}

}  // namespace

cudaError_t launch_w8a8_tc(const W8A8Launch& a, int num_sms, cudaStream_t s) {
    const bool lm = a.epi == Epi::LmHead;
    WsLayout L = ws_layout(a.MP, a.N, lm);
    W8A8Params p;
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.KT = ceil_div(a.K, BKB);
    p.NT = ceil_div(a.N, BN);
    p.T = (long long)p.KT * p.NT;
    p.sx = a.sx; p.sw = a.sw; p.y = a.y; p.y_bf16 = a.y_bf16; p.acc_debug = a.acc_debug;
    p.tokens = a.tokens; p.max_logit = a.max_logit;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    p.slots = reinterpret_cast<unsigned long long*>(ws + L.slots);
    p.slot_wait_ns = kWaitLimitNs;
    p.drop_partials = 0;
    p.keys = reinterpret_cast<unsigned long long*>(ws + L.keys);
    p.done = reinterpret_cast<unsigned*>(ws + L.done);
    const int grid = tc_grid(p.T, p.KT, a.MP, num_sms);
#define QV_TC_LAUNCH(MPV, EPIV) \
    launch_tc(w8a8_tc_kernel<MPV, (int)EPIV>, grid, TcCfg<MPV>::SmemBytes, s, a.tmap_w, a.tmap_x, p)
#define QV_TC_CASE(MPV)                                                                           \
    case MPV:                                                                                     \
        return lm ? QV_TC_LAUNCH(MPV, Epi::LmHead)                                                \
                  : a.epi == Epi::SwiGLU ? QV_TC_LAUNCH(MPV, Epi::SwiGLU) : QV_TC_LAUNCH(MPV, Epi::Linear);
    switch (a.MP) {   // fewer tokens go to the mma.sync streaming kernel
        QV_TC_CASE(32)
        QV_TC_CASE(64)
        QV_TC_CASE(80)
        default: return cudaErrorInvalidValue;
    }
#undef QV_TC_CASE
#undef QV_TC_LAUNCH
}

cudaError_t read_and_clear_tc_gemm_error(unsigned* code) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_tc_gemm_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_tc_gemm_error, &zero, sizeof(unsigned));
}

}  // namespace qv
