// k_stream_gemm.cu -- weight-streaming GEMMs for skinny M on sm_103a.
//
//  * w8a8_stream_kernel: y = dequant(xq . wq^T) (qv_w8a8_linear) and the LM
//    head fused with the greedy argmax (qv_lm_head_argmax).
//      Quasar, gist.science/ja summary, section 2.2 item 3 (INT8 GEMM with
//      INT32 accumulation, dequantization to high precision);
//      gist.science/it summary, section 2 item 3 (logits kept precise for
//      the acceptance test).
//  * bf16_stream_kernel: the BF16-weight verifier used as the traffic
//    comparator (gist.science/ja summary, section 2.3; gist.science/de
//    summary, section 3 item 4).
//
// Design (both kernels):
//  - The weight matrix [N][K] is cut into tiles of 128 output channels x 128
//    bytes of K. Tiles are ordered channel-tile major, K minor, and each CTA
//    takes one contiguous, equally sized range of that order (stream-K), so
//    every SM streams the same number of bytes whatever N and K are.
//  - One producer thread moves tiles with 2-D TMA (128-byte swizzle) into a
//    ring of shared-memory stages guarded by mbarriers. The activation slice
//    of the same K range (M rows padded to MP, out-of-range rows zero-filled
//    by TMA) travels with each weight tile.
//  - Eight consumer warps each own 16 output channels of a tile and run
//    mma.sync with the output channels as the MMA's M and the tokens as its
//    N (token count padded to a multiple of 8).
//  - W8A8 with up to 8 tokens: int8 m16n8k32 MMA, exact int32 accumulation,
//    the ldmatrix words being the MMA fragments as they are. With more
//    tokens: int8 codes are widened exactly to binary16 in registers and run
//    through the f16 m16n8k16 MMA; products are at most 128^2 = 2^14, one
//    tile sums 128 of them (|sum| <= 2^21), so every fp32 partial is an
//    exact integer; after each tile it is converted to int32 and added.
//  - A channel tile whose K range is split over CTAs is combined through
//    per-CTA slots of tagged 64-bit words (stream_common.cuh): the segment
//    that starts at K-tile 0 (the head, the last segment of its CTA) waits,
//    with a 1 s %globaltimer limit, for the partial sums that the later CTAs
//    covering the rest of the tile publish into their slots, adds them
//    (exact integer sums), zeroes the slots and runs the epilogue, so the
//    workspace is left zeroed. A CTA only ever waits on CTAs with a higher
//    index, which publish before they wait on anything; a wait that runs
//    out sets kErrSlotWait in the device error word.
//  - The LM head reduces each finished channel tile to one 64-bit key per
//    token, (order-preserving bits of y) << 32 | (0xFFFFFFFF - v), combined
//    with atomicMax: the largest key is the largest logit and, among equal
//    logits, the lowest index. The last tile to finish decodes the keys.
//  - Programmatic dependent launch: weight tiles (never written by the
//    preceding kernels of this library) are requested before waiting for the
//    preceding kernel; activations, scales and workspace only afterwards.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "qv.h"
#include "qv_internal.h"
#include "qv_ptx.cuh"
#include "stream_common.cuh"

static_assert(qv::kErrFullWait == QV_DEVICE_ERR_FULL_WAIT && qv::kErrEmptyWait == QV_DEVICE_ERR_EMPTY_WAIT &&
                  qv::kErrDrainWait == QV_DEVICE_ERR_DRAIN_WAIT && qv::kErrGridWait == QV_DEVICE_ERR_GRID_WAIT &&
                  qv::kErrTcWait == QV_DEVICE_ERR_TC_WAIT && qv::kErrSlotWait == QV_DEVICE_ERR_SLOT_WAIT,
              "device error bits of qv.h");

namespace qv {

__device__ unsigned int g_stream_gemm_error;

namespace {


// Consumer warps per CTA (one more warp produces), and how many of the four
// 32-byte chunk pairs of each tile row go through the int8 tensor path; the
// rest are widened to binary16 and go through the f16 path. With 8 tokens or
// fewer the int8 path alone keeps up with HBM; with more tokens it would be
// the bottleneck and the f16 path is faster (measured on GB300).
constexpr int kW8A8Warps = 8;
constexpr int kBf16Warps = 8;
template <int NG>
__host__ __device__ constexpr int s8_pairs() { return NG == 1 ? 4 : 0; }

template <int NG, int XB = 1>
struct Cfg {
    static constexpr int MP = 8 * NG;                        // padded tokens
    static constexpr int XBytes = MP * BKB * XB;             // activation slice (XB boxes)
    static constexpr int XSlot = ((XBytes + 1023) / 1024) * 1024;
    static constexpr int StageBytes = kWTileBytes + XSlot;
    // Seven stages for up to 16 tokens also make a CTA need more than half of
    // an SM's shared memory, so no SM ever holds two CTAs of one launch (two
    // would share the SM's bandwidth and finish last).
    static constexpr int Stages = NG == 1 ? 7 : NG == 2 ? 7 : NG == 4 ? 5 : 4;
    // Epilogue staging [channel][token], row stride MP + 2: even, for the
    // 8-byte pair stores, and two words off a multiple of 32 so that the
    // per-channel reads of a warp spread over the banks.
    static constexpr int SP = MP + 2;
    static constexpr int StgWords = BN * SP;
    // W4A8 f16 path: the tile's activation codes as f16 MMA fragments, one
    // 16-byte word per (chunk, token group, lane), two tiles' worth
    static constexpr int XfBytes = XB == 2 ? 2 * 8 * NG * 32 * 16 : 0;
    static constexpr int SmemBytes =
        1024 /*alignment slack*/ + Stages * StageBytes + StgWords * 4 +
        2 * Stages * 8 + kMaxConsumerWarps * MP * 8 + MP * 4 + 64 + 16 + XfBytes;
    static_assert(SmemBytes > (int)kMinSmemOneCtaPerSm, "one CTA per SM");
};


// Shared-memory carve-up common to both kernels.
template <int Stages, int StageBytes, int StgWords, int MP>
struct Smem {
    static constexpr int SP = MP + 2;   // staging row stride (Cfg::SP)
    uint8_t* stages;          // Stages x StageBytes, 1024-aligned
    int32_t* stg;             // BN x MP staging words
    uint64_t* full;
    uint64_t* empty;
    unsigned long long* red;  // kMaxConsumerWarps x MP
    float* sx;                // MP
    volatile int* abort;
    volatile int* flag;
    uint8_t* xf;              // W4A8 f16 path: activation fragments (Cfg::XfBytes)

    __device__ __forceinline__ explicit Smem(uint8_t* raw) {
        uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023);
        uint8_t* p = reinterpret_cast<uint8_t*>(base);
        stages = p;
        p += Stages * StageBytes;
        stg = reinterpret_cast<int32_t*>(p);
        p += StgWords * 4;
        full = reinterpret_cast<uint64_t*>(p);
        p += Stages * 8;
        empty = reinterpret_cast<uint64_t*>(p);
        p += Stages * 8;
        red = reinterpret_cast<unsigned long long*>(p);
        p += kMaxConsumerWarps * MP * 8;
        sx = reinterpret_cast<float*>(p);
        p += MP * 4;
        abort = reinterpret_cast<volatile int*>(p);
        flag = reinterpret_cast<volatile int*>(p + 4);
        xf = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p + 64) + 15) & ~uintptr_t(15));
    }
    __device__ __forceinline__ uint8_t* w_tile(int s) { return stages + s * StageBytes; }
    __device__ __forceinline__ uint8_t* x_tile(int s) { return stages + s * StageBytes + kWTileBytes; }
    // box j of the activation slice: MP rows x 128 bytes, 1024-byte aligned
    __device__ __forceinline__ uint8_t* x_box(int s, int j) { return x_tile(s) + j * MP * BKB; }
};


// ---------------------------------------------------------------------------
// One weight tile (128 channels x 128 bytes of K, 128-byte swizzled) against
// the activation tile (MP tokens x the same 128 bytes, same swizzle), both in
// shared memory: acci += exact int32 partial sums of this warp's channels.
// Chunk pairs P < S8P use the int8 m16n8k32 MMA directly on the ldmatrix
// words; the others widen the codes exactly to binary16 and use the f16
// m16n8k16 MMA, whose fp32 partials (|sum| <= 2^21) are exact integers.
// The f16 products use a fixed permutation of K within each 16-byte chunk
// (logical k 2t,2t+1 <-> bytes 4t,4t+1 and 2t+8,2t+9 <-> bytes 4t+2,4t+3),
// applied identically to both operands, which leaves every sum unchanged.
// ---------------------------------------------------------------------------
template <int BPW>
struct TileLanes {
    uint32_t w_row_off[BPW];   // byte offset of this lane's ldmatrix row, per 16-row block
    uint32_t w_chunk_off[4];   // swizzled chunk offset per chunk pair
    uint32_t x_chunk_off[2];   // swizzled chunk offset per group of four chunks
    uint32_t x_row_off;        // byte offset of this lane's activation row
    __device__ __forceinline__ TileLanes(int first_row, int lane) {
        const int li = lane & 7, lj = lane >> 3;
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk)
            w_row_off[blk] = (uint32_t)((first_row + 16 * blk + li + 8 * (lj & 1)) * BKB);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp)
            w_chunk_off[cp] = (uint32_t)((((2 * cp) + (lj >> 1)) ^ li) << 4);
#pragma unroll
        for (int cq = 0; cq < 2; ++cq) x_chunk_off[cq] = (uint32_t)(((4 * cq + lj) ^ li) << 4);
        x_row_off = (uint32_t)(li * BKB);
    }
};

template <int NG, int BPW, int S8P>
__device__ __forceinline__ void w8a8_tile_mma(uint32_t wb, uint32_t xb, const TileLanes<BPW>& L,
                                              int32_t (&acci)[BPW][NG][4]) {
    float accf[BPW][NG][4];
#pragma unroll
    for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
        for (int gr = 0; gr < NG; ++gr)
#pragma unroll
            for (int e = 0; e < 4; ++e) accf[blk][gr][e] = 0.f;
#pragma unroll
    for (int cq = 0; cq < 2; ++cq) {
        // Activation words (tokens = MMA columns) for chunks 4cq .. 4cq+3.
        uint32_t bw[NG][4];
#pragma unroll
        for (int gr = 0; gr < NG; ++gr)
            ldmatrix_x4(xb + (uint32_t)(8 * gr * BKB) + L.x_row_off + L.x_chunk_off[cq],
                        bw[gr][0], bw[gr][1], bw[gr][2], bw[gr][3]);
        uint32_t bh[NG][4][2];
#pragma unroll
        for (int gr = 0; gr < NG; ++gr)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (2 * cq + c / 2 >= S8P) widen_i8x4_f16(bw[gr][c], bh[gr][c][0], bh[gr][c][1]);
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk) {
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) {
                const int P = 2 * cq + cp;      // chunk pair: chunks 2P, 2P+1
                uint32_t r0, r1, r2, r3;
                ldmatrix_x4(wb + L.w_row_off[blk] + L.w_chunk_off[P], r0, r1, r2, r3);
                if (P < S8P) {
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr)
                        mma_s8_16832(acci[blk][gr], r0, r1, r2, r3, bw[gr][2 * cp], bw[gr][2 * cp + 1]);
                } else {
                    uint32_t a0l, a0h, a1l, a1h;
                    widen_i8x4_f16(r0, a0l, a0h);   // row g,   chunk 2P
                    widen_i8x4_f16(r1, a1l, a1h);   // row g+8, chunk 2P
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr)
                        mma_f16_16816(accf[blk][gr], a0l, a1l, a0h, a1h,
                                      bh[gr][2 * cp][0], bh[gr][2 * cp][1]);
                    widen_i8x4_f16(r2, a0l, a0h);   // row g,   chunk 2P+1
                    widen_i8x4_f16(r3, a1l, a1h);   // row g+8, chunk 2P+1
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr)
                        mma_f16_16816(accf[blk][gr], a0l, a1l, a0h, a1h,
                                      bh[gr][2 * cp + 1][0], bh[gr][2 * cp + 1][1]);
                }
            }
        }
    }
    if (S8P < 4) {
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
            for (int gr = 0; gr < NG; ++gr)
#pragma unroll
                for (int e = 0; e < 4; ++e) acci[blk][gr][e] += __float2int_rn(accf[blk][gr][e]);
    }
}

// ---------------------------------------------------------------------------
// W4A8 tile: 128 channels x 128 bytes of packed int4 codes (256 codes of K per
// channel; byte j holds code 2j in its low nibble and 2j+1 in its high one)
// against the activation tile, two 128-byte swizzled boxes of MP tokens x
// 128 codes. A 32-bit ldmatrix word holds codes 32c + 8t .. 32c + 8t + 7 of
// one row (t = lane % 4); the matching activation codes of each token come
// from one 8-byte load. Chunk pairs P < S8P run on the int8 MMA, the others
// on the f16 MMA:
//  - int8 m16n8k32: masking a high nibble in place gives 16 * code(2j+1)
//    and shifting a low nibble up gives 16 * code(2j), both exact int8
//    operands; the activation bytes are split into even and odd codes to
//    match (K slots carry even codes in the first half, odd codes in the
//    second); the sums are 16 times the true ones and are shifted back
//    exactly after the tile;
//  - f16 m16n8k16: (w & 0x000F000F) ^ 0x64086408 is the f16 pair 1032 + code
//    for the nibbles at bits 0 and 16 (two's complement nibble with bit 3
//    flipped under the exponent of 1024), minus 1032 exactly; the nibbles at
//    bits 4 and 20 give 1024 + 16 (code ^ 8) and one fused multiply-add by
//    1/16 and -72 (exact) gives the code; the word shifted by 8 gives the
//    other two pairs. Activation codes are regrouped into the same pairs and
//    widened exactly to f16. Products are at most 7 * 127 and a tile sums at
//    most 256 of them per output (|sum| < 2^24): every fp32 partial is an
//    exact integer, converted to int32 after the tile.
// On GB300 the int8 MMA runs at a quarter of the f16 rate and the f16 path
// pays for its conversions in issue slots; the two costs add up rather than
// overlap (measured: splitting a tile between them, interleaved or not, and
// independent accumulator chains all land between the two). With one token
// group (up to 8 tokens) the int8 path is faster, with more the f16 path.
// ---------------------------------------------------------------------------
template <int NG>
__host__ __device__ constexpr int w4_s8_pairs() { return NG == 1 ? 4 : 0; }

// f16 pairs (code 8t+s, code 8t+4+s), s = 0..3, of one packed word
__device__ __forceinline__ void int4x8_f16(uint32_t w, uint32_t (&h)[4]) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t v = q ? (w >> 8) : w;
        uint32_t lo = (v & 0x000F000Fu) ^ 0x64086408u;    // 1032 + code
        uint32_t hi = (v & 0x00F000F0u) ^ 0x64806480u;    // 1024 + 16 (code ^ 8)
        asm("sub.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64086408u));
        asm("fma.rn.f16x2 %0, %0, %1, %2;" : "+r"(hi) : "r"(0x2C002C00u), "r"(0xD480D480u));   // * 1/16 - 72
        h[2 * q] = lo;
        h[2 * q + 1] = hi;
    }
}

template <int NG, int BPW, int MP, int CW>
__device__ __forceinline__ void w4a8_tile_mma(uint32_t wb, uint32_t xb, const TileLanes<BPW>& L,
                                              const uint32_t (&x_off)[4], uint32_t xfb, int warp, int lane,
                                              int32_t (&acci)[BPW][NG][4]) {
    constexpr int S8P = w4_s8_pairs<NG>();
    if constexpr (S8P < 4) {
        // The f16 chunks' activation fragments are the same for every warp:
        // warp w widens chunk w once for the CTA into shared memory (two
        // tiles' buffers: a warp can run at most one tile ahead of the
        // others, since each tile's barrier waits for all of them).
        static_assert(CW == 8, "one 32-code chunk per consumer warp");
        if (warp >= 2 * S8P) {
            const int c = warp, g = lane >> 2, t4 = lane & 3;
            const uint32_t off = (uint32_t)((c >> 2) * MP * BKB + g * BKB +
                                            ((((2 * (c & 3)) + (t4 >> 1)) ^ g) << 4) + ((t4 & 1) << 3));
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                uint32_t lo, hi, f0, f1, f2, f3;
                lds_v2_u32(xb + off + (uint32_t)(8 * gr * BKB), lo, hi);
                widen_i8x4_f16(__byte_perm(lo, hi, 0x5140), f0, f1);
                widen_i8x4_f16(__byte_perm(lo, hi, 0x7362), f2, f3);
                sts_v4_u32(xfb + (uint32_t)(((c * NG + gr) * 32 + lane) * 16), f0, f1, f2, f3);
            }
        }
        consumer_sync<CW>();
    }
    float accf[BPW][NG][4];
    int32_t acc16[BPW][NG][4];
#pragma unroll
    for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
        for (int gr = 0; gr < NG; ++gr)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                accf[blk][gr][e] = 0.f;
                acc16[blk][gr][e] = 0;
            }
#pragma unroll
    for (int P = 0; P < 4; ++P) {                 // packed chunks 2P, 2P+1: codes 64P .. 64P+63
        if (P < S8P) {
            uint32_t be[2][NG], bo[2][NG];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = 2 * P + h;
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    uint32_t lo, hi;
                    lds_v2_u32(xb + (uint32_t)((c >> 2) * MP * BKB + 8 * gr * BKB) + x_off[c & 3], lo, hi);
                    be[h][gr] = __byte_perm(lo, hi, 0x6420);   // codes 8t, 8t+2, 8t+4, 8t+6
                    bo[h][gr] = __byte_perm(lo, hi, 0x7531);   // codes 8t+1, 8t+3, 8t+5, 8t+7
                }
            }
#pragma unroll
            for (int blk = 0; blk < BPW; ++blk) {
                uint32_t r0, r1, r2, r3;     // rows g, g+8 of chunk 2P; rows g, g+8 of chunk 2P+1
                ldmatrix_x4(wb + L.w_row_off[blk] + L.w_chunk_off[P], r0, r1, r2, r3);
                const uint32_t e0 = (r0 << 4) & 0xF0F0F0F0u, o0 = r0 & 0xF0F0F0F0u;
                const uint32_t e1 = (r1 << 4) & 0xF0F0F0F0u, o1 = r1 & 0xF0F0F0F0u;
                const uint32_t e2 = (r2 << 4) & 0xF0F0F0F0u, o2 = r2 & 0xF0F0F0F0u;
                const uint32_t e3 = (r3 << 4) & 0xF0F0F0F0u, o3 = r3 & 0xF0F0F0F0u;
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    mma_s8_16832(acc16[blk][gr], e0, e1, o0, o1, be[0][gr], bo[0][gr]);
                    mma_s8_16832(acc16[blk][gr], e2, e3, o2, o3, be[1][gr], bo[1][gr]);
                }
            }
        } else {
            uint32_t bx[2][NG][4];                // f16 pairs (x[8t+s], x[8t+4+s])
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c = 2 * P + h;
#pragma unroll
                for (int gr = 0; gr < NG; ++gr)
                    lds_v4_u32(xfb + (uint32_t)(((c * NG + gr) * 32 + lane) * 16), bx[h][gr][0], bx[h][gr][1],
                               bx[h][gr][2], bx[h][gr][3]);
            }
#pragma unroll
            for (int blk = 0; blk < BPW; ++blk) {
                uint32_t r[4];
                ldmatrix_x4(wb + L.w_row_off[blk] + L.w_chunk_off[P], r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t ag[4], ag8[4];
                    int4x8_f16(r[2 * h], ag);
                    int4x8_f16(r[2 * h + 1], ag8);
#pragma unroll
                    for (int gr = 0; gr < NG; ++gr) {
                        mma_f16_16816(accf[blk][gr], ag[0], ag8[0], ag[1], ag8[1], bx[h][gr][0],
                                      bx[h][gr][1]);
                        mma_f16_16816(accf[blk][gr], ag[2], ag8[2], ag[3], ag8[3], bx[h][gr][2],
                                      bx[h][gr][3]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
        for (int gr = 0; gr < NG; ++gr)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acci[blk][gr][e] += (S8P > 0 ? (acc16[blk][gr][e] >> 4) : 0) +
                                    (S8P < 4 ? __float2int_rn(accf[blk][gr][e]) : 0);
}


// ---------------------------------------------------------------------------
// W8A8 kernel (W4 = 1: the W4A8 kernel, packed int4 weights, same pipeline
// and epilogue)
// ---------------------------------------------------------------------------
template <int NG, int EPI, int W4>
__global__ void __launch_bounds__((kW8A8Warps + 1) * 32, 1)
w8a8_stream_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const W8A8Params p) {
    using C = Cfg<NG, W4 ? 2 : 1>;
    constexpr int MP = C::MP;
    constexpr int Stages = C::Stages;
    constexpr int CW = kW8A8Warps;
    constexpr int RW = BN / CW;          // output channels per consumer warp
    constexpr int BPW = RW / 16;         // 16-channel MMA blocks per warp
    constexpr int S8P = s8_pairs<NG>();
    extern __shared__ uint8_t smem_raw[];
    Smem<Stages, C::StageBytes, C::StgWords, MP> sm(smem_raw);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const long long G = gridDim.x;
    const int a = (int)((long long)blockIdx.x * p.T / G);
    const int b = (int)((long long)(blockIdx.x + 1) * p.T / G);

    if (tid == 0) {
        for (int s = 0; s < Stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], CW);
        }
        *sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    allow_dependent_launch();

    if (warp == CW) {
        if (lane == 0)
            produce<Stages, W4 ? 2 : 1>(&g_stream_gemm_error, sm, &tmap_w, &tmap_x, a, b, p.KT, BKB,
                                        (unsigned)(kWTileBytes + C::XBytes));
        return;
    }

    // ---------------- consumers ----------------
    EpiState est;
    est.c2 = split_contributors_end(p.T, p.KT, b);
    grid_dependency_wait();
    if (tid < MP) sm.sx[tid] = tid < p.M ? p.sx[tid] : 0.f;
    consumer_sync<CW>();

    const int g = lane >> 2, t4 = lane & 3;
    const TileLanes<BPW> L(RW * warp, lane);
    // W4: this lane's 8-byte activation word of each 32-code chunk of a box
    uint32_t x_off[4];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
        x_off[cc] = (uint32_t)(g * BKB + ((((2 * cc) + (t4 >> 1)) ^ g) << 4) + ((t4 & 1) << 3));

    int32_t acci[BPW][NG][4];
    int s = 0, phase = 0;
    int i = a;
    while (i < b) {
        const int nt = i / p.KT;
        const int seg_begin = i;
        const int seg_end = min(b, (nt + 1) * p.KT);
        segment_start<EPI>(est, p, nt, tid);
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
            for (int gr = 0; gr < NG; ++gr)
#pragma unroll
                for (int e = 0; e < 4; ++e) acci[blk][gr][e] = 0;

        for (; i < seg_end; ++i) {
            if (!mbar_wait_bounded(&sm.full[s], phase, sm.abort))
                atomicOr(&g_stream_gemm_error, kErrFullWait);
            if constexpr (W4)
                w4a8_tile_mma<NG, BPW, MP, CW>(smem_u32(sm.w_tile(s)), smem_u32(sm.x_tile(s)), L, x_off,
                                               smem_u32(sm.xf) + (uint32_t)((i & 1) * (C::XfBytes / 2)), warp,
                                               lane, acci);
            else
                w8a8_tile_mma<NG, BPW, S8P>(smem_u32(sm.w_tile(s)), smem_u32(sm.x_tile(s)), L, acci);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            if (++s == Stages) { s = 0; phase ^= 1; }
        }

        // -------- segment end: stage the int32 sums [row][token] --------
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk) {
            const int r0 = RW * warp + 16 * blk + g;
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                const int col = 8 * gr + 2 * t4;
                *reinterpret_cast<int2*>(&sm.stg[r0 * C::SP + col]) = make_int2(acci[blk][gr][0], acci[blk][gr][1]);
                *reinterpret_cast<int2*>(&sm.stg[(r0 + 8) * C::SP + col]) = make_int2(acci[blk][gr][2], acci[blk][gr][3]);
            }
        }
        consumer_sync<CW>();

        segment_end<MP, CW, EPI>(sm, p, nt, seg_begin, seg_end - seg_begin, tid, est, &g_stream_gemm_error);
    }
    range_end<MP, CW, EPI>(sm, p, tid, est);
}

// ---------------------------------------------------------------------------
// BF16 comparator kernel: same pipeline, bf16 operands, fp32 accumulation.
// A tile holds 128 channels x 64 bf16 (128 bytes) of K.
// ---------------------------------------------------------------------------
struct Bf16Params {
    int M, N, K, KT, NT;
    long long T;
    float* y;
    unsigned long long* slots;   // split-K partials (fp32 bits), one slot per CTA
};

template <int NG>
__global__ void __launch_bounds__((kBf16Warps + 1) * 32, 1)
bf16_stream_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const Bf16Params p) {
    using C = Cfg<NG>;
    constexpr int MP = C::MP;
    constexpr int Stages = C::Stages;
    constexpr int CW = kBf16Warps;
    constexpr int RW = BN / CW;
    constexpr int BPW = RW / 16;
    extern __shared__ uint8_t smem_raw[];
    Smem<Stages, C::StageBytes, C::StgWords, MP> sm(smem_raw);
    float* stgf = reinterpret_cast<float*>(sm.stg);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const long long G = gridDim.x;
    const int a = (int)((long long)blockIdx.x * p.T / G);
    const int b = (int)((long long)(blockIdx.x + 1) * p.T / G);

    if (tid == 0) {
        for (int s = 0; s < Stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], CW);
        }
        *sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    allow_dependent_launch();

    if (warp == CW) {
        if (lane == 0)
            produce<Stages>(&g_stream_gemm_error, sm, &tmap_w, &tmap_x, a, b, p.KT, BKB / 2,
                            (unsigned)(kWTileBytes + C::XBytes));
        return;
    }
    const int c2 = split_contributors_end(p.T, p.KT, b);
    grid_dependency_wait();

    const int li = lane & 7, lj = lane >> 3;
    const int g = lane >> 2, t4 = lane & 3;
    uint32_t w_row_off[BPW];
#pragma unroll
    for (int blk = 0; blk < BPW; ++blk)
        w_row_off[blk] = (uint32_t)((RW * warp + 16 * blk + li + 8 * (lj & 1)) * BKB);
    uint32_t w_chunk_off[4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) w_chunk_off[ks] = (uint32_t)((((2 * ks) + (lj >> 1)) ^ li) << 4);
    uint32_t x_chunk_off[2];
#pragma unroll
    for (int cq = 0; cq < 2; ++cq) x_chunk_off[cq] = (uint32_t)(((4 * cq + lj) ^ li) << 4);

    float acc[BPW][NG][4];
    int s = 0, phase = 0;
    int i = a;
    while (i < b) {
        const int nt = i / p.KT;
        const int seg_begin = i;
        const int seg_end = min(b, (nt + 1) * p.KT);
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
            for (int gr = 0; gr < NG; ++gr)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[blk][gr][e] = 0.f;

        for (; i < seg_end; ++i) {
            if (!mbar_wait_bounded(&sm.full[s], phase, sm.abort))
                atomicOr(&g_stream_gemm_error, kErrFullWait);
            const uint32_t wb = smem_u32(sm.w_tile(s));
            const uint32_t xb = smem_u32(sm.x_tile(s));
#pragma unroll
            for (int cq = 0; cq < 2; ++cq) {
                // x chunks 4cq..4cq+3 = k-steps 2cq (chunks 0,1) and 2cq+1 (chunks 2,3)
                uint32_t bx[NG][4];
#pragma unroll
                for (int gr = 0; gr < NG; ++gr)
                    ldmatrix_x4(xb + (uint32_t)((8 * gr + li) * BKB) + x_chunk_off[cq],
                                bx[gr][0], bx[gr][1], bx[gr][2], bx[gr][3]);
#pragma unroll
                for (int blk = 0; blk < BPW; ++blk) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int ks = 2 * cq + h;
                        uint32_t r0, r1, r2, r3;
                        ldmatrix_x4(wb + w_row_off[blk] + w_chunk_off[ks], r0, r1, r2, r3);
#pragma unroll
                        for (int gr = 0; gr < NG; ++gr)
                            mma_bf16_16816(acc[blk][gr], r0, r1, r2, r3, bx[gr][2 * h], bx[gr][2 * h + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            if (++s == Stages) { s = 0; phase ^= 1; }
        }

#pragma unroll
        for (int blk = 0; blk < BPW; ++blk) {
            const int r0 = RW * warp + 16 * blk + g;
#pragma unroll
            for (int gr = 0; gr < NG; ++gr) {
                const int col = 8 * gr + 2 * t4;
                *reinterpret_cast<float2*>(&stgf[r0 * C::SP + col]) = make_float2(acc[blk][gr][0], acc[blk][gr][1]);
                *reinterpret_cast<float2*>(&stgf[(r0 + 8) * C::SP + col]) = make_float2(acc[blk][gr][2], acc[blk][gr][3]);
            }
        }
        consumer_sync<CW>();
        // split tiles combine through per-CTA slots, as in the W8A8 kernels;
        // the head's CTA sums the partials in K order
        if (seg_end - seg_begin != p.KT) {
            if (seg_begin != nt * p.KT) {
                publish_partial<MP, CW>(sm, p.slots, p.M, tid);
                consumer_sync<CW>();
                continue;
            }
            gather_partials<MP, CW, true>(sm, p.slots, p.M, c2, tid, &g_stream_gemm_error);
            consumer_sync<CW>();
        }
        // two threads per channel, as in the W8A8 finish: thread h takes tokens h, h + 2, ...
        constexpr int TH = CW * 32 >= 2 * BN ? 2 : 1;
        const int r = tid & (BN - 1), h = tid / BN;
        const int n = nt * BN + r;
        if (h < TH && n < p.N) {
            for (int m = h; m < p.M; m += TH) p.y[(size_t)m * p.N + n] = stgf[r * C::SP + m];
        }
        consumer_sync<CW>();
    }
}

template <class... Args, class... Params>
cudaError_t launch_ex(void (*kern)(Args...), int grid, int threads, int smem, cudaStream_t s,
                      const Params&... params) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, params...);
}

// ---------------------------------------------------------------------------
// Persistent verify-stack kernel: a sequence of quantize -> W8A8 linear phases
// and (optionally) the LM head with the greedy argmax and the acceptance, in
// one cooperative launch (one CTA per SM, all resident).
//
//  - The producer warp streams the weight tiles of every phase, in phase
//    order, through a 6-stage ring; weights never depend on activations, so
//    it runs ahead across phase boundaries while consumers wait for the
//    previous phase.
//  - Consumers start phase p once every CTA has finished phase p-1 (a grid
//    barrier: an arrival counter in the workspace, read with acquire loads,
//    waited on for at most kWaitLimitNs). They compute the per-token scales of
//    the phase input (every CTA computes the same bits), quantize the
//    128-byte activation chunks their tiles need into shared memory (all
//    loads of a phase issued together), then run the same tile MMA and
//    stream-K epilogue as the single-linear kernel.
//  - The LM head's last finishing tile decodes the argmax keys and the same
//    threads apply the acceptance rule.
// ---------------------------------------------------------------------------
struct StackPhase {
    const void* x;            // [M][K] fp32 or bf16 input of the phase
    const float* act_mul;     // [K] smoothing multipliers or null
    const float* sw;          // [N]
    float* y;                 // [M][N] fp32 output or null (LM head: unused)
    int K, N, KT, NT;
};

struct StackParams {
    CUtensorMap tmap_w[kMaxStackPhases];   // int8 [N rows][K], box {128, 128}, 128B swizzle
    CUtensorMap tmap_x;                    // int8 codes [M rows][kmax], box {128, MP}, 128B swizzle
    StackPhase ph[kMaxStackPhases];
    int n_phases;             // phases in this launch
    int lm_last;              // the last phase is the LM head (argmax + accept)
    int M, x_bf16, kmax;
    int B, gamma;
    const int32_t* draft;
    int32_t* tokens;
    float* max_logit;
    int32_t* accept_len;
    int32_t* out_tokens;
    int32_t* ws_acc;
    unsigned* ws_cnt;
    unsigned long long* keys;
    unsigned* sync;           // [0] B arrivals [1] exits [3] LM tiles done; [32] B flag; [64] A flag;
                              // [96] abort; [128] A arrivals (each group on its own 128-byte line)
    int8_t* xq;               // [M][kmax] int8 codes of the current phase input
};

template <int NG>
struct StackCfg {
    static constexpr int MP = 8 * NG;
    static constexpr int XBytes = MP * BKB;
    static constexpr int XSlot = ((XBytes + 1023) / 1024) * 1024;
    static constexpr int StageBytes = kWTileBytes + XSlot;
    // A deeper ring (12 stages, with a warp prefetching 24 tiles further into
    // L2) made the step slower, 3.81 against 3.09 ms at 5 tokens: CTAs that
    // finish a phase early stream the next one and take bandwidth from the
    // ones the grid barrier waits for. 4 to 7 stages measured alike.
    static constexpr int Stages = 6;
    static constexpr int StgWords = BN * MP;
    static constexpr int SmemBytes = 1024 + Stages * StageBytes + StgWords * 4 + 2 * Stages * 8 +
                                     kMaxConsumerWarps * MP * 8 + 3 * MP * 4 +
                                     kMaxConsumerWarps * MP * 4 + 64;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Device-wide barriers of the stack kernel: B(p) "the phase-p input is
// quantized" and A(p) "every output of phase p is written". Arrivals only
// increment the barrier's own counter; the CTA whose arrival completes it
// publishes p+1 on the barrier's flag, on a cache line of its own, so waiters
// poll a line that changes once per barrier. B and A have separate counters: a
// CTA without tiles in a phase reaches A(p) before others reach B(p).
constexpr int kCountB = 0, kFlagB = 32, kFlagA = 64, kAbort = 96, kCountA = 128;

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Thread 0 of a CTA: arrive on sync[count]; the arrival that makes it reach
// `target` publishes `flag_value` on sync[flag].
__device__ __forceinline__ void grid_arrive(unsigned* sync, int count, unsigned target, int flag,
                                            unsigned flag_value) {
    __threadfence();
    const unsigned prev = atomicAdd(&sync[count], 1u);
    if (prev + 1u == target) {
        __threadfence();
        st_release_gpu(&sync[flag], flag_value);
    }
}

// Thread 0 of the consumers waits until sync[flag] >= value (or the launch was
// aborted); returns false when the wait was cut short.
__device__ __forceinline__ bool grid_wait(unsigned* sync, int flag, unsigned value) {
    if (ld_acquire_gpu(&sync[flag]) >= value) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        __nanosleep(64);
        if (ld_acquire_gpu(&sync[flag]) >= value) return true;
        if (ld_acquire_gpu(&sync[kAbort])) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_stream_gemm_error, kErrGridWait);
            atomicExch(&sync[kAbort], 1u);
            return false;
        }
    }
}

// The 8 bf16 or 4 fp32 elements of one 16-byte vector as binary32 (bf16 widened).
__device__ __forceinline__ void unpack_vec(const uint4& r, bool bf16, float (&e)[8]) {
    if (bf16) {
        const uint32_t w4[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            e[2 * j] = __uint_as_float(w4[j] << 16);
            e[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
        }
    } else {
        e[0] = __uint_as_float(r.x); e[1] = __uint_as_float(r.y);
        e[2] = __uint_as_float(r.z); e[3] = __uint_as_float(r.w);
        e[4] = e[5] = e[6] = e[7] = 0.f;
    }
}

template <int NG>
__global__ void __launch_bounds__((kW8A8Warps + 1) * 32, 1)
verify_stack_kernel(const __grid_constant__ StackParams sp) {
    using C = StackCfg<NG>;
    constexpr int MP = C::MP;
    constexpr int Stages = C::Stages;
    constexpr int CW = kW8A8Warps;
    constexpr int CT = CW * 32;
    constexpr int RW = BN / CW;
    constexpr int BPW = RW / 16;
    constexpr int S8P = s8_pairs<NG>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = base;                                        // Stages x (W tile + X tile)
    int32_t* stg = reinterpret_cast<int32_t*>(ring + Stages * C::StageBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(stg + C::StgWords);
    uint64_t* empty = full + Stages;
    unsigned long long* red = reinterpret_cast<unsigned long long*>(empty + Stages);
    float* s_sx = reinterpret_cast<float*>(red + kMaxConsumerWarps * MP);
    float* s_rx = s_sx + MP;                                     // fl32(1 / sx)
    int32_t* s_tok = reinterpret_cast<int32_t*>(s_rx + MP);
    float* s_amax = reinterpret_cast<float*>(s_tok + MP);        // [warp][MP]
    volatile int* abort = reinterpret_cast<volatile int*>(s_amax + kMaxConsumerWarps * MP);
    volatile int* flag = abort + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x;
    const int P = sp.n_phases;
    const int M = sp.M;
    const bool xbf = sp.x_bf16 != 0;
    const int esz = xbf ? 2 : 4;                                 // input element bytes
    const int E = 16 / esz;                                      // elements per 16-byte vector

    if (tid == 0) {
        for (int st = 0; st < Stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], CW);
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // Grid barriers: every CTA arrives once per phase on B (its share of the
    // phase input is quantized) and once on A (its tiles of the phase are done).
    if (warp == CW) {
        // ---------------- producer ----------------
        // Weight tiles of every phase stream in phase order, ahead of the
        // consumers; a stage's activation tile is requested once the phase's
        // quantized input is complete (B(p) observed), possibly after its
        // weight tile, so weights never wait for activations.
        if (lane != 0) return;
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        prefetch_tensormap(&sp.tmap_x);
        int pend_st[Stages] = {}, pend_ph[Stages] = {}, pend_kt[Stages] = {};   // activation loads not yet issued
        int pend_head = 0, pend_n = 0;
        int ready = -1;                                           // last phase with B(p) complete
        // Polls the barrier counter (one L2 round trip) only while an
        // activation load waits for its phase, then issues what became ready.
        auto refresh = [&]() {
            if (pend_n == 0) return;
            if (pend_ph[pend_head] > ready) {
                const int rp = (int)ld_acquire_gpu(&sp.sync[kFlagB]) - 1;
                if (rp > ready) {
                    ready = rp;
                    fence_proxy_async_global();
                }
            }
            while (pend_n > 0 && pend_ph[pend_head] <= ready) {
                const int s2 = pend_st[pend_head];
                tma_load_2d(ring + s2 * C::StageBytes + kWTileBytes, &sp.tmap_x, pend_kt[pend_head] * BKB, 0,
                            &full[s2], pol_x);
                pend_head = (pend_head + 1) % Stages;
                --pend_n;
            }
        };
        int st = 0, round = 0;
        long long issued = 0;
        bool ok = true;
        for (int p = 0; p < P && ok; ++p) {
            const StackPhase& ph = sp.ph[p];
            const CUtensorMap* tmap = &sp.tmap_w[p];
            prefetch_tensormap(tmap);
            const long long T = (long long)ph.KT * ph.NT;
            const int a = (int)((long long)blockIdx.x * T / G);
            const int b = (int)((long long)(blockIdx.x + 1) * T / G);
            for (int j = a; j < b; ++j) {
                if (issued >= Stages && !mbar_test_wait(&empty[st], (round - 1) & 1)) {
                    // poll without suspending: pending activation loads must go
                    // out as soon as their phase's codes are complete
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_test_wait(&empty[st], (round - 1) & 1)) {
                        refresh();
                        if (*abort || ld_acquire_gpu(&sp.sync[kAbort])) { ok = false; break; }
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            atomicOr(&g_stream_gemm_error, kErrEmptyWait);
                            atomicExch(&sp.sync[kAbort], 1u);
                            *abort = 1;
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                }
                const int nt = j / ph.KT, kt = j - nt * ph.KT;
                mbar_arrive_expect_tx(&full[st], (unsigned)(kWTileBytes + C::XBytes));
                tma_load_2d(ring + st * C::StageBytes, tmap, kt * BKB, nt * BN, &full[st], pol_w);
                if (p <= ready && pend_n == 0) {
                    tma_load_2d(ring + st * C::StageBytes + kWTileBytes, &sp.tmap_x, kt * BKB, 0, &full[st], pol_x);
                } else {
                    const int tail = (pend_head + pend_n) % Stages;
                    pend_st[tail] = st; pend_ph[tail] = p; pend_kt[tail] = kt;
                    ++pend_n;
                    if (pend_n == 1 || (issued & 3) == 0) refresh();
                }
                ++issued;
                if (++st == Stages) { st = 0; ++round; }
            }
        }
        // the last activation loads, then no copy may still be landing at exit
        if (pend_n > 0) {
            const unsigned long long t0 = global_timer_ns();
            while (pend_n > 0) {
                refresh();
                if (pend_n == 0) break;
                if (ld_acquire_gpu(&sp.sync[kAbort]) || global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(&g_stream_gemm_error, kErrDrainWait);
                    break;
                }
                __nanosleep(64);
            }
        }
        const long long first = issued > Stages ? issued - Stages : 0;
        for (long long j = first; j < issued; ++j) {
            const int s2 = (int)(j % Stages), par = (int)((j / Stages) & 1);
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&full[s2], par)) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(&g_stream_gemm_error, kErrDrainWait);
                    return;
                }
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int g = lane >> 2, t4 = lane & 3;
    const TileLanes<BPW> L(RW * warp, lane);
    int st = 0, phase_bit = 0;
    int32_t acci[BPW][NG][4];

    for (int p = 0; p < P; ++p) {
        const StackPhase& ph = sp.ph[p];
        const bool lm = sp.lm_last && p == P - 1;
        const int K = ph.K, KT = ph.KT;
        const long long T = (long long)KT * ph.NT;
        const int a = (int)((long long)blockIdx.x * T / G);
        const int b = (int)((long long)(blockIdx.x + 1) * T / G);
        const uint8_t* xin = static_cast<const uint8_t*>(ph.x);

        // ---- A(p-1): every CTA finished phase p-1 (its outputs may feed this input)
        if (p > 0) {
            if (tid == 0 && !grid_wait(sp.sync, kFlagA, (unsigned)p)) *abort = 1;
            consumer_sync<CW>();
        }

        // ---- per-token scales of the phase input (amax / 127): every CTA
        // computes the same bits; one memory round trip per round of loads
        {
            const int vpr = K / E;                                   // vectors per row
            float part[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m) part[m] = 0.f;
            for (int v0 = 0; v0 < vpr; v0 += CT) {
                const int v = v0 + tid;
                uint4 r[MP];
#pragma unroll
                for (int m = 0; m < MP; ++m)
                    if (m < M && v < vpr)
                        r[m] = __ldg(reinterpret_cast<const uint4*>(xin + ((size_t)m * K + (size_t)v * E) * esz));
                if (v < vpr) {
                    float c[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
                    if (ph.act_mul) {
                        const float4* cm = reinterpret_cast<const float4*>(ph.act_mul + (size_t)v * E);
                        const float4 c0 = __ldg(cm);
                        c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
                        if (xbf) {
                            const float4 c1 = __ldg(cm + 1);
                            c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
                        }
                    }
#pragma unroll
                    for (int m = 0; m < MP; ++m) {
                        if (m >= M) break;
                        float e[8];
                        unpack_vec(r[m], xbf, e);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (j >= E) break;
                            const float xx = ph.act_mul ? __fmul_rn(e[j], c[j]) : e[j];
                            part[m] = fmaxf(part[m], fabsf(xx));
                        }
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MP; ++m) {
                float v = part[m];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                if (lane == 0) s_amax[warp * MP + m] = v;
            }
            consumer_sync<CW>();
            if (tid < MP) {
                float v = 0.f;
                for (int w = 0; w < CW; ++w) v = fmaxf(v, s_amax[w * MP + tid]);
                const float sx = tid < M ? __fdiv_rn(v, 127.0f) : 0.f;
                s_sx[tid] = sx;
                s_rx[tid] = sx != 0.f ? __frcp_rn(sx) : 0.f;
            }
            consumer_sync<CW>();
        }

        // ---- this CTA's share of the codes: (chunk, token) rows round-robin
        // over the CTAs, one row of 128 codes per warp, 4 per lane
        {
            const int items = KT * M;
            for (int it = blockIdx.x + G * warp; it < items; it += G * CW) {
                const int kt = it / M, m = it - (it / M) * M;
                const int k0 = kt * BKB + 4 * lane;
                if (k0 < K) {
                    float v[4];
                    if (xbf) {
                        const uint2 r = __ldg(reinterpret_cast<const uint2*>(xin + ((size_t)m * K + k0) * 2));
                        v[0] = __uint_as_float(r.x << 16); v[1] = __uint_as_float(r.x & 0xFFFF0000u);
                        v[2] = __uint_as_float(r.y << 16); v[3] = __uint_as_float(r.y & 0xFFFF0000u);
                    } else {
                        const uint4 r = __ldg(reinterpret_cast<const uint4*>(xin + ((size_t)m * K + k0) * 4));
                        v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y);
                        v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
                    }
                    float c[4] = {1.f, 1.f, 1.f, 1.f};
                    if (ph.act_mul) {
                        const float4 c0 = __ldg(reinterpret_cast<const float4*>(ph.act_mul + k0));
                        c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
                    }
                    const float sxm = s_sx[m], rxm = s_rx[m];
                    uint32_t word = 0;
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float xx = ph.act_mul ? __fmul_rn(v[jj], c[jj]) : v[jj];
                        word |= (uint32_t)(uint8_t)(int8_t)quant_code(xx, sxm, rxm) << (8 * jj);
                    }
                    *reinterpret_cast<uint32_t*>(sp.xq + (size_t)m * sp.kmax + k0) = word;
                }
            }
            // B(p): the codes are visible to the other CTAs' TMA loads
            fence_proxy_async_global();
            consumer_sync<CW>();
            if (tid == 0) grid_arrive(sp.sync, kCountB, (unsigned)((p + 1) * G), kFlagB, (unsigned)(p + 1));
        }

        // ---- this CTA's tiles
        int seg_begin = a;
#pragma unroll
        for (int blk = 0; blk < BPW; ++blk)
#pragma unroll
            for (int gr = 0; gr < NG; ++gr)
#pragma unroll
                for (int e = 0; e < 4; ++e) acci[blk][gr][e] = 0;

        for (int i = a; i < b; ++i) {
            const int nt = i / KT;
            const int kt = i - nt * KT;
            if (!mbar_wait_bounded(&full[st], phase_bit, abort))
                atomicOr(&g_stream_gemm_error, kErrFullWait);
            uint8_t* stage = ring + st * C::StageBytes;
            w8a8_tile_mma<NG, BPW, S8P>(smem_u32(stage), smem_u32(stage + kWTileBytes), L, acci);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (++st == Stages) { st = 0; phase_bit ^= 1; }

            if (kt != KT - 1 && i != b - 1) continue;
            // -------- segment end: stage [row][token] sums, combine, epilogue
#pragma unroll
            for (int blk = 0; blk < BPW; ++blk) {
                const int r0 = RW * warp + 16 * blk + g;
#pragma unroll
                for (int gr = 0; gr < NG; ++gr) {
                    const int col = 8 * gr + 2 * t4;
                    *reinterpret_cast<int2*>(&stg[r0 * MP + col]) = make_int2(acci[blk][gr][0], acci[blk][gr][1]);
                    *reinterpret_cast<int2*>(&stg[(r0 + 8) * MP + col]) = make_int2(acci[blk][gr][2], acci[blk][gr][3]);
                    acci[blk][gr][0] = acci[blk][gr][1] = acci[blk][gr][2] = acci[blk][gr][3] = 0;
                }
            }
            consumer_sync<CW>();
            const int seg_len = i + 1 - seg_begin;
            seg_begin = i + 1;
            const bool whole = seg_len == KT;
            int32_t* gacc = sp.ws_acc + (size_t)nt * BN * MP;
            if (!whole) {
                for (int e = tid; e < BN * MP; e += CT) {
                    const int r = e / MP, m = e - (e / MP) * MP;
                    if (m < M && nt * BN + r < ph.N) atomicAdd(&gacc[e], stg[e]);
                }
                // one gpu-scope fence by the publishing thread after the CTA
                // barrier orders every thread's adds before the count (the
                // pattern of a grid-wide barrier); its acquire side likewise
                consumer_sync<CW>();
                if (tid == 0) {
                    __threadfence();
                    const unsigned prev = atomicAdd(&sp.ws_cnt[nt], (unsigned)seg_len);
                    const bool last = prev + (unsigned)seg_len == (unsigned)KT;
                    if (last) __threadfence();
                    *flag = last ? 1 : 0;
                }
                consumer_sync<CW>();
            }
            if (whole || *flag) {
                const int r = tid;
                const int n = nt * BN + r;
                const bool valid = r < BN && n < ph.N;
                const float swn = valid ? ph.sw[n] : 0.f;
                // the finished tile's sums: from staging, or read from the
                // workspace in one batch and cleared (no other CTA touches it now)
                int32_t accs[MP];
#pragma unroll
                for (int m = 0; m < MP; ++m) accs[m] = 0;
                if (valid) {
                    if (whole) {
#pragma unroll
                        for (int m = 0; m < MP; ++m) accs[m] = stg[r * MP + m];
                    } else {
#pragma unroll
                        for (int m = 0; m < MP; ++m) accs[m] = m < M ? __ldcg(&gacc[r * MP + m]) : 0;
#pragma unroll
                        for (int m = 0; m < MP; ++m)
                            if (m < M) __stcg(&gacc[r * MP + m], 0);
                    }
                }
                if (!lm) {
                    if (valid && ph.y) {
#pragma unroll
                        for (int m = 0; m < MP; ++m) {
                            if (m >= M) break;
                            ph.y[(size_t)m * ph.N + n] = __fmul_rn(__int2float_rn(accs[m]), __fmul_rn(s_sx[m], swn));
                        }
                    }
                } else {
                    if (r < BN) {
#pragma unroll
                        for (int m = 0; m < MP; ++m) {
                            if (m >= M) break;
                            unsigned long long key = 0ull;
                            if (valid) {
                                const float yv = __fmul_rn(__int2float_rn(accs[m]), __fmul_rn(s_sx[m], swn));
                                key = ((unsigned long long)ordered_bits(yv) << 32) |
                                      (unsigned long long)(0xFFFFFFFFu - (unsigned)n);
                            }
                            key = warp_max_u64(key);
                            if (lane == 0) red[warp * MP + m] = key;
                        }
                    }
                    consumer_sync<CW>();
                    if (tid < M) {
                        unsigned long long k = red[tid];
#pragma unroll
                        for (int w = 1; w < BN / 32; ++w) {
                            const unsigned long long o = red[w * MP + tid];
                            k = o > k ? o : k;
                        }
                        atomicMax(&sp.keys[tid], k);
                    }
                    consumer_sync<CW>();
                    if (tid == 0) {
                        __threadfence();
                        const unsigned prev = atomicAdd(&sp.sync[3], 1u);
                        const bool last = prev + 1u == (unsigned)ph.NT;
                        if (last) __threadfence();
                        *flag = last ? 2 : 0;
                    }
                    consumer_sync<CW>();
                    if (*flag == 2) {
                        // last LM tile: decode the argmax, then accept
                        if (tid < M) {
                            const unsigned long long k = atomicExch(&sp.keys[tid], 0ull);
                            const int32_t t = (int32_t)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull));
                            s_tok[tid] = t;
                            sp.tokens[tid] = t;
                            if (sp.max_logit) sp.max_logit[tid] = unordered_bits((unsigned)(k >> 32));
                        }
                        if (tid == 0) atomicExch(&sp.sync[3], 0u);
                        consumer_sync<CW>();
                        if (sp.accept_len) {
                            const int Gm = sp.gamma + 1;
                            for (int bq = tid; bq < sp.B; bq += CT) {
                                const int32_t* tb = s_tok + bq * Gm;
                                const int32_t* db = sp.draft + (size_t)bq * sp.gamma;
                                int k = 0;
                                while (k < sp.gamma && db[k] == tb[k]) ++k;
                                sp.accept_len[bq] = k + 1;
                                for (int jq = 0; jq < Gm; ++jq)
                                    sp.out_tokens[(size_t)bq * Gm + jq] = jq <= k ? tb[jq] : -1;
                            }
                        }
                    }
                }
                if (!whole && tid == 0) atomicExch(&sp.ws_cnt[nt], 0u);
            }
            consumer_sync<CW>();
        }
        // ---- A(p): this CTA is done with phase p
        consumer_sync<CW>();
        if (tid == 0) grid_arrive(sp.sync, kCountA, (unsigned)((p + 1) * G), kFlagA, (unsigned)(p + 1));
    }
    // last CTA out resets the barrier words for the next launch
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&sp.sync[1], 1u);
        if (prev + 1u == (unsigned)G) {
            atomicExch(&sp.sync[kCountB], 0u);
            atomicExch(&sp.sync[kCountA], 0u);
            atomicExch(&sp.sync[kAbort], 0u);
            atomicExch(&sp.sync[kFlagB], 0u);
            atomicExch(&sp.sync[kFlagA], 0u);
            __threadfence();
            atomicExch(&sp.sync[1], 0u);
        }
    }
}

}  // namespace

WsLayout ws_layout(int mp, int n, bool lm_head, bool stack) {
    WsLayout L;
    const int nt = ceil_div(n, BN);
    auto al16 = [](size_t v) { return (v + 15) & ~size_t(15); };
    size_t off = 0;
    L.slots = off;
    if (!stack) off = al16(off + (size_t)kMaxStreamCtas * BN * mp * 8);
    L.acc = off;
    if (stack) off = al16(off + (size_t)nt * BN * mp * 4);
    L.counters = off;
    if (stack) off = al16(off + (size_t)nt * 4);
    L.keys = off;
    if (lm_head) off = al16(off + (size_t)mp * 8);
    L.done = off;
    if (lm_head) off = al16(off + 5 * 128);   // counters and flags on separate 128-byte lines
    L.total = off;
    return L;
}

cudaError_t launch_w8a8_stream(const W8A8Launch& a, int num_sms, cudaStream_t s) {
    const bool lm = a.epi == Epi::LmHead;
    WsLayout L = ws_layout(a.MP, a.N, lm);
    W8A8Params p;
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.KT = ceil_div(a.w4 ? a.K / 2 : a.K, BKB);   // weight bytes of K per tile row
    p.NT = ceil_div(a.N, BN);
    p.T = (long long)p.KT * p.NT;
    p.sx = a.sx; p.sw = a.sw; p.y = a.y; p.y_bf16 = a.y_bf16; p.acc_debug = a.acc_debug;
    p.tokens = a.tokens; p.max_logit = a.max_logit;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    p.slots = reinterpret_cast<unsigned long long*>(ws + L.slots);
    p.keys = reinterpret_cast<unsigned long long*>(ws + L.keys);
    p.done = reinterpret_cast<unsigned*>(ws + L.done);
    p.slot_wait_ns = debug_slot_wait_ns();
    p.drop_partials = debug_take_drop_partials() ? 1 : 0;
    const int grid = stream_grid(p.T, num_sms);
#define QV_W8A8_LAUNCH(NGV, EPIV, W4V)                                                       \
    launch_ex(w8a8_stream_kernel<NGV, (int)EPIV, W4V>, grid, (kW8A8Warps + 1) * 32,          \
              Cfg<NGV, W4V ? 2 : 1>::SmemBytes, s, a.tmap_w, a.tmap_x, p)
#define QV_W8A8_EPI(NGV, W4V)                                                                \
        (lm ? QV_W8A8_LAUNCH(NGV, Epi::LmHead, W4V)                                          \
            : a.epi == Epi::SwiGLU ? QV_W8A8_LAUNCH(NGV, Epi::SwiGLU, W4V)                   \
                                   : QV_W8A8_LAUNCH(NGV, Epi::Linear, W4V))
#define QV_W8A8_CASE(NGV)                                                                    \
    case NGV:                                                                                \
        return a.w4 ? QV_W8A8_EPI(NGV, 1) : QV_W8A8_EPI(NGV, 0);
    switch (a.MP / 8) {   // W8A8 up to 16 tokens (more go to the tcgen05 kernel), W4A8 up to 32
        QV_W8A8_CASE(1)
        QV_W8A8_CASE(2)
        QV_W8A8_CASE(4)
        default: return cudaErrorInvalidValue;
    }
#undef QV_W8A8_CASE
#undef QV_W8A8_EPI
#undef QV_W8A8_LAUNCH
}

cudaError_t launch_bf16_stream(const Bf16Launch& a, int num_sms, cudaStream_t s) {
    const int NG = a.MP / 8;
    WsLayout L = ws_layout(a.MP, a.N, false);
    Bf16Params p;
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.KT = ceil_div(a.K, BKB / 2);
    p.NT = ceil_div(a.N, BN);
    p.T = (long long)p.KT * p.NT;
    p.y = a.y;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    p.slots = reinterpret_cast<unsigned long long*>(ws + L.slots);
    const int grid = stream_grid(p.T, num_sms);
#define QV_BF16_CASE(NGV) \
    case NGV: return launch_ex(bf16_stream_kernel<NGV>, grid, (kBf16Warps + 1) * 32, Cfg<NGV>::SmemBytes, s, a.tmap_w, a.tmap_x, p);
    switch (NG) {
        QV_BF16_CASE(1)
        QV_BF16_CASE(2)
        QV_BF16_CASE(4)
        QV_BF16_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef QV_BF16_CASE
}

cudaError_t launch_verify_stack(const StackLaunch& a, int num_sms, cudaStream_t s) {
    if (a.n_phases < 1 || a.n_phases > kMaxStackPhases) return cudaErrorInvalidValue;
    static thread_local StackParams sp;     // ~27 KB: kept off the stack
    memset(&sp, 0, sizeof sp);
    for (int i = 0; i < a.n_phases; ++i) {
        const StackLaunchPhase& h = a.phases[i];
        StackPhase& d = sp.ph[i];
        sp.tmap_w[i] = h.tmap_w;
        d.x = h.x; d.act_mul = h.act_mul; d.sw = h.sw; d.y = h.y;
        d.K = h.K; d.N = h.N;
        d.KT = ceil_div(h.K, BKB);
        d.NT = ceil_div(h.N, BN);
    }
    sp.n_phases = a.n_phases;
    sp.lm_last = a.lm_last ? 1 : 0;
    sp.M = a.M; sp.x_bf16 = a.x_bf16 ? 1 : 0;
    sp.B = a.B; sp.gamma = a.gamma; sp.draft = a.draft;
    sp.tokens = a.tokens; sp.max_logit = a.max_logit;
    sp.accept_len = a.accept_len; sp.out_tokens = a.out_tokens;
    WsLayout L = ws_layout(a.MP, a.n_max, true, true);
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    sp.ws_acc = reinterpret_cast<int32_t*>(ws + L.acc);
    sp.ws_cnt = reinterpret_cast<unsigned*>(ws + L.counters);
    sp.keys = reinterpret_cast<unsigned long long*>(ws + L.keys);
    sp.sync = reinterpret_cast<unsigned*>(ws + L.done);
    sp.xq = reinterpret_cast<int8_t*>(ws + stack_xq_offset(a.MP, a.n_max));
    sp.kmax = a.kmax;
    sp.tmap_x = a.tmap_x;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3((kW8A8Warps + 1) * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (a.MP == 8) {
        cfg.dynamicSmemBytes = StackCfg<1>::SmemBytes;
        e = cudaFuncSetAttribute(verify_stack_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 StackCfg<1>::SmemBytes);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, verify_stack_kernel<1>, sp);
    }
    if (a.MP == 16) {
        cfg.dynamicSmemBytes = StackCfg<2>::SmemBytes;
        e = cudaFuncSetAttribute(verify_stack_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 StackCfg<2>::SmemBytes);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, verify_stack_kernel<2>, sp);
    }
    return cudaErrorInvalidValue;
}

size_t stack_xq_offset(int mp, int n_max) {
    return (ws_layout(mp, n_max, true, true).total + 255) & ~size_t(255);
}

size_t stack_ws_bytes(int mp, int M, int n_max, int kmax) {
    return stack_xq_offset(mp, n_max) + (((size_t)M * kmax + 15) & ~size_t(15));
}

cudaError_t read_and_clear_stream_gemm_error(unsigned* code) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_stream_gemm_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_stream_gemm_error, &zero, sizeof(unsigned));
}

}  // namespace qv
