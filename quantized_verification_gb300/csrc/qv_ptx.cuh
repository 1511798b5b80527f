// qv_ptx.cuh -- inline-PTX building blocks for the sm_103a kernels of libqv:
// mbarriers with bounded waits, 2-D TMA loads, ldmatrix, f16 mma.sync, the
// tcgen05 tensor-memory and MMA instructions, programmatic-dependent-launch
// controls and the exact int8 -> f16 widening.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "qv_internal.h"

namespace qv {


// Device error word bits.
constexpr unsigned kErrFullWait = 1u;    // consumer waited too long for a stage
constexpr unsigned kErrEmptyWait = 2u;   // producer waited too long for a slot
constexpr unsigned kErrDrainWait = 4u;   // copies still in flight at exit
constexpr unsigned kErrGridWait = 8u;    // a CTA waited too long at a grid barrier
constexpr unsigned kErrTcWait = 16u;     // tensor-core pipeline wait (operands / MMA completion)
constexpr unsigned kErrSlotWait = 32u;   // split-K head waited too long for a partial sum

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the TMA unit and the other threads.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy global writes before later async-proxy
// (TMA) accesses, and the reverse.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking probe of the phase with the given parity (never suspends).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, unsigned parity) {
    unsigned ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// kWaitLimitNs. Returns false (without waiting) once *abort is set, and sets
// *abort itself when the limit runs out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                                  volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = global_timer_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}

// mbar_wait_bounded for a single thread that shares its SM sub-partition with
// compute warps (a producer or an MMA issuer): between probes it sleeps for
// about sleep_ns, so that its polling does not take their issue slots.
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint64_t* bar, unsigned parity,
                                                        volatile int* abort, unsigned sleep_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    unsigned long long t0 = global_timer_ns();
    while (true) {
        __nanosleep(sleep_ns);
        if (mbar_test_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];"
                 :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled load of the box at (x = inner coordinate, y = row) into shared
// memory; completion is signalled on `bar` as transaction bytes. The caller
// guarantees x * element size is a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map,
                                            int x, int y, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)),
           "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Prefetch the box at (x, y) of a 2-D tensor map into L2 (no shared memory,
// no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}

// ---------------------------------------------------------------- PDL
// Wait until every kernel this grid depends on has completed and its memory
// operations are visible (no-op when launched without a programmatic edge).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel on the stream to begin launching.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- warp MMA
// Two consecutive 32-bit words of shared memory (8-byte aligned address).
__device__ __forceinline__ void lds_v2_u32(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// Four consecutive 32-bit words of shared memory (16-byte aligned address).
__device__ __forceinline__ void lds_v4_u32(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                           uint32_t& r3) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void sts_v4_u32(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" :: "r"(addr), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A(16x16, f16) * B(16x8, f16), fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A(16x16, bf16) * B(16x8, bf16), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A(16x32, s8) * B(32x8, s8), exact int32 accumulate.
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Exact widening of four int8 codes (one 32-bit word, element 0 in the low
// byte) to four binary16 values, returned as two f16x2 words {e0, e1} and
// {e2, e3}. Derivation from the binary16 format: flipping the sign bit of a
// two's-complement byte b gives u = b + 128 in [0, 255]; the binary16 pattern
// 0x6400 | u has exponent 10 and encodes 1024 + u exactly; subtracting
// 1152 = 1024 + 128 (pattern 0x6480) leaves b, which is exact because b is a
// small integer.
__device__ __forceinline__ void widen_i8x4_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x4140);
    hi = __byte_perm(u, 0x64646464u, 0x4342);
    asm("sub.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
    asm("sub.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// ---------------------------------------------------------------- quantization
// q = clamp(rne(fl32(x / s)), -127, 127) (0 when s == 0), decided from t = fl32(x * r)
// with r = fl32(1 / s) when t is far from every half-integer, else from the
// IEEE quotient. Error bound: r = (1/s)(1+d1), t = (x/s)(1+d1)(1+d2) and
// fl32(x/s) = (x/s)(1+d3) with |di| <= 2^-24, so |t - fl32(x/s)| < 2^-22 |t|.
// If the distance from t to the nearest half-integer exceeds 2^-20 |t|, both
// lie strictly on the same side of it and round to the same integer.
// The IEEE-quotient decision, kept out of line so that the compiler branches
// to it (rarely) instead of evaluating the division for every element.
static __device__ __noinline__ int quant_code_div(float x, float s) {
    const int qi = __float2int_rn(rintf(__fdiv_rn(x, s)));
    return qi > 127 ? 127 : (qi < -127 ? -127 : qi);
}
// The fast rule alone, for callers that batch the rare exact decisions: t is
// rounded half-even by adding and removing 1.5 * 2^23 (exact for |t| < 2^22;
// here |t| <= 127 (1 + 2^-22) unless s is subnormal, when r and t overflow and
// `near` is set), the code is read from the sum's low bits and clamped, and
// `near` is set when t lies within 2^-20 |t| of a half-integer (or is not
// finite): the caller must then take quant_code_exact(x, s) instead.
__device__ __forceinline__ int quant_code_fast(float x, float r, bool& near) {
    const float t = __fmul_rn(x, r);
    const float y = __fadd_rn(t, 12582912.0f);
    const float n = __fsub_rn(y, 12582912.0f);
    const float margin = __fsub_rn(0.5f, fabsf(__fsub_rn(t, n)));
    near = !(margin > __fmul_rn(fabsf(t), 0x1p-20f));
    const int qi = __float_as_int(y) - 0x4B400000;
    return qi > 127 ? 127 : (qi < -127 ? -127 : qi);
}
// The IEEE-quotient decision, inline (callers branch to it rarely).
__device__ __forceinline__ int quant_code_exact(float x, float s) {
    const int qi = __float2int_rn(rintf(__fdiv_rn(x, s)));
    return qi > 127 ? 127 : (qi < -127 ? -127 : qi);
}

__device__ __forceinline__ int quant_code(float x, float s, float r) {
    if (s == 0.f) return 0;
    const float t = __fmul_rn(x, r);
    const float q = rintf(t);
    const float margin = __fsub_rn(0.5f, fabsf(__fsub_rn(t, q)));
    if (!(margin > __fmul_rn(fabsf(t), 0x1p-20f))) return quant_code_div(x, s);
    const int qi = __float2int_rn(q);
    return qi > 127 ? 127 : (qi < -127 ? -127 : qi);
}

// ---------------------------------------------------------------- SiLU
// The decoder layer's SiLU, shared by the SwiGLU steps (the fused
// quantization kernel and the gate|up GEMM epilogue).
// exp(x): x > 88 -> +inf, x < -87 -> 0; otherwise k = rne(fl(x * log2 e)),
// r = fl(fl(x - fl(k * LN2_HI)) - fl(k * LN2_LO)), p = the degree-7 Taylor
// polynomial of e^r by Horner (coefficients fl(1/n!)), E = fl(p * 2^k).
// LN2_HI has 16 significant bits, so k * LN2_HI is exact for |k| <= 127.
__device__ __forceinline__ float layer_exp(float x) {
    if (x > 88.0f) return __uint_as_float(0x7F800000u);
    if (x < -87.0f) return 0.0f;
    const float k = rintf(__fmul_rn(x, 1.44269504088896341f));
    float r = __fsub_rn(x, __fmul_rn(k, 0.693145751953125f));
    r = __fsub_rn(r, __fmul_rn(k, 1.42860682030941723212e-6f));
    float p = 1.0f / 5040.0f;
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
    p = __fadd_rn(__fmul_rn(p, r), 0.5f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    p = __fadd_rn(__fmul_rn(p, r), 1.0f);
    const float two_k = __uint_as_float((uint32_t)((int)k + 127) << 23);
    return __fmul_rn(p, two_k);
}

__device__ __forceinline__ float silu(float v) {
    const float den = __fadd_rn(1.0f, layer_exp(-v));
    return __fmul_rn(v, __fdiv_rn(1.0f, den));
}

// ---------------------------------------------------------------- tcgen05
// Tensor memory (TMEM): 128 lanes x 512 columns of 32-bit cells per SM. An
// address is (lane << 16) | column; a warp reaches only the 32 lanes
// 32 * (warp id % 4) .. +31.

// Allocate `ncols` columns (a power of two >= 32); the whole warp executes it
// and the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
// Order tcgen05 operations before / after a thread synchronisation.
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's generic shared-memory writes visible to the async proxy
// (the tensor core reading an operand from shared memory).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand stored as rows of 128
// bytes with the 128-byte swizzle (16-byte chunk c of row r at position
// c ^ (r % 8)), 8-row groups 1024 bytes apart; `saddr` is the group-aligned
// start plus the byte offset of the K step inside the 128-byte row.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);      // start address / 16
    d |= (uint64_t)1u << 16;                      // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;            // stride byte offset: 8 rows x 128 bytes
    d |= (uint64_t)1u << 46;                      // descriptor version for tcgen05
    d |= (uint64_t)2u << 61;                      // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with f16 A and B (both K-major) and an
// f32 accumulator, for an M x N tile.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, one K = 16 step, issued by one thread.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// Store 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                    "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
                    "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
                    "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
                    "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Load NC consecutive columns of this thread's lane (NC = 8, 16 or 32).
template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[NC]);
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr) : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                 "%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(taddr) : "memory");
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                 "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
                 "%30,%31}, [%32];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                   "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
                   "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
                   "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
                   "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
                   "=r"(v[30]), "=r"(v[31])
                 : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

}  // namespace qv
