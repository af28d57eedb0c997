// common.cuh -- sm_103a building blocks shared by the fp8kv kernels:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (TMEM allocation,
// FP8 MMAs, TMEM loads/stores), shared-memory and instruction descriptors,
// and host helpers (status checks, tensor maps, the device error word).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "../../include/fp8kv.h"

namespace fp8kv {

// ---------------------------------------------------------------------------
// Constants
// ---------------------------------------------------------------------------
constexpr float kE4M3Max = 448.0f;           // largest finite e4m3 value
constexpr int kTile = 128;                    // keys per KV tile (= MMA M/N)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded-wait limit: 2 s

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two fp32 -> packed e4m3x2 (lo byte = a, hi byte = b), round to nearest
// even, saturating to +-448 (NaN stays NaN).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
    float2 f = make_float2(a, b);
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3));
}

// A per-tensor scale as the kernels use it.  x / s is the IEEE fp32 quotient;
// when s is a power of two (1.0 included) x * (1 / s) is the same real
// number rounded the same way (1 / s is exact and both operations round
// once to nearest), so the kernels multiply instead of dividing.
struct QScale {
    float scale;
    float inv;       // 1 / scale, used when pow2 != 0
    uint32_t pow2;
};

inline QScale make_qscale(float s) {
    int e = 0;
    const float m = frexpf(s, &e);
    const float inv = 1.0f / s;
    QScale q;
    q.scale = s;
    q.inv = inv;
    q.pow2 = (m == 0.5f && isnormal(inv) && isnormal(s)) ? 1u : 0u;
    return q;
}

__device__ __forceinline__ float scale_div(float x, const QScale &q) {
    return q.pow2 ? x * q.inv : __fdiv_rn(x, q.scale);
}

// Convert two quotients x / s to nearest-even e4m3 with saturation (the
// satfinite conversion maps +-Inf and every magnitude beyond 448 to +-448 and
// NaN to NaN, which is the clamp to +-448 that keeps NaN) and set the sign
// bits `sign_a` / `sign_b` of the inputs, so that -NaN and -0 keep their sign
// (the division returns the canonical positive NaN).  Returns lo byte = a,
// hi byte = b.
__device__ __forceinline__ uint32_t pack_quotients(float a, float b, uint32_t sign_a,
                                                   uint32_t sign_b) {
    return static_cast<uint32_t>(f32x2_to_e4m3x2(a, b)) | (sign_a << 7) | (sign_b << 15);
}

// Quantize two fp32 values (already in the value domain) by a per-tensor
// scale: IEEE fp32 division (an exact multiply for a power-of-two scale),
// then pack_quotients.
__device__ __forceinline__ uint32_t quantize_pair(float a, float b, const QScale &scale,
                                                  uint32_t sign_a, uint32_t sign_b) {
    return pack_quotients(scale_div(a, scale), scale_div(b, scale), sign_a, sign_b);
}

// Quantize the two bf16 elements packed in `word` (element 0 in the low half).
__device__ __forceinline__ uint32_t quantize_bf16x2(uint32_t word, const QScale &scale) {
    return quantize_pair(__uint_as_float(word << 16), __uint_as_float(word & 0xFFFF0000u), scale,
                         (word >> 15) & 1u, word >> 31);
}

// quantize_bf16x2 with the scale's form fixed at compile time (kPow2: the
// scale is a power of two and scale.inv its exact reciprocal), for loops
// where the compiler would otherwise evaluate both the multiply and the
// division for every element.
// Query quantization inside the attention kernels: the same quotient and
// conversion without the NaN sign fix-up.  Q8 is never stored, and a NaN
// query gives NaN scores whichever NaN code it gets, so -NaN need not stay
// 0xFF here (-0 keeps its sign through the multiply or divide).
template <bool kPow2>
__device__ __forceinline__ uint32_t quantize_q_bf16x2(uint32_t word, const QScale &scale) {
    const float2 v = make_float2(__uint_as_float(word << 16), __uint_as_float(word & 0xFFFF0000u));
    const float2 q = kPow2 ? __fmul2_rn(v, make_float2(scale.inv, scale.inv))
                           : make_float2(__fdiv_rn(v.x, scale.scale), __fdiv_rn(v.y, scale.scale));
    return static_cast<uint32_t>(f32x2_to_e4m3x2(q.x, q.y));
}

template <bool kPow2>
__device__ __forceinline__ uint32_t quantize_bf16x2_as(uint32_t word, const QScale &scale) {
    const float a = __uint_as_float(word << 16), b = __uint_as_float(word & 0xFFFF0000u);
    const float qa = kPow2 ? a * scale.inv : __fdiv_rn(a, scale.scale);
    const float qb = kPow2 ? b * scale.inv : __fdiv_rn(b, scale.scale);
    return pack_quotients(qa, qb, (word >> 15) & 1u, word >> 31);
}

// max(a, b, c) in one instruction (sm_100 and later); a NaN operand is
// ignored like fmaxf does.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// packed e4m3x2 -> two halves (exact: every e4m3 value is an fp16 value).
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint16_t v) {
    __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
    return *reinterpret_cast<__half2 *>(&r);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase has not completed
// sleeps until it completes or `hint_ns` elapses, instead of spinning on the
// issue slots that the other warps of its scheduler need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t addr, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Longest sleep of one try_wait in a bounded wait: the abort flag and the
// time limit are checked after each.
constexpr uint32_t kWaitSleepNs = 100000;   // 0.1 ms

// Shared state of one CTA's failure handling: the first wait that runs out
// sets `abort`; every later wait in the CTA then gives up at once, so all
// roles reach the teardown without waiting out the limit again.
struct CtaFail {
    volatile uint32_t abort;
};

// Bounded wait for the phase with the given parity.  Returns false (and
// records FP8KV_DEVERR_WAIT_TIMEOUT) when the limit ran out or another role
// of the CTA gave up already.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, CtaFail *fail,
                                          uint32_t *err_word) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(addr, parity, kWaitSleepNs)) return true;
        if (fail->abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            fail->abort = 1;
            atomicOr(err_word, FP8KV_DEVERR_WAIT_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Proxy fences
// ---------------------------------------------------------------------------
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy for data read exactly once (streamed KV).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 4-D tiled load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 3-D tiled load into shared memory, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and MMA
// ---------------------------------------------------------------------------
// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the base
// address is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Whole warp: give up the CTA's right to allocate TMEM without allocating
// (a CTA that returns before its allocation).
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far has
// completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], e4m3 x e4m3 -> fp32.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], e4m3 x e4m3 -> fp32, with A read from
// tensor memory: row i of A in lane i, each 32-bit column holding four
// consecutive K elements (lowest byte first); one MMA of K = 32 reads eight
// columns from a_tmem.
__device__ __forceinline__ void mma_e4m3_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor, kind::f8f6f4: A and B e4m3, D fp32, M x N tile.
// a_mn / b_mn select the MN-major ("transposed") operand layout.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                   // D format: f32
           | (0u << 7) | (0u << 10)                    // A, B format: e4m3
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle.  Operand tiles are
// stored in "atoms" of 8 rows x 128 bytes (1024 bytes, 1024-aligned), the
// 16-byte chunk c of row r sitting at chunk position c ^ (r % 8).
//   K-major:  rows are M/N indices, 128 bytes of K per row; sbo = bytes
//             between 8-row groups (1024 when dense); lbo unused.
//   MN-major: rows are K indices, 128 bytes of M/N per row; sbo = bytes
//             between 8-row groups along K; lbo = bytes between 128-byte
//             column blocks along M/N.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;   // descriptor version for tcgen05
    d |= 2ull << 61;   // 128-byte swizzle
    return d;
}

// Byte offset of (row, byte) inside a 128-byte-swizzled tile whose rows are
// 128 bytes long (row r, 16-byte chunk c -> chunk c ^ (r & 7)).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t byte) {
    return row * 128u + ((((byte >> 4) ^ (row & 7u)) << 4) | (byte & 15u));
}

// --- TMEM loads / stores (32 lanes x 32 bits shape: thread i of warp w reads
//     TMEM lane 32*(w%4)+i, one column per register).  The wait is part of the
//     same asm statement, so the registers are valid when it returns.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape),
// one wait for the whole load.
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, float *v) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive 32-bit TMEM columns of this thread's lane (32x32b shape),
// one wait for the whole load.
__device__ __forceinline__ void tmem_ld_x128(uint32_t taddr, float *v) {
    uint32_t r[128];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// Store 64 consecutive 32-bit TMEM columns of this thread's lane and wait
// for the store to complete.
__device__ __forceinline__ void tmem_st_x64(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])), "r"(__float_as_uint(v[32])), "r"(__float_as_uint(v[33])), "r"(__float_as_uint(v[34])), "r"(__float_as_uint(v[35])), "r"(__float_as_uint(v[36])), "r"(__float_as_uint(v[37])), "r"(__float_as_uint(v[38])), "r"(__float_as_uint(v[39])), "r"(__float_as_uint(v[40])), "r"(__float_as_uint(v[41])), "r"(__float_as_uint(v[42])), "r"(__float_as_uint(v[43])), "r"(__float_as_uint(v[44])), "r"(__float_as_uint(v[45])), "r"(__float_as_uint(v[46])), "r"(__float_as_uint(v[47])), "r"(__float_as_uint(v[48])), "r"(__float_as_uint(v[49])), "r"(__float_as_uint(v[50])), "r"(__float_as_uint(v[51])), "r"(__float_as_uint(v[52])), "r"(__float_as_uint(v[53])), "r"(__float_as_uint(v[54])), "r"(__float_as_uint(v[55])), "r"(__float_as_uint(v[56])), "r"(__float_as_uint(v[57])), "r"(__float_as_uint(v[58])), "r"(__float_as_uint(v[59])), "r"(__float_as_uint(v[60])), "r"(__float_as_uint(v[61])), "r"(__float_as_uint(v[62])), "r"(__float_as_uint(v[63]))
        : "memory");
}

// Store 128 consecutive 32-bit TMEM columns of this thread's lane and wait
// for the store to complete.
__device__ __forceinline__ void tmem_st_x128(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x128.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127,%128};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31])), "r"(__float_as_uint(v[32])), "r"(__float_as_uint(v[33])), "r"(__float_as_uint(v[34])), "r"(__float_as_uint(v[35])), "r"(__float_as_uint(v[36])), "r"(__float_as_uint(v[37])), "r"(__float_as_uint(v[38])), "r"(__float_as_uint(v[39])), "r"(__float_as_uint(v[40])), "r"(__float_as_uint(v[41])), "r"(__float_as_uint(v[42])), "r"(__float_as_uint(v[43])), "r"(__float_as_uint(v[44])), "r"(__float_as_uint(v[45])), "r"(__float_as_uint(v[46])), "r"(__float_as_uint(v[47])), "r"(__float_as_uint(v[48])), "r"(__float_as_uint(v[49])), "r"(__float_as_uint(v[50])), "r"(__float_as_uint(v[51])), "r"(__float_as_uint(v[52])), "r"(__float_as_uint(v[53])), "r"(__float_as_uint(v[54])), "r"(__float_as_uint(v[55])), "r"(__float_as_uint(v[56])), "r"(__float_as_uint(v[57])), "r"(__float_as_uint(v[58])), "r"(__float_as_uint(v[59])), "r"(__float_as_uint(v[60])), "r"(__float_as_uint(v[61])), "r"(__float_as_uint(v[62])), "r"(__float_as_uint(v[63])), "r"(__float_as_uint(v[64])), "r"(__float_as_uint(v[65])), "r"(__float_as_uint(v[66])), "r"(__float_as_uint(v[67])), "r"(__float_as_uint(v[68])), "r"(__float_as_uint(v[69])), "r"(__float_as_uint(v[70])), "r"(__float_as_uint(v[71])), "r"(__float_as_uint(v[72])), "r"(__float_as_uint(v[73])), "r"(__float_as_uint(v[74])), "r"(__float_as_uint(v[75])), "r"(__float_as_uint(v[76])), "r"(__float_as_uint(v[77])), "r"(__float_as_uint(v[78])), "r"(__float_as_uint(v[79])), "r"(__float_as_uint(v[80])), "r"(__float_as_uint(v[81])), "r"(__float_as_uint(v[82])), "r"(__float_as_uint(v[83])), "r"(__float_as_uint(v[84])), "r"(__float_as_uint(v[85])), "r"(__float_as_uint(v[86])), "r"(__float_as_uint(v[87])), "r"(__float_as_uint(v[88])), "r"(__float_as_uint(v[89])), "r"(__float_as_uint(v[90])), "r"(__float_as_uint(v[91])), "r"(__float_as_uint(v[92])), "r"(__float_as_uint(v[93])), "r"(__float_as_uint(v[94])), "r"(__float_as_uint(v[95])), "r"(__float_as_uint(v[96])), "r"(__float_as_uint(v[97])), "r"(__float_as_uint(v[98])), "r"(__float_as_uint(v[99])), "r"(__float_as_uint(v[100])), "r"(__float_as_uint(v[101])), "r"(__float_as_uint(v[102])), "r"(__float_as_uint(v[103])), "r"(__float_as_uint(v[104])), "r"(__float_as_uint(v[105])), "r"(__float_as_uint(v[106])), "r"(__float_as_uint(v[107])), "r"(__float_as_uint(v[108])), "r"(__float_as_uint(v[109])), "r"(__float_as_uint(v[110])), "r"(__float_as_uint(v[111])), "r"(__float_as_uint(v[112])), "r"(__float_as_uint(v[113])), "r"(__float_as_uint(v[114])), "r"(__float_as_uint(v[115])), "r"(__float_as_uint(v[116])), "r"(__float_as_uint(v[117])), "r"(__float_as_uint(v[118])), "r"(__float_as_uint(v[119])), "r"(__float_as_uint(v[120])), "r"(__float_as_uint(v[121])), "r"(__float_as_uint(v[122])), "r"(__float_as_uint(v[123])), "r"(__float_as_uint(v[124])), "r"(__float_as_uint(v[125])), "r"(__float_as_uint(v[126])), "r"(__float_as_uint(v[127]))
        : "memory");
}

// Store 16 consecutive 32-bit TMEM columns of this thread's lane without
// waiting; tmem_wait_st() waits for every store the thread issued.
__device__ __forceinline__ void tmem_st_x16_nowait(uint32_t taddr, const uint32_t *w) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]),
        "r"(w[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Host helpers (defined in api.cu)
// ---------------------------------------------------------------------------
// The device error word of the current device (a device address), or NULL.
uint32_t *device_error_word();
// 0 when the current device is compute capability 10.3; also returns the SM
// count.  Cached per device.
fp8kv_status check_device(int *num_sms);
bool scale_ok(float s);
// Tensor map over one cache array [block][head][row][d], viewed as a 4-D
// tensor (head_dim bytes, block rows, kv heads, blocks), box
// (128, block_size, 1, 1), 128-byte swizzle.  Returns false when the driver
// rejects it.
bool make_cache_map(CUtensorMap *map, const uint8_t *base, int64_t num_blocks, int block_size,
                    int num_kv_heads, int head_dim);
// Tensor map over a bf16 array [rows][heads][head_dim] (rows a bound on the
// rows that are read), box (64 values, 1 head, 32 rows) = 32 rows of 128
// bytes, 128-byte swizzle.  Returns false when the driver rejects it.
bool make_rows_map(CUtensorMap *map, const void *base, int64_t rows, int heads, int head_dim);

// Sets a kernel's dynamic shared-memory size (and, with max_carveout, the
// preference for the whole unified L1 as shared memory) once per device;
// `done` holds one bit per device already set.  False on a CUDA error.
bool func_attrs_once(const void *func, std::atomic<uint64_t> *done, int smem_bytes,
                     bool max_carveout);

}  // namespace fp8kv
