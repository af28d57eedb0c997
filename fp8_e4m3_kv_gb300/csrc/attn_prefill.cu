// attn_prefill.cu -- varlen causal / sliding-window prefill attention over
// the e4m3 paged cache on FP8 tensor cores (vLLM PR 54705: "Purpose",
// descale handling; evidence document Tier 0: P formed in e4m3 pre-scaled by
// 2^max_offset with max_offset = 8 and a lazy-rescale threshold of 0.75,
// below the log2(448) - 8 = 0.807 slack that keeps P from clipping).
//
// One CTA computes one tile of 128 query rows of one query head of one
// sequence.  Keys stream in tiles of 128 from the paged cache:
//   warp 4  (producer)  TMA-loads the K and V tiles (one box per block and
//                       128-byte column) into a 3-stage ring (2 for D = 256);
//   warp 5  (MMA)       one thread issues tcgen05 kind::f8f6f4 MMAs:
//                       S  = Q8 . K_tile^T            (128 x 128, fp32 in TMEM,
//                                                      double-buffered)
//                       O += P_hi . V_tile + P_lo . V_tile   (128 x D in TMEM)
//   warps 0-3 (softmax) thread r owns query row r (TMEM lane r): folded
//                       descale, exact bf16 relative bias, causal / window
//                       mask, running max with the lazy rescale, P, row sum,
//                       and at the end out = v_scale * O / l in bf16.
// P = exp2(z - m + 8) <= 2^(8 + 0.75) < 448 is stored as two e4m3 terms,
// P_hi = e4m3(P) and P_lo = e4m3(P - P_hi), so that the PV product stays on
// the FP8 tensor cores while the weights keep about 8 significant bits.
#include <math.h>

#include <atomic>

#include "common.cuh"

namespace fp8kv {
namespace {

constexpr int kPreThreads = 192;
constexpr float kLog2eP = 1.4426950408889634f;
// P = 2^(z - m + kPOffset) with a lazy reference m: the row's reference max
// moves only when its max grew by more than kRescaleTau, so P stays below
// 2^(kPOffset + kRescaleTau) < 448 (the pages' rule tau < log2(448) -
// max_offset).  The pages' kernel uses max_offset 8 with tau 0.75; here the
// head_dim-128 kernel takes max_offset 6 with tau 2.75, the same rule: a
// rescale of O in tensor memory is warp-wide (any of its 32 rows), and at
// tau 0.75 about half of all 64-key halves paid one.  The e4m3 weights keep
// their 3-bit precision down to 2^-12 of the row max (2^-14 at offset 8).
constexpr float kRescaleTau = 0.75f;   // one-query-tile kernel (head_dim 256)
constexpr float kPOffset = 8.0f;
constexpr float kRescaleTau2 = 2.75f;  // two-pipeline kernel (head_dim 128)
constexpr float kPOffset2 = 6.0f;
static_assert(kPOffset + kRescaleTau < 8.807f && kPOffset2 + kRescaleTau2 < 8.807f,
              "P must stay below 448");
// One-term P budget.  Rounding P to one e4m3 term moves each weight by at
// most 2^-4 of itself, independently per key, so the output error it causes
// has a variance proportional to (sum of p^2 over the one-term keys) / l^2.
// A row keeps P in one term for a 64-key half while the running sum of
// p_max * l_half (>= sum of p^2) over its one-term halves stays within
// kPBudget * l^2, l being the row sum so far (it only grows, relative to the
// reference max, so the bound holds for the final l as well); otherwise the
// half gets the second term e4m3(P - P_hi) as well.  Rows with few visible
// keys or a few dominant weights take two terms, long flat rows one.
constexpr float kPBudget = 0.01f;

template <int D>
struct PreCfg {
    static constexpr int kCB = D / 128;
    static constexpr int kStages = D == 128 ? 3 : 2;
    static constexpr int kTileBytes = kTile * D;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = kTile * D;
    static constexpr int kPBytes = kTile * kTile;          // one P term, 16 KB
    static constexpr int kOffQ = 0;
    static constexpr int kOffStages = kQBytes;
    static constexpr int kOffP = kOffStages + kStages * kStageBytes;   // [hi, lo]
    static constexpr int kOffMisc = kOffP + 2 * kPBytes;
    static constexpr int kSmemBytes = kOffMisc + 1024 + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;                   // S buffers: cols 0, 128
    static constexpr uint32_t kColO = 256;                 // O: cols 256 .. 256 + D
};

struct PrefillParams {
    const uint16_t *q;
    const int32_t *cu_q;
    const int32_t *lens_k;
    const int32_t *block_table;
    const uint16_t *rel;
    uint16_t *out;
    uint32_t *err;
    int64_t bias_tok_stride;
    int64_t num_blocks;
    int32_t max_blocks;
    int32_t Hq;
    int32_t G;
    int32_t block_size;
    int32_t bs_shift;       // log2(block_size) (a power of two)
    int32_t rel_extent;
    int32_t window;
    int32_t n_qtiles;
    int32_t bias_vec;   // rows 16-byte aligned with an extent that is a multiple of 8
    int32_t num_seqs;
    int32_t persist;    // head_dim 128: one CTA per SM walking the sorted item list
    QScale q_scale;
    float score_log2;   // softmax_scale * q_scale * k_scale * log2(e)
    float v_scale;
    float bias_fold;    // log2(e) / score_log2, or 0 where that is not a safe finite factor
    // per-token scales (the per-token variant only):
    // float[num_blocks][num_kv_heads][block_size], one per cached token and head
    const float *k_tok_scale;
    const float *v_tok_scale;
    int32_t num_kv_heads;
    // head_dim-128 kernel: each softmax warp copies the next item's Q rows
    // with the tensor map qmap (only when its 32 rows are all the item's)
    int32_t q_tma;
};

__device__ __forceinline__ void mbar_drain_p(uint64_t *bar, uint32_t parity, uint32_t *err) {
    CtaFail never{0};
    mbar_wait(bar, parity, &never, err);
}

__device__ __forceinline__ bool warp_wait_p(uint64_t *bar, uint32_t parity, CtaFail *fail,
                                            uint32_t *err) {
    const bool ok = mbar_wait(bar, parity, fail, err);
    return __all_sync(0xffffffffu, ok);
}

// 16 consecutive P values of one row -> 16 e4m3 bytes of P_hi and of P_lo
// (P_lo = e4m3(P - P_hi), the difference taken in fp16).
__device__ __forceinline__ void split_p16(const float *pv, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t hw = 0, lw = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __half2 ph = __floats2half2_rn(pv[4 * w + 2 * k], pv[4 * w + 2 * k + 1]);
            const __half2_raw phr = ph;
            const uint32_t h8 = __nv_cvt_halfraw2_to_fp8x2(phr, __NV_SATFINITE, __NV_E4M3);
            const __half2 hh = e4m3x2_to_half2(static_cast<uint16_t>(h8));
            const __half2_raw rr = __hsub2(ph, hh);
            const uint32_t l8 = __nv_cvt_halfraw2_to_fp8x2(rr, __NV_SATFINITE, __NV_E4M3);
            hw |= (h8 & 0xFFFFu) << (16 * k);
            lw |= (l8 & 0xFFFFu) << (16 * k);
        }
        h[w] = hw;
        l[w] = lw;
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

template <int D>
__global__ void __launch_bounds__(kPreThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const PrefillParams p) {
    using C = PreCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x);   // longest tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int kvh = h / p.G;
    const int q_first = p.cu_q[b];
    const int len_q = p.cu_q[b + 1] - q_first;
    if (qt * kTile >= len_q) return;
    const int64_t len_k = p.lens_k[b];
    const int n_rows = min(kTile, len_q - qt * kTile);
    const int64_t P0 = len_k - len_q + static_cast<int64_t>(qt) * kTile;   // position of row 0
    const int64_t pos_last = P0 + n_rows - 1;
    int64_t key_lo = 0;
    if (p.window > 0 && P0 - p.window + 1 > 0) key_lo = P0 - p.window + 1;
    const int64_t kt0 = key_lo / kTile;
    const int ntiles = static_cast<int>((pos_last + 1 + kTile - 1) / kTile - kt0);
    if (ntiles <= 0 || P0 < 0) return;   // (seq_lens_k smaller than the query count)

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffMisc);
    uint64_t *full = bars;              // [3]
    uint64_t *empty = bars + 3;         // [3]
    uint64_t *s_full = bars + 6;        // [2]
    uint64_t *s_free = bars + 8;        // [2]
    uint64_t *p_full = bars + 10;       // P of the current tile written
    uint64_t *o_done = bars + 11;       // PV of a tile complete
    uint64_t *mma_done = bars + 12;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc + 128);
    CtaFail *fail = reinterpret_cast<CtaFail *>(smem + C::kOffMisc + 132);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(mma_done, 1);
        fail->abort = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(tmem_slot, C::kTmemCols);
    if (warp < 4) {
        // Q8 row r = e4m3(q / q_scale), 128-byte swizzled K-major; rows past
        // the sequence's queries are zero.
        const int r = threadIdx.x;
        const uint16_t *qrow = p.q + (static_cast<int64_t>(q_first) + qt * kTile + r) * p.Hq * D +
                               static_cast<int64_t>(h) * D;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            uint4 packed = make_uint4(0, 0, 0, 0);
            if (r < n_rows) {
                const uint4 w0 = *reinterpret_cast<const uint4 *>(qrow + c * 16);
                const uint4 w1 = *reinterpret_cast<const uint4 *>(qrow + c * 16 + 8);
                packed.x = quantize_bf16x2(w0.x, p.q_scale) | (quantize_bf16x2(w0.y, p.q_scale) << 16);
                packed.y = quantize_bf16x2(w0.z, p.q_scale) | (quantize_bf16x2(w0.w, p.q_scale) << 16);
                packed.z = quantize_bf16x2(w1.x, p.q_scale) | (quantize_bf16x2(w1.y, p.q_scale) << 16);
                packed.w = quantize_bf16x2(w1.z, p.q_scale) | (quantize_bf16x2(w1.w, p.q_scale) << 16);
            }
            const int cb = c / 8, cc = c % 8;
            *reinterpret_cast<uint4 *>(smem + C::kOffQ + cb * (kTile * 128) + r * 128 +
                                       ((cc ^ (r & 7)) << 4)) = packed;
        }
        fence_proxy_async_smem();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_map(&kmap);
        tma_prefetch_map(&vmap);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = l2_policy_evict_first();
        const int nb = kTile / p.block_size;
        int last_issued[C::kStages];
#pragma unroll
        for (int s = 0; s < C::kStages; ++s) last_issued[s] = -1;
        for (int i = 0; i < ntiles; ++i) {
            const int s = i % C::kStages;
            int32_t phys = static_cast<int32_t>(p.num_blocks);   // out of range: zero fill
            if (lane < nb) {
                const int64_t lb = (kt0 + i) * nb + lane;
                if (lb * p.block_size < len_k) {
                    // a length past the block table is flagged like a bad id
                    const int32_t id =
                        lb < p.max_blocks
                            ? __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + lb)
                            : -1;
                    if (id >= 0 && id < p.num_blocks)
                        phys = id;
                    else
                        atomicOr(p.err, FP8KV_DEVERR_BAD_BLOCK);
                }
            }
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, fail, p.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            __syncwarp();
            if (lane < nb) {
                uint8_t *kdst = smem + C::kOffStages + s * C::kStageBytes + lane * p.block_size * 128;
                uint8_t *vdst = kdst + C::kTileBytes;
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb) {
                    tma_load_4d(kdst + cb * (kTile * 128), &kmap, &full[s], cb * 128, 0, kvh, phys, pol);
                    tma_load_4d(vdst + cb * (kTile * 128), &vmap, &full[s], cb * 128, 0, kvh, phys, pol);
                }
            }
            last_issued[s] = i;
        }
        if (lane == 0 && fail->abort) {
            for (int s = 0; s < C::kStages; ++s)
                if (last_issued[s] >= 0)
                    mbar_drain_p(&full[s], (last_issued[s] / C::kStages) & 1, p.err);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_e4m3_f32(128, 128, false, false);
            const uint32_t idesc_pv = idesc_e4m3_f32(128, 128, false, true);
            const uint32_t q_addr = smem_u32(smem + C::kOffQ);
            const uint32_t p_addr = smem_u32(smem + C::kOffP);
            for (int i = 0; i <= ntiles; ++i) {
                if (i < ntiles) {
                    const int s = i % C::kStages, sb = i & 1;
                    if (!mbar_wait(&full[s], (i / C::kStages) & 1, fail, p.err)) break;
                    if (!mbar_wait(&s_free[sb], ((i >> 1) & 1) ^ 1, fail, p.err)) break;
                    tc_fence_after_sync();
                    const uint32_t k_addr = smem_u32(smem + C::kOffStages + s * C::kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk) {
                        const uint32_t cb = kk / 4, ko = (kk % 4) * 32;
                        const uint64_t a = sdesc_sw128(q_addr + cb * (kTile * 128) + ko, 16, 1024);
                        const uint64_t bd = sdesc_sw128(k_addr + cb * (kTile * 128) + ko, 16, 1024);
                        mma_e4m3(tmem + C::kColS + sb * 128, a, bd, idesc_qk, kk > 0);
                    }
                    tc_commit(&s_full[sb]);
                }
                if (i >= 1) {
                    const int j = i - 1, s = j % C::kStages;
                    if (!mbar_wait(p_full, j & 1, fail, p.err)) break;
                    tc_fence_after_sync();
                    const uint32_t v_addr =
                        smem_u32(smem + C::kOffStages + s * C::kStageBytes + C::kTileBytes);
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb) {
#pragma unroll
                        for (int part = 0; part < 2; ++part) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                // A = P (K-major, 128 keys per row); B = V tile
                                // (MN-major: key rows of 128 d-bytes, 8-row groups
                                // 1024 bytes apart), 32 keys per MMA.
                                const uint64_t a =
                                    sdesc_sw128(p_addr + part * C::kPBytes + kk * 32, 16, 1024);
                                const uint64_t bd = sdesc_sw128(
                                    v_addr + cb * (kTile * 128) + kk * 32 * 128, kTile * 128, 1024);
                                mma_e4m3(tmem + C::kColO + cb * 128, a, bd, idesc_pv,
                                         (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    }
                    tc_commit(o_done);
                    tc_commit(&empty[s]);
                }
            }
            tc_commit(mma_done);
            mbar_drain_p(mma_done, 0, p.err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int r = threadIdx.x;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        const int64_t pos = P0 + r;
        const bool row_ok = r < n_rows;
        const uint16_t *bias_row =
            (p.rel && row_ok) ? p.rel + (static_cast<int64_t>(q_first) + qt * kTile + r) *
                                            p.bias_tok_stride + static_cast<int64_t>(h) * p.rel_extent
                              : nullptr;
        uint8_t *p_hi = smem + C::kOffP;
        uint8_t *p_lo = p_hi + C::kPBytes;
        float m_used = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int sb = i & 1;
            if (!warp_wait_p(&s_full[sb], (i >> 1) & 1, fail, p.err)) { ok = false; break; }
            tc_fence_after_sync();
            float z[128];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld_x32(tmem + lane_base + C::kColS + sb * 128 + c * 32, z + c * 32);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[sb]);

            const int64_t k0 = (kt0 + i) * kTile;
            const bool full_tile = (k0 + kTile - 1 <= P0) &&
                                   (p.window == 0 || pos_last - k0 < p.window) &&
                                   (k0 + kTile - 1 < len_k);
            const bool bias_tile = bias_row != nullptr && pos - k0 >= 0 &&
                                   pos - k0 - (kTile - 1) < p.rel_extent;
            float mx = -INFINITY;
            if (full_tile && !bias_tile) {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    z[c] *= p.score_log2;
                    mx = fmaxf(mx, z[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    const int64_t kidx = k0 + c;
                    float zz = z[c] * p.score_log2;
                    const int64_t d = pos - kidx;
                    if (bias_tile && d >= 0 && d < p.rel_extent)
                        zz = fmaf(bf16_bits_to_float(__ldg(bias_row + d)), kLog2eP, zz);
                    const bool valid = d >= 0 && (p.window == 0 || d < p.window) && kidx < len_k;
                    zz = valid ? zz : -INFINITY;
                    z[c] = zz;
                    mx = fmaxf(mx, zz);
                }
            }
            // lazy rescale: move the reference max only when the row max grew
            // by more than tau, so P <= 2^(8 + tau) stays below 448
            const bool resc = mx > m_used + kRescaleTau;
            const float m_new = resc ? mx : m_used;
            const float alpha = (resc && m_used != -INFINITY) ? exp2f(m_used - m_new) : 1.0f;
            if (i >= 1) {
                if (!warp_wait_p(o_done, (i - 1) & 1, fail, p.err)) { ok = false; break; }
                tc_fence_after_sync();
                if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        const uint32_t ta = tmem + lane_base + C::kColO + c * 32;
                        tmem_ld_x32(ta, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= alpha;
                        tmem_st_x32(ta, o);
                    }
                }
            }
            l *= alpha;
            m_used = m_new;
            const float m8 = (m_used == -INFINITY) ? 0.0f : m_used - kPOffset;
            const int sw = r & 7;
#pragma unroll
            for (int c16 = 0; c16 < 8; ++c16) {
                float pv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    pv[e] = exp2f(z[c16 * 16 + e] - m8);
                    l += pv[e];
                }
                uint4 hi, lo;
                split_p16(pv, hi, lo);
                const uint32_t off = r * 128 + ((c16 ^ sw) << 4);
                *reinterpret_cast<uint4 *>(p_hi + off) = hi;
                *reinterpret_cast<uint4 *>(p_lo + off) = lo;
            }
            // keys past the end of the sequence may hold stale bytes (NaN codes
            // included): zero their V rows so that 0 * V stays 0 in the MMA
            if (k0 + r >= len_k) {
                uint8_t *vrow = smem + C::kOffStages + (i % C::kStages) * C::kStageBytes +
                                C::kTileBytes + r * 128;
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb) {
                    uint4 *q4 = reinterpret_cast<uint4 *>(vrow + cb * (kTile * 128));
#pragma unroll
                    for (int c = 0; c < 8; ++c) q4[c] = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && warp_wait_p(o_done, (ntiles - 1) & 1, fail, p.err)) {
            tc_fence_after_sync();
            const float f = (l > 0.0f) ? p.v_scale / l : 0.0f;
            uint16_t *orow = p.out + (static_cast<int64_t>(q_first) + qt * kTile + r) * p.Hq * D +
                             static_cast<int64_t>(h) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld_x32(tmem + lane_base + C::kColO + c * 32, o);
                if (row_ok) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[2 * e] * f, o[2 * e + 1] * f);
                        w[e] = *reinterpret_cast<const uint32_t *>(&v2);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// head_dim 128: two independent query-tile pipelines per CTA
//
// A work item is one query tile (128 rows) of one head of one sequence.  A
// CTA runs two pipelines, k = 0 and 1, each with its own items, K/V ring, Q8
// and P buffers and TMEM columns (S_k: 128, O_k: 128), sharing only the
// tensor cores and the issue slots; neither waits on the other, so one
// pipeline's per-item work (loading and quantizing Q, writing the output)
// overlaps the other's MMAs and softmax.  Pipeline k: warp 8 + 3k is its
// producer (TMA-loads the item's key tiles into a 2-stage ring), warp 9 + k
// its MMA issuer, warps 4k .. 4k + 3 its softmax warpgroup.  For up to 64
// sequences the kernel is persistent: one CTA per SM, each pipeline working
// through a list of items; within a pipeline the producer runs on into the
// next item's key tiles, and the softmax warpgroup, as soon as the last P of
// an item is written, loads the next item's Q (the issuer starts its QKs)
// and then writes the finished item's output while those QKs run.  Each key
// tile is worked in two halves of 64 keys, each with its own half of S and
// of P, so that S and P are double-buffered within the same TMEM and shared
// memory and the lazy rescale is decided per half.  Per element the softmax
// is one FMA (the folded score scale and the running max), one ex2, the row
// sum, and the two-term e4m3 split done on packed f16 pairs.
// ---------------------------------------------------------------------------
// Three warpgroups: two softmax warpgroups, then the two producer warps and
// the two MMA warps.  The kernel is built for 384 threads at 168 registers;
// at run time the third warpgroup gives registers back (setmaxnreg.dec to
// kRegsIo) and the softmax warpgroups take them (setmaxnreg.inc to
// kRegsSoftmax): 2*128*224 + 128*56 = 384*168.
constexpr int kPre2Threads = 384;
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 224;
constexpr int kRegsIo = 56;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsIo <= kPre2Threads * kRegsLaunch,
              "register split exceeds the launch's registers");
// Batches of up to this many sequences run persistent (each CTA sorts them by
// query count); larger ones get one CTA per two query tiles.
constexpr int kPre2SchedSeqs = 64;

struct Pre2Cfg {
    static constexpr int kStages = 2;                       // per pipeline
    static constexpr int kTileBytes = kTile * 128;          // K or V tile, 16 KB
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = kTile * 128;             // one Q8 tile, 16 KB
    static constexpr int kPBytes = kTile * kTile;           // one P term, 16 KB
    static constexpr int kOffQ = 0;                         // [pipeline] Q8
    static constexpr int kOffStages = 2 * kQBytes;          // [pipeline][stage]
    // [pipeline] 32 KB: the output staging of the epilogue (and the sort's
    // scratch at the start); P itself lives in tensor memory
    static constexpr int kOffP = kOffStages + 2 * kStages * kStageBytes;
    static constexpr int kOffMisc = kOffP + 2 * 2 * kPBytes;
    static constexpr int kOffSched = kOffMisc + 512;        // sorted sequence tables
    static constexpr int kSmemBytes = kOffSched + 4 * 4 * kPre2SchedSeqs + 1024;
    static constexpr uint32_t kTmemCols = 512;              // S0 O0 | S1 O1
    static constexpr int kHalf = kTile / 2;                 // keys per unit
    // per-token variant: per pipeline and ring stage, three float[128] key
    // tables (score factor, log2 of the V scale, its reciprocal) in the
    // staging area, which that variant's epilogue does not use
    static constexpr int kOffTab = kOffP;
};
static_assert(2 * Pre2Cfg::kStages * 2048 <= 2 * 2 * Pre2Cfg::kPBytes, "per-token tables");
static_assert(Pre2Cfg::kSmemBytes <= 227 * 1024, "shared memory");

// 16 x 8 bf16 -> 16 x 8 e4m3 bytes, the scale's form fixed at compile time.
template <bool kPow2>
__device__ __forceinline__ void quantize_q16(const uint4 (&v)[16], uint2 (&o)[16],
                                             const QScale &s) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        o[i].x = quantize_q_bf16x2<kPow2>(v[i].x, s) | (quantize_q_bf16x2<kPow2>(v[i].y, s) << 16);
        o[i].y = quantize_q_bf16x2<kPow2>(v[i].z, s) | (quantize_q_bf16x2<kPow2>(v[i].w, s) << 16);
    }
}

__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16 consecutive P values of one row -> their 16 e4m3 bytes, nearest even,
// straight from fp32 (P <= 2^(8 + tau) never reaches the saturation bound).
__device__ __forceinline__ uint4 p_hi16(const float *pv) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = static_cast<uint32_t>(f32x2_to_e4m3x2(pv[4 * i], pv[4 * i + 1])) |
               (static_cast<uint32_t>(f32x2_to_e4m3x2(pv[4 * i + 2], pv[4 * i + 3])) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The second terms e4m3(P - P_hi) of the same 16 values, given their P_hi
// bytes; the difference is taken in fp16, where it is exact.
__device__ __forceinline__ uint4 p_lo16(const float *pv, const uint4 hi) {
    const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t half_words[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const __half2 ph = __floats2half2_rn(pv[4 * i + 2 * k], pv[4 * i + 2 * k + 1]);
            const __half2 hh = e4m3x2_to_half2(static_cast<uint16_t>(hw[i] >> (16 * k)));
            half_words[k] =
                __nv_cvt_halfraw2_to_fp8x2(__hsub2(ph, hh), __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
        }
        w[i] = half_words[0] | (half_words[1] << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The bias of 64 consecutive keys of one row, fetched before any of it is
// used: Y holds row[lo + i] at half i (i = 0 .. 63, lo = d0 - 63, so key e of
// the half, at distance d0 - e, is half 63 - e) and 0 where lo + i is outside
// [0, extent) or row is null.  With vec the row is read as 16-byte chunks
// from the multiple of 8 at or below lo (a chunk lies wholly inside or
// outside the extent) and shifted down by the remainder; otherwise as 64
// independent 2-byte loads.
__device__ __forceinline__ void load_bias64(const uint16_t *row, int32_t d0, int32_t extent,
                                            bool vec, uint32_t (&Y)[32]) {
    const int32_t lo = d0 - 63;
    if (vec) {
        const int32_t base = lo & ~7;
        const int32_t rem = lo - base;   // 0 .. 7 halves
        uint32_t w[36];
#pragma unroll
        for (int c = 0; c < 9; ++c) {
            const int32_t i0 = base + 8 * c;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (row != nullptr && i0 >= 0 && i0 + 8 <= extent)
                v = __ldg(reinterpret_cast<const uint4 *>(row + i0));
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
        }
        // shift by rem halves: whole words by rem / 2 (two select stages),
        // then the odd half with a funnel shift
        const bool by1 = rem & 2, by2 = rem & 4, odd = rem & 1;
#pragma unroll
        for (int m = 0; m < 35; ++m) w[m] = by1 ? w[m + 1] : w[m];
#pragma unroll
        for (int m = 0; m < 33; ++m) w[m] = by2 ? w[m + 2] : w[m];
#pragma unroll
        for (int m = 0; m < 32; ++m) Y[m] = odd ? __funnelshift_r(w[m], w[m + 1], 16) : w[m];
    } else {
        uint16_t hv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const int32_t j = lo + i;
            hv[i] = (row != nullptr && j >= 0 && j < extent) ? __ldg(row + j) : uint16_t(0);
        }
#pragma unroll
        for (int m = 0; m < 32; ++m)
            Y[m] = static_cast<uint32_t>(hv[2 * m]) | (static_cast<uint32_t>(hv[2 * m + 1]) << 16);
    }
}

// One work item: query tile qt (128 rows) of head h of sequence b, and the
// key tiles kt_lo .. kt_hi it reads.
struct Pre2Item {
    int32_t b, h, qt, q_first, n_rows;
    int32_t len_k, P0, kt_lo, kt_hi;   // positions fit in int32: key counts are int32
};

// Fills the item; false when it holds no query (past the sequence's queries,
// or fewer keys than queries).
__device__ __forceinline__ bool pre2_item(const PrefillParams &p, int32_t b, int32_t q_first,
                                          int32_t len_q, int32_t len_k, int32_t h, int32_t qt,
                                          Pre2Item &it) {
    if (qt < 0 || qt * kTile >= len_q || len_k < len_q) return false;
    it.b = b;
    it.h = h;
    it.qt = qt;
    it.q_first = q_first;
    it.len_k = len_k;
    it.n_rows = min(kTile, len_q - qt * kTile);
    it.P0 = len_k - len_q + qt * kTile;
    const int32_t key_lo = (p.window > 0 && it.P0 - p.window + 1 > 0) ? it.P0 - p.window + 1 : 0;
    it.kt_lo = key_lo / kTile;
    it.kt_hi = (it.P0 + it.n_rows - 1) / kTile;
    return true;
}

// The sorted sequence table of a persistent launch: entry r describes the
// sequence with the r-th most queries (ties by index).
struct Pre2Seqs {
    int32_t *seq, *q_first, *len_q, *len_k;   // len_q 0: no query to compute
};

// The items of one pipeline.  Every role of the pipeline walks them with
// its own copy of this state and gets the same items in the same order.
//
// Persistent launch: the items are ordered by query tile index, highest first
// (for causal and windowed rows, the items with the most key tiles first),
// then by sequence in table order, then by head; empty items are left out.
// With V = 2 x CTAs pipelines, pipeline v takes positions v, 2V - 1 - v,
// 2V + v, 4V - 1 - v, ... of that list, so that each gets one of the
// costliest and one of the cheapest items of every 2V.
//
// Flat launch (more sequences than the table holds): CTA (x, h, b) has query
// tiles 2 x' and 2 x' + 1 of head h of sequence b, x' = pairs - 1 - x, one per
// pipeline.
struct Pre2Sched {
    int32_t step = 0;        // items taken so far
    int32_t lev_start = 0;   // list position of the current query tile level
    int32_t lev_n = 0;       // items in it
    int32_t lev = -1;        // levels passed, highest query tile first
};

__device__ __forceinline__ bool pre2_next(const PrefillParams &p, const Pre2Seqs &t, int k,
                                          Pre2Sched &sc, Pre2Item &it) {
    if (!p.persist) {
        if (sc.step++ > 0) return false;
        const int b = static_cast<int>(blockIdx.z);
        const int q_first = __ldg(p.cu_q + b);
        const int n_pairs = (p.n_qtiles + 1) / 2;
        return pre2_item(p, b, q_first, __ldg(p.cu_q + b + 1) - q_first, __ldg(p.lens_k + b),
                         static_cast<int>(blockIdx.y),
                         2 * (n_pairs - 1 - static_cast<int>(blockIdx.x)) + k, it);
    }
    // list positions fit in int32 (checked when the launch is set up)
    const int32_t V = 2 * static_cast<int32_t>(gridDim.x), v = 2 * blockIdx.x + k;
    const int32_t blk = sc.step++;
    const int32_t i = blk * V + ((blk & 1) ? V - 1 - v : v);
    while (i >= sc.lev_start + sc.lev_n) {
        if (sc.lev + 1 >= p.n_qtiles) return false;
        sc.lev_start += sc.lev_n;
        ++sc.lev;
        // sequences with more than kTile * qt queries: a prefix of the table
        const int32_t floor_q = kTile * (p.n_qtiles - 1 - sc.lev);
        int lo = 0, hi = p.num_seqs;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (t.len_q[mid] > floor_q)
                lo = mid + 1;
            else
                hi = mid;
        }
        sc.lev_n = lo * p.Hq;
    }
    const int32_t rem = i - sc.lev_start;
    const int32_t r = rem / p.Hq;
    return pre2_item(p, t.seq[r], t.q_first[r], t.len_q[r], t.len_k[r], rem - r * p.Hq,
                     p.n_qtiles - 1 - sc.lev, it);
}

// kPT: per-token scales.  Key j's score is x_j * score_log2 * k_scale_j; its
// V scale is folded into the exponent, P_j = 2^(z_j + log2 v_scale_j - m +
// offset), so that the MMA weights are p_j * v_scale_j, and the row sum adds
// P_j / v_scale_j.  The producer writes the three per-key factors of each
// key tile into its stage's table.
// kUnfold: the bias is added to the scaled score (the q / k scales are too
// extreme for the folded factor bias_fold); else as bias * bias_fold with the
// score scale kept in the FMA of P.  Each is its own instantiation, so that
// the softmax loop holds only the code it runs.
template <bool kPT, bool kUnfold>
__global__ void __launch_bounds__(kPre2Threads, 1)
prefill2_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const __grid_constant__ CUtensorMap qmap, const PrefillParams p) {
    using C = Pre2Cfg;
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // barriers of pipeline k at bars + 16 k
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffMisc);
    auto full = [&](int k, int s) { return bars + 16 * k + s; };         // stage loaded
    auto empty = [&](int k, int s) { return bars + 16 * k + 2 + s; };    // stage consumed
    auto s_full = [&](int k, int hh) { return bars + 16 * k + 4 + hh; }; // S half written by QK
    auto p_full = [&](int k, int hh) { return bars + 16 * k + 8 + hh; }; // P half written
    auto o_done = [&](int k, int hh) { return bars + 16 * k + 10 + hh; };// PV of P half done
    auto q_full = [&](int k) { return bars + 16 * k + 12; };             // Q8 of next item
    auto mma_done = [&](int k) { return bars + 16 * k + 13; };
    // softmax warp w of pipeline k: its copy of the next item's Q rows landed
    auto qbar = [&](int k, int w) { return bars + 36 + 4 * k + w; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc + 256);
    CtaFail *fail = reinterpret_cast<CtaFail *>(smem + C::kOffMisc + 260);
    // byte wq of lo_flag(k, hh): softmax warp wq of pipeline k wrote a second
    // P term for its rows of the current unit of half hh (written before the
    // warp arrives on p_full, read by the MMA thread after it waits there)
    auto lo_flag = [&](int k, int hh) {
        return reinterpret_cast<volatile uint8_t *>(smem + C::kOffMisc + 264 + 8 * k + 4 * hh);
    };
    // per-token key tables of pipeline k's ring stage s: [factor | log2 sv | 1 / sv]
    auto key_tab = [&](int k, int s) {
        return reinterpret_cast<float *>(smem + C::kOffTab + (2 * k + s) * 2048);
    };
    Pre2Seqs tab;
    tab.seq = reinterpret_cast<int32_t *>(smem + C::kOffSched);
    tab.q_first = tab.seq + kPre2SchedSeqs;
    tab.len_q = tab.q_first + kPre2SchedSeqs;
    tab.len_k = tab.len_q + kPre2SchedSeqs;

    if (p.persist) {
        // sort the sequences by query count, most first (ties by index): the
        // rank of each is the number of sequences ahead of it.  The counts
        // are staged in the P buffers, unused until the first item.
        int32_t *eff = reinterpret_cast<int32_t *>(smem + C::kOffP);
        for (int b = threadIdx.x; b < p.num_seqs; b += blockDim.x) {
            const int32_t q0 = __ldg(p.cu_q + b), lq = __ldg(p.cu_q + b + 1) - q0;
            eff[b] = (lq > 0 && __ldg(p.lens_k + b) >= lq) ? lq : 0;
        }
        __syncthreads();
        for (int b = threadIdx.x; b < p.num_seqs; b += blockDim.x) {
            const int32_t e = eff[b];
            int r = 0;
            for (int o = 0; o < p.num_seqs; ++o) {
                const int32_t eo = eff[o];
                r += (eo > e || (eo == e && o < b)) ? 1 : 0;
            }
            tab.seq[r] = b;
            tab.q_first[r] = __ldg(p.cu_q + b);
            tab.len_q[r] = e;
            tab.len_k[r] = __ldg(p.lens_k + b);
        }
    }
    if (threadIdx.x == 0) {
        for (int k = 0; k < 2; ++k) {
            for (int s = 0; s < C::kStages; ++s) {
                mbar_init(full(k, s), 1);
                mbar_init(empty(k, s), 1);
            }
            for (int hh = 0; hh < 2; ++hh) {
                mbar_init(s_full(k, hh), 1);
                mbar_init(p_full(k, hh), 4);
                mbar_init(o_done(k, hh), 1);
            }
            mbar_init(q_full(k), 4);
            mbar_init(mma_done(k), 1);
            for (int w = 0; w < 4; ++w) mbar_init(qbar(k, w), 1);
        }
        fail->abort = 0;
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(tmem_slot, C::kTmemCols);
    if ((warp == 8 || warp == 11) && lane == 0) {
        tma_prefetch_map(&kmap);
        tma_prefetch_map(&vmap);
        if (p.q_tma) tma_prefetch_map(&qmap);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // Per pipeline, counters that run across its items give every barrier
    // phase: stages of its ring (each item's key tiles pass through it once),
    // 64-key units (two per key tile; unit u uses S and P half u & 1), and
    // items.
    if (warp >= 8) {
      // the third warpgroup (producers and MMA issuers) gives registers back
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIo));
      if (warp == 8 || warp == 11) {
        // ------------------------------------------------------------ producer
        const int k = warp == 8 ? 0 : 1;
        const uint64_t pol = l2_policy_evict_first();
        const int nb = kTile / p.block_size;
        uint8_t *ring = smem + C::kOffStages + k * C::kStages * C::kStageBytes;
        int last_issued[C::kStages];
#pragma unroll
        for (int s = 0; s < C::kStages; ++s) last_issued[s] = -1;
        int g = 0;   // stages filled
        bool ok = true;
        Pre2Sched sc;
        Pre2Item it;
        while (ok && pre2_next(p, tab, k, sc, it)) {
            const int kvh = it.h / p.G;
            for (int32_t t = it.kt_lo; t <= it.kt_hi; ++t, ++g) {
                const int s = g % C::kStages;
                int32_t phys = static_cast<int32_t>(p.num_blocks);   // out of range: zero fill
                if (lane < nb) {
                    const int64_t lb = static_cast<int64_t>(t) * nb + lane;
                    if (lb * p.block_size < it.len_k) {
                        // a length past the block table is flagged like a bad id
                        const int32_t id =
                            lb < p.max_blocks
                                ? __ldg(p.block_table + static_cast<int64_t>(it.b) * p.max_blocks + lb)
                                : -1;
                        if (id >= 0 && id < p.num_blocks)
                            phys = id;
                        else
                            atomicOr(p.err, FP8KV_DEVERR_BAD_BLOCK);
                    }
                }
                int w_ok = 1;
                if (lane == 0)
                    w_ok = mbar_wait(empty(k, s), ((g / C::kStages) & 1) ^ 1, fail, p.err);
                if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
                    ok = false;
                    break;
                }
                if constexpr (kPT) {
                    // the stage's key table (its previous tile's softmax is
                    // done with it: the stage is empty); four keys per lane.
                    // Keys outside the sequence get factors that keep their
                    // masked -inf scores -inf and add nothing to the sum.
                    float4 fk = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
                    float4 lv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    float4 iv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    float *fkp = &fk.x, *lvp = &lv.x, *ivp = &iv.x;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int32_t key = t * kTile + 4 * lane + i;
                        const int32_t lb = key >> p.bs_shift;
                        if (key < it.len_k && lb < p.max_blocks) {
                            const int32_t id =
                                __ldg(p.block_table + static_cast<int64_t>(it.b) * p.max_blocks + lb);
                            if (id >= 0 && id < p.num_blocks) {
                                const int64_t si = (static_cast<int64_t>(id) * p.num_kv_heads + kvh) *
                                                       p.block_size + (key & (p.block_size - 1));
                                const float sv = __ldg(p.v_tok_scale + si);
                                const float lv = log2f(sv);
                                fkp[i] = p.score_log2 * __ldg(p.k_tok_scale + si);
                                // below 2^-60 the exponent takes 2^-60 (and the
                                // sum its reciprocal): P stays far from fp32
                                // underflow, at an error below p * 2^-60 * 448
                                lvp[i] = fmaxf(lv, -60.0f);
                                ivp[i] = lv > -60.0f ? __frcp_rn(sv) : 0x1p60f;
                            }
                        }
                    }
                    float *tb = key_tab(k, s);
                    reinterpret_cast<float4 *>(tb)[lane] = fk;
                    reinterpret_cast<float4 *>(tb + kTile)[lane] = lv;
                    reinterpret_cast<float4 *>(tb + 2 * kTile)[lane] = iv;
                    __syncwarp();   // the table before lane 0's arrive releases it
                }
                if (lane == 0) mbar_arrive_expect_tx(full(k, s), C::kStageBytes);
                __syncwarp();
                if (lane < nb) {
                    uint8_t *kdst = ring + s * C::kStageBytes + lane * p.block_size * 128;
                    tma_load_4d(kdst, &kmap, full(k, s), 0, 0, kvh, phys, pol);
                    tma_load_4d(kdst + C::kTileBytes, &vmap, full(k, s), 0, 0, kvh, phys, pol);
                }
                last_issued[s] = g;
            }
        }
        if (lane == 0 && fail->abort) {
            for (int s = 0; s < C::kStages; ++s)
                if (last_issued[s] >= 0)
                    mbar_drain_p(full(k, s), (last_issued[s] / C::kStages) & 1, p.err);
        }
      } else {
        // ------------------------------------------------------------ MMA issuer
        // After the QK of unit u the thread issues the PV of unit u - 1, so
        // the softmax of one half overlaps the QK of the next and the PV of
        // the last; an item's last PV is issued before the thread moves on.
        // The PV of a key tile's second half releases its stage.  The first
        // PV of an item overwrites O: its P being written means the softmax
        // warps have read the previous item's O.
        const int k = warp - 9;
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_e4m3_f32(128, C::kHalf, false, false);
            const uint32_t idesc_pv = idesc_e4m3_f32(128, 128, false, true);
            const uint32_t q_addr = smem_u32(smem + C::kOffQ + k * C::kQBytes);
            const uint32_t ring = smem_u32(smem + C::kOffStages + k * C::kStages * C::kStageBytes);
            const uint32_t col_s = k * 256, col_o = k * 256 + 128;
            int g = 0;   // stages seen
            int U = 0;   // units whose QK was issued
            int A = 0;   // items
            bool ok = true;
            Pre2Sched sc;
            Pre2Item it;
            while (ok && pre2_next(p, tab, k, sc, it)) {
                const int g0 = g;
                const int n = it.kt_hi - it.kt_lo + 1;
                int ui = 0;   // units of this item issued
                bool q_ready = false;
                // O += P[:, half] . V_j[half, :] for unit v (half v & 1 of the
                // item's key tile j), P read from tensor memory, where the
                // softmax wrote it over the half's S columns (P_hi in the
                // first 16, P_lo in the next 16); the second half releases
                // the stage
                auto issue_pv = [&](int v, bool first, int j) -> bool {
                    const int hv = v & 1;
                    if (!mbar_wait(p_full(k, hv), (v >> 1) & 1, fail, p.err)) return false;
                    tc_fence_after_sync();
                    const int s = (g0 + j) % C::kStages;
                    const uint32_t v_addr = ring + s * C::kStageBytes + C::kTileBytes;
                    // the P_lo product only when a softmax warp wrote a second term
                    const int parts = *reinterpret_cast<volatile uint32_t *>(lo_flag(k, hv)) ? 2 : 1;
#pragma unroll 1
                    for (int part = 0; part < parts; ++part) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const int ks = 2 * hv + kk;   // 32-key step within the tile
                            const uint64_t bd = sdesc_sw128(v_addr + ks * 32 * 128, kTile * 128, 1024);
                            mma_e4m3_tmem_a(tmem + col_o, tmem + col_s + hv * C::kHalf + part * 16 + kk * 8,
                                            bd, idesc_pv, (!first || part > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(o_done(k, hv));
                    if (hv == 1) tc_commit(empty(k, s));
                    return true;
                };
                for (int j = 0; j < n && ok; ++j) {
                    const int s = (g0 + j) % C::kStages;
                    if (!mbar_wait(full(k, s), ((g0 + j) / C::kStages) & 1, fail, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t k_addr = ring + s * C::kStageBytes;
                    for (int hh = 0; hh < 2; ++hh) {
                        if (!q_ready && !(q_ready = mbar_wait(q_full(k), A & 1, fail, p.err))) {
                            ok = false;
                            break;
                        }
                        // S half hh last held P of unit U - 2, whose PV was
                        // issued before this QK: MMAs of this thread run in
                        // issue order, so the PV reads P before the QK writes
                        tc_fence_after_sync();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = sdesc_sw128(q_addr + kk * 32, 16, 1024);
                            const uint64_t bd =
                                sdesc_sw128(k_addr + hh * C::kHalf * 128 + kk * 32, 16, 1024);
                            mma_e4m3(tmem + col_s + hh * C::kHalf, a, bd, idesc_qk, kk > 0);
                        }
                        tc_commit(s_full(k, hh));
                        ++U;
                        ++ui;
                        if (ui >= 2 && !issue_pv(U - 2, ui == 2, hh == 1 ? j : j - 1)) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (ok && ui > 0) ok = issue_pv(U - 1, ui == 1, n - 1);
                g = g0 + n;
                ++A;
            }
            tc_commit(mma_done(k));
            mbar_drain_p(mma_done(k), 0, p.err);
        }
        __syncwarp();
      }
    } else {
        // ------------------------------------------------------------ softmax
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        const int k = warp >> 2, wq = warp & 3;
        const int r = threadIdx.x & 127;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t col_s = k * 256, col_o = k * 256 + 128;
        const int sw = r & 7;
        uint8_t *p_hi = smem + C::kOffP + k * 2 * C::kPBytes;
        uint8_t *p_lo = p_hi + C::kPBytes;
        uint8_t *ring = smem + C::kOffStages + k * C::kStages * C::kStageBytes;
        int g = 0;   // stages seen
        int c = 0;   // key tiles processed
        bool ok = true;
        // the previous item, whose output is still in O
        bool have_prev = false;
        int64_t prev_tok = 0;   // token of its first query row
        int prev_rows = 0, prev_h = 0;
        float2 prev_l = make_float2(0.0f, 0.0f);

        // out = bf16(v_scale * O / l) of the previous item, once the PV of
        // its last unit (the second half of its last key tile; its completion
        // means every earlier MMA of the pipeline completed too) is done.
        // Staged through this pipeline's P buffers, row r in its own P_hi and
        // P_lo rows (chunks 0-7 and 8-15), so that each warp stages and
        // stores its own 32 rows, two rows per coalesced store instruction.
        auto epilogue = [&]() -> bool {
            if (!warp_wait_p(o_done(k, 1), (c - 1) & 1, fail, p.err)) return false;
            tc_fence_after_sync();
            const float l = prev_l.x + prev_l.y;
            const float f = (l > 0.0f) ? p.v_scale / l : 0.0f;
            float o[D];
            tmem_ld_x128(tmem + lane_base + col_o, o);
            if constexpr (kPT) {
                // the staging area holds the key tables: each thread stores
                // its own row
                if (r < prev_rows) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + (prev_tok + r) * p.Hq * D +
                                                           static_cast<int64_t>(prev_h) * D);
#pragma unroll
                    for (int cch = 0; cch < D / 8; ++cch) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 v2 = __floats2bfloat162_rn(
                                o[8 * cch + 2 * e] * f, o[8 * cch + 2 * e + 1] * f);
                            w[e] = *reinterpret_cast<const uint32_t *>(&v2);
                        }
                        dst[cch] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            } else {
#pragma unroll
            for (int cch = 0; cch < D / 8; ++cch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 v2 =
                        __floats2bfloat162_rn(o[8 * cch + 2 * e] * f, o[8 * cch + 2 * e + 1] * f);
                    w[e] = *reinterpret_cast<const uint32_t *>(&v2);
                }
                *reinterpret_cast<uint4 *>((cch < 8 ? p_hi : p_lo) + r * 128 +
                                           (((cch & 7) ^ sw) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            __syncwarp();
            const int row_in_pair = lane >> 4, col = lane & 15;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int row = 32 * wq + 2 * i + row_in_pair;
                if (row < prev_rows) {
                    const uint4 val = *reinterpret_cast<const uint4 *>(
                        (col < 8 ? p_hi : p_lo) + row * 128 + (((col & 7) ^ (row & 7)) << 4));
                    *reinterpret_cast<uint4 *>(p.out + (prev_tok + row) * p.Hq * D +
                                               static_cast<int64_t>(prev_h) * D + col * 8) = val;
                }
            }
            // the rows are read back before the next item's P overwrites them
            __syncwarp();
            }
            return true;
        };

        // this warp's copy of the next item's Q rows into its staging rows
        // (P_hi / P_lo rows 32 wq .. 32 wq + 31: the epilogue's layout)
        bool q_pending = false;
        int q_copies = 0;
        Pre2Sched sc;
        Pre2Item it;
        while (ok && pre2_next(p, tab, k, sc, it)) {
            const int g0 = g;
            const int n = it.kt_hi - it.kt_lo + 1;
            g += n;
            const int32_t pos = it.P0 + r;   // positions are int32
            const bool row_ok = r < it.n_rows;
            const int32_t pos_first = it.P0, pos_last = it.P0 + it.n_rows - 1;
            const int64_t tok0 = static_cast<int64_t>(it.q_first) + it.qt * kTile;
            const uint16_t *bias_row =
                (p.rel && row_ok) ? p.rel + (tok0 + r) * p.bias_tok_stride +
                                        static_cast<int64_t>(it.h) * p.rel_extent
                                  : nullptr;
            {
                // Q8 of this item = e4m3(q / q_scale), rows past the
                // sequence's queries zero.  Q8 is free: every QK of the
                // previous item has completed, its S having been read.  Warp
                // wq loads rows 32 wq .. 32 wq + 31, two rows per load
                // instruction (16 lanes x 16 bytes per row), with all sixteen
                // loads in flight; the producer is already filling the ring.
                uint8_t *q8 = smem + C::kOffQ + k * C::kQBytes;
                const int row_in_pair = lane >> 4, col = lane & 15;   // 8 bf16 per lane
                uint4 v[16];
                if (!kPT && q_pending) {
                    // copied during the previous item: all 32 rows are this
                    // item's, in the staging rows (swizzled like the epilogue's)
                    if (!warp_wait_p(qbar(k, wq), (q_copies - 1) & 1, fail, p.err)) {
                        ok = false;
                        break;
                    }
                    q_pending = false;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int row = 32 * wq + 2 * i + row_in_pair;
                        v[i] = *reinterpret_cast<const uint4 *>(
                            (col < 8 ? p_hi : p_lo) + row * 128 + (((col & 7) ^ (row & 7)) << 4));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int row = 32 * wq + 2 * i + row_in_pair;
                        v[i] = make_uint4(0, 0, 0, 0);
                        if (row < it.n_rows)
                            v[i] = __ldg(reinterpret_cast<const uint4 *>(
                                p.q + (tok0 + row) * p.Hq * D + static_cast<int64_t>(it.h) * D +
                                col * 8));
                    }
                }
                // this row's bias is read on the diagonal key tiles: start it
                // toward L2 now
                if (bias_row != nullptr) {
                    for (int off = 0; off < p.rel_extent; off += 64) prefetch_l2(bias_row + off);
                    prefetch_l2(bias_row + p.rel_extent - 1);
                }
                uint2 q8w[16];
                if (p.q_scale.pow2)
                    quantize_q16<true>(v, q8w, p.q_scale);
                else
                    quantize_q16<false>(v, q8w, p.q_scale);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int row = 32 * wq + 2 * i + row_in_pair;
                    *reinterpret_cast<uint2 *>(q8 + row * 128 + (((col >> 1) ^ (row & 7)) << 4) +
                                               (col & 1) * 8) = q8w[i];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(q_full(k));
            }
            // the pipeline's next item: its Q rows are copied into this
            // warp's staging rows once the epilogue below is done with them
            // (when all 32 are the item's), else started toward L2
            int32_t nq_row = -1, nq_h = 0;
            {
                Pre2Sched peek = sc;
                Pre2Item nx;
                if (pre2_next(p, tab, k, peek, nx)) {
                    if (!kPT && p.q_tma && 32 * wq + 32 <= nx.n_rows) {
                        nq_row = nx.q_first + nx.qt * kTile + 32 * wq;
                        nq_h = nx.h;
                    } else if (r < nx.n_rows) {
                        const uint16_t *nq =
                            p.q + (static_cast<int64_t>(nx.q_first) + nx.qt * kTile + r) * p.Hq * D +
                            static_cast<int64_t>(nx.h) * D;
                        prefetch_l2(nq);
                        prefetch_l2(nq + 64);
                    }
                }
            }
            // the previous item's output, while the QKs of this one run
            if (have_prev && !(ok = epilogue())) break;
            if (!kPT && nq_row >= 0) {
                // the staging rows' generic reads and writes come before the
                // copy writes them
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(qbar(k, wq), 2 * 32 * 128);
                    tma_load_3d(p_hi + 32 * wq * 128, &qmap, qbar(k, wq), 0, nq_h, nq_row);
                    tma_load_3d(p_lo + 32 * wq * 128, &qmap, qbar(k, wq), 64, nq_h, nq_row);
                }
                ++q_copies;
                q_pending = true;
            }

            float m_used = -INFINITY;
            float2 lsum = make_float2(0.0f, 0.0f);   // two partial row sums
            float err_bound = 0.0f;   // sum of p_max * l_half over single-term halves
            for (int j = 0; j < n && ok; ++j) {
                const int32_t k0 = (it.kt_lo + j) * kTile;
                for (int hh = 0; hh < 2; ++hh) {
                    const int u = 2 * c + hh;   // unit: key half hh of this key tile
                    const int32_t kh = k0 + hh * C::kHalf;
                    const bool full_half = (kh + C::kHalf - 1 <= pos_first) &&
                                           (p.window == 0 || pos_last - kh < p.window);
                    const bool bias_half = bias_row != nullptr && pos - kh >= 0 &&
                                           pos - kh - (C::kHalf - 1) < p.rel_extent;
                    const int32_t d0 = static_cast<int32_t>(pos - kh);   // positions are int32
                    if (!warp_wait_p(s_full(k, hh), c & 1, fail, p.err)) { ok = false; break; }
                    tc_fence_after_sync();
                    if (hh == 0 && k0 + r >= it.len_k) {
                        // keys past the end of the sequence may hold stale
                        // bytes (NaN codes included): zero their V rows so
                        // that 0 * V stays 0 in the MMA.  S of this tile being
                        // written means the stage's TMA copies have landed.
                        uint4 *q4 = reinterpret_cast<uint4 *>(
                            ring + ((g0 + j) % C::kStages) * C::kStageBytes + C::kTileBytes +
                            r * 128);
#pragma unroll
                        for (int e = 0; e < 8; ++e) q4[e] = make_uint4(0, 0, 0, 0);
                        fence_proxy_async_smem();   // before the PV reads the rows
                    }
                    float x[C::kHalf];
                    tmem_ld_x64(tmem + lane_base + col_s + hh * C::kHalf, x);
                    const float *ktab = key_tab(k, (g0 + j) % C::kStages) + hh * C::kHalf;
                    if constexpr (kPT) {
                        // the producer's table of this stage: its full barrier
                        // (complete, since S of the tile exists) orders it
                        if (hh == 0 && !warp_wait_p(full(k, (g0 + j) % C::kStages),
                                                    ((g0 + j) / C::kStages) & 1, fail, p.err)) {
                            ok = false;
                            break;
                        }
                        // z = x * score_log2 * k_scale + log2(v_scale)
#pragma unroll
                        for (int e = 0; e < C::kHalf; e += 4) {
                            const float4 f4 = *reinterpret_cast<const float4 *>(ktab + e);
                            const float4 l4 = *reinterpret_cast<const float4 *>(ktab + kTile + e);
                            const float2 za = __ffma2_rn(make_float2(x[e], x[e + 1]),
                                                         make_float2(f4.x, f4.y), make_float2(l4.x, l4.y));
                            const float2 zb = __ffma2_rn(make_float2(x[e + 2], x[e + 3]),
                                                         make_float2(f4.z, f4.w), make_float2(l4.z, l4.w));
                            x[e] = za.x;
                            x[e + 1] = za.y;
                            x[e + 2] = zb.x;
                            x[e + 3] = zb.y;
                        }
                    }

                    // Scores to log2 units: z = x * score_log2 (+ bias *
                    // log2(e)), -inf where masked.  The scale stays folded
                    // into the FMA of P (mult): the bias is added as bias *
                    // log2(e) / score_log2; masking and the max do not need
                    // the scale, it being positive.
                    float mult = kPT ? 1.0f : p.score_log2;
                    const bool any_bias = __any_sync(0xffffffffu, bias_half);
                    if (any_bias) {
                        uint32_t Y[32];
                        load_bias64(bias_half ? bias_row : nullptr, d0, p.rel_extent,
                                    p.bias_vec != 0, Y);
                        if constexpr (kPT) {
                            // the scores are already in log2 units
#pragma unroll
                            for (int e = 0; e < C::kHalf; ++e) {
                                const uint32_t wd = Y[(63 - e) >> 1];
                                const float bv = __uint_as_float(((63 - e) & 1) ? (wd & 0xFFFF0000u)
                                                                                 : (wd << 16));
                                x[e] = fmaf(bv, kLog2eP, x[e]);
                            }
                        } else if constexpr (!kUnfold) {
                            // x + bias * log2(e) / score_log2: the score scale
                            // stays folded into the FMA of P (packed pairs;
                            // key e takes the upper half of its word for even e)
                            const float2 c2 = make_float2(p.bias_fold, p.bias_fold);
#pragma unroll
                            for (int e = 0; e < C::kHalf; e += 2) {
                                const uint32_t wd = Y[(63 - e) >> 1];
                                const float2 r2 = __ffma2_rn(
                                    make_float2(__uint_as_float(wd & 0xFFFF0000u), __uint_as_float(wd << 16)),
                                    c2, make_float2(x[e], x[e + 1]));
                                x[e] = r2.x;
                                x[e + 1] = r2.y;
                            }
                        } else {
                            // scales too extreme for the factor: unfold
#pragma unroll
                            for (int e = 0; e < C::kHalf; ++e) {
                                const uint32_t wd = Y[(63 - e) >> 1];
                                const float bv = __uint_as_float(((63 - e) & 1) ? (wd & 0xFFFF0000u)
                                                                                 : (wd << 16));
                                x[e] = fmaf(bv, kLog2eP, x[e] * p.score_log2);
                            }
                            mult = 1.0f;
                        }
                    }
                    if (!full_half) {
                        // key e of the half sits at distance d0 - e from this
                        // row: visible for e in [e_lo, e_hi] (causal, window,
                        // sequence end)
                        const int32_t keys_left = static_cast<int32_t>(
                            it.len_k - kh < C::kHalf ? it.len_k - kh : C::kHalf);
                        const int32_t e_hi = min(d0, keys_left - 1);
                        const int32_t e_lo = p.window > 0 ? max(0, d0 - p.window + 1) : 0;
#pragma unroll
                        for (int e = 0; e < C::kHalf; ++e)
                            x[e] = (e >= e_lo && e <= e_hi) ? x[e] : -INFINITY;
                    }
                    float mx = -INFINITY, m2 = -INFINITY;
#pragma unroll
                    for (int e = 0; e < C::kHalf; e += 4) {
                        mx = fmax3(mx, x[e], x[e + 1]);
                        m2 = fmax3(m2, x[e + 2], x[e + 3]);
                    }
                    mx = fmaxf(mx, m2) * mult;
                    // lazy rescale: a row must move its reference max when
                    // its max grew by more than tau (P <= 2^(8 + tau) stays
                    // below 448).  O is rescaled a whole warp at a time, so
                    // once any row of the warp needs it, every row whose max
                    // grew moves too.
                    const bool resc = mx > m_used + kRescaleTau2;
                    const bool rescale_o = __any_sync(0xffffffffu, resc && m_used != -INFINITY);
                    const bool move = resc || (rescale_o && mx > m_used);
                    const float m_new = move ? mx : m_used;
                    const float alpha =
                        (move && m_used != -INFINITY) ? ex2_fast(m_used - m_new) : 1.0f;
                    lsum = __fmul2_rn(lsum, make_float2(alpha, alpha));
                    err_bound *= alpha * alpha;
                    m_used = m_new;
                    const float neg_m8 = (m_used == -INFINITY) ? 0.0f : kPOffset2 - m_used;
                    // P = 2^(x * mult - m8) of the half, kept in x
                    float2 lu = make_float2(0.0f, 0.0f);
                    {
                        const float2 mult2 = make_float2(mult, mult), off2 = make_float2(neg_m8, neg_m8);
#pragma unroll
                        for (int e = 0; e < C::kHalf; e += 2) {
                            const float2 z = __ffma2_rn(make_float2(x[e], x[e + 1]), mult2, off2);
                            x[e] = ex2_fast(z.x);
                            x[e + 1] = ex2_fast(z.y);
                            if constexpr (kPT)   // the row sum takes P / v_scale
                                lu = __ffma2_rn(make_float2(x[e], x[e + 1]),
                                                make_float2(ktab[2 * kTile + e], ktab[2 * kTile + e + 1]), lu);
                            else
                                lu = __fadd2_rn(lu, make_float2(x[e], x[e + 1]));
                        }
                    }
                    lsum = __fadd2_rn(lsum, lu);
                    // One e4m3 term for this half's P when the row's bound
                    // stays within the budget; the warp takes two terms if
                    // any of its rows needs them (sum p^2 <= p_max * l_half).
                    const float l_row = lsum.x + lsum.y;
                    const float s2 = ex2_fast(mx + neg_m8) * (lu.x + lu.y);
                    // (the per-token variant always takes two terms)
                    const bool two =
                        kPT || __any_sync(0xffffffffu, err_bound + s2 > kPBudget * l_row * l_row);
                    if (!two) err_bound += s2;
                    // P over the half's own S columns (read above): P_hi in
                    // the first 16 columns, P_lo (or zeros, when another warp
                    // makes the PV take the second term) in the next 16
                    {
                        uint32_t w[16];
#pragma unroll
                        for (int q = 0; q < C::kHalf / 16; ++q) {
                            const uint4 hi = p_hi16(x + q * 16);
                            w[4 * q] = hi.x;
                            w[4 * q + 1] = hi.y;
                            w[4 * q + 2] = hi.z;
                            w[4 * q + 3] = hi.w;
                        }
                        const uint32_t pcol = tmem + lane_base + col_s + hh * C::kHalf;
                        tmem_st_x16_nowait(pcol, w);
                        uint32_t wl[16];
                        if (two) {
#pragma unroll
                            for (int q = 0; q < C::kHalf / 16; ++q) {
                                const uint4 lo = p_lo16(x + q * 16, make_uint4(w[4 * q], w[4 * q + 1],
                                                                               w[4 * q + 2], w[4 * q + 3]));
                                wl[4 * q] = lo.x;
                                wl[4 * q + 1] = lo.y;
                                wl[4 * q + 2] = lo.z;
                                wl[4 * q + 3] = lo.w;
                            }
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; ++q) wl[q] = 0u;
                        }
                        tmem_st_x16_nowait(pcol + 16, wl);
                    }
                    if (lane == 0) lo_flag(k, hh)[wq] = two ? 1 : 0;
                    if (rescale_o) {
                        // O holds the products up to unit u - 1 against the
                        // old reference: scale it by alpha once the PV of unit
                        // u - 1 (the other half) is done, before this unit's
                        // PV is issued.  Done after P so that the PV has had
                        // the whole P phase to finish.
                        if (!warp_wait_p(o_done(k, hh ^ 1), ((u - 1) >> 1) & 1, fail, p.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
                        for (int q = 0; q < D / 64; ++q) {
                            float o[64];
                            tmem_ld_x64(tmem + lane_base + col_o + q * 64, o);
#pragma unroll
                            for (int e = 0; e < 64; e += 2) {
                                const float2 s2 = __fmul2_rn(make_float2(o[e], o[e + 1]), a2);
                                o[e] = s2.x;
                                o[e + 1] = s2.y;
                            }
                            tmem_st_x64(tmem + lane_base + col_o + q * 64, o);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(p_full(k, hh));
                }
                if (ok) ++c;
            }
            have_prev = ok;
            prev_tok = tok0;
            prev_rows = it.n_rows;
            prev_h = it.h;
            prev_l = lsum;
        }
        if (ok && have_prev) epilogue();
        // a copy still in flight (the loop ended early) lands before the CTA ends
        if (!kPT && q_pending) {
            if (lane == 0) mbar_drain_p(qbar(k, wq), (q_copies - 1) & 1, p.err);
            __syncwarp();
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// The register split relies on the kernel being launched with kRegsLaunch
// registers per thread: with fewer, setmaxnreg.inc would wait for registers
// that do not exist.  Checked once per process against the built kernel.
template <bool kPT, bool kUnfold>
bool prefill2_registers_ok() {
    static int ok = -1;
    if (ok < 0) {
        cudaFuncAttributes attr;
        ok = (cudaFuncGetAttributes(&attr, prefill2_kernel<kPT, kUnfold>) == cudaSuccess &&
              attr.numRegs >= kRegsLaunch && attr.maxThreadsPerBlock >= kPre2Threads)
                 ? 1
                 : 0;
        if (!ok) cudaGetLastError();
    }
    return ok == 1;
}

// CTAs of a persistent launch at most (0: one per SM).
std::atomic<int> g_prefill_max_ctas{0};

template <bool kPT, bool kUnfold>
fp8kv_status launch_prefill2(const CUtensorMap &km, const CUtensorMap &vm, const CUtensorMap &qm,
                             const PrefillParams &p, int num_seqs, int sms, cudaStream_t stream) {
    const int cap = g_prefill_max_ctas.load(std::memory_order_relaxed);
    if (cap > 0 && cap < sms) sms = cap;
    auto kern = prefill2_kernel<kPT, kUnfold>;
    if (!prefill2_registers_ok<kPT, kUnfold>()) return FP8KV_ERR_UNSUPPORTED;
    static std::atomic<uint64_t> attrs_set{0};
    if (!func_attrs_once(reinterpret_cast<const void *>(kern), &attrs_set,
                         Pre2Cfg::kSmemBytes, false))
        return FP8KV_ERR_LAUNCH;
    // persistent: two pipelines per CTA, at most one CTA per SM
    const int64_t n_pairs = (p.n_qtiles + 1) / 2;
    const int64_t n_items = n_pairs * p.Hq * num_seqs;
    const dim3 grid = p.persist ? dim3(static_cast<unsigned>(n_items < sms ? n_items : sms))
                                : dim3(static_cast<unsigned>(n_pairs), p.Hq, num_seqs);
    kern<<<grid, kPre2Threads, Pre2Cfg::kSmemBytes, stream>>>(km, vm, qm, p);
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}

template <int D>
fp8kv_status launch_prefill(const CUtensorMap &km, const CUtensorMap &vm, const PrefillParams &p,
                            int num_seqs, cudaStream_t stream) {
    using C = PreCfg<D>;
    auto kern = prefill_kernel<D>;
    static std::atomic<uint64_t> attrs_set{0};
    if (!func_attrs_once(reinterpret_cast<const void *>(kern), &attrs_set, C::kSmemBytes, false))
        return FP8KV_ERR_LAUNCH;
    dim3 grid(p.n_qtiles, p.Hq, num_seqs);
    kern<<<grid, kPreThreads, C::kSmemBytes, stream>>>(km, vm, p);
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}

}  // namespace
}  // namespace fp8kv

using namespace fp8kv;

namespace {
// k_scales / v_scales non-null: the per-token variant (k_scale = v_scale = 1).
fp8kv_status prefill_impl(const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads,
                          const int32_t *cu_seqlens_q, const int32_t *seq_lens_k,
                          const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_seqs,
                          int32_t max_seqlen_q, float q_scale, float k_scale, float v_scale,
                          float softmax_scale, const float *k_scales, const float *v_scales,
                          const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride, int32_t rel_extent,
                          int32_t window, fp8kv_bf16 *out, void *stream) {
    const bool per_token = k_scales != nullptr;
    if (!cache || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || window < 0 ||
        max_seqlen_q < 0)
        return FP8KV_ERR_ARG;
    if (!scale_ok(q_scale) || !scale_ok(k_scale) || !scale_ok(v_scale) || !scale_ok(softmax_scale))
        return FP8KV_ERR_SCALE;
    const int D = cache->head_dim, bs = cache->block_size, Hkv = cache->num_kv_heads;
    if (Hkv <= 0 || cache->num_blocks < 0 || num_q_heads % Hkv != 0) return FP8KV_ERR_ARG;
    if ((D != 128 && D != 256) || (bs != 16 && bs != 32 && bs != 64 && bs != 128) ||
        num_seqs > 65535 || num_q_heads > 65535 || cache->num_blocks >= (1ll << 31) ||
        static_cast<int64_t>(max_blocks_per_seq) * bs > (1ll << 31) - 256)   // int32 positions
        return FP8KV_ERR_UNSUPPORTED;
    if (rel_bias && (rel_extent <= 0 || bias_tok_stride < 0)) return FP8KV_ERR_ARG;
    if (num_seqs == 0 || max_seqlen_q == 0) return FP8KV_OK;
    if (!q || !cu_seqlens_q || !seq_lens_k || !block_table || !out || !cache->k || !cache->v)
        return FP8KV_ERR_ARG;
    if (per_token && (D != 128 || !v_scales || (reinterpret_cast<uintptr_t>(k_scales) & 3) ||
                      (reinterpret_cast<uintptr_t>(v_scales) & 3)))
        return D != 128 ? FP8KV_ERR_UNSUPPORTED : FP8KV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(out) & 15) ||
        (reinterpret_cast<uintptr_t>(cache->k) & 15) || (reinterpret_cast<uintptr_t>(cache->v) & 15))
        return FP8KV_ERR_ARG;
    int sms = 0;
    fp8kv_status st = check_device(&sms);
    if (st != FP8KV_OK) return st;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, cache->k, cache->num_blocks, bs, Hkv, D) ||
        !make_cache_map(&vm, cache->v, cache->num_blocks, bs, Hkv, D))
        return FP8KV_ERR_LAUNCH;
    PrefillParams p;
    p.q = q;
    p.cu_q = cu_seqlens_q;
    p.lens_k = seq_lens_k;
    p.block_table = block_table;
    p.rel = rel_bias;
    p.out = out;
    p.err = device_error_word();
    p.bias_tok_stride = bias_tok_stride;
    p.num_blocks = cache->num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.Hq = num_q_heads;
    p.G = num_q_heads / Hkv;
    p.block_size = bs;
    p.bs_shift = __builtin_ctz(static_cast<unsigned>(bs));
    p.rel_extent = rel_bias ? rel_extent : 0;
    p.bias_vec = rel_bias && (reinterpret_cast<uintptr_t>(rel_bias) & 15) == 0 &&
                 bias_tok_stride % 8 == 0 && rel_extent % 8 == 0;
    p.window = window;
    p.num_seqs = num_seqs;
    p.n_qtiles = (max_seqlen_q + kTile - 1) / kTile;
    // the persistent schedule counts list positions in int32
    p.persist = D == 128 && num_seqs <= kPre2SchedSeqs && sms > 0 &&
                static_cast<int64_t>(p.n_qtiles) * num_seqs * num_q_heads < (1ll << 30);
    p.q_scale = make_qscale(q_scale);
    p.score_log2 = static_cast<float>(static_cast<double>(softmax_scale) * q_scale * k_scale *
                                      1.4426950408889634);
    p.v_scale = v_scale;
    {
        const double c = 1.0 / (static_cast<double>(softmax_scale) * q_scale * k_scale);
        p.bias_fold = (c < 0x1p60 && c > 0x1p-60) ? static_cast<float>(c) : 0.0f;
    }
    p.k_tok_scale = k_scales;
    p.v_tok_scale = v_scales;
    p.num_kv_heads = Hkv;
    // Q rows by tensor map (head_dim-128 kernel without per-token tables):
    // rows are bounded by num_seqs * max_seqlen_q, and a warp copies only
    // rows of its item's own queries
    CUtensorMap qm = km;
    p.q_tma = !per_token && D == 128 &&
              make_rows_map(&qm, q, static_cast<int64_t>(num_seqs) * max_seqlen_q, num_q_heads, D);
    if (!p.q_tma) qm = km;   // unused
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (per_token) return launch_prefill2<true, false>(km, vm, qm, p, num_seqs, sms, s);
    if (D != 128) return launch_prefill<256>(km, vm, p, num_seqs, s);
    const bool unfold = p.rel_extent > 0 && !(p.bias_fold > 0.0f);
    return unfold ? launch_prefill2<false, true>(km, vm, qm, p, num_seqs, sms, s)
                  : launch_prefill2<false, false>(km, vm, qm, p, num_seqs, sms, s);
}
}  // namespace

extern "C" fp8kv_status attn_fp8_varlen_prefill(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads,
    const int32_t *cu_seqlens_q, const int32_t *seq_lens_k, const int32_t *block_table,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t max_seqlen_q, float q_scale,
    float k_scale, float v_scale, float softmax_scale, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *workspace,
    size_t workspace_bytes, void *stream) {
    (void)workspace;
    (void)workspace_bytes;
    return prefill_impl(cache, q, num_q_heads, cu_seqlens_q, seq_lens_k, block_table,
                        max_blocks_per_seq, num_seqs, max_seqlen_q, q_scale, k_scale, v_scale,
                        softmax_scale, nullptr, nullptr, rel_bias, bias_tok_stride, rel_extent,
                        window, out, stream);
}

extern "C" fp8kv_status attn_fp8_varlen_prefill_per_token(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads,
    const int32_t *cu_seqlens_q, const int32_t *seq_lens_k, const int32_t *block_table,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t max_seqlen_q, float q_scale,
    float softmax_scale, const float *k_scales, const float *v_scales, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *stream) {
    if (num_seqs > 0 && max_seqlen_q > 0 && (!k_scales || !v_scales)) return FP8KV_ERR_ARG;
    // the per-token scales replace k_scale and v_scale (1 in the fold and the epilogue)
    return prefill_impl(cache, q, num_q_heads, cu_seqlens_q, seq_lens_k, block_table,
                        max_blocks_per_seq, num_seqs, max_seqlen_q, q_scale, 1.0f, 1.0f,
                        softmax_scale, k_scales ? k_scales : nullptr, v_scales, rel_bias,
                        bias_tok_stride, rel_extent, window, out, stream);
}


extern "C" fp8kv_status fp8kv_set_prefill_max_ctas(int32_t max_ctas) {
    if (max_ctas < 0) return FP8KV_ERR_ARG;
    g_prefill_max_ctas.store(max_ctas, std::memory_order_relaxed);
    return FP8KV_OK;
}
