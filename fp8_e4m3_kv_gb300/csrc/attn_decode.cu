// attn_decode.cu -- split-KV paged decode attention over the e4m3 cache
// (vLLM PR 54705 "Purpose": query quantization, descale fold into the
// softmax scale before the exact bf16 relative bias, v_scale post-multiply;
// full-causal or sliding-window layers).
//
// One CTA handles one (split of the key range, KV head, sequence) and all
// query heads of that KV head (the GQA group, padded to 16).  Keys stream in
// tiles of 128:
//   producer warp   TMA-loads the K and V tiles of the split's blocks (one box
//                   of block_size rows x 128 bytes per block and 128-byte
//                   column) into a ring of stages;
//   MMA warp        one thread issues the tcgen05 FP8 MMAs:
//                     S^T[key][head] = K_tile . Q8^T              (M=128, N=16)
//                     O^T[d][n]     = V_tile^T . P^T        (M=128, N=2*GMAX)
//                   into TMEM (S^T double-, O^T triple-buffered), where the
//                   rows n of P hold both e4m3 terms of every head (P_hi
//                   and P_lo of a warpgroup's heads side by side), so the
//                   PV takes as many MMAs as one term of P would;
//   consumer        thread t owns key row t of S^T and value row d = t of
//   warpgroups      O^T; warpgroup hs takes its share of the query heads:
//                   folded descale, bias, mask, block-wide max per head
//                   (warp shuffles and a 4-warp exchange), P, and O
//                   accumulated in registers with the online rescale, two
//                   tiles behind the MMAs.
// The per-tile chain is latency-bound; splitting the heads over warpgroups
// halves each thread's serial work.  P is exp2(z - m + 8) (at most 256) split
// into two e4m3 terms, P_hi = e4m3(P) and P_lo = e4m3(P - P_hi), so the PV
// product runs on the FP8 tensor cores while the weights keep ~8 significant
// bits (the consumers add the two terms' columns of O^T).  The partial
// (o, m, l) of each split goes to the workspace; a second
// kernel merges the splits with the log-sum-exp rule and writes
// v_scale * o / l in bf16.
#include <math.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace fp8kv {
namespace {

constexpr int kNPad = 16;          // query heads per KV head, padded to the MMA N
constexpr float kMinLog2VScale = -60.0f;   // per-token V scales folded into exponents
constexpr float kLog2e = 1.4426950408889634f;

// Consumer warpgroups, pipeline depth, keys per tile and resident CTAs per SM
// (tuning knobs, fixed at build time).
#ifndef FP8KV_DECODE_HS
#define FP8KV_DECODE_HS 2
#endif
#ifndef FP8KV_DECODE_STAGES_D128
#define FP8KV_DECODE_STAGES_D128 3
#endif
#ifndef FP8KV_DECODE_CTAS_D128
#define FP8KV_DECODE_CTAS_D128 2
#endif
#ifndef FP8KV_DECODE_KEYS_D128
#define FP8KV_DECODE_KEYS_D128 128
#endif
#ifndef FP8KV_DECODE_STAGES_D256
#define FP8KV_DECODE_STAGES_D256 3
#endif

template <int D>
struct DecCfg {
    static constexpr int kCB = D / 128;               // 128-byte column blocks per row
    // consumer warpgroups; warpgroup hs owns query heads [hs*GH, (hs+1)*GH) of
    // the group, GH = GMAX / kHS, for every key of the tile
    static constexpr int kHS = FP8KV_DECODE_HS;
    static constexpr int kStages = D == 128 ? FP8KV_DECODE_STAGES_D128 : FP8KV_DECODE_STAGES_D256;
    static constexpr int kCtasPerSm = D == 128 ? FP8KV_DECODE_CTAS_D128 : 1;
    static constexpr int kConsumers = kHS * 128;
    static constexpr int kThreads = kConsumers + 64;
    static constexpr int kProducerWarp = kHS * 4;
    static constexpr int kMmaWarp = kHS * 4 + 1;
    // keys per tile (a multiple of 128: one QK MMA with M = 128 per 128 keys)
    static constexpr int kKeys = D == 128 ? FP8KV_DECODE_KEYS_D128 : 128;
    static constexpr int kKB = kKeys / 128;           // 128-key sub-tiles (QK MMAs, M = 128)
    static constexpr int kCBBytes = kKeys * 128;      // one 128-byte column block of a tile
    static constexpr int kTileBytes = kKeys * D;      // one K (or V) tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kQBytes = kNPad * D;         // Q8: 16 rows x D bytes
    static constexpr int kPBytes = kNPad * kKeys;     // one P term: 16 rows x kKeys keys
    // P of one tile: per 128-key column block, up to 32 rows of 128 bytes
    // (both terms of up to 16 heads), 128-byte swizzled
    static constexpr int kPBlock = 2 * kNPad * 128;
    // P and O^T buffers: a tile's O^T is read back two tiles later, so the
    // PV latency stays off the softmax chain
    static constexpr int kOBuf = 3;
    static constexpr int kOffQ = kStages * kStageBytes;
    static constexpr int kOffP = kOffQ + kQBytes;     // [kOBuf][kKB][P rows]
    static constexpr int kOffMisc = kOffP + kOBuf * 2 * kPBytes;
    // misc: barriers, tmem slot, abort flag, then per warpgroup the tile-max
    // exchange [2][4][16] and row-sum exchange [4][16] floats
    static constexpr int kOffRed = 512;
    static constexpr int kMiscBytes = kOffRed + kHS * 768;
    static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;   // + alignment slack
    // TMEM: S^T 2 buffers x kKB x 16 columns, then O^T kOBuf buffers x kCB x
    // np columns (np = rows of P: 16 for up to 8 heads, 32 for 16)
    static constexpr uint32_t kColO = 2 * kKB * kNPad;
    __host__ __device__ static constexpr uint32_t cols(int np) { return kColO + kOBuf * kCB * np + kNPad; }   // + over-read room
    __host__ __device__ static constexpr uint32_t tmem_cols(int np) {
        return cols(np) <= 64 ? 64 : cols(np) <= 128 ? 128 : 256;
    }
    static_assert(cols(2 * kNPad) <= 256, "TMEM columns");
    static_assert(kStages >= 2 && kStages <= 8, "stages");
    static_assert(kHS >= 1 && kHS <= 4, "head split");
};

struct DecodeParams {
    const uint16_t *q;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const uint16_t *rel;
    float *part_o;          // [B][Hq][S][D]
    float *part_ml;         // [B][Hq][S][2]  (running max in log2 units, sum)
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
    int32_t split_tiles;
    // the first fine_splits splits of a sequence (in key order) take
    // fine_tiles tiles each, the rest split_tiles (fine_splits 0: all equal)
    int32_t fine_splits;
    int32_t fine_tiles;
    int32_t num_slots;      // partial slots per (sequence, head) = splits
    QScale q_scale;
    float score_log2;       // softmax_scale * q_scale * k_scale * log2(e)
    // fused store of the step's new token (k_new == nullptr: none): row
    // [b][kv head][D] of k_new / v_new goes to the cache slot of position
    // seq_len - 1, quantized exactly as kv_store_e4m3 does
    const uint16_t *k_new;
    const uint16_t *v_new;
    uint8_t *cache_k;
    uint8_t *cache_v;
    float *amax_k;          // nullable: running max |k_new|
    float *amax_v;
    int32_t num_kv_heads;
    QScale k_scale;
    QScale v_scale;
    // per-token scales (the per-token variant of the kernel only):
    // float[num_blocks][num_kv_heads][block_size], one per cached token and head
    const float *k_tok_scale;
    const float *v_tok_scale;
    // test hook (fp8kv_test_drop_first_copy): the producer issues neither
    // the copy nor the expected-bytes arrival of its first key tile, so the
    // MMA warp's wait for that tile runs out
    int32_t drop_first_copy;
    // one split per (sequence, KV head): the decode kernel writes
    // out = bf16(v_scale * o / l) itself, the merge's arithmetic for one split
    uint16_t *out;
    float out_scale;    // v_scale (1 for per-token scales)
    int32_t direct_out;
    // work items: num_kv_heads x num_seqs x num_slots, taken in order from
    // the counter *sched (zero at launch); sched == nullptr: one CTA per
    // item, CTA c takes item c
    uint32_t *sched;
    int32_t num_items;
    int32_t num_seqs;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Bounded wait that ignores the CTA's abort flag: used only in the teardown
// to let copies and MMAs that are already in flight finish.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, uint32_t *err) {
    CtaFail never{0};
    mbar_wait(bar, parity, &never, err);
}

// Every lane of the warp waits on the barrier (each thread then observes the
// phase), and the warp agrees on the outcome, so that the .sync.aligned
// tcgen05 loads that follow never run diverged.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, CtaFail *fail,
                                          uint32_t *err) {
    const bool ok = mbar_wait(bar, parity, fail, err);
    return __all_sync(0xffffffffu, ok);
}

// Eight bf16 values -> eight e4m3 bytes, as the store quantizes them (the
// multiply and the divide give the same IEEE quotient for a power-of-two
// scale, so either branch is bit-exact).
__device__ __forceinline__ uint2 store_quantize8(const uint4 w, const QScale &s) {
    uint2 r;
    if (s.pow2) {
        r.x = quantize_bf16x2_as<true>(w.x, s) | (quantize_bf16x2_as<true>(w.y, s) << 16);
        r.y = quantize_bf16x2_as<true>(w.z, s) | (quantize_bf16x2_as<true>(w.w, s) << 16);
    } else {
        r.x = quantize_bf16x2_as<false>(w.x, s) | (quantize_bf16x2_as<false>(w.y, s) << 16);
        r.y = quantize_bf16x2_as<false>(w.z, s) | (quantize_bf16x2_as<false>(w.w, s) << 16);
    }
    return r;
}

__device__ __forceinline__ float absmax8(const uint4 w) {
    // fmaxf ignores NaN operands, so NaN elements never win
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(a[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(a[i] & 0xFFFF0000u)));
    }
    return m;
}

// Q8 = e4m3(q / q_scale) for one KV head's group of query heads (rows >= G
// zero), 128-byte swizzled K-major (row = head, D bytes per row), written by
// kThreads threads with 8 elements each per step.  The scale's form is a
// template argument so that only one of multiply / divide is evaluated.
template <bool kPow2, int D, int kThreads>
__device__ __forceinline__ void load_q8(uint8_t *q8, const uint16_t *q_group, int G,
                                        const QScale &s) {
    for (int e = threadIdx.x * 8; e < kNPad * D; e += kThreads * 8) {
        const int g = e / D, d = e % D;
        uint2 packed = make_uint2(0u, 0u);
        if (g < G) {
            const uint4 w = *reinterpret_cast<const uint4 *>(q_group + static_cast<int64_t>(g) * D + d);
            packed.x = quantize_q_bf16x2<kPow2>(w.x, s) | (quantize_q_bf16x2<kPow2>(w.y, s) << 16);
            packed.y = quantize_q_bf16x2<kPow2>(w.z, s) | (quantize_q_bf16x2<kPow2>(w.w, s) << 16);
        }
        *reinterpret_cast<uint2 *>(q8 + (d / 128) * (kNPad * 128) + sw128_offset(g, d % 128)) =
            packed;
    }
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One work item: a split of one (sequence, KV head); ntiles < 0 ends the
// list.
struct DecItem {
    int32_t b, kvh, split, ntiles;
};
constexpr int kItemSlots = 4;   // item records in flight between the roles

// The key range of split `split` of sequence b: keys [lo, len) (the window's
// keys for a sliding-window layer) in tiles of kKeys, this split's tiles
// [t0, t0 + ntiles) (ntiles <= 0: none).
struct ItemGeom {
    int64_t len, lo, t0, t_end;
    int ntiles;
};

template <int kKeys>
__device__ __forceinline__ ItemGeom item_geom(const DecodeParams &p, int b, int split) {
    ItemGeom g;
    g.len = p.seq_lens[b];
    g.lo = (p.window > 0 && g.len > p.window) ? g.len - p.window : 0;
    int64_t off, n;
    if (split < p.fine_splits) {
        off = static_cast<int64_t>(split) * p.fine_tiles;
        n = p.fine_tiles;
    } else {
        off = static_cast<int64_t>(p.fine_splits) * p.fine_tiles +
              static_cast<int64_t>(split - p.fine_splits) * p.split_tiles;
        n = p.split_tiles;
    }
    g.t0 = g.lo / kKeys + off;
    g.t_end = (g.len + kKeys - 1) / kKeys;
    g.ntiles = static_cast<int>(g.t_end - g.t0 < n ? g.t_end - g.t0 : n);
    return g;
}

// kPT: per-token scales.  Key j's score is multiplied by its K scale, and
// its V scale is folded into the exponent: z_j + log2(v_scale_j) takes part
// in the block-wide max like any score, so P_j = 2^(z_j + log2 v_scale_j -
// m + 8) <= 2^8 is p_j * v_scale_j (up to the common factor) and the row
// sum adds P_j / v_scale_j.
//
// The launch is persistent: up to kCtasPerSm CTAs per SM, each taking work
// items from a counter in global memory until none is left.  Items are
// numbered KV heads fastest, then sequences, then splits in descending
// order (the first splits, full-length ones, come last and fill the tail).
// The producer warp takes the items, marks the empty ones itself and hands
// the others to the MMA thread and the consumers through a ring of item
// records in shared memory; it loads each item's key tiles right after the
// previous item's, so the pipeline does not drain between items, and the
// consumers quantize the next item's Q while the last P of an item is
// multiplied.
template <int D, int GMAX, bool kPT>
__global__ void __launch_bounds__(DecCfg<D>::kThreads, DecCfg<D>::kCtasPerSm)
decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const DecodeParams p) {
    using C = DecCfg<D>;
    constexpr int HS = C::kHS;
    constexpr int GH = GMAX / HS;                      // heads per consumer warpgroup
    static_assert(GH * HS == GMAX && GH % 2 == 0, "head split: an even number of heads per warpgroup");
    // rows of P (= the PV's N): warpgroup hs writes P_hi of its head g in row
    // hs * 2GH + g and P_lo in row hs * 2GH + GH + g
    constexpr int NP = 2 * GMAX < 16 ? 16 : 2 * GMAX;
    static_assert(NP % 16 == 0 && NP <= 2 * kNPad && 2 * GH <= 16, "P rows");
    constexpr uint32_t kTmemCols = C::tmem_cols(NP);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffMisc);
    uint64_t *full = bars;          // [kStages] TMA landed
    uint64_t *empty = bars + 8;     // [kStages] stage consumed (PV committed)
    uint64_t *s_full = bars + 16;   // [2] S^T in TMEM
    uint64_t *s_free = bars + 18;   // [2] S^T read by all consumer warps
    uint64_t *p_full = bars + 20;   // [3] P in shared memory
    uint64_t *o_full = bars + 23;   // [3] O^T in TMEM
    uint64_t *o_free = bars + 26;   // [3] O^T read by all consumer warps
    uint64_t *mma_done = bars + 29; // teardown: all MMAs complete
    // per warpgroup hs: red_bar[2] at bars + 30 + 3*hs, l_bar at + 2
    uint64_t *q_full = bars + 42;      // Q8 of the next item written by every consumer warp
    uint64_t *item_full = bars + 43;   // [kItemSlots] item record written
    uint64_t *item_free = bars + 47;   // [kItemSlots] record read by the MMA thread and every consumer warp
    DecItem *items = reinterpret_cast<DecItem *>(smem + C::kOffMisc + 416);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffMisc + 480);
    CtaFail *fail = reinterpret_cast<CtaFail *>(smem + C::kOffMisc + 484);
    static_assert(30 + 3 * 4 <= 42 && (47 + kItemSlots) * 8 <= 416 &&
                      416 + kItemSlots * sizeof(DecItem) <= 480,
                  "barrier area");

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4 * HS);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(&p_full[i], 4 * HS);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_free[i], 4 * HS);
        }
        mbar_init(mma_done, 1);
        for (int hs = 0; hs < HS; ++hs) {
            mbar_init(bars + 30 + 3 * hs, 4);
            mbar_init(bars + 31 + 3 * hs, 4);
            mbar_init(bars + 32 + 3 * hs, 4);
        }
        mbar_init(q_full, 4 * HS);
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_free[i], 1 + 4 * HS);
        }
        fail->abort = 0;
        fence_mbar_init();
    }
    if (warp == C::kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
    if (warp == C::kProducerWarp) {
        // zero the P buffers: rows past the group are never written
        uint4 *pz = reinterpret_cast<uint4 *>(smem + C::kOffP);
        for (int i = lane; i < C::kOBuf * 2 * C::kPBytes / 16; i += 32) pz[i] = make_uint4(0, 0, 0, 0);
        if (lane == 0) {
            tma_prefetch_map(&kmap);
            tma_prefetch_map(&vmap);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // the merge launch that follows may be scheduled now: it waits for this
    // whole grid's completion (and its writes) before reading any partial
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == C::kProducerWarp) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = l2_policy_evict_first();
        const int nb = C::kKeys / p.block_size;   // blocks per tile (<= 16)
        int last_issued[C::kStages];
#pragma unroll
        for (int s = 0; s < C::kStages; ++s) last_issued[s] = -1;
        int T = 0;   // key tiles of this CTA so far
        int J = 0;   // item records written
        bool ok = true;
        bool fetched = false;
        while (ok) {
            int idx = 0;
            if (lane == 0)
                idx = p.sched ? static_cast<int>(atomicAdd(p.sched, 1u))
                              : (fetched ? p.num_items : static_cast<int>(blockIdx.x));
            idx = __shfl_sync(0xffffffffu, idx, 0);
            fetched = true;
            DecItem it{0, 0, 0, -1};
            ItemGeom gm{};
            if (idx < p.num_items) {
                const int kvh = idx % p.num_kv_heads;
                const int rest = idx / p.num_kv_heads;
                const int b = rest % p.num_seqs;
                const int split = p.num_slots - 1 - rest / p.num_seqs;
                gm = item_geom<C::kKeys>(p, b, split);
                if (gm.ntiles <= 0) {   // nothing to attend in this split: mark it empty
                    const int h0 = kvh * p.G;
                    if (p.direct_out) {   // the only split: the output is zero
                        for (int e = lane; e < p.G * D; e += 32)
                            p.out[(static_cast<int64_t>(b) * p.Hq + h0 + e / D) * D + e % D] = 0;
                    } else if (lane < p.G) {
                        float *ml = p.part_ml + ((static_cast<int64_t>(b) * p.Hq + h0 + lane) *
                                                     p.num_slots + split) * 2;
                        ml[0] = -INFINITY;
                        ml[1] = 0.0f;
                    }
                    continue;
                }
                it = DecItem{b, kvh, split, gm.ntiles};
            }
            const int slot = J % kItemSlots;
            int w = 1;
            if (lane == 0) w = mbar_wait(&item_free[slot], ((J / kItemSlots) & 1) ^ 1, fail, p.err);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            if (lane == 0) {
                items[slot] = it;
                mbar_arrive(&item_full[slot]);
            }
            ++J;
            if (it.ntiles < 0) break;
            if (p.k_new != nullptr && gm.len > 0 && gm.t0 + it.ntiles == gm.t_end) {
                // Fused store: this item holds the sequence's last tile, so the
                // warp writes the step's new token (position len - 1) for its
                // KV head before loading the tile; the proxy fence orders these
                // generic writes before the warp's TMA copies.
                const int64_t lb = (gm.len - 1) / p.block_size;
                const int32_t id =
                    lb < p.max_blocks
                        ? __ldg(p.block_table + static_cast<int64_t>(it.b) * p.max_blocks + lb)
                        : -1;
                if (id >= 0 && id < p.num_blocks) {
                    if (lane < D / 8) {
                        const int d = lane * 8;
                        const int64_t src = (static_cast<int64_t>(it.b) * p.num_kv_heads + it.kvh) * D + d;
                        const int64_t dst = ((static_cast<int64_t>(id) * p.num_kv_heads + it.kvh) *
                                                 p.block_size + (gm.len - 1) % p.block_size) * D + d;
                        const uint4 kw = *reinterpret_cast<const uint4 *>(p.k_new + src);
                        const uint4 vw = *reinterpret_cast<const uint4 *>(p.v_new + src);
                        *reinterpret_cast<uint2 *>(p.cache_k + dst) = store_quantize8(kw, p.k_scale);
                        *reinterpret_cast<uint2 *>(p.cache_v + dst) = store_quantize8(vw, p.v_scale);
                        // non-negative floats order like their bit patterns
                        if (p.amax_k)
                            atomicMax(reinterpret_cast<unsigned int *>(p.amax_k), __float_as_uint(absmax8(kw)));
                        if (p.amax_v)
                            atomicMax(reinterpret_cast<unsigned int *>(p.amax_v), __float_as_uint(absmax8(vw)));
                    }
                } else if (lane == 0) {
                    atomicOr(p.err, FP8KV_DEVERR_BAD_BLOCK);
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
            }
            for (int i = 0; i < it.ntiles; ++i, ++T) {
                const int s = T % C::kStages;
                int32_t phys = static_cast<int32_t>(p.num_blocks);   // out of range: zero fill
                if (lane < nb) {
                    const int64_t lb = (gm.t0 + i) * nb + lane;
                    if (lb * p.block_size < gm.len) {
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
                int okw = 1;
                if (lane == 0) okw = mbar_wait(&empty[s], ((T / C::kStages) & 1) ^ 1, fail, p.err);
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    ok = false;
                    break;
                }
                if (T == 0 && p.drop_first_copy) continue;
                if (lane == 0) mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                __syncwarp();
                if (lane < nb) {
                    uint8_t *kdst = smem + s * C::kStageBytes + lane * p.block_size * 128;
                    uint8_t *vdst = kdst + C::kTileBytes;
#pragma unroll
                    for (int cb = 0; cb < C::kCB; ++cb) {
                        tma_load_4d(kdst + cb * C::kCBBytes, &kmap, &full[s], cb * 128, 0, it.kvh, phys, pol);
                        tma_load_4d(vdst + cb * C::kCBBytes, &vmap, &full[s], cb * 128, 0, it.kvh, phys, pol);
                    }
                }
                last_issued[s] = T;
            }
        }
        if (lane == 0 && fail->abort) {   // let copies already issued land
            for (int s = 0; s < C::kStages; ++s)
                if (last_issued[s] >= 0) mbar_drain(&full[s], (last_issued[s] / C::kStages) & 1, p.err);
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Per item, step i issues QK of tile i, then PV of tile i - 1 (whose P
        // the consumers produced while QK of tile i was in flight).
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_e4m3_f32(128, kNPad, false, false);
            const uint32_t idesc_pv = idesc_e4m3_f32(128, NP, true, false);
            const uint32_t q_addr = smem_u32(smem + C::kOffQ);
            int T = 0, J = 0, A = 0;
            bool ok = true;
            while (ok) {
                const int slot = J % kItemSlots;
                if (!mbar_wait(&item_full[slot], (J / kItemSlots) & 1, fail, p.err)) break;
                const int ntiles = reinterpret_cast<volatile DecItem *>(items)[slot].ntiles;
                mbar_arrive(&item_free[slot]);
                ++J;
                if (ntiles < 0) break;
                if (!mbar_wait(q_full, A & 1, fail, p.err)) break;
                ++A;
                for (int i = 0; i <= ntiles; ++i) {
                    if (i < ntiles) {
                        const int TT = T + i;
                        const int s = TT % C::kStages, sb = TT & 1;
                        if (!mbar_wait(&full[s], (TT / C::kStages) & 1, fail, p.err) ||
                            !mbar_wait(&s_free[sb], ((TT >> 1) & 1) ^ 1, fail, p.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t k_addr = smem_u32(smem + s * C::kStageBytes);
#pragma unroll
                        for (int kb = 0; kb < C::kKB; ++kb) {
                            const uint32_t dcol = tmem + (sb * C::kKB + kb) * kNPad;
#pragma unroll
                            for (int kk = 0; kk < D / 32; ++kk) {
                                const uint32_t cb = kk / 4, ko = (kk % 4) * 32;
                                const uint64_t a = sdesc_sw128(
                                    k_addr + cb * C::kCBBytes + kb * (128 * 128) + ko, 16, 1024);
                                const uint64_t bd =
                                    sdesc_sw128(q_addr + cb * (kNPad * 128) + ko, 16, 1024);
                                mma_e4m3(dcol, a, bd, idesc_qk, kk > 0);
                            }
                        }
                        tc_commit(&s_full[sb]);
                    }
                    if (i >= 1) {
                        const int j = T + i - 1, s = j % C::kStages;
                        const int pb = j % C::kOBuf, ph = (j / C::kOBuf) & 1;
                        if (!mbar_wait(&p_full[pb], ph, fail, p.err) ||
                            !mbar_wait(&o_free[pb], ph ^ 1, fail, p.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t v_addr = smem_u32(smem + s * C::kStageBytes + C::kTileBytes);
                        const uint32_t p_addr = smem_u32(smem + C::kOffP + pb * 2 * C::kPBytes);
#pragma unroll
                        for (int mh = 0; mh < C::kCB; ++mh) {
                            const uint32_t dcol = tmem + C::kColO + (pb * C::kCB + mh) * NP;
#pragma unroll
                            for (int kk = 0; kk < C::kKeys / 32; ++kk) {
                                // V tile, MN-major: rows are keys (128 bytes of d
                                // each), 8-row groups 1024 bytes apart; 32 keys per
                                // MMA.  P: NP rows of 128 keys per column block.
                                const uint64_t a = sdesc_sw128(
                                    v_addr + mh * C::kCBBytes + kk * 32 * 128, C::kCBBytes, 1024);
                                const uint64_t bd = sdesc_sw128(
                                    p_addr + (kk / 4) * C::kPBlock + (kk % 4) * 32, 16, 1024);
                                mma_e4m3(dcol, a, bd, idesc_pv, kk != 0);
                            }
                        }
                        tc_commit(&o_full[pb]);
                        tc_commit(&empty[s]);
                    }
                }
                T += ntiles;
            }
            tc_commit(mma_done);
            mbar_drain(mma_done, 0, p.err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const int hs = warp >> 2, wq = warp & 3;            // warpgroup (head half), TMEM quadrant
        const int t = threadIdx.x & 127;                    // key row / value row
        const int gbase = hs * GH;                          // this warpgroup's first head
        uint64_t *red_bar = bars + 30 + 3 * hs, *l_bar = bars + 32 + 3 * hs;
        float *red = reinterpret_cast<float *>(smem + C::kOffMisc + C::kOffRed + hs * 768);  // [2][4][16]
        float *lred = red + 128;                                                          // [4][16]
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        int T = 0, J = 0, A = 0;
        bool ok = true;

        // the next item record (every lane reads it; lane 0 releases it)
        auto pop_item = [&](DecItem &it) -> bool {
            const int slot = J % kItemSlots;
            if (!warp_wait(&item_full[slot], (J / kItemSlots) & 1, fail, p.err)) return false;
            const volatile DecItem *r = reinterpret_cast<volatile DecItem *>(items) + slot;
            it.b = r->b;
            it.kvh = r->kvh;
            it.split = r->split;
            it.ntiles = r->ntiles;
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_free[slot]);
            ++J;
            return true;
        };
        // Q rows of an item's group (8 bf16 per thread and step; rows >= G
        // zero), then Q8 = e4m3(q / q_scale), 128-byte swizzled, K-major (row =
        // head, D bytes per row), handed to the MMA thread
        constexpr int kQV = kNPad * D / 8 / C::kConsumers;
        static_assert(kQV * 8 * C::kConsumers == kNPad * D, "Q split");
        uint4 qreg[kQV];
        auto load_q = [&](const DecItem &it) {
            const uint16_t *qb = p.q + (static_cast<int64_t>(it.b) * p.Hq + it.kvh * p.G) * D;
#pragma unroll
            for (int v = 0; v < kQV; ++v) {
                const int e = (threadIdx.x + v * C::kConsumers) * 8;
                const int g = e / D, d = e % D;
                qreg[v] = g < p.G ? *reinterpret_cast<const uint4 *>(qb + static_cast<int64_t>(g) * D + d)
                                  : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        auto store_q8 = [&]() {
            uint8_t *q8 = smem + C::kOffQ;
#pragma unroll
            for (int v = 0; v < kQV; ++v) {
                const int e = (threadIdx.x + v * C::kConsumers) * 8;
                const int g = e / D, d = e % D;
                const uint4 w = qreg[v];
                uint2 packed;
                if (p.q_scale.pow2) {
                    packed.x = quantize_q_bf16x2<true>(w.x, p.q_scale) | (quantize_q_bf16x2<true>(w.y, p.q_scale) << 16);
                    packed.y = quantize_q_bf16x2<true>(w.z, p.q_scale) | (quantize_q_bf16x2<true>(w.w, p.q_scale) << 16);
                } else {
                    packed.x = quantize_q_bf16x2<false>(w.x, p.q_scale) | (quantize_q_bf16x2<false>(w.y, p.q_scale) << 16);
                    packed.y = quantize_q_bf16x2<false>(w.z, p.q_scale) | (quantize_q_bf16x2<false>(w.w, p.q_scale) << 16);
                }
                *reinterpret_cast<uint2 *>(q8 + (d / 128) * (kNPad * 128) + sw128_offset(g, d % 128)) = packed;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        };

        DecItem it{0, 0, 0, -1};
        ok = pop_item(it);
        if (ok && it.ntiles > 0) {
            load_q(it);
            store_q8();
        }
        while (ok && it.ntiles > 0) {
            const int ntiles = it.ntiles;
            const ItemGeom gm = item_geom<C::kKeys>(p, it.b, it.split);
            // positions fit in int32 (the host bounds the block table's keys)
            const int32_t len = static_cast<int32_t>(gm.len), lo = static_cast<int32_t>(gm.lo),
                          t0 = static_cast<int32_t>(gm.t0);
            const int b = it.b, split = it.split, h0 = it.kvh * p.G;
            const uint16_t *bias = p.rel ? p.rel + static_cast<int64_t>(b) * p.bias_tok_stride +
                                               static_cast<int64_t>(h0 + gbase) * p.rel_extent
                                         : nullptr;

            // rescale factors of the two previous tiles (a tile's O^T is taken two
            // tiles later): alpha_1 of tile j - 1, alpha_2 of tile j - 2
            float m_run[GH], l_part[GH], alpha_1[GH], alpha_2[GH], o_acc[C::kCB][GH];
#pragma unroll
            for (int g = 0; g < GH; ++g) {
                m_run[g] = -INFINITY;
                l_part[g] = 0.0f;
                alpha_1[g] = alpha_2[g] = 1.0f;
#pragma unroll
                for (int mh = 0; mh < C::kCB; ++mh) o_acc[mh][g] = 0.0f;
            }
            // Accumulate this warpgroup's heads of O^T of the CTA's tile j
            // (rescaled) into the registers.
            auto take_o = [&](int j, const float *alpha) -> bool {
                const int ob = j % C::kOBuf;
                if (!warp_wait(&o_full[ob], (j / C::kOBuf) & 1, fail, p.err)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int mh = 0; mh < C::kCB; ++mh) {
                    // this warpgroup's columns: the P_hi product of head g in
                    // o[g], the P_lo product in o[GH + g]
                    float o[16];
                    tmem_ld_x16(tmem + lane_base + C::kColO + (ob * C::kCB + mh) * NP + 2 * gbase, o);
#pragma unroll
                    for (int g = 0; g < GH; ++g)
                        o_acc[mh][g] = fmaf(o_acc[mh][g], alpha[g], o[g] + o[GH + g]);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_free[ob]);
                return true;
            };

            // kPT: the raw scales of this thread's keys of tile i (ksc, vsc),
            // loaded a tile ahead so that their latency stays off the chain
            float ksc[C::kKB], vsc[C::kKB];
            auto load_scales = [&](int i) {
#pragma unroll
                for (int kb = 0; kb < C::kKB; ++kb) {
                    const int32_t key = (t0 + i) * C::kKeys + kb * 128 + t;
                    const int32_t lb = key >> p.bs_shift;
                    ksc[kb] = 1.0f;
                    vsc[kb] = 0.0f;   // marks a key that is not visible
                    if (i < ntiles && key < len && key >= lo && lb < p.max_blocks) {
                        const int32_t id =
                            __ldg(p.block_table + static_cast<int64_t>(b) * p.max_blocks + lb);
                        if (id >= 0 && id < p.num_blocks) {
                            const int64_t si = (static_cast<int64_t>(id) * p.num_kv_heads + it.kvh) *
                                                   p.block_size + (key & (p.block_size - 1));
                            ksc[kb] = __ldg(p.k_tok_scale + si);
                            vsc[kb] = __ldg(p.v_tok_scale + si);
                        }
                    }
                }
            };
            if constexpr (kPT) load_scales(0);
            DecItem nx{0, 0, 0, -1};
            for (int i = 0; i < ntiles; ++i) {
                const int TT = T + i;
                if (i == ntiles - 1) {
                    // the next item: its record and its Q rows, in flight
                    // during this tile
                    if (!pop_item(nx)) { ok = false; break; }
                    if (nx.ntiles > 0) load_q(nx);
                }
                // per-token factors of this thread's keys: K scale, log2 and
                // reciprocal of the V scale (1, 0, 0 where not visible; the
                // score of such a key is -inf anyway)
                float tsk[C::kKB], tlv[C::kKB], tiv[C::kKB];
                if constexpr (kPT) {
#pragma unroll
                    for (int kb = 0; kb < C::kKB; ++kb) {
                        const float sv = vsc[kb];
                        // the hardware log2 and reciprocal: their ~2^-22 relative
                        // errors move a key's weight by ~1e-5 of itself, far
                        // below the e4m3 rounding of P
                        const float lv = __log2f(sv);
                        tsk[kb] = ksc[kb];
                        // below 2^-60 the exponent takes 2^-60 (and the sum its
                        // reciprocal): P stays far from fp32 underflow, at an
                        // error below p * 2^-60 * 448
                        tlv[kb] = sv > 0.0f ? fmaxf(lv, kMinLog2VScale) : 0.0f;
                        tiv[kb] = sv > 0.0f ? (lv > kMinLog2VScale ? __fdividef(1.0f, sv) : 0x1p60f) : 0.0f;
                    }
                    load_scales(i + 1);   // the next tile's, in flight during this one
                }
                if (!warp_wait(&s_full[TT & 1], (TT >> 1) & 1, fail, p.err)) { ok = false; break; }
                tc_fence_after_sync();
                float sc[C::kKB][16];
#pragma unroll
                for (int kb = 0; kb < C::kKB; ++kb)
                    tmem_ld_x16(tmem + lane_base + ((TT & 1) * C::kKB + kb) * kNPad + gbase, sc[kb]);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[TT & 1]);

                // this thread's keys: t, t + 128, ... of the tile
                float z[C::kKB][GH];
                bool any_past_end = false;
#pragma unroll
                for (int kb = 0; kb < C::kKB; ++kb) {
                    const int32_t key = (t0 + i) * C::kKeys + kb * 128 + t;
                    const bool valid = key < len && key >= lo;
                    any_past_end |= key >= len;
                    const int32_t dist = len - 1 - key;
                    const bool has_bias = bias && valid && dist < p.rel_extent;
#pragma unroll
                    for (int g = 0; g < GH; ++g) {
                        float zz = -INFINITY;
                        if (valid && gbase + g < p.G) {
                            zz = kPT ? fmaf(sc[kb][g], p.score_log2 * tsk[kb], tlv[kb])
                                     : sc[kb][g] * p.score_log2;
                            if (has_bias)
                                zz = fmaf(bf16_bits_to_float(__ldg(bias + g * p.rel_extent + dist)),
                                          kLog2e, zz);
                        }
                        z[kb][g] = zz;
                    }
                }
                // block-wide max per head: warp shuffles, then the 4 warps of the
                // warpgroup via shared memory and a (bounded) mbarrier exchange
                float *rb = red + (TT & 1) * 64;
#pragma unroll
                for (int g = 0; g < GH; ++g) {
                    float mx = z[0][g];
#pragma unroll
                    for (int kb = 1; kb < C::kKB; ++kb) mx = fmaxf(mx, z[kb][g]);
                    mx = warp_max(mx);
                    if (lane == 0) rb[wq * 16 + g] = mx;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&red_bar[TT & 1]);
                if (!warp_wait(&red_bar[TT & 1], (TT >> 1) & 1, fail, p.err)) { ok = false; break; }
                float alpha[GH], neg_m8[GH];
                uint8_t *pt = smem + C::kOffP + (TT % C::kOBuf) * 2 * C::kPBytes;
#pragma unroll
                for (int g = 0; g < GH; ++g) {
                    const float tile_max =
                        fmaxf(fmaxf(rb[g], rb[16 + g]), fmaxf(rb[32 + g], rb[48 + g]));
                    const float m_new = fmaxf(m_run[g], tile_max);
                    alpha[g] = (m_new == -INFINITY) ? 1.0f : exp2f(m_run[g] - m_new);
                    // P = 2^(z - m + 8); with no visible key yet (m = -inf) every
                    // z is -inf and P is 0
                    neg_m8[g] = (m_new == -INFINITY) ? 0.0f : 8.0f - m_new;
                    m_run[g] = m_new;
                }
                // Two heads at a time: P of heads g and g + 1 for this key as a
                // packed f16 pair, split into two e4m3 terms, hi = e4m3(P) and
                // lo = e4m3(P - hi) (the difference is exact in f16).
#pragma unroll
                for (int g = 0; g < GH; g += 2) {
                    float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll
                    for (int kb = 0; kb < C::kKB; ++kb) {
                        const float p0 = ex2_approx(z[kb][g] + neg_m8[g]);
                        const float p1 = ex2_approx(z[kb][g + 1] + neg_m8[g + 1]);
                        if constexpr (kPT) {   // the row sum takes P / v_scale
                            ls0 = fmaf(p0, tiv[kb], ls0);
                            ls1 = fmaf(p1, tiv[kb], ls1);
                        } else {
                            ls0 += p0;
                            ls1 += p1;
                        }
                        const __half2 ph = __floats2half2_rn(p0, p1);
                        const uint32_t h8 = __nv_cvt_halfraw2_to_fp8x2(ph, __NV_SATFINITE, __NV_E4M3);
                        const __half2 hh = e4m3x2_to_half2(static_cast<uint16_t>(h8));
                        const uint32_t l8 =
                            __nv_cvt_halfraw2_to_fp8x2(__hsub2(ph, hh), __NV_SATFINITE, __NV_E4M3);
                        uint8_t *blk = pt + kb * C::kPBlock;
                        const int r_hi = 2 * gbase + g, r_lo = 2 * gbase + GH + g;
                        blk[sw128_offset(r_hi, t)] = static_cast<uint8_t>(h8 & 0xFF);
                        blk[sw128_offset(r_hi + 1, t)] = static_cast<uint8_t>((h8 >> 8) & 0xFF);
                        blk[sw128_offset(r_lo, t)] = static_cast<uint8_t>(l8 & 0xFF);
                        blk[sw128_offset(r_lo + 1, t)] = static_cast<uint8_t>((l8 >> 8) & 0xFF);
                    }
                    l_part[g] = fmaf(l_part[g], alpha[g], ls0);
                    l_part[g + 1] = fmaf(l_part[g + 1], alpha[g + 1], ls1);
                }
                // Keys past the sequence end may hold stale bytes (NaN codes
                // included); zero their V rows so that 0 * V stays 0 in the MMA.
                // (Warpgroup 0 does it; the PV waits for every consumer warp.)
                if (hs == 0 && any_past_end) {
                    uint8_t *vtile = smem + (TT % C::kStages) * C::kStageBytes + C::kTileBytes;
#pragma unroll
                    for (int kb = 0; kb < C::kKB; ++kb) {
                        if ((t0 + i) * C::kKeys + kb * 128 + t < len) continue;
#pragma unroll
                        for (int cb = 0; cb < C::kCB; ++cb) {
                            uint4 *r = reinterpret_cast<uint4 *>(vtile + cb * C::kCBBytes +
                                                                 (kb * 128 + t) * 128);
#pragma unroll
                            for (int c = 0; c < 8; ++c) r[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[TT % C::kOBuf]);
                // the MMA thread takes the next item's Q8 after this item's last P
                if (i == ntiles - 1 && nx.ntiles > 0) store_q8();
                if (i >= 2 && !take_o(TT - 2, alpha_2)) { ok = false; break; }
#pragma unroll
                for (int g = 0; g < GH; ++g) {
                    alpha_2[g] = alpha_1[g];
                    alpha_1[g] = alpha[g];
                }
            }
            if (ok && ntiles >= 2) ok = take_o(T + ntiles - 2, alpha_2);
            if (ok && ntiles >= 1) ok = take_o(T + ntiles - 1, alpha_1);

            // l per head: sum of the thread partials of the warpgroup
#pragma unroll
            for (int g = 0; g < GH; ++g) {
                const float s = warp_sum(l_part[g]);
                if (lane == 0) lred[wq * 16 + g] = s;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(l_bar);
            if (ok && !warp_wait(l_bar, A & 1, fail, p.err)) ok = false;
            if (p.direct_out) {
                // the only split: out = bf16(v_scale * o / l), as the merge computes it
#pragma unroll
                for (int g = 0; g < GH; ++g) {
                    if (gbase + g < p.G) {
                        const float L = lred[g] + lred[16 + g] + lred[32 + g] + lred[48 + g];
                        const bool live = ok && m_run[g] != -INFINITY;
                        const float f = (live && L > 0.0f) ? p.out_scale / L : 0.0f;
                        uint16_t *o = p.out + (static_cast<int64_t>(b) * p.Hq + h0 + gbase + g) * D;
#pragma unroll
                        for (int mh = 0; mh < C::kCB; ++mh)
                            o[mh * 128 + t] = __bfloat16_as_ushort(
                                __float2bfloat16_rn((live ? o_acc[mh][g] : 0.0f) * f));
                    }
                }
            }
            const int64_t row0 = (static_cast<int64_t>(b) * p.Hq + h0 + gbase) * p.num_slots + split;
            if (!p.direct_out && t == 0) {
#pragma unroll
                for (int g = 0; g < GH; ++g) {
                    if (gbase + g < p.G) {
                        float *ml = p.part_ml + (row0 + static_cast<int64_t>(g) * p.num_slots) * 2;
                        ml[0] = ok ? m_run[g] : -INFINITY;
                        ml[1] = lred[g] + lred[16 + g] + lred[32 + g] + lred[48 + g];
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < GH && !p.direct_out; ++g) {
                if (gbase + g < p.G) {
                    float *po = p.part_o + (row0 + static_cast<int64_t>(g) * p.num_slots) * D;
#pragma unroll
                    for (int mh = 0; mh < C::kCB; ++mh) po[mh * 128 + t] = o_acc[mh][g];
                }
            }
            T += ntiles;
            ++A;
            it = nx;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge the splits of one (sequence, query head): m = max m_s,
// l = sum l_s 2^(m_s - m), o = sum o_s 2^(m_s - m); out = v_scale * o / l.
// Eight warps take the splits round-robin (lane = 4 consecutive d per 128),
// then the warp partials are summed in a fixed order.
constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
decode_merge_kernel(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                    uint16_t *__restrict__ out, int32_t Hq, int32_t S, float v_scale) {
    constexpr int kV = D / 128;   // float4 per lane
    // launched as a programmatic dependent of the decode grid: its partials
    // are complete and visible once this returns
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float red_m[kMergeWarps];
    __shared__ float red_l[kMergeWarps];
    __shared__ __align__(16) float red_acc[kMergeWarps][D];
    const int h = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(b) * Hq + h;
    const float *ml = part_ml + row * S * 2;
    float m = -INFINITY;
    for (int s = threadIdx.x; s < S; s += kMergeWarps * 32) m = fmaxf(m, ml[2 * s]);
    m = warp_max(m);
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    m = red_m[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) m = fmaxf(m, red_m[w]);
    float4 acc[kV];
#pragma unroll
    for (int c = 0; c < kV; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.0f;
    if (m != -INFINITY) {
#pragma unroll 2
        for (int s = warp; s < S; s += kMergeWarps) {
            const float ms = ml[2 * s];
            if (ms == -INFINITY) continue;
            const float w = exp2f(ms - m);
            l = fmaf(ml[2 * s + 1], w, l);
            const float4 *po = reinterpret_cast<const float4 *>(part_o + (row * S + s) * D);
#pragma unroll
            for (int c = 0; c < kV; ++c) {
                const float4 v = po[c * 32 + lane];
                acc[c].x = fmaf(v.x, w, acc[c].x);
                acc[c].y = fmaf(v.y, w, acc[c].y);
                acc[c].z = fmaf(v.z, w, acc[c].z);
                acc[c].w = fmaf(v.w, w, acc[c].w);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kV; ++c)
        reinterpret_cast<float4 *>(red_acc[warp])[c * 32 + lane] = acc[c];
    if (lane == 0) red_l[warp] = l;
    __syncthreads();
    float L = 0.0f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) L += red_l[w];
    const float f = L > 0.0f ? v_scale / L : 0.0f;
    uint16_t *o = out + row * D;
    for (int d = threadIdx.x; d < D; d += kMergeWarps * 32) {
        float a = 0.0f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) a += red_acc[w][d];
        o[d] = __bfloat16_as_ushort(__float2bfloat16_rn(a * f));
    }
}

// The same merge for launches with few (sequence, query head) rows and many
// splits (a single long sequence): a CTA takes one row and one of
// `gridDim.z` slices of its D values, so that the GPU has enough loads in
// flight.  Lane l of a warp holds float4 l % L of
// the slice (L = slice / 4) for split (l / L) of the warp's group of
// 32 / L splits; the warps take the groups round-robin, four splits per
// thread in flight.  Empty splits (m = -inf) are skipped by a select, so
// their never-written partials are loaded but not used.  The thread
// partials are then summed in a fixed order.
constexpr int kMergeUnroll = 4;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
decode_merge_sliced_kernel(const float *__restrict__ part_o, const float *__restrict__ part_ml,
                    uint16_t *__restrict__ out, int32_t Hq, int32_t S, float v_scale) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // as in decode_merge_kernel
    __shared__ float red_m[kMergeWarps];
    __shared__ __align__(16) float4 red_acc[kMergeWarps * 32];
    __shared__ float red_l[kMergeWarps * 32];
    const int h = blockIdx.x, b = blockIdx.y;
    const int slice = D / static_cast<int>(gridDim.z);   // D values of this CTA
    const int L = slice / 4;                             // lanes per split row
    const int G = 32 / L;                                // splits per warp step
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sg = lane / L, qd = lane % L;
    const int64_t row = static_cast<int64_t>(b) * Hq + h;
    const float *ml = part_ml + row * S * 2;
    float m = -INFINITY;
    for (int s = threadIdx.x; s < S; s += kMergeWarps * 32) m = fmaxf(m, ml[2 * s]);
    m = warp_max(m);
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    m = red_m[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) m = fmaxf(m, red_m[w]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.0f;
    if (m != -INFINITY) {
        const int step = kMergeWarps * G;
        const float4 *pbase = reinterpret_cast<const float4 *>(part_o + row * S * D) +
                              (blockIdx.z * slice) / 4 + qd;
        for (int s0 = warp * G + sg; s0 < S; s0 += kMergeUnroll * step) {
            float ms[kMergeUnroll], ls[kMergeUnroll];
            float4 ov[kMergeUnroll];
#pragma unroll
            for (int u = 0; u < kMergeUnroll; ++u) {
                const int s = s0 + u * step;
                const bool in = s < S;
                ms[u] = in ? ml[2 * s] : -INFINITY;
                ls[u] = in ? ml[2 * s + 1] : 0.0f;
                ov[u] = in ? pbase[static_cast<int64_t>(s) * (D / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kMergeUnroll; ++u) {
                const bool live = ms[u] != -INFINITY;
                const float w = live ? exp2f(ms[u] - m) : 0.0f;
                l = live ? fmaf(ls[u], w, l) : l;
                acc.x = live ? fmaf(ov[u].x, w, acc.x) : acc.x;
                acc.y = live ? fmaf(ov[u].y, w, acc.y) : acc.y;
                acc.z = live ? fmaf(ov[u].z, w, acc.z) : acc.z;
                acc.w = live ? fmaf(ov[u].w, w, acc.w) : acc.w;
            }
        }
    }
    red_acc[threadIdx.x] = acc;
    red_l[threadIdx.x] = qd == 0 ? l : 0.0f;   // one l per split row
    __syncthreads();
    // output float4 q of the slice: the threads with qd == q, in order
    if (threadIdx.x < L) {
        float L_sum = 0.0f;
        for (int t = 0; t < kMergeWarps * 32; t += L) L_sum += red_l[t];
        const float f = L_sum > 0.0f ? v_scale / L_sum : 0.0f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int t = threadIdx.x; t < kMergeWarps * 32; t += L) {
            const float4 v = red_acc[t];
            a.x += v.x;
            a.y += v.y;
            a.z += v.z;
            a.w += v.w;
        }
        uint16_t *o = out + row * D + blockIdx.z * slice + 4 * threadIdx.x;
        o[0] = __bfloat16_as_ushort(__float2bfloat16_rn(a.x * f));
        o[1] = __bfloat16_as_ushort(__float2bfloat16_rn(a.y * f));
        o[2] = __bfloat16_as_ushort(__float2bfloat16_rn(a.z * f));
        o[3] = __bfloat16_as_ushort(__float2bfloat16_rn(a.w * f));
    }
}

struct SplitPlan {
    int num_splits;
    int split_tiles;
    int fine_splits;   // leading splits of fine_tiles tiles each
    int fine_tiles;
};

// Split plan: ~8 work items per resident CTA of the persistent launch (the
// counter hands them out, so short last items even out the tail), at least
// 2048 keys per split and a whole number of quarter splits; the first split
// of each sequence is then cut into quarters (below).  A single sequence
// instead takes the split length that fills whole rounds of the CTA slots.
bool plan_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim,
                 int32_t max_blocks_per_seq, int32_t block_size, int32_t window,
                 int32_t split_tokens, int num_sms, SplitPlan *plan) {
    const int64_t keys = head_dim == 128 ? DecCfg<128>::kKeys : DecCfg<256>::kKeys;
    const int64_t max_len = static_cast<int64_t>(max_blocks_per_seq) * block_size;
    int64_t tiles = (max_len + keys - 1) / keys;
    if (window > 0) {
        const int64_t wt = (static_cast<int64_t>(window) - 1) / keys + 2;
        if (wt < tiles) tiles = wt;
    }
    if (tiles < 1) tiles = 1;
    int64_t st;
    if (split_tokens > 0) {
        if (split_tokens % keys) return false;
        st = split_tokens / keys;
    } else {
        const int64_t ctas_per_sm = head_dim == 128 ? DecCfg<128>::kCtasPerSm : 1;
        const int64_t target = static_cast<int64_t>(num_sms) * ctas_per_sm * 8;
        int64_t pairs = static_cast<int64_t>(num_seqs) * num_kv_heads;
        if (pairs < 1) pairs = 1;
        const int64_t want = (target + pairs - 1) / pairs;
        st = (tiles + want - 1) / want;
        // at least 2048 keys per split: each split costs a partial result
        // (written and merged) and a Q quantization
        const int64_t min_st = (2048 + keys - 1) / keys;
        if (st < min_st) st = min_st;
        st = (st + 3) / 4 * 4;   // whole quarters for the cut below
        if (num_seqs == 1 && (tiles + st - 1) / st >= 2) {
            // One sequence: every item has the same length, so take the
            // split (up to twice as long) whose items fill whole rounds of
            // the CTA slots best, i.e. the least rounds x split length.
            const int64_t slots = static_cast<int64_t>(num_sms) * ctas_per_sm;
            int64_t best = st, best_cost = -1;
            for (int64_t c = st; c <= 2 * st; ++c) {
                const int64_t items = pairs * ((tiles + c - 1) / c);
                const int64_t cost = (items + slots - 1) / slots * c;
                if (best_cost < 0 || cost < best_cost) {
                    best = c;
                    best_cost = cost;
                }
            }
            st = best;
        }
    }
    int64_t S = (tiles + st - 1) / st;
    // Automatic plans with several splits over more than one sequence: the
    // first split of each sequence (in key order) is cut into four.  Items go
    // out last splits first, so these are the launch's last items, and the
    // tail ends in quarter-size pieces.
    int64_t F = 0, ft = 0;
    if (split_tokens <= 0 && S >= 2 && st % 4 == 0 && num_seqs > 1) {
        F = 4;
        ft = st / 4;
        S += F - 1;
    }
    if (S > 65535 || st > (1 << 24)) return false;
    plan->num_splits = static_cast<int>(S);
    plan->split_tiles = static_cast<int>(st);
    plan->fine_splits = static_cast<int>(F);
    plan->fine_tiles = static_cast<int>(ft);
    return true;
}

// Partial-result slots per (sequence, query head): one per split.
int slots_for(int32_t head_dim, int num_splits) {
    (void)head_dim;
    return num_splits;
}

// Workspace: the partial o and (m, l) of every split, then the work-item
// counter of the persistent launch (kSchedBytes).
constexpr size_t kSchedBytes = 256;

size_t workspace_bytes_for(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim, int slots) {
    return static_cast<size_t>(num_seqs) * num_q_heads * slots * (head_dim + 2) * sizeof(float) +
           kSchedBytes;
}

template <int D, int GMAX, bool kPT>
fp8kv_status launch_decode(const CUtensorMap &km, const CUtensorMap &vm, const DecodeParams &p,
                           int num_sms, cudaStream_t stream) {
    using C = DecCfg<D>;
    auto kern = decode_kernel<D, GMAX, kPT>;
    // The whole unified L1 as shared memory: without this preference an SM
    // may take a carveout that holds only one of the kCtasPerSm CTAs.
    static std::atomic<uint64_t> attrs_set{0};
    if (!func_attrs_once(reinterpret_cast<const void *>(kern), &attrs_set, C::kSmemBytes, true))
        return FP8KV_ERR_LAUNCH;
    // persistent: kCtasPerSm CTAs per SM at most; with no more items than
    // that, one CTA per item and no counter
    const int64_t slots = static_cast<int64_t>(num_sms) * C::kCtasPerSm;
    int grid = static_cast<int>(slots);
    DecodeParams q = p;
    if (p.num_items <= slots) {
        grid = p.num_items;
        q.sched = nullptr;
    } else if (cudaMemsetAsync(p.sched, 0, sizeof(uint32_t), stream) != cudaSuccess) {
        cudaGetLastError();
        return FP8KV_ERR_LAUNCH;
    }
    kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(km, vm, q);
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}

}  // namespace
}  // namespace fp8kv

using namespace fp8kv;

extern "C" size_t fp8kv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                              int32_t num_kv_heads, int32_t head_dim,
                                              int32_t max_blocks_per_seq, int32_t block_size,
                                              int32_t window, int32_t split_tokens) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        block_size <= 0 || window < 0 || split_tokens < 0 || (head_dim != 128 && head_dim != 256))
        return 0;
    int sms = 0;
    if (split_tokens == 0 && check_device(&sms) != FP8KV_OK) return 0;
    SplitPlan plan;
    if (!plan_splits(num_seqs, num_kv_heads, head_dim, max_blocks_per_seq, block_size, window,
                     split_tokens, sms, &plan))
        return 0;
    return workspace_bytes_for(num_seqs, num_q_heads, head_dim, slots_for(head_dim, plan.num_splits));
}

namespace {
// One-shot request of fp8kv_test_drop_first_copy, taken by the next decode launch.
std::atomic<int> g_drop_first_copy{0};

// The step's new tokens, stored by the decode launch itself.
struct FusedStore {
    const fp8kv_bf16 *k_new;
    const fp8kv_bf16 *v_new;
    float *amax_k;
    float *amax_v;
};

// Per-token scales of the cached K and V (float[num_blocks][Hkv][block_size]).
struct PerToken {
    const float *k_scales;
    const float *v_scales;
};

fp8kv_status decode_impl(const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads,
                         const int32_t *block_table, int32_t max_blocks_per_seq,
                         const int32_t *seq_lens, int32_t num_seqs, float q_scale, float k_scale,
                         float v_scale, float softmax_scale, const fp8kv_bf16 *rel_bias,
                         int64_t bias_tok_stride, int32_t rel_extent, int32_t window,
                         fp8kv_bf16 *out, void *workspace, size_t workspace_bytes,
                         int32_t split_tokens, const FusedStore *fs, const PerToken *pt,
                         void *stream) {
    if (!cache || num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || window < 0 ||
        split_tokens < 0)
        return FP8KV_ERR_ARG;
    if (!scale_ok(q_scale) || !scale_ok(k_scale) || !scale_ok(v_scale) || !scale_ok(softmax_scale))
        return FP8KV_ERR_SCALE;
    const int D = cache->head_dim, bs = cache->block_size, Hkv = cache->num_kv_heads;
    if (Hkv <= 0 || cache->num_blocks < 0 || num_q_heads % Hkv != 0) return FP8KV_ERR_ARG;
    const int G = num_q_heads / Hkv;
    if ((D != 128 && D != 256) || G > kNPad || (bs != 16 && bs != 32 && bs != 64 && bs != 128) ||
        num_seqs > 65535 || Hkv > 65535 || num_q_heads > 65535 || cache->num_blocks >= (1ll << 31) ||
        static_cast<int64_t>(max_blocks_per_seq) * bs > (1ll << 31) - 256)   // int32 positions
        return FP8KV_ERR_UNSUPPORTED;
    if (rel_bias && (rel_extent <= 0 || bias_tok_stride < 0)) return FP8KV_ERR_ARG;
    if (split_tokens % (D == 128 ? DecCfg<128>::kKeys : DecCfg<256>::kKeys)) return FP8KV_ERR_ARG;
    if (num_seqs == 0) return FP8KV_OK;
    if (!q || !block_table || !seq_lens || !out || !cache->k || !cache->v) return FP8KV_ERR_ARG;
    if (pt && (!pt->k_scales || !pt->v_scales || (reinterpret_cast<uintptr_t>(pt->k_scales) & 3) ||
               (reinterpret_cast<uintptr_t>(pt->v_scales) & 3)))
        return FP8KV_ERR_ARG;
    if (fs && (!fs->k_new || !fs->v_new || (reinterpret_cast<uintptr_t>(fs->k_new) & 15) ||
               (reinterpret_cast<uintptr_t>(fs->v_new) & 15) ||
               (reinterpret_cast<uintptr_t>(fs->amax_k) & 3) ||
               (reinterpret_cast<uintptr_t>(fs->amax_v) & 3)))
        return FP8KV_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(cache->k) & 15) ||
        (reinterpret_cast<uintptr_t>(cache->v) & 15) || (reinterpret_cast<uintptr_t>(out) & 1))
        return FP8KV_ERR_ARG;
    int sms = 0;
    fp8kv_status st = check_device(&sms);
    if (st != FP8KV_OK) return st;
    SplitPlan plan;
    if (!plan_splits(num_seqs, Hkv, D, max_blocks_per_seq, bs, window, split_tokens, sms, &plan))
        return FP8KV_ERR_ARG;
    const int slots = slots_for(D, plan.num_splits);
    const size_t need = workspace_bytes_for(num_seqs, num_q_heads, D, slots);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 15))
        return FP8KV_ERR_WORKSPACE;
    CUtensorMap km, vm;
    if (!make_cache_map(&km, cache->k, cache->num_blocks, bs, Hkv, D) ||
        !make_cache_map(&vm, cache->v, cache->num_blocks, bs, Hkv, D))
        return FP8KV_ERR_LAUNCH;

    DecodeParams p;
    p.q = q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.rel = rel_bias;
    p.part_o = static_cast<float *>(workspace);
    p.part_ml = p.part_o + static_cast<size_t>(num_seqs) * num_q_heads * slots * D;
    p.err = device_error_word();
    p.bias_tok_stride = bias_tok_stride;
    p.num_blocks = cache->num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.Hq = num_q_heads;
    p.G = G;
    p.block_size = bs;
    p.bs_shift = __builtin_ctz(static_cast<unsigned>(bs));
    p.rel_extent = rel_bias ? rel_extent : 0;
    p.window = window;
    p.split_tiles = plan.split_tiles;
    p.fine_splits = plan.fine_splits;
    p.fine_tiles = plan.fine_tiles;
    p.num_slots = slots;
    p.q_scale = make_qscale(q_scale);
    p.score_log2 = static_cast<float>(static_cast<double>(softmax_scale) * q_scale * k_scale *
                                      1.4426950408889634);
    p.k_new = fs ? fs->k_new : nullptr;
    p.v_new = fs ? fs->v_new : nullptr;
    p.cache_k = cache->k;
    p.cache_v = cache->v;
    p.amax_k = fs ? fs->amax_k : nullptr;
    p.amax_v = fs ? fs->amax_v : nullptr;
    p.num_kv_heads = Hkv;
    p.k_scale = make_qscale(k_scale);
    p.v_scale = make_qscale(v_scale);
    p.k_tok_scale = pt ? pt->k_scales : nullptr;
    p.v_tok_scale = pt ? pt->v_scales : nullptr;
    p.drop_first_copy = g_drop_first_copy.exchange(0, std::memory_order_relaxed);
    p.out = out;
    p.out_scale = v_scale;
    p.direct_out = slots == 1 ? 1 : 0;
    p.sched = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + need - kSchedBytes);
    p.num_seqs = num_seqs;
    const int64_t items = static_cast<int64_t>(Hkv) * num_seqs * slots;
    if (items >= (1ll << 31)) return FP8KV_ERR_UNSUPPORTED;
    p.num_items = static_cast<int32_t>(items);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pt) {
        if (D == 128)
            st = G <= 8 ? launch_decode<128, 8, true>(km, vm, p, sms, s)
                        : launch_decode<128, 16, true>(km, vm, p, sms, s);
        else
            st = G <= 8 ? launch_decode<256, 8, true>(km, vm, p, sms, s)
                        : launch_decode<256, 16, true>(km, vm, p, sms, s);
    } else if (D == 128) {
        st = G <= 8 ? launch_decode<128, 8, false>(km, vm, p, sms, s)
                    : launch_decode<128, 16, false>(km, vm, p, sms, s);
    } else {
        st = G <= 8 ? launch_decode<256, 8, false>(km, vm, p, sms, s)
                    : launch_decode<256, 16, false>(km, vm, p, sms, s);
    }
    if (st != FP8KV_OK) return st;
    if (p.direct_out) return FP8KV_OK;   // one split: the decode kernel wrote out
    // slices of D per (sequence, head) for the sliced merge: enough CTAs for
    // two per SM, with at least 32 values (8 lanes of float4) per split row
    int zs = 1;
    while (zs < D / 32 && static_cast<int64_t>(num_q_heads) * num_seqs * zs < 2ll * sms) zs *= 2;
    const dim3 mgrid(num_q_heads, num_seqs, zs);
    // a programmatic dependent launch: the merge's CTAs may be scheduled while
    // the decode grid drains, and wait (griddepcontrol.wait) for its end
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = mgrid;
    cfg.blockDim = dim3(kMergeWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto merge = zs == 1 ? (D == 128 ? decode_merge_kernel<128> : decode_merge_kernel<256>)
                         : (D == 128 ? decode_merge_sliced_kernel<128> : decode_merge_sliced_kernel<256>);
    if (cudaLaunchKernelEx(&cfg, merge, static_cast<const float *>(p.part_o),
                           static_cast<const float *>(p.part_ml), out, num_q_heads, slots,
                           v_scale) != cudaSuccess) {
        cudaGetLastError();
        return FP8KV_ERR_LAUNCH;
    }
    return FP8KV_OK;
}
}  // namespace

extern "C" fp8kv_status paged_attn_fp8_decode_ex(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, float q_scale,
    float k_scale, float v_scale, float softmax_scale, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *workspace,
    size_t workspace_bytes, int32_t split_tokens, void *stream) {
    return decode_impl(cache, q, num_q_heads, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                       q_scale, k_scale, v_scale, softmax_scale, rel_bias, bias_tok_stride,
                       rel_extent, window, out, workspace, workspace_bytes, split_tokens, nullptr,
                       nullptr, stream);
}

extern "C" fp8kv_status paged_attn_fp8_decode_store(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads, const fp8kv_bf16 *k_new,
    const fp8kv_bf16 *v_new, const int32_t *block_table, int32_t max_blocks_per_seq,
    const int32_t *seq_lens, int32_t num_seqs, float q_scale, float k_scale, float v_scale,
    float softmax_scale, const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride, int32_t rel_extent,
    int32_t window, float *amax_k_inout, float *amax_v_inout, fp8kv_bf16 *out, void *workspace,
    size_t workspace_bytes, void *stream) {
    if (num_seqs > 0 && (!k_new || !v_new)) return FP8KV_ERR_ARG;
    const FusedStore fs{k_new, v_new, amax_k_inout, amax_v_inout};
    return decode_impl(cache, q, num_q_heads, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                       q_scale, k_scale, v_scale, softmax_scale, rel_bias, bias_tok_stride,
                       rel_extent, window, out, workspace, workspace_bytes, 0, &fs, nullptr,
                       stream);
}

extern "C" fp8kv_status paged_attn_fp8_decode_per_token(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, float q_scale,
    float softmax_scale, const float *k_scales, const float *v_scales, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *workspace,
    size_t workspace_bytes, void *stream) {
    if (num_seqs > 0 && (!k_scales || !v_scales)) return FP8KV_ERR_ARG;
    const PerToken pt{k_scales, v_scales};
    // the per-token scales replace k_scale and v_scale (1 in the fold and the merge)
    return decode_impl(cache, q, num_q_heads, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                       q_scale, 1.0f, 1.0f, softmax_scale, rel_bias, bias_tok_stride, rel_extent,
                       window, out, workspace, workspace_bytes, 0, nullptr, &pt, stream);
}

extern "C" fp8kv_status fp8kv_test_drop_first_copy(int32_t on) {
    g_drop_first_copy.store(on ? 1 : 0, std::memory_order_relaxed);
    return FP8KV_OK;
}

extern "C" fp8kv_status paged_attn_fp8_decode(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, float q_scale,
    float k_scale, float v_scale, float softmax_scale, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *workspace,
    size_t workspace_bytes, void *stream) {
    return paged_attn_fp8_decode_ex(cache, q, num_q_heads, block_table, max_blocks_per_seq,
                                    seq_lens, num_seqs, q_scale, k_scale, v_scale, softmax_scale,
                                    rel_bias, bias_tok_stride, rel_extent, window, out, workspace,
                                    workspace_bytes, 0, stream);
}

// ---------------------------------------------------------------------------
// Decode without a caller-supplied workspace.
//
// Some callers cannot give the library scratch memory: an engine that hands
// all free device memory to its KV-cache pool at start-up has none left, and a
// latency-critical decode loop must not call cudaMalloc, which can
// synchronize the whole device.  For them the per-split partial results live
// in one fixed buffer compiled into the library: kNoAllocScratchBytes on every
// GPU that loads the library, held until the process exits.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices];
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch buffer on the current device.  The host-side
// name g_noalloc_scratch is only a stand-in, so the address is looked up once
// per device (with that device current) and cached.
static fp8kv_status noalloc_scratch(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return FP8KV_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FP8KV_ERR_LAUNCH;
        }
        g_noalloc_addr[dev] = p;
    }
    *addr = g_noalloc_addr[dev];
    return FP8KV_OK;
}

extern "C" fp8kv_status paged_attn_fp8_decode_noalloc(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, float q_scale,
    float k_scale, float v_scale, float softmax_scale, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *stream) {
    // Argument and device checks of the regular entry point: with no workspace
    // it stops at the workspace check when everything else is valid.
    fp8kv_status st = paged_attn_fp8_decode_ex(
        cache, q, num_q_heads, block_table, max_blocks_per_seq, seq_lens, num_seqs, q_scale,
        k_scale, v_scale, softmax_scale, rel_bias, bias_tok_stride, rel_extent, window, out,
        nullptr, 0, 0, stream);
    if (st != FP8KV_ERR_WORKSPACE) return st;   // an error, or nothing to do
    const size_t need = fp8kv_decode_workspace_size(num_seqs, num_q_heads, cache->num_kv_heads,
                                                    cache->head_dim, max_blocks_per_seq,
                                                    cache->block_size, window, 0);
    if (need == 0 || need > kNoAllocScratchBytes) return FP8KV_ERR_WORKSPACE;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != FP8KV_OK) return st;
    return paged_attn_fp8_decode_ex(cache, q, num_q_heads, block_table, max_blocks_per_seq,
                                    seq_lens, num_seqs, q_scale, k_scale, v_scale, softmax_scale,
                                    rel_bias, bias_tok_stride, rel_extent, window, out, scratch,
                                    kNoAllocScratchBytes, 0, stream);
}
