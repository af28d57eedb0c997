// kv_store.cu -- quant-on-store of bf16 K/V into the e4m3 paged cache and the
// amax calibration pass (vLLM PR 54705 "Purpose", quant-on-store;
// Qwen3.8-27B-FP8-KVcal "What it fixes", amax/448 at the cache-write point).
//
// Both kernels are HBM-bound streams: each thread owns 16 consecutive
// elements of one token row (two 16-byte bf16 loads), so a warp reads 1 KiB
// of one or two rows contiguously; the store writes one 16-byte e4m3 vector
// per K and per V.  Grids are a multiple of the SM count and grid-stride.
#include "common.cuh"

namespace fp8kv {
namespace {

constexpr int kStoreThreads = 256;
constexpr int kChunk = 16;   // elements per thread-step

// 16 bf16 elements -> 16 e4m3 bytes (IEEE fp32 x / s, an exact multiply for
// a power-of-two scale; clamp to +-448 keeping NaN, nearest-even saturating
// conversion, sign kept).  The scale's form is a template argument so that
// only one of multiply / divide is evaluated.
template <bool kPow2>
__device__ __forceinline__ uint4 quantize16(const uint4 lo, const uint4 hi, const QScale &s) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out[i] = quantize_bf16x2_as<kPow2>(w[2 * i], s) |
                 (quantize_bf16x2_as<kPow2>(w[2 * i + 1], s) << 16);
    return make_uint4(out[0], out[1], out[2], out[3]);
}

template <bool kPowK, bool kPowV>
__global__ void __launch_bounds__(kStoreThreads)
kv_store_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, int64_t k_stride,
                int64_t v_stride, const int64_t *__restrict__ slots, int64_t num_tokens,
                int32_t row_elems, int32_t head_dim, int32_t num_kv_heads, int32_t block_size,
                int64_t capacity, uint8_t *__restrict__ ck, uint8_t *__restrict__ cv,
                const QScale k_scale, const QScale v_scale, uint32_t *err) {
    const int32_t chunks = row_elems / kChunk;
    const int64_t total = num_tokens * chunks;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / chunks;
        const int32_t c = static_cast<int32_t>(i - t * chunks);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= capacity) {
            atomicOr(err, FP8KV_DEVERR_BAD_SLOT);
            continue;
        }
        const uint4 *ks = reinterpret_cast<const uint4 *>(k + t * k_stride + c * kChunk);
        const uint4 *vs = reinterpret_cast<const uint4 *>(v + t * v_stride + c * kChunk);
        const uint4 k0 = __ldcs(ks), k1 = __ldcs(ks + 1);
        const uint4 v0 = __ldcs(vs), v1 = __ldcs(vs + 1);
        // cache[block][head][row][d]: head h's row of the block
        const int32_t e = c * kChunk, h = e / head_dim, d = e - h * head_dim;
        const int64_t blk = slot / block_size, row = slot - blk * block_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * head_dim + d;
        *reinterpret_cast<uint4 *>(ck + dst) = quantize16<kPowK>(k0, k1, k_scale);
        *reinterpret_cast<uint4 *>(cv + dst) = quantize16<kPowV>(v0, v1, v_scale);
    }
}

__device__ __forceinline__ float absmax16(const uint4 lo, const uint4 hi, float m) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // fmaxf ignores NaN operands, so NaN elements never win.
        m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    return m;
}

__device__ __forceinline__ float block_max(float m, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = (threadIdx.x < blockDim.x / 32) ? red[threadIdx.x] : 0.0f;
    if (warp == 0)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

__global__ void __launch_bounds__(kStoreThreads)
kv_amax_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, int64_t k_stride,
               int64_t v_stride, const int64_t *__restrict__ slots, int64_t num_tokens,
               int32_t row_elems, float *amax_k, float *amax_v) {
    __shared__ float red[2][kStoreThreads / 32];
    const int32_t chunks = row_elems / kChunk;
    const int64_t total = num_tokens * chunks;
    float mk = 0.0f, mv = 0.0f;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / chunks;
        const int32_t c = static_cast<int32_t>(i - t * chunks);
        if (slots && __ldg(slots + t) < 0) continue;
        if (k) {
            const uint4 *p = reinterpret_cast<const uint4 *>(k + t * k_stride + c * kChunk);
            mk = absmax16(__ldcs(p), __ldcs(p + 1), mk);
        }
        if (v) {
            const uint4 *p = reinterpret_cast<const uint4 *>(v + t * v_stride + c * kChunk);
            mv = absmax16(__ldcs(p), __ldcs(p + 1), mv);
        }
    }
    mk = block_max(mk, red[0]);
    mv = block_max(mv, red[1]);
    // Non-negative floats order like their bit patterns.
    if (threadIdx.x == 0) {
        if (k) atomicMax(reinterpret_cast<unsigned int *>(amax_k), __float_as_uint(mk));
        if (v) atomicMax(reinterpret_cast<unsigned int *>(amax_v), __float_as_uint(mv));
    }
}

int grid_for(int64_t work_items, int num_sms) {
    int64_t blocks = (work_items + kStoreThreads - 1) / kStoreThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // 8 resident CTAs per SM
    if (blocks > cap) blocks = cap;
    return static_cast<int>(blocks < 1 ? 1 : blocks);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Band counts of two elements (one bf16 word, a = low half): their quotients
// and codes as quantize16 makes them, the finite / non-zero / clipped /
// flushed counts, and the relative round-trip errors added to e.  The error
// |s dec(c) - x| / |x| is taken in the quotient's domain, |dec(c) - q| / |q|
// (q = x / s; the two are equal in exact arithmetic and q carries one
// rounding), which keeps the fast division in range without rescaling:
// |q| >= 2^-10 for an element that is not flushed, and a quotient beyond
// 2^100 (an overflowed one included) counts as 2^100.  A flushed element
// decodes to 0, so its term is exactly 1.
template <bool kPow2>
__device__ __forceinline__ void band_pair(uint32_t wd, const QScale &s, uint32_t &n_fin,
                                          uint32_t &n_nz, uint32_t &n_clip, uint32_t &n_flush,
                                          float &e) {
    const float xa = __uint_as_float(wd << 16), xb = __uint_as_float(wd & 0xFFFF0000u);
    const bool fa = (wd & 0x7F80u) != 0x7F80u;             // not NaN or +-Inf
    const bool fb = (wd & 0x7F800000u) != 0x7F800000u;
    const bool za = fa && (wd & 0x7FFFu) != 0u;
    const bool zb = fb && (wd & 0x7FFF0000u) != 0u;
    float qa, qb;
    if (kPow2) {
        const float2 q = __fmul2_rn(make_float2(xa, xb), make_float2(s.inv, s.inv));
        qa = q.x;
        qb = q.y;
    } else {
        qa = __fdiv_rn(xa, s.scale);
        qb = __fdiv_rn(xb, s.scale);
    }
    const uint32_t code = f32x2_to_e4m3x2(qa, qb);
    const float2 d = __half22float2(e4m3x2_to_half2(static_cast<uint16_t>(code)));
    const bool la = za && (code & 0x7Fu) == 0u;
    const bool lb = zb && (code & 0x7F00u) == 0u;
    const float aa = fabsf(qa), ab = fabsf(qb);
    n_fin += static_cast<uint32_t>(fa) + static_cast<uint32_t>(fb);
    n_nz += static_cast<uint32_t>(za) + static_cast<uint32_t>(zb);
    n_clip += static_cast<uint32_t>(za && aa > kE4M3Max) + static_cast<uint32_t>(zb && ab > kE4M3Max);
    n_flush += static_cast<uint32_t>(la) + static_cast<uint32_t>(lb);
    const float ca = fminf(aa, 0x1p100f), cb = fminf(ab, 0x1p100f);
    e += la ? 1.0f : (za ? __fdividef(fabsf(fabsf(d.x) - ca), ca) : 0.0f);
    e += lb ? 1.0f : (zb ? __fdividef(fabsf(fabsf(d.y) - cb), cb) : 0.0f);
}

// Band counters of one stream at one scale, through a table.  An element's
// error term and its clip and flush tests depend only on its magnitude bits
// t = bits & 0x7FFF (the quotient and the e4m3 code are sign-symmetric), so
// each CTA first evaluates band_pair once per t into a table of 32,768 fp32
// terms in shared memory, and the stream reads each element's term from it
// (the same value, added in the same order as band_pair over the element's
// word).  Both tests are monotone in t, the quotient and the nearest-even
// conversion being non-decreasing in |x|: an element is flushed iff
// 0 < t <= t_flush and clipped iff t_clip <= t < 0x7F80, with the two bounds
// taken from the table's own entries.  The counts are then four comparisons
// per element: not finite (t >= 0x7F80), zero, t >= t_clip, t <= t_flush.
// The error terms are summed in fp32 over a thread's 16 elements, then in
// fp64.  chunk_shift is log2 of the chunks per row when that is a power of
// two, else -1.  One 64-bit atomic per counter and block.
constexpr int kBandThreads = 1024;
constexpr int kBandTab = 1 << 15;
constexpr int kBandSmem = kBandTab * static_cast<int>(sizeof(float));

template <bool kPow2>
__global__ void __launch_bounds__(kBandThreads, 1)
kv_band_kernel(const uint16_t *__restrict__ x, int64_t stride, const int64_t *__restrict__ slots,
               int64_t num_tokens, int32_t row_elems, int32_t chunk_shift, const QScale s,
               fp8kv_band_counts *out) {
    extern __shared__ float tab[];   // [kBandTab] error term of magnitude bits t
    __shared__ unsigned long long red_n[4][kBandThreads / 32];
    __shared__ double red_e[kBandThreads / 32];
    __shared__ uint32_t t_flush, t_clip;
    if (threadIdx.x == 0) {
        t_flush = 0u;        // no flushed magnitude: only t = 0 is <= t_flush
        t_clip = 0x7F80u;    // no clipped magnitude: only non-finite t are >= t_clip
    }
    __syncthreads();
    for (uint32_t t = threadIdx.x; t < static_cast<uint32_t>(kBandTab); t += blockDim.x) {
        uint32_t fin = 0, nz = 0, clip = 0, flush = 0;
        float e = 0.0f;
        band_pair<kPow2>(t, s, fin, nz, clip, flush, e);   // (t, +0): the +0 adds nothing
        tab[t] = e;
        if (flush) atomicMax(&t_flush, t);
        if (clip) atomicMin(&t_clip, t);
    }
    __syncthreads();
    const uint32_t tf = t_flush, tc = t_clip;

    const int32_t chunks = row_elems / kChunk;
    const int64_t total = num_tokens * chunks;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint32_t c_all = 0, c_inf = 0, c_zero = 0, c_hi = 0, c_lo = 0;   // this thread's counts
    double err = 0.0;
    // two chunks per iteration, both loaded before either is counted
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += 2 * step) {
        uint4 v[2][2];
        bool use[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t ci = i + u * step;
            use[u] = ci < total;
            if (!use[u]) continue;
            const int64_t t = chunk_shift >= 0 ? (ci >> chunk_shift) : ci / chunks;
            const int32_t c = static_cast<int32_t>(ci - t * chunks);
            if (slots && __ldg(slots + t) < 0) {
                use[u] = false;
                continue;
            }
            const uint4 *p = reinterpret_cast<const uint4 *>(x + t * stride + c * kChunk);
            v[u][0] = __ldcs(p);
            v[u][1] = __ldcs(p + 1);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (!use[u]) continue;
            const uint32_t w[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                                   v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
            float e16 = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t t = (w[k] >> (16 * h)) & 0x7FFFu;
                    e16 += tab[t];
                    c_inf += t >= 0x7F80u ? 1u : 0u;
                    c_zero += t == 0u ? 1u : 0u;
                    c_hi += t >= tc ? 1u : 0u;
                    c_lo += t <= tf ? 1u : 0u;
                }
            }
            c_all += 16u;
            err += static_cast<double>(e16);
        }
    }
    // finite, non-zero, clipped (finite and t >= t_clip), flushed (non-zero
    // and t <= t_flush)
    unsigned long long n_fin = c_all - c_inf, n_nz = c_all - c_inf - c_zero, n_clip = c_hi - c_inf,
                       n_flush = c_lo - c_zero;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        n_fin += __shfl_xor_sync(0xffffffffu, n_fin, o);
        n_nz += __shfl_xor_sync(0xffffffffu, n_nz, o);
        n_clip += __shfl_xor_sync(0xffffffffu, n_clip, o);
        n_flush += __shfl_xor_sync(0xffffffffu, n_flush, o);
        err += __shfl_xor_sync(0xffffffffu, err, o);
    }
    if (lane == 0) {
        red_n[0][warp] = n_fin;
        red_n[1][warp] = n_nz;
        red_n[2][warp] = n_clip;
        red_n[3][warp] = n_flush;
        red_e[warp] = err;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long a[4] = {0, 0, 0, 0};
        double e = 0.0;
        for (int w2 = 0; w2 < kBandThreads / 32; ++w2) {
#pragma unroll
            for (int f = 0; f < 4; ++f) a[f] += red_n[f][w2];
            e += red_e[w2];
        }
        if (a[0]) {
            atomicAdd(&out->count, a[0]);
            atomicAdd(&out->nonzero, a[1]);
            atomicAdd(&out->clipped, a[2]);
            atomicAdd(&out->flushed, a[3]);
            atomicAdd(&out->rt_err_sum, e);
        }
    }
}

// Per-token store: one warp per (token, KV head) row of D values.  The
// row's scale is max |x| / 448 over its finite values (the IEEE quotient; 1
// for an all-zero row), then every value is quantized with it exactly as
// quantize16 does (division).  Lane l holds D/32 consecutive values.
template <int D>
__global__ void __launch_bounds__(kStoreThreads)
kv_store_pt_kernel(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                   int64_t k_stride, int64_t v_stride, const int64_t *__restrict__ slots,
                   int64_t num_tokens, int32_t num_kv_heads, int32_t block_size, int64_t capacity,
                   uint8_t *__restrict__ ck, uint8_t *__restrict__ cv, float *__restrict__ sk,
                   float *__restrict__ sv, uint32_t *err) {
    constexpr int kPer = D / 32;                  // values per lane (4 or 8)
    const int lane = threadIdx.x & 31;
    const int64_t rows = num_tokens * num_kv_heads;
    for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < rows;
         w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t t = w / num_kv_heads;
        const int32_t h = static_cast<int32_t>(w - t * num_kv_heads);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= capacity) {
            if (lane == 0) atomicOr(err, FP8KV_DEVERR_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size, row = slot - blk * block_size;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * D + lane * kPer;
        const int64_t sdst = (blk * num_kv_heads + h) * block_size + row;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint16_t *src = (which ? v + t * v_stride : k + t * k_stride) + h * D + lane * kPer;
            uint32_t wd[kPer / 2];
            if constexpr (kPer == 4) {
                const uint2 a = *reinterpret_cast<const uint2 *>(src);
                wd[0] = a.x;
                wd[1] = a.y;
            } else {
                const uint4 a = *reinterpret_cast<const uint4 *>(src);
                wd[0] = a.x;
                wd[1] = a.y;
                wd[2] = a.z;
                wd[3] = a.w;
            }
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const uint32_t bits = (wd[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
                if ((bits & 0x7F80u) != 0x7F80u) m = fmaxf(m, fabsf(__uint_as_float(bits << 16)));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            QScale qs;
            qs.scale = m > 0.0f ? __fdiv_rn(m, kE4M3Max) : 1.0f;
            qs.inv = 0.0f;
            qs.pow2 = 0u;
            uint32_t out[kPer / 4];
#pragma unroll
            for (int i = 0; i < kPer / 4; ++i)
                out[i] = quantize_bf16x2_as<false>(wd[2 * i], qs) |
                         (quantize_bf16x2_as<false>(wd[2 * i + 1], qs) << 16);
            uint8_t *c = which ? cv : ck;
            if constexpr (kPer == 4)
                *reinterpret_cast<uint32_t *>(c + dst) = out[0];
            else
                *reinterpret_cast<uint2 *>(c + dst) = make_uint2(out[0], out[1]);
            if (lane == 0) (which ? sv : sk)[sdst] = qs.scale;
        }
    }
}

}  // namespace
}  // namespace fp8kv

using namespace fp8kv;

extern "C" fp8kv_status kv_store_e4m3(const fp8kv_cache *cache, const fp8kv_bf16 *k,
                                      const fp8kv_bf16 *v, int64_t k_tok_stride,
                                      int64_t v_tok_stride, const int64_t *slot_mapping,
                                      int64_t num_tokens, float k_scale, float v_scale,
                                      void *stream) {
    if (!cache || num_tokens < 0) return FP8KV_ERR_ARG;
    if (!scale_ok(k_scale) || !scale_ok(v_scale)) return FP8KV_ERR_SCALE;
    if (cache->num_blocks < 0 || cache->block_size <= 0 || cache->num_kv_heads <= 0 ||
        cache->head_dim <= 0)
        return FP8KV_ERR_ARG;
    const int64_t row = static_cast<int64_t>(cache->num_kv_heads) * cache->head_dim;
    if (row % kChunk != 0 || cache->head_dim % kChunk != 0 || row > (1 << 30))
        return FP8KV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return FP8KV_OK;
    if (!cache->k || !cache->v || !k || !v || !slot_mapping) return FP8KV_ERR_ARG;
    if (k_tok_stride < row || v_tok_stride < row || (k_tok_stride % 8) || (v_tok_stride % 8))
        return FP8KV_ERR_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(cache->k) || !aligned16(cache->v))
        return FP8KV_ERR_ARG;
    int sms = 0;
    fp8kv_status st = check_device(&sms);
    if (st != FP8KV_OK) return st;
    uint32_t *err = device_error_word();
    const int64_t capacity = cache->num_blocks * cache->block_size;
    const int grid = grid_for(num_tokens * (row / kChunk), sms);
    const QScale ks = make_qscale(k_scale), vs = make_qscale(v_scale);
    auto kernel = ks.pow2 ? (vs.pow2 ? kv_store_kernel<true, true> : kv_store_kernel<true, false>)
                          : (vs.pow2 ? kv_store_kernel<false, true> : kv_store_kernel<false, false>);
    kernel<<<grid, kStoreThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        k, v, k_tok_stride, v_tok_stride, slot_mapping, num_tokens, static_cast<int32_t>(row),
        cache->head_dim, cache->num_kv_heads, cache->block_size, capacity, cache->k, cache->v, ks,
        vs, err);
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}

extern "C" fp8kv_status kv_amax_calibrate(const fp8kv_bf16 *k, const fp8kv_bf16 *v,
                                          int64_t k_tok_stride, int64_t v_tok_stride,
                                          const int64_t *slot_mapping, int64_t num_tokens,
                                          int32_t num_kv_heads, int32_t head_dim,
                                          float *amax_k_inout, float *amax_v_inout,
                                          void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0) return FP8KV_ERR_ARG;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (row % kChunk != 0 || row > (1 << 30)) return FP8KV_ERR_UNSUPPORTED;
    if (k && (!amax_k_inout || k_tok_stride < row || (k_tok_stride % 8) || !aligned16(k)))
        return FP8KV_ERR_ARG;
    if (v && (!amax_v_inout || v_tok_stride < row || (v_tok_stride % 8) || !aligned16(v)))
        return FP8KV_ERR_ARG;
    if (num_tokens == 0 || (!k && !v)) return FP8KV_OK;
    int sms = 0;
    fp8kv_status st = check_device(&sms);
    if (st != FP8KV_OK) return st;
    const int grid = grid_for(num_tokens * (row / kChunk), sms);
    kv_amax_kernel<<<grid, kStoreThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        k, v, k_tok_stride, v_tok_stride, slot_mapping, num_tokens, static_cast<int32_t>(row),
        amax_k_inout, amax_v_inout);
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}

extern "C" fp8kv_status kv_band_counts(const fp8kv_bf16 *x, int64_t tok_stride,
                                       const int64_t *slot_mapping, int64_t num_tokens,
                                       int32_t row_elems, float scale, fp8kv_band_counts *counts,
                                       void *stream) {
    if (num_tokens < 0 || row_elems <= 0) return FP8KV_ERR_ARG;
    if (!scale_ok(scale)) return FP8KV_ERR_SCALE;
    if (row_elems % kChunk != 0 || row_elems > (1 << 30)) return FP8KV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return FP8KV_OK;
    if (!x || !counts || tok_stride < row_elems || (tok_stride % 8) || !aligned16(x) ||
        (reinterpret_cast<uintptr_t>(counts) & 7))
        return FP8KV_ERR_ARG;
    int sms = 0;
    fp8kv_status st = check_device(&sms);
    if (st != FP8KV_OK) return st;
    const int32_t chunks = row_elems / kChunk;
    int32_t chunk_shift = -1;
    if ((chunks & (chunks - 1)) == 0)
        for (chunk_shift = 0; (1 << chunk_shift) < chunks; ++chunk_shift) {
        }
    // one CTA per SM (the table fills most of its shared memory), fewer for
    // small inputs
    int64_t blocks = (num_tokens * chunks + kBandThreads - 1) / kBandThreads;
    if (blocks > sms) blocks = sms;
    const int grid = static_cast<int>(blocks);
    const QScale qs = make_qscale(scale);
    auto kernel = qs.pow2 ? kv_band_kernel<true> : kv_band_kernel<false>;
    static std::atomic<uint64_t> attrs_set[2];
    if (!func_attrs_once(reinterpret_cast<const void *>(kernel), &attrs_set[qs.pow2 ? 1 : 0],
                         kBandSmem, true))
        return FP8KV_ERR_LAUNCH;
    kernel<<<grid, kBandThreads, kBandSmem, static_cast<cudaStream_t>(stream)>>>(
        x, tok_stride, slot_mapping, num_tokens, row_elems, chunk_shift, qs, counts);
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}

extern "C" fp8kv_status kv_store_e4m3_per_token(const fp8kv_cache *cache, const fp8kv_bf16 *k,
                                                const fp8kv_bf16 *v, int64_t k_tok_stride,
                                                int64_t v_tok_stride,
                                                const int64_t *slot_mapping, int64_t num_tokens,
                                                float *k_scales, float *v_scales, void *stream) {
    if (!cache || num_tokens < 0) return FP8KV_ERR_ARG;
    const int32_t D = cache->head_dim, Hkv = cache->num_kv_heads, bs = cache->block_size;
    if (Hkv <= 0 || bs <= 0 || cache->num_blocks < 0) return FP8KV_ERR_ARG;
    if (D != 128 && D != 256) return FP8KV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return FP8KV_OK;
    const int64_t row = static_cast<int64_t>(Hkv) * D;
    if (!k || !v || !slot_mapping || !k_scales || !v_scales || !cache->k || !cache->v ||
        k_tok_stride < row || v_tok_stride < row || (k_tok_stride % 8) || (v_tok_stride % 8))
        return FP8KV_ERR_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(cache->k) || !aligned16(cache->v) ||
        (reinterpret_cast<uintptr_t>(k_scales) & 3) || (reinterpret_cast<uintptr_t>(v_scales) & 3))
        return FP8KV_ERR_ARG;
    int sms = 0;
    fp8kv_status st = check_device(&sms);
    if (st != FP8KV_OK) return st;
    const int64_t warps = num_tokens * Hkv;
    const int grid = grid_for(warps * 32, sms);
    const int64_t capacity = cache->num_blocks * bs;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (D == 128)
        kv_store_pt_kernel<128><<<grid, kStoreThreads, 0, s>>>(
            k, v, k_tok_stride, v_tok_stride, slot_mapping, num_tokens, Hkv, bs, capacity,
            cache->k, cache->v, k_scales, v_scales, device_error_word());
    else
        kv_store_pt_kernel<256><<<grid, kStoreThreads, 0, s>>>(
            k, v, k_tok_stride, v_tok_stride, slot_mapping, num_tokens, Hkv, bs, capacity,
            cache->k, cache->v, k_scales, v_scales, device_error_word());
    if (cudaGetLastError() != cudaSuccess) return FP8KV_ERR_LAUNCH;
    return FP8KV_OK;
}
