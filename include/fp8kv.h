/*
 * fp8kv.h -- C ABI of libfp8kv: an FP8 e4m3 paged KV cache and attention
 * over it, as hand-written CUDA kernels for one NVIDIA GB300 (sm_103).
 *
 * The method is the one of vLLM pull request 54705 ("fp8 e4m3 KV cache for
 * Inkling on SM100"), section "Purpose":
 *   - quant-on-store: K and V are divided by a per-tensor scale, clamped to
 *     the e4m3 finite range +-448 and stored as e4m3 bytes in a paged cache;
 *   - query quantization: q is statically quantized to e4m3 with q_scale;
 *   - descale handling: the QK descale is folded into softmax_scale
 *     (softmax_scale * q_scale * k_scale), the scores are descaled before an
 *     exact bf16 relative-position bias is added, and the output is
 *     multiplied by v_scale;
 *   - full-causal or 512-token sliding-window attention layers.
 * Scale calibration (amax/448) follows the model card "Qwen3.8-27B-FP8-KVcal",
 * section "What it fixes".
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers on the current
 *     device; the caller owns all memory, including workspaces.  The library
 *     never allocates device memory and never synchronizes the stream.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on it.
 *   - bf16 data is passed as raw 16-bit patterns (fp8kv_bf16).
 *   - Scales are host floats, passed by value; they must be finite and > 0
 *     (vLLM PR 54705 "Purpose": loaded scales are validated finite and
 *     positive; scalar descales stay on the host so the hot path never syncs
 *     on a GPU scalar).
 *   - Errors are returned as fp8kv_status; nothing aborts or throws.
 *     Arguments are checked on the host before any CUDA call.  A kernel that
 *     meets an inconsistency it can detect (a bounded wait that ran out, a
 *     block id outside the pool) records a bit in a device error word, skips
 *     the faulty access and finishes; fp8kv_device_error() reads the word.
 *   - Only e4m3 (OCP "e4m3fn", max 448) is supported; the gate of vLLM PR
 *     54705 ("Purpose", first bullet) rejects other fp8 variants and other
 *     devices, and so does this library (FP8KV_ERR_UNSUPPORTED when the
 *     device is not compute capability 10.3).
 *
 * Cache layout (fp8kv_cache): two byte arrays, K and V, each
 *   uint8[num_blocks][num_kv_heads][block_size][head_dim]  (row-major),
 * every byte an e4m3 code: one head's rows of a block are contiguous
 * (block_size * head_dim bytes).  Token slot s lives in block s / block_size,
 * row s % block_size, of every head.  A sequence's keys are listed by its block-table row:
 * logical block i of sequence b is physical block block_table[b][i].
 * Supported: block_size in {16, 32, 64, 128}, head_dim in {128, 256}.
 * head_dim 64 is not supported (FP8KV_ERR_UNSUPPORTED): the kernels move
 * K/V rows as 128-byte swizzled TMA boxes and feed the MMAs 128-byte rows.
 */
#ifndef FP8KV_H
#define FP8KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8KV_OK = 0,
    FP8KV_ERR_ARG = 1,          /* null pointer, negative size, bad stride or shape  */
    FP8KV_ERR_SCALE = 2,        /* a scale that is not finite and > 0                 */
    FP8KV_ERR_UNSUPPORTED = 3,  /* device not sm_103, head_dim / block size / GQA     */
    FP8KV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required        */
    FP8KV_ERR_LAUNCH = 5,       /* a CUDA runtime call or kernel launch failed       */
    FP8KV_ERR_DEVICE = 6        /* the device error word is set (see below)          */
} fp8kv_status;

typedef uint16_t fp8kv_bf16;    /* raw bfloat16 bit pattern */

/* Device error word bits (fp8kv_device_error). */
#define FP8KV_DEVERR_WAIT_TIMEOUT 0x1u   /* a bounded pipeline wait ran out       */
#define FP8KV_DEVERR_BAD_BLOCK    0x2u   /* a block id outside [0, num_blocks), or a
                                            sequence length past its block-table row  */
#define FP8KV_DEVERR_BAD_SLOT     0x4u   /* a slot outside the pool                */

typedef struct {
    uint8_t *k;            /* device, num_blocks*num_kv_heads*block_size*head_dim bytes */
    uint8_t *v;            /* device, same size as k                                    */
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
} fp8kv_cache;

/*
 * kv_store_e4m3 -- quantize bf16 K and V and scatter them into the cache
 * (vLLM PR 54705 "Purpose", quant-on-store).
 *   byte = e4m3_rn_sat( fp32(x) / scale )   -- IEEE fp32 division, clamp to
 *   +-448 (NaN stays NaN, +-Inf saturates), round to nearest even.
 * k, v:        device bf16, token t's row of num_kv_heads*head_dim elements
 *              starts at k + t*k_tok_stride (v + t*v_tok_stride); rows must be
 *              contiguous, strides are in elements and multiples of 8.
 * slot_mapping: device int64 [num_tokens]; slot < 0 skips the token; a slot
 *              >= num_blocks*block_size is skipped and sets
 *              FP8KV_DEVERR_BAD_SLOT.
 * num_tokens:  >= 0 (0 is a no-op).
 */
fp8kv_status kv_store_e4m3(const fp8kv_cache *cache, const fp8kv_bf16 *k,
                           const fp8kv_bf16 *v, int64_t k_tok_stride,
                           int64_t v_tok_stride, const int64_t *slot_mapping,
                           int64_t num_tokens, float k_scale, float v_scale,
                           void *stream);

/*
 * paged_attn_fp8_decode -- one query token per sequence attends over its
 * cached keys (vLLM PR 54705 "Purpose", descale handling and query
 * quantization), split over the KV length with a log-sum-exp merge.
 *   q8    = e4m3_rn_sat(q / q_scale)
 *   z_j   = (softmax_scale*q_scale*k_scale) * <q8, k8_j> + bias(j)
 *   out   = bf16( v_scale * sum_j softmax(z)_j * v8_j )
 * q:            device bf16 [num_seqs][num_q_heads][head_dim], contiguous.
 * num_q_heads:  a multiple of num_kv_heads with at most 16 query heads per KV
 *               head (q head h reads KV head h / (num_q_heads/num_kv_heads)).
 * block_table:  device int32 [num_seqs][max_blocks_per_seq].
 * seq_lens:     device int32 [num_seqs], keys per sequence,
 *               0 <= len <= max_blocks_per_seq*block_size.  The query sits at
 *               position len-1 (it is the newest stored token).  len = 0
 *               yields zeros.  Keys whose block lies past the table row (a
 *               longer len) or whose table entry is outside [0, num_blocks)
 *               are read as zeros and set FP8KV_DEVERR_BAD_BLOCK.
 * rel_bias:     NULL, or device bf16; the bias of sequence b, query head h,
 *               distance d = (len-1) - j is rel_bias[b*bias_tok_stride +
 *               h*rel_extent + d] for 0 <= d < rel_extent, else 0.  It is
 *               added after the descale and not multiplied by softmax_scale.
 * window:       0 = full causal; W > 0 = only keys with (len-1) - j < W.
 * out:          device bf16 [num_seqs][num_q_heads][head_dim].
 * workspace:    device, >= fp8kv_decode_workspace_size(...) bytes, 16-byte
 *               aligned; holds the per-split partial results and the work
 *               counter of the persistent launch (the call zeroes it on the
 *               stream before the launch).  Calls that overlap on the GPU
 *               must not share a workspace.
 * Launch: one persistent kernel of at most two CTAs per SM that take the
 * splits from that counter, then (with more than one split) a merge kernel,
 * launched as a programmatic dependent of the first (it waits for the first
 * grid's completion before reading the partials).
 */
fp8kv_status paged_attn_fp8_decode(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                   int32_t num_q_heads, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                   int32_t num_seqs, float q_scale, float k_scale,
                                   float v_scale, float softmax_scale,
                                   const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride,
                                   int32_t rel_extent, int32_t window, fp8kv_bf16 *out,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attn_fp8_decode_ex -- paged_attn_fp8_decode with an explicit split
 * length: split_tokens > 0 makes every split cover that many keys and must be
 * a multiple of the kernel's key tile (128 keys);
 * 0 chooses it from the device's SM count (the plain call).
 */
fp8kv_status paged_attn_fp8_decode_ex(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                      int32_t num_q_heads, const int32_t *block_table,
                                      int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                      int32_t num_seqs, float q_scale, float k_scale,
                                      float v_scale, float softmax_scale,
                                      const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride,
                                      int32_t rel_extent, int32_t window, fp8kv_bf16 *out,
                                      void *workspace, size_t workspace_bytes,
                                      int32_t split_tokens, void *stream);

/*
 * paged_attn_fp8_decode_store -- one decode step in one call: quantize and
 * write each sequence's new token into the cache (as kv_store_e4m3 does),
 * optionally raise the running amax over it (as kv_amax_calibrate does), and
 * attend (as paged_attn_fp8_decode does).  The pages' write path quantizes
 * K/V on store inside the fused small-batch prep kernel that also emits q
 * (vLLM PR 54705 "Purpose", quant-on-store); here the store rides on the
 * decode launch that reads the token's tile, so the step costs the decode
 * and merge launches only.
 * k_new, v_new:  device bf16 [num_seqs][num_kv_heads][head_dim], contiguous,
 *                16-byte aligned: the step's new token of each sequence.  It
 *                is the sequence's last key: position seq_lens[b] - 1, in
 *                cache block block_table[b][(seq_lens[b]-1) / block_size],
 *                row (seq_lens[b]-1) % block_size.  A sequence with
 *                seq_lens[b] == 0 stores nothing.
 * amax_k_inout, amax_v_inout: NULL, or device float >= 0: raised to the max
 *                |k_new| (|v_new|) over all sequences (NaN ignored).
 * Other arguments and the result are those of paged_attn_fp8_decode; the
 * cache bytes written are bit-identical to kv_store_e4m3's, and the output
 * equals that of kv_store_e4m3 followed by paged_attn_fp8_decode.  An
 * invalid block-table entry for the new token's block sets
 * FP8KV_DEVERR_BAD_BLOCK and stores nothing.
 */
fp8kv_status paged_attn_fp8_decode_store(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                         int32_t num_q_heads, const fp8kv_bf16 *k_new,
                                         const fp8kv_bf16 *v_new, const int32_t *block_table,
                                         int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                         int32_t num_seqs, float q_scale, float k_scale,
                                         float v_scale, float softmax_scale,
                                         const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride,
                                         int32_t rel_extent, int32_t window, float *amax_k_inout,
                                         float *amax_v_inout, fp8kv_bf16 *out, void *workspace,
                                         size_t workspace_bytes, void *stream);

/*
 * paged_attn_fp8_decode_noalloc -- paged_attn_fp8_decode for callers that
 * cannot provide a workspace.  (The pages describe no such call; it exists
 * for users of this library.)  Some callers cannot allocate device memory at
 * all: an engine that gives every free byte of HBM to its KV-cache pool at
 * start-up has nothing left to lend, and a latency-critical decode loop must
 * not call cudaMalloc, which can synchronize the device.  This entry point
 * keeps the per-split partial results in one fixed 16 MiB buffer that is part
 * of the library's device image (every GPU that loads the library holds it
 * until the process exits) and allocates nothing.
 *   - Arguments, layout and results are those of paged_attn_fp8_decode.
 *   - Returns FP8KV_ERR_WORKSPACE when the sizes would need more than the
 *     16 MiB buffer (fp8kv_decode_workspace_size(..., split_tokens = 0)
 *     larger than 16 MiB).
 *   - The first call on a device looks up the buffer's device address (a
 *     CUDA runtime query) and keeps it for later calls.
 *   - Every call on a device shares the one buffer and may overwrite what
 *     the previous call left there; nothing in it needs clearing between
 *     calls.  Calls that can overlap on the GPU (on different streams, or
 *     from different threads) race on it: serialize them.
 */
fp8kv_status paged_attn_fp8_decode_noalloc(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                           int32_t num_q_heads, const int32_t *block_table,
                                           int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                           int32_t num_seqs, float q_scale, float k_scale,
                                           float v_scale, float softmax_scale,
                                           const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride,
                                           int32_t rel_extent, int32_t window, fp8kv_bf16 *out,
                                           void *stream);

/* Workspace bytes paged_attn_fp8_decode(_ex) needs for these sizes (split_tokens
 * as in _ex; 0 = automatic).  Returns 0 for invalid sizes. */
size_t fp8kv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim,
                                   int32_t max_blocks_per_seq, int32_t block_size,
                                   int32_t window, int32_t split_tokens);

/*
 * attn_fp8_varlen_prefill -- causal (optionally sliding-window) attention of
 * a chunk of query tokens per sequence over the cached keys, on FP8 tensor
 * cores (vLLM PR 54705 "Purpose" descale handling; evidence document Tier 0:
 * P is formed in e4m3 pre-scaled by 2^8 with a lazy-rescale threshold of
 * 0.75 < log2(448) - 8).  P of a 64-key half of a row is one e4m3 term
 * while a bound on the rounding error it adds to the row stays within a
 * fixed budget; rows with few visible keys or a few dominant weights get a
 * second term e4m3(P - P_hi) as well.
 * q:             device bf16 [total_q][num_q_heads][head_dim], contiguous;
 *                sequence b's queries are rows cu_seqlens_q[b] ..
 *                cu_seqlens_q[b+1]-1.
 * cu_seqlens_q:  device int32 [num_seqs+1], non-decreasing, starting at 0.
 * seq_lens_k:    device int32 [num_seqs]; keys per sequence, >= the
 *                sequence's query count.  The queries are the last ones:
 *                query i of a chunk of n sits at position seq_len_k - n + i.
 *                Keys past the block-table row, or with a table entry outside
 *                [0, num_blocks), are read as zeros and set
 *                FP8KV_DEVERR_BAD_BLOCK.
 * max_seqlen_q:  an upper bound of the per-sequence query counts (sizes the
 *                grid and bounds the rows of q that are read, num_seqs *
 *                max_seqlen_q; rows beyond a sequence's count do nothing).
 * rel_bias:      NULL, or device bf16; bias of query row t (global index),
 *                head h, distance d = pos_q - pos_k is
 *                rel_bias[t*bias_tok_stride + h*rel_extent + d] for
 *                0 <= d < rel_extent, else 0.
 * window, out:   as for decode; out is [total_q][num_q_heads][head_dim].
 * workspace:     not used (may be NULL / 0).
 */
fp8kv_status attn_fp8_varlen_prefill(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                     int32_t num_q_heads, const int32_t *cu_seqlens_q,
                                     const int32_t *seq_lens_k, const int32_t *block_table,
                                     int32_t max_blocks_per_seq, int32_t num_seqs,
                                     int32_t max_seqlen_q, float q_scale, float k_scale,
                                     float v_scale, float softmax_scale,
                                     const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride,
                                     int32_t rel_extent, int32_t window, fp8kv_bf16 *out,
                                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * fp8kv_set_prefill_max_ctas -- caps the grid of attn_fp8_varlen_prefill at
 * head_dim 128.  For batches of up to 64 sequences that prefill is
 * persistent: one CTA per SM, each running two pipelines that work through
 * the (query tile, head, sequence) items, so that one item's Q load and
 * output overlap the MMAs of the next item and of the other pipeline.  A cap
 * below the SM count leaves SMs to work on other streams; 0 (the default)
 * restores one CTA per SM.  The results do not depend on the cap.
 * Process-wide, read at each launch.
 * Returns FP8KV_ERR_ARG for a negative cap.
 */
fp8kv_status fp8kv_set_prefill_max_ctas(int32_t max_ctas);

/*
 * kv_store_e4m3_per_token -- quant-on-store with a dynamic scale per token
 * and KV head, kept beside the cache (local-inference-lab/vllm PR 189: a
 * per-token scale stored with each cached token, so that no calibrated
 * per-tensor scale is needed).  For each stored token and KV head h, over
 * the head's head_dim values x:
 *   s = max |x| / 448 over the finite values (fp32 IEEE quotient; 1 if they
 *       are all zero)
 *   code = e4m3(x / s) exactly as kv_store_e4m3 quantizes at scale s
 * The codes go to the cache like kv_store_e4m3's; s goes to
 * k_scales[blk][h][row] (v_scales likewise), blk = slot / block_size,
 * row = slot % block_size: float[num_blocks][num_kv_heads][block_size],
 * device, 4-byte aligned, owned by the caller.
 * k, v, strides, slot_mapping: as for kv_store_e4m3 (slot_mapping required);
 * head_dim 128 or 256.
 */
fp8kv_status kv_store_e4m3_per_token(const fp8kv_cache *cache, const fp8kv_bf16 *k,
                                     const fp8kv_bf16 *v, int64_t k_tok_stride,
                                     int64_t v_tok_stride, const int64_t *slot_mapping,
                                     int64_t num_tokens, float *k_scales, float *v_scales,
                                     void *stream);

/*
 * paged_attn_fp8_decode_per_token -- paged_attn_fp8_decode over a cache
 * written by kv_store_e4m3_per_token: key j of a sequence is
 * k_j = k_scales[j] * dec(k8_j) and v_j = v_scales[j] * dec(v8_j) (its
 * block's entries of the scale arrays), so the score is
 * softmax_scale * q_scale * k_scales[j] * (q8 . k8_j) (+ bias) and the output
 * sum_j P_j * v_scales[j] * v8_j.  In the kernel the V scale is folded into
 * the exponent of P (z_j + log2 v_scales[j] takes part in the running max,
 * so P_j = p_j * v_scales[j] up to a common factor stays in the e4m3 range)
 * and the row sum adds P_j / v_scales[j].
 * Other arguments, the workspace (fp8kv_decode_workspace_size with
 * split_tokens 0) and the result are those of paged_attn_fp8_decode.
 */
fp8kv_status paged_attn_fp8_decode_per_token(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                             int32_t num_q_heads, const int32_t *block_table,
                                             int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                             int32_t num_seqs, float q_scale, float softmax_scale,
                                             const float *k_scales, const float *v_scales,
                                             const fp8kv_bf16 *rel_bias, int64_t bias_tok_stride,
                                             int32_t rel_extent, int32_t window, fp8kv_bf16 *out,
                                             void *workspace, size_t workspace_bytes,
                                             void *stream);

/*
 * attn_fp8_varlen_prefill_per_token -- attn_fp8_varlen_prefill over a cache
 * written by kv_store_e4m3_per_token (local-inference-lab/vllm PR 189: a
 * per-token scale stored with each cached token, read by decode and by the
 * chunked prefill over the cached prefix): key j of a sequence is
 * k_j = k_scales[j] * dec(k8_j) and v_j = v_scales[j] * dec(v8_j) (its
 * block's entries of the scale arrays), so the score is
 * softmax_scale * q_scale * k_scales[j] * (q8 . k8_j) (+ bias) and the
 * output sum_j softmax_j * v_scales[j] * v8_j.  In the kernel the V scale is
 * folded into the exponent of P (P_j = p_j * v_scales[j]), the row sum adds
 * P_j / v_scales[j], and P is always kept in two e4m3 terms.
 * k_scales, v_scales: device float[num_blocks][num_kv_heads][block_size],
 *                4-byte aligned, finite and > 0 where the sequences' keys
 *                are (kv_store_e4m3_per_token writes such values).
 * Other arguments and the result are those of attn_fp8_varlen_prefill (no
 * workspace).  head_dim 128 only (FP8KV_ERR_UNSUPPORTED for 256).
 */
fp8kv_status attn_fp8_varlen_prefill_per_token(const fp8kv_cache *cache, const fp8kv_bf16 *q,
                                               int32_t num_q_heads, const int32_t *cu_seqlens_q,
                                               const int32_t *seq_lens_k,
                                               const int32_t *block_table,
                                               int32_t max_blocks_per_seq, int32_t num_seqs,
                                               int32_t max_seqlen_q, float q_scale,
                                               float softmax_scale, const float *k_scales,
                                               const float *v_scales, const fp8kv_bf16 *rel_bias,
                                               int64_t bias_tok_stride, int32_t rel_extent,
                                               int32_t window, fp8kv_bf16 *out, void *stream);

/*
 * kv_band_counts -- clip and flush-to-zero counters and the round-trip error
 * of quantizing the stored values at one scale: the KV value-range
 * instrument of vLLM PR 54705 (evidence document, Tier 2: exact e4m3 band
 * counters at scale 1.0 and 3.0 over exactly the values at each call's slot
 * mapping).  For every finite element x of a stored token:
 *   count    += 1
 *   nonzero  += x != 0
 *   clipped  += |x / scale| > 448   (the store saturates it to +-448)
 *   flushed  += x != 0 and its e4m3 code is +-0
 *   rt_err_sum += |scale * dec(enc(x / scale)) - x| / |x|   (x != 0)
 * The quotient x / scale and the code are bit-identical to kv_store_e4m3's,
 * so the counts are exact; rt_err_sum is added in parallel, so its last bits
 * depend on the order of the additions.
 * x:             device bf16 [num_tokens] rows of row_elems elements (a
 *                multiple of 16), tok_stride elements apart (a multiple of
 *                8, >= row_elems), 16-byte aligned; NaN and +-Inf are not
 *                counted.
 * slot_mapping:  NULL (every token counts) or device int64 [num_tokens];
 *                tokens with slot < 0 are skipped.
 * scale:         finite and > 0, else FP8KV_ERR_SCALE.
 * counts:        device fp8kv_band_counts, 8-byte aligned; added into, so
 *                zero it before the first call of a measurement.
 * Runs asynchronously on `stream`.
 */
typedef struct {
    unsigned long long count;
    unsigned long long nonzero;
    unsigned long long clipped;
    unsigned long long flushed;
    double rt_err_sum;
} fp8kv_band_counts;

fp8kv_status kv_band_counts(const fp8kv_bf16 *x, int64_t tok_stride, const int64_t *slot_mapping,
                            int64_t num_tokens, int32_t row_elems, float scale,
                            fp8kv_band_counts *counts, void *stream);

/*
 * kv_amax_calibrate -- running max |x| over the tokens that are stored
 * (model card "Qwen3.8-27B-FP8-KVcal", "What it fixes": amax at the
 * cache-write point; vLLM PR 54705 Tier 2: only the values at each call's
 * slot mapping count).
 *   *amax_k_inout = max(*amax_k_inout, max |k|)   (same for v)
 * k, v:          device bf16 rows as in kv_store_e4m3; either may be NULL
 *                (its amax is then left alone).  Strides multiples of 8.
 * slot_mapping:  NULL (every token counts) or device int64 [num_tokens];
 *                tokens with slot < 0 are skipped.
 * amax_*_inout:  device float, >= 0 on entry (e.g. 0 before the first call).
 * NaN elements are ignored.
 */
fp8kv_status kv_amax_calibrate(const fp8kv_bf16 *k, const fp8kv_bf16 *v,
                               int64_t k_tok_stride, int64_t v_tok_stride,
                               const int64_t *slot_mapping, int64_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim,
                               float *amax_k_inout, float *amax_v_inout, void *stream);

/*
 * fp8kv_scale_from_amax -- host-only scale rule.
 *   rule 0: amax/448                (Qwen3.8-27B-FP8-KVcal, "What it fixes")
 *   rule 1: ceil_to_bfloat16(amax/448), as fp32
 *                                   (Qwen3.8-27B-FP8-KVcal, "Rebuild / reproduce")
 *   rule 2: max(1, amax*1.3/448)    (vLLM PR 54705, calibration paragraph)
 * Returns FP8KV_ERR_SCALE when amax is negative, NaN or Inf, or the scale
 * would not be finite and > 0 (amax = 0 under rules 0 and 1),
 * FP8KV_ERR_ARG for an unknown rule or NULL out.
 */
fp8kv_status fp8kv_scale_from_amax(float amax, int32_t rule, float *scale);

/* Bytes of one cache array (K or V): num_blocks*block_size*num_kv_heads*head_dim. */
size_t fp8kv_cache_bytes(int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim);

/*
 * fp8kv_test_drop_first_copy -- test hook for the failure path of the
 * kernels' bounded waits.  With on != 0, the next paged_attn_fp8_decode*
 * launch (one launch only; the request is then cleared) has each CTA's
 * producer skip the TMA copy of its first key tile and the expected-bytes
 * arrival that goes with it.  The MMA warp's wait for that tile then runs
 * out after the wait limit (2 s), the CTA gives up with no copy or MMA in
 * flight, frees its tensor memory and finishes; the call returns normally,
 * its output is unspecified, and the device error word gets
 * FP8KV_DEVERR_WAIT_TIMEOUT.  Nothing faults, traps or hangs, and later
 * calls are unaffected.  on = 0 withdraws a pending request.
 */
fp8kv_status fp8kv_test_drop_first_copy(int32_t on);

/* Reads (and with clear != 0 resets) the current device's error word.
 * Synchronizes the device. */
fp8kv_status fp8kv_device_error(uint32_t *flags, int32_t clear);

/* Static text for a status code. */
const char *fp8kv_status_string(fp8kv_status status);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H */
