// attn_prefill.cu -- varlen prefill attention over the e4m3 cache (kernel to
// follow; the entry point validates and reports the path as unsupported).
#include "common.cuh"

extern "C" fp8kv_status attn_fp8_varlen_prefill(
    const fp8kv_cache *cache, const fp8kv_bf16 *q, int32_t num_q_heads,
    const int32_t *cu_seqlens_q, const int32_t *seq_lens_k, const int32_t *block_table,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t max_seqlen_q, float q_scale,
    float k_scale, float v_scale, float softmax_scale, const fp8kv_bf16 *rel_bias,
    int64_t bias_tok_stride, int32_t rel_extent, int32_t window, fp8kv_bf16 *out, void *workspace,
    size_t workspace_bytes, void *stream) {
    (void)cache; (void)q; (void)num_q_heads; (void)cu_seqlens_q; (void)seq_lens_k;
    (void)block_table; (void)max_blocks_per_seq; (void)num_seqs; (void)max_seqlen_q;
    (void)q_scale; (void)k_scale; (void)v_scale; (void)softmax_scale; (void)rel_bias;
    (void)bias_tok_stride; (void)rel_extent; (void)window; (void)out; (void)workspace;
    (void)workspace_bytes; (void)stream;
    return FP8KV_ERR_UNSUPPORTED;
}
