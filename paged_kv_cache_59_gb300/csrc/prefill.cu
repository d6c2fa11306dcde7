// Chunked causal prefill over the paged cache (tcgen05 path): placeholder
// until the tensor-core kernel lands; reports the configuration as
// unsupported so no caller mistakes it for a result.
#include "pa_common.cuh"

extern "C" int pa_prefill_paged(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* q_start_loc, float scale, int n_heads, int n_kv_heads,
                                int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                                int max_chunk_len, int num_blocks, pa_stream_t stream) {
    (void)out; (void)q; (void)k_pool; (void)v_pool; (void)block_tables; (void)context_lens;
    (void)q_start_loc; (void)scale; (void)n_heads; (void)n_kv_heads; (void)head_dim;
    (void)block_size; (void)n_seqs; (void)max_blocks_per_seq; (void)max_chunk_len;
    (void)num_blocks; (void)stream;
    return PA_ERR_UNSUPPORTED;
}
