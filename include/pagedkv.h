/*
 * pagedkv.h - C ABI of libpagedkv.so: PagedAttention decode over a paged
 * bf16 (or fp8 E4M3) KV cache on NVIDIA GB300 (sm_103a), the kernels that
 * keep the cache valid, a chunked causal prefill over the same cache, and a
 * host-side block manager that builds the tables.
 *
 * Sources (page title, section):
 *  [PA]  "PagedAttention vs Traditional KV Cache: How vLLM Reinvented GPU
 *        Memory for LLM Inference", Section 4 "PagedAttention: How It Works".
 *  [LD]  "LLM Inference Optimization: KV-Cache, PagedAttention, and GPU
 *        Memory Efficiency", section "PagedAttention: OS Concepts Meet GPU
 *        Memory" (block table, kernel outline, copy-on-write).
 *  [KE]  "KV Cache Explained Like You're an LLM Engineer", sections
 *        "Transformer Attention: A Quick Refresher", "What KV Cache Stores",
 *        "Prefill Phase vs. Decode Phase".
 *  [MA]  "Modern AI Infrastructure and Agentic System Design", 9.1 "The key
 *        and value cache" (closed form, copy-on-write figure), "Two workloads
 *        wearing one name" (chunked prefill).
 *  [DR]  "Inference serving: the KV-cache machine", sections "Paged KV:
 *        virtual memory for tokens" and "Continuous batching: the server as
 *        an allocator".
 *
 * Common conventions
 *  - Every pointer argument of the kernel entry points (pa_decode*,
 *    pa_reshape_and_cache*, pa_copy_blocks, pa_prefill_paged*) is DEVICE
 *    memory owned by the caller, 16-byte aligned unless stated otherwise;
 *    bf16 tensors are raw 16-bit patterns. The one exception is the host
 *    side of pa_swap_out_blocks / pa_swap_in_blocks (page-locked HOST
 *    memory). The library allocates no device memory in these calls; it
 *    owns a 4-byte device error word per device and the fixed scratch of
 *    pa_decode_noalloc. The pa_bm_* block manager works on host memory only.
 *  - KV pool layout: k_pool and v_pool are bf16 (or, for the fp8 entry
 *    points, E4M3 bytes)
 *        [num_blocks][n_kv_heads][block_size][head_dim]
 *    so that one (block, kv-head) tile - block_size tokens of one head - is a
 *    contiguous block_size*head_dim*element_size bytes. block_size must be 16 (the
 *    pages' block size), head_dim 64 or 128, n_heads a multiple of
 *    n_kv_heads with group n_heads/n_kv_heads in {1, 2, 4, 8}; query head h
 *    reads KV head h / (n_heads / n_kv_heads).
 *  - A slot is physical_block * block_size + offset ([LD]: logical position p
 *    lives at table[p / block_size], offset p % block_size).
 *  - All kernels run asynchronously on `stream` (NULL = legacy default
 *    stream). Argument errors are returned synchronously and nothing is
 *    launched. A launch failure returns PA_ERR_CUDA. Faults the kernels can
 *    detect only on the device (a block id or slot outside the pool, a wait
 *    that timed out) skip the offending work and set a bit in the device
 *    error word, read and cleared with pa_get_device_error().
 */
#ifndef PAGEDKV_H_
#define PAGEDKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1, /* null/misaligned pointer, negative size, ... */
    PA_ERR_UNSUPPORTED = -2, /* valid but not built: head_dim, block_size, group */
    PA_ERR_WORKSPACE = -3,   /* workspace missing or too small */
    PA_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
    PA_ERR_DEVICE = -5,      /* device error word was non-zero */
    PA_ERR_OOM = -6,         /* block manager: free list cannot supply the blocks */
    PA_ERR_REFCOUNT = -7,    /* block manager: unknown sequence / refcount misuse */
    PA_ERR_CAPACITY = -8     /* an output buffer given by the caller is too small */
};

/* Bits of the device error word. */
enum pa_device_error {
    PA_DEVERR_BLOCK_ID = 1, /* a block-table entry outside [0, num_blocks) */
    PA_DEVERR_SLOT = 2,     /* a slot >= num_blocks * block_size */
    PA_DEVERR_TIMEOUT = 4,  /* an mbarrier / async-copy wait ran out */
    PA_DEVERR_PAIR = 8,     /* a copy_blocks pair outside the pool */
    PA_DEVERR_CONTEXT = 16, /* a context length beyond 16*max_blocks_per_seq or
                               max_context_len (the excess is not attended), or a
                               prefill chunk longer than its context */
    PA_DEVERR_LAYOUT = 32,  /* the shared-memory base was not 1024-byte aligned
                               (prefill; nothing computed) */
    PA_DEVERR_RANGE = 64,   /* a prefill output (or split partial) was not finite:
                               a V element beyond +-65504*2^8 in a key tile the
                               chunk reads (the P.V product stages V in fp16), or
                               non-finite inputs */
    PA_DEVERR_PLAN = 128    /* a pa_decode_planned item outside the call's bounds
                               (that CTA did nothing) */
};

/* ------------------------------------------------------------------ decode */

/*
 * Workspace bytes pa_decode needs for this batch shape (0 when every context
 * fits in one partition, in which case workspace may be NULL). The workspace
 * holds fp32 split-K partials: running max m and sum l per (seq, q-head,
 * partition) and the unnormalised output per (seq, q-head, partition, dim).
 * partition_tokens: tokens per context partition, a multiple of 64 in
 * [64, 2048]; 0 selects the library default (pa_decode_partition_tokens),
 * and sizes the workspace for 512 tokens, which covers every default (fewer,
 * larger partitions fit in the same bytes).
 */
size_t pa_decode_workspace_bytes(int n_seqs, int n_heads, int head_dim,
                                 int max_context_len, int partition_tokens);

/*
 * The partition size (tokens per context partition) pa_decode, pa_decode_fp8
 * (elem_bytes 1) and pa_decode_window (window >= 0; -1 for none) use when
 * partition_tokens is 0, for this batch shape on the current device: 1024 on
 * the tensor-core kernel. On the CUDA-core kernel, with context =
 * max_context_len (or the window's span): when n_seqs x n_kv_heads is at
 * least the device's SM count and at most its CTA slots (one wave) and the
 * context is at most 2048 tokens, the context rounded up to 64 (one
 * partition per sequence, no split-K merge); otherwise the multiple of 64 in
 * [512, 1024] whose grid of n_seqs x n_kv_heads x ceil(context / size) CTAs
 * fills the last wave of the device's CTA slots best, the smallest on ties.
 * Every such size needs no more workspace than
 * pa_decode_workspace_bytes(..., 0) gives. Negative status for arguments the
 * decode entry points would reject.
 */
int pa_decode_partition_tokens(int n_seqs, int n_heads, int n_kv_heads, int head_dim,
                               int max_context_len, int window, int elem_bytes);

/*
 * PagedAttention decode ([LD] kernel outline; [KE] attention formula):
 * for every sequence b and query head h,
 *     out[b][h][:] = softmax_t( scale * q[b][h] . K_b[t] ) . V_b[t],
 *                    t = 0 .. context_lens[b]-1,
 * where K_b[t] / V_b[t] is token t of sequence b, stored in physical block
 * block_tables[b][t / 16] at offset t % 16, for KV head h / group.
 *
 *  out            bf16 [n_seqs][n_heads][head_dim]   (written; must not alias q)
 *  q              bf16 [n_seqs][n_heads][head_dim]
 *  k_pool, v_pool bf16 pool layout above (read only)
 *  block_tables   int32 [n_seqs][max_blocks_per_seq]; entries past
 *                 ceil(context_lens[b]/16) are never read
 *  context_lens   int32 [n_seqs]: valid tokens of each sequence, including
 *                 any token written this step; <= 0 gives a zero output row;
 *                 must be <= max_context_len and <= 16*max_blocks_per_seq
 *  scale          softmax scale (typically 1/sqrt(head_dim))
 *  max_context_len upper bound of context_lens (sizes the partition grid)
 *  num_blocks     pool size in blocks (bounds check of table entries)
 *  workspace      device scratch of >= pa_decode_workspace_bytes(...) bytes,
 *                 caller-owned; contents need no initialisation
 * Arithmetic: bf16 inputs, fp32 dot products, fp32 online softmax (base-2
 * exponent with scale*log2(e) folded into q), fp32 split-K merge, bf16 output
 * rounded to nearest even.
 * Kernels: groups of up to 4 query heads per KV head use warp-shuffle fp32 dot
 * products on the CUDA cores. A group of 8 at head_dim 128 would make that
 * kernel bound by its FMA work, far below HBM speed, so it runs its two
 * products as warp-level tensor-core MMAs (see pa_decode_tc), unless the pool
 * has more than 2^31 - 16 rows of 16 tokens x KV heads. pa_decode_fp8 does the
 * same for every group at head_dim 128.
 */
int pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
              const int32_t* block_tables, const int32_t* context_lens, float scale,
              int n_heads, int n_kv_heads, int head_dim, int block_size,
              int n_seqs, int max_blocks_per_seq, int max_context_len, int num_blocks,
              void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* pa_decode with an explicit partition size (see pa_decode_workspace_bytes). */
int pa_decode_ex(void* out, const void* q, const void* k_pool, const void* v_pool,
                 const int32_t* block_tables, const int32_t* context_lens, float scale,
                 int n_heads, int n_kv_heads, int head_dim, int block_size,
                 int n_seqs, int max_blocks_per_seq, int max_context_len, int num_blocks,
                 int partition_tokens, void* workspace, size_t workspace_bytes,
                 pa_stream_t stream);

/*
 * pa_decode_ex on the tensor-core partition kernel at every group size. Each
 * 16-token block's products are warp-level mma.sync instructions:
 *     S[16 x 16] = Q[16 x 128] . K^T  (the group's G heads are the first G of
 *                                      16 rows; the rest are zero)
 *     O[16 x 128] += P . V            (P as two bf16 terms, P_hi = p
 *                                      truncated and P_lo = the rounded rest)
 * with fp32 accumulation. K and V tiles arrive by 2-D TMA in 128-byte-swizzled
 * shared memory. Softmax, partitions, workspace, errors and the split-K merge
 * are as for pa_decode_ex.
 * Requires head_dim 128 and a pool of at most 2^31 - 16 rows (num_blocks *
 * n_kv_heads * 16), else PA_ERR_UNSUPPORTED.
 */
int pa_decode_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                 const int32_t* block_tables, const int32_t* context_lens, float scale,
                 int n_heads, int n_kv_heads, int head_dim, int block_size,
                 int n_seqs, int max_blocks_per_seq, int max_context_len, int num_blocks,
                 int partition_tokens, void* workspace, size_t workspace_bytes,
                 pa_stream_t stream);

/*
 * Allocation-free pa_decode. The pages have no counterpart: this entry point
 * exists for callers that cannot allocate device memory for pa_decode's
 * workspace - a runtime that gave all free HBM to its KV pool, a decode loop
 * that must not call cudaMalloc/cudaFree (they can synchronize the device),
 * or a host that only holds raw pointers. Same arguments and result as
 * pa_decode (default partition size), minus the workspace: the split-K
 * scratch is a fixed 32 MiB device array inside the library, held by every
 * device that loads it until the process exits. The call allocates nothing.
 *  - Returns PA_ERR_WORKSPACE, launching nothing, when
 *    pa_decode_workspace_bytes(n_seqs, n_heads, head_dim, max_context_len, 0)
 *    exceeds 32 MiB.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents (nothing in it needs to start at zero); calls whose kernels
 *    overlap on the GPU race on it.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *    The lookup is cached per device and per context, and is thread-safe;
 *    after a device reset the first call in the new context looks the
 *    address up again (and the array's contents start over).
 */
int pa_decode_noalloc(void* out, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, const int32_t* context_lens, float scale,
                      int n_heads, int n_kv_heads, int head_dim, int block_size,
                      int n_seqs, int max_blocks_per_seq, int max_context_len, int num_blocks,
                      pa_stream_t stream);

/* --------------------------------------------------------- cache upkeep */

/*
 * reshape_and_cache ([KE] "What KV Cache Stores": append the new token's K/V;
 * [DR] slot = table[p / 16], offset p % 16): for t < n_tokens with
 * slot_mapping[t] >= 0, copy k[t][h][:] to k_pool[slot/16][h][slot%16][:] and
 * v[t][h][:] to v_pool likewise, for every KV head h. Bit copy.
 *  k, v          bf16 [n_tokens][n_kv_heads][head_dim]
 *  slot_mapping  int64 [n_tokens]; negative = skip (padding);
 *                >= num_blocks*16 sets PA_DEVERR_SLOT and is skipped
 * Two tokens naming the same slot race (one of them wins).
 */
int pa_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                         const int64_t* slot_mapping, int n_tokens, int n_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_stream_t stream);

/*
 * copy_blocks ([MA] copy-on-write figure; [LD] only the diverging block is
 * copied): for each pair i, the whole block block_mapping[2i] (all KV heads,
 * all 16 slots) is copied to block block_mapping[2i+1], in k_pool and v_pool.
 * Bit copy. Destinations must be distinct and must not be sources of other
 * pairs. A pair outside [0, num_blocks) sets PA_DEVERR_PAIR and is skipped.
 *  block_mapping int64 [n_pairs][2] (src, dst), device memory
 * The pools are bf16 (2-byte elements); an fp8 pool takes pa_copy_blocks_ex.
 */
int pa_copy_blocks(void* k_pool, void* v_pool, const int64_t* block_mapping, int n_pairs,
                   int n_kv_heads, int head_dim, int block_size, int num_blocks,
                   pa_stream_t stream);

/*
 * pa_copy_blocks for a pool of either element size: elem_bytes 2 for a bf16
 * pool (the same as pa_copy_blocks), 1 for an fp8 (E4M3) pool, whose blocks
 * hold n_kv_heads * 16 * head_dim bytes. Any other elem_bytes returns
 * PA_ERR_INVALID_ARG. Pools 16-byte aligned. The copy-on-write pairs the
 * block manager emits do not depend on the cache's element type.
 */
int pa_copy_blocks_ex(void* k_pool, void* v_pool, const int64_t* block_mapping, int n_pairs,
                      int n_kv_heads, int head_dim, int block_size, int elem_bytes, int num_blocks,
                      pa_stream_t stream);

/* ----------------------------------------------------- swap (preemption) */

/*
 * Whole-block copies between the pools and host memory for preemption by
 * swapping ([MA] 9.1 "Batching and the scheduler": swapping costs a transfer
 * and no compute; [DR] "Paged KV: virtual memory for tokens": swap out the
 * private blocks, reload them anywhere). One launch moves n_blocks blocks,
 * K and V, every KV head and slot of each, in bits.
 *  block_ids     int32 [n_blocks] pool block ids, DEVICE memory (e.g. the
 *                ids pa_bm_swap_out / pa_bm_swap_in returned, copied over);
 *                an id outside [0, num_blocks) sets PA_DEVERR_BLOCK_ID and
 *                that block is skipped
 *  host_k,host_v HOST memory, page-locked (cudaHostAlloc, or registered with
 *                cudaHostRegister) so that the device reaches it directly;
 *                16-byte aligned; block i of the transfer occupies bytes
 *                [i * B, (i + 1) * B), B = n_kv_heads * 16 * head_dim *
 *                elem_bytes (the pool's block layout)
 *  elem_bytes    2 for a bf16 pool, 1 for an fp8 pool
 * pa_swap_out_blocks: host[i] := pool block block_ids[i].
 * pa_swap_in_blocks:  pool block block_ids[i] := host[i].
 * Asynchronous on stream: the host copy is complete once the stream is; a
 * swap-in must be ordered before any kernel that reads those blocks.
 */
int pa_swap_out_blocks(const void* k_pool, const void* v_pool, const int32_t* block_ids, int n_blocks,
                       void* host_k, void* host_v, int n_kv_heads, int head_dim, int block_size,
                       int elem_bytes, int num_blocks, pa_stream_t stream);
int pa_swap_in_blocks(const void* host_k, const void* host_v, void* k_pool, void* v_pool,
                      const int32_t* block_ids, int n_blocks, int n_kv_heads, int head_dim,
                      int block_size, int elem_bytes, int num_blocks, pa_stream_t stream);

/* ------------------------------------------------------ sliding window */

/*
 * Sliding-window decode ([KE] "Sliding Window Attention": token i attends to
 * tokens [i - W, i], so the cache it needs is O(W)): as pa_decode_ex, but the
 * query at position i = context_lens[b] - 1 attends only to positions
 * max(0, i - window) .. i (window >= 0, else PA_ERR_INVALID_ARG).
 *     out[b][h] = sum_{i-W <= t <= i} softmax_t(scale * q[b][h] . K_b[t]) V_b[t]
 * Table entries of blocks that lie wholly before the window are never read
 * (they may be -1, see pa_bm_release_before); the block that holds position
 * i - W must be present. Workspace as for pa_decode_ex (sized by
 * max_context_len, an upper bound for any window).
 */
int pa_decode_window(void* out, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, const int32_t* context_lens, float scale,
                     int n_heads, int n_kv_heads, int head_dim, int block_size, int n_seqs,
                     int max_blocks_per_seq, int max_context_len, int num_blocks, int window,
                     int partition_tokens, void* workspace, size_t workspace_bytes,
                     pa_stream_t stream);

/* ------------------------------------------------- fp8 (E4M3) KV cache */

/*
 * An fp8 cache stores every K and V element as one E4M3 code (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, 0x7F/0xFF NaN,
 * largest magnitude 448) with one fp32 scale per KV head for K and one for V;
 * an element stands for decode(code) * scale ([DR] "What insiders know": fp8
 * KV with per-head scale factors; [KE] "KV Cache Quantization": one byte per
 * element and a scale). The pool layout is the bf16 one with 1-byte elements:
 *     uint8 [num_blocks][n_kv_heads][block_size][head_dim]
 * so a block holds half the bytes.
 *  k_scale, v_scale  fp32 [n_kv_heads], device memory, 4-byte aligned, > 0.
 */

/*
 * Cache write for an fp8 cache: as pa_reshape_and_cache, but element x of
 * k[t][h][:] (bf16) is stored as the E4M3 code of the fp32 quotient
 * x / k_scale[h] (IEEE division, round to nearest even, finite values beyond
 * +-448 saturate to +-448), and likewise for v with v_scale.
 *  k, v          bf16 [n_tokens][n_kv_heads][head_dim], 16-byte aligned
 *  k_pool,v_pool uint8 pools (8-byte aligned)
 *  slot_mapping  int64 [n_tokens]; negative = skip; out of range sets
 *                PA_DEVERR_SLOT and is skipped
 */
int pa_reshape_and_cache_fp8(const void* k, const void* v, void* k_pool, void* v_pool,
                             const int64_t* slot_mapping, const float* k_scale,
                             const float* v_scale, int n_tokens, int n_kv_heads, int head_dim,
                             int block_size, int num_blocks, pa_stream_t stream);

/*
 * Decode over an fp8 cache: pa_decode_ex with K and V read as E4M3 codes
 * times their KV head's scale,
 *     out[b][h] = sum_t softmax_t(scale * q[b][h] . Kd_b[t]) Vd_b[t],
 *     Kd = decode(k code) * k_scale[kv head], Vd = decode(v code) * v_scale.
 * q and out are bf16 as in pa_decode; the workspace is sized by
 * pa_decode_workspace_bytes (the same formula); partition_tokens as in
 * pa_decode_ex. Pools must be 16-byte aligned.
 * At head_dim 128 the products run on the tensor-core kernel (fp16 MMAs with
 * fp32 accumulate: every E4M3 value is an fp16 value, q is converted to fp16
 * once, exact for |q| within the fp16 range, and P enters as one fp16 term,
 * within 2^-12 of p, which adds at most 2^-12 * max|v| to an output);
 * at head_dim 64 on the CUDA-core kernel (fp32 dot products).
 */
int pa_decode_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                  const float* k_scale, const float* v_scale, const int32_t* block_tables,
                  const int32_t* context_lens, float scale, int n_heads, int n_kv_heads,
                  int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                  int max_context_len, int num_blocks, int partition_tokens, void* workspace,
                  size_t workspace_bytes, pa_stream_t stream);

/*
 * Host-side work plan for one decode call, for callers that hold the batch's
 * context lengths on the host (a block manager does): the call's work items,
 * one per CTA, each a (partition, KV head, sequence) of the partition
 * kernel, the longest partitions first (the short last partitions of the
 * sequences run at the end, where a grid in plain order can end on full
 * partitions that started late). No device work; the plan stays valid for
 * any call whose lengths give every sequence the same number of partitions.
 *  context_lens   HOST int32 [n_seqs]: the lengths the call will get
 *  other arguments as the decode entry points (num_blocks and elem_bytes
 *                 pick the kernel and so the default partition size;
 *                 window -1 for none; partition_tokens 0 = default)
 *  items          HOST int32 [cap][4], written as (partition, kv head,
 *                 sequence, 0); NULL to query the count
 * Returns the item count, or a negative status (PA_ERR_CAPACITY when cap is
 * too small).
 */
int pa_decode_plan(const int32_t* context_lens, int n_seqs, int n_heads, int n_kv_heads, int head_dim,
                   int max_blocks_per_seq, int max_context_len, int num_blocks, int window,
                   int elem_bytes, int partition_tokens, int32_t* items, int cap);

/*
 * pa_decode_ex (k_scale, v_scale NULL), pa_decode_fp8 (both given) or, with
 * window >= 0, pa_decode_window, run from a plan: CTA i computes item i of
 * items (DEVICE int32 [n_items][4], 16-byte aligned), which must be
 * pa_decode_plan's output for the same lengths and arguments. The results
 * are bit-identical to the unplanned call's. An item outside the call's
 * bounds sets PA_DEVERR_PLAN and is skipped; a plan missing items leaves
 * their outputs unwritten.
 */
int pa_decode_planned(void* out, const void* q, const void* k_pool, const void* v_pool,
                      const float* k_scale, const float* v_scale, const int32_t* block_tables,
                      const int32_t* context_lens, float scale, int n_heads, int n_kv_heads,
                      int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                      int max_context_len, int num_blocks, int window, int partition_tokens,
                      const int32_t* items, int n_items, void* workspace, size_t workspace_bytes,
                      pa_stream_t stream);

/* ------------------------------------------------------- chunked prefill */

/*
 * Causal attention of prompt chunks over the paged cache ([MA] "Two workloads
 * wearing one name": chunked prefill; [KE] "Prefill Phase vs. Decode Phase").
 * Sequence s owns query rows q_start_loc[s] .. q_start_loc[s+1]-1 (L_s rows);
 * its chunk occupies the last L_s of its context_lens[s] tokens, which must
 * already be in the cache (write them with pa_reshape_and_cache first). Row
 * i of the chunk sits at position p = context_lens[s] - L_s + i and attends to
 * positions 0..p:
 *     out[r][h][:] = softmax_{t<=p}( scale * q[r][h] . K_s[t] ) . V_s[t].
 *  out, q        bf16 [q_start_loc[n_seqs]][n_heads][head_dim]
 *  q_start_loc   int32 [n_seqs+1], non-decreasing, q_start_loc[0] = 0
 *  context_lens  int32 [n_seqs], >= L_s
 *  max_chunk_len upper bound of L_s
 * head_dim 64 or 128 and the group n_heads/n_kv_heads 1, 2, 4 or 8, else
 * PA_ERR_UNSUPPORTED. The workspace size of pa_prefill_paged_ex does not
 * depend on head_dim (a partial row holds up to 128 dims).
 * QK^T and PV run on the tcgen05 tensor cores with fp32 accumulation in
 * tensor memory; softmax in fp32. QK^T takes bf16 q and K. PV takes P rounded
 * to fp16 (within 2^-12 of p) and V staged in fp16 as v * 2^-8, which holds
 * every bf16 significand for 2^-6 <= |v| <= 65504 * 2^8. The P rounding adds
 * at most 2^-12 * max|v| to an output. Smaller |v| lose bits, at an absolute
 * error of at most 2^-17. Larger |v| in a key tile the chunk reads make the
 * output non-finite and set PA_DEVERR_RANGE.
 */
int pa_prefill_paged(void* out, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, const int32_t* context_lens,
                     const int32_t* q_start_loc, float scale, int n_heads, int n_kv_heads,
                     int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                     int max_chunk_len, int num_blocks, pa_stream_t stream);

/*
 * pa_prefill_paged with the key range of query-tile pairs split into pieces,
 * so that the work fills the GPU's SMs evenly (one prefill CTA runs per SM).
 * Each piece keeps its un-normalised output, reference maximum and sum in
 * the workspace; a merge kernel combines the pieces (O = sum_p O_p 2^(m_p -
 * M), l = sum_p l_p 2^(m_p - M), out = O / l).
 *  splits     0 = balanced: a small planning kernel lists the pairs with
 *             rows; all but the last partial wave's run whole, those of the
 *             last partial wave are cut into a few equal key ranges, and one
 *             CTA per SM takes list entries in order from a counter;
 *             1 = no split (no workspace needed); 2..64 = every pair cut
 *             into that many equal pieces
 *  workspace  DEVICE memory, 16-byte aligned, of at least
 *             pa_prefill_workspace_bytes(n_seqs, n_heads, n_kv_heads,
 *             max_chunk_len, splits) bytes (query it with the same
 *             arguments and the same current device); PA_ERR_WORKSPACE if
 *             missing or too small. Contents need no initialisation.
 * pa_prefill_workspace_bytes returns 0 for arguments pa_prefill_paged_ex
 * would reject, for splits = 1, and for splits = 0 when no device is
 * visible (the balanced size depends on the device's SM count).
 */
size_t pa_prefill_workspace_bytes(int n_seqs, int n_heads, int n_kv_heads, int max_chunk_len, int splits);
int pa_prefill_paged_ex(void* out, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* block_tables, const int32_t* context_lens,
                        const int32_t* q_start_loc, float scale, int n_heads, int n_kv_heads,
                        int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                        int max_chunk_len, int num_blocks, int splits, void* workspace,
                        size_t workspace_bytes, pa_stream_t stream);

/* ----------------------------------------------------------- diagnostics */

/* Reads the current device's error word into *flags_out (a PA_DEVERR_* mask)
 * and clears it. Synchronises with the device. */
int pa_get_device_error(int* flags_out);

/* Self-test of failure detection (no counterpart on the pages): launches a
 * one-thread kernel that waits on an mbarrier nothing arrives on, bounded to
 * limit_us microseconds (1 .. 10^7). The wait gives up, sets PA_DEVERR_TIMEOUT
 * in the device error word and returns; the context stays usable. Used by
 * the tests to show that every bounded wait ends without a fault or hang. */
int pa_selftest_wait_timeout(int limit_us, pa_stream_t stream);

/* Static string for a status code. */
const char* pa_status_string(int status);

/* ------------------------------------------------------ host block manager */
/*
 * Builds block tables, slot mappings and copy-on-write pairs on the host
 * ([PA] free list and append-allocates-on-full; [DR] refcounts, fork aliasing,
 * copy-on-write; [MA] copy-on-write figure). Not thread-safe; one manager per
 * pool. refcount(b) = number of block tables that reference block b; a block
 * returns to the free list when its refcount reaches 0. Allocation pops the
 * most recently freed block (LIFO). Every call that can fail is all-or-nothing.
 */
typedef struct pa_bm pa_bm;

/* NULL on bad sizes or allocation failure. */
pa_bm* pa_bm_create(int num_blocks, int block_size);
void pa_bm_destroy(pa_bm* bm);

/* New empty sequence. PA_ERR_REFCOUNT if seq_id exists. */
int pa_bm_add_seq(pa_bm* bm, int64_t seq_id);

/*
 * Appends n tokens to seq_id. slots_out[0..n) receives each token's slot.
 * If the sequence's last block is partially filled and shared (refcount > 1),
 * it is first copied: a fresh block replaces it in this table, the old one is
 * decref'd, and the pair (old, fresh) is written to cow_pairs_out (int64
 * [cap][2]); *n_cow_out receives the number of pairs (0 or 1). New blocks are
 * taken from the free list when the last block is full. PA_ERR_OOM (no state
 * change) if the free list cannot supply every block needed; PA_ERR_CAPACITY
 * if cow_cap < 1 and a copy would be needed.
 */
int pa_bm_append_tokens(pa_bm* bm, int64_t seq_id, int n, int64_t* slots_out,
                        int64_t* cow_pairs_out, int cow_cap, int* n_cow_out);

/* Forces logical block `logical_block` of seq_id to be private: if shared it is
 * copied to a fresh block (pair written to pair_out[2], *n_out = 1), else
 * *n_out = 0. */
int pa_bm_make_private(pa_bm* bm, int64_t seq_id, int logical_block, int64_t* pair_out,
                       int* n_out);

/* child's table aliases parent's blocks; each block's refcount += 1. */
int pa_bm_fork(pa_bm* bm, int64_t parent, int64_t child);

/* Drops seq_id; each of its blocks is decref'd and freed at refcount 0. */
int pa_bm_free_seq(pa_bm* bm, int64_t seq_id);

/*
 * Window release ([KE] "Sliding Window Attention"): drops every block of the
 * sequence that lies wholly before logical position first_pos (clamped to
 * [0, len]); its table entry becomes -1 (a hole, kept so positions keep
 * their logical block) and its refcount drops (free list at zero). Holes are
 * skipped by fork and free and reported as -1 by pa_bm_block_table and
 * pa_bm_build_batch; pa_bm_make_private on a hole returns
 * PA_ERR_INVALID_ARG. *n_released_out = entries dropped by this call.
 */
int pa_bm_release_before(pa_bm* bm, int64_t seq_id, int64_t first_pos, int* n_released_out);

/*
 * Preemption by swapping ([MA] 9.1 "Batching and the scheduler": a preempted
 * sequence is recomputed or swapped to host memory; [DR] "Paged KV: virtual
 * memory for tokens": swap out the private blocks, reload them anywhere).
 * pa_bm_swap_out releases the sequence's private tail - the longest run of
 * trailing blocks only its table holds - writes those block ids to
 * blocks_out (logical order; copy their contents out with pa_swap_out_blocks
 * before anything reuses them) and marks the sequence swapped: it keeps its
 * length and shared head, and append, copy, fork, release, cache
 * registration and pa_bm_build_batch on it return PA_ERR_INVALID_ARG until
 * pa_bm_swap_in allocates that many fresh blocks (all-or-nothing: PA_ERR_OOM
 * changes nothing), appends them and writes them to blocks_out (copy the
 * contents back with pa_swap_in_blocks). *n_out = the tail's block count;
 * PA_ERR_CAPACITY (nothing changed) when cap is smaller.
 */
int pa_bm_swap_out(pa_bm* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n_out);
int pa_bm_swap_in(pa_bm* bm, int64_t seq_id, int32_t* blocks_out, int cap, int* n_out);

/*
 * Prefix caching ("Modular LLM Inference Engine from Scratch", section
 * "Prefix caching - skip recomputing the same prompt": a hash-based LRU cache
 * whose lookup finds the longest cached prefix of whole blocks; [DR], [KE]
 * "Prefix Caching": a shared prompt's KV is computed once). An entry is one
 * full block, identified by all tokens from position 0 through its last
 * (a 128-bit chained hash of them); each entry holds one reference to its
 * block. When an allocation (append, copy-on-write, make_private) finds the
 * free list empty it evicts entries from the least-recently-used end,
 * skipping blocks a table still holds; appends stay all-or-nothing over
 * free + evictable blocks.
 *
 * pa_bm_cache_blocks: registers the sequence's full blocks (the first
 * min(n_tokens, len) / block_size, tokens = the sequence's token ids from
 * position 0); new entries go to the most-recently-used end, entries that
 * exist are left in place; *n_added_out = entries added.
 * pa_bm_add_seq_cached: creates seq_id on the longest run of leading blocks
 * whose prefixes of tokens[0..n_tokens) are cached (incref'd, refreshed in
 * block order); *n_cached_out = tokens it already holds (a multiple of the
 * block size) - append the rest with pa_bm_append_tokens.
 * pa_bm_num_cached: number of entries.
 */
int pa_bm_cache_blocks(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int64_t n_tokens,
                       int* n_added_out);
int pa_bm_add_seq_cached(pa_bm* bm, int64_t seq_id, const int32_t* tokens, int64_t n_tokens,
                         int64_t* n_cached_out);
int pa_bm_num_cached(const pa_bm* bm);

/* Copies seq_id's table into out[0..cap); *n_out = its length. PA_ERR_CAPACITY
 * (with *n_out set) if cap is too small. */
int pa_bm_block_table(const pa_bm* bm, int64_t seq_id, int32_t* out, int cap, int* n_out);

/* Number of tokens held by seq_id, or a negative status. */
int64_t pa_bm_seq_len(const pa_bm* bm, int64_t seq_id);

int pa_bm_num_free(const pa_bm* bm);
/* Refcount of block_id, or a negative status if out of range. */
int pa_bm_refcount(const pa_bm* bm, int block_id);

/*
 * Fills a padded int32 [n][max_blocks] table array (row i = seq_ids[i]'s
 * table, -1 padded) and int32 context_lens[n] for a batch, ready for a
 * host->device copy. PA_ERR_CAPACITY if a table is longer than max_blocks.
 */
int pa_bm_build_batch(const pa_bm* bm, const int64_t* seq_ids, int n, int max_blocks,
                      int32_t* tables_out, int32_t* context_lens_out);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H_ */
