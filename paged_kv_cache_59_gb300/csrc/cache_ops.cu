// Cache upkeep kernels: new-token scatter (reshape_and_cache, and its fp8
// variant that encodes while it scatters), the copy-on-write block copy
// (copy_blocks), and the swap of whole blocks to and from page-locked host
// memory for preemption ("Modern AI Infrastructure and Agentic System Design",
// 9.1 "Batching and the scheduler"; "Inference serving: the KV-cache machine",
// section "Paged KV: virtual memory for tokens"). The first three are bound
// by HBM bandwidth, the swap by the host link.
//
// reshape_and_cache: each decode step appends the new token's K and V to the
// cache ("KV Cache Explained Like You're an LLM Engineer", section "What KV
// Cache Stores"); in the paged cache the destination is the token's slot,
// block table[p / 16] at offset p % 16 ("Inference serving: the KV-cache
// machine", section "Paged KV: virtual memory for tokens").
// copy_blocks: a write to a shared block first copies the whole block to a
// fresh one ("Modern AI Infrastructure and Agentic System Design", 9.1, the
// copy-on-write figure).
#include "pa_common.cuh"

namespace {

constexpr int kBS = 16;

// One thread moves one 16-byte chunk (8 dims) of one (token, KV head) row of
// K and the same chunk of V. Threads of a warp cover consecutive chunks of
// consecutive rows, so loads and stores are fully coalesced.
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                         uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                         const int64_t* __restrict__ slots, long long n_chunks, int n_kv_heads,
                         int chunks_per_head, long long pool_slots, unsigned int* err) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    pa::launch_dependents();     // the next kernel (decode, prefill) may be scheduled
    pa::grid_dependency_wait();  // earlier readers of the pool are complete
    if (i >= n_chunks) return;
    const int per_token = n_kv_heads * chunks_per_head;
    const long long t = i / per_token;
    const int rem = (int)(i - t * per_token);
    const int h = rem / chunks_per_head;
    const int c = rem - h * chunks_per_head;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= pool_slots) {
        if (rem == 0) pa::set_error(err, PA_DEVERR_SLOT);
        return;
    }
    const long long blk = slot / kBS, off = slot % kBS;
    const long long dst = ((blk * n_kv_heads + h) * kBS + off) * chunks_per_head + c;
    k_pool[dst] = k[i];
    v_pool[dst] = v[i];
}

// fp8 (E4M3) cache write: one thread encodes one 8-element chunk of one
// (token, KV head) row of K and the same chunk of V. Each bf16 element x
// becomes the E4M3 code of the fp32 quotient x / scale[head] (IEEE division,
// then round to nearest even with saturation at +-448), 8 bytes per chunk.
__device__ __forceinline__ uint32_t e4m3x4_from_f32(float a, float b, float c, float d) {
    // cvt.rn.satfinite.e4m3x2.f32 puts its first source in the upper byte
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 t;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\t"
        "cvt.u32.u16 %0, t;\n\t}"
        : "=r"(lo)
        : "f"(a), "f"(b));
    asm("{\n\t.reg .b16 t;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\t"
        "cvt.u32.u16 %0, t;\n\t}"
        : "=r"(hi)
        : "f"(c), "f"(d));
    return lo | (hi << 16);
}

__device__ __forceinline__ uint2 encode_chunk(const uint4 w, float s) {
    const float2 x0 = pa::bf16x2_to_float2(w.x), x1 = pa::bf16x2_to_float2(w.y);
    const float2 x2 = pa::bf16x2_to_float2(w.z), x3 = pa::bf16x2_to_float2(w.w);
    uint2 r;
    r.x = e4m3x4_from_f32(__fdiv_rn(x0.x, s), __fdiv_rn(x0.y, s), __fdiv_rn(x1.x, s), __fdiv_rn(x1.y, s));
    r.y = e4m3x4_from_f32(__fdiv_rn(x2.x, s), __fdiv_rn(x2.y, s), __fdiv_rn(x3.x, s), __fdiv_rn(x3.y, s));
    return r;
}

__global__ void __launch_bounds__(256)
reshape_and_cache_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             uint2* __restrict__ k_pool, uint2* __restrict__ v_pool,
                             const int64_t* __restrict__ slots, const float* __restrict__ k_scale,
                             const float* __restrict__ v_scale, long long n_chunks, int n_kv_heads,
                             int chunks_per_head, long long pool_slots, unsigned int* err) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    pa::launch_dependents();
    pa::grid_dependency_wait();
    if (i >= n_chunks) return;
    const int per_token = n_kv_heads * chunks_per_head;
    const long long t = i / per_token;
    const int rem = (int)(i - t * per_token);
    const int h = rem / chunks_per_head;
    const int c = rem - h * chunks_per_head;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= pool_slots) {
        if (rem == 0) pa::set_error(err, PA_DEVERR_SLOT);
        return;
    }
    const long long blk = slot / kBS, off = slot % kBS;
    const long long dst = ((blk * n_kv_heads + h) * kBS + off) * chunks_per_head + c;
    k_pool[dst] = encode_chunk(k[i], k_scale[h]);
    v_pool[dst] = encode_chunk(v[i], v_scale[h]);
}

// grid.x = pair, grid.y = slice of the block; each CTA copies its slice of K
// and of V for one pair. A block is n_kv_heads*16*head_dim*2 bytes.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                   const int64_t* __restrict__ pairs, int chunks_per_block, int num_blocks,
                   unsigned int* err) {
    const int pr = blockIdx.x;
    const int64_t src = pairs[2 * pr], dst = pairs[2 * pr + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) pa::set_error(err, PA_DEVERR_PAIR);
        return;
    }
    const long long s0 = src * (long long)chunks_per_block, d0 = dst * (long long)chunks_per_block;
    for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < chunks_per_block;
         c += gridDim.y * blockDim.x) {
        const uint4 kk = k_pool[s0 + c];
        const uint4 vv = v_pool[s0 + c];
        k_pool[d0 + c] = kk;
        v_pool[d0 + c] = vv;
    }
}

// Swap of whole blocks between the pool and page-locked host memory.
// grid.x = block index i, grid.y = slice; each CTA moves its slice of block
// ids[i]'s K and V (all KV heads, all 16 slots) in 16-byte vectors. out == true:
// pool -> host (host_k[i] is block i of the host copy); else host -> pool.
__global__ void __launch_bounds__(256)
swap_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, uint4* __restrict__ host_k,
                   uint4* __restrict__ host_v, const int32_t* __restrict__ ids, long long chunks_per_block,
                   int num_blocks, bool out, unsigned int* err) {
    pa::grid_dependency_wait();
    const int i = blockIdx.x;
    const int32_t b = ids[i];
    if (b < 0 || b >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) pa::set_error(err, PA_DEVERR_BLOCK_ID);
        return;
    }
    const long long p0 = (long long)b * chunks_per_block, h0 = (long long)i * chunks_per_block;
    for (long long c = (long long)blockIdx.y * blockDim.x + threadIdx.x; c < chunks_per_block;
         c += (long long)gridDim.y * blockDim.x) {
        if (out) {
            host_k[h0 + c] = k_pool[p0 + c];
            host_v[h0 + c] = v_pool[p0 + c];
        } else {
            k_pool[p0 + c] = host_k[h0 + c];
            v_pool[p0 + c] = host_v[h0 + c];
        }
    }
}

}  // namespace

namespace {
int swap_blocks(void* k_pool, void* v_pool, void* host_k, void* host_v, const int32_t* block_ids, int n_blocks,
                int n_kv_heads, int head_dim, int block_size, int elem_bytes, int num_blocks, bool out,
                pa_stream_t stream) {
    if (n_blocks < 0 || n_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (block_size != kBS) return PA_ERR_UNSUPPORTED;
    if (elem_bytes != 1 && elem_bytes != 2) return PA_ERR_UNSUPPORTED;
    const long long block_bytes = (long long)n_kv_heads * kBS * head_dim * elem_bytes;
    if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (n_blocks == 0) return PA_OK;
    if (!k_pool || !v_pool || !host_k || !host_v || !block_ids) return PA_ERR_INVALID_ARG;
    if (!pa_aligned16(k_pool) || !pa_aligned16(v_pool) || !pa_aligned16(host_k) || !pa_aligned16(host_v) ||
        (reinterpret_cast<uintptr_t>(block_ids) & 3u))
        return PA_ERR_INVALID_ARG;
    if (n_blocks > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    const long long chunks = block_bytes / 16;
    const int threads = 256;
    int slices = (int)((chunks + threads - 1) / threads);
    if (slices > 64) slices = 64;
    return pa_launch_pdl(swap_blocks_kernel, dim3((unsigned)n_blocks, slices), dim3(threads), 0,
                         reinterpret_cast<cudaStream_t>(stream), static_cast<uint4*>(k_pool),
                         static_cast<uint4*>(v_pool), static_cast<uint4*>(host_k), static_cast<uint4*>(host_v),
                         block_ids, chunks, num_blocks, out, err);
}
}  // namespace

extern "C" int pa_swap_out_blocks(const void* k_pool, const void* v_pool, const int32_t* block_ids, int n_blocks,
                                  void* host_k, void* host_v, int n_kv_heads, int head_dim, int block_size,
                                  int elem_bytes, int num_blocks, pa_stream_t stream) {
    return swap_blocks(const_cast<void*>(k_pool), const_cast<void*>(v_pool), host_k, host_v, block_ids, n_blocks,
                       n_kv_heads, head_dim, block_size, elem_bytes, num_blocks, true, stream);
}

extern "C" int pa_swap_in_blocks(const void* host_k, const void* host_v, void* k_pool, void* v_pool,
                                 const int32_t* block_ids, int n_blocks, int n_kv_heads, int head_dim,
                                 int block_size, int elem_bytes, int num_blocks, pa_stream_t stream) {
    return swap_blocks(k_pool, v_pool, const_cast<void*>(host_k), const_cast<void*>(host_v), block_ids, n_blocks,
                       n_kv_heads, head_dim, block_size, elem_bytes, num_blocks, false, stream);
}

extern "C" int pa_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                                    const int64_t* slot_mapping, int n_tokens, int n_kv_heads,
                                    int head_dim, int block_size, int num_blocks, pa_stream_t stream) {
    if (n_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (block_size != kBS) return PA_ERR_UNSUPPORTED;
    if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return PA_OK;
    if (!k || !v || !k_pool || !v_pool || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!pa_aligned16(k) || !pa_aligned16(v) || !pa_aligned16(k_pool) || !pa_aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    const int cph = head_dim / 8;
    const long long n_chunks = (long long)n_tokens * n_kv_heads * cph;
    const int threads = 256;
    const long long blocks = (n_chunks + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return pa_launch_pdl(reshape_and_cache_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                         reinterpret_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                         static_cast<const uint4*>(v), static_cast<uint4*>(k_pool),
                         static_cast<uint4*>(v_pool), slot_mapping, n_chunks, n_kv_heads, cph,
                         (long long)num_blocks * kBS, err);
}

extern "C" int pa_reshape_and_cache_fp8(const void* k, const void* v, void* k_pool, void* v_pool,
                                        const int64_t* slot_mapping, const float* k_scale,
                                        const float* v_scale, int n_tokens, int n_kv_heads, int head_dim,
                                        int block_size, int num_blocks, pa_stream_t stream) {
    if (n_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (block_size != kBS) return PA_ERR_UNSUPPORTED;
    if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return PA_OK;
    if (!k || !v || !k_pool || !v_pool || !slot_mapping || !k_scale || !v_scale) return PA_ERR_INVALID_ARG;
    if (!pa_aligned16(k) || !pa_aligned16(v) || (reinterpret_cast<uintptr_t>(k_pool) & 7u) ||
        (reinterpret_cast<uintptr_t>(v_pool) & 7u) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_ERR_INVALID_ARG;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    const int cph = head_dim / 8;
    const long long n_chunks = (long long)n_tokens * n_kv_heads * cph;
    const int threads = 256;
    const long long blocks = (n_chunks + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return pa_launch_pdl(reshape_and_cache_fp8_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                         reinterpret_cast<cudaStream_t>(stream), static_cast<const uint4*>(k),
                         static_cast<const uint4*>(v), static_cast<uint2*>(k_pool),
                         static_cast<uint2*>(v_pool), slot_mapping, k_scale, v_scale, n_chunks, n_kv_heads,
                         cph, (long long)num_blocks * kBS, err);
}

namespace {
int copy_blocks(void* k_pool, void* v_pool, const int64_t* block_mapping, int n_pairs, int n_kv_heads,
                int head_dim, int block_size, int elem_bytes, int num_blocks, pa_stream_t stream) {
    if (n_pairs < 0 || n_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (elem_bytes != 1 && elem_bytes != 2) return PA_ERR_INVALID_ARG;
    if (block_size != kBS) return PA_ERR_UNSUPPORTED;
    if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (n_pairs == 0) return PA_OK;
    if (n_pairs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
    if (!k_pool || !v_pool || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!pa_aligned16(k_pool) || !pa_aligned16(v_pool) ||
        (reinterpret_cast<uintptr_t>(block_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    // 16-byte chunks per block: n_kv_heads * 16 tokens * head_dim * elem_bytes
    // (a multiple of 16 for every head_dim that is a multiple of 8)
    const long long chunks = (long long)n_kv_heads * kBS * head_dim * elem_bytes / 16;
    if (chunks > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    const int threads = 256;
    int slices = (int)((chunks + threads - 1) / threads);
    if (slices > 64) slices = 64;
    dim3 grid(n_pairs, slices);
    copy_blocks_kernel<<<grid, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), block_mapping, (int)chunks, num_blocks,
        err);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
}  // namespace

extern "C" int pa_copy_blocks(void* k_pool, void* v_pool, const int64_t* block_mapping, int n_pairs,
                              int n_kv_heads, int head_dim, int block_size, int num_blocks,
                              pa_stream_t stream) {
    return copy_blocks(k_pool, v_pool, block_mapping, n_pairs, n_kv_heads, head_dim, block_size, 2, num_blocks,
                       stream);
}

extern "C" int pa_copy_blocks_ex(void* k_pool, void* v_pool, const int64_t* block_mapping, int n_pairs,
                                 int n_kv_heads, int head_dim, int block_size, int elem_bytes, int num_blocks,
                                 pa_stream_t stream) {
    return copy_blocks(k_pool, v_pool, block_mapping, n_pairs, n_kv_heads, head_dim, block_size, elem_bytes,
                       num_blocks, stream);
}
