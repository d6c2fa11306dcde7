// PagedAttention decode for sm_103a.
//
// What is computed ("LLM Inference Optimization: KV-Cache, PagedAttention,
// and GPU Memory Efficiency", section "PagedAttention: OS Concepts Meet GPU
// Memory": for each query, walk the sequence's block table, load K and V of
// each physical block, compute partial scores and accumulate with an online
// softmax; "KV Cache Explained Like You're an LLM Engineer", section
// "Transformer Attention: A Quick Refresher": softmax(q K^T / sqrt(d)) V):
//
//   out[b][h] = sum_t softmax_t(scale * q[b][h] . K_b[t]) V_b[t]
//
// Work decomposition (a GB300 design; the pages give none):
//  * One CTA per (context partition, KV head, sequence). All G = n_heads /
//    n_kv_heads query heads of the KV head's group are handled by the CTA, so
//    every K/V byte read from HBM serves the whole group.
//  * Each warp of the CTA streams its own share of the partition's blocks
//    through a private ring of S shared-memory stages. A (block, KV head)
//    tile of K and of V is block_size*head_dim*2 contiguous bytes in the pool
//    layout [blocks][kv_heads][16][head_dim]; lane 0 moves each with one
//    bulk asynchronous copy (cp.async.bulk, completion counted on an
//    mbarrier), so several tiles per warp are in flight while the warp
//    computes on an earlier one. Block ids come from the block table, read
//    once per warp (one entry per lane) and broadcast with a shuffle.
//  * Dot products: LPT lanes share one token row, each holding head_dim/LPT
//    dims of q (pre-multiplied by scale*log2(e)) in registers; partial dots
//    for all (head, token) pairs of the tile are combined with a
//    transposing butterfly (each shuffle level halves the values a lane
//    keeps), which costs far fewer shuffles than one reduction per dot.
//  * Online softmax in fp32 (base-2): running max and sum per head; the
//    probabilities of a tile are exchanged through a small per-warp shared
//    buffer and the PV product accumulates fp32 outputs with packed
//    fp32x2 FMAs.
//  * Warps of a CTA are merged through shared memory. If the sequence fits in
//    one partition the CTA writes the bf16 output directly; otherwise it
//    writes (max, sum, unnormalised output) to the workspace and a second
//    kernel merges the partitions (split-K).
//  * Groups of 8 query heads and E4M3 caches (head_dim 128) make the dot
//    products above bound by their instructions, not by HBM. Those run the
//    tensor-core variant further down: the same decomposition, with each
//    block's two products as warp-level MMAs over TMA-staged, swizzled tiles.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <vector>

#include "pa_common.cuh"
#include "tc_sm100.cuh"

namespace {

constexpr int kBS = 16;          // tokens per block
constexpr unsigned kFull = 0xffffffffu;

struct DecodeParams {
    uint16_t* out;
    const uint16_t* q;
    const unsigned char* k_pool;  // bf16 or E4M3 elements (see the kernel's EB)
    const unsigned char* v_pool;
    const float* k_scale;         // E4M3 cache: per-KV-head scales (else unused)
    const float* v_scale;
    const int32_t* tables;
    const int32_t* ctx;
    float* ws_ml;  // [B][H][P][2]
    float* ws_o;   // [B][H][P][D]
    float scale_log2;
    int n_heads;
    int n_kv_heads;
    int max_blocks;
    int num_blocks;
    int part_blocks;
    int max_parts;
    int window;  // >= 0: the query at position ctx-1 sees positions ctx-1-window .. ctx-1
    unsigned int* err;
    // optional plan (pa_decode_planned): CTA i runs item i = (partition, KV head,
    // sequence, unused) instead of the one its grid position names
    const int4* items;
    int n_items;
    int n_seqs;
};

// The (partition, KV head, sequence) of this CTA: its grid position, or its
// plan item. A plan item outside the call's bounds sets PA_DEVERR_PLAN and
// the CTA does nothing.
__device__ __forceinline__ bool cta_item(const DecodeParams& P, int& p, int& kvh, int& b) {
    if (!P.items) {
        p = blockIdx.x;
        kvh = blockIdx.y;
        b = blockIdx.z;
        return true;
    }
    const int4 it = P.items[blockIdx.x];
    p = it.x;
    kvh = it.y;
    b = it.z;
    if (b < 0 || b >= P.n_seqs || kvh < 0 || kvh >= P.n_kv_heads || p < 0 || p >= P.max_parts) {
        if (threadIdx.x == 0) pa::set_error(P.err, PA_DEVERR_PLAN);
        return false;
    }
    return true;
}

// First block and partition count of a sequence's (windowed) context.
__device__ __forceinline__ int first_position(const DecodeParams& P, int ctx) {
    return P.window >= 0 ? max(0, ctx - 1 - P.window) : 0;
}

// Transposing butterfly: N values per lane are summed across the lanes that
// differ in bits M, M/2, ..., 1; each level keeps half of the values.
template <int N, int M>
struct TransposeReduce {
    static __device__ __forceinline__ void run(float* v, int lane) {
        if constexpr (M >= 1) {
            if constexpr (N > 1) {
                constexpr int H2 = N / 2;
                const bool up = (lane & M) != 0;
#pragma unroll
                for (int k = 0; k < H2; ++k) {
                    float send = up ? v[k] : v[k + H2];
                    float keep = up ? v[k + H2] : v[k];
                    v[k] = keep + __shfl_xor_sync(kFull, send, M);
                }
                TransposeReduce<H2, M / 2>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(kFull, v[0], M);
                TransposeReduce<1, M / 2>::run(v, lane);
            }
        }
    }
};

// EB = bytes per cached element: 2 (bf16) or 1 (E4M3 codes with per-head scales).
template <int D, int G, int LPT, int EB>
struct Shape {
    static constexpr int NCH = D / (8 * LPT);      // 16-byte chunks per lane per token row
    static constexpr int TPP = 32 / LPT;           // tokens per warp pass
    static constexpr int NPASS = kBS / TPP;        // passes per tile
    static constexpr int NV = NPASS * G;           // partial dots per lane
    static constexpr int NKEEP = NV / LPT > 0 ? NV / LPT : 1;
    static constexpr int TILE_ELEMS = kBS * D;
    static constexpr int TILE_BYTES = TILE_ELEMS * EB;
    // lane-bit masks (within a warp) that do not select the head of the kept
    // values, and the subset on which kept values are duplicated
    static constexpr int HEAD_LO = LPT / G;        // masks >= HEAD_LO and < LPT select the head
    static constexpr int nonhead_mask() {
        int r = 0;
        for (int m = 1; m < 32; m <<= 1)
            if (m >= LPT || m < HEAD_LO) r |= m;
        return r;
    }
    static constexpr int dup_mask() {              // levels run after a single value is left
        int r = 0, n = NV;
        for (int m = LPT / 2; m >= 1; m >>= 1) {
            if (n > 1) n /= 2;
            else r |= m;
        }
        return r;
    }
    static_assert(D % (8 * LPT) == 0, "head_dim must split into 16-byte chunks per lane");
    static_assert(G <= LPT, "kept values of a lane must belong to one head");
};

template <int D, int G, int LPT, int EB, int NW, int S>
struct Smem {
    using SH = Shape<D, G, LPT, EB>;
    static constexpr size_t STAGES = (size_t)NW * S * 2 * SH::TILE_BYTES;
    static constexpr size_t BARS = (size_t)NW * S * 8;
    static constexpr size_t PBUF = (size_t)NW * G * kBS * 4;
    static constexpr size_t ABUF = (size_t)NW * ((G + 3) / 4) * 16;
    static constexpr size_t MERGE = (size_t)NW * (G * D + 2 * G) * 4;
    static_assert(MERGE <= STAGES, "merge buffers reuse the stage ring");
    static constexpr size_t TOTAL = STAGES + BARS + PBUF + ABUF;
};

// Eight cached elements of a row chunk -> four float2 (element pairs 0-1,
// 2-3, 4-5, 6-7). bf16 widens exactly by a shift; an E4M3 code widens exactly
// to fp16 (every E4M3 value is an fp16 value) and then to fp32.
template <int EB>
struct Chunk8;
template <>
struct Chunk8<2> {
    static __device__ __forceinline__ void load(const unsigned char* p, float2 (&f)[4]) {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        f[0] = pa::bf16x2_to_float2(w.x);
        f[1] = pa::bf16x2_to_float2(w.y);
        f[2] = pa::bf16x2_to_float2(w.z);
        f[3] = pa::bf16x2_to_float2(w.w);
    }
};
template <>
struct Chunk8<1> {
    static __device__ __forceinline__ void load(const unsigned char* p, float2 (&f)[4]) {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        pa::e4m3x4_to_float2x2(w.x, f[0], f[1]);
        pa::e4m3x4_to_float2x2(w.y, f[2], f[3]);
    }
};

template <int D, int G, int LPT, int EB, int NW, int S, int MINB>
__global__ void __launch_bounds__(NW * 32, MINB)
pa_decode_partition_kernel(const DecodeParams P) {
    using SH = Shape<D, G, LPT, EB>;
    using SM = Smem<D, G, LPT, EB, NW, S>;
    constexpr int NCH = SH::NCH, TPP = SH::TPP, NPASS = SH::NPASS, NV = SH::NV;
    constexpr int NKEEP = SH::NKEEP;
    constexpr int NONHEAD = SH::nonhead_mask();
    constexpr int LSUM = NONHEAD & ~SH::dup_mask();

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::STAGES);
    float* pbuf_all = reinterpret_cast<float*>(smem + SM::STAGES + SM::BARS);
    float* abuf_all = reinterpret_cast<float*>(smem + SM::STAGES + SM::BARS + SM::PBUF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = P.n_heads, Hk = P.n_kv_heads;
    pa::launch_dependents();     // the merge kernel may be scheduled now
    pa::grid_dependency_wait();  // the previous kernel (e.g. the cache write) is complete
    int p, kvh, b;
    if (!cta_item(P, p, kvh, b)) return;
    const int h0 = kvh * G;
    const int ctx = P.ctx[b];

    if (ctx <= 0) {  // empty sequence: zero output rows, written once
        if (p == 0) {
            for (int e = threadIdx.x; e < G * D / 2; e += NW * 32) {
                int h = e / (D / 2), d2 = e % (D / 2);
                reinterpret_cast<uint32_t*>(P.out + ((size_t)b * H + h0 + h) * D)[d2] = 0u;
            }
        }
        return;
    }
    int nblk = (ctx + kBS - 1) / kBS;
    // sliding window: blocks wholly before the window are never read (their
    // table entries may be released); positions before it are masked
    const int first_pos = first_position(P, ctx);
    int blk_first = first_pos / kBS;
    int nparts = (nblk - blk_first + P.part_blocks - 1) / P.part_blocks;
    if (nblk > P.max_blocks || nparts > P.max_parts) {  // caller broke the bounds it passed
        if (p == 0 && threadIdx.x == 0) pa::set_error(P.err, PA_DEVERR_CONTEXT);
        nblk = min(nblk, P.max_blocks);
        blk_first = min(blk_first, nblk);
        nparts = min((nblk - blk_first + P.part_blocks - 1) / P.part_blocks, P.max_parts);
        nblk = min(nblk, blk_first + nparts * P.part_blocks);
    }
    if (p >= nparts) return;
    const int blk_begin = blk_first + p * P.part_blocks;
    const int nb_local = min(blk_begin + P.part_blocks, nblk) - blk_begin;
    const int my_n = nb_local > warp ? (nb_local - warp + NW - 1) / NW : 0;  // <= 32

    const int c = lane % LPT;   // chunk lane within a token row
    const int tg = lane / LPT;  // token group within a pass

    unsigned char* my_stages = stages + (size_t)warp * S * 2 * SH::TILE_BYTES;
    uint64_t* my_bars = bars + warp * S;
    float* pbuf = pbuf_all + warp * G * kBS;
    float* abuf = abuf_all + warp * ((G + 3) / 4) * 4;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) pa::mbar_init(&my_bars[s], 1);
        pa::fence_mbar_init();
    }
    __syncwarp();

    // one block-table entry per lane: local block warp + NW*lane
    int my_bid = -1;
    if (lane < my_n) my_bid = P.tables[(size_t)b * P.max_blocks + blk_begin + warp + NW * lane];

    const uint64_t pol = pa::l2_evict_first_policy();
    const size_t head_stride = (size_t)SH::TILE_BYTES;
    auto issue = [&](int i) {  // all lanes call (shuffle); lane 0 issues the copies
        const int bid = __shfl_sync(kFull, my_bid, i);
        if (lane == 0) {
            const int st = i % S;
            uint64_t* bar = &my_bars[st];
            unsigned char* dk = my_stages + (size_t)st * 2 * SH::TILE_BYTES;
            if (bid >= 0 && bid < P.num_blocks) {
                const size_t off = ((size_t)bid * Hk + kvh) * head_stride;
                pa::mbar_arrive_expect_tx(bar, 2 * SH::TILE_BYTES);
                pa::bulk_g2s(dk, P.k_pool + off, SH::TILE_BYTES, bar, pol);
                pa::bulk_g2s(dk + SH::TILE_BYTES, P.v_pool + off, SH::TILE_BYTES, bar, pol);
            } else {
                pa::set_error(P.err, PA_DEVERR_BLOCK_ID);
                pa::mbar_arrive(bar);  // completes the phase with no data
            }
        }
    };

    // q for the G heads, this lane's dims, pre-scaled into the base-2 domain
    // (an E4M3 cache folds the KV head's K scale in here: q.(code*s) = (q*s).code)
    const float qscale = EB == 1 ? P.scale_log2 * P.k_scale[kvh] : P.scale_log2;
    float2 qf[G][NCH][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint16_t* qrow = P.q + ((size_t)b * H + h0 + h) * D;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
            uint4 w = *reinterpret_cast<const uint4*>(qrow + (c + LPT * j) * 8);
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float2 f = pa::bf16x2_to_float2(ws[k]);
                qf[h][j][k] = make_float2(f.x * qscale, f.y * qscale);
            }
        }
    }

    // which (head, pass) values this lane keeps after the transposing butterfly
    int base = 0;
    {
        int n = NV;
#pragma unroll
        for (int m = LPT / 2; m >= 1; m >>= 1) {
            if (n > 1) {
                n /= 2;
                if (lane & m) base += n;
            }
        }
    }
    const int h_own = base / NPASS;
    const int ip0 = base % NPASS;
    const bool alpha_writer = (lane & NONHEAD) == 0;

    float m_run = -INFINITY;  // running max of this lane's head (base-2 units)
    float l_run = 0.f;        // partial sum of p over this lane's kept tokens
    float2 o[G][NCH][4];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
            for (int k = 0; k < 4; ++k) o[h][j][k] = make_float2(0.f, 0.f);

    for (int s = 0; s < S && s < my_n; ++s) issue(s);

    int consumed = 0;
    bool aborted = false;
    for (int i = 0; i < my_n; ++i) {
        const int st = i % S;
        const bool ok = pa::mbar_wait(&my_bars[st], (uint32_t)((i / S) & 1), P.err);
        if (__any_sync(kFull, !ok)) {
            aborted = true;
            break;
        }
        consumed = i + 1;
        const int bid = __shfl_sync(kFull, my_bid, i);
        if (bid >= 0 && bid < P.num_blocks) {
            const unsigned char* sK = my_stages + (size_t)st * 2 * SH::TILE_BYTES;
            const unsigned char* sV = sK + SH::TILE_BYTES;
            const int tok0 = (blk_begin + warp + NW * i) * kBS;

            // ---- scores: partial dots over this lane's dims
            float sc[NV];
#pragma unroll
            for (int ip = 0; ip < NPASS; ++ip) {
                const int t = ip * TPP + tg;
                float2 acc[G];
#pragma unroll
                for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    float2 kf[4];
                    Chunk8<EB>::load(sK + (t * D + (c + LPT * j) * 8) * EB, kf);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        acc[h] = __ffma2_rn(qf[h][j][0], kf[0], acc[h]);
                        acc[h] = __ffma2_rn(qf[h][j][1], kf[1], acc[h]);
                        acc[h] = __ffma2_rn(qf[h][j][2], kf[2], acc[h]);
                        acc[h] = __ffma2_rn(qf[h][j][3], kf[3], acc[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < G; ++h) sc[h * NPASS + ip] = acc[h].x + acc[h].y;
            }
            TransposeReduce<NV, LPT / 2>::run(sc, lane);

            // ---- online softmax for this lane's head
            float tmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < NKEEP; ++k) {
                const int t = (ip0 + k) * TPP + tg;
                sc[k] = (tok0 + t < ctx && tok0 + t >= first_pos) ? sc[k] : -INFINITY;
                tmax = fmaxf(tmax, sc[k]);
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1)
                if (NONHEAD & m) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, m));
            const float m_new = fmaxf(m_run, tmax);
            const bool changed = m_new > m_run;
            const float alpha = pa::fast_exp2(m_run - m_new);
            float psum = 0.f;
#pragma unroll
            for (int k = 0; k < NKEEP; ++k) {
                const float pk = pa::fast_exp2(sc[k] - m_new);
                psum += pk;
                pbuf[h_own * kBS + tg * NPASS + ip0 + k] = pk;
            }
            l_run = l_run * alpha + psum;
            m_run = m_new;
            if (alpha_writer) abuf[h_own] = alpha;
            const bool any_changed = __any_sync(kFull, changed);
            __syncwarp();

            // ---- rescale and accumulate p . V
            if (any_changed) {
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float a = abuf[h];
                    const float2 a2 = make_float2(a, a);
#pragma unroll
                    for (int j = 0; j < NCH; ++j)
#pragma unroll
                        for (int k = 0; k < 4; ++k) o[h][j][k] = __fmul2_rn(o[h][j][k], a2);
                }
            }
            float pl[G][NPASS];
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int ip = 0; ip < NPASS; ip += 4) {
                    const float4 v4 = *reinterpret_cast<const float4*>(pbuf + h * kBS + tg * NPASS + ip);
                    pl[h][ip] = v4.x;
                    pl[h][ip + 1] = v4.y;
                    pl[h][ip + 2] = v4.z;
                    pl[h][ip + 3] = v4.w;
                }
#pragma unroll
            for (int ip = 0; ip < NPASS; ++ip) {
                const int t = ip * TPP + tg;
                if (tok0 + t < ctx && tok0 + t >= first_pos) {
#pragma unroll
                    for (int j = 0; j < NCH; ++j) {
                        float2 vf[4];
                        Chunk8<EB>::load(sV + (t * D + (c + LPT * j) * 8) * EB, vf);
#pragma unroll
                        for (int h = 0; h < G; ++h) {
                            const float2 pp = make_float2(pl[h][ip], pl[h][ip]);
                            o[h][j][0] = __ffma2_rn(pp, vf[0], o[h][j][0]);
                            o[h][j][1] = __ffma2_rn(pp, vf[1], o[h][j][1]);
                            o[h][j][2] = __ffma2_rn(pp, vf[2], o[h][j][2]);
                            o[h][j][3] = __ffma2_rn(pp, vf[3], o[h][j][3]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (i + S < my_n) issue(i + S);
    }
    if (aborted) {
        // drain copies still in flight (bounded) before the stage memory is reused
        for (int i = consumed; i < my_n && i < consumed + S; ++i)
            pa::mbar_wait(&my_bars[i % S], (uint32_t)((i / S) & 1), P.err, 10000000ull);
    }

    // ---- merge within the warp: sum o over token groups, l over head lanes
#pragma unroll
    for (int m = LPT; m < 32; m <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < NCH; ++j)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o[h][j][k].x += __shfl_xor_sync(kFull, o[h][j][k].x, m);
                    o[h][j][k].y += __shfl_xor_sync(kFull, o[h][j][k].y, m);
                }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1)
        if (LSUM & m) l_run += __shfl_xor_sync(kFull, l_run, m);

    __syncthreads();  // every warp is done with its ring: reuse it for the merge
    float* mo = reinterpret_cast<float*>(stages);            // [NW][G][D]
    float* mm = mo + NW * G * D;                               // [NW][G] max
    float* ml = mm + NW * G;                                   // [NW][G] sum
    if (tg == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
                float* dst = mo + ((size_t)warp * G + h) * D + (c + LPT * j) * 8;
                reinterpret_cast<float4*>(dst)[0] =
                    make_float4(o[h][j][0].x, o[h][j][0].y, o[h][j][1].x, o[h][j][1].y);
                reinterpret_cast<float4*>(dst)[1] =
                    make_float4(o[h][j][2].x, o[h][j][2].y, o[h][j][3].x, o[h][j][3].y);
            }
    }
    if (alpha_writer) {
        mm[warp * G + h_own] = m_run;
        ml[warp * G + h_own] = l_run;
    }
    __syncthreads();

    const bool single = (nparts == 1);
    const float vscale = EB == 1 ? P.v_scale[kvh] : 1.f;  // sum p (code*s) = s * sum p code
    for (int e = threadIdx.x; e < G * D / 2; e += NW * 32) {
        const int h = e / (D / 2), d = (e % (D / 2)) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * G + h]);
        float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = (mm[w * G + h] == -INFINITY) ? 0.f : pa::fast_exp2(mm[w * G + h] - M);
            L += ml[w * G + h] * f;
            const float2 ov = *reinterpret_cast<const float2*>(mo + ((size_t)w * G + h) * D + d);
            O0 += ov.x * f;
            O1 += ov.y * f;
        }
        O0 *= vscale;
        O1 *= vscale;
        const size_t row = (size_t)b * H + h0 + h;
        if (single) {
            const float inv = 1.f / L;
            reinterpret_cast<uint32_t*>(P.out + row * D)[d / 2] = pa::float2_to_bf16x2(O0 * inv, O1 * inv);
        } else {
            const size_t slot = row * P.max_parts + p;
            *reinterpret_cast<float2*>(P.ws_o + slot * D + d) = make_float2(O0, O1);
            if (d == 0) *reinterpret_cast<float2*>(P.ws_ml + slot * 2) = make_float2(M, L);
        }
    }
}

// ------------------------------------------------------------------------
// Tensor-core variant of the partition kernel for large query groups
// (head_dim 128, bf16 cache). With G = 8 query heads per KV head the CUDA-core
// kernel above needs 255 registers, runs 8 warps per SM and is bound by its
// FMA work, not by HBM. Here each tile's two products are warp-level
// mma.sync tensor-core instructions (m16n8k16): a tile costs 16 (QK^T, the
// G query heads in the first G of 16 rows) + 16 (PV, two P terms x 8 m-tiles
// of 16 dims) of them instead of ~1,000 FMA and shuffle instructions. tcgen05 needs M >= 64, which would
// waste 7/8 of every instruction on padding rows for this shape.
//   S[16 x 16 tokens] = Q[16 x 128] . K^T   (A = q in registers, B = K via ldmatrix;
//                                            with an E4M3 cache S^T = K . Q^T instead:
//                                            the 16 tokens as M, the heads as N, one
//                                            MMA per k-step, and P^T for the P.V
//                                            product from two movmatrix transposes)
//   O^T[128 x 8]     += V^T . P^T           (A = V^T via ldmatrix.trans; with an
//                                            E4M3 cache V's codes widened in
//                                            registers and transposed by movmatrix;
//                                            B = P^T, which is S's accumulator
//                                            layout as it stands; the 8 head rows
//                                            fill N = 8)
// With a bf16 cache P enters as two bf16 terms (P_hi = p truncated, P_lo =
// the rounded remainder), so the weights keep ~16 significant bits. (A single
// fp16 P, as the prefill uses, would need V widened to fp16 element by element
// in registers here, which costs more instructions than the P_lo MMAs save.)
// With an E4M3 cache, whose V codes are widened to fp16 anyway, P enters as
// one fp16 term, rounded to nearest (within 2^-12 of p).
// K and V tiles arrive by 2-D TMA in 128B-swizzled layout (16 rows x 64 dims
// per box), so the ldmatrix row reads are free of bank conflicts.
namespace mma {

constexpr int kNW = 4;  // warps per CTA
// Per warp, bf16 cache: 2 stages of K 4 KiB + V 4 KiB (each two 2 KiB boxes,
// 16 rows x 64 dims): 64 KiB per CTA, three CTAs per SM. E4M3 cache: 2
// stages of K 2 KiB + V 2 KiB (one box of 16 rows x 128 codes each; both are
// widened in registers, straight from the stage): 32 KiB per CTA and four
// CTAs per SM, the most its registers allow (its per-block work is
// latency-bound, so more warps per SM beat a deeper ring).
template <int EB>
struct Lay {
    static constexpr int kStage = EB == 2 ? 8192 : 4096;
    static constexpr int kStages = 2;  // ring stages per warp
    static constexpr int kWarp = kStages * kStage;
    static constexpr int kSmem = kNW * kWarp + kNW * kStages * 8;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// the same with fp16 operands (an E4M3 cache widened exactly to fp16)
__device__ __forceinline__ void mma16816_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <int EB>
__device__ __forceinline__ void mma_t(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    if constexpr (EB == 2) mma16816(c, a0, 0u, a2, 0u, b0, b1);
    else mma16816_f16(c, a0, 0u, a2, 0u, b0, b1);
}
template <int EB>
__device__ __forceinline__ void mma_full(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    if constexpr (EB == 2) mma16816(c, a0, a1, a2, a3, b0, b1);
    else mma16816_f16(c, a0, a1, a2, a3, b0, b1);
}
__device__ __forceinline__ uint32_t f2_to_h2(float a, float b) {  // fp16x2, a in the low half
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
// transposes an 8 x 8 matrix of 16-bit elements held in the m8n8 fragment
// layout (lane l: row l / 4, columns 2 (l % 4), +1)
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint16_t c) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
    return r;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// byte offset of (row, 8-element chunk `dims8` of 0..15) in a tile stored as
// two 128B-swizzled boxes of 16 rows x 64 dims
__device__ __forceinline__ uint32_t sw_off(int row, int dims8) {
    return (uint32_t)((dims8 >> 3) * 2048 + row * 128 + (((dims8 & 7) ^ (row & 7)) << 4));
}

}  // namespace mma

template <int G, int EB>
__global__ void __launch_bounds__(mma::kNW * 32, EB == 1 ? 4 : 3)
pa_decode_mma_kernel(const DecodeParams P, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
    using namespace mma;
    constexpr int D = 128, NW = kNW, S = Lay<EB>::kStages;
    constexpr int kStage = Lay<EB>::kStage, kWarp = Lay<EB>::kWarp;
    static_assert(G <= 8, "query heads of a group fill the first G of 16 MMA rows");
    extern __shared__ __align__(1024) unsigned char smem_mma[];
    unsigned char* stages = smem_mma;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_mma + NW * kWarp);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;  // MMA fragment row group and column pair
    const int H = P.n_heads, Hk = P.n_kv_heads;
    pa::launch_dependents();
    pa::grid_dependency_wait();
    int p, kvh, b;
    if (!cta_item(P, p, kvh, b)) return;
    const int h0 = kvh * G;
    if (pa::smem_u32(smem_mma) & 1023u) {  // never expected; refuse rather than mis-swizzle
        if (threadIdx.x == 0) pa::set_error(P.err, PA_DEVERR_LAYOUT);
        return;
    }
    const int ctx = P.ctx[b];
    if (ctx <= 0) {  // empty sequence: zero output rows, written once
        if (p == 0) {
            for (int e = threadIdx.x; e < G * D / 2; e += NW * 32) {
                int h = e / (D / 2), d2 = e % (D / 2);
                reinterpret_cast<uint32_t*>(P.out + ((size_t)b * H + h0 + h) * D)[d2] = 0u;
            }
        }
        return;
    }
    int nblk = (ctx + kBS - 1) / kBS;
    const int first_pos = first_position(P, ctx);
    int blk_first = first_pos / kBS;
    int nparts = (nblk - blk_first + P.part_blocks - 1) / P.part_blocks;
    if (nblk > P.max_blocks || nparts > P.max_parts) {  // caller broke the bounds it passed
        if (p == 0 && threadIdx.x == 0) pa::set_error(P.err, PA_DEVERR_CONTEXT);
        nblk = min(nblk, P.max_blocks);
        blk_first = min(blk_first, nblk);
        nparts = min((nblk - blk_first + P.part_blocks - 1) / P.part_blocks, P.max_parts);
        nblk = min(nblk, blk_first + nparts * P.part_blocks);
    }
    if (p >= nparts) return;
    const int blk_begin = blk_first + p * P.part_blocks;
    const int nb_local = min(blk_begin + P.part_blocks, nblk) - blk_begin;
    const int my_n = nb_local > warp ? (nb_local - warp + NW - 1) / NW : 0;  // <= 32

    unsigned char* my_stages = stages + (size_t)warp * kWarp;
    uint64_t* my_bars = bars + warp * S;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) pa::mbar_init(&my_bars[s], 1);
        pa::fence_mbar_init();
    }
    __syncwarp();

    int my_bid = -1;  // one block-table entry per lane: local block warp + NW*lane
    if (lane < my_n) my_bid = P.tables[(size_t)b * P.max_blocks + blk_begin + warp + NW * lane];

    const uint64_t pol = pa::l2_evict_first_policy();
    auto issue = [&](int i) {  // all lanes call (shuffle); lanes 0..3 issue the four boxes
        const int bid = __shfl_sync(kFull, my_bid, i);
        const int st = i % S;
        uint64_t* bar = &my_bars[st];
        unsigned char* dst = my_stages + (size_t)st * kStage;
        if (bid >= 0 && bid < P.num_blocks) {
            if (lane == 0) pa::mbar_arrive_expect_tx(bar, kStage);
            __syncwarp();
            const int y = (bid * Hk + kvh) * kBS;
            if constexpr (EB == 2) {
                if (lane < 4)  // lane: bit 1 = V, bit 0 = dims 64..127
                    tc::tma_load_2d_hint(dst + (lane >> 1) * 4096 + (lane & 1) * 2048,
                                         (lane >> 1) ? &tmV : &tmK, (lane & 1) * 64, y, bar, pol);
            } else {
                if (lane < 2)  // lane 1 = V; one box of 16 rows x 128 codes
                    tc::tma_load_2d_hint(dst + lane * 2048, lane ? &tmV : &tmK, 0, y, bar, pol);
            }
        } else if (lane == 0) {
            pa::set_error(P.err, PA_DEVERR_BLOCK_ID);
            pa::mbar_arrive(bar);  // completes the phase with no data
        }
    };

    // q as the A operand: rows g < G are the group's heads, rows g+8 are zero;
    // per k-step of 16 dims a lane holds dims 2t, 2t+1 and 2t+8, 2t+9
    uint32_t qa[8][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(P.q + ((size_t)b * H + h0 + (g < G ? g : 0)) * D);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            // bf16 cache: k = 2t, 2t+1 | 2t+8, 2t+9 are dims 16ks + 2t.. | 16ks + 2t + 8..; E4M3
            // cache: the same k are dims 16ks + 4t, +1 | +2, +3, so that a lane's K codes are
            // four consecutive bytes (the sum over the k-step is unchanged)
            qa[ks][0] = g < G ? qrow[EB == 2 ? ks * 8 + t : ks * 8 + 2 * t] : 0u;
            qa[ks][1] = g < G ? qrow[EB == 2 ? ks * 8 + 4 + t : ks * 8 + 2 * t + 1] : 0u;
            if constexpr (EB == 1) {  // bf16 -> fp16 for the fp16 MMA (exact for |q| in the fp16 range)
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float2 f = pa::bf16x2_to_float2(qa[ks][k]);
                    qa[ks][k] = f2_to_h2(f.x, f.y);
                }
            }
        }
    }
    // O^T fragments: m-tile mt holds dims 16mt + g (c0, c1) and 16mt + g + 8 (c2, c3)
    // of heads 2t (c0, c2) and 2t + 1 (c1, c3)
    float o[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[n][k] = 0.f;
    float m_used = -INFINITY, l_run = 0.f;  // row g, base-2 units; l over this lane's columns
    // E4M3 cache: scores are computed transposed (S^T, tokens x heads), so a
    // lane holds heads 2t and 2t + 1: their reference maxima and its part of
    // their sums (the same reference on the 8 lanes of a head)
    float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
    // E4M3 cache: q.(code*s_k) = s_k (q.code), folded into the score scale
    const float sc = EB == 1 ? P.scale_log2 * P.k_scale[kvh] : P.scale_log2;

    for (int s = 0; s < S && s < my_n; ++s) issue(s);
    int consumed = 0;
    bool aborted = false;
    for (int i = 0; i < my_n; ++i) {
        const int st = i % S;
        const bool ok = pa::mbar_wait(&my_bars[st], (uint32_t)((i / S) & 1), P.err);
        if (__any_sync(kFull, !ok)) {
            aborted = true;
            break;
        }
        consumed = i + 1;
        const int bid = __shfl_sync(kFull, my_bid, i);
        if (bid >= 0 && bid < P.num_blocks) {
            const uint32_t kb = pa::smem_u32(my_stages + (size_t)st * kStage);
            const uint32_t vb = kb + 4096;  // bf16 cache: the V tile
            const int tok0 = (blk_begin + warp + NW * i) * kBS;
            // ---- S = Q K^T: two n-tiles of 8 tokens
            float s_acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            if constexpr (EB == 2) {
                const int m = lane >> 3, row = 8 * (m >> 1) + (lane & 7), kh = m & 1;  // matrix: (token half, k half)
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(kb + sw_off(row, 2 * ks + kh), b00, b01, b10, b11);
                    mma_t<EB>(s_acc[0], qa[ks][0], qa[ks][1], b00, b01);
                    mma_t<EB>(s_acc[1], qa[ks][0], qa[ks][1], b10, b11);
                }
            }
            // E4M3: S^T = K Q^T with the tile's 16 tokens as M and the group's heads as
            // N: one MMA per k-step of 16 dims; the lane's k = 2t, 2t+1 | 2t+8, 2t+9 are
            // dims 16ks + 4t, +1 | +2, +3 (four consecutive codes of each of its token
            // rows g and g + 8, widened in registers); two accumulators (even and odd
            // k-steps) halve the dependent chain
            float sT[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (EB == 1) {
                const unsigned char* rk = my_stages + (size_t)st * kStage;
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int off = ((ks ^ (g & 7)) << 4) + 4 * t;  // rows g and g + 8 share the swizzle
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(rk + g * 128 + off);
                    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(rk + (g + 8) * 128 + off);
                    mma16816_f16(ks & 1 ? sb : sa, e4m3x2_to_h2((uint16_t)(w0 & 0xffffu)),
                                 e4m3x2_to_h2((uint16_t)(w1 & 0xffffu)), e4m3x2_to_h2((uint16_t)(w0 >> 16)),
                                 e4m3x2_to_h2((uint16_t)(w1 >> 16)), qa[ks][0], qa[ks][1]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) sT[k] = sa[k] + sb[k];
            }
            uint32_t ph[2], pl[2];
            if constexpr (EB == 1) {
                // ---- online softmax per head over the tile's 16 tokens: this lane holds
                // tokens g, g + 8 (sT[0..1], sT[2..3]) of heads 2t, 2t + 1 (even, odd k).
                // p = 2^(s*scale - m) against the head's reference m, set to the maximum
                // so far on the head's first visible keys and whenever a p could leave
                // fp16's range (the key at the maximum gets p = 1 exactly)
                float sv[4], pv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int pos = tok0 + g + 8 * (u >> 1);
                    sv[u] = (pos < ctx && pos >= first_pos) ? sT[u] * sc : -INFINITY;
                }
                auto exps = [&]() {
#pragma unroll
                    for (int u = 0; u < 4; ++u) pv[u] = pa::fast_exp2(sv[u] - (m2[u & 1] == -INFINITY ? 0.f : m2[u & 1]));
                };
                exps();
                int need[2];
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    need[k] = !(pv[k] <= 32768.f && pv[2 + k] <= 32768.f) ||
                              (m2[k] == -INFINITY && (sv[k] != -INFINITY || sv[2 + k] != -INFINITY));
                if (__any_sync(kFull, need[0] | need[1])) {
                    // rare: a new reference for the heads that need one (uniform over a head's lanes)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float hm = fmaxf(sv[k], sv[2 + k]);
                        int nd = need[k];
#pragma unroll
                        for (int o2 = 4; o2 <= 16; o2 <<= 1) {
                            hm = fmaxf(hm, __shfl_xor_sync(kFull, hm, o2));
                            nd |= __shfl_xor_sync(kFull, nd, o2);
                        }
                        if (nd && hm > m2[k]) {
                            const float a = pa::fast_exp2(m2[k] - hm);  // 0 on the head's first keys
                            m2[k] = hm;
                            l2[k] *= a;
#pragma unroll
                            for (int n = 0; n < 8; ++n) {
                                o[n][k] *= a;
                                o[n][2 + k] *= a;
                            }
                        }
                    }
                    exps();
                }
                l2[0] += pv[0] + pv[2];
                l2[1] += pv[1] + pv[3];
                // P^T as the B operand (tokens 2t, 2t+1 | 2t+8, 2t+9 of head g): the
                // fp16 pairs (token g; heads 2t, 2t+1) of each 8 x 8 half, transposed
                ph[0] = movmatrix_t(f2_to_h2(pv[0], pv[1]));
                ph[1] = movmatrix_t(f2_to_h2(pv[2], pv[3]));
                pl[0] = pl[1] = 0u;
            } else {
                // ---- online softmax of row g over the tile's 16 tokens (this lane: 2t, 2t+1, 8+2t, 9+2t)
                float sv[4];
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int pos = tok0 + 8 * n + 2 * t + k;
                        sv[2 * n + k] = (pos < ctx && pos >= first_pos) ? s_acc[n][k] * sc : -INFINITY;
                    }
                float tmax = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
                tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 1));
                tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 2));
                float alpha = 1.f;
                if (tmax > m_used + 8.f) {  // lazy rescale: p <= 2^8 un-normalised
                    alpha = pa::fast_exp2(m_used - tmax);  // 0 on the first tile
                    l_run *= alpha;
                    m_used = tmax;
                }
                if (__any_sync(kFull, alpha != 1.f)) {  // O^T columns are heads: head h's factor from lane 4h
                    const float a0 = __shfl_sync(kFull, alpha, 8 * t), a1 = __shfl_sync(kFull, alpha, 8 * t + 4);
#pragma unroll
                    for (int n = 0; n < 8; ++n) {
                        o[n][0] *= a0;
                        o[n][1] *= a1;
                        o[n][2] *= a0;
                        o[n][3] *= a1;
                    }
                }
                const float mref = m_used == -INFINITY ? 0.f : m_used;  // a row with no visible key yet
                float pv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    pv[k] = pa::fast_exp2(sv[k] - mref);
                    l_run += pv[k];
                }
                // P as the B operand (tokens of head g), as two bf16 terms: P_hi truncated
                // and P_lo the rounded rest, two MMAs (a single bf16 term, within 2^-9 of p,
                // can miss an absolute 2e-3 on short rows)
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    const uint32_t bx = __float_as_uint(pv[2 * n]), by = __float_as_uint(pv[2 * n + 1]);
                    ph[n] = __byte_perm(bx, by, 0x7632);
                    pl[n] = pa::float2_to_bf16x2(pv[2 * n] - __uint_as_float(bx & 0xffff0000u),
                                                 pv[2 * n + 1] - __uint_as_float(by & 0xffff0000u));
                }
            }
            // V rows of the sequence's last, partial block past the context hold
            // whatever the pool has there (p = 0 must not meet a NaN): zero them
            // (E4M3: in registers, below)
            if (EB == 2 && ctx < tok0 + kBS) {
                const int r0 = ctx - tok0;
                unsigned char* vt = my_stages + (size_t)st * kStage + 4096;
                for (int e = lane; e < (kBS - r0) * 32; e += 32)  // a row: 2 boxes x 128 B
                    *reinterpret_cast<uint2*>(vt + ((e & 31) >> 4) * 2048 + (r0 + (e >> 5)) * 128 + (e & 15) * 8) =
                        make_uint2(0u, 0u);
                tc::fence_async_smem();  // before the stage's next TMA fill
                __syncwarp();
            }
            // ---- O^T += V^T P^T: 8 m-tiles of 16 dims, k = the tile's 16 tokens, n = the 8 head
            // rows; P's accumulator layout is already the B operand (tokens 2t.. and 2t+8.. of head g)
            if constexpr (EB == 2) {
                const int m = lane >> 3, row = 8 * (m >> 1) + (lane & 7), dh = m & 1;  // matrix: (token half, dim half)
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vb + sw_off(row, 2 * mt + dh), a0, a1, a2, a3);
                    mma_full<EB>(o[mt], a0, a1, a2, a3, ph[0], ph[1]);
                    mma_full<EB>(o[mt], a0, a1, a2, a3, pl[0], pl[1]);
                }
            } else {
                // E4M3: V^T's fragments straight from the codes. Within m-tile mt the
                // 16 rows of O^T are the dims in the order that gives lane (g, t) the
                // four consecutive codes 16mt + 4t .. +3 of its token rows g and g + 8:
                // codes 4t, 4t+1 are rows 2t, 2t+1 and codes 4t+2, 4t+3 rows 8+2t,
                // 9+2t. Widened to fp16 pairs they are the m8n8 fragments of V's
                // four 8 x 8 (token, dim) blocks; a movmatrix transpose makes each
                // the matching block of V^T, the A operand. Token rows past the
                // context are zero (p = 0 must not meet a NaN).
                const unsigned char* rv = my_stages + (size_t)st * kStage + 2048;
                const bool lo_ok = tok0 + g < ctx, hi_ok = tok0 + g + 8 < ctx;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int off = ((mt ^ (g & 7)) << 4) + 4 * t;  // rows g and g + 8 share the swizzle
                    const uint32_t w0 = lo_ok ? *reinterpret_cast<const uint32_t*>(rv + g * 128 + off) : 0u;
                    const uint32_t w1 = hi_ok ? *reinterpret_cast<const uint32_t*>(rv + (g + 8) * 128 + off) : 0u;
                    const uint32_t a0 = movmatrix_t(e4m3x2_to_h2((uint16_t)(w0 & 0xffffu)));
                    const uint32_t a1 = movmatrix_t(e4m3x2_to_h2((uint16_t)(w0 >> 16)));
                    const uint32_t a2 = movmatrix_t(e4m3x2_to_h2((uint16_t)(w1 & 0xffffu)));
                    const uint32_t a3 = movmatrix_t(e4m3x2_to_h2((uint16_t)(w1 >> 16)));
                    mma_full<EB>(o[mt], a0, a1, a2, a3, ph[0], ph[1]);
                }
            }
        }
        __syncwarp();
        if (i + S < my_n) issue(i + S);
    }
    if (aborted) {
        // drain copies still in flight (bounded) before the stage memory is reused
        for (int i = consumed; i < my_n && i < consumed + S; ++i)
            pa::mbar_wait(&my_bars[i % S], (uint32_t)((i / S) & 1), P.err, 10000000ull);
    }
    l_run += __shfl_xor_sync(kFull, l_run, 1);
    l_run += __shfl_xor_sync(kFull, l_run, 2);
#pragma unroll
    for (int k = 0; k < 2; ++k)  // E4M3: a head's sum over its 8 lanes
#pragma unroll
        for (int o2 = 4; o2 <= 16; o2 <<= 1) l2[k] += __shfl_xor_sync(kFull, l2[k], o2);

    __syncthreads();  // every warp is done with its ring: reuse it for the merge
    float* mo = reinterpret_cast<float*>(stages);  // [NW][G][D]
    float* mm = mo + NW * G * D;                   // [NW][G] max
    float* ml = mm + NW * G;                       // [NW][G] sum
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // heads 2t and 2t + 1
        const int h = 2 * t + k;
        if (h < G) {
            // O^T rows g and g + 8 of an m-tile: dims g and g + 8 (bf16 cache); with an
            // E4M3 cache the rows' dims as ordered above: 2g, 2g + 2 (g even) or
            // 2g - 1, 2g + 1 (g odd)
            const int d_lo = EB == 2 ? g : ((g & 1) ? 2 * g - 1 : 2 * g);
            const int d_hi = EB == 2 ? g + 8 : ((g & 1) ? 2 * g + 1 : 2 * g + 2);
            float* dst = mo + ((size_t)warp * G + h) * D;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                dst[16 * mt + d_lo] = o[mt][k];
                dst[16 * mt + d_hi] = o[mt][2 + k];
            }
        }
    }
    if constexpr (EB == 1) {
        if (g == 0) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (2 * t + k < G) {
                    mm[warp * G + 2 * t + k] = m2[k];
                    ml[warp * G + 2 * t + k] = l2[k];
                }
        }
    } else if (g < G && t == 0) {
        mm[warp * G + g] = m_used;
        ml[warp * G + g] = l_run;
    }
    __syncthreads();

    const bool single = (nparts == 1);
    for (int e = threadIdx.x; e < G * D / 2; e += NW * 32) {
        const int h = e / (D / 2), d = (e % (D / 2)) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * G + h]);
        float L = 0.f, O0 = 0.f, O1 = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = (mm[w * G + h] == -INFINITY) ? 0.f : pa::fast_exp2(mm[w * G + h] - M);
            L += ml[w * G + h] * f;
            const float2 ov = *reinterpret_cast<const float2*>(mo + ((size_t)w * G + h) * D + d);
            O0 += ov.x * f;
            O1 += ov.y * f;
        }
        if constexpr (EB == 1) {  // sum p (code * s_v) = s_v * sum p code
            O0 *= P.v_scale[kvh];
            O1 *= P.v_scale[kvh];
        }
        const size_t row = (size_t)b * H + h0 + h;
        if (single) {
            const float inv = 1.f / L;
            reinterpret_cast<uint32_t*>(P.out + row * D)[d / 2] = pa::float2_to_bf16x2(O0 * inv, O1 * inv);
        } else {
            const size_t slot = row * P.max_parts + p;
            *reinterpret_cast<float2*>(P.ws_o + slot * D + d) = make_float2(O0, O1);
            if (d == 0) *reinterpret_cast<float2*>(P.ws_ml + slot * 2) = make_float2(M, L);
        }
    }
}

}  // namespace

namespace {

// Split-K merge: one warp per (sequence, query head) row. Lane p reads the
// (m, l) of partitions p, p+32, ...; a warp reduction gives M and L; then the
// partitions' output slices are loaded eight at a time, so a row costs two
// rounds of memory latency rather than one per partition.
template <int D>
__global__ void __launch_bounds__(128)
pa_decode_merge_kernel(const DecodeParams P, int n_rows) {
    constexpr int PER = D / 32;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // (seq, head) row
    const int lane = threadIdx.x & 31;
    pa::grid_dependency_wait();  // every partition's partial is written
    if (row >= n_rows) return;
    const int H = P.n_heads;
    const int b = row / H;
    const int ctx = P.ctx[b];
    if (ctx <= 0) return;
    const int nblk = min((ctx + kBS - 1) / kBS, P.max_blocks);
    const int blk_first = min(first_position(P, ctx) / kBS, nblk);
    const int nparts = min((nblk - blk_first + P.part_blocks - 1) / P.part_blocks, P.max_parts);
    if (nparts <= 1) return;  // the partition kernel wrote this row
    const size_t slot0 = (size_t)row * P.max_parts;
    float m_mine = -INFINITY, l_mine = 0.f;  // this lane's partitions, relative to m_mine
    for (int p = lane; p < nparts; p += 32) {
        const float2 ml = *reinterpret_cast<const float2*>(P.ws_ml + (slot0 + p) * 2);
        if (ml.x > m_mine) {
            l_mine = (m_mine == -INFINITY ? 0.f : l_mine * pa::fast_exp2(m_mine - ml.x)) + ml.y;
            m_mine = ml.x;
        } else if (ml.x != -INFINITY) {
            l_mine += ml.y * pa::fast_exp2(ml.x - m_mine);
        }
    }
    float M = m_mine;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float L = m_mine == -INFINITY ? 0.f : l_mine * pa::fast_exp2(m_mine - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
    float acc[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) acc[k] = 0.f;
    for (int p0 = 0; p0 < nparts; p0 += 8) {
        float f[8], v[8][PER];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = p0 + u;
            f[u] = 0.f;
#pragma unroll
            for (int k = 0; k < PER; ++k) v[u][k] = 0.f;
            if (p < nparts) {
                const float m = P.ws_ml[(slot0 + p) * 2];
                f[u] = m == -INFINITY ? 0.f : pa::fast_exp2(m - M);
                const float* op = P.ws_o + (slot0 + p) * D + lane * PER;
                if constexpr (PER == 4) {
                    const float4 w = *reinterpret_cast<const float4*>(op);
                    v[u][0] = w.x; v[u][1] = w.y; v[u][2] = w.z; v[u][3] = w.w;
                } else {
                    const float2 w = *reinterpret_cast<const float2*>(op);
                    v[u][0] = w.x; v[u][1] = w.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int k = 0; k < PER; ++k) acc[k] += v[u][k] * f[u];
    }
    const float inv = 1.f / L;
    uint32_t* dst = reinterpret_cast<uint32_t*>(P.out + (size_t)row * D + lane * PER);
#pragma unroll
    for (int k = 0; k < PER; k += 2) dst[k / 2] = pa::float2_to_bf16x2(acc[k] * inv, acc[k + 1] * inv);
}

constexpr int kNW = 4;  // warps per CTA


// Per (head_dim, group) launch shape. Twelve resident warps per SM (three
// CTAs of four warps, three warps per scheduler) hide the latency of the
// per-tile dependency chains best; that caps a thread at 168 registers, so
// G = 4 at head_dim 128 spreads a token row over 16 lanes (q and the
// accumulators then take 32 registers each). G = 8 needs more registers and
// runs two CTAs per SM. S stages of K+V tiles per warp fill the shared memory
// of the resident CTAs (2 or 3 stages of 8 KiB at head_dim 128, 4 or 6 of
// 4 KiB at head_dim 64).
// An E4M3 cache (EB = 1) has half-size tiles and keeps the same bytes in
// flight with twice the stages; at head_dim 128 and G = 4 its kernel fits in
// 128 registers, so it runs four CTAs (16 warps) per SM with two stages
// instead (measured 2% faster: the kernel is latency-bound there).
template <int D, int G, int EB>
struct Launch {
    static constexpr bool FP8_WIDE = EB == 1 && D == 128 && G == 4;
    static constexpr int LPT = (D == 128 && G >= 4) ? 16 : 8;
    static constexpr int MINB = FP8_WIDE ? 4 : (G == 8 ? 2 : 3);
    static constexpr int S = FP8_WIDE ? 2 : (D == 128 ? 2 : 4) * (MINB == 3 ? 1 : 3) / (MINB == 3 ? 1 : 2) * (2 / EB);
};

template <int D, int G, int EB>
int launch_partition(const DecodeParams& P, int n_seqs, cudaStream_t stream) {
    using LC = Launch<D, G, EB>;
    using SM = Smem<D, G, LC::LPT, EB, kNW, LC::S>;
    auto kern = pa_decode_partition_kernel<D, G, LC::LPT, EB, kNW, LC::S, LC::MINB>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SM::TOTAL) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        attr_done[dev] = true;
    }
    const dim3 grid = P.items ? dim3((unsigned)P.n_items) : dim3(P.max_parts, P.n_kv_heads, n_seqs);
    return pa_launch_pdl(kern, grid, dim3(kNW * 32), SM::TOTAL, stream, P);
}

template <int D, int EB>
int dispatch_group(int G, const DecodeParams& P, int n_seqs, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_partition<D, 1, EB>(P, n_seqs, stream);
        case 2: return launch_partition<D, 2, EB>(P, n_seqs, stream);
        case 4: return launch_partition<D, 4, EB>(P, n_seqs, stream);
        case 8: return launch_partition<D, 8, EB>(P, n_seqs, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

// The tensor-core partition kernel (head_dim 128, bf16 cache): K and V pools
// as 2-D TMA maps of [num_blocks * n_kv_heads * 16 rows][128 dims].
template <int G, int EB>
int launch_partition_mma(const DecodeParams& P, int n_seqs, cudaStream_t stream) {
    auto kern = pa_decode_mma_kernel<G, EB>;
    constexpr int kSmem = mma::Lay<EB>::kSmem;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_done[dev] = true;
    }
    const uint64_t rows = (uint64_t)P.num_blocks * P.n_kv_heads * kBS;
    CUtensorMap tk, tv;
    const bool maps = EB == 2 ? pa_make_tmap_2d_bf16(&tk, P.k_pool, 128, rows, 256, 64, kBS) &&
                                    pa_make_tmap_2d_bf16(&tv, P.v_pool, 128, rows, 256, 64, kBS)
                              : pa_make_tmap_2d_u8(&tk, P.k_pool, 128, rows, 128, 128, kBS) &&
                                    pa_make_tmap_2d_u8(&tv, P.v_pool, 128, rows, 128, 128, kBS);
    if (!maps) return PA_ERR_CUDA;
    const dim3 grid = P.items ? dim3((unsigned)P.n_items) : dim3(P.max_parts, P.n_kv_heads, n_seqs);
    return pa_launch_pdl(kern, grid, dim3(mma::kNW * 32), kSmem, stream, P, tk, tv);
}

constexpr int kDefaultPartitionTokens = 512;

// CTAs of the CUDA-core partition kernel resident per SM (its launch bounds).
int k1_ctas_per_sm(int head_dim, int G, int eb) {
    if (head_dim == 128) {
        if (eb == 1 && G == 4) return Launch<128, 4, 1>::MINB;
        return G == 8 ? Launch<128, 8, 2>::MINB : Launch<128, 4, 2>::MINB;
    }
    return G == 8 ? Launch<64, 8, 2>::MINB : Launch<64, 4, 2>::MINB;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;  // every thread that races here writes the same value
    }
    return cached[dev];
}

// Default partition size of the CUDA-core kernel. One CTA streams one
// partition of one (sequence, KV head); when the grid is a few waves of CTA
// slots deep, a last wave that fills only part of the slots leaves SMs idle.
// When one CTA per (sequence, KV head) gives every SM at least one and fits
// a single wave (sms <= n_seqs x n_kv_heads <= slots) and a context fits one
// partition (<= 2048 tokens), each sequence takes a single partition: one
// wave of HBM-bound streams, no split-K partials and no merge. Otherwise,
// among the multiples of 64 tokens in [512, 1024] (each needs no more
// workspace than 512), take the one whose grid - n_seqs x n_kv_heads x
// ceil(context / size) CTAs, exact when every context is `context` - fills
// its last wave best (waves / ceil(waves)), the smallest on ties.
int wave_partition_tokens(int n_seqs, int n_kv_heads, int context, int sms, int slots) {
    const long long groups = (long long)n_seqs * n_kv_heads;
    if (sms > 0 && groups >= sms && groups <= slots && context > kDefaultPartitionTokens &&
        context <= 4 * kDefaultPartitionTokens)
        return (context + 63) / 64 * 64;
    if (slots <= 0 || context <= kDefaultPartitionTokens) return kDefaultPartitionTokens;
    int best = kDefaultPartitionTokens;
    double best_fill = -1.0;
    for (int pt = kDefaultPartitionTokens; pt <= 2 * kDefaultPartitionTokens; pt += 64) {
        const double ctas = (double)n_seqs * n_kv_heads * ((context + pt - 1) / pt);
        const double waves = ctas / slots;
        const double fill = waves / ceil(waves);
        if (fill > best_fill + 1e-9) {
            best_fill = fill;
            best = pt;
        }
    }
    return best;
}

int default_partition_tokens(bool tensor, int eb, int n_seqs, int n_kv_heads, int G, int head_dim,
                             int max_context_len, int window) {
    if (tensor) return 2 * kDefaultPartitionTokens;
    const int span = window >= 0 && window + 2 * kBS < max_context_len ? window + 2 * kBS : max_context_len;
    const int sms = sm_count();
    return wave_partition_tokens(n_seqs, n_kv_heads, span, sms, sms * k1_ctas_per_sm(head_dim, G, eb));
}

int resolve_partition_tokens(int pt) {
    if (pt == 0) return kDefaultPartitionTokens;
    if (pt < 64 || pt > 2048 || pt % 64 != 0) return -1;
    return pt;
}

size_t workspace_bytes_for(int n_seqs, int n_heads, int head_dim, int max_parts) {
    if (max_parts <= 1) return 0;
    const size_t rows = (size_t)n_seqs * n_heads * max_parts;
    const size_t ml = (rows * 2 * sizeof(float) + 255) & ~(size_t)255;
    return ml + rows * head_dim * sizeof(float);
}

}  // namespace

extern "C" size_t pa_decode_workspace_bytes(int n_seqs, int n_heads, int head_dim,
                                            int max_context_len, int partition_tokens) {
    const int pt = resolve_partition_tokens(partition_tokens);
    if (pt < 0 || n_seqs <= 0 || n_heads <= 0 || head_dim <= 0 || max_context_len <= 0) return 0;
    const int max_parts = (max_context_len + pt - 1) / pt;
    return workspace_bytes_for(n_seqs, n_heads, head_dim, max_parts);
}

extern "C" int pa_decode_partition_tokens(int n_seqs, int n_heads, int n_kv_heads, int head_dim,
                                          int max_context_len, int window, int elem_bytes) {
    if (n_seqs < 0 || n_heads <= 0 || n_kv_heads <= 0 || max_context_len < 0 || n_heads % n_kv_heads != 0 ||
        (elem_bytes != 1 && elem_bytes != 2))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    const int G = n_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    const bool tensor = head_dim == 128 && (G == 8 || elem_bytes == 1);
    return default_partition_tokens(tensor, elem_bytes, n_seqs, n_kv_heads, G, head_dim, max_context_len, window);
}

namespace {

// Shared body of the bf16 (eb = 2) and E4M3 (eb = 1) decode entry points.
int decode_impl(int eb, void* out, const void* q, const void* k_pool, const void* v_pool,
                const float* k_scale, const float* v_scale, const int32_t* block_tables,
                const int32_t* context_lens, float scale, int n_heads, int n_kv_heads, int head_dim,
                int block_size, int n_seqs, int max_blocks_per_seq, int max_context_len, int num_blocks,
                int window, int partition_tokens, void* workspace, size_t workspace_bytes,
                pa_stream_t stream, bool force_tc = false, const int32_t* items = nullptr, int n_items = 0) {
    if (n_seqs < 0 || max_context_len < 0 || num_blocks < 0 || max_blocks_per_seq < 0 ||
        n_heads <= 0 || n_kv_heads <= 0)
        return PA_ERR_INVALID_ARG;
    if (block_size != kBS) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (n_heads % n_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int G = n_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    if (n_kv_heads > 65535 || n_seqs > 65535) return PA_ERR_UNSUPPORTED;
    const bool tc_rows_ok = (long long)num_blocks * n_kv_heads * kBS + kBS <= 0x7fffffffLL;  // TMA coordinates
    if (force_tc && (eb != 2 || head_dim != 128 || !tc_rows_ok)) return PA_ERR_UNSUPPORTED;
    if ((long long)max_blocks_per_seq * kBS < (long long)max_context_len) return PA_ERR_INVALID_ARG;
    // At head_dim 128, groups of 8 heads and every E4M3 cache run on the tensor
    // cores (the CUDA-core kernel is bound by its instructions there, not by
    // HBM), unless the pool has too many rows for a TMA coordinate;
    // pa_decode_tc asks for the tensor-core kernel at every group size
    const bool tensor = force_tc || (head_dim == 128 && tc_rows_ok && (G == 8 || eb == 1));
    // default partitions: on the CUDA-core kernel the size in [512, 1024]
    // whose grid fills its last wave of CTA slots best (wave_partition_tokens);
    // 1024 tokens on the tensor-core kernel, whose shorter blocks amortise a
    // CTA's fixed cost over more of them (measured 3-5% faster). The workspace
    // for 512 covers every one of them.
    const int pt = partition_tokens == 0
                       ? default_partition_tokens(tensor, eb, n_seqs, n_kv_heads, G, head_dim, max_context_len, window)
                       : resolve_partition_tokens(partition_tokens);
    if (pt < 0) return PA_ERR_INVALID_ARG;
    if (pt / kBS > 32 * kNW) return PA_ERR_INVALID_ARG;  // one table entry per lane
    if (n_seqs == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!pa_aligned16(out) || !pa_aligned16(q) || !pa_aligned16(k_pool) || !pa_aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    if (eb == 1 && (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
                    (reinterpret_cast<uintptr_t>(v_scale) & 3u)))
        return PA_ERR_INVALID_ARG;
    if (out == q) return PA_ERR_INVALID_ARG;
    int max_parts = max_context_len > 0 ? (max_context_len + pt - 1) / pt : 1;
    if (window >= 0) {  // W + 1 positions touch at most ceil((W + 16) / 16) blocks
        const int wblocks = (window + 2 * kBS - 1) / kBS;
        const int wparts = (wblocks + pt / kBS - 1) / (pt / kBS);
        if (wparts < max_parts) max_parts = wparts;
    }
    const size_t need = workspace_bytes_for(n_seqs, n_heads, head_dim, max_parts);
    if (need > 0 && (!workspace || workspace_bytes < need || !pa_aligned16(workspace)))
        return PA_ERR_WORKSPACE;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;

    DecodeParams P;
    P.out = static_cast<uint16_t*>(out);
    P.q = static_cast<const uint16_t*>(q);
    P.k_pool = static_cast<const unsigned char*>(k_pool);
    P.v_pool = static_cast<const unsigned char*>(v_pool);
    P.k_scale = k_scale;
    P.v_scale = v_scale;
    P.tables = block_tables;
    P.ctx = context_lens;
    const size_t rows = (size_t)n_seqs * n_heads * max_parts;
    P.ws_ml = need ? static_cast<float*>(workspace) : nullptr;
    P.ws_o = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             ((rows * 2 * sizeof(float) + 255) & ~(size_t)255))
                  : nullptr;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.n_heads = n_heads;
    P.n_kv_heads = n_kv_heads;
    P.max_blocks = max_blocks_per_seq;
    P.num_blocks = num_blocks;
    P.part_blocks = pt / kBS;
    P.max_parts = max_parts;
    P.window = window;
    P.err = err;
    P.items = reinterpret_cast<const int4*>(items);
    P.n_items = n_items;
    P.n_seqs = n_seqs;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int st;
    if (tensor) {
        if (eb == 2) {
            switch (G) {
                case 1: st = launch_partition_mma<1, 2>(P, n_seqs, s); break;
                case 2: st = launch_partition_mma<2, 2>(P, n_seqs, s); break;
                case 4: st = launch_partition_mma<4, 2>(P, n_seqs, s); break;
                default: st = launch_partition_mma<8, 2>(P, n_seqs, s); break;
            }
        } else {
            switch (G) {
                case 1: st = launch_partition_mma<1, 1>(P, n_seqs, s); break;
                case 2: st = launch_partition_mma<2, 1>(P, n_seqs, s); break;
                case 4: st = launch_partition_mma<4, 1>(P, n_seqs, s); break;
                default: st = launch_partition_mma<8, 1>(P, n_seqs, s); break;
            }
        }
    } else if (eb == 1)
        st = head_dim == 128 ? dispatch_group<128, 1>(G, P, n_seqs, s) : dispatch_group<64, 1>(G, P, n_seqs, s);
    else
        st = head_dim == 128 ? dispatch_group<128, 2>(G, P, n_seqs, s) : dispatch_group<64, 2>(G, P, n_seqs, s);
    if (st != PA_OK || max_parts <= 1) return st;
    const int n_rows = n_seqs * n_heads;
    dim3 grid((n_rows + 3) / 4);
    if (head_dim == 128) return pa_launch_pdl(pa_decode_merge_kernel<128>, grid, dim3(128), 0, s, P, n_rows);
    return pa_launch_pdl(pa_decode_merge_kernel<64>, grid, dim3(128), 0, s, P, n_rows);
}

}  // namespace

extern "C" int pa_decode_ex(void* out, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const int32_t* context_lens, float scale,
                            int n_heads, int n_kv_heads, int head_dim, int block_size, int n_seqs,
                            int max_blocks_per_seq, int max_context_len, int num_blocks,
                            int partition_tokens, void* workspace, size_t workspace_bytes,
                            pa_stream_t stream) {
    return decode_impl(2, out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens, scale,
                       n_heads, n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq,
                       max_context_len, num_blocks, -1, partition_tokens, workspace, workspace_bytes,
                       stream);
}

extern "C" int pa_decode_tc(void* out, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const int32_t* context_lens, float scale,
                            int n_heads, int n_kv_heads, int head_dim, int block_size, int n_seqs,
                            int max_blocks_per_seq, int max_context_len, int num_blocks,
                            int partition_tokens, void* workspace, size_t workspace_bytes,
                            pa_stream_t stream) {
    return decode_impl(2, out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens, scale,
                       n_heads, n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq,
                       max_context_len, num_blocks, -1, partition_tokens, workspace, workspace_bytes,
                       stream, true);
}

extern "C" int pa_decode_window(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* context_lens, float scale,
                                int n_heads, int n_kv_heads, int head_dim, int block_size, int n_seqs,
                                int max_blocks_per_seq, int max_context_len, int num_blocks, int window,
                                int partition_tokens, void* workspace, size_t workspace_bytes,
                                pa_stream_t stream) {
    if (window < 0) return PA_ERR_INVALID_ARG;
    return decode_impl(2, out, q, k_pool, v_pool, nullptr, nullptr, block_tables, context_lens, scale,
                       n_heads, n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq,
                       max_context_len, num_blocks, window, partition_tokens, workspace, workspace_bytes,
                       stream);
}

extern "C" int pa_decode_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                             const float* k_scale, const float* v_scale, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, int n_heads, int n_kv_heads,
                             int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                             int max_context_len, int num_blocks, int partition_tokens, void* workspace,
                             size_t workspace_bytes, pa_stream_t stream) {
    return decode_impl(1, out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens, scale,
                       n_heads, n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq,
                       max_context_len, num_blocks, -1, partition_tokens, workspace, workspace_bytes,
                       stream);
}

extern "C" int pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                         int n_heads, int n_kv_heads, int head_dim, int block_size, int n_seqs,
                         int max_blocks_per_seq, int max_context_len, int num_blocks, void* workspace,
                         size_t workspace_bytes, pa_stream_t stream) {
    return pa_decode_ex(out, q, k_pool, v_pool, block_tables, context_lens, scale, n_heads, n_kv_heads,
                        head_dim, block_size, n_seqs, max_blocks_per_seq, max_context_len, num_blocks, 0,
                        workspace, workspace_bytes, stream);
}

// Host-side plan: the decode call's work items (one CTA each), the longest
// partitions first. The partition size and count follow decode_impl, and
// each sequence's partitions follow the partition kernels' own count, with
// the same clamps; a sequence with no partition keeps one item (p = 0),
// whose CTA writes its zero rows or flags its bounds. A grid in plain order
// ends on whichever CTAs start last, full or short; longest-first puts the
// short last partitions of the sequences at the end (measured 97.5 -> 94.3
// us on 64 sequences of 128..4,096 tokens).
extern "C" int pa_decode_plan(const int32_t* context_lens, int n_seqs, int n_heads, int n_kv_heads,
                              int head_dim, int max_blocks_per_seq, int max_context_len, int num_blocks,
                              int window, int elem_bytes, int partition_tokens, int32_t* items, int cap) {
    if (n_seqs < 0 || n_heads <= 0 || n_kv_heads <= 0 || max_context_len < 0 || max_blocks_per_seq < 0 ||
        num_blocks < 0 || window < -1 || cap < 0 || n_heads % n_kv_heads != 0 ||
        (elem_bytes != 1 && elem_bytes != 2) || (n_seqs > 0 && !context_lens))
        return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    const int G = n_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    const bool tc_rows_ok = (long long)num_blocks * n_kv_heads * kBS + kBS <= 0x7fffffffLL;
    const bool tensor = head_dim == 128 && tc_rows_ok && (G == 8 || elem_bytes == 1);
    const int pt = partition_tokens == 0
                       ? default_partition_tokens(tensor, elem_bytes, n_seqs, n_kv_heads, G, head_dim,
                                                  max_context_len, window)
                       : resolve_partition_tokens(partition_tokens);
    if (pt < 0 || pt / kBS > 32 * kNW) return PA_ERR_INVALID_ARG;
    const int part_blocks = pt / kBS;
    int max_parts = max_context_len > 0 ? (max_context_len + pt - 1) / pt : 1;
    if (window >= 0) {
        const int wblocks = (window + 2 * kBS - 1) / kBS;
        const int wparts = (wblocks + part_blocks - 1) / part_blocks;
        if (wparts < max_parts) max_parts = wparts;
    }
    // per sequence: its partition count and the blocks of its last partition
    std::vector<int> nparts(n_seqs), last_blocks(n_seqs);
    long long total = 0;
    for (int b = 0; b < n_seqs; ++b) {
        const int ctx = context_lens[b];
        int np = 0, last = 0;
        if (ctx > 0) {
            int nblk = (ctx + kBS - 1) / kBS;
            int blk_first = (window >= 0 ? std::max(0, ctx - 1 - window) : 0) / kBS;
            np = (nblk - blk_first + part_blocks - 1) / part_blocks;
            if (nblk > max_blocks_per_seq || np > max_parts) {
                nblk = std::min(nblk, max_blocks_per_seq);
                blk_first = std::min(blk_first, nblk);
                np = std::min((nblk - blk_first + part_blocks - 1) / part_blocks, max_parts);
                nblk = std::min(nblk, blk_first + np * part_blocks);
            }
            if (np > 0) last = (nblk - blk_first) - (np - 1) * part_blocks;
        }
        if (np <= 0) {  // one item: the zero rows, or the bounds flag
            np = 1;
            last = 0;
        }
        nparts[b] = np;
        last_blocks[b] = last;
        total += (long long)np * n_kv_heads;
    }
    if (total > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (!items) return (int)total;  // size query
    if (total > cap) return PA_ERR_CAPACITY;
    // counting sort by the item's blocks, descending; (sequence, KV head,
    // partition) order within a length
    std::vector<long long> start(part_blocks + 2, 0);
    auto blocks_of = [&](int b, int p) { return p + 1 < nparts[b] ? part_blocks : last_blocks[b]; };
    for (int b = 0; b < n_seqs; ++b)
        for (int p = 0; p < nparts[b]; ++p) start[part_blocks - blocks_of(b, p) + 1] += n_kv_heads;
    for (int l = 1; l <= part_blocks + 1; ++l) start[l] += start[l - 1];
    for (int b = 0; b < n_seqs; ++b)
        for (int kvh = 0; kvh < n_kv_heads; ++kvh)
            for (int p = 0; p < nparts[b]; ++p) {
                const long long i = start[part_blocks - blocks_of(b, p)]++;
                items[4 * i + 0] = p;
                items[4 * i + 1] = kvh;
                items[4 * i + 2] = b;
                items[4 * i + 3] = 0;
            }
    return (int)total;
}

extern "C" int pa_decode_planned(void* out, const void* q, const void* k_pool, const void* v_pool,
                                 const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                 const int32_t* context_lens, float scale, int n_heads, int n_kv_heads,
                                 int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                                 int max_context_len, int num_blocks, int window, int partition_tokens,
                                 const int32_t* items, int n_items, void* workspace, size_t workspace_bytes,
                                 pa_stream_t stream) {
    if (window < -1 || (k_scale == nullptr) != (v_scale == nullptr)) return PA_ERR_INVALID_ARG;
    if (n_seqs > 0 && (!items || n_items <= 0 || !pa_aligned16(items))) return PA_ERR_INVALID_ARG;
    return decode_impl(k_scale ? 1 : 2, out, q, k_pool, v_pool, k_scale, v_scale, block_tables, context_lens,
                       scale, n_heads, n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq,
                       max_context_len, num_blocks, window, partition_tokens, workspace, workspace_bytes, stream,
                       false, items, n_items);
}

// ---------------------------------------------------------------------------
// Allocation-free decode (pa_decode_noalloc).
//
// pa_decode needs a caller-provided scratch workspace for its split-K
// partials. Some callers cannot allocate one: a serving runtime that has
// handed all free HBM to its KV-cache pool, an integration that must not call
// cudaMalloc/cudaFree on its decode loop because those calls can synchronize
// the device and stall every stream, or a host that only passes raw pointers
// and has no allocator to offer. For them the scratch lives in the fixed
// array below, which every device that loads this library holds until the
// process exits.
//
// Limits and sharing: the array is kNoAllocScratchBytes (32 MiB); a batch
// whose decode workspace would be larger is rejected with PA_ERR_WORKSPACE
// before anything is launched. Every call on a device uses the same array
// and it keeps the previous call's contents; nothing in it has to start at
// zero (each call writes every partial it later reads). Two calls whose
// kernels overlap on the GPU (for example on two streams without ordering
// between them) race on the array and may produce wrong outputs.
//
// Host code cannot use the array's name as a device address (on the host it
// only names a stand-in). The first call on each device, with that device
// current, resolves the real address with cudaGetSymbolAddress and caches it
// (thread-safe, per device and per context: after a device reset the new
// context's address is looked up again on its first call); make that first
// call before any stream capture on that device.
static constexpr size_t kNoAllocScratchBytes = 32ull << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

extern "C" int pa_decode_noalloc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_tables, const int32_t* context_lens, float scale,
                                 int n_heads, int n_kv_heads, int head_dim, int block_size, int n_seqs,
                                 int max_blocks_per_seq, int max_context_len, int num_blocks,
                                 pa_stream_t stream) {
    static PaSymbolCache* cache = pa_symbol_cache_new();
    if (n_seqs < 0 || n_heads <= 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
    if (n_seqs > 0 && max_context_len > 0 &&
        pa_decode_workspace_bytes(n_seqs, n_heads, head_dim, max_context_len, 0) > kNoAllocScratchBytes)
        return PA_ERR_WORKSPACE;  // this batch needs more scratch than the fixed array holds
    void* scratch = pa_symbol_address(cache, &g_noalloc_scratch);
    if (!scratch) return PA_ERR_CUDA;
    return pa_decode_ex(out, q, k_pool, v_pool, block_tables, context_lens, scale, n_heads, n_kv_heads,
                        head_dim, block_size, n_seqs, max_blocks_per_seq, max_context_len, num_blocks, 0,
                        scratch, kNoAllocScratchBytes, stream);
}
