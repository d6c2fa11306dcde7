// Chunked causal prefill over the paged KV cache on the tcgen05 tensor cores.
//
// What is computed ("Modern AI Infrastructure and Agentic System Design",
// 9.1 "Two workloads wearing one name": a long prompt is processed in chunks
// interleaved with decode; "KV Cache Explained Like You're an LLM Engineer",
// "Prefill Phase vs. Decode Phase"; causal masking as in "What Happens Inside
// an LLM During Inference ...", "Self-Attention Mechanism"): sequence s's
// chunk of L new tokens occupies the last L of its context_lens[s] cached
// positions; chunk row i sits at position p = ctx - L + i and
//     out[i][h] = sum_{t <= p} softmax_t(scale * q[i][h] . K[t]) V[t].
//
// Design (GB300), for head_dim D = 64 or 128 (one instantiation each; the
// K/V block rows are D bf16 values, moved as D/64 boxes of 64 dims). A query
// tile is 128 matrix rows = QT = 128/G chunk tokens x
// the G query heads of one KV head's group, so every K/V byte staged in
// shared memory feeds all G heads. One CTA owns two query tiles (A and B) of
// the same (sequence, KV head): both use every K/V tile it loads, and the
// tensor core alternates between them so that one tile's MMAs run while the
// other tile's softmax works. Per key tile j of 128 keys (8 blocks of 16),
// five roles in 14 warps, each waiting only on mbarriers or, for the
// hand-over of P, on a named barrier:
//   - a producer warp moves the 8 K and 8 V blocks with 2-D TMA loads into
//     128B-swizzled shared memory: two K stages and three V stages, each
//     refilled as soon as the tensor core is done with it (blocks past the
//     end of the sequence load out of bounds and arrive as zeros);
//   - four converter warps (one per scheduler) rewrite each landed V tile in
//     place as fp16 values of v * 2^-8 (rows past the context, which hold
//     whatever the pool has there, become zeros);
//   - one thread of an MMA warp issues, per query tile X, S_X = Q_X K_j^T
//     (tcgen05.mma kind::f16, bf16 in, fp32 accumulator in tensor memory,
//     M = N = 128, K = D) and, once X's softmax has written P, O_X += P V_j (fp16
//     in: P read from tensor memory, V as an MN-major shared-memory operand)
//     with S_X(j+1) right behind it. The MMAs of one thread execute in issue
//     order, so S_X(j+1) may follow the PV MMA that still reads P(j) out of
//     the same columns, and the completion of S_X(j+1) covers that PV MMA;
//   - one softmax warpgroup per query tile (thread = row) reads S_X from
//     tensor memory once, a quarter of 32 columns at a time, applies the
//     scale, the causal mask (diagonal tiles only) and an online softmax in
//     fp32 (base 2) against the row's integer reference maximum m (changed
//     only on a row's first visible keys or before any p = 2^(s*scale - m)
//     could leave the fp16 range, so every rescale of O, l and the tile's
//     earlier P is an exact power of two), and writes P back into S_X's
//     columns as fp16 (rounded to nearest: within 2^-12 of p relative).
//     A bf16 P (within 2^-9) would exceed an absolute error of 2e-3 on short
//     causal rows with cancelling values; the tensor core takes A and B of
//     one type, hence V in fp16 too. Every bf16 value is an fp16 value
//     inside fp16's exponent range; the factor 2^-8 moves that range up to
//     |v| <= 65504 * 2^8 (larger values become infinite and the output
//     non-finite, which is flagged), at an absolute error of at most 2^-17
//     for |v| < 2^-6, where the scaled value is subnormal. The four warps
//     hand P over to the MMA warp through a named barrier (arrive/sync).
// The normalised output 2^8 O / l is written once at the end.
//
// Scheduling. Per-pair mode: one CTA per (pair, KV head, sequence), or per
// piece of its key range. Balanced mode: one CTA per SM takes entries of a
// work list in order (whole pairs for the full waves, pieces of the pairs of
// the last partial wave) and runs them one after another, re-initialising
// its barriers between entries; pieces leave partials for a merge kernel.
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "tc_sm100.cuh"

namespace {

constexpr int kBS = 16;          // tokens per block
constexpr int kKT = 128;         // keys per key tile
constexpr int kBPT = kKT / kBS;  // blocks per key tile
constexpr int kRows = 128;       // MMA M
constexpr unsigned kFull = 0xffffffffu;

constexpr int kKS = 2;  // K tile stages
constexpr int kVS = 3;  // V tile stages
constexpr int kThreads = 448;  // 8 softmax warps, MMA warp (8), producer (9), 4 converter warps (10..13)
// Shared memory map for head_dim D (64 or 128): a Q tile (128 rows) and a
// K or V tile (128 keys) are 128 x D bf16 values each, stored as D / 64
// 128B-swizzled halves of 64 dims (16 KiB each). The dynamic shared memory
// base must be 1024-byte aligned (swizzle atoms of TMA and of the matrix
// descriptors): checked.
template <int D>
struct PfLay {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static constexpr int kHalves = D / 64;               // 64-dim halves of a row
    static constexpr uint32_t kTile = kKT * D * 2;       // K or V tile bytes
    static constexpr uint32_t kQTile = kRows * D * 2;    // Q tile bytes
    static constexpr uint32_t kQ = 0;                    // Q_A, Q_B
    static constexpr uint32_t kK0 = 2 * kQTile;          // K stages
    static constexpr uint32_t kV0 = kK0 + kKS * kTile;   // V stages
    static constexpr uint32_t kBars = kV0 + kVS * kTile; // mbarriers
    static constexpr uint32_t kMisc = kBars + 256;       // tmem slot, abort flag, segment entries
    static constexpr uint32_t kSmem = kMisc + 64;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};
constexpr uint32_t kTmemCols = 512;  // tile X: S at 256X, O at 256X + 128 (D columns)

struct PrefillParams {
    uint16_t* out;
    const uint16_t* q;
    const int32_t* tables;
    const int32_t* ctx;
    const int32_t* qsl;
    float scale_log2;
    int n_heads;
    int n_kv_heads;
    int max_blocks;
    int num_blocks;
    int oob_row;  // a TMA row coordinate past the end of the pool (zero fill)
    int splits;   // per-pair mode: pieces per query-tile pair (1: no split)
    float* part;  // partials of pieces: [item][piece] (per-pair mode) or [slot] (balanced mode),
                  // each [tile][row][kPartStride]
    // Balanced mode (work null in per-pair mode). Item it = (sequence *
    // n_kv_heads + kv head) * n_qp + pair. The planning kernel writes the
    // work list: every non-empty item whole, in item order, except the items
    // of the last partial wave, which are cut into sched[2] equal key ranges
    // (piece-major); CTAs take entries in order from the counter sched[0].
    int4* work;      // entries (item, first key tile, end key tile, partial slot or -1); sched[1] of them
    int* sched;      // counter, entries, pieces per cut item, cut items
    int n_items;
    int n_qp;
    int n_cta;
    unsigned int* err;
};

// A piece's partial for one row: the un-normalised O (head_dim floats from
// offset 0), and at offset 128 the reference maximum m (base-2 units) and the
// sum l of 2^(s*scale - m); the same row size for both head dims.
constexpr int kPartStride = 132;  // floats, 16-byte aligned rows
constexpr int kPartML = 128;      // offset of (m, l) in a partial row

// Key tiles [kt0, kt1) of piece sp out of `splits` over a pair's n_kt tiles.
__host__ __device__ inline void piece_range(int n_kt, int sp, int splits, int& kt0, int& kt1) {
    kt0 = (int)((long long)sp * n_kt / splits);
    kt1 = (int)((long long)(sp + 1) * n_kt / splits);
}

// fp32 -> fp16 round to nearest even; a in the low half, b in the high half
// (beyond the fp16 range: infinity).
__device__ __forceinline__ uint32_t float2_to_f16x2(float a, float b) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp16 A and B (the
// kind takes one type for both operands) and an fp32 accumulator; fields as
// in tc::idesc_bf16_f32 with the A and B format fields 0 (fp16).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Bounded wait (1 s) that also gives up once another role has aborted. A
// waiting thread sleeps inside try_wait (up to 20 us per try, woken when the
// phase completes), so idle roles take no issue slots from busy ones.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, unsigned int* err,
                                         volatile int* abort_flag) {
    if (pa::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    const uint64_t t0 = pa::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (pa::mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (pa::globaltimer_ns() - t0 > PA_WAIT_LIMIT_NS) {
                pa::set_error(err, PA_DEVERR_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

template <int G, int D>
__global__ void __launch_bounds__(kThreads, 1)
pa_prefill_tc_kernel(const PrefillParams P, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
    using L_ = PfLay<D>;
    constexpr uint32_t kQ = L_::kQ, kK0 = L_::kK0, kV0 = L_::kV0, kBars = L_::kBars, kMisc = L_::kMisc;
    constexpr uint32_t kTile = L_::kTile, kQTile = L_::kQTile;
    constexpr int kNH = L_::kHalves;
    constexpr int QT = kRows / G;  // chunk tokens per query tile
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBars);
    uint64_t* k_full = bars;          // [kKS] K tile landed
    uint64_t* k_free = k_full + kKS;  // [kKS] QK_B, the last reader of the K stage, is done
    uint64_t* v_full = k_free + kKS;  // [kVS] V tile landed (bf16)
    uint64_t* v_free = v_full + kVS;  // [kVS] PV_B, the last reader of the V stage, is done
    uint64_t* s_full = v_free + kVS;  // [2] per query tile: S_X(j) and every earlier MMA done
    uint64_t* pv_done = s_full + 2;   // [2] per query tile
    uint64_t* drain = pv_done + 2;    // every MMA issued in the segment is done
    uint64_t* v_conv = drain + 1;     // [kVS] V tile rewritten as fp16, 4 arrivals (one per converter warp)
    constexpr int kNumBars = 2 * kKS + 3 * kVS + 5;
    static_assert(kNumBars * 8 <= 256, "barrier area");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMisc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = P.n_heads, Hk = P.n_kv_heads;
    if (pa::smem_u32(sm) & 1023u) {  // never expected; refuse rather than mis-swizzle
        if (threadIdx.x == 0) pa::set_error(P.err, PA_DEVERR_LAYOUT);
        return;
    }
    // Segments. Per-pair mode: piece sp of pair (qp, kv head, sequence) from
    // the grid position. Balanced mode: the work-list entries this CTA takes
    // from the counter, one at a time.
    int* next = reinterpret_cast<int*>(sm + kMisc + 8);  // [2] the entry taken, by segment parity
    bool have_tmem = false;
    uint32_t tbase = 0;
    int n_run = 0;  // segments run so far
    for (int seg = 0;; ++seg) {
        int s, kvh, qp, kt0 = 0, kt1 = 0;
        bool direct = true;
        float* part_base = nullptr;
        if (P.work) {
            if (threadIdx.x == 0) next[seg & 1] = atomicAdd(&P.sched[0], 1);
            __syncthreads();
            const int w = next[seg & 1];
            if (w >= P.sched[1]) break;
            const int4 e = P.work[w];
            kt0 = e.y;
            kt1 = e.z;
            direct = e.w < 0;
            if (!direct) part_base = P.part + (size_t)e.w * 2 * 128 * kPartStride;
            s = e.x / (Hk * P.n_qp);
            kvh = (e.x / P.n_qp) % Hk;
            qp = e.x % P.n_qp;
        } else {
            if (seg > 0) break;
            qp = blockIdx.x / P.splits;
            kvh = blockIdx.y;
            s = blockIdx.z;
        }
        const int h0 = kvh * G;
        const int q0 = P.qsl[s];
        const int L = P.qsl[s + 1] - q0;
        const int i0 = qp * 2 * QT;  // first chunk token of query tile A; tile B follows
        if (i0 >= L) continue;       // segment-uniform, before any barrier or TMEM use
        const int ctx = P.ctx[s];
        if (ctx < L) {  // the chunk must be in the cache already
            if (threadIdx.x == 0) pa::set_error(P.err, PA_DEVERR_CONTEXT);
            continue;
        }
        const int nblk = min((ctx + kBS - 1) / kBS, P.max_blocks);
        const int first_pos = ctx - L;
        // both tiles walk the key tiles up to the last row of the pair (tile A's
        // extra tiles beyond its own rows are fully masked)
        const int p_last = first_pos + min(i0 + 2 * QT, L) - 1;
        const int n_kt_all = p_last / kKT + 1;
        if (!P.work) {  // this CTA's piece of the key tiles (all of them when not split)
            const int sp = blockIdx.x % P.splits;
            piece_range(n_kt_all, sp, P.splits, kt0, kt1);
            direct = P.splits <= 1;
            if (!direct) {
                const size_t item = ((size_t)s * Hk + kvh) * (gridDim.x / P.splits) + qp;
                part_base = P.part + (item * P.splits + sp) * 2 * 128 * kPartStride;
            }
        }
        kt1 = min(kt1, n_kt_all);
        const int n_kt = kt1 - kt0;  // tiles this segment walks; local tile j is key tile kt0 + j
        if (n_kt <= 0) continue;     // segment-uniform; the merge skips empty pieces

        if (threadIdx.x == 0) {
            if (n_run > 0) {  // every phase of the last segment has completed
                for (int b = 0; b < kNumBars; ++b) pa::mbar_inval(&bars[b]);
            } else {
                *abort_flag = 0;
            }
            for (int i = 0; i < kKS; ++i) {
                pa::mbar_init(&k_full[i], 1);
                pa::mbar_init(&k_free[i], 1);
            }
            for (int i = 0; i < kVS; ++i) {
                pa::mbar_init(&v_full[i], 1);
                pa::mbar_init(&v_free[i], 1);
                pa::mbar_init(&v_conv[i], 4);
            }
            for (int x = 0; x < 2; ++x) {
                pa::mbar_init(&s_full[x], 1);
                pa::mbar_init(&pv_done[x], 1);
            }
            pa::mbar_init(drain, 1);
            pa::fence_mbar_init();
        }
        if (warp == 0 && !have_tmem) {
            tc::tmem_alloc(tslot, kTmemCols);
            tc::tmem_relinquish();
        }
        // ---- Q tiles: tile X row r = (chunk token i0 + X*QT + r/G, head h0 + r%G)
        if (warp < 8) {
            const int x = warp >> 2, r = threadIdx.x & 127;
            const int i = i0 + x * QT + r / G;
            const uint4* src = reinterpret_cast<const uint4*>(P.q + ((size_t)(q0 + i) * H + h0 + r % G) * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = i < L ? src[c] : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + kQ + x * kQTile + (c >> 3) * 16384 + tc::sw128_offset(r, c & 7)) = v;
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        tbase = *tslot;
        have_tmem = true;

        constexpr uint32_t ID_QK = tc::idesc_bf16_f32(128, 128, 0, 0);
        constexpr uint32_t ID_PV = idesc_f16_f32(128, D, 0, 1);

        if (warp == 9) {
            // ------------------------------------------------------- TMA producer
            // K(j) goes to K stage j%2 once both QKs of K(j-2) are done (k_free);
            // V(j) to V stage j%3 once PV_B(j-3), the last reader of V(j-3), is
            // done. K(j) is issued before V(j), and V(j) before K(j+1).
            const int32_t* trow = P.tables + (size_t)s * P.max_blocks;
            struct Ids { int ids = -1, group = -1; };  // block ids of key tiles 4g..4g+3, one per lane
            Ids idk, idv;
            auto issue_tile = [&](Ids& w, const CUtensorMap* map, unsigned char* dst, uint64_t* bar, int j) {
                if ((j >> 2) != w.group) {  // warp-collective
                    w.group = j >> 2;
                    const int blk = w.group * 32 + lane;
                    w.ids = blk < nblk ? trow[blk] : -1;
                }
                // lane l < 8 * kNH moves box (block b = l / kNH, dims 64 g .. 64 g + 63, g = l % kNH)
                const int b = (lane / kNH) & (kBPT - 1), g = lane % kNH;
                const int bid = __shfl_sync(kFull, w.ids, (j & 3) * kBPT + b);
                const int blk = j * kBPT + b;
                bool ok = blk < nblk;
                if (ok && (bid < 0 || bid >= P.num_blocks)) {
                    if (lane < kNH * kBPT && g == 0) pa::set_error(P.err, PA_DEVERR_BLOCK_ID);
                    ok = false;
                }
                const int y = ok ? (bid * Hk + kvh) * kBS : P.oob_row;  // out of range: zero fill
                if (lane == 0) pa::mbar_arrive_expect_tx(bar, kTile);
                __syncwarp();
                if (lane < kNH * kBPT) tc::tma_load_2d(dst + g * 16384 + b * 2048, map, g * 64, y, bar);
                __syncwarp();
            };
            auto issue_k = [&](int j) {
                issue_tile(idk, &tmK, sm + kK0 + (j % kKS) * kTile, &k_full[j % kKS], kt0 + j);
            };
            auto issue_v = [&](int j) {
                issue_tile(idv, &tmV, sm + kV0 + (j % kVS) * kTile, &v_full[j % kVS], kt0 + j);
            };
            int nk = 0, nv = 0;  // loads issued
            bool ok = true;
            for (; nk < kKS && nk < n_kt; ++nk) issue_k(nk);
            for (; nv < kVS && nv < n_kt; ++nv) issue_v(nv);
            while (ok && (nk < n_kt || nv < n_kt)) {
                if (nk < n_kt && nk <= nv) {  // K(nk) replaces K(nk-2)
                    ok = wait_bar(&k_free[nk % kKS], (uint32_t)(((nk - kKS) / kKS) & 1), P.err, abort_flag);
                    if (!ok) break;
                    issue_k(nk++);
                } else {  // V(nv) replaces V(nv-3)
                    ok = wait_bar(&v_free[nv % kVS], (uint32_t)(((nv - kVS) / kVS) & 1), P.err, abort_flag);
                    if (!ok) break;
                    issue_v(nv++);
                }
            }
            // every issued copy has landed before the CTA may exit (bounded; in
            // the normal case the MMA warp has already consumed them all)
            for (int t = (nk > kKS ? nk - kKS : 0); t < nk; ++t)
                pa::mbar_wait(&k_full[t % kKS], (uint32_t)((t / kKS) & 1), nullptr, 5000000ull);
            for (int t = (nv > kVS ? nv - kVS : 0); t < nv; ++t)
                pa::mbar_wait(&v_full[t % kVS], (uint32_t)((t / kVS) & 1), nullptr, 5000000ull);
        } else if (warp == 8) {
            // ---------------------------------------------------------- MMA issuer
            // One thread issues every MMA. Its waits for data that is normally
            // ready long before (the V tile's conversion, the next K tile) come
            // before its wait for a tile's P, so that P.V and the next Q.K^T of a
            // tile are issued back to back once the softmax hands P over.
            // Matrix descriptors differ only in the start-address field (bits
            // 0-13, byte address / 16); every operand lies inside the shared
            // allocation, so offsets added to the low word never leave the field.
            // The hand-over of each tile's P is a named barrier (ids 1 and 2, the
            // four softmax warps arrive, this warp syncs): every segment has
            // exactly n_kt arrivals of each softmax warpgroup and n_kt syncs here,
            // also after a failed wait, so neither side can be left waiting.
            const uint64_t dq = tc::smem_desc(pa::smem_u32(sm + kQ), 16, 1024);
            const uint64_t dk = tc::smem_desc(pa::smem_u32(sm + kK0), 16, 1024);
            const uint64_t dv = tc::smem_desc(pa::smem_u32(sm + kV0), 16384, 1024);
            auto at = [](uint64_t d, uint32_t off16) {
                return ((uint64_t)(uint32_t)(d >> 32) << 32) | (uint32_t)((uint32_t)d + off16);
            };
            auto issue_qk = [&](int x, int kst) {  // S_x = Q_x K^T, K in stage kst (one thread)
                const uint32_t qo = x * (kQTile >> 4), ko = kst * (kTile >> 4);
                const uint32_t dst = tbase + x * 256;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t o = ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4;
                    tc::mma_bf16(dst, at(dq, qo + o), at(dk, ko + o), ID_QK, ks > 0 ? 1u : 0u);
                }
                if (x == 1) tc::mma_commit(&k_free[kst]);  // the stage's last reader
                tc::mma_commit(&s_full[x]);
            };
            auto issue_pv = [&](int x, int vst, bool first) {  // O_x += P V (fp16), V in stage vst (one thread)
                const uint32_t vo = vst * (kTile >> 4);
                const uint32_t pcol = tbase + x * 256, dst = pcol + 128;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16_ts(dst, pcol + (ks >> 1) * 32 + (ks & 1) * 8, at(dv, vo + ks * (2048 >> 4)),
                                    ID_PV, (!first || ks > 0) ? 1u : 0u);  // fp16 operands per ID_PV
                if (x == 1) tc::mma_commit(&v_free[vst]);  // the stage's last reader
                tc::mma_commit(&pv_done[x]);
            };
            // The tensor core runs the MMAs of this thread in issue order, so
            // QK_x(j+1) may follow PV_x(j) (which reads P out of S_x's columns)
            // without a wait.
            bool ok = wait_bar(&k_full[0], 0, P.err, abort_flag);
            ok = __all_sync(kFull, ok);
            if (ok && lane == 0) {
                tc::fence_after_sync();
                issue_qk(0, 0);
                issue_qk(1, 0);
            }
            __syncwarp();
            int kst = 1, kph = 0;  // stage and phase parity of K(j+1)
            int vst = 0, vph = 0;  // stage and phase parity of V(j)
            for (int j = 0; j < n_kt; ++j) {
                const bool more = j + 1 < n_kt;
                if (ok) ok = wait_bar(&v_conv[vst], (uint32_t)vph, P.err, abort_flag);
                if (ok && more) ok = wait_bar(&k_full[kst], (uint32_t)kph, P.err, abort_flag);
                ok = __all_sync(kFull, ok);
                asm volatile("bar.sync 1, 160;" ::: "memory");  // tile A's P is in tensor memory
                if (ok && lane == 0) {
                    tc::fence_after_sync();
                    issue_pv(0, vst, j == 0);
                    if (more) issue_qk(0, kst);
                }
                __syncwarp();
                asm volatile("bar.sync 2, 160;" ::: "memory");  // tile B's P
                if (ok && lane == 0) {
                    tc::fence_after_sync();
                    issue_pv(1, vst, j == 0);
                    if (more) issue_qk(1, kst);
                }
                __syncwarp();
                if (++vst == kVS) { vst = 0; vph ^= 1; }
                if (++kst == kKS) { kst = 0; kph ^= 1; }
            }
            // drain: every issued MMA has completed before the CTA can release its
            // shared and tensor memory (bounded wait)
            if (lane == 0) tc::mma_commit(drain);
            __syncwarp();
            pa::mbar_wait(drain, 0, nullptr, 10000000ull);
            if (ok && lane == 0) {  // the stages' last frees (never waited for) land before the barriers are reused
                for (int t = max(0, n_kt - kKS); t < n_kt; ++t)
                    pa::mbar_wait(&k_free[t % kKS], (uint32_t)((t / kKS) & 1), nullptr, 10000000ull);
                for (int t = max(0, n_kt - kVS); t < n_kt; ++t)
                    pa::mbar_wait(&v_free[t % kVS], (uint32_t)((t / kVS) & 1), nullptr, 10000000ull);
            }
            __syncwarp();
        } else if (warp >= 10) {
            // ------------------------------------------------------ V converters
            // Thread t of 128 (four warps, one per scheduler) rewrites the 16-byte
            // chunks t, t + 128, ... of the landed tile (consecutive threads,
            // consecutive chunks). A chunk holds
            // 8 consecutive values of one key row: row (chunk % 1024) / 8 of
            // either 64-dim half, wherever the swizzle put the chunk in the row.
            const int t = threadIdx.x - 320;  // 0..127
            const float2 k2 = make_float2(0.00390625f, 0.00390625f);  // 2^-8
            auto cvt = [&](uint32_t u) {  // bf16 pair -> fp16 pair of v * 2^-8
                const float2 f = __fmul2_rn(make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u)), k2);
                return float2_to_f16x2(f.x, f.y);
            };
            bool ok = true;
            for (int j = 0; j < n_kt && ok; ++j) {
                ok = wait_bar(&v_full[j % kVS], (uint32_t)((j / kVS) & 1), P.err, abort_flag);
                ok = __all_sync(kFull, ok);
                if (!ok) break;
                const int kb = (kt0 + j) * kKT;
                uint4* vs = reinterpret_cast<uint4*>(sm + kV0 + (j % kVS) * kTile);
                const int valid = ctx - kb;  // key rows of this tile inside the context (may exceed 128)
                auto convert = [&](auto partial) {
#pragma unroll 4
                    for (int c = 0; c < (int)(kTile / 2048); ++c) {
                        const int e = t + 128 * c;
                        uint4 w = vs[e];
                        if constexpr (decltype(partial)::value)
                            if (((e & 1023) >> 3) >= valid) w = make_uint4(0, 0, 0, 0);
                        w.x = cvt(w.x);
                        w.y = cvt(w.y);
                        w.z = cvt(w.z);
                        w.w = cvt(w.w);
                        vs[e] = w;
                    }
                };
                if (valid < kKT) convert(std::true_type{});  // the context ends inside this tile
                else convert(std::false_type{});
                tc::fence_async_smem();  // generic-proxy writes, read next by the tensor core
                __syncwarp();
                if (lane == 0) pa::mbar_arrive(&v_conv[j % kVS]);
            }
        } else {
            // --------------------------------------- softmax warpgroup of tile x
            // warp w serves TMEM lanes 32*(w%4) .. +31 (rows). After a failed wait
            // (timeout) the warps keep iterating without waiting.
            //
            // One pass over S per key tile, a quarter of 32 columns at a time:
            // p = 2^(s*scale - m) against the row's current reference m, which is
            // an integer (or -inf before the row has seen a key), so every change
            // of m rescales by an exact power of two. m changes only when a
            // quarter's sum of p exceeds 2^15, i.e. before any p could leave the
            // fp16 range (65504), and on a row's first visible quarter (m = -inf
            // gives p = inf): the quarter is then recomputed against
            // m = ceil(max s*scale of the quarter) (its p <= 1), and the P of the
            // tile's earlier quarters, already in tensor memory, is rescaled in
            // place (fp16 times a power of two: exact down to the subnormals).
            const int x = warp >> 2;
            const int r = threadIdx.x & 127;  // matrix row = TMEM lane
            const int i = i0 + x * QT + r / G;
            const int pos = first_pos + i;  // this row's position (padding rows: beyond the chunk)
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t tS = tbase + x * 256 + lane_base;
            const uint32_t tO = tS + 128;
            const float sc = P.scale_log2;
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = 0; j < n_kt; ++j) {
                if (ok) ok = wait_bar(&s_full[x], (uint32_t)(j & 1), P.err, abort_flag);
                ok = __all_sync(kFull, ok);
                tc::fence_after_sync();
                const int kb = (kt0 + j) * kKT;
                // Keys beyond a row's position are masked. Only the tiles on the
                // diagonal have such keys; a warp takes the masking code only when
                // one of its rows needs it (a warp-uniform branch), so the other
                // tiles run the plain loop.
                const bool mask_warp = __any_sync(kFull, kb + kKT - 1 > pos);
                const int lim0 = pos - kb;  // keys k > lim0 of the tile are not visible
                float2 psum2 = make_float2(0.f, 0.f);  // this tile's sum of p against m_used
                float alpha = 1.f;                     // this tile's rescale of l and O
                const float2 sc2 = make_float2(sc, sc);
                // p of one quarter (raw scores in columns 32q..32q+31) -> fp16 pairs;
                // P of keys 2w, 2w+1 goes to column 32q + w, so a quarter only
                // overwrites columns it has already read.
                auto exps = [&](auto masked, const uint32_t (&raw)[32], int qd, uint32_t (&ph)[16]) {
                    const float2 nm2 = make_float2(-m_used, -m_used);
                    float2 qs = make_float2(0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < 16; ++w) {
                        float2 e = __ffma2_rn(make_float2(__uint_as_float(raw[2 * w]), __uint_as_float(raw[2 * w + 1])),
                                              sc2, nm2);
                        if constexpr (decltype(masked)::value) {  // masked keys give p = 0 (also for a zero scale)
                            const int k = 32 * qd + 2 * w;
                            if (k > lim0) e.x = -INFINITY;
                            if (k + 1 > lim0) e.y = -INFINITY;
                        }
                        e.x = pa::fast_exp2(e.x);
                        e.y = pa::fast_exp2(e.y);
                        qs = __fadd2_rn(qs, e);
                        ph[w] = float2_to_f16x2(e.x, e.y);
                    }
                    return qs.x + qs.y;
                };
                auto sweep = [&](auto masked) {
#pragma unroll 1
                    for (int qd = 0; qd < 4; ++qd) {
                        uint32_t raw[32];
                        tc::tmem_ld32(tS + 32 * qd, raw);
                        tc::tmem_wait_ld();
                        uint32_t ph[16];
                        float qs = exps(masked, raw, qd, ph);
                        const bool big = !(qs <= 32768.f);  // also inf (no reference yet) and NaN
                        if (__any_sync(kFull, big)) {
                            // rare: a new reference for the rows that need one
                            float a = 1.f;
                            if (big) {
                                float qmax = -INFINITY;
#pragma unroll
                                for (int k = 0; k < 32; ++k) {
                                    const bool vis = !decltype(masked)::value || 32 * qd + k <= lim0;
                                    if (vis) qmax = fmaxf(qmax, __uint_as_float(raw[k]));
                                }
                                const float mq = ceilf(qmax * sc);
                                if (mq > m_used) {
                                    // 2^(m_used - mq) built from its exponent bits (0 below 2^-126)
                                    const float d = m_used - mq;
                                    a = d < -126.f ? 0.f : __int_as_float(((int)d + 127) << 23);
                                    m_used = mq;
                                    qs = exps(masked, raw, qd, ph);
                                }
                            }
                            psum2.x *= a;
                            psum2.y *= a;
                            alpha *= a;
                            if (qd > 0) {  // P of the earlier quarters, in place (warp-collective)
                                tc::tmem_wait_st();
                                // in fp32: the factor itself may lie below fp16's range
                                // (2^-25 would round to 0 as a half) while the products
                                // (P <= 2^15) do not
#pragma unroll 1
                                for (int q2 = 0; q2 < qd; ++q2) {
                                    uint32_t pp[16];
                                    tc::tmem_ld16(tS + 32 * q2, pp);
                                    tc::tmem_wait_ld();
#pragma unroll
                                    for (int w = 0; w < 16; ++w) {
                                        const float2 f = __half22float2(*reinterpret_cast<__half2*>(&pp[w]));
                                        pp[w] = float2_to_f16x2(f.x * a, f.y * a);
                                    }
                                    tc::tmem_st16(tS + 32 * q2, pp);
                                }
                            }
                        }
                        psum2.x += qs;
                        tc::tmem_st16(tS + 32 * qd, ph);
                    }
                };
                if (mask_warp) sweep(std::true_type{});
                else sweep(std::false_type{});
                l = l * alpha + (psum2.x + psum2.y);
                // a new reference rescales O_x: PV_x(j-1) must have landed first
                if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
                    if (ok) ok = wait_bar(&pv_done[x], (uint32_t)((j - 1) & 1), P.err, abort_flag);
                    ok = __all_sync(kFull, ok);
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t raw[32];
                        tc::tmem_ld32(tO + c * 32, raw);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) raw[k] = __float_as_uint(__uint_as_float(raw[k]) * alpha);
                        tc::tmem_st32(tO + c * 32, raw);
                    }
                }
                tc::tmem_wait_st();
                tc::fence_before_sync();
                __syncwarp();
                asm volatile("bar.arrive %0, 160;" ::"r"(1 + x) : "memory");  // P handed to the MMA warp
            }
            tc::tmem_wait_st();  // no store may be pending when the columns are released
            if (ok) ok = wait_bar(&pv_done[x], (uint32_t)((n_kt - 1) & 1), P.err, abort_flag);
            ok = __all_sync(kFull, ok);
            if (ok && !direct) {
                // a piece: keep O, m and l for the merge
                tc::fence_after_sync();
                float* dst = part_base + ((size_t)x * 128 + r) * kPartStride;
                bool finite = true;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t raw[32];
                    tc::tmem_ld32(tO + c * 32, raw);
                    tc::tmem_wait_ld();
                    if (i < L) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            raw[k] = __float_as_uint(__uint_as_float(raw[k]) * 256.f);  // undo V's 2^-8
                            finite &= (raw[k] & 0x7f800000u) != 0x7f800000u;
                        }
#pragma unroll
                        for (int k = 0; k < 32; k += 4)
                            *reinterpret_cast<float4*>(dst + c * 32 + k) =
                                make_float4(__uint_as_float(raw[k]), __uint_as_float(raw[k + 1]),
                                            __uint_as_float(raw[k + 2]), __uint_as_float(raw[k + 3]));
                    }
                }
                if (!finite) pa::set_error(P.err, PA_DEVERR_RANGE);
                if (i < L) *reinterpret_cast<float2*>(dst + kPartML) = make_float2(m_used, l);
            } else if (ok) {
                tc::fence_after_sync();
                const float inv = 256.f / l;  // with V's 2^-8 undone
                uint4* dst = reinterpret_cast<uint4*>(P.out + ((size_t)(q0 + i) * H + h0 + r % G) * D);
                bool finite = true;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t raw[32];
                    tc::tmem_ld32(tO + c * 32, raw);
                    tc::tmem_wait_ld();
                    if (i < L) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) finite &= (raw[k] & 0x7f800000u) != 0x7f800000u;
#pragma unroll
                        for (int k = 0; k < 32; k += 8) {
                            uint4 w;
                            w.x = pa::float2_to_bf16x2(__uint_as_float(raw[k]) * inv, __uint_as_float(raw[k + 1]) * inv);
                            w.y = pa::float2_to_bf16x2(__uint_as_float(raw[k + 2]) * inv, __uint_as_float(raw[k + 3]) * inv);
                            w.z = pa::float2_to_bf16x2(__uint_as_float(raw[k + 4]) * inv, __uint_as_float(raw[k + 5]) * inv);
                            w.w = pa::float2_to_bf16x2(__uint_as_float(raw[k + 6]) * inv, __uint_as_float(raw[k + 7]) * inv);
                            dst[(c * 32 + k) / 8] = w;
                        }
                    }
                }
                if (!finite) pa::set_error(P.err, PA_DEVERR_RANGE);
            }
        }
        tc::fence_before_sync();
        __syncthreads();  // end of the segment: every role is done with smem, TMEM and the barriers
        ++n_run;
    }  // segments
    if (have_tmem && warp == 0) tc::tmem_dealloc(tbase, kTmemCols);
}

// Key tiles of item it = (sequence * n_kv_heads + kv head) * n_qp + pair:
// 0 if the pair has no rows. A chunk that is not in the cache (ctx < L) has
// none either, and flags the device error once per sequence.
template <int G>
__device__ int item_tiles(const PrefillParams& P, int it) {
    constexpr int QT = kRows / G;
    const int per_seq = P.n_kv_heads * P.n_qp;
    const int s = it / per_seq, qp = it % P.n_qp;
    const int q0 = P.qsl[s], L = P.qsl[s + 1] - q0, i0 = qp * 2 * QT;
    if (i0 >= L) return 0;
    const int ctx = P.ctx[s];
    if (ctx < L) {
        if (it % per_seq == 0) pa::set_error(P.err, PA_DEVERR_CONTEXT);
        return 0;
    }
    return (ctx - L + min(i0 + 2 * QT, L) - 1) / kKT + 1;
}

// Balanced mode: the work list. One block of 1024 threads, each a run of
// consecutive items. With P non-empty items and C CTAs (one per SM), the
// first P - R items run whole (full waves, in item order so that the pairs of
// one KV head run side by side and share their K/V tiles in L2); the last
// R = P mod C items would fill only part of a wave, so each is cut into S
// equal key ranges, S (1..8, R*S <= 4C) minimising ceil(R*S/C)/S + 0.03 S
// (the wave fraction the tail takes plus a per-piece cost); its pieces are
// listed piece-major, so the pieces running together again share key ranges.
template <int G>
__global__ void __launch_bounds__(1024) pa_prefill_plan_kernel(const PrefillParams P) {
    __shared__ int wsum[32];
    __shared__ int sh[3];  // P, R, S
    const int n = P.n_items, t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int per = (n + 1023) / 1024;
    const int b0 = min(n, t * per), b1 = min(n, b0 + per);
    int mine = 0;
    for (int it = b0; it < b1; ++it) mine += item_tiles<G>(P, it) > 0;
    int incl = mine;  // inclusive count within the warp
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += y;
        }
        wsum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    if (t == 0) {
        const int np = wsum[31], C = P.n_cta;
        int R = np % C, S = 1;
        float best = 2.f;
        for (int c = 1; c <= 8 && R * c <= 4 * C; ++c) {
            const float cost = (float)((R * c + C - 1) / C) / c + 0.03f * c;
            if (cost < best) {
                best = cost;
                S = c;
            }
        }
        if (S == 1) R = 0;  // no cut: the tail runs whole
        sh[0] = np;
        sh[1] = R;
        sh[2] = S;
        P.sched[0] = 0;
        P.sched[1] = np - R + R * S;
        P.sched[2] = S;
        P.sched[3] = R;
    }
    __syncthreads();
    const int np = sh[0], R = sh[1], S = sh[2], whole = np - R;
    int rank = incl - mine + (wid > 0 ? wsum[wid - 1] : 0);
    for (int it = b0; it < b1; ++it) {
        const int nk = item_tiles<G>(P, it);
        if (nk <= 0) continue;
        if (rank < whole) {
            P.work[rank] = make_int4(it, 0, nk, -1);
        } else {
            const int ti = rank - whole;
            for (int sp = 0; sp < S; ++sp) {
                int a, b;
                piece_range(nk, sp, S, a, b);
                P.work[whole + sp * R + ti] = make_int4(it, a, b, ti * S + sp);
            }
        }
        ++rank;
    }
}

// Combines the pieces of one output row: O = sum_k O_k 2^(m_k - M),
// l = sum_k l_k 2^(m_k - M), out = O / l (lane: D / 32 consecutive dims).
// Piece k covers key tiles piece_range(n_kt_all, k, n_pieces); empty ones
// wrote nothing and are skipped. Up to 8 pieces: every lane loads every
// piece's (m, l) (one broadcast load each) and its O slices, all at once, so
// the row costs one round of memory latency. More pieces (n_pieces <= 64):
// lane k reads piece k's (m, l), then the O slices are loaded 8 pieces at a
// time.
template <int NV>
__device__ __forceinline__ void store_row(const float (&acc)[NV], float inv, int lane, uint16_t* out_row) {
    if constexpr (NV == 4) {
        uint2 pk;
        pk.x = pa::float2_to_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pa::float2_to_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(out_row + lane * 4) = pk;
    } else {
        *reinterpret_cast<uint32_t*>(out_row + lane * 2) = pa::float2_to_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}
template <int NV>
__device__ __forceinline__ void load_slice(const float* src, int lane, float (&v)[NV]) {
    if constexpr (NV == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src + lane * 4);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2*>(src + lane * 2);
        v[0] = t.x; v[1] = t.y;
    }
}
template <int D, typename PartOf>
__device__ __forceinline__ void merge_row(int n_pieces, int n_kt_all, PartOf part_of, int lane, uint16_t* out_row) {
    constexpr int NV = D / 32;  // dims per lane: 4 or 2
    if (n_pieces <= 8) {
        float v[8][NV];
        float2 ml[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            int a = 0, b = 0;
            if (k < n_pieces) piece_range(n_kt_all, k, n_pieces, a, b);
            ml[k] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int e = 0; e < NV; ++e) v[k][e] = 0.f;
            if (b > a) {
                const float* src = part_of(k);
                ml[k] = *reinterpret_cast<const float2*>(src + kPartML);
                load_slice<NV>(src, lane, v[k]);
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < 8; ++k) M = fmaxf(M, ml[k].x);
        float l = 0.f, acc[NV] = {};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float f = ml[k].x == -INFINITY ? 0.f : pa::fast_exp2(ml[k].x - M);
            l += ml[k].y * f;
#pragma unroll
            for (int e = 0; e < NV; ++e) acc[e] += v[k][e] * f;
        }
        store_row<NV>(acc, 1.f / l, lane, out_row);
        return;
    }
    float m_mine = -INFINITY, l_mine = 0.f;
    for (int k = lane; k < n_pieces; k += 32) {
        int a, b;
        piece_range(n_kt_all, k, n_pieces, a, b);
        if (b > a) {
            const float2 ml = *reinterpret_cast<const float2*>(part_of(k) + kPartML);
            if (ml.x > m_mine) {  // keep the larger reference; rescale the other sum
                l_mine = l_mine * (m_mine == -INFINITY ? 0.f : pa::fast_exp2(m_mine - ml.x)) + ml.y;
                m_mine = ml.x;
            } else {
                l_mine += ml.x == -INFINITY ? 0.f : ml.y * pa::fast_exp2(ml.x - m_mine);
            }
        }
    }
    float M = m_mine;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    float l = m_mine == -INFINITY ? 0.f : l_mine * pa::fast_exp2(m_mine - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
    float acc[NV] = {};
    for (int k0 = 0; k0 < n_pieces; k0 += 8) {
        float v[8][NV];
        float f[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int k = k0 + u;
            int a = 0, b = 0;
            if (k < n_pieces) piece_range(n_kt_all, k, n_pieces, a, b);
            f[u] = 0.f;
#pragma unroll
            for (int e = 0; e < NV; ++e) v[u][e] = 0.f;
            if (b > a) {
                const float* src = part_of(k);
                const float m = src[kPartML];
                f[u] = m == -INFINITY ? 0.f : pa::fast_exp2(m - M);
                load_slice<NV>(src, lane, v[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int e = 0; e < NV; ++e) acc[e] += v[u][e] * f[u];
    }
    store_row<NV>(acc, 1.f / l, lane, out_row);
}

// Per-pair mode with splits > 1: one warp per (chunk row, query head).
template <int G, int D>
__global__ void __launch_bounds__(128)
pa_prefill_merge_kernel(const PrefillParams P, int n_seqs, int n_rows_total, int n_qp) {
    constexpr int QT = kRows / G;
    pa::grid_dependency_wait();  // every piece's partial is written
    const long long w = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int H = P.n_heads, Hk = P.n_kv_heads;
    if (w >= (long long)n_rows_total * H) return;
    const int t = (int)(w / H), h = (int)(w % H);
    // the sequence whose chunk holds row t: the last s with qsl[s] <= t
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.qsl[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int q0 = P.qsl[s], L = P.qsl[s + 1] - q0, ctx = P.ctx[s];
    const int i = t - q0;
    if (i < 0 || i >= L || ctx < L) return;
    const int qp = i / (2 * QT), x = (i % (2 * QT)) / QT, r = (i % QT) * G + h % G, kvh = h / G;
    const int i0 = qp * 2 * QT;
    const int n_kt_all = (ctx - L + min(i0 + 2 * QT, L) - 1) / kKT + 1;
    const size_t item = ((size_t)s * Hk + kvh) * n_qp + qp;
    merge_row<D>(P.splits, n_kt_all,
                 [&](int k) { return P.part + (((item * P.splits + k) * 2 + x) * 128 + r) * kPartStride; }, lane,
                 P.out + ((size_t)t * H + h) * D);
}

// Balanced mode: one warp per (row, head) of the cut pairs, warp w = 256 *
// (cut pair) + 128 * (query tile) + (tile row); the cut pairs are the
// piece-0 entries of the work list's tail.
template <int G, int D>
__global__ void __launch_bounds__(128) pa_prefill_merge_cut_kernel(const PrefillParams P) {
    constexpr int QT = kRows / G;
    pa::grid_dependency_wait();  // every piece's partial is written
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int S = P.sched[2], R = P.sched[3];
    const int t = w >> 8, x = (w >> 7) & 1, r = w & 127;
    if (t >= R) return;
    const int item = P.work[P.sched[1] - R * S + t].x;
    const int Hk = P.n_kv_heads;
    const int s = item / (Hk * P.n_qp), kvh = (item / P.n_qp) % Hk, qp = item % P.n_qp;
    const int q0 = P.qsl[s], L = P.qsl[s + 1] - q0, ctx = P.ctx[s];
    const int i0 = qp * 2 * QT, i = i0 + x * QT + r / G;
    if (i >= L) return;
    const int n_kt_all = (ctx - L + min(i0 + 2 * QT, L) - 1) / kKT + 1;
    const size_t slot0 = (size_t)t * S;
    merge_row<D>(S, n_kt_all, [&](int k) { return P.part + (((slot0 + k) * 2 + x) * 128 + r) * kPartStride; },
                 lane, P.out + ((size_t)(q0 + i) * P.n_heads + kvh * G + r % G) * D);
}

template <int G, int D>
int launch_prefill(const PrefillParams& Pp, const CUtensorMap& tk, const CUtensorMap& tv, int n_seqs,
                   int max_chunk_len, int n_rows, cudaStream_t stream) {
    auto kern = pa_prefill_tc_kernel<G, D>;
    constexpr uint32_t kSmemBytes = PfLay<D>::kSmem;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        attr_done[dev] = true;
    }
    constexpr int QT = kRows / G;
    const int n_qp = (max_chunk_len + 2 * QT - 1) / (2 * QT);
    if (Pp.work) {  // balanced mode: plan, then one CTA per SM taking work-list entries
        pa_prefill_plan_kernel<G><<<1, 1024, 0, stream>>>(Pp);
        kern<<<Pp.n_cta, kThreads, kSmemBytes, stream>>>(Pp, tk, tv);
    } else {
        dim3 grid(n_qp * Pp.splits, Pp.n_kv_heads, n_seqs);
        kern<<<grid, kThreads, kSmemBytes, stream>>>(Pp, tk, tv);
    }
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (Pp.work)  // the cut pairs (fewer than one per CTA): 256 rows each
        return pa_launch_pdl(pa_prefill_merge_cut_kernel<G, D>, dim3((unsigned)Pp.n_cta * 64), dim3(128), 0, stream,
                             Pp);
    if (Pp.splits <= 1) return PA_OK;
    // rows of all chunks: the merge finds each row's sequence in q_start_loc
    const long long warps = (long long)n_rows * Pp.n_heads;
    return pa_launch_pdl(pa_prefill_merge_kernel<G, D>, dim3((unsigned)((warps + 3) / 4)), dim3(128), 0, stream, Pp,
                         n_seqs, n_rows, n_qp);
}

}  // namespace

namespace {

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev] && cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        cached[dev] = 0;
    return cached[dev];
}

int pairs_per_seq(int G, int max_chunk_len) {
    const int QT = kRows / G;
    return (max_chunk_len + 2 * QT - 1) / (2 * QT);
}

size_t part_bytes(long long n_items, int splits) {
    return splits > 1 ? (size_t)n_items * splits * 2 * 128 * kPartStride * sizeof(float) : 0;
}

// Balanced mode (splits = 0): partial slots for the cut items (at most 4
// per CTA), the work list (n_items + 4 * n_cta entries) and the counters,
// each part 16-byte aligned.
struct BalancedLayout {
    size_t part, work, sched, total;
};
BalancedLayout balanced_layout(long long n_items, int n_cta) {
    BalancedLayout b;
    b.part = 0;
    b.work = (size_t)4 * n_cta * 2 * 128 * kPartStride * sizeof(float);
    b.sched = b.work + (size_t)(n_items + 4LL * n_cta) * sizeof(int4);
    b.total = b.sched + 16;
    return b;
}

int prefill_impl(void* out, const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                 const int32_t* context_lens, const int32_t* q_start_loc, float scale, int n_heads,
                 int n_kv_heads, int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                 int max_chunk_len, int num_blocks, int splits, void* workspace, size_t workspace_bytes,
                 pa_stream_t stream) {
    if (n_seqs < 0 || max_chunk_len < 0 || num_blocks < 0 || max_blocks_per_seq < 0 || n_heads <= 0 ||
        n_kv_heads <= 0 || splits < 0 || splits > 64)
        return PA_ERR_INVALID_ARG;
    if ((head_dim != 64 && head_dim != 128) || block_size != kBS) return PA_ERR_UNSUPPORTED;
    if (n_heads % n_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int G = n_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    if (n_seqs == 0 || max_chunk_len == 0) return PA_OK;
    if (n_kv_heads > 65535 || n_seqs > 65535) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens || !q_start_loc)
        return PA_ERR_INVALID_ARG;
    if (!pa_aligned16(out) || !pa_aligned16(q) || !pa_aligned16(k_pool) || !pa_aligned16(v_pool))
        return PA_ERR_INVALID_ARG;
    if (out == q) return PA_ERR_INVALID_ARG;
    const long long rows = (long long)num_blocks * n_kv_heads * kBS;
    if (rows + kBS > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
    const int n_qp = pairs_per_seq(G, max_chunk_len);
    const long long n_items = (long long)n_qp * n_kv_heads * n_seqs;
    if (n_items > 0x3fffffffLL) return PA_ERR_UNSUPPORTED;
    const int n_cta = splits == 0 ? sm_count() : 0;
    if (splits == 0 && n_cta <= 0) return PA_ERR_CUDA;
    if ((long long)n_qp * (splits > 0 ? splits : 1) > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    const size_t need = splits == 0 ? balanced_layout(n_items, n_cta).total : part_bytes(n_items, splits);
    if (need > 0 && (!workspace || workspace_bytes < need || !pa_aligned16(workspace))) return PA_ERR_WORKSPACE;
    unsigned int* err = pa_device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    CUtensorMap tk, tv;
    if (!pa_make_tmap_2d_bf16(&tk, k_pool, head_dim, (uint64_t)rows, head_dim * 2, 64, kBS) ||
        !pa_make_tmap_2d_bf16(&tv, v_pool, head_dim, (uint64_t)rows, head_dim * 2, 64, kBS))
        return PA_ERR_CUDA;
    PrefillParams Pp;
    Pp.out = static_cast<uint16_t*>(out);
    Pp.q = static_cast<const uint16_t*>(q);
    Pp.tables = block_tables;
    Pp.ctx = context_lens;
    Pp.qsl = q_start_loc;
    Pp.scale_log2 = scale * 1.4426950408889634f;
    Pp.n_heads = n_heads;
    Pp.n_kv_heads = n_kv_heads;
    Pp.max_blocks = max_blocks_per_seq;
    Pp.num_blocks = num_blocks;
    Pp.oob_row = (int)rows;
    Pp.splits = splits > 0 ? splits : 1;
    Pp.part = need ? static_cast<float*>(workspace) : nullptr;
    Pp.work = nullptr;
    Pp.sched = nullptr;
    if (splits == 0) {
        const BalancedLayout bl = balanced_layout(n_items, n_cta);
        char* w = static_cast<char*>(workspace);
        Pp.work = reinterpret_cast<int4*>(w + bl.work);
        Pp.sched = reinterpret_cast<int*>(w + bl.sched);
    }
    Pp.n_items = (int)n_items;
    Pp.n_qp = n_qp;
    Pp.n_cta = n_cta;
    Pp.err = err;
    // chunk rows bound for the merge grid (rows past the last chunk exit)
    const long long n_rows = (long long)n_seqs * max_chunk_len;
    if (n_rows > 0x7fffffffLL || n_rows * n_heads > 0x7fffffffLL * 4LL) return PA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int nr = (int)n_rows;
    if (head_dim == 64) {
        switch (G) {
            case 1: return launch_prefill<1, 64>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
            case 2: return launch_prefill<2, 64>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
            case 4: return launch_prefill<4, 64>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
            default: return launch_prefill<8, 64>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
        }
    }
    switch (G) {
        case 1: return launch_prefill<1, 128>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
        case 2: return launch_prefill<2, 128>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
        case 4: return launch_prefill<4, 128>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
        default: return launch_prefill<8, 128>(Pp, tk, tv, n_seqs, max_chunk_len, nr, st);
    }
}

}  // namespace

extern "C" size_t pa_prefill_workspace_bytes(int n_seqs, int n_heads, int n_kv_heads, int max_chunk_len,
                                             int splits) {
    if (n_seqs <= 0 || n_heads <= 0 || n_kv_heads <= 0 || max_chunk_len <= 0 || splits < 0 || splits > 64 ||
        n_heads % n_kv_heads != 0)
        return 0;
    const int G = n_heads / n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return 0;
    const long long n_items = (long long)pairs_per_seq(G, max_chunk_len) * n_kv_heads * n_seqs;
    if (splits > 0) return part_bytes(n_items, splits);
    const int n_cta = sm_count();
    return n_cta > 0 ? balanced_layout(n_items, n_cta).total : 0;
}

extern "C" int pa_prefill_paged_ex(void* out, const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_tables, const int32_t* context_lens,
                                   const int32_t* q_start_loc, float scale, int n_heads, int n_kv_heads,
                                   int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                                   int max_chunk_len, int num_blocks, int splits, void* workspace,
                                   size_t workspace_bytes, pa_stream_t stream) {
    return prefill_impl(out, q, k_pool, v_pool, block_tables, context_lens, q_start_loc, scale, n_heads,
                        n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq, max_chunk_len, num_blocks,
                        splits, workspace, workspace_bytes, stream);
}

extern "C" int pa_prefill_paged(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* q_start_loc, float scale, int n_heads, int n_kv_heads,
                                int head_dim, int block_size, int n_seqs, int max_blocks_per_seq,
                                int max_chunk_len, int num_blocks, pa_stream_t stream) {
    return prefill_impl(out, q, k_pool, v_pool, block_tables, context_lens, q_start_loc, scale, n_heads,
                        n_kv_heads, head_dim, block_size, n_seqs, max_blocks_per_seq, max_chunk_len, num_blocks,
                        1, nullptr, 0, stream);
}
