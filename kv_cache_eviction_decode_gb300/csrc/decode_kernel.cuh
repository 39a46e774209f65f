// decode_kernel.cuh -- the fused decode step over a budget-bounded KV cache.
//
// One persistent launch per layer-step. The grid is n_clusters thread-block
// clusters of `split` CTAs. Cluster c processes the units (sequence, KV head)
// c, c + n_clusters, ...; inside a cluster the CTAs divide each unit's
// occupied slots into contiguous ranges of 32-slot tiles.
//
// Memory pipeline: a ring of NST shared-memory stages, each filled by TMA
// copies of one 32-slot K or V tile that complete on the stage's mbarrier:
// one 1-D bulk copy (CUDA-core path), or two 2-D tensor-map boxes of 32 x 64
// bf16 with the 128-byte swizzle (tensor-core path; conflict-free ldmatrix).
// The CTA's tiles form one sequence over all of its units (unit 0's K tiles,
// its V tiles, unit 1's K tiles, ...). Thread 0 issues the first NST copies;
// after that, the warp that consumes tile s issues the copy of tile s + NST
// into the stage it has just freed, so the ring keeps streaming across unit
// boundaries: the next unit's first tiles land while the current unit's
// combine and score epilogue run. The next unit's slot positions (and H2O
// scores) are prefetched into a shared-memory area as soon as the current
// unit is done with it, and its q / k_new into registers.
//
// Per unit, every CTA:
//   K phase   logits z = q.k / sqrt(d) of the G query heads for each slot,
//             kept in shared memory (log2 units):
//               CUDA cores   every lane holds d/32 coordinates of q and of
//                            each key; a 31-shuffle butterfly transposes the
//                            partial sums so lane i ends with one logit;
//               tensor cores S^T = K Q^T with mma.sync m16n8k16 (bf16 in,
//                            fp32 accumulate): 16 slots are M, the G heads
//                            (padded to 8) are N, head_dim is K; K rows come
//                            in by ldmatrix, q is the B operand in registers.
//   V phase   with the CTA-local max m_c known, p = 2^(z - m_c) is written
//             back over z and o += p v is accumulated (tensor cores:
//             O^T = V^T P^T with 16 head_dim rows as M, V by ldmatrix.trans,
//             P as the B operand in registers; the warps' partial outputs
//             are summed in a tree in fragment order).
//   combine   (m_c, l_c, o_c) of every CTA in the cluster are read through
//             distributed shared memory; each CTA writes its share of
//             out = sum_c o_c 2^(m_c - m) / l. Rank 0 adds the new token.
//   scores    (H2O) every retained slot's cumulative score grows by
//             (1/G) sum_g p_g 2^(m_c - m) / l; the eligible slot with the
//             smallest (score, position) is the CTA's candidate, and a
//             second cluster exchange picks the victim.
//   insert    the new token's K/V, position and score are written in place
//             into the victim's slot (H2O), the closed-form ring slot
//             (StreamingLLM), the next empty slot, or the next entry of the
//             unit's free list (Random after a cut).
//
// Method (page title and section): attention over the retained cache, then
// the cumulative-score update, then eviction -- "KV Cache 驱逐策略：从 LRU 到
// H2O" flowchart and "Attention Sinks 与 KV Cache 淘汰策略" section 4.2 loop;
// greedy removal of the lowest-score candidate -- "h2o: heavy-hitter oracle"
// summary, Algorithm 1; sink + ring window -- same page section 4.1; the GQA
// score is the mean over the query heads of one KV head.
#pragma once

#include <cfloat>
#include <climits>
#include <cmath>

#include <cuda_fp16.h>

#include "device_common.cuh"

namespace kvevict {

constexpr int kTile = 32;  // slots per pipeline stage
constexpr int kMaxSplit = 16;

// Warps per CTA. 8 everywhere: 16 warps for the one-CTA-per-SM kernels
// (G >= 4) were measured slower -- the 128-register cap and the larger
// partial-output buffer cost more than the extra latency hiding gained.
template <int G, bool MMA> constexpr int warps_for() { return 8; }
constexpr int kSmemAlign = 1024;  // 128-byte swizzle atoms are 1 KB
constexpr int kMaxStages = 32;    // ring stages (the host fills the shared-memory budget)
constexpr int kMinStages = 4;

enum InsertMode : int {
    kInsertAt = 0,     // the host gives the slot (empty slot, or the ring slot)
    kH2OEvict = 1,     // cache full: evict the lowest-score eligible token
    kFromFreeList = 2, // Random after a cut: next entry of the unit's free list
    kH2OFill = 3,      // H2O with per-unit empty slots (after a SnapKV prefill): the unit's
                       // lowest empty slot if it has one, else evict as kH2OEvict
    kTwoPool = 4       // two-pool H2O: a recent pool and a heavy-hitter pool (per-slot pool flags)
};

// Opaque 128-byte tensor map (CUtensorMap), 64-byte aligned as a kernel
// parameter requires.
struct alignas(64) TensorMapBytes {
    uint64_t word[16];
};

struct DecodeParams {
    TensorMapBytes tmk, tmv;  // tensor maps of this layer's K and V (tensor-core path)
    const void *q;       // [B][Hkv*G][D]
    const void *k_new;   // [B][Hkv][D]
    const void *v_new;   // [B][Hkv][D]
    void *out;           // [B][Hkv*G][D]
    void *kc, *vc;       // this layer's cache, [B][Hkv][C][D]
    int32_t *pos;        // [B][Hkv][cstride]
    void *score;         // [B][Hkv][cstride] fp32 (fp16 with score_half), or null when the policy keeps no scores
    const int32_t *freelist;  // [B][Hkv][freelist_len]
    int32_t *trace;      // [B][Hkv][4] or null: slot, evicted position, evicted score, new score
    uint32_t *err;
    double *ledger;      // [B][Hkv] evicted score mass of this layer (policies with scores), or null
    int units;           // B * Hkv
    int C;
    int cstride;         // per-unit stride of pos/score (C rounded up to 4: 16-byte rows)
    int n_active;        // slots [0, n_active) may hold tokens
    int p;               // position of the new token
    int mode, dest_slot, freelist_idx, freelist_len;
    int n_sink, n_recent;
    int split;           // CTAs per cluster
    int tail_split;      // 1: a cluster's CTAs process whole units alone and split only the units left over
                         // (n_units mod split, processed first); 0: every unit is split over the cluster
    int zcap;            // per-head stride of the logit buffer (and aux slots)
    int nst;             // ring stages, kMinStages..kMaxStages
    int part_alias;      // the warps' partial outputs are written over the logits (after the score pass)
    int prefetch_early;  // the launch before this one did not touch this layer: cache tiles may be
                         // fetched before the programmatic-dependency wait (inputs still after it)
    float scale_log2;    // log2(e) / sqrt(D)
    float score_keep;    // each step s <- score_keep * s + a (1: the exact cumulative score)
    int score_half;      // scores stored as IEEE binary16 (cstride a multiple of 8)
    int score_int8;      // scores stored as 8-bit codes, one scale per unit (cstride a multiple of 16; split 1)
    float *qscale;       // score_int8: [B][Hkv] each unit's scale, its largest score / 255
    // two-pool H2O (kTwoPool)
    uint8_t *pool;       // [B][Hkv][pstride]: 0 recent pool, 1 heavy-hitter pool (slots holding a token)
    int pstride;         // per-unit stride of the pool flags (C rounded up to 16)
    int recent_full;     // every unit's recent pool holds n_recent tokens before this step
    float hh_threshold;  // a token leaving the recent pool is promoted iff its score is above this
};

// The standalone H2O selector (h2o_select_kernel).
struct SelectParams {
    const float *score;    // [units][C] fp32 scores supplied by the caller
    const int32_t *pos;    // this layer's slot positions [units][cstride]
    int32_t *victim;       // [units] the slot to evict, -1 if no slot is a candidate
    int C, cstride, n_active;
    int n_sink, n_recent;
    int p;                 // position of the token the next decode step appends
};

// Stored cumulative scores: fp32, or binary16 rounded to nearest even.
__device__ __forceinline__ float score_load(const DecodeParams &P, size_t i)
{
    return P.score_half ? __half2float(static_cast<const __half *>(P.score)[i]) : static_cast<const float *>(P.score)[i];
}
// Stores v and returns the value stored (v rounded when binary16).
__device__ __forceinline__ float score_store(const DecodeParams &P, size_t i, float v)
{
    if (P.score_half) {
        const __half h = __float2half_rn(v);
        static_cast<__half *>(P.score)[i] = h;
        return __half2float(h);
    }
    static_cast<float *>(P.score)[i] = v;
    return v;
}
__device__ __forceinline__ float score_round(const DecodeParams &P, float v)
{
    return P.score_half ? __half2float(__float2half_rn(v)) : v;
}

// Shared-memory layout, shared by host (size) and device (offsets). All
// offsets are from a base aligned up to kSmemAlign inside the allocation.
template <typename T, int D, int G, bool MMA> struct DecodeLayout {
    static constexpr int kWarps = warps_for<G, MMA>();
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kEPL = D / 32;  // key/value coordinates per lane (CUDA-core path)
    static constexpr int kR = 32 / G;    // slots per butterfly chunk (CUDA-core path)
    static constexpr int kStageBytes = kTile * D * static_cast<int>(sizeof(T));
    // warp partial outputs [warp][head][kPS]; the row stride D + 4 puts the
    // 32 lanes of one mma-fragment store on 32 different banks
    static constexpr int kPS = D + 4;
    static constexpr int kPartBytes = kWarps * G * kPS * 4;
    static_assert((2 * kThreads) % D == 0, "a thread owns the same coordinate pair of every head it sums");
    static_assert(G >= 1 && G <= 8 && (G & (G - 1)) == 0, "G in {1,2,4,8}");
    static_assert(!MMA || (sizeof(T) == 2 && D % 64 == 0), "tensor-core path: bf16, head_dim multiple of 64");

    struct Misc {
        uint64_t full[kMaxStages];
        uint64_t auxbar;
        uint32_t issued[kMaxStages];  // copies issued per stage
        uint32_t aux_issued;
        int abort;
        float wmax[kWarps][G];
        float wsum[kWarps][G];
        float m[G];        // this CTA's max logit per head (log2 units)
        float znew[G];     // the new token's logits (rank 0)
        float pnew[G];     // 2^(znew - m) (rank 0)
        float fac[kMaxSplit][G];  // 2^(m_c - m_global) / l_global per CTA c
        // cluster exchange, double-buffered by unit parity: (m, l) of every
        // CTA per head; from every CTA, its partial output over the
        // coordinates this CTA owns; every CTA's eviction candidate; rank
        // 0's new-token score
        float2 xml[2][kMaxSplit][G];
        alignas(16) float xo[2][G * D];
        uint64_t xkey[2][kMaxSplit];
        int32_t xslot[2][kMaxSplit];
        int32_t xempty[2][kMaxSplit];  // fill and two-pool modes: every CTA's lowest empty slot
        uint64_t xkey2[2][kMaxSplit];  // two-pool mode: every CTA's heavy-hitter candidate
        int32_t xslot2[2][kMaxSplit];
        float xanew[2];
        float anew;  // the new token's score (one CTA per unit)
        float wqmax[kWarps];  // INT8 scores: every warp's largest updated score
        uint64_t wkey[kWarps];
        int32_t wslot[kWarps];
        int32_t wempty[kWarps];
        uint64_t wkey2[kWarps];
        int32_t wslot2[kWarps];
    };

    // zcap = slots per CTA rounded to whole tiles, padded so that the head
    // rows of the logit buffer start on different banks: == R (mod 32) for
    // the butterfly's lane groups, == 8 (mod 32) for the mma path's float2
    // accesses by (head = lane / 4, slot pair = lane % 4).
    __host__ __device__ static int zcap(int max_slots_per_cta)
    {
        int z = ((max_slots_per_cta + kTile - 1) / kTile) * kTile;
        return MMA ? z + 8 : (G > 1 ? z + kR : z);
    }
    // Layout: [ring: nst stages][logits][warp partials][aux][misc]. With
    // `alias` the warp partials have no area of their own: they are written
    // over the logits once every read of those is done (alias_fits: they fit).
    __host__ __device__ static size_t off_z(int nst) { return static_cast<size_t>(nst) * kStageBytes; }
    __host__ __device__ static size_t off_part(int zc, int nst) { return off_z(nst) + ((static_cast<size_t>(G) * zc * 4 + 127) / 128) * 128; }
    __host__ __device__ static bool alias_fits(int zc) { return static_cast<size_t>(kPartBytes) <= static_cast<size_t>(G) * zc * 4; }
    // aux: the unit's slot positions, with scores (H2O) the cumulative scores,
    // and in two-pool mode the pool flags: n_arrays = 0 (none), 1, 2 or 3.
    __host__ __device__ static size_t off_aux(int zc, int nst, bool alias) { return off_part(zc, nst) + (alias ? 0 : kPartBytes); }
    __host__ __device__ static size_t aux_bytes(int zc) { return ((static_cast<size_t>(zc) * 4 + 15) / 16) * 16; }
    __host__ __device__ static size_t off_misc(int zc, int n_arrays, int nst, bool alias) { return off_aux(zc, nst, alias) + n_arrays * aux_bytes(zc); }
    __host__ __device__ static size_t bytes(int zc, int n_arrays, int nst, bool alias) { return off_misc(zc, n_arrays, nst, alias) + sizeof(Misc) + kSmemAlign; }
    // Shared memory besides the ring.
    __host__ __device__ static size_t fixed_bytes(int zc, int n_arrays, bool alias) { return bytes(zc, n_arrays, 0, alias); }
};

// Butterfly transpose-reduce: lane L holds 32 partial sums v[0..31]; after
// 31 shuffles lane L holds the full sum (over all lanes) of entry L.
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

template <int N> __device__ __forceinline__ float dot_n(const float (&a)[N], const float (&b)[N])
{
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) s = fmaf(a[i], b[i], s);
    return s;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Butterfly argmin over the warp of (key, slot); keys are distinct except the
// empty candidate (~0, -1), so every lane ends with the same pair.
__device__ __forceinline__ void warp_argmin(uint64_t &key, int32_t &slot)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const uint64_t ok = __shfl_xor_sync(0xffffffffu, key, off);
        const int32_t os = __shfl_xor_sync(0xffffffffu, slot, off);
        if (ok < key) {
            key = ok;
            slot = os;
        }
    }
}

__device__ __forceinline__ int32_t warp_min_s32(int32_t v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// ------------------------------------------------------------ H2O selector
// The pieces of the H2O eviction decision ("h2o: heavy-hitter oracle" summary,
// Algorithm 1: remove the token whose removal leaves the remaining set with
// the highest cumulative score -- with an additive score, the lowest-score
// token). The fused decode epilogue and the standalone selector kernel
// (h2o_select_kernel) decide with this same code.
//
// A retained token at position ps is a candidate at the step that appends
// position p iff it is neither a sink nor inside the recent window.
__device__ __forceinline__ bool h2o_candidate(int32_t ps, int n_sink, int p, int n_recent)
{
    return ps >= n_sink && ps <= p - n_recent;
}
// The eviction order: the lower score first, then the older position. Scores
// are >= 0, so their fp32 bit patterns order as the values do, and (score
// bits << 32 | position) orders as (score, position).
__device__ __forceinline__ uint64_t h2o_key(float score, int32_t ps)
{
    return (static_cast<uint64_t>(__float_as_uint(score)) << 32) | static_cast<uint32_t>(ps);
}
// Folds the token in `slot` (stored score `score`, position ps) into this
// thread's running minimum (best, bslot) if it is a candidate.
__device__ __forceinline__ void h2o_fold(uint64_t &best, int32_t &bslot, float score, int32_t ps, int slot,
                                         int n_sink, int p, int n_recent)
{
    if (h2o_candidate(ps, n_sink, p, n_recent)) {
        const uint64_t key = h2o_key(score, ps);
        if (key < best) {
            best = key;
            bslot = slot;
        }
    }
}
// The smallest of n <= 32 candidates (one per warp or per CTA) in shared
// memory, in every lane: (~0, -1) when none is a candidate.
__device__ __forceinline__ void argmin_of(const uint64_t *key, const int32_t *slot, int n, int lane, uint64_t &k,
                                          int32_t &sl)
{
    k = lane < n ? key[lane] : ~0ull;
    sl = lane < n ? slot[lane] : -1;
    warp_argmin(k, sl);
}

// Adds an evicted token's stored score to its unit's fp64 ledger. One thread
// per unit and step adds, and steps of a layer run in stream order, so the
// sum is deterministic; the reduction is issued without waiting for it
// (a plain load-add-store would hold the thread, and at the next barrier its
// CTA, for a global load's latency).
__device__ __forceinline__ void ledger_add(double *slot, float v)
{
    asm volatile("red.relaxed.gpu.global.add.f64 [%0], %1;" ::"l"(slot), "d"(static_cast<double>(v)) : "memory");
}

// A compile-time flag as a value (selects a specialisation of a generic lambda).
template <bool B> struct Flag {
    static constexpr bool value = B;
};

// Two consecutive elements, moved as one naturally aligned access.
template <typename T> struct alignas(2 * sizeof(T)) TPair {
    T x, y;
};

constexpr uint64_t kEmptyKey = 0x00000000FFFFFFFFull;  // no token leaves: position -1, score 0

// Two-pool H2O, the add step of the H2OCache class ("KV Cache 驱逐策略：从 LRU
// 到 H2O", section "实现要点"). The new token joins the recent pool; when that
// pool overflows, its lowest (score, position) member v leaves it -- the new
// token is a member -- and is promoted to the heavy-hitter pool iff its score
// is above hh_threshold, else it leaves the cache; an overfull heavy-hitter
// pool drops its lowest member, v included. Inputs: the recent pool's lowest
// key kv at slot sv, the heavy-hitter pool's lowest kw at slot sw (~0 when
// it is empty), the unit's lowest empty slot em (INT_MAX: none) and the new
// token's key kn. A key is (score bits << 32 | position); scores are >= 0.
struct PoolDecision {
    int dest;          // slot that receives the new token; -1: the new token leaves
    int new_pool;      // the pool it joins
    int promote;       // slot of a held token moved to the heavy-hitter pool; -1: none
    uint64_t evicted;  // key of the token that leaves the cache; kEmptyKey: none
};

__device__ __forceinline__ PoolDecision pool_decide(bool recent_full, float theta, uint64_t kv, int sv, uint64_t kw,
                                                    int sw, int em, uint64_t kn)
{
    PoolDecision d{-1, 0, -1, kEmptyKey};
    if (!recent_full) {  // room in the recent pool
        d.dest = em;
        return d;
    }
    const bool v_new = kn < kv;
    const uint64_t k = v_new ? kn : kv;
    if (!(__uint_as_float(static_cast<uint32_t>(k >> 32)) > theta) || (em == INT_MAX && k < kw)) {
        d.evicted = k;  // v leaves the cache: below the threshold, or the lowest of a full pool
        d.dest = v_new ? -1 : sv;
        return d;
    }
    if (em != INT_MAX) {
        d.dest = em;  // room in the heavy-hitter pool
    } else {
        d.dest = sw;  // the heavy-hitter pool's lowest leaves
        d.evicted = kw;
    }
    if (v_new) d.new_pool = 1;
    else d.promote = sv;
    return d;
}

// The CTA's share of one launch. Cluster c (of n_clusters, S CTAs each)
// owns the units c, c + n_clusters, ... (n_units of them). The CTA works
// through a sequence of items:
//   - first n_split "split" items, units k = 0 .. n_split - 1 of the
//     cluster, each divided over the cluster's S CTAs (this CTA: the slots
//     [s_lo, s_hi), nt tiles) and combined through distributed shared memory;
//   - then its "whole" units, k = n_split + j S + rank, each processed by
//     this CTA alone (slots [0, n_all), ntw tiles).
// Without tail splitting every unit is a split item (n_split = n_units; at
// S = 1 a split item is the whole unit). With it (tail = 1), a cluster
// splits only the n_units mod S units left over once every CTA has an equal
// number of whole units: the grid's load then differs by less than one unit
// between CTAs, and only those few units pay for the cluster exchange.
struct Work {
    int cluster_id, n_clusters, n_units;  // units this cluster processes
    int S, rank;                          // cluster size, this CTA's rank
    int n_split, n_items;                 // split items (first), all items of this CTA
    int nt, s_lo, s_hi, n_mine;           // a split item: this CTA's tiles / slot range
    int ntw, n_all;                       // a whole unit: its tiles / slots
    int total_seq;                        // K and V tiles over all items
};

// Item i of the CTA: its unit.
__device__ __forceinline__ size_t item_unit(const Work &W, int i)
{
    const int k = i < W.n_split ? i : W.n_split + (i - W.n_split) * W.S + W.rank;
    return static_cast<size_t>(W.cluster_id) + static_cast<size_t>(k) * W.n_clusters;
}

// Tile s of the CTA's sequence: unit, K or V, which 32 slots.
struct TileAt {
    size_t unit;
    bool is_k;
    int slot0, rows;
};

template <bool FLEX> __device__ __forceinline__ TileAt tile_at(const Work &W, int s)
{
    const int split_seq = W.n_split * 2 * W.nt;
    TileAt t;
    if (!FLEX || s < split_seq) {
        const int two_nt = 2 * W.nt;
        const int i = s / two_nt, loc = s - i * two_nt;
        t.unit = item_unit(W, i);
        t.is_k = loc < W.nt;
        t.slot0 = W.s_lo + (t.is_k ? loc : loc - W.nt) * kTile;
        t.rows = min(kTile, W.s_hi - t.slot0);
    } else {
        const int two_nt = 2 * W.ntw;
        const int j = (s - split_seq) / two_nt, loc = (s - split_seq) - j * two_nt;
        t.unit = item_unit(W, W.n_split + j);
        t.is_k = loc < W.ntw;
        t.slot0 = (t.is_k ? loc : loc - W.ntw) * kTile;
        t.rows = min(kTile, W.n_all - t.slot0);
    }
    return t;
}

// CUDA-core path: one contiguous bulk copy per tile (only the valid rows).
template <typename T, int D, bool FLEX> struct BulkTileSource {
    const T *kc, *vc;
    size_t C;
    __device__ __forceinline__ void issue(const Work &W, int s, T *stage, uint64_t *bar) const
    {
        const TileAt t = tile_at<FLEX>(W, s);
        const uint32_t bytes = static_cast<uint32_t>(t.rows * D * sizeof(T));
        const T *src = (t.is_k ? kc : vc) + (t.unit * C + t.slot0) * D;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_stream(stage, src, bytes, bar, l2_policy_evict_first());
    }
};

// Tensor-core path: D/64 tensor-map boxes of 32 rows x 64 bf16 per tile,
// 128-byte swizzled. A box always moves 32 full rows (rows past the unit's
// range belong to the next unit or are zero-filled past the tensor's end).
template <int D, bool FLEX> struct TmaTileSource {
    const void *tmk, *tmv;
    size_t C;
    __device__ __forceinline__ void issue(const Work &W, int s, __nv_bfloat16 *stage, uint64_t *bar) const
    {
        const TileAt t = tile_at<FLEX>(W, s);
        const int row = static_cast<int>(t.unit * C + t.slot0);
        const void *tm = t.is_k ? tmk : tmv;
        const uint64_t pol = l2_policy_evict_first();
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kTile * D * 2));
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
            tma_load_2d(reinterpret_cast<uint8_t *>(stage) + b * kTile * 128, tm, b * 64, row, bar, pol);
    }
};

// Two CTAs per SM (registers <= 128) for G <= 2; for larger G shared memory
// holds one CTA and the registers are left free.
template <int G, bool MMA> __host__ __device__ constexpr int min_blocks() { return G <= 2 ? 2 : 1; }
// Tail splitting and partials over the logits are built into the kernels
// that run one CTA per SM only: the two-CTA kernels (G <= 2) gain nothing from
// them (measured) and run at the 128-register limit, where the extra state
// cost them about 2% per launch.
template <int G, bool MMA> __host__ __device__ constexpr bool flex_layout() { return min_blocks<G, MMA>() == 1; }

template <typename T, int D, int G, bool HOLES, bool MMA>
__global__ void __launch_bounds__((warps_for<G, MMA>() * 32), (min_blocks<G, MMA>()))
    decode_step_kernel(const __grid_constant__ DecodeParams P)
{
    using L = DecodeLayout<T, D, G, MMA>;
    constexpr int kWarps = L::kWarps, kThreads = L::kThreads;
    constexpr int EPL = L::kEPL, R = L::kR, kPS = L::kPS;
    const int NST = P.nst;
    constexpr int KSTEPS = D / 16;  // mma k-steps over head_dim
    using E = Elem<T>;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + kSmemAlign - 1) &
                                                ~static_cast<uintptr_t>(kSmemAlign - 1));
    T *ring = reinterpret_cast<T *>(smem);
    const int zc = P.zcap;
    float *zbuf = reinterpret_cast<float *>(smem + L::off_z(NST));
    constexpr bool kFlex = flex_layout<G, MMA>();
    const bool alias = kFlex && P.part_alias != 0;
    float *part = alias ? zbuf : reinterpret_cast<float *>(smem + L::off_part(zc, NST));
    uint8_t *aux = smem + L::off_aux(zc, NST, alias);
    const size_t auxb = L::aux_bytes(zc);
    // slot positions (and H2O scores, pool flags) are prefetched per unit only when used
    const bool need_aux = P.score != nullptr || HOLES;
    const bool pools = P.mode == kTwoPool;
    const int n_aux = pools ? 3 : (P.score != nullptr ? 2 : (HOLES ? 1 : 0));
    auto &M = *reinterpret_cast<typename L::Misc *>(smem + L::off_misc(zc, n_aux, NST, alias));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_rank());
    const int S = P.split;
    // INT8 scores need the unit's largest score before any code is written:
    // one CTA per unit only (the host refuses a split); a cluster leaves at once
    if (S > 1 && P.score_int8) {
        if (tid == 0 && blockIdx.x == 0) atomicOr(P.err, KVEVICT_DEV_BAD_SLOT);
        return;
    }
    const size_t C = static_cast<size_t>(P.C);
    const size_t CS = static_cast<size_t>(P.cstride);
    const bool has_score = P.score != nullptr;

    Work W;
    W.cluster_id = blockIdx.x / S;
    W.n_clusters = gridDim.x / S;
    W.n_units = W.cluster_id < P.units ? (P.units - W.cluster_id + W.n_clusters - 1) / W.n_clusters : 0;
    W.S = S;
    W.rank = rank;
    {
        const int nt_all = (P.n_active + kTile - 1) / kTile;
        const int t_lo = static_cast<int>(static_cast<long long>(rank) * nt_all / S);
        const int t_hi = static_cast<int>(static_cast<long long>(rank + 1) * nt_all / S);
        W.nt = t_hi - t_lo;
        W.s_lo = t_lo * kTile;
        W.s_hi = min(t_hi * kTile, P.n_active);
        W.n_mine = max(0, W.s_hi - W.s_lo);
        W.ntw = nt_all;
        W.n_all = P.n_active;
        W.n_split = (kFlex && P.tail_split) ? W.n_units % S : W.n_units;
        W.n_items = W.n_split + (W.n_units - W.n_split) / S;
        W.total_seq = W.n_split * 2 * W.nt + (W.n_items - W.n_split) * 2 * W.ntw;
    }
    // item i's slots: [lo, lo + n) and the index of its aux copy among the
    // items that copy any (a CTA with no slots of a split item copies none)
    auto item_slots = [&](int i, int &lo, int &n) {
        lo = i < W.n_split ? W.s_lo : 0;
        n = i < W.n_split ? W.n_mine : W.n_all;
    };
    auto aux_index = [&](int i) {
        return i < W.n_split ? (W.n_mine > 0 ? i : 0) : (W.n_mine > 0 ? W.n_split : 0) + (i - W.n_split);
    };
    BulkTileSource<T, D, kFlex> bulk_src{static_cast<const T *>(P.kc), static_cast<const T *>(P.vc), C};
    TmaTileSource<D, kFlex> tma_src{&P.tmk, &P.tmv, C};
    auto issue_tile = [&](int s, int st) {
        T *stage = ring + static_cast<size_t>(st) * kTile * D;
        if constexpr (MMA)
            tma_src.issue(W, s, reinterpret_cast<__nv_bfloat16 *>(stage), &M.full[st]);
        else
            bulk_src.issue(W, s, stage, &M.full[st]);
    };


    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&M.full[i], 1);
            M.issued[i] = 0;
        }
        mbar_init(&M.auxbar, 1);
        M.aux_issued = 0;
        M.abort = 0;
        mbar_fence_init();
        if constexpr (MMA) {
            prefetch_tensormap(&P.tmk);
            prefetch_tensormap(&P.tmv);
        }
    }
    __syncthreads();

    // Bulk copy of the i-th unit's slot positions (and scores) into the aux
    // area; it completes phase i of the aux mbarrier.
    auto issue_aux = [&](int i) {
        const size_t unit = item_unit(W, i);
        int lo, n;
        item_slots(i, lo, n);
        if (n <= 0) return;
        const uint32_t bytes = static_cast<uint32_t>(((n * 4 + 15) / 16) * 16);
        const uint32_t sbytes = P.score_int8   ? static_cast<uint32_t>(((n + 15) / 16) * 16)
                                : P.score_half ? static_cast<uint32_t>(((n * 2 + 15) / 16) * 16)
                                               : bytes;
        const uint32_t pbytes = pools ? static_cast<uint32_t>(((n + 15) / 16) * 16) : 0u;
        const uint32_t tx = (has_score ? bytes + sbytes : bytes) + pbytes;
        mbar_arrive_expect_tx(&M.auxbar, tx);
        bulk_g2s(aux, P.pos + unit * CS + lo, bytes, &M.auxbar);
        if (has_score)
            bulk_g2s(aux + auxb,
                     static_cast<const uint8_t *>(P.score) +
                         (unit * CS + lo) * (P.score_int8 ? 1 : (P.score_half ? 2 : 4)),
                     sbytes,
                     &M.auxbar);
        if (pools)
            bulk_g2s(aux + 2 * auxb, P.pool + unit * static_cast<size_t>(P.pstride) + lo, pbytes, &M.auxbar);
        M.aux_issued++;
    };

    auto issue_first = [&]() {
        for (int s = 0; s < min(NST, W.total_seq); ++s) issue_tile(s, s);
        if (need_aux && W.n_items > 0) issue_aux(0);
        for (int s = 0; s < min(NST, W.total_seq); ++s) st_release_cta(&M.issued[s], 1u);
    };
    // This layer's cache (and positions/scores) can only be written by a
    // launch for this layer. When the launch before this one was for another
    // layer, the first tiles are fetched while that launch is still running;
    // the inputs q/k/v (which a preceding kernel may produce) are read only
    // after the programmatic-dependency wait.
    if (P.prefetch_early && tid == 0) issue_first();
    grid_dependency_wait();
    grid_launch_dependents();
    if (!P.prefetch_early && tid == 0) issue_first();

    bool ok = true;  // false after a timed-out wait: skip work, keep barriers
    volatile int *abort_flag = &M.abort;
    // Tile s is copy number c = s / NST into stage s % NST. Its consumer
    // first waits until that copy has been issued (by the consumer of tile
    // s - NST, usually another warp): the stage's mbarrier is then in phase c
    // or c + 1 -- never behind -- so the parity wait below tests phase c. The
    // copy after it (tile s + NST) is only issued once tile s is consumed.
    auto wait_stage = [&](int s) -> bool {
        if (!ok || *abort_flag) {
            ok = false;
            return false;
        }
        const int st = s % NST;
        const uint32_t need = static_cast<uint32_t>(s / NST) + 1;
        if (ld_acquire_cta(&M.issued[st]) < need) {
            const uint64_t t0 = global_timer_ns();
            for (uint32_t it = 1; ld_acquire_cta(&M.issued[st]) < need; ++it) {
                if ((it & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || *abort_flag)) {
                    atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
                    ok = false;
                    *abort_flag = 1;
                    return false;
                }
            }
        }
        if (!mbar_wait(&M.full[st], (s / NST) & 1)) {
            atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
            ok = false;
            *abort_flag = 1;
            return false;
        }
        return true;
    };
    auto release_stage = [&](int s) {
        __syncwarp();
        const int nx = s + NST;
        if (lane == 0 && nx < W.total_seq && ok) {
            const int st = s % NST;
            issue_tile(nx, st);
            st_release_cta(&M.issued[st], M.issued[st] + 1);  // after the arrive.expect_tx
        }
    };

    // Per-lane view of the logits: the CUDA-core butterfly gives lane L the
    // head L / R; the mma fragments give lane L the head L / 4 (valid if < G).
    const int g_lane = MMA ? (lane >> 2) : (lane / R);
    const int t4 = lane & 3;
    const bool lane_has_head = g_lane < G;
    constexpr int kHeadLanes = MMA ? 4 : R;  // lanes sharing one head's partials

    // Register prefetch of a unit's q (CUDA-core path: d-slices; mma path: A
    // fragments) and, for warp 0, the new token's key in the same layout
    // (used where this CTA is the unit's rank 0).
    constexpr int QG = MMA ? 1 : G, QE = MMA ? 1 : EPL, QK = MMA ? KSTEPS : 1;
    float qn[QG][QE];
    uint32_t qan[QK][2];
    float kn_next[QE];
    uint32_t kan[QK][2];
    // Every thread: the new token's k and v at the coordinate pair (dp, dp + 1)
    // -- rank 0 adds p_new v_new there, and the threads tid < D/2 of the CTA
    // that stores the new token write them -- and the slot the new token goes
    // to when the host or the free list names it.
    const int dp = 2 * (tid % (D / 2));
    TPair<T> kpair_next, vpair_next;
    int dest_next = -1;
    auto load_unit_inputs = [&](size_t u) {
        const T *qp = static_cast<const T *>(P.q) + u * G * D;
        if constexpr (MMA) {
            const T *kp = static_cast<const T *>(P.k_new) + u * D + 2 * t4;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                if (lane_has_head) {
                    const T *row = qp + g_lane * D + 16 * kk + 2 * t4;
                    qan[kk][0] = *reinterpret_cast<const uint32_t *>(row);
                    qan[kk][1] = *reinterpret_cast<const uint32_t *>(row + 8);
                } else {
                    qan[kk][0] = qan[kk][1] = 0u;
                }
                if (warp == 0) {
                    kan[kk][0] = *reinterpret_cast<const uint32_t *>(kp + 16 * kk);
                    kan[kk][1] = *reinterpret_cast<const uint32_t *>(kp + 16 * kk + 8);
                }
            }
        } else {
#pragma unroll
            for (int g = 0; g < G; ++g) load_f32<T, EPL>(qp + g * D + lane * EPL, qn[g]);
            if (warp == 0) load_f32<T, EPL>(static_cast<const T *>(P.k_new) + u * D + lane * EPL, kn_next);
        }
        kpair_next = *reinterpret_cast<const TPair<T> *>(static_cast<const T *>(P.k_new) + u * D + dp);
        vpair_next = *reinterpret_cast<const TPair<T> *>(static_cast<const T *>(P.v_new) + u * D + dp);
        dest_next = P.mode == kFromFreeList ? P.freelist[u * P.freelist_len + P.freelist_idx] : P.dest_slot;
    };
    if (W.n_items > 0) load_unit_inputs(item_unit(W, 0));

    for (int i = 0; i < W.n_items; ++i) {
        const size_t unit = item_unit(W, i);
        // this item: split over the cluster (Si CTAs, this one rank ri) or
        // this CTA's whole unit (Si = 1, ri = 0); its slots, tiles and first
        // tile in the CTA's sequence
        const bool split_item = !kFlex || i < W.n_split;
        const int Si = split_item ? S : 1, ri = split_item ? rank : 0;
        const int s_lo = split_item ? W.s_lo : 0, s_hi = split_item ? W.s_hi : W.n_all;
        const int n_mine = split_item ? W.n_mine : W.n_all;
        const int nt = split_item ? W.nt : W.ntw;
        const int seq0 = split_item ? i * 2 * W.nt : W.n_split * 2 * W.nt + (i - W.n_split) * 2 * W.ntw;
        const int32_t *apos = reinterpret_cast<const int32_t *>(aux);
        const float *ascore = reinterpret_cast<const float *>(aux + auxb);
        const __half *ascore_h = reinterpret_cast<const __half *>(aux + auxb);
        const uint8_t *ascore8 = aux + auxb;
        const uint8_t *apool = aux + 2 * auxb;
        // INT8 scores: this unit's scale before this step (0 before its first step)
        const float qscale_u = P.score_int8 ? P.qscale[unit] : 0.f;
        // this unit's stored score of local slot j, before this step
        auto stored_score = [&](int j) {
            return P.score_int8   ? static_cast<float>(ascore8[j]) * qscale_u
                   : P.score_half ? __half2float(ascore_h[j])
                                  : ascore[j];
        };

        // This unit's q (prefetched during the previous unit); start the
        // next unit's loads.
        float qf[QG][QE], kf_new[QE];
        uint32_t qa[QK][2], ka[QK][2];
        const TPair<T> kpair = kpair_next, vpair = vpair_next;
        const int dest_mine = dest_next;
        if constexpr (MMA) {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                qa[kk][0] = qan[kk][0];
                qa[kk][1] = qan[kk][1];
                ka[kk][0] = kan[kk][0];
                ka[kk][1] = kan[kk][1];
            }
        } else {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < EPL; ++e) qf[g][e] = qn[g][e];
#pragma unroll
            for (int e = 0; e < EPL; ++e) kf_new[e] = kn_next[e];
        }
        if (i + 1 < W.n_items) load_unit_inputs(item_unit(W, i + 1));
        // the new token's logits (rank 0, warp 0)
        if (ri == 0 && warp == 0) {
            if constexpr (MMA) {
                // lane (g, t) holds q[g][16kk + 2t + {0,1,8,9}] and the same
                // coordinates of k_new: partial dot, then sum over t.
                float s = 0.f;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float q0, q1, k0, k1;
                        bf16x2_to_f32(qa[kk][h], q0, q1);
                        bf16x2_to_f32(ka[kk][h], k0, k1);
                        s = fmaf(q0, k0, fmaf(q1, k1, s));
                    }
                s += __shfl_xor_sync(0xffffffffu, s, 1);
                s += __shfl_xor_sync(0xffffffffu, s, 2);
                if (t4 == 0 && lane_has_head) M.znew[g_lane] = s * P.scale_log2;
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float s = warp_sum(dot_n(qf[g], kf_new));
                    if (lane == 0) M.znew[g] = s * P.scale_log2;
                }
            }
        }
        // positions (and scores) of this unit's slots; every unit that
        // prefetched them waits for them exactly once
        bool aux_ready = false;
        auto wait_aux = [&]() {
            if (aux_ready || n_mine == 0 || !need_aux) return;
            aux_ready = true;
            if (!ok || *abort_flag) {
                ok = false;
                return;
            }
            if (!mbar_wait(&M.auxbar, aux_index(i) & 1)) {
                atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
                ok = false;
                *abort_flag = 1;
            }
        };
        if (HOLES) wait_aux();

        // ---------------------------------------------------------- K phase
        float mx = -INFINITY;   // max of this lane's head (mma path: head 2t)
        float mx1 = -INFINITY;  // mma path: head 2t + 1
        for (int s_loc = warp; s_loc < nt; s_loc += kWarps) {
            const int s = seq0 + s_loc;
            if (!wait_stage(s)) break;
            const T *tk = ring + static_cast<size_t>(s % NST) * kTile * D;
            const int base = s_loc * kTile;
            const int rows = min(kTile, n_mine - base);
            if constexpr (MMA) {
                // S^T (32 slots x 8 heads) = K (32 x D) Q^T, two 16-slot
                // m-tiles; fragment c = (slot g, heads 2t, 2t+1), (slot g+8, ...)
                const uint32_t sb = smem_u32(tk);
                const int mi = lane >> 3, ri = lane & 7;
                // four independent accumulation chains: (m-tile, k-step parity)
                float cc[2][2][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int par = 0; par < 2; ++par) cc[mt][par][0] = cc[mt][par][1] = cc[mt][par][2] = cc[mt][par][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        uint32_t a[4];
                        ldsm_x4(sb + swz128_offset(mt * 16 + (mi & 1) * 8 + ri, 2 * kk + (mi >> 1)), a[0], a[1], a[2],
                                a[3]);
                        mma_bf16_16816(cc[mt][kk & 1], a, qa[kk][0], qa[kk][1]);
                    }
                // fragment: (slot r0 = mt*16 + g | r0 + 8, heads 2t, 2t+1).
                // Branch-free: slot validity once per row (the aux buffer covers
                // the whole tile, rows past `rows` are masked), head validity
                // is a per-lane constant.
                const bool h0_ok = 2 * t4 < G, h1_ok = 2 * t4 + 1 < G;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int r0 = mt * 16 + g_lane, r1 = r0 + 8;
                    bool v0 = r0 < rows, v1 = r1 < rows;
                    if (HOLES) {
                        v0 = v0 && apos[base + r0] >= 0;
                        v1 = v1 && apos[base + r1] >= 0;
                    }
                    const float z00 = v0 ? (cc[mt][0][0] + cc[mt][1][0]) * P.scale_log2 : -INFINITY;
                    const float z01 = v0 ? (cc[mt][0][1] + cc[mt][1][1]) * P.scale_log2 : -INFINITY;
                    const float z10 = v1 ? (cc[mt][0][2] + cc[mt][1][2]) * P.scale_log2 : -INFINITY;
                    const float z11 = v1 ? (cc[mt][0][3] + cc[mt][1][3]) * P.scale_log2 : -INFINITY;
                    if (h0_ok) {
                        zbuf[(2 * t4) * zc + base + r0] = z00;
                        zbuf[(2 * t4) * zc + base + r1] = z10;
                        mx = fmaxf(mx, fmaxf(z00, z10));
                    }
                    if (h1_ok) {
                        zbuf[(2 * t4 + 1) * zc + base + r0] = z01;
                        zbuf[(2 * t4 + 1) * zc + base + r1] = z11;
                        mx1 = fmaxf(mx1, fmaxf(z01, z11));
                    }
                }
            } else {
#pragma unroll
                for (int c = 0; c < G; ++c) {
                    float vals[32];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float kf[EPL];
                        load_f32<T, EPL>(tk + (c * R + r) * D + lane * EPL, kf);
#pragma unroll
                        for (int g = 0; g < G; ++g) vals[g * R + r] = dot_n(qf[g], kf);
                    }
                    const float sum = transpose_reduce32(vals, lane);
                    const int row = c * R + (lane % R);
                    bool valid = row < rows;
                    if (HOLES && valid) valid = apos[base + row] >= 0;
                    const float z = valid ? sum * P.scale_log2 : -INFINITY;
                    zbuf[g_lane * zc + base + row] = z;
                    mx = fmaxf(mx, z);
                }
            }
            release_stage(s);
        }
        // per-warp max per head
        if constexpr (MMA) {
            // lanes with the same t hold heads 2t, 2t+1 for different slots
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            if (g_lane == 0) {
                if (2 * t4 < G) M.wmax[warp][2 * t4] = mx;
                if (2 * t4 + 1 < G) M.wmax[warp][2 * t4 + 1] = mx1;
            }
        } else {
            // the lanes of one head form an aligned group
#pragma unroll
            for (int off = 1; off < kHeadLanes; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane % kHeadLanes == 0 && lane_has_head) M.wmax[warp][g_lane] = mx;
        }
        __syncthreads();
        if (warp == 0 && lane < G) {
            float m = -INFINITY;
            for (int w = 0; w < kWarps; ++w) m = fmaxf(m, M.wmax[w][lane]);
            if (ri == 0) m = fmaxf(m, M.znew[lane]);
            M.m[lane] = m;
        }
        __syncthreads();
        const float m_mine = lane_has_head ? M.m[g_lane] : 0.f;

        // ---------------------------------------------------------- V phase
        float lsum = 0.f;
        float acc[MMA ? 1 : G][MMA ? 1 : EPL];  // CUDA-core accumulators
        float oacc[MMA ? D / 16 : 1][4];        // mma accumulators: O^T (16 head_dim rows x 8 heads) per m-tile
        if constexpr (MMA) {
#pragma unroll
            for (int md = 0; md < D / 16; ++md) oacc[md][0] = oacc[md][1] = oacc[md][2] = oacc[md][3] = 0.f;
        } else {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
        }
        const int first_v = nt + ((warp - nt % kWarps) % kWarps + kWarps) % kWarps;
        for (int s_loc = first_v; s_loc < 2 * nt; s_loc += kWarps) {
            const int s = seq0 + s_loc;
            if (!wait_stage(s)) break;
            const int base = (s_loc - nt) * kTile;
            const int rows = min(kTile, n_mine - base);
            const T *tv = ring + static_cast<size_t>(s % NST) * kTile * D;
            if constexpr (MMA) {
                const uint32_t sb = smem_u32(tv);
                const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    // B = P^T fragment: (slots 2t, 2t+1 | 2t+8, 2t+9 of this
                    // 16-slot step, head g); this lane computes those p.
                    uint32_t pa[4] = {0u, 0u, 0u, 0u};
                    if (lane_has_head) {
                        float pr[4];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            float2 *zp = reinterpret_cast<float2 *>(zbuf + g_lane * zc + base + ks * 16 + hh * 8 + 2 * t4);
                            const float2 z = *zp;
                            const float p0 = (z.x == -INFINITY) ? 0.f : exp2f(z.x - m_mine);
                            const float p1 = (z.y == -INFINITY) ? 0.f : exp2f(z.y - m_mine);
                            *zp = make_float2(p0, p1);
                            lsum += p0 + p1;
                            pr[2 * hh] = p0;
                            pr[2 * hh + 1] = p1;
                        }
                        pa[0] = pack_bf16x2(pr[0], pr[1]);
                        pa[2] = pack_bf16x2(pr[2], pr[3]);
                    }
#pragma unroll
                    for (int md = 0; md < D / 16; ++md) {
                        // A = V^T (16 head_dim rows x 16 slots) from the [slot][d] tile
                        uint32_t a[4];
                        ldsm_x4_trans(sb + swz128_offset(ks * 16 + (mi >> 1) * 8 + ri, 2 * md + (mi & 1)), a[0], a[1],
                                      a[2], a[3]);
                        mma_bf16_16816(oacc[md], a, pa[0], pa[2]);
                    }
                }
            } else {
                // probabilities of this tile: lane L owns (head L/R, slots L%R + c*R)
#pragma unroll
                for (int c = 0; c < G; ++c) {
                    float *zp = zbuf + g_lane * zc + base + c * R + (lane % R);
                    const float z = *zp;
                    const float pr = (z == -INFINITY) ? 0.f : exp2f(z - m_mine);
                    *zp = pr;
                    lsum += pr;
                }
                __syncwarp();
                int r = 0;
                if (!HOLES) {
                    for (; r + 4 <= rows; r += 4) {
                        float4 p4[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) p4[g] = *reinterpret_cast<const float4 *>(zbuf + g * zc + base + r);
#pragma unroll
                        for (int rr = 0; rr < 4; ++rr) {
                            float vf[EPL];
                            load_f32<T, EPL>(tv + (r + rr) * D + lane * EPL, vf);
#pragma unroll
                            for (int g = 0; g < G; ++g) {
                                const float pv = rr == 0 ? p4[g].x : rr == 1 ? p4[g].y : rr == 2 ? p4[g].z : p4[g].w;
#pragma unroll
                                for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pv, vf[e], acc[g][e]);
                            }
                        }
                    }
                }
                for (; r < rows; ++r) {
                    float pr[G];
                    bool any = false;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        pr[g] = zbuf[g * zc + base + r];
                        any |= pr[g] != 0.f;
                    }
                    if (HOLES && !any) continue;  // an empty slot (same for every lane)
                    float vf[EPL];
                    load_f32<T, EPL>(tv + r * D + lane * EPL, vf);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pr[g], vf[e], acc[g][e]);
                }
            }
            release_stage(s);
        }
#pragma unroll
        for (int off = 1; off < kHeadLanes; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        if (lane % kHeadLanes == 0 && lane_has_head) M.wsum[warp][g_lane] = lsum;
        // rank 0 adds the new token: p_new = 2^(z_new - m)
        if (ri == 0 && tid < G) M.pnew[tid] = exp2f(M.znew[tid] - M.m[tid]);
        // every warp's partial output, compact: part[warp][head][kPS]; with
        // `alias` over the logits, once the score pass has read them
        auto write_partials = [&]() {
            if constexpr (MMA) {
                // O^T fragment: (d = 16 md + g | + 8, heads 2t, 2t + 1)
#pragma unroll
                for (int md = 0; md < D / 16; ++md)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = 2 * t4 + (e & 1), d = md * 16 + g_lane + (e >> 1) * 8;
                        if (h < G) part[(warp * G + h) * kPS + d] = oacc[md][e];
                    }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < EPL; ++e) part[(warp * G + g) * kPS + lane * EPL + e] = acc[g][e];
            }
        };
        if (!alias) write_partials();
        __syncthreads();  // (A) sums, p_new (and unaliased partials) visible; every read of this unit's tiles is done

        // This CTA's totals of head g: l_g = sum over the warps (+ p_new on
        // rank 0), o_g[d] likewise (+ p_new v_new[d] on rank 0). A thread
        // owns the coordinate pairs (g, dp), (g, dp + 1) of its pair indices
        // jp = tid, tid + kThreads, ... (g = 2 jp / D).
        auto cta_l = [&](int g) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) l += M.wsum[w][g];
            if (ri == 0) l += M.pnew[g];
            return l;
        };
        auto cta_o = [&](int g, float &ox, float &oy) {
            ox = 0.f;
            oy = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float2 v = *reinterpret_cast<const float2 *>(part + (w * G + g) * kPS + dp);
                ox += v.x;
                oy += v.y;
            }
            if (ri == 0) {
                ox = fmaf(M.pnew[g], E::to_f32(vpair.x), ox);
                oy = fmaf(M.pnew[g], E::to_f32(vpair.y), oy);
            }
        };
        constexpr int kPairs = G * D / 2;
        const bool fill = P.mode == kH2OFill;
        // a victim is chosen (fill: unless a slot is empty; two-pool: per the pools)
        const bool evict = P.mode == kH2OEvict || fill || pools;
        int dest = -1;             // slot that receives the new token
        bool writer = false;       // this CTA writes it
        uint64_t win_key = ~0ull;  // H2O eviction: (score bits, position) of the evicted token
        float anew = 0.f;          // the new token's score (rank 0)
        uint8_t anew_code = 0;     // INT8 scores: its code
        PoolDecision pd{-1, 0, -1, kEmptyKey};  // two-pool mode
        // The score pass over this CTA's slots [s_lo, s_lo + n_mine): every retained
        // score s <- keep * s + a (a: this step's probability, mean over the G heads,
        // from the logits and the factors fself), and, evicting, the lowest
        // (score, position) candidate (two-pool: one per pool) and the lowest empty
        // slot. GEN = false is the plain H2O eviction with fp32 scores (no binary16,
        // fill or pool branches in the loop); GEN = true handles every mode.
        // INT8 (one CTA per unit): this pass only updates, keeping the value in
        // the slot's head-0 logit cell (read by this thread alone) and the
        // largest retained one in qmax; the codes and candidates follow once
        // the unit's largest score is known.
        const bool general_scores = P.score_half || P.score_int8 || fill || pools;
        auto score_pass = [&](auto gen, const float(&fself)[G], uint64_t &best, int32_t &bslot, uint64_t &best2,
                              int32_t &bslot2, int32_t &emin, float &qmax) {
            constexpr bool GEN = decltype(gen)::value;
            if constexpr (!GEN) {
                // plain H2O, fp32 scores: four consecutive slots per thread, with
                // 16-byte accesses to the logits, the scores (shared and global) and
                // the positions (every row and offset here is a multiple of 4 floats);
                // the same fmaf order per slot as the general loop
                float *sp = static_cast<float *>(P.score) + unit * CS + s_lo;
                for (int j0 = 4 * tid; j0 < n_mine; j0 += 4 * kThreads) {
                    float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float4 z = *reinterpret_cast<const float4 *>(zbuf + g * zc + j0);
                        a4.x = fmaf(z.x, fself[g], a4.x);
                        a4.y = fmaf(z.y, fself[g], a4.y);
                        a4.z = fmaf(z.z, fself[g], a4.z);
                        a4.w = fmaf(z.w, fself[g], a4.w);
                    }
                    const float4 s4 = *reinterpret_cast<const float4 *>(ascore + j0);
                    const float4 n4 = make_float4(fmaf(P.score_keep, s4.x, a4.x), fmaf(P.score_keep, s4.y, a4.y),
                                                  fmaf(P.score_keep, s4.z, a4.z), fmaf(P.score_keep, s4.w, a4.w));
                    const int left = n_mine - j0;  // valid slots in this group of four
                    if (left >= 4) {
                        *reinterpret_cast<float4 *>(sp + j0) = n4;
                    } else {
                        sp[j0] = n4.x;
                        if (left > 1) sp[j0 + 1] = n4.y;
                        if (left > 2) sp[j0 + 2] = n4.z;
                    }
                    if (evict) {
                        const int4 p4 = *reinterpret_cast<const int4 *>(apos + j0);
                        h2o_fold(best, bslot, n4.x, p4.x, s_lo + j0, P.n_sink, P.p, P.n_recent);
                        if (left > 1) h2o_fold(best, bslot, n4.y, p4.y, s_lo + j0 + 1, P.n_sink, P.p, P.n_recent);
                        if (left > 2) h2o_fold(best, bslot, n4.z, p4.z, s_lo + j0 + 2, P.n_sink, P.p, P.n_recent);
                        if (left > 3) h2o_fold(best, bslot, n4.w, p4.w, s_lo + j0 + 3, P.n_sink, P.p, P.n_recent);
                    }
                }
                return;
            }
            for (int j = tid; j < n_mine; j += kThreads) {
                float a = 0.f;
#pragma unroll
                for (int g = 0; g < G; ++g) a = fmaf(zbuf[g * zc + j], fself[g], a);
                const size_t si = unit * CS + s_lo + j;
                if (P.score_int8) {
                    const float v = fmaf(P.score_keep, stored_score(j), a);
                    zbuf[j] = v;
                    if (apos[j] >= 0) qmax = fmaxf(qmax, v);
                    continue;
                }
                const float sc = score_store(P, si, fmaf(P.score_keep, stored_score(j), a));
                if (evict) {
                    const int ps = apos[j];
                    if ((fill || pools) && ps < 0 && s_lo + j < emin) emin = s_lo + j;
                    if (pools) {
                        // two-pool: every held token is a candidate of the pool its flag names
                        if (ps >= 0) {
                            const uint64_t key = h2o_key(sc, ps);
                            if (apool[j] != 0) {
                                if (key < best2) {
                                    best2 = key;
                                    bslot2 = s_lo + j;
                                }
                            } else if (key < best) {
                                best = key;
                                bslot = s_lo + j;
                            }
                        }
                    } else {
                        h2o_fold(best, bslot, sc, ps, s_lo + j, P.n_sink, P.p, P.n_recent);
                    }
                }
            }
        };

        if (Si == 1) {
            // ------------------------------ output, one CTA per unit: o / l
            auto write_output = [&]() {
                T *outp = static_cast<T *>(P.out) + unit * (G * D);
                for (int jp = tid; jp < kPairs; jp += kThreads) {
                    const int g = (2 * jp) / D;
                    float ox, oy;
                    cta_o(g, ox, oy);
                    const float inv = 1.f / cta_l(g);
                    TPair<T> o2;
                    o2.x = E::from_f32(ox * inv);
                    o2.y = E::from_f32(oy * inv);
                    *reinterpret_cast<TPair<T> *>(outp + 2 * jp) = o2;
                }
            };
            if (!alias) write_output();
            if (tid < G) {
                const float l = cta_l(tid);
                if (!(l > 0.f && l <= FLT_MAX)) atomicOr(P.err, KVEVICT_DEV_NONFINITE);
            }
            if (has_score) {
                // ------------------------------ cumulative scores (H2O)
                wait_aux();
                float invl[G], fself[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    invl[g] = 1.f / cta_l(g);
                    fself[g] = invl[g] * (1.0f / G);
                }
                uint64_t best = ~0ull, best2 = ~0ull;
                int32_t bslot = -1, bslot2 = -1, emin = INT_MAX;
                float qmax = 0.f;
                // INT8 with at most kI8Groups groups of four slots per thread: the
                // updated values stay in registers across the barrier that finds the
                // unit's largest score (no second pass over the logit cells)
                constexpr int kI8Groups = 1;
                const bool int8_regs = P.score_int8 && n_mine <= 4 * kI8Groups * kThreads;
                float v8[kI8Groups][4];
                if (int8_regs) {
                    const uint8_t *codes = ascore8;
#pragma unroll
                    for (int it = 0; it < kI8Groups; ++it) {
                        const int j0 = 4 * tid + it * 4 * kThreads;
                        if (j0 >= n_mine) break;
                        float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const float4 z = *reinterpret_cast<const float4 *>(zbuf + g * zc + j0);
                            a4[0] = fmaf(z.x, fself[g], a4[0]);
                            a4[1] = fmaf(z.y, fself[g], a4[1]);
                            a4[2] = fmaf(z.z, fself[g], a4[2]);
                            a4[3] = fmaf(z.w, fself[g], a4[3]);
                        }
                        const uint32_t c4 = *reinterpret_cast<const uint32_t *>(codes + j0);
                        const int4 p4 = *reinterpret_cast<const int4 *>(apos + j0);
                        const int pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float old = static_cast<float>((c4 >> (8 * e)) & 0xFFu) * qscale_u;
                            v8[it][e] = fmaf(P.score_keep, old, a4[e]);
                            if (j0 + e < n_mine && pp[e] >= 0) qmax = fmaxf(qmax, v8[it][e]);
                        }
                    }
                } else if (general_scores) {
                    score_pass(Flag<true>{}, fself, best, bslot, best2, bslot2, emin, qmax);
                } else {
                    score_pass(Flag<false>{}, fself, best, bslot, best2, bslot2, emin, qmax);
                }
                if (P.score_int8) {
                    // the unit's largest score, the new token's included (every
                    // thread forms that one as thread 0 does); then the codes
                    // c = round(s * 255 / max) (0..255) and the stored values c * scale
                    float a = 0.f;
#pragma unroll
                    for (int g = 0; g < G; ++g) a = fmaf(M.pnew[g], invl[g], a);
                    a *= 1.0f / G;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
                    if (lane == 0) M.wqmax[warp] = qmax;
                    __syncthreads();  // every warp's largest; every read of the old scale is done
                    float mx = a;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, M.wqmax[w]);
                    const float inv = mx > 0.f ? 255.f / mx : 0.f;
                    const float scl = mx / 255.f;
                    auto code = [&](float v) {
                        const float c = fminf(rintf(v * inv), 255.f);
                        return c >= 0.f ? c : 0.f;
                    };
                    uint8_t *codes_out = static_cast<uint8_t *>(P.score) + unit * CS + s_lo;
                    if (int8_regs) {
#pragma unroll
                        for (int it = 0; it < kI8Groups; ++it) {
                            const int j0 = 4 * tid + it * 4 * kThreads;
                            if (j0 >= n_mine) break;
                            const int left = n_mine - j0;
                            const int4 p4 = *reinterpret_cast<const int4 *>(apos + j0);
                            const int pp[4] = {p4.x, p4.y, p4.z, p4.w};
                            uint32_t packed = 0;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float c = code(v8[it][e]);
                                packed |= static_cast<uint32_t>(c) << (8 * e);
                                if (evict && e < left) h2o_fold(best, bslot, c * scl, pp[e], s_lo + j0 + e, P.n_sink, P.p, P.n_recent);
                            }
                            if (left >= 4) {
                                *reinterpret_cast<uint32_t *>(codes_out + j0) = packed;
                            } else {
                                for (int e = 0; e < left; ++e) codes_out[j0 + e] = static_cast<uint8_t>(packed >> (8 * e));
                            }
                        }
                    } else {
                        for (int j = tid; j < n_mine; j += kThreads) {
                            const float c = code(zbuf[j]);
                            codes_out[j] = static_cast<uint8_t>(c);
                            if (evict) h2o_fold(best, bslot, c * scl, apos[j], s_lo + j, P.n_sink, P.p, P.n_recent);
                        }
                    }
                    anew_code = static_cast<uint8_t>(code(a));
                    anew = code(a) * scl;
                    if (tid == 0) {
                        M.anew = anew;
                        P.qscale[unit] = scl;
                    }
                } else if (tid == 0) {
                    float a = 0.f;
#pragma unroll
                    for (int g = 0; g < G; ++g) a = fmaf(M.pnew[g], invl[g], a);
                    anew = score_round(P, a * (1.0f / G));
                    M.anew = anew;
                }
                if (evict) {
                    warp_argmin(best, bslot);
                    if (pools) warp_argmin(best2, bslot2);
                    if (fill || pools) emin = warp_min_s32(emin);
                    if (lane == 0) {
                        M.wkey[warp] = best;
                        M.wslot[warp] = bslot;
                        M.wempty[warp] = emin;
                        M.wkey2[warp] = best2;
                        M.wslot2[warp] = bslot2;
                    }
                }
                __syncthreads();  // (B) candidates visible; every read of this unit's aux data and logits is done
                if (alias) {
                    write_partials();
                    __syncthreads();
                    write_output();
                }
                if (evict) {
                    // every warp reduces the warps' candidates itself
                    uint64_t k;
                    int32_t sl;
                    argmin_of(M.wkey, M.wslot, kWarps, lane, k, sl);
                    int32_t em = (fill || pools) ? warp_min_s32(lane < kWarps ? M.wempty[lane] : INT_MAX) : INT_MAX;
                    if (pools) {
                        uint64_t k2;
                        int32_t sl2;
                        argmin_of(M.wkey2, M.wslot2, kWarps, lane, k2, sl2);
                        if (P.n_active < P.C) em = min(em, P.n_active);  // the slots past the scanned ones are empty
                        const uint64_t kn = h2o_key(M.anew, P.p);
                        pd = pool_decide(P.recent_full != 0, P.hh_threshold, k, sl, k2, sl2, em, kn);
                        if (pd.dest == INT_MAX) {  // no room where the rule needs an empty slot
                            if (tid == 0) atomicOr(P.err, KVEVICT_DEV_NO_CANDIDATE);
                            pd.dest = -1;
                            pd.promote = -1;
                        }
                        win_key = pd.evicted;
                        dest = pd.dest;
                    } else if (em != INT_MAX) {  // an empty slot: no eviction
                        win_key = kEmptyKey;
                        dest = em;
                    } else {
                        win_key = k;
                        dest = sl;
                        if (sl < 0 && tid == 0) atomicOr(P.err, KVEVICT_DEV_NO_CANDIDATE);
                    }
                }
            } else if (alias) {  // no score pass: every read of the logits was done by (A)
                write_partials();
                __syncthreads();
                write_output();
            }
            // the next unit's positions/scores may come in
            if (tid == 0 && need_aux && i + 1 < W.n_items) issue_aux(i + 1);
            if (!evict) dest = dest_mine;
            writer = true;
        } else {
            // ------------------------------------------ cluster exchange
            // Every CTA pushes its (m, l) to all CTAs of the cluster and its
            // output partial to the CTA that owns those coordinates (CTA r
            // owns the slice [r SL, (r + 1) SL), SL = G D / S). Unaliased, both
            // go before barrier (1); aliased, the output partials exist only
            // after the score pass and go, with the eviction candidates,
            // before barrier (2). The buffers alternate between units: a CTA
            // writes a peer's buffer of parity b again only after both passed
            // barrier (1) of the next unit, when the peer has finished reading it.
            const int b = i & 1;
            constexpr int GD = G * D;
            const int SL = GD / S;
            auto push_partials = [&]() {
                for (int jp = tid; jp < kPairs; jp += kThreads) {
                    const int g = (2 * jp) / D;
                    float ox, oy;
                    cta_o(g, ox, oy);
                    const int j = 2 * jp, r = j / SL;
                    st_peer_f32x2(peer_addr(&M.xo[b][ri * SL + (j - r * SL)], r), make_float2(ox, oy));
                }
            };
            if (!alias) push_partials();
            if (tid < G) {
                const float2 ml = make_float2(M.m[tid], cta_l(tid));
                for (int c = 0; c < S; ++c) st_peer_f32x2(peer_addr(&M.xml[b][ri][tid], c), ml);
            }
            cluster_sync();  // (1) every CTA's (m, l) (and unaliased partials) are here

            // -------------------------------------------------------- combine
            if (tid < G) {
                float mg = -INFINITY;
                for (int c = 0; c < S; ++c) mg = fmaxf(mg, M.xml[b][c][tid].x);
                float lg = 0.f;
                for (int c = 0; c < S; ++c) {
                    const float2 ml = M.xml[b][c][tid];
                    if (ml.x != -INFINITY) lg += ml.y * exp2f(ml.x - mg);
                }
                if (ri == 0 && !(lg > 0.f && lg <= FLT_MAX)) atomicOr(P.err, KVEVICT_DEV_NONFINITE);
                const float inv = 1.f / lg;
                for (int c = 0; c < S; ++c) {
                    const float mc = M.xml[b][c][tid].x;
                    M.fac[c][tid] = (mc == -INFINITY) ? 0.f : exp2f(mc - mg) * inv;
                }
            }
            __syncthreads();
            auto write_slice = [&]() {
                const int i0 = ri * SL;
                T *outp = static_cast<T *>(P.out) + unit * GD;
                for (int k = tid; k < SL; k += kThreads) {
                    const int g = (i0 + k) / D;
                    float o = 0.f;
                    for (int c = 0; c < S; ++c) o = fmaf(M.xo[b][c * SL + k], M.fac[c][g], o);
                    outp[i0 + k] = E::from_f32(o);
                }
            };
            if (!alias) write_slice();

            // ------------------------------------------ cumulative scores (H2O)
            if (has_score) {
                wait_aux();
                float fself[G];
#pragma unroll
                for (int g = 0; g < G; ++g) fself[g] = M.fac[ri][g] * (1.0f / G);
                uint64_t best = ~0ull, best2 = ~0ull;
                int32_t bslot = -1, bslot2 = -1, emin = INT_MAX;
                float qmax = 0.f;  // (INT8 scores never reach a cluster)
                if (general_scores) score_pass(Flag<true>{}, fself, best, bslot, best2, bslot2, emin, qmax);
                else score_pass(Flag<false>{}, fself, best, bslot, best2, bslot2, emin, qmax);
                if (ri == 0 && tid == 0) {
                    float a = 0.f;
#pragma unroll
                    for (int g = 0; g < G; ++g) a = fmaf(M.pnew[g], M.fac[0][g], a);
                    anew = score_round(P, a * (1.0f / G));
                }
                if (evict) {
                    warp_argmin(best, bslot);
                    if (pools) warp_argmin(best2, bslot2);
                    if (fill || pools) emin = warp_min_s32(emin);
                    if (lane == 0) {
                        M.wkey[warp] = best;
                        M.wslot[warp] = bslot;
                        M.wempty[warp] = emin;
                        M.wkey2[warp] = best2;
                        M.wslot2[warp] = bslot2;
                    }
                }
                __syncthreads();  // candidates visible; every read of this unit's aux data is done
                if (evict && warp == 0) {
                    // this CTA's candidates (and, filling, its lowest empty slot) to every
                    // CTA; rank 0's new-token score too
                    uint64_t k, k2 = ~0ull;
                    int32_t sl, sl2 = -1;
                    argmin_of(M.wkey, M.wslot, kWarps, lane, k, sl);
                    if (pools) argmin_of(M.wkey2, M.wslot2, kWarps, lane, k2, sl2);
                    const int32_t em =
                        (fill || pools) ? warp_min_s32(lane < kWarps ? M.wempty[lane] : INT_MAX) : INT_MAX;
                    if (lane < S) {
                        st_peer_u64(peer_addr(&M.xkey[b][ri], lane), k);
                        st_peer_s32(peer_addr(&M.xslot[b][ri], lane), sl);
                        st_peer_s32(peer_addr(&M.xempty[b][ri], lane), em);
                        if (pools) {
                            st_peer_u64(peer_addr(&M.xkey2[b][ri], lane), k2);
                            st_peer_s32(peer_addr(&M.xslot2[b][ri], lane), sl2);
                        }
                    }
                    if (ri == 0 && lane == 0)
                        for (int c = 0; c < S; ++c) st_peer_f32(peer_addr(&M.xanew[b], c), anew);
                }
            }
            if (alias) {
                // every read of the logits is done: the score pass ended with a
                // barrier, and without scores nothing read them after (A)
                write_partials();
                __syncthreads();
                push_partials();
                cluster_sync();  // (2) every CTA's partials (and candidates) are here
                write_slice();
            }
            // the next unit's positions/scores may come in
            if (tid == 0 && need_aux && i + 1 < W.n_items) issue_aux(i + 1);

            // --------------------------------------------------------- victim
            if (evict) {
                if (!alias) cluster_sync();  // (2) every CTA's candidate is here
                uint64_t k;
                int32_t sl;
                argmin_of(M.xkey[b], M.xslot[b], S, lane, k, sl);
                int32_t em = (fill || pools) ? warp_min_s32(lane < S ? M.xempty[b][lane] : INT_MAX) : INT_MAX;
                if (pools) {
                    uint64_t k2;
                    int32_t sl2;
                    argmin_of(M.xkey2[b], M.xslot2[b], S, lane, k2, sl2);
                    if (P.n_active < P.C) em = min(em, P.n_active);  // the slots past the scanned ones are empty
                    const uint64_t kn = h2o_key(M.xanew[b], P.p);
                    pd = pool_decide(P.recent_full != 0, P.hh_threshold, k, sl, k2, sl2, em, kn);
                    if (pd.dest == INT_MAX) {  // no room where the rule needs an empty slot
                        if (ri == 0 && tid == 0) atomicOr(P.err, KVEVICT_DEV_NO_CANDIDATE);
                        pd.dest = -1;
                        pd.promote = -1;
                    }
                    win_key = pd.evicted;
                    dest = pd.dest;
                } else if (em != INT_MAX) {  // an empty slot: no eviction
                    win_key = kEmptyKey;
                    dest = em;
                } else {
                    win_key = k;
                    dest = sl;
                    if (sl < 0 && ri == 0 && tid == 0) atomicOr(P.err, KVEVICT_DEV_NO_CANDIDATE);
                }
                // the CTA that attended the victim; a slot past the scanned ones: rank 0
                writer = (dest >= s_lo && dest < s_hi) || (dest >= P.n_active && ri == 0);
                if (has_score) anew = M.xanew[b];
            } else {
                dest = dest_mine;
                writer = ri == 0;
            }
        }

        // ------------------------------------------------------------- insert
        // The new token's K/V row (prefetched pairs), position and score go
        // in place into slot `dest`.
        if (!evict && (dest < 0 || dest >= P.C)) {
            if (writer && tid == 0) atomicOr(P.err, KVEVICT_DEV_BAD_SLOT);
            dest = -1;
        }
        // two-pool: the promotion record of the trace (-2: the new token itself)
        const int prec = pd.promote >= 0 ? pd.promote : (pd.new_pool ? -2 : -1);
        if (pools && tid == 0) {
            const bool mine = Si == 1 || (pd.promote >= s_lo && pd.promote < s_hi);
            if (pd.promote >= 0 && mine) P.pool[unit * P.pstride + pd.promote] = 1;
            if (dest < 0 && ri == 0) {  // the new token itself left: its score leaves the cache
                if (P.ledger) ledger_add(P.ledger + unit, __uint_as_float(static_cast<uint32_t>(win_key >> 32)));
                if (P.trace != nullptr)
                    reinterpret_cast<int4 *>(P.trace)[unit] = make_int4(
                        -1, static_cast<int32_t>(static_cast<uint32_t>(win_key)),
                        static_cast<int32_t>(static_cast<uint32_t>(win_key >> 32)), prec);
            }
        }
        if (writer && dest >= 0) {
            if (tid < D / 2) {
                *reinterpret_cast<TPair<T> *>(static_cast<T *>(P.kc) + (unit * C + dest) * D + dp) = kpair;
                *reinterpret_cast<TPair<T> *>(static_cast<T *>(P.vc) + (unit * C + dest) * D + dp) = vpair;
            }
            if (tid == 0) {
                // the evicted token's position and score are the winning key;
                // otherwise they are read only when a trace is kept
                int32_t old_pos = static_cast<int32_t>(static_cast<uint32_t>(win_key));
                float old_score = __uint_as_float(static_cast<uint32_t>(win_key >> 32));
                // an evicted token's stored score leaves the cache: the ledger keeps it
                if (evict && old_pos >= 0 && P.ledger) ledger_add(P.ledger + unit, old_score);
                if (!evict && P.trace != nullptr) {
                    old_pos = P.pos[unit * CS + dest];
                    // (INT8: the codes were rewritten above; the slot is an empty one, score 0)
                    old_score = has_score && !P.score_int8 ? score_load(P, unit * CS + dest) : 0.f;
                }
                P.pos[unit * CS + dest] = P.p;
                if (P.score_int8) static_cast<uint8_t *>(P.score)[unit * CS + dest] = anew_code;
                else if (has_score) score_store(P, unit * CS + dest, anew);
                if (pools) P.pool[unit * P.pstride + dest] = static_cast<uint8_t>(pd.new_pool);
                if (P.trace != nullptr)
                    reinterpret_cast<int4 *>(P.trace)[unit] =
                        make_int4(dest, old_pos, __float_as_int(old_score), pools ? prec : __float_as_int(anew));
            }
        }
    }
    // No CTA leaves while a peer might still store into its shared memory.
    if (S > 1) cluster_sync();

    // After a timed-out wait some copies may still be landing: wait for them
    // (bounded) before the CTA exits.
    if (tid == 0 && M.abort) {
        for (int st = 0; st < NST; ++st)
            if (M.issued[st] > 0) mbar_wait(&M.full[st], (M.issued[st] - 1) & 1);
        if (M.aux_issued > 0) mbar_wait(&M.auxbar, (M.aux_issued - 1) & 1);
    }
}

// The H2O eviction decision alone, on caller-supplied fp32 scores: for every
// unit (one CTA), the candidate with the smallest (score, position) among
// slots [0, n_active) -- the victim the fused decode epilogue would take with
// these scores. Same candidate rule, key and reductions (h2o_fold,
// warp_argmin, argmin_of) as that epilogue, same CTA shape.
template <int kWarps> __global__ void __launch_bounds__(kWarps * 32) h2o_select_kernel(const SelectParams P)
{
    __shared__ uint64_t wkey[kWarps];
    __shared__ int32_t wslot[kWarps];
    const size_t unit = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t best = ~0ull;
    int32_t bslot = -1;
    for (int j = tid; j < P.n_active; j += kWarps * 32)
        h2o_fold(best, bslot, P.score[unit * P.C + j], P.pos[unit * P.cstride + j], j, P.n_sink, P.p, P.n_recent);
    warp_argmin(best, bslot);
    if (lane == 0) {
        wkey[warp] = best;
        wslot[warp] = bslot;
    }
    __syncthreads();
    if (warp == 0) {
        uint64_t k;
        int32_t sl;
        argmin_of(wkey, wslot, kWarps, lane, k, sl);
        if (lane == 0) P.victim[unit] = sl;
    }
}

}  // namespace kvevict
