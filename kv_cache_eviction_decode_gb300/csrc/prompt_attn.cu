// prompt_attn.cu -- Q-seeded prefill: the prompt's causal attention scores the
// prompt, then the budget is enforced by the greedy rule of Algorithm 1
// ("h2o: heavy-hitter oracle" summary: the cumulative attention a token
// receives is its score; remove the token whose removal keeps the highest
// total). With z_gij = q_gi . k_j / sqrt(d) over j <= i:
//   pass 1  per query row i of head g: ms_gi = m_gi + log2(l_gi), the log2 of
//           its softmax normaliser (m the row max, l the row sum, log2 units),
//           stored negated;
//   pass 2  per key j: score_j = (1/G) sum_g sum_{i >= j} 2^(z_gij - ms_gi);
//   cut     keep the n_sink first and n_recent last positions and, of the
//           rest, all but the P - K with the smallest (score, position).
//
// Passes 1 and 2 are one kernel body on the 5th-generation tensor cores: a
// CTA keeps one 128-row tile A (pass 1: 128 queries; pass 2: 128 keys) in
// shared memory and streams 128-row tiles B (pass 1: the keys up to the
// diagonal; pass 2: the queries from the diagonal on, for each of the G query
// heads). tcgen05.mma computes A B^T (128 x 128, fp32) into one of two TMEM
// accumulators while the epilogue warps read the other; every thread owns one
// row of A, so both reductions (over a query row, over a key column of the
// attention matrix) stay inside a thread.
//
// Warps: 0-15 epilogue (four per TMEM lane quadrant, each taking 32 of the
// 128 columns), 16 TMA producer (and TMEM allocation), 17 MMA issuer.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include "device_common.cuh"
#include "prompt_attn.h"
#include "tc5_common.cuh"

namespace kvevict {

namespace {

constexpr int kPT = kPromptTile;
constexpr int kPStages = 4;
constexpr int kEpiWarps = 16;
constexpr int kSlices = kEpiWarps / 4;  // column slices per row (warps sharing a lane quadrant)
// Pass 2 (unstacked): each B tile's 128 query normalisers are copied into one
// of kNrmSlots shared-memory slots, beside the tile, completing on the slot's
// own mbarrier. The copy for tile t is issued once the producer has seen the
// MMAs of tile t - 4 complete (one ring turn), and those were issued after the
// epilogue released tile t - 6: with 6 slots or more, the slot's previous tile
// (t - kNrmSlots) is always released before its next copy starts.
constexpr int kNrmSlots = 8;
constexpr int kProdWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
constexpr int kPThreads = (kEpiWarps + 2) * 32;
constexpr uint32_t kTmemCols = 256;  // two 128-column fp32 accumulators

enum PromptMode : int { kRowStats = 0, kColSum = 1 };

template <int D> struct PromptLayout {
    static constexpr int kTileBytes = kPT * D * 2;
    static constexpr int kBoxBytes = kPT * 128;  // one 128-row x 64-column box
    static constexpr int kOffA = 0;              // two A tiles: the current item's and the next one's
    static constexpr int kOffB = 2 * kTileBytes;
    static constexpr int kOffBar = kOffB + kPStages * kTileBytes;
    static constexpr int kOffXchg = kOffBar + 512;  // [2 items][kSlices - 1][128]
    static constexpr int kOffPart = kOffXchg + 2 * (kSlices - 1) * kPT * 8;  // per-head partials [8][kSlices][128]
    static constexpr int kOffNrm = kOffPart + 8 * kSlices * kPT * 4;          // pass 2: [kNrmSlots][128] normalisers
    static constexpr int kBytes = kOffNrm + kNrmSlots * kPT * 4 + 1024;  // + slack to align the base to 1 KB
};

__device__ __forceinline__ void flag_timeout(uint32_t *err) { atomicOr(err, KVEVICT_DEV_WAIT_TIMEOUT); }

// 2^x by the special-function unit (PTX ex2.approx, subnormal results flushed
// to zero); x = -inf gives 0.
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (the three-input max.f32 of sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 lanes per instruction (Blackwell's packed f32x2 FMA and add).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// sum over e < 32 of 2^(r_e * c + a_e) (r the raw fp32 bits of 32 TMEM
// columns, a[e] from `add`), in four independent packed chains.
__device__ __forceinline__ float exp2_sum32(const uint32_t (&r)[32], float c, const float4 *add)
{
    const float2 c2 = make_float2(c, c);
    float2 s[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const float4 nms = __ldg(add + e4);
        const int e = e4 * 4;
        const float2 za = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2, make_float2(nms.x, nms.y));
        const float2 zb = ffma2(make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), c2, make_float2(nms.z, nms.w));
        s[(e4 & 1) * 2] = fadd2(s[(e4 & 1) * 2], make_float2(ex2(za.x), ex2(za.y)));
        s[(e4 & 1) * 2 + 1] = fadd2(s[(e4 & 1) * 2 + 1], make_float2(ex2(zb.x), ex2(zb.y)));
    }
    const float2 t = fadd2(fadd2(s[0], s[1]), fadd2(s[2], s[3]));
    return t.x + t.y;
}

// STACK (SnapKV, window a multiple of 32): the G query heads' window rows,
// contiguous in Q, form one stacked row axis r = g * w + t per unit (query
// head g, query position P - w + t), tiled by 128 across heads.
template <int D, int MODE, bool STACK>
__global__ void __launch_bounds__(kPThreads, 1) prompt_attn_kernel(const __grid_constant__ PromptAttnParams p)
{
    using L = PromptLayout<D>;
    extern __shared__ uint8_t praw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(praw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    uint64_t *a_full = bars;                 // [2] an item's A tile landed
    uint64_t *a_empty = a_full + 2;          // [2] every MMA on that A tile completed
    uint64_t *b_full = a_empty + 2;          // [kPStages]
    uint64_t *b_empty = b_full + kPStages;   // [kPStages]
    uint64_t *s_full = b_empty + kPStages;   // [2] accumulators
    uint64_t *s_empty = s_full + 2;          // [2]
    uint64_t *i_full = s_empty + 2;          // [2] the next item's index is posted
    uint64_t *i_empty = i_full + 2;          // [2] every consumer has read it
    uint64_t *n_full = i_empty + 2;          // [kNrmSlots] pass 2: a B tile's normalisers landed
    int *item_idx = reinterpret_cast<int *>(n_full + kNrmSlots);  // [2]
    int *eagree = item_idx + 2;                            // [kEpiWarps] what each epilogue warp read
    uint32_t *tslot = reinterpret_cast<uint32_t *>(eagree + kEpiWarps);
    float2 *xchg_all = reinterpret_cast<float2 *>(sm + L::kOffXchg);
    float *hpart = reinterpret_cast<float *>(sm + L::kOffPart);
    float *nrm = reinterpret_cast<float *>(sm + L::kOffNrm);
    constexpr bool kNrm = MODE == kColSum && !STACK;  // normalisers staged in shared memory

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nT = (p.P + kPT - 1) / kPT;
    const int qlo_t = p.q_lo / kPT;
    const int qs0 = qlo_t * kPT;  // first query row with statistics
    const int Lq = p.G * p.q_stride;  // STACK: stacked rows per unit
    const int nLq = (Lq + kPT - 1) / kPT;
    // Persistent: the CTAs take items of p.nheads x p.ntiles, head-major, from
    // a work counter (the producer fetches the next index while the current
    // item streams and posts it to the MMA and epilogue warps), so the items in
    // flight at one time are consecutive: a few heads, whose B tiles are read
    // once into L2. Each head's tiles come the most work first. An item: pass 1 --
    // query tile `tile` of query head `head` (= b * Hq + qh), B tiles = key
    // tiles 0..tile of its KV head; pass 2 -- key tile `tile` of unit `head`
    // (= b * Hkv + kvh), B tiles = (query head g, query tile qt) for g < G and
    // qt from max(tile, first query tile) on.
    const int n_items = p.ntiles * p.nheads;
    struct Item {
        int tile, head, qt0, nq, n_b, a_row;
    };
    auto item_at = [&](int k) {
        Item it;
        it.head = k / p.ntiles;
        const int ti = k - it.head * p.ntiles;
        it.tile = MODE == kRowStats && !STACK ? nT - 1 - ti : ti;
        it.qt0 = max(it.tile, qlo_t);
        it.nq = nT - it.qt0;
        it.n_b = STACK ? (MODE == kRowStats ? nT : nLq) : (MODE == kRowStats ? it.tile + 1 : p.G * it.nq);
        // Q rows: query i of query head h is row h * q_stride + i - q_first (rows
        // before a head's first given query belong to the previous head or lie
        // before the tensor: they only feed masked rows and columns)
        it.a_row = STACK ? (MODE == kRowStats ? it.head * Lq + it.tile * kPT : it.head * p.P + it.tile * kPT)
                         : (MODE == kRowStats ? it.head * p.q_stride + it.tile * kPT - p.q_first
                                              : it.head * p.P + it.tile * kPT);
        return it;
    };
    auto b_row = [&](const Item &it, int n) -> int {
        if (STACK) return MODE == kRowStats ? it.head * p.P + n * kPT : it.head * Lq + n * kPT;
        if (MODE == kRowStats) {
            const int b = it.head / p.Hq, qh = it.head - b * p.Hq;
            return (b * p.Hkv + qh / p.G) * p.P + n * kPT;
        } else {
            const int b = it.head / p.Hkv, kvh = it.head - b * p.Hkv;
            const int g = n / it.nq, qt = it.qt0 + (n - g * it.nq);
            return (b * p.Hq + kvh * p.G + g) * p.q_stride + qt * kPT - p.q_first;
        }
    };

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], kEpiWarps);
        }
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&i_full[s], 1);
            mbar_init(&i_empty[s], kEpiWarps + 1);
        }
        for (int s = 0; s < kNrmSlots; ++s) mbar_init(&n_full[s], 1);
        mbar_fence_init();
    }
    if (warp == kProdWarp) tmem_alloc(tslot, kTmemCols);
    // The i-th item of this CTA (slot i & 1): its index, or -1 when the work is
    // done. `whole_warp`: every lane of the warp calls (the epilogue warps; one
    // arrival per warp after all lanes have read), else lane 0 alone (the MMA issuer).
    auto take_item = [&](int i, bool &ok, bool whole_warp) -> int {
        const int ib = i & 1;
        if (!mbar_wait(&i_full[ib], (i >> 1) & 1)) {
            ok = false;
            return -1;
        }
        const int k = *reinterpret_cast<volatile int *>(&item_idx[ib]);
        if (whole_warp) __syncwarp();
        if (lane == 0) mbar_arrive(&i_empty[ib]);
        return k;
    };
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tslot);

    // Counters over the CTA's whole run: B tiles (ring stage and phase) and
    // MMA tiles (accumulator and phase) continue across items; A tiles
    // alternate between two buffers by item.
    int issued_b = 0;     // producer: B tiles whose copies were issued
    int issued_a = 0;     // producer: A tiles whose copies were issued
    int issued_mma = 0;   // MMA issuer: tiles whose MMAs were issued
    int freed_a = 0;      // MMA issuer: items whose A tile release was committed

    if (warp == kProdWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool ok = true;
            for (int i = 0;; ++i) {
                const int ib = i & 1;
                if (i >= 2 && !mbar_wait(&i_empty[ib], ((i >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                int k = atomicAdd(p.work, 1);
                if (k >= n_items) k = -1;
                item_idx[ib] = k;
                mbar_arrive(&i_full[ib]);
                if (k < 0) break;
                const Item it = item_at(k);
                const int ab = i & 1;
                if (i >= 2 && !mbar_wait(&a_empty[ab], ((i >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&a_full[ab], L::kTileBytes);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d_plain(sm + L::kOffA + ab * L::kTileBytes + c * L::kBoxBytes, &p.tma, c * 64, it.a_row,
                                      &a_full[ab]);
                issued_a = i + 1;
                for (int n = 0; n < it.n_b; ++n) {
                    const int g = issued_b, s = g % kPStages;
                    if (g >= kPStages && !mbar_wait(&b_empty[s], ((g / kPStages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&b_full[s], L::kTileBytes);
                    const int row = b_row(it, n);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d_plain(sm + L::kOffB + s * L::kTileBytes + c * L::kBoxBytes, &p.tmb, c * 64, row,
                                          &b_full[s]);
                    if constexpr (kNrm) {
                        // the 128 queries' normalisers of this tile (query head gq, query tile qt)
                        const int b = it.head / p.Hkv, kvh = it.head - b * p.Hkv;
                        const int gq = n / it.nq, qt = it.qt0 + (n - gq * it.nq);
                        const float *src = p.stats + static_cast<size_t>(b * p.Hq + kvh * p.G + gq) * p.Ps + (qt * kPT - qs0);
                        const int ns = g % kNrmSlots;
                        mbar_arrive_expect_tx(&n_full[ns], kPT * 4);
                        bulk_g2s(nrm + ns * kPT, src, kPT * 4, &n_full[ns]);
                    }
                    issued_b = g + 1;
                }
            }
            if (!ok) flag_timeout(p.err);
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kPT, kPT);
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int k = take_item(i, ok, false);
                if (k < 0) break;
                const Item it = item_at(k);
                const int ab = i & 1;
                if (!mbar_wait(&a_full[ab], (i >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const uint32_t a0 = smem_u32(sm + L::kOffA + ab * L::kTileBytes);
                for (int n = 0; n < it.n_b; ++n) {
                    const int g = issued_mma, s = g % kPStages, acc = g & 1;
                    if (!mbar_wait(&b_full[s], (g / kPStages) & 1)) ok = false;
                    else if (g >= 2 && !mbar_wait(&s_empty[acc], ((g >> 1) - 1) & 1)) ok = false;
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t b0 = smem_u32(sm + L::kOffB + s * L::kTileBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = static_cast<uint32_t>((kk >> 2) * L::kBoxBytes + (kk & 3) * 32);
                        tc_mma_bf16(tmem + static_cast<uint32_t>(acc * kPT), smem_desc_sw128(a0 + koff),
                                    smem_desc_sw128(b0 + koff), idesc, kk > 0);
                    }
                    tc_commit(&b_empty[s]);
                    tc_commit(&s_full[acc]);
                    issued_mma = g + 1;
                }
                if (ok) {
                    tc_commit(&a_empty[ab]);  // the A tile is free once these MMAs complete
                    freed_a = i + 1;
                }
            }
            if (!ok) flag_timeout(p.err);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int quad = warp & 3, slice = warp >> 2;
        const int row = quad * 32 + lane;      // TMEM lane = row of the A tile
        const uint32_t lane_field = static_cast<uint32_t>(quad * 32) << 16;
        const int col0 = slice * 32;           // this warp's 32 columns of each tile
        const float c = p.scale_log2;
        bool ok = true;
        int gt = 0;                            // tiles consumed over the CTA's run
        for (int i = 0;; ++i) {
            // Every epilogue warp takes the posted index (bounded wait), then they all
            // agree on one through a barrier every warp reaches, so that they leave
            // the loop together: -1 (no more work) or a failed wait ends it for all.
            bool okk = true;
            const int kw = take_item(i, okk, true);
            if (lane == 0) eagree[warp] = okk ? kw : -2;
            named_bar_sync(3, kEpiWarps * 32);
            int k = eagree[0];
            for (int w = 1; w < kEpiWarps; ++w)
                if (eagree[w] != k) k = -2;
            named_bar_sync(3, kEpiWarps * 32);  // eagree may be written again
            if (k == -2 && lane == 0) flag_timeout(p.err);
            if (k < 0) break;
            const Item it = item_at(k);
            const int tile = it.tile, head = it.head, qt0 = it.qt0, nq = it.nq, n_b = it.n_b;
            const int a_idx = tile * kPT + row;    // pass 1: query i; pass 2: key j
            float2 *xchg = xchg_all + (i & 1) * (kSlices - 1) * kPT;
            float m = -INFINITY, l = 0.f;          // pass 1: running max and sum (log2 units)
            float acc = 0.f;                       // pass 2: mass received
            int cur_g = 0;                         // STACK pass 2: query head of the running sum
            if (MODE == kColSum && (STACK || p.per_head)) {
                // the previous item's per-head partials have been read (slice 0, after its barrier)
                if (i > 0) named_bar_sync(2, kEpiWarps * 32);
                if (STACK)
                    for (int g = 0; g < p.G; ++g) hpart[(g * kSlices + slice) * kPT + row] = 0.f;
            }
            // STACK pass 1: a warp whose 32 rows all lie past the stacked rows has nothing to do
            const bool idle = MODE == kRowStats && STACK && tile * kPT + quad * 32 >= Lq;
            int gq = 0, jq = 0;  // pass 2 (unstacked): tile n is query tile qt0 + jq of query head gq
            for (int n = 0; n < n_b; ++n, ++gt) {
                const int sb = gt & 1;
                // the TMEM load below is warp-collective: the whole warp agrees on `ok`
                if (ok && !__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (gt >> 1) & 1))) {
                    ok = false;
                    if (lane == 0) flag_timeout(p.err);
                }
                if (kNrm && ok &&
                    !__all_sync(0xffffffffu, mbar_wait(&n_full[gt % kNrmSlots], (gt / kNrmSlots) & 1))) {
                    ok = false;
                    if (lane == 0) flag_timeout(p.err);
                }
                tc_fence_after();
                if (ok && !idle) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_field + static_cast<uint32_t>(sb * kPT + col0), r);
                    tc_wait_ld();
                    if (MODE == kRowStats) {
                        // keys j = n * 128 + col0 + e; only the diagonal tile is masked (STACK: the
                        // keys from the window on, against this row's query position)
                        const int j0 = n * kPT + col0;
                        const int qi = STACK ? p.P - p.q_stride + a_idx % p.q_stride : a_idx;
                        float v[32];
                        if (STACK ? j0 + 32 > p.P - p.q_stride : n == tile) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                v[e] = (j0 + e <= qi && j0 + e < p.P) ? __uint_as_float(r[e]) : -INFINITY;
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
                        }
                        // the tile's max, two values per three-input max
                        float cm = fmax3(v[0], v[1], v[2]);
#pragma unroll
                        for (int e = 3; e < 31; e += 2) cm = fmax3(cm, v[e], v[e + 1]);
                        cm = fmaxf(cm, v[31]);
                        cm *= c;  // c > 0: the max of the scaled logits
                        if (cm > m) {
                            l *= ex2(m - cm);
                            m = cm;
                        }
                        if (m != -INFINITY) {
                            const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
                            float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float2 z = ffma2(make_float2(v[e], v[e + 1]), c2, nm2);
                                s2 = fadd2(s2, make_float2(ex2(z.x), ex2(z.y)));
                            }
                            l += s2.x + s2.y;
                        }
                    } else if (STACK) {
                        // stacked rows r0 .. r0 + 31 (one query head: w is a multiple of 32)
                        const int r0 = n * kPT + col0;
                        if (r0 < Lq) {
                            const int g = r0 / p.q_stride, i0 = p.P - p.q_stride + (r0 - g * p.q_stride);
                            if (g != cur_g) {
                                hpart[(cur_g * kSlices + slice) * kPT + row] = acc;
                                acc = 0.f;
                                cur_g = g;
                            }
                            const float4 *st = reinterpret_cast<const float4 *>(p.stats + static_cast<size_t>(head) * p.Ps + r0);
                            const float2 c2 = make_float2(c, c);
                            float2 s2 = make_float2(0.f, 0.f);
                            if (a_idx < p.P - p.q_stride) {  // a key before the window: every window query sees it
#pragma unroll
                                for (int e4 = 0; e4 < 8; ++e4) {
                                    const float4 nms = __ldg(st + e4);
                                    const int e = e4 * 4;
                                    const float2 za = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                                            c2, make_float2(nms.x, nms.y));
                                    const float2 zb = ffma2(make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])),
                                                            c2, make_float2(nms.z, nms.w));
                                    s2 = fadd2(s2, make_float2(ex2(za.x), ex2(za.y)));
                                    s2 = fadd2(s2, make_float2(ex2(zb.x), ex2(zb.y)));
                                }
                            } else {
#pragma unroll
                                for (int e4 = 0; e4 < 8; ++e4) {
                                    const float4 nms = __ldg(st + e4);
                                    const float mv[4] = {nms.x, nms.y, nms.z, nms.w};
#pragma unroll
                                    for (int t = 0; t < 4; ++t) {
                                        const int e = e4 * 4 + t;
                                        const float pr = ex2(fmaf(__uint_as_float(r[e]), c, mv[t]));
                                        const float add = (i0 + e >= a_idx) ? pr : 0.f;
                                        if (t & 1) s2.y += add;
                                        else s2.x += add;
                                    }
                                }
                            }
                            acc += s2.x + s2.y;
                        }
                    } else {
                        // queries i = qt * 128 + col0 + e of query head g
                        const int g = gq, qt = qt0 + jq;
                        const int i0 = qt * kPT + col0;
                        // minus the log2 normalisers of these 32 queries, staged by the producer
                        const float4 *st = reinterpret_cast<const float4 *>(nrm + (gt % kNrmSlots) * kPT + col0);
                        const bool full = qt > tile && i0 + 32 <= p.P && i0 >= p.q_lo;
                        const float2 c2 = make_float2(c, c);
                        float2 s2 = make_float2(0.f, 0.f);
                        if (full) {  // every query of these 32 columns attends this key
#pragma unroll
                            for (int e4 = 0; e4 < 8; ++e4) {
                                const float4 nms = st[e4];
                                const int e = e4 * 4;
                                const float2 za = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2,
                                                        make_float2(nms.x, nms.y));
                                const float2 zb = ffma2(make_float2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])),
                                                        c2, make_float2(nms.z, nms.w));
                                s2 = fadd2(s2, make_float2(ex2(za.x), ex2(za.y)));
                                s2 = fadd2(s2, make_float2(ex2(zb.x), ex2(zb.y)));
                            }
                        } else {
#pragma unroll
                            for (int e4 = 0; e4 < 8; ++e4) {
                                const float4 nms = st[e4];
                                const float mv[4] = {nms.x, nms.y, nms.z, nms.w};
#pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    const int e = e4 * 4 + t, i = i0 + e;
                                    const float pr = ex2(fmaf(__uint_as_float(r[e]), c, mv[t]));
                                    const float add = (i >= a_idx && i < p.P && i >= p.q_lo) ? pr : 0.f;
                                    if (t & 1) s2.y += add;
                                    else s2.x += add;
                                }
                            }
                        }
                        acc += s2.x + s2.y;
                        if (p.per_head && jq == nq - 1) {  // the last tile of query head g
                            hpart[(g * kSlices + slice) * kPT + row] = acc;
                            acc = 0.f;
                        }
                    }
                } else if (MODE == kColSum && p.per_head && !STACK) {
                    if (jq == nq - 1) hpart[(gq * kSlices + slice) * kPT + row] = 0.f;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                if (++jq == nq) {
                    jq = 0;
                    ++gq;
                }
            }
            if (MODE == kColSum && STACK) hpart[(cur_g * kSlices + slice) * kPT + row] = acc;
            // the column slices of each row meet: slices 1.. hand over to slice 0
            if (slice > 0) xchg[(slice - 1) * kPT + row] = MODE == kRowStats ? make_float2(m, l) : make_float2(acc, 0.f);
            named_bar_sync(1, kEpiWarps * 32);
            if (slice == 0 && ok) {
                if (MODE == kRowStats) {
                    float mm = m;
#pragma unroll
                    for (int k = 0; k < kSlices - 1; ++k) mm = fmaxf(mm, xchg[k * kPT + row].x);
                    float ll = m == -INFINITY ? 0.f : l * ex2(m - mm);
#pragma unroll
                    for (int k = 0; k < kSlices - 1; ++k) {
                        const float2 o = xchg[k * kPT + row];
                        if (o.x != -INFINITY) ll += o.y * ex2(o.x - mm);
                    }
                    if (STACK ? a_idx < Lq : a_idx < p.P)
                        p.stats[static_cast<size_t>(head) * p.Ps + (STACK ? a_idx : a_idx - qs0)] = -(mm + log2f(ll));
                } else if (p.per_head || STACK) {
                    if (a_idx < p.P) {
                        const int b = head / p.Hkv, kvh = head - b * p.Hkv;
                        for (int g = 0; g < p.G; ++g) {
                            float tot = 0.f;
#pragma unroll
                            for (int k = 0; k < kSlices; ++k) tot += hpart[(g * kSlices + k) * kPT + row];
                            p.score[static_cast<size_t>(b * p.Hq + kvh * p.G + g) * p.P + a_idx] = tot;
                        }
                    }
                } else {
                    float tot = acc;
#pragma unroll
                    for (int k = 0; k < kSlices - 1; ++k) tot += xchg[k * kPT + row].x;
                    if (a_idx < p.P) p.score[static_cast<size_t>(head) * p.P + a_idx] = tot * (1.f / p.G);
                }
            }
        }
    }

    // Teardown. After a timed-out wait, let the copies and MMAs already issued
    // finish (bounded) before the TMEM and the shared memory go away.
    if (warp == kProdWarp && lane == 0) {
        for (int n = max(0, issued_b - kPStages); n < issued_b; ++n)
            mbar_wait(&b_full[n % kPStages], (n / kPStages) & 1);
        if (kNrm)
            for (int n = max(0, issued_b - kNrmSlots); n < issued_b; ++n)
                mbar_wait(&n_full[n % kNrmSlots], (n / kNrmSlots) & 1);
        for (int i = max(0, issued_a - 2); i < issued_a; ++i) mbar_wait(&a_full[i & 1], (i >> 1) & 1);
    }
    if (warp == kMmaWarp && lane == 0) {
        for (int n = max(0, issued_mma - 2); n < issued_mma; ++n) mbar_wait(&s_full[n & 1], (n >> 1) & 1);
        for (int i = max(0, freed_a - 2); i < freed_a; ++i) mbar_wait(&a_empty[i & 1], (i >> 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProdWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------- SnapKV votes, streamed
// votes_gj = sum over the window's queries t of head g of 2^(z_gtj * c - ms_gt),
// z = q . k (bf16 in, fp32 accumulate), ms_gt the row's log2 normaliser from
// the row-statistics pass, for every prompt key j (masked causally inside the
// window). One persistent CTA per SM takes a contiguous range of items (unit,
// key tile of 128). The unit's Lq = G * w stacked window rows stay in shared
// memory as the B operand (reloaded when the range crosses into the next
// unit); the key tiles stream through a TMA ring as A. One tcgen05.mma of
// M = 128 keys, N = Lq rows per K step fills one of two TMEM accumulators
// while the epilogue reads the other: thread (quad, slice) owns key row
// quad * 32 + lane and the query heads slice, slice + 4, ... (every 32-row
// chunk of each), so it writes those heads' votes of its key itself.
constexpr int kVStages = 4;

template <int D> struct VotesLayout {
    static constexpr int kATile = kPT * D * 2;           // one key tile
    static constexpr int kBBytes = kSnapVotesMaxRows * D * 2;
    static constexpr int kOffB = 0;
    static constexpr int kOffA = kBBytes;
    static constexpr int kOffBar = kOffA + kVStages * kATile;
    static constexpr int kBytes = kOffBar + 256 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kPThreads, 1) snap_votes_kernel(const __grid_constant__ SnapVotesParams p)
{
    using L = VotesLayout<D>;
    extern __shared__ uint8_t vraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(vraw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::kOffBar);
    uint64_t *a_full = bars;                   // [kVStages]
    uint64_t *a_empty = a_full + kVStages;     // [kVStages]
    uint64_t *s_full = a_empty + kVStages;     // [2]
    uint64_t *s_empty = s_full + 2;            // [2]
    uint64_t *b_full = s_empty + 2;            // the unit's window rows landed
    uint64_t *b_free = b_full + 1;             // every MMA on the previous unit's rows completed
    uint32_t *tslot = reinterpret_cast<uint32_t *>(b_free + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = p.Lq;                        // MMA N: stacked window rows (multiple of 32, <= 256)
    const uint32_t tcols = N <= 16 ? 32u : (N <= 32 ? 64u : (N <= 64 ? 128u : (N <= 128 ? 256u : 512u)));
    const int nT = (p.P + kPT - 1) / kPT;
    const long long n_items = static_cast<long long>(p.units) * nT;
    const int it0 = static_cast<int>(n_items * blockIdx.x / gridDim.x);
    const int it1 = static_cast<int>(n_items * (blockIdx.x + 1) / gridDim.x);

    if (tid == 0) {
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], kEpiWarps);
        }
        mbar_init(b_full, 1);
        mbar_init(b_free, 1);
        mbar_fence_init();
    }
    if (warp == kProdWarp) tmem_alloc(tslot, tcols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tslot);

    int issued_a = 0, issued_mma = 0, loads_b = 0;

    if (warp == kProdWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int cur = -1;
            for (int it = it0; it < it1; ++it) {
                const int u = it / nT, kt = it - u * nT, n = it - it0;
                if (u != cur) {
                    // the previous unit's rows are overwritten once its MMAs are done
                    if (loads_b > 0 && !mbar_wait(b_free, (loads_b - 1) & 1)) {
                        flag_timeout(p.err);
                        break;
                    }
                    mbar_arrive_expect_tx(b_full, static_cast<uint32_t>(N * D * 2));
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d_plain(sm + L::kOffB + c * N * 128, &p.tmq, c * 64, u * N, b_full);
                    ++loads_b;
                    cur = u;
                }
                const int s = n % kVStages;
                if (n >= kVStages && !mbar_wait(&a_empty[s], ((n / kVStages) - 1) & 1)) {
                    flag_timeout(p.err);
                    break;
                }
                mbar_arrive_expect_tx(&a_full[s], static_cast<uint32_t>(L::kATile));
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d_plain(sm + L::kOffA + s * L::kATile + c * kPT * 128, &p.tmk, c * 64,
                                      u * p.P + kt * kPT, &a_full[s]);
                issued_a = n + 1;
            }
        }
    } else if (warp == kMmaWarp) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kPT, N);
            bool ok = true;
            int cur = -1, nb = 0;
            for (int it = it0; ok && it < it1; ++it) {
                const int u = it / nT, n = it - it0, s = n % kVStages, acc = n & 1;
                if (u != cur) {
                    if (nb > 0) tc_commit(b_free);  // completes once the previous unit's MMAs have
                    if (!mbar_wait(b_full, nb & 1)) {
                        ok = false;
                        break;
                    }
                    ++nb;
                    cur = u;
                }
                if (!mbar_wait(&a_full[s], (n / kVStages) & 1)) ok = false;
                else if (n >= 2 && !mbar_wait(&s_empty[acc], ((n >> 1) - 1) & 1)) ok = false;
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(sm + L::kOffA + s * L::kATile), b0 = smem_u32(sm + L::kOffB);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t ka = static_cast<uint32_t>((k >> 2) * kPT * 128 + (k & 3) * 32);
                    const uint32_t kb = static_cast<uint32_t>((k >> 2) * N * 128 + (k & 3) * 32);
                    tc_mma_bf16(tmem + static_cast<uint32_t>(acc * N), smem_desc_sw128(a0 + ka),
                                smem_desc_sw128(b0 + kb), idesc, k > 0);
                }
                tc_commit(&a_empty[s]);
                tc_commit(&s_full[acc]);
                issued_mma = n + 1;
            }
            if (!ok) flag_timeout(p.err);
        }
    } else {
        // ----------------------------------------------------------- epilogue
        const int quad = warp & 3, slice = warp >> 2;
        const int row = quad * 32 + lane;
        const uint32_t lane_field = static_cast<uint32_t>(quad * 32) << 16;
        const int per_head = p.w / 32;  // 32-row chunks per query head
        const float c = p.scale_log2;
        const int pre = p.P - p.w;  // keys before the window: every window query sees them
        bool ok = true;
        // item it = (unit u, key tile kt), u = it / nT, kept by counters
        int u = it0 / nT, kt = it0 - u * nT;
        int b = u / p.Hkv, kvh = u - b * p.Hkv;
        for (int it = it0; it < it1; ++it) {
            const int n = it - it0, sb = n & 1;
            const int j = kt * kPT + row;  // this thread's key
            // the TMEM loads below are warp-collective: the whole warp agrees on `ok`
            if (ok && !__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (n >> 1) & 1))) {
                ok = false;
                if (lane == 0) flag_timeout(p.err);
            }
            tc_fence_after();
            float *vout = p.votes + static_cast<size_t>(b * p.Hq + kvh * p.G) * p.P + j;
            // this slice's query heads: g = slice, slice + 4, ... (all chunks of each)
            for (int g = slice; ok && g < p.G; g += kSlices) {
                float tot = 0.f;
                for (int k = 0; k < per_head; ++k) {
                    const int ch = g * per_head + k;
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_field + static_cast<uint32_t>(sb * N + ch * 32), r);
                    tc_wait_ld();
                    const float4 *st = reinterpret_cast<const float4 *>(p.stats + static_cast<size_t>(u) * p.Ps + ch * 32);
                    if (kt * kPT + kPT <= pre) {  // a tile wholly before the window: no mask
                        tot += exp2_sum32(r, c, st);
                    } else {
                        // query position of stacked row ch * 32 + e: P - w + (row mod w)
                        const int i0 = pre + (ch * 32) % p.w;
                        float s0 = 0.f, s1 = 0.f;
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 nms = __ldg(st + e4);
                            const float mv[4] = {nms.x, nms.y, nms.z, nms.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int e = e4 * 4 + t;
                                const float pr = ex2(fmaf(__uint_as_float(r[e]), c, mv[t]));
                                const float add = (j <= i0 + e) ? pr : 0.f;
                                if (t & 1) s1 += add;
                                else s0 += add;
                            }
                        }
                        tot += s0 + s1;
                    }
                }
                if (j < p.P) vout[static_cast<size_t>(g) * p.P] = tot;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[sb]);
            if (++kt == nT) {
                kt = 0;
                ++u;
                if (++kvh == p.Hkv) {
                    kvh = 0;
                    ++b;
                }
            }
        }
    }

    // Teardown: let the copies and MMAs already issued finish (bounded) before
    // the TMEM and the shared memory go away.
    if (warp == kProdWarp && lane == 0) {
        for (int n = max(0, issued_a - kVStages); n < issued_a; ++n)
            mbar_wait(&a_full[n % kVStages], (n / kVStages) & 1);
        if (loads_b > 0) mbar_wait(b_full, (loads_b - 1) & 1);
    }
    if (warp == kMmaWarp && lane == 0) {
        for (int n = max(0, issued_mma - 2); n < issued_mma; ++n) mbar_wait(&s_full[n & 1], (n >> 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProdWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, tcols);
    }
}

// ------------------------------------------------------------------ cut
constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelCand = 2 * kSelThreads;  // patterns the in-register search gathers once its interval is narrow

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// Block-wide reductions of the selection kernels (kSelThreads threads; `red`
// holds kSelWarps ints, `total` one; both free again on return).
struct BlockOps {
    int *red, *total;
    int lane, warp;
    // exclusive prefix of v over the threads in order (x) and the total (y)
    __device__ int2 scan(int v) const
    {
        const int inc = warp_incl_scan(v, lane);
        if (lane == 31) red[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            const int w = lane < kSelWarps ? red[lane] : 0;
            const int winc = warp_incl_scan(w, lane);
            if (lane < kSelWarps) red[lane] = winc - w;  // exclusive warp offsets
            if (lane == kSelWarps - 1) *total = winc;
        }
        __syncthreads();
        const int2 r = make_int2(red[warp] + inc - v, *total);
        __syncthreads();
        return r;
    }
};

// Warp w owns the positions [base, end) of [lo, hi): consecutive spans of a
// multiple of 32 positions, in warp order. Its walk visits 32 consecutive
// positions per step (lane l: base + 32 i + l): conflict-free in shared
// memory, and in position order across steps, lanes and warps.
struct WarpRange {
    int base, end;
    __device__ WarpRange(int lo, int hi, int warp)
    {
        const int span = 32 * ((hi - lo + 32 * kSelWarps - 1) / (32 * kSelWarps));
        base = min(hi, lo + warp * span);
        end = min(hi, base + span);
    }
};

__device__ __forceinline__ unsigned lanes_below(int lane) { return (1u << lane) - 1u; }

// The E-th smallest bit pattern T among bits[lo, hi) (1 <= E <= hi - lo) and
// how many of the E smallest equal T (`need`), by radix selection: four
// passes over 8-bit digits, most significant first, each a histogram of the
// digit among the patterns that share the digits found so far (increments
// aggregated over the lanes holding the same digit).
__device__ void radix_threshold(const uint32_t *bits, int lo, int hi, int E, int *hist, int *bc, uint32_t &T,
                                int &need)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const WarpRange R(lo, hi, warp);
    uint32_t prefix = 0, mask = 0;
    int rank = E;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
        __syncthreads();
        for (int j0 = R.base; j0 < R.end; j0 += 32) {
            const int j = j0 + lane;
            const uint32_t bt = j < R.end ? bits[j] : 0u;
            const bool m = j < R.end && (bt & mask) == prefix;
            const unsigned act = __ballot_sync(0xffffffffu, m);
            if (m) {
                const uint32_t d = (bt >> shift) & 255u;
                const unsigned peers = __match_any_sync(act, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[d], __popc(peers));
            }
        }
        __syncthreads();
        if (warp == 0) {  // lane l holds bins 8 l .. 8 l + 7; the one holding the rank-th picks the digit
            int c[8], sum = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                c[k] = hist[lane * 8 + k];
                sum += c[k];
            }
            const int incl = warp_incl_scan(sum, lane), excl = incl - sum;
            if (excl < rank && rank <= incl) {
                int acc = excl, d = 7;
                for (int k = 0; k < 8; ++k) {
                    if (acc + c[k] >= rank) {
                        d = k;
                        break;
                    }
                    acc += c[k];
                }
                bc[0] = lane * 8 + d;
                bc[1] = rank - acc;
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(bc[0]) << shift;
        mask |= 255u << shift;
        rank = bc[1];
    }
    T = prefix;
    need = rank;
}

// Exclusive prefix over the warps (in order) of one value per warp, and the
// total; every lane of a warp gets its warp's prefix.
__device__ __forceinline__ int2 warp_prefix(const BlockOps &ops, int v, int lane)
{
    const int2 r = ops.scan(lane == 0 ? v : 0);
    return make_int2(__shfl_sync(0xffffffffu, r.x, 0), r.y);
}

// Copies K and V rows of the slots [0, kept) from the prompt rows named by
// pos; each warp moves four rows per step (all loads, then all stores).
__device__ void copy_kept_rows(const void *K, const void *V, void *kc, void *vc, const int32_t *pos, size_t unit,
                               int P, int C, int row_bytes, int kept, int warp, int lane)
{
    constexpr int kRows = 4;
    const int vecs = row_bytes / 16;
    for (int s0 = warp * kRows; s0 < kept; s0 += kSelWarps * kRows) {
        for (int vi = lane; vi < 2 * vecs; vi += 32) {
            const int which = vi / vecs, off = vi - which * vecs;
            const uint8_t *src = static_cast<const uint8_t *>(which ? V : K);
            uint8_t *dst = static_cast<uint8_t *>(which ? vc : kc);
            uint4 v[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                if (s0 + r < kept)
                    v[r] = reinterpret_cast<const uint4 *>(src + (unit * P + pos[s0 + r]) * static_cast<size_t>(row_bytes))[off];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
                if (s0 + r < kept)
                    reinterpret_cast<uint4 *>(dst + (unit * C + s0 + r) * static_cast<size_t>(row_bytes))[off] = v[r];
        }
    }
}

// Keeps the first n_sink and last n_recent positions and, of the others, all
// but the P - K smallest (score, position) keys; the kept tokens fill slots
// 0, 1, ... in ascending position order. One CTA per unit: the unit's score
// bits (non-negative floats, so their bit patterns order like the values) in
// shared memory; the cut threshold by radix selection on the bit pattern;
// ties at the threshold go in position order, oldest first.
__global__ void __launch_bounds__(kSelThreads) prompt_select_kernel(const PromptSelectParams p)
{
    extern __shared__ uint32_t sbits[];
    __shared__ int red[kSelWarps];
    __shared__ int total;
    __shared__ int hist[256];
    __shared__ int bc[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const BlockOps ops{red, &total, lane, warp};
    const size_t unit = blockIdx.x;
    const int P = p.P;
    const int e_lo = p.n_sink, e_hi = P - p.n_recent;  // eligible positions [e_lo, e_hi)
    for (int j = tid; j < P; j += kSelThreads) {
        const float sv = p.score[unit * P + j];
        if (!(sv >= 0.f && sv <= FLT_MAX)) atomicOr(p.err, KVEVICT_DEV_NONFINITE);
        sbits[j] = __float_as_uint(sv);
    }
    __syncthreads();

    const int E = P > p.budget ? P - p.budget : 0;  // tokens to remove
    uint32_t T = 0;
    int need = 0;
    if (E > 0) radix_threshold(sbits, e_lo, e_hi, E, hist, bc, T, need);

    // leaves: eligible and (below T, or among the first `need` ties in position order)
    const WarpRange R(0, P, warp);
    auto walk = [&](int tie_base, int slot_base, bool write) {  // returns (ties, kept) of this warp
        int ties = 0, kept = 0;
        for (int j0 = R.base; j0 < R.end; j0 += 32) {
            const int j = j0 + lane;
            const bool in = j < R.end;
            const bool elig = in && j >= e_lo && j < e_hi;
            const uint32_t bt = in ? sbits[j] : 0u;
            const bool tie = E > 0 && elig && bt == T;
            const unsigned tm = __ballot_sync(0xffffffffu, tie);
            const bool leave = E > 0 && elig && (bt < T || (tie && tie_base + ties + __popc(tm & lanes_below(lane)) < need));
            const bool keep = in && !leave;
            const unsigned km = __ballot_sync(0xffffffffu, keep);
            if (write && keep) {
                const int slot = slot_base + kept + __popc(km & lanes_below(lane));
                if (slot < p.C) {
                    p.pos[unit * p.cstride + slot] = j;
                    p.cscore[unit * p.cstride + slot] = __uint_as_float(bt);
                }
            }
            ties += __popc(tm);
            kept += __popc(km);
        }
        return make_int2(ties, kept);
    };
    int ties = 0;
    for (int j0 = R.base; j0 < R.end; j0 += 32) {
        const int j = j0 + lane;
        ties += __popc(__ballot_sync(0xffffffffu, E > 0 && j < R.end && j >= e_lo && j < e_hi && sbits[j] == T));
    }
    const int tie_base = warp_prefix(ops, ties, lane).x;
    const int2 kb = warp_prefix(ops, walk(tie_base, 0, false).y, lane);
    walk(tie_base, kb.x, true);
    __syncthreads();  // the positions written above are visible to the whole CTA
    copy_kept_rows(p.K, p.V, p.kc, p.vc, p.pos + unit * p.cstride, unit, P, p.C, p.row_bytes, min(kb.y, p.C),
                   warp, lane);
}

// SnapKV ("Attention Sinks 与 KV Cache 淘汰策略" section 4.3): for each query
// head g of the unit's KV head, the votes of the prefix [0, P - window) are
// max-pooled over 7 positions (within the prefix) and the head keeps its topk
// largest pooled votes (ties: the newer position); the unit keeps the union
// over its G query heads plus the window, in slots 0, 1, ... in ascending
// position order, each token with the mean over g of its votes. One CTA per
// unit: a head's pooled bits and the kept bitmap in shared memory; each head's
// cut by radix selection, its ties in position order through one scan over
// the warps' spans.
__device__ void snap_union_tail(const SnapSelectParams &p, const uint32_t *keep, const BlockOps &ops, size_t unit,
                                int b, int kvh);

__global__ void __launch_bounds__(kSelThreads) snapkv_select_kernel(const SnapSelectParams p)
{
    extern __shared__ uint32_t ssm[];
    const int P = p.P, n_pre = P - p.window;
    uint32_t *pbits = ssm;               // [n_pre]
    uint32_t *keep = ssm + n_pre;        // [ceil(P / 32)] bitmap
    __shared__ int red[kSelWarps];
    __shared__ int total;
    __shared__ int hist[256];
    __shared__ int bc[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const BlockOps ops{red, &total, lane, warp};
    const size_t unit = blockIdx.x;
    const int b = static_cast<int>(unit) / p.Hkv, kvh = static_cast<int>(unit) - b * p.Hkv;
    const int nw = (P + 31) / 32;
    for (int i = tid; i < nw; i += kSelThreads) keep[i] = 0u;
    __syncthreads();
    for (int j = n_pre + tid; j < P; j += kSelThreads) atomicOr(&keep[j >> 5], 1u << (j & 31));  // the window

    const int take = min(p.topk, n_pre);
    const int E = n_pre - take;  // prefix positions a head does not take
    const WarpRange R(0, n_pre, warp);
    for (int g = 0; g < p.G; ++g) {
        const float *vg = p.votes + static_cast<size_t>(b * p.Hq + kvh * p.G + g) * P;
        __syncthreads();  // the previous head is done with pbits
        for (int j = tid; j < n_pre; j += kSelThreads) {
            float mx = vg[j];
            for (int jj = max(0, j - 3); jj <= min(n_pre - 1, j + 3); ++jj) mx = fmaxf(mx, vg[jj]);
            if (!(mx >= 0.f && mx <= FLT_MAX)) atomicOr(p.err, KVEVICT_DEV_NONFINITE);
            pbits[j] = __float_as_uint(mx);
        }
        __syncthreads();
        if (take == 0) continue;
        uint32_t T = 0;
        int need = 0;
        if (E > 0) radix_threshold(pbits, 0, n_pre, E, hist, bc, T, need);
        // taken: not among the E smallest (bits, position); a warp's span starts on a
        // multiple of 32, so each step of its walk fills one bitmap word
        int ties = 0;
        for (int j0 = R.base; j0 < R.end; j0 += 32) {
            const int j = j0 + lane;
            ties += __popc(__ballot_sync(0xffffffffu, E > 0 && j < R.end && pbits[j] == T));
        }
        int tb = warp_prefix(ops, ties, lane).x;
        for (int j0 = R.base; j0 < R.end; j0 += 32) {
            const int j = j0 + lane;
            const bool in = j < R.end;
            const uint32_t bt = in ? pbits[j] : 0u;
            const bool tie = E > 0 && in && bt == T;
            const unsigned tm = __ballot_sync(0xffffffffu, tie);
            const bool left = E > 0 && in && (bt < T || (tie && tb + __popc(tm & lanes_below(lane)) < need));
            const unsigned km = __ballot_sync(0xffffffffu, in && !left);
            if (lane == 0 && km) keep[j0 >> 5] |= km;
            tb += __popc(tm);
        }
    }
    __syncthreads();
    snap_union_tail(p, keep, ops, unit, b, kvh);
}

// The union's tail, shared by both selection kernels: the kept positions (the
// bitmap) in ascending order fill slots 0, 1, ..., each with the mean over
// its G heads of its votes; then the K/V rows are copied.
__device__ void snap_union_tail(const SnapSelectParams &p, const uint32_t *keep, const BlockOps &ops, size_t unit,
                                int b, int kvh)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = p.P, nw = (P + 31) / 32;
    // slots: the kept positions in ascending order, one bitmap word per lane and step
    const WarpRange RW(0, nw, warp);
    int cnt = 0;
    for (int w0 = RW.base; w0 < RW.end; w0 += 32) {
        const int w = w0 + lane;
        cnt += __reduce_add_sync(0xffffffffu, w < RW.end ? __popc(keep[w]) : 0);
    }
    const int2 sb = warp_prefix(ops, cnt, lane);
    int slot_base = sb.x;
    for (int w0 = RW.base; w0 < RW.end; w0 += 32) {
        const int w = w0 + lane;
        uint32_t word = w < RW.end ? keep[w] : 0u;
        const int c = __popc(word);
        const int incl = warp_incl_scan(c, lane);
        int slot = slot_base + incl - c;
        while (word) {
            const int j = w * 32 + __ffs(word) - 1;
            word &= word - 1u;
            if (slot < p.C) {
                float sc = 0.f;
                for (int g = 0; g < p.G; ++g) sc += p.votes[static_cast<size_t>(b * p.Hq + kvh * p.G + g) * P + j];
                p.pos[unit * p.cstride + slot] = j;
                p.cscore[unit * p.cstride + slot] = sc * (1.f / p.G);
            }
            ++slot;
        }
        slot_base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (sb.y > p.C && tid == 0) atomicOr(p.err, KVEVICT_DEV_BAD_SLOT);
    __syncthreads();
    copy_kept_rows(p.K, p.V, p.kc, p.vc, p.pos + unit * p.cstride, unit, P, p.C, p.row_bytes, min(sb.y, p.C),
                   warp, lane);
}

// The same selection with a head's pooled votes in registers: warp w owns the
// prefix positions [32 R w, 32 R (w + 1)), its lane l the positions
// 32 R w + 32 r + l (r < R). The pooling loads every vote once, with three
// halo values on each side of the warp's span, and builds the 7-wide max by
// doubling: m1(s) = max x[s, s+1], m2(s) = max m1(s), m1(s+2) = max x[s, s+3],
// then max m2(s-3), m2(s) = max x[s-3, s+3]; each shifted read takes the value
// from the lanes and registers around it (two shuffles). The cut threshold is
// a binary search on the bit pattern (the E-th smallest), each step counting
// with per-thread compares, a warp reduction, one barrier and a reduction of
// the warps' counts (double-buffered by step parity). For n_pre <= 512 R.
template <int R>
__global__ void __launch_bounds__(kSelThreads) snapkv_select_reg_kernel(const SnapSelectParams p)
{
    extern __shared__ uint32_t keep[];  // [ceil(P / 32)] bitmap
    __shared__ int red[kSelWarps];
    __shared__ int total;
    __shared__ int wcnt[2][kSelWarps];
    __shared__ uint32_t wlim[2][kSelWarps];
    __shared__ uint32_t cand[kSelCand];  // the patterns inside the search interval, once few enough
    __shared__ int ncand_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const BlockOps ops{red, &total, lane, warp};
    const size_t unit = blockIdx.x;
    const int P = p.P, n_pre = P - p.window;
    const int b = static_cast<int>(unit) / p.Hkv, kvh = static_cast<int>(unit) - b * p.Hkv;
    const int nw = (P + 31) / 32;
    for (int i = tid; i < nw; i += kSelThreads) keep[i] = 0u;
    __syncthreads();
    for (int j = n_pre + tid; j < P; j += kSelThreads) atomicOr(&keep[j >> 5], 1u << (j & 31));  // the window

    const int take = min(p.topk, n_pre);
    const int E = n_pre - take;
    const int base = warp * 32 * R + lane;
    constexpr uint32_t kNone = 0xFFFFFFFFu;  // past the prefix: above every finite pattern, never counted
    for (int g = 0; g < p.G && take > 0; ++g) {
        const float *vg = p.votes + static_cast<size_t>(b * p.Hq + kvh * p.G + g) * P;
        // raw votes (0 outside the prefix: neutral for the max of non-negative
        // values); x holds them, then m1, then m2
        float x[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int j = base + 32 * r;
            x[r] = j < n_pre ? __ldg(vg + j) : 0.f;
        }
        // lanes 0-2: the three positions before the span (hl) and after it (hr)
        const int span0 = base - lane;
        const int jl = span0 - 3 + lane, jr = span0 + 32 * R + lane;
        const float hl = (lane < 3 && jl >= 0 && jl < n_pre) ? __ldg(vg + jl) : 0.f;
        const float hr = (lane < 3 && jr < n_pre) ? __ldg(vg + jr) : 0.f;
        // span offsets s = 32 r + lane; the halos hold s = -3..-1 (left, lanes
        // 0-2) and s = 32 R.. (right, lanes 0-2 for x, 0-1 for m1)
        // m1 at s = -3..-1: x(s) and x(s + 1), the latter hl of the next lane or x(0)
        float m1l;
        {
            const float t = __shfl_sync(0xffffffffu, hl, (lane + 1) & 31);
            const float u = __shfl_sync(0xffffffffu, x[0], 0);
            m1l = fmaxf(hl, lane < 2 ? t : u);
        }
        const float m1r = fmaxf(hr, __shfl_sync(0xffffffffu, hr, (lane + 1) & 31));
        // m1 in place, ascending r (x[r + 1] is still raw when m1[r] reads it)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float same = __shfl_sync(0xffffffffu, x[r], (lane + 1) & 31);
            const float next = __shfl_sync(0xffffffffu, r + 1 < R ? x[r + 1 < R ? r + 1 : r] : hr, 0);
            x[r] = fmaxf(x[r], lane < 31 ? same : next);
        }
        // m2 at s = -3..-1: m1(s) and m1(s + 2), the latter m1l two lanes up or m1(lane - 1)
        float m2l;
        {
            const float t = __shfl_sync(0xffffffffu, m1l, (lane + 2) & 31);
            const float u = __shfl_sync(0xffffffffu, x[0], (lane - 1) & 31);
            m2l = fmaxf(m1l, lane == 0 ? t : u);
        }
        // m2 in place, ascending r
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float same = __shfl_sync(0xffffffffu, x[r], (lane + 2) & 31);
            const float next = __shfl_sync(0xffffffffu, r + 1 < R ? x[r + 1 < R ? r + 1 : r] : m1r, (lane - 30) & 31);
            x[r] = fmaxf(x[r], lane < 30 ? same : next);
        }
        // the pooled vote max(m2(s - 3), m2(s)) as a bit pattern
        uint32_t v[R];
        uint32_t lo = kNone, hi = 0;
        bool bad = false;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float same = __shfl_sync(0xffffffffu, x[r], (lane - 3) & 31);
            const float prev = r > 0 ? __shfl_sync(0xffffffffu, x[r > 0 ? r - 1 : 0], (lane + 29) & 31)
                                     : __shfl_sync(0xffffffffu, m2l, lane & 31);
            const float mx = fmaxf(x[r], lane >= 3 ? same : prev);
            const int j = base + 32 * r;
            v[r] = kNone;
            if (j < n_pre) {
                bad |= !(mx >= 0.f && mx <= FLT_MAX);
                v[r] = __float_as_uint(mx);
                lo = min(lo, v[r]);
                hi = max(hi, v[r]);
            }
        }
        if (bad) atomicOr(p.err, KVEVICT_DEV_NONFINITE);
        if (E == 0) {  // every prefix position is taken
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const unsigned km = __ballot_sync(0xffffffffu, v[r] != kNone);
                if (lane == 0 && km) atomicOr(&keep[(base - lane + 32 * r) >> 5], km);
            }
            continue;
        }
        // the search interval [a, bb] from the block's smallest and largest pattern
        lo = __reduce_min_sync(0xffffffffu, lo);
        hi = __reduce_max_sync(0xffffffffu, hi);
        if (lane == 0) {
            wlim[0][warp] = lo;
            wlim[1][warp] = hi;
        }
        if (tid == 0) ncand_s = 0;  // the previous head read it before its tie scan's barriers
        __syncthreads();
        static_assert(kSelWarps <= 32, "one warp reduces the per-warp values");
        uint32_t a = __reduce_min_sync(0xffffffffu, lane < kSelWarps ? wlim[0][lane] : kNone);
        uint32_t bb = __reduce_max_sync(0xffffffffu, lane < kSelWarps ? wlim[1][lane] : 0u);
        // smallest T in [a, bb] with #{v <= T} >= E. lt_a = #{v < a} and
        // le_bb = #{v <= bb} are exact (block-uniform); once [a, bb] holds at most
        // kSelCand patterns they are gathered into shared memory, and every later
        // step (its mid inside that interval) counts them plus the lt_a of the
        // gather, lt_g.
        int lt_a = 0, le_bb = n_pre, ncand = -1, lt_g = 0;  // ncand < 0: counting in registers
        for (int it = 0; a < bb; ++it) {
            const uint32_t mid = a + (bb - a) / 2;
            int cnt;
            if (ncand < 0) {
                int c0 = 0, c1 = 0;
#pragma unroll
                for (int r = 0; r < R; r += 2) {
                    c0 += v[r] <= mid;
                    if (r + 1 < R) c1 += v[r + 1] <= mid;
                }
                cnt = c0 + c1;
            } else {
                cnt = 0;
                for (int i = tid; i < ncand; i += kSelThreads) cnt += cand[i] <= mid;
            }
            const int c = __reduce_add_sync(0xffffffffu, cnt);
            if (lane == 0) wcnt[it & 1][warp] = c;
            __syncthreads();
            const int tot = (ncand < 0 ? 0 : lt_g) +
                            __reduce_add_sync(0xffffffffu, lane < kSelWarps ? wcnt[it & 1][lane] : 0);
            if (tot >= E) {
                bb = mid;
                le_bb = tot;
            } else {
                a = mid + 1;
                lt_a = tot;
            }
            if (ncand < 0 && a < bb && le_bb - lt_a <= kSelCand) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (v[r] >= a && v[r] <= bb) {
                        const int k = atomicAdd(&ncand_s, 1);
                        if (k < kSelCand) cand[k] = v[r];
                    }
                }
                __syncthreads();
                ncand = min(ncand_s, kSelCand);
                lt_g = lt_a;
            }
        }
        const uint32_t T = a;
        // ties at T: the first `need` in position order leave, the newer ones are taken
        int below = 0, ties = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            below += v[r] < T;
            ties += v[r] == T;
        }
        below = __reduce_add_sync(0xffffffffu, below);
        ties = __reduce_add_sync(0xffffffffu, ties);
        const int2 bs = warp_prefix(ops, below, lane);  // (synchronises: wcnt of the search is free again)
        const int need = E - bs.y;
        int tb = warp_prefix(ops, ties, lane).x;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const bool tie = v[r] == T;
            const unsigned tm = __ballot_sync(0xffffffffu, tie);
            const bool left = v[r] < T || (tie && tb + __popc(tm & lanes_below(lane)) < need);
            const unsigned km = __ballot_sync(0xffffffffu, v[r] != kNone && !left);
            if (lane == 0 && km) atomicOr(&keep[(base - lane + 32 * r) >> 5], km);
            tb += __popc(tm);
        }
    }
    __syncthreads();
    snap_union_tail(p, keep, ops, unit, b, kvh);
}

template <int D, int MODE, bool STACK> cudaError_t launch_attn_t(const PromptAttnParams &p0, int B, cudaStream_t st)
{
    const int smem = PromptLayout<D>::kBytes;
    cudaError_t e =
        cudaFuncSetAttribute(prompt_attn_kernel<D, MODE, STACK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    PromptAttnParams p = p0;
    const int nT = (p.P + kPT - 1) / kPT;
    const int nLq = (p.G * p.q_stride + kPT - 1) / kPT;
    p.ntiles = STACK ? (MODE == kRowStats ? nLq : nT) : (MODE == kRowStats ? nT - p.q_lo / kPT : nT);
    p.nheads = STACK ? B * p.Hkv : (MODE == kRowStats ? B * p.Hq : B * p.Hkv);
    if (p.ntiles <= 0 || p.nheads <= 0) return cudaSuccess;
    // persistent: one CTA per SM (the shared memory admits one), at most one per item
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long items = static_cast<long long>(p.ntiles) * p.nheads;
    const int grid = static_cast<int>(std::min<long long>(items, std::max(sms, 1)));
    prompt_attn_kernel<D, MODE, STACK><<<grid, kPThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <int D, int MODE> cudaError_t launch_attn(const PromptAttnParams &p, int B, cudaStream_t st)
{
    return p.stacked ? launch_attn_t<D, MODE, true>(p, B, st) : launch_attn_t<D, MODE, false>(p, B, st);
}

}  // namespace

size_t prompt_attn_smem(int head_dim) { return head_dim == 64 ? PromptLayout<64>::kBytes : PromptLayout<128>::kBytes; }

cudaError_t launch_prompt_rowstats(const PromptAttnParams &p, int head_dim, int B, cudaStream_t st)
{
    return head_dim == 64 ? launch_attn<64, kRowStats>(p, B, st) : launch_attn<128, kRowStats>(p, B, st);
}

cudaError_t launch_prompt_colsum(const PromptAttnParams &p, int head_dim, int B, cudaStream_t st)
{
    return head_dim == 64 ? launch_attn<64, kColSum>(p, B, st) : launch_attn<128, kColSum>(p, B, st);
}

cudaError_t launch_snapkv_votes(const SnapVotesParams &p, int head_dim, int sms, cudaStream_t st)
{
    if (p.Lq < 32 || p.Lq > kSnapVotesMaxRows || p.Lq % 32 || p.w % 32) return cudaErrorInvalidValue;
    const long long items = static_cast<long long>(p.units) * ((p.P + kPT - 1) / kPT);
    const int grid = static_cast<int>(std::min<long long>(sms, items));
    if (grid <= 0) return cudaSuccess;
    auto go = [&](auto kern, int smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kPThreads, smem, st>>>(p);
        return cudaGetLastError();
    };
    return head_dim == 64 ? go(snap_votes_kernel<64>, VotesLayout<64>::kBytes)
                          : go(snap_votes_kernel<128>, VotesLayout<128>::kBytes);
}

template <int R> cudaError_t launch_select_reg(const SnapSelectParams &p, int units, cudaStream_t st)
{
    const size_t smem = static_cast<size_t>((p.P + 31) / 32) * 4;
    cudaError_t e = cudaFuncSetAttribute(snapkv_select_reg_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    snapkv_select_reg_kernel<R><<<units, kSelThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_snapkv_select(const SnapSelectParams &p, int units, cudaStream_t st)
{
    const int n_pre = p.P - p.window;
    if (n_pre <= kSelThreads * 4) return launch_select_reg<4>(p, units, st);
    if (n_pre <= kSelThreads * 16) return launch_select_reg<16>(p, units, st);
    if (n_pre <= kSelThreads * 64) return launch_select_reg<64>(p, units, st);
    const size_t smem = static_cast<size_t>(p.P - p.window) * 4 + static_cast<size_t>((p.P + 31) / 32) * 4;
    cudaError_t e = cudaFuncSetAttribute(snapkv_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    snapkv_select_kernel<<<units, kSelThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prompt_select(const PromptSelectParams &p, int units, cudaStream_t st)
{
    const size_t smem = static_cast<size_t>(p.P) * 4;
    cudaError_t e = cudaFuncSetAttribute(prompt_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    prompt_select_kernel<<<units, kSelThreads, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace kvevict
