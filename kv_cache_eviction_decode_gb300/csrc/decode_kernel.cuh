// decode_kernel.cuh -- the fused decode step over a budget-bounded KV cache.
//
// One launch per layer-step. Grid (split, Hkv, B): the `split` CTAs of one
// thread-block cluster share one (sequence, KV head) unit and divide its
// occupied slots into contiguous ranges of 32-slot tiles. Per CTA:
//
//   producer warp   one elected lane streams the CTA's K tiles, then its V
//                   tiles, global -> shared with bulk (TMA) copies into a
//                   ring of stages, each completing on a full-mbarrier; the
//                   consumers free a stage through its empty-mbarrier.
//   K phase         each consumer warp takes whole K tiles and forms the
//                   logits z = q.k / sqrt(d) of the G query heads for the 32
//                   slots: every lane holds d/32 coordinates of q and of each
//                   key, and a 31-shuffle butterfly transposes the partial
//                   sums so lane i ends with one (head, slot) logit. The
//                   logits stay in shared memory (the score pass needs them).
//   V phase         with the CTA-local max m_c known, p = 2^(z - m_c) is
//                   written back over z and o += p v is accumulated.
//   combine         (m_c, l_c, o_c) of every CTA in the cluster are read
//                   through distributed shared memory; each CTA writes its
//                   share of out = sum_c o_c 2^(m_c - m) / l.
//   scores (H2O)    every retained slot's cumulative score grows by
//                   (1/G) sum_g p_g 2^(m_c - m) / l; the eligible slot with the
//                   smallest (score, position) is the CTA's candidate, and a
//                   second cluster exchange picks the victim.
//   insert          the new token's K/V, position and score are written in
//                   place into the victim's slot (H2O), the closed-form ring
//                   slot (StreamingLLM), the next empty slot, or the next
//                   entry of the unit's free list (Random after a cut).
//
// Method (page title and section): attention over the retained cache then
// cumulative-score update then eviction, "KV Cache 驱逐策略：从 LRU 到 H2O"
// flowchart and "Attention Sinks 与 KV Cache 淘汰策略" section 4.2 loop;
// greedy removal of the lowest-score candidate, "h2o: heavy-hitter oracle"
// summary, Algorithm 1; sink + ring window, same page section 4.1; GQA score =
// mean over the query heads of one KV head.
#pragma once

#include <cfloat>
#include <cmath>

#include "device_common.cuh"

namespace kvevict {

constexpr int kTile = 32;           // slots per pipeline stage
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kMaxSplit = 16;

enum InsertMode : int {
    kInsertAt = 0,     // the host gives the slot (empty slot, or the ring slot)
    kH2OEvict = 1,     // cache full: evict the lowest-score eligible token
    kFromFreeList = 2  // Random after a cut: next entry of the unit's free list
};

struct DecodeParams {
    const void *q;       // [B][Hkv*G][D]
    const void *k_new;   // [B][Hkv][D]
    const void *v_new;   // [B][Hkv][D]
    void *out;           // [B][Hkv*G][D]
    void *kc, *vc;       // this layer's cache, [B][Hkv][C][D]
    int32_t *pos;        // [B][Hkv][C]
    float *score;        // [B][Hkv][C], or null when the policy keeps no scores
    const int32_t *freelist;  // [B][Hkv][freelist_len]
    int32_t *trace;      // [B][Hkv][4] or null: slot, evicted position, evicted score, new score
    uint32_t *err;
    int Hkv, C;
    int n_active;        // slots [0, n_active) may hold tokens
    int p;               // position of the new token
    int mode, dest_slot, freelist_idx, freelist_len;
    int n_sink, n_recent;
    int split;           // CTAs per unit (cluster size)
    int zcap;            // per-head stride of the logit buffer
    float scale_log2;    // log2(e) / sqrt(D)
};

// Shared-memory layout, shared by host (size) and device (offsets).
template <typename T, int D, int G> struct DecodeLayout {
    static constexpr int kEPL = D / 32;  // key/value coordinates per lane
    static constexpr int kR = 32 / G;    // slots per butterfly chunk
    static constexpr int kStageBytes = kTile * D * static_cast<int>(sizeof(T));
    static constexpr int kStages = (65536 / kStageBytes) < 4 ? 4 : (65536 / kStageBytes);
    static constexpr int kStageArea = kStages * kStageBytes;
    static_assert(kConsumerWarps * G * D * 4 <= kStageArea, "partial outputs must fit the stage area");
    static_assert(G >= 1 && G <= 8 && (G & (G - 1)) == 0, "G in {1,2,4,8}");

    struct Misc {
        uint64_t full[kStages];
        uint64_t empty[kStages];
        float wmax[kConsumerWarps][G];
        float wsum[kConsumerWarps][G];
        float m[G];        // this CTA's max logit per head (log2 units)
        float l[G];        // this CTA's softmax denominator relative to m
        float o[G][D];     // this CTA's unnormalised output relative to m
        float znew[G];     // the new token's logits (rank 0)
        float pnew[G];     // 2^(znew - m) (rank 0)
        float fac[kMaxSplit][G];  // 2^(m_c - m_global) / l_global per CTA c
        float anew;        // the new token's score (rank 0)
        int dest;
        uint64_t best_key;
        int32_t best_slot;
        uint64_t wkey[kConsumerWarps + 1];
        int32_t wslot[kConsumerWarps + 1];
    };

    // zcap = C-per-CTA rounded to whole tiles; for G > 1 padded so that
    // zcap == R (mod 32): the G lanes groups then hit distinct banks.
    __host__ __device__ static int zcap(int max_slots_per_cta)
    {
        int z = ((max_slots_per_cta + kTile - 1) / kTile) * kTile;
        return G > 1 ? z + kR : z;
    }
    __host__ __device__ static size_t off_z() { return kStageArea; }
    __host__ __device__ static size_t off_misc(int zc)
    {
        return kStageArea + ((static_cast<size_t>(G) * zc * 4 + 127) / 128) * 128;
    }
    __host__ __device__ static size_t bytes(int zc) { return off_misc(zc) + sizeof(Misc); }
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

template <typename T, int D, int G, bool HOLES>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ DecodeParams P)
{
    using L = DecodeLayout<T, D, G>;
    constexpr int EPL = L::kEPL, R = L::kR, NST = L::kStages;
    using E = Elem<T>;

    extern __shared__ __align__(128) uint8_t smem[];
    T *stage = reinterpret_cast<T *>(smem);
    const int zc = P.zcap;
    float *zbuf = reinterpret_cast<float *>(smem + L::off_z());
    auto &M = *reinterpret_cast<typename L::Misc *>(smem + L::off_misc(zc));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_rank());
    const int S = P.split;
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t unit = static_cast<size_t>(b) * P.Hkv + h;
    const size_t C = static_cast<size_t>(P.C);

    // This CTA's contiguous range of whole tiles among the occupied slots.
    const int nt_all = (P.n_active + kTile - 1) / kTile;
    const int t_lo = static_cast<int>(static_cast<long long>(rank) * nt_all / S);
    const int t_hi = static_cast<int>(static_cast<long long>(rank + 1) * nt_all / S);
    const int nt = t_hi - t_lo;
    const int s_lo = t_lo * kTile;
    const int s_hi = min(t_hi * kTile, P.n_active);
    const int n_mine = max(0, s_hi - s_lo);

    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&M.full[i], 1);
            mbar_init(&M.empty[i], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();

    // Everything below reads memory the previous launch on the stream may
    // have written.
    grid_dependency_wait();
    grid_launch_dependents();

    const T *kbase = static_cast<const T *>(P.kc) + unit * C * D;
    const T *vbase = static_cast<const T *>(P.vc) + unit * C * D;
    const int g_lane = lane / R;  // the head this lane's logits belong to

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int issued = 0;
            for (int s = 0; s < 2 * nt; ++s) {
                const int st = s % NST, round = s / NST;
                if (round > 0 && !mbar_wait(&M.empty[st], (round - 1) & 1)) {
                    atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
                    break;
                }
                const int tile = s < nt ? s : s - nt;
                const int slot0 = s_lo + tile * kTile;
                const int rows = min(kTile, s_hi - slot0);
                const uint32_t bytes = static_cast<uint32_t>(rows * D * sizeof(T));
                const T *src = (s < nt ? kbase : vbase) + static_cast<size_t>(slot0) * D;
                mbar_arrive_expect_tx(&M.full[st], bytes);
                bulk_g2s_stream(stage + static_cast<size_t>(st) * kTile * D, src, bytes, &M.full[st], pol);
                issued = s + 1;
            }
            // No copy may still be landing in shared memory when the CTA
            // leaves: wait for the last stages issued (earlier ones were
            // consumed before their stage was reused).
            for (int s = max(0, issued - NST); s < issued; ++s)
                if (!mbar_wait(&M.full[s % NST], (s / NST) & 1)) atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------ consumers
        const T *qp = static_cast<const T *>(P.q) + unit * G * D;
        float qf[G][EPL];
#pragma unroll
        for (int g = 0; g < G; ++g) load_f32<T, EPL>(qp + g * D + lane * EPL, qf[g]);

        if (rank == 0 && warp == 0) {  // the new token's logits
            float kf[EPL];
            load_f32<T, EPL>(static_cast<const T *>(P.k_new) + unit * D + lane * EPL, kf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float s = warp_sum(dot_n(qf[g], kf));
                if (lane == 0) M.znew[g] = s * P.scale_log2;
            }
        }

        // K phase: logits of this CTA's slots, kept in shared memory.
        float mx = -INFINITY;
        bool ok = true;
        for (int s = warp; s < nt; s += kConsumerWarps) {
            const int st = s % NST;
            if (!mbar_wait(&M.full[st], (s / NST) & 1)) {
                atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
                ok = false;
                break;
            }
            const T *tk = stage + static_cast<size_t>(st) * kTile * D;
            const int base = s * kTile;
            const int rows = min(kTile, n_mine - base);
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
                if (HOLES && valid) valid = P.pos[unit * C + s_lo + base + row] >= 0;
                const float z = valid ? sum * P.scale_log2 : -INFINITY;
                zbuf[g_lane * zc + base + row] = z;
                mx = fmaxf(mx, z);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&M.empty[st]);
        }
#pragma unroll
        for (int off = 1; off < R; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane % R == 0) M.wmax[warp][g_lane] = mx;
        named_sync(1, kConsumerThreads);
        if (warp == 0 && lane < G) {
            float m = -INFINITY;
            for (int w = 0; w < kConsumerWarps; ++w) m = fmaxf(m, M.wmax[w][lane]);
            if (rank == 0) m = fmaxf(m, M.znew[lane]);
            M.m[lane] = m;
        }
        named_sync(1, kConsumerThreads);
        const float m_mine = M.m[g_lane];

        // V phase.
        float acc[G][EPL];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
        float lsum = 0.f;
        if (rank == 0 && warp == 0) {
            float vf[EPL];
            load_f32<T, EPL>(static_cast<const T *>(P.v_new) + unit * D + lane * EPL, vf);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pn = exp2f(M.znew[g] - M.m[g]);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(pn, vf[e], acc[g][e]);
                if (lane == g * R) lsum += pn;
                if (lane == 0) M.pnew[g] = pn;
            }
        }
        const int first_v = nt + ((warp - nt % kConsumerWarps) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
        for (int s = first_v; ok && s < 2 * nt; s += kConsumerWarps) {
            const int st = s % NST;
            if (!mbar_wait(&M.full[st], (s / NST) & 1)) {
                atomicOr(P.err, KVEVICT_DEV_WAIT_TIMEOUT);
                break;
            }
            const int base = (s - nt) * kTile;
            const int rows = min(kTile, n_mine - base);
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
            const T *tv = stage + static_cast<size_t>(st) * kTile * D;
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
            __syncwarp();
            if (lane == 0) mbar_arrive(&M.empty[st]);
        }
#pragma unroll
        for (int off = 1; off < R; off <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        if (lane % R == 0) M.wsum[warp][g_lane] = lsum;

        // Reduce the consumer warps' partial outputs through the (now idle)
        // stage area.
        named_sync(1, kConsumerThreads);
        float *part = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EPL; ++e) part[(warp * G + g) * D + lane * EPL + e] = acc[g][e];
        named_sync(1, kConsumerThreads);
        for (int i = tid; i < G * D; i += kConsumerThreads) {
            float o = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) o += part[w * G * D + i];
            M.o[i / D][i % D] = o;
        }
        if (tid < G) {
            float l = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) l += M.wsum[w][tid];
            M.l[tid] = l;
        }
    }
    __syncthreads();
    cluster_sync();  // (1) every CTA's (m, l, o) is ready

    // ---------------------------------------------------------------- combine
    if (tid < G) {
        float mg = -INFINITY;
        for (int c = 0; c < S; ++c) mg = fmaxf(mg, ld_peer_f32(peer_addr(&M.m[tid], c)));
        float lg = 0.f;
        for (int c = 0; c < S; ++c) {
            const float mc = ld_peer_f32(peer_addr(&M.m[tid], c));
            const float lc = ld_peer_f32(peer_addr(&M.l[tid], c));
            if (mc != -INFINITY) lg += lc * exp2f(mc - mg);
        }
        if (rank == 0 && !(lg > 0.f && lg <= FLT_MAX)) atomicOr(P.err, KVEVICT_DEV_NONFINITE);
        const float inv = 1.f / lg;
        for (int c = 0; c < S; ++c) {
            const float mc = ld_peer_f32(peer_addr(&M.m[tid], c));
            M.fac[c][tid] = (mc == -INFINITY) ? 0.f : exp2f(mc - mg) * inv;
        }
    }
    __syncthreads();
    {
        constexpr int GD = G * D;
        const int i0 = rank * GD / S, i1 = (rank + 1) * GD / S;
        T *outp = static_cast<T *>(P.out) + unit * GD;
        for (int i = i0 + tid; i < i1; i += kThreads) {
            const int g = i / D, e = i % D;
            float o = 0.f;
            for (int c = 0; c < S; ++c) o = fmaf(ld_peer_f32(peer_addr(&M.o[g][e], c)), M.fac[c][g], o);
            outp[i] = E::from_f32(o);
        }
    }

    // ------------------------------------------------ cumulative scores (H2O)
    if (P.score != nullptr) {
        float fself[G];
#pragma unroll
        for (int g = 0; g < G; ++g) fself[g] = M.fac[rank][g] * (1.0f / G);
        uint64_t best = ~0ull;
        int32_t bslot = -1;
        const bool evict = P.mode == kH2OEvict;
        for (int j = tid; j < n_mine; j += kThreads) {
            float a = 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) a = fmaf(zbuf[g * zc + j], fself[g], a);
            const size_t gi = unit * C + s_lo + j;
            const float sc = P.score[gi] + a;
            P.score[gi] = sc;
            if (evict) {
                const int ps = P.pos[gi];
                if (ps >= P.n_sink && ps <= P.p - P.n_recent) {
                    const uint64_t key = (static_cast<uint64_t>(__float_as_uint(sc)) << 32) | static_cast<uint32_t>(ps);
                    if (key < best) {
                        best = key;
                        bslot = s_lo + j;
                    }
                }
            }
        }
        if (rank == 0 && tid == 0) {
            float a = 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) a = fmaf(M.pnew[g], M.fac[0][g], a);
            M.anew = a * (1.0f / G);
        }
        if (evict) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const uint64_t ok = __shfl_xor_sync(0xffffffffu, best, off);
                const int32_t os = __shfl_xor_sync(0xffffffffu, bslot, off);
                if (ok < best) {
                    best = ok;
                    bslot = os;
                }
            }
            if (lane == 0) {
                M.wkey[warp] = best;
                M.wslot[warp] = bslot;
            }
            __syncthreads();
            if (tid == 0) {
                uint64_t k = ~0ull;
                int32_t sl = -1;
                for (int w = 0; w <= kConsumerWarps; ++w)
                    if (M.wkey[w] < k) {
                        k = M.wkey[w];
                        sl = M.wslot[w];
                    }
                M.best_key = k;
                M.best_slot = sl;
            }
        }
    }

    // ------------------------------------------------------------- insert
    int dest = -1;
    bool writer = false;
    if (P.mode == kH2OEvict) {
        cluster_sync();  // (2) every CTA's candidate is ready
        if (tid == 0) {
            uint64_t k = ~0ull;
            int32_t sl = -1;
            for (int c = 0; c < S; ++c) {
                const uint64_t kc = ld_peer_u64(peer_addr(&M.best_key, c));
                const int32_t sc = ld_peer_s32(peer_addr(&M.best_slot, c));
                if (kc < k) {
                    k = kc;
                    sl = sc;
                }
            }
            if (sl < 0 && rank == 0) atomicOr(P.err, KVEVICT_DEV_NO_CANDIDATE);
            M.dest = sl;
        }
        __syncthreads();
        dest = M.dest;
        writer = dest >= s_lo && dest < s_hi;  // the CTA that attended the victim
    } else {
        __syncthreads();
        dest = P.mode == kInsertAt ? P.dest_slot
                                   : P.freelist[unit * P.freelist_len + P.freelist_idx];
        writer = rank == 0;
        if (dest < 0 || dest >= P.C) {
            if (writer && tid == 0) atomicOr(P.err, KVEVICT_DEV_BAD_SLOT);
            dest = -1;
        }
    }
    if (writer && dest >= 0) {
        const T *kn = static_cast<const T *>(P.k_new) + unit * D;
        const T *vn = static_cast<const T *>(P.v_new) + unit * D;
        T *kd = static_cast<T *>(P.kc) + (unit * C + dest) * D;
        T *vd = static_cast<T *>(P.vc) + (unit * C + dest) * D;
        for (int i = tid; i < D; i += kThreads) {
            kd[i] = kn[i];
            vd[i] = vn[i];
        }
        if (tid == 0) {
            const int32_t old_pos = P.pos[unit * C + dest];
            const float old_score = P.score != nullptr ? P.score[unit * C + dest] : 0.f;
            const float an = P.score != nullptr ? ld_peer_f32(peer_addr(&M.anew, 0)) : 0.f;
            P.pos[unit * C + dest] = P.p;
            if (P.score != nullptr) P.score[unit * C + dest] = an;
            if (P.trace != nullptr)
                reinterpret_cast<int4 *>(P.trace)[unit] = make_int4(dest, old_pos, __float_as_int(old_score),
                                                                    __float_as_int(an));
        }
    }
    cluster_sync();  // (last) no CTA leaves while a peer may still read its shared memory
}

}  // namespace kvevict
