// prompt_attn.h -- host-visible parameters of the prompt-scoring kernels
// (Q-seeded prefill): causal attention statistics of the prompt on the
// tcgen05 tensor cores, then the cut to the budget.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace kvevict {

constexpr int kPromptTile = 128;          // query / key rows per MMA tile (M and N)
constexpr int kPromptMaxLen = 49152;      // selection keeps one unit's score bits in shared memory

// Opaque 128-byte tensor map (CUtensorMap), 64-byte aligned as a kernel
// parameter requires.
struct alignas(64) PromptTmap {
    uint64_t word[16];
};

struct PromptAttnParams {
    PromptTmap tma, tmb;  // A-side rows (the tile a CTA keeps) and B-side rows (the tiles it streams)
    float *stats;         // [B * Hq][Ps]: per query row i >= qs0 (q_lo rounded down to a tile),
                          // -(m + log2(l)) of its softmax (log2 units), at index i - qs0
    float *score;         // per key, the mass it receives from the queries i >= q_lo:
                          // [B * Hkv][P], mean over the G query heads, or, with per_head,
                          // [B * Hq][P], one row per query head
    int P, Ps, G, Hq, Hkv;
    int q_lo;             // first query that takes part
    int q_stride;         // rows per query head in the Q tensor
    int q_first;          // query index of each head's first Q row (queries before it are not given)
    int per_head;
    int stacked;          // SnapKV with a window of a multiple of 32: the G heads' window rows stacked
                          // (row g * q_stride + t); stats then [B * Hkv][Ps] over the stacked rows
    float scale_log2;     // log2(e) / sqrt(d)
    uint32_t *err;
    int ntiles, nheads;   // set by the launcher: the items (tile, head) of the persistent grid
    int *work;            // the launch's work counter (zero before it; the CTAs take items from it)
};

struct PromptSelectParams {
    const float *score;   // [B * Hkv][P]
    const void *K, *V;    // prompt [B][Hkv][P][d]
    void *kc, *vc;        // layer cache [B][Hkv][C][d]
    int32_t *pos;         // layer [B][Hkv][cstride]
    float *cscore;        // layer [B][Hkv][cstride]
    int P, C, cstride, row_bytes;
    int budget, n_sink, n_recent;
    uint32_t *err;
};

struct SnapSelectParams {
    const float *votes;   // [B * Hq][P]: per query head, the window's softmax mass on every key
    const void *K, *V;    // prompt [B][Hkv][P][d]
    void *kc, *vc;        // layer cache [B][Hkv][C][d]
    int32_t *pos;         // layer [B][Hkv][cstride]
    float *cscore;        // layer [B][Hkv][cstride]
    int P, C, cstride, row_bytes;
    int G, Hq, Hkv, window, topk;
    uint32_t *err;
};

// SnapKV votes, streamed: one persistent CTA per SM walks a contiguous range of
// (unit, 128-key tile) items. The unit's stacked window queries (Lq = G * w
// rows, a multiple of 32, at most 256) stay in shared memory as the MMA's B
// operand; key tiles stream through a TMA ring as A.
struct SnapVotesParams {
    PromptTmap tmk;       // prompt K, rows [B * Hkv * P], boxes of 128 rows x 64
    PromptTmap tmq;       // window queries, rows [B * Hq * w] (a unit's Lq rows are contiguous), boxes of Lq rows x 64
    const float *stats;   // [B * Hkv][Ps]: minus the log2 normaliser of each stacked window row
    float *votes;         // [B * Hq][P]
    int P, Ps, w, G, Hq, Hkv, Lq;
    int units;
    float scale_log2;
    uint32_t *err;
};
constexpr int kSnapVotesMaxRows = 256;  // Lq limit of the streamed votes kernel (one MMA's N)

// Bytes of shared memory the scoring kernels use for head_dim d.
size_t prompt_attn_smem(int head_dim);
// Pass 1 (row statistics) and pass 2 (column sums); d in {64, 128}.
cudaError_t launch_prompt_rowstats(const PromptAttnParams &p, int head_dim, int B, cudaStream_t st);
cudaError_t launch_prompt_colsum(const PromptAttnParams &p, int head_dim, int B, cudaStream_t st);
// SnapKV votes with the stacked window resident (Lq <= kSnapVotesMaxRows); `sms` CTAs.
cudaError_t launch_snapkv_votes(const SnapVotesParams &p, int head_dim, int sms, cudaStream_t st);
// The cut to the budget and the copy of the kept rows into the cache.
cudaError_t launch_prompt_select(const PromptSelectParams &p, int units, cudaStream_t st);
// SnapKV: pooling, per-head top-k, the union with the window, the copy.
cudaError_t launch_snapkv_select(const SnapSelectParams &p, int units, cudaStream_t st);

}  // namespace kvevict
