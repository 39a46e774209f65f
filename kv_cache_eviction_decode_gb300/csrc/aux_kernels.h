// aux_kernels.h -- host-visible parameters of the prefill and Random-cut kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace kvevict {

constexpr int kCutThreads = 512;
constexpr int kMaxRandomCandidates = 8192;  // K + r, sorted in shared memory

struct PrefillParams {
    const void *K, *V;  // [B][Hkv][n_tok][D]
    void *kc, *vc;      // layer cache [B][Hkv][C][D]
    int32_t *pos;
    void *score;        // fp32, binary16 (score_half) or 8-bit codes (score_int8), or null
    int score_half;
    int score_int8;
    int n_tok, p0, C, cstride, Hkv, head_dim, elem_bytes;
    int n_sink, ring_len;  // ring_len = C - n_sink for ring policies, 0 for Random
    int a0, a1, b0, b1;    // chunk rows to copy
    uint8_t *pool;         // two-pool H2O: pool flags [B][Hkv][pstride], else null
    int pstride, hh_below; // positions below hh_below go to the heavy-hitter pool
};

struct CutParams {
    int32_t *pos;       // layer [B][Hkv][cstride]
    int32_t *freelist;  // layer [B][Hkv][r]
    void *kc, *vc;      // layer cache [B][Hkv][C][D]: freed rows are zeroed
    int row_bytes;
    uint64_t seed;
    int layer, step, Hkv, C, cstride;
    int first_slot, n_cand, n_pow2, r;
};

// Block-granular H2O prefill: the slot-centric closed form of admitting the
// prompt one token at a time with score 0 (see prefill_block_kernel).
struct BlockPrefillParams {
    const void *K, *V;  // [B][Hkv][n_tok][D]
    void *kc, *vc;      // layer cache [B][Hkv][C][D]
    int32_t *pos;       // [B][Hkv][cstride]
    float *score;
    int n_tok, C, cstride, Hkv, row_bytes;
    int bs, nsb;        // block size, blocks holding sinks
};

// Block-granular H2O release: frees one block per unit and lists its slots.
struct BlockReleaseParams {
    int32_t *pos;       // layer [B][Hkv][cstride]
    float *score;
    int32_t *freelist;  // layer [B][Hkv][bs]
    void *kc, *vc;      // layer cache [B][Hkv][C][D]: freed rows are zeroed
    int row_bytes, C, cstride, bs;
    int n_sink, n_recent, p;  // p: position of the token the release makes room for
    double *ledger;     // layer [B][Hkv]: evicted score mass, the released block's added
    uint32_t *err;
};

// Validation mode: the near-ties of one H2O decode step's eviction decisions.
struct TieAuditParams {
    const int32_t *pos;          // layer [B][Hkv][cstride], after the step
    const void *score;           // layer scores after the step: fp32, binary16 or 8-bit codes
    const float *qscale;         // score_int8: layer [B][Hkv] scales after the step
    const int32_t *trace;        // [B][Hkv][4] the step's records: slot, evicted position, evicted score bits, ...
    unsigned long long *count;   // this layer's count of near-ties
    int score_half, score_int8;
    int n_active, cstride, p, n_sink, n_recent;
    float rel;                   // relative gap below which two scores are a near-tie
};

void launch_prefill(const PrefillParams &p, int rows, int B, cudaStream_t st);
// binary16 scores [units][cstride] -> fp32 [units][C]
cudaError_t launch_scores_to_f32(float *dst, const void *src, int C, int cstride, size_t units, cudaStream_t st);
// One thread's bounded wait on an mbarrier nothing completes: records
// KVEVICT_DEV_WAIT_TIMEOUT in err after the wait limit.
cudaError_t launch_wait_timeout_probe(uint32_t *err, cudaStream_t st);
// INT8 score storage read back as fp32: code * the unit's scale.
cudaError_t launch_scores_int8_to_f32(float *dst, const void *src, const float *scale, int C, int cstride,
                                      size_t units, cudaStream_t st);
void launch_block_prefill(const BlockPrefillParams &p, int B, cudaStream_t st);
cudaError_t launch_block_release(const BlockReleaseParams &p, int units, cudaStream_t st);
size_t cut_smem_bytes(int n_pow2, int r);
cudaError_t launch_random_cut(const CutParams &p, int B, cudaStream_t st);
cudaError_t launch_tie_audit(const TieAuditParams &p, int units, cudaStream_t st);

}  // namespace kvevict
