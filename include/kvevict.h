/*
 * kvevict.h -- C ABI of libkvevict.so: the decode step of attention over a
 * budget-bounded KV cache with eviction, on one NVIDIA GB300 (sm_103a).
 *
 * One handle holds the KV cache of a whole model for B sequences: for every
 * (layer, sequence, KV head) "unit" a fixed array of C slots, each slot
 * holding one retained token's key, value, position and (H2O only) its
 * cumulative attention score. A decode step for one layer does, for every
 * unit, in one launch:
 *   1. attention of the unit's G query heads over the retained tokens plus
 *      the new token (split over the CTAs of a thread-block cluster, softmax
 *      partials combined through distributed shared memory);
 *   2. H2O: each retained token's cumulative score grows by its normalised
 *      attention probability (mean over the G query heads); the new token
 *      starts with its own;
 *   3. the eviction decision (H2O: lowest score among non-sink tokens
 *      outside the recent window; StreamingLLM: the token leaving the ring
 *      window; Random Attention: a periodic uniform-random cut);
 *   4. the new token's key/value written in place into the freed slot.
 *
 * Sources (page title and section):
 *  - "KV Cache 驱逐策略：从 LRU 到 H2O" (wiblog.cn): cumulative attention
 *    score as the eviction signal, eviction only when the pool is full, the
 *    eviction flowchart.
 *  - "h2o: heavy-hitter oracle for efficient generative inference" summary
 *    (fmread.com): Algorithm 1 -- budget K, candidate set S_{i-1} + {i},
 *    remove the element whose removal keeps the highest cumulative score.
 *  - "Attention Sinks 与 KV Cache 淘汰策略" (10100.com): section 4.1
 *    (StreamingLLM: 4 sink tokens locked + rolling window, ring buffer),
 *    section 4.2 (H2O: sink + heavy hitters + recent window).
 *  - "Random Attention" summary (ai-feeds.com), 方法: keep the prompt; evict
 *    generated tokens uniformly at random, independently per head, with a
 *    periodic budget K and buffer r.
 *
 * Conventions for every call:
 *  - Returns KVEVICT_OK (0) or a negative kvevict_status. Argument and state
 *    errors are found on the host before anything is launched; the call then
 *    has no effect. Nothing in the device code traps: anomalies found on the
 *    GPU set bits of a device error word that kvevict_check() reads.
 *  - All work is queued asynchronously on the handle's CUDA stream; device
 *    pointers passed in must stay valid until the stream has passed the call.
 *  - Device tensors are dense, row-major, of the handle's dtype (fp32 or
 *    bf16), 16-byte aligned.
 *  - Calls are made with the handle's device current: the device that holds
 *    the state buffer given to kvevict_create (its stream belongs to it).
 *  - Not thread-safe: one host thread drives one handle at a time.
 */
#ifndef KVEVICT_H
#define KVEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVEVICT_API_VERSION 1

typedef struct kvevict_handle *kvevict_t;

typedef enum {
    KVEVICT_H2O = 0,          /* sink + heavy hitters + recent window */
    KVEVICT_SINK_WINDOW = 1,  /* StreamingLLM: sink + ring window, no scores */
    KVEVICT_RANDOM = 2,       /* Random Attention: prompt kept, periodic random cut */
    KVEVICT_H2O_BLOCK = 3,    /* H2O scores, whole blocks of r slots released at a time */
    KVEVICT_H2O_POOLS = 4     /* H2O scores, a recent pool and a heavy-hitter pool (hh_threshold) */
} kvevict_policy;

typedef enum { KVEVICT_F32 = 0, KVEVICT_BF16 = 1 } kvevict_dtype;

typedef enum {
    KVEVICT_OK = 0,
    KVEVICT_ERR_INVALID_ARG = -1, /* bad argument, shape, pointer or alignment */
    KVEVICT_ERR_CAPACITY = -2,    /* prompt beyond max_prompt (Random), state buffer too small */
    KVEVICT_ERR_STATE = -3,       /* call out of order (prefill after decode, layer out of range) */
    KVEVICT_ERR_CUDA = -4,        /* a CUDA runtime call failed */
    KVEVICT_ERR_DEVICE = -5       /* kvevict_check found device error bits */
} kvevict_status;

/* Bits of the device error word (kvevict_check). */
#define KVEVICT_DEV_NONFINITE 0x1u    /* a softmax denominator was not finite or not positive */
#define KVEVICT_DEV_NO_CANDIDATE 0x2u /* H2O found no evictable token; the new token was dropped */
#define KVEVICT_DEV_WAIT_TIMEOUT 0x4u /* a pipeline wait gave up after its time limit */
#define KVEVICT_DEV_BAD_SLOT 0x8u     /* a free-list entry was out of range; the new token was dropped */

/*
 * Whole configuration of a handle.
 *   policy, n_sink, n_heavy, n_recent, budget, r, seed: the eviction method.
 *     H2O:         budget K = n_sink + n_heavy + n_recent, n_recent >= 1; a
 *                  token at position j is a candidate at the step that
 *                  appends position p iff n_sink <= j <= p - n_recent.
 *     SINK_WINDOW: budget = n_sink + n_recent, n_heavy = 0, n_recent >= 1.
 *     RANDOM:      budget K = generated tokens kept after a cut, r >= 1 the
 *                  buffer/period, K + r <= 8192; n_sink = n_heavy =
 *                  n_recent = 0; seed keys the Philox4x64-10 draws.
 *     H2O_BLOCK:   as H2O, with r >= 1 the block size: the slots form blocks
 *                  of r consecutive slots, budget a multiple of r, and at
 *                  least one block besides those holding sinks lies outside
 *                  the recent window ((budget / r - ceil(n_sink / r) - 1) r
 *                  >= n_recent). When a token needs a slot and the cache is
 *                  full, the block wholly outside the sinks and the recent
 *                  window (n_sink <= pos <= p - n_recent) with the smallest
 *                  (sum of cumulative scores, oldest position) is released
 *                  before the token attends ("Attention Sinks 与 KV Cache 淘汰
 *                  策略" section 5: a paged cache frees whole blocks); the token
 *                  and the next r - 1 fill its slots in order.
 *     H2O_POOLS:   the H2OCache class of "KV Cache 驱逐策略：从 LRU 到 H2O"
 *                  (section "实现要点"): n_sink = 0, budget = n_recent +
 *                  n_heavy, n_recent >= 1. Each held token belongs to the
 *                  recent pool or the heavy-hitter pool. The new token joins
 *                  the recent pool; when that pool then holds more than
 *                  n_recent tokens, its member with the lowest (score,
 *                  position) leaves it, the new token included. That token is
 *                  promoted to the heavy-hitter pool iff its score is strictly
 *                  above hh_threshold, and leaves the cache otherwise; a
 *                  heavy-hitter pool above n_heavy tokens drops its lowest
 *                  member, the promoted one included. The new token takes the
 *                  slot of the token that left, else the lowest empty slot;
 *                  when it leaves itself, no slot changes. Scores as H2O.
 *   batch, n_layers, n_q_heads, n_kv_heads, head_dim: model shape;
 *     n_q_heads / n_kv_heads = G in {1, 2, 4, 8}; head_dim in {64, 128}.
 *   dtype: KVEVICT_F32 or KVEVICT_BF16 for K, V, q and out.
 *   max_prompt: RANDOM only, the longest prompt a unit may hold.
 *   score_forget, score_half: how H2O stores its cumulative scores ("Attention
 *     Sinks 与 KV Cache 淘汰策略" section 6.2: FP16 storage, or a moving average
 *     in place of the exact sum). Each step s <- (1 - score_forget) s + a, with
 *     0 <= score_forget < 1 (0, the default: the exact cumulative score; H2O
 *     and H2O_BLOCK). score_half = 1 stores every score as IEEE binary16
 *     (rounded to nearest even after each update; eviction compares the stored
 *     values), halving the score traffic; H2O and H2O_POOLS, and not with
 *     kvevict_prefill_scored / kvevict_prefill_snapkv. kvevict_scores still
 *     returns fp32. score_forget also applies to H2O_POOLS.
 *   hh_threshold: H2O_POOLS only, the promotion threshold (any value but NaN;
 *     the pages leave it open; -INFINITY promotes every token).
 *   score_int8: 1 stores the H2O scores as unsigned 8-bit codes with one fp32
 *     scale per (sequence, KV head) unit (the same section names INT8
 *     quantisation of the scores and gives no scale; the reading is absmax
 *     per unit, zero point 0): after each step's update (score_forget applies)
 *     every score becomes c = round(s * 255 / M), M the unit's largest score
 *     (the new token's included), stored as c * M / 255; eviction compares
 *     the stored values, ties to the older position. A quarter of the fp32
 *     score traffic. H2O only, not with score_half, nor with
 *     kvevict_prefill_scored / kvevict_prefill_snapkv; one CTA per unit
 *     (kvevict_create and kvevict_set_split refuse a split above 1 with
 *     INVALID_ARG). kvevict_scores returns c * scale as fp32.
 * Slot capacity per unit: C = budget (H2O, SINK_WINDOW, H2O_BLOCK) or
 * max_prompt + budget + r (RANDOM).
 */
typedef struct {
    int policy;
    int n_sink, n_heavy, n_recent, budget, r;
    uint64_t seed;
    int batch, n_layers, n_q_heads, n_kv_heads, head_dim;
    int dtype;
    int max_prompt;
    float score_forget;
    int score_half;
    float hh_threshold;
    int score_int8;
} kvevict_config;

typedef struct {
    int64_t decode_steps;   /* layer-steps issued (one per kvevict_decode_step call) */
    int64_t prefill_tokens; /* prompt tokens appended, summed over layers */
    int64_t evictions;      /* tokens evicted, summed over units and layers (H2O_POOLS: unit-steps in which the
                               recent pool overflowed; a promotion into a pool with room evicts nothing) */
    int64_t cuts;           /* Random cuts or H2O_BLOCK releases, summed over layers (each over every unit) */
    int split;              /* CTAs per unit in the decode launch (thread-block cluster size) */
    int capacity;           /* slots per unit */
    int clusters;           /* clusters in the last decode launch's persistent grid (0 before any) */
    int tensor_cores;       /* 1 if the decode path uses the tensor cores (mma), 0 for CUDA cores */
    int ring_stages;        /* shared-memory ring stages of the last decode launch (32 slots of K or V each) */
    int tail_split;         /* 1 if clusters split only their leftover units (kvevict_set_tail_split) */
    int partials_alias;     /* 1 if the last decode launch wrote its warps' partial outputs over the logits */
    double evicted_mass;    /* policies with scores: the stored scores of every token that left the cache,
                               summed over layers and units in fp64 (kvevict_evicted_mass per unit) */
    int64_t near_ties;      /* validation mode (kvevict_set_tie_audit): H2O eviction decisions whose runner-up
                               candidate's stored score was within 1e-5 relative of the evicted token's,
                               summed over layers and units; 0 when the mode was never on */
} kvevict_stats;

/* Bytes of device memory a handle with this configuration needs (cache,
 * positions, scores, the evicted-mass ledger and the near-tie counters of
 * policies with scores, free lists, error word, two slots of host-path
 * staging). Host only:
 * launches nothing, needs no GPU. Returns INVALID_ARG for a configuration
 * the library does not accept. */
int kvevict_state_bytes(const kvevict_config *cfg, size_t *bytes);

/* Creates a handle. `state` is device memory of at least
 * kvevict_state_bytes() bytes, 256-byte aligned, owned by the caller (the
 * Python binding allocates it with PyTorch) and used by the handle until
 * kvevict_destroy. `cuda_stream` is a cudaStream_t (NULL: the legacy default
 * stream). The cache starts empty (every position -1, every score 0); that
 * initialisation is queued on the stream. */
int kvevict_create(kvevict_t *out, const kvevict_config *cfg, void *state, size_t state_bytes,
                   void *cuda_stream);

/* Appends n_tokens prompt tokens to every unit of `layer`, with no attention
 * (the API gives the prompt no queries): each enters with score 0 through the
 * policy's admission rule, so H2O and SINK_WINDOW keep the n_sink first and
 * the newest C - n_sink prompt tokens, and RANDOM keeps them all.
 * K, V: device, [batch][n_kv_heads][n_tokens][head_dim]. May be called several
 * times (chunks) before the layer's first decode step; STATE after it.
 * RANDOM: CAPACITY if the layer's prompt would exceed max_prompt.
 * H2O_POOLS: the whole prompt in one call (STATE otherwise); with every score
 * 0 the recent pool's oldest member leaves each time, so hh_threshold >= 0
 * keeps the last n_recent prompt tokens and hh_threshold < 0 the last C, the
 * ones before the last n_recent in the heavy-hitter pool. */
int kvevict_prefill(kvevict_t h, int layer, const void *K, const void *V, int n_tokens);

/* Q-seeded prefill of an empty H2O layer ("h2o: heavy-hitter oracle" summary,
 * Algorithm 1: a token's score is the cumulative attention it receives; over
 * budget, remove the token whose removal leaves the highest total). The prompt
 * scores itself with its own causal attention:
 *   score_j = (1/G) sum over the G query heads g of the KV head, sum over
 *             prompt queries i >= j, of softmax_j(q_gi . k_j / sqrt(d)) (j <= i),
 * then, if prompt_len > budget, the n_sink first and n_recent last positions
 * stay and, of the others, the prompt_len - budget with the smallest (score,
 * position) leave (the greedy rule with scores that do not change during the
 * cut). The kept tokens fill slots 0, 1, ... in ascending position order, with
 * their scores; decode steps then add to those scores. (Calling
 * kvevict_decode_step for each prompt token instead applies Algorithm 1 from
 * the first token, with eviction during the prompt.)
 *   Q:    device, [batch][n_q_heads][prompt_len][head_dim] bf16;
 *   K, V: device, [batch][n_kv_heads][prompt_len][head_dim] bf16;
 *   workspace: device, 256-byte aligned, at least
 *         kvevict_prefill_scored_workspace_bytes() bytes, owned by the caller.
 *         Layout: per query row minus the log2 of its softmax normaliser, fp32
 *         [batch * n_q_heads][Ps] with Ps = prompt_len rounded up to 128; then,
 *         at the next 256-byte boundary, every prompt token's score before the
 *         cut, fp32 [batch][n_kv_heads][prompt_len]; then, at the next 256-byte
 *         boundary, 256 bytes of work counters that the call zeroes and the
 *         scoring kernels use. The first two are valid once the stream has
 *         passed the call; the caller may reuse the memory after.
 * The attention statistics run on the tcgen05 tensor cores (bf16 in, fp32
 * accumulate). INVALID_ARG unless the policy is H2O and the dtype bf16, for
 * prompt_len outside 1..49152, for null or misaligned pointers or a short
 * workspace; STATE if the layer already holds tokens or has decoded. */
int kvevict_prefill_scored_workspace_bytes(kvevict_t h, int prompt_len, size_t *bytes);
int kvevict_prefill_scored(kvevict_t h, int layer, const void *Q, const void *K, const void *V, int prompt_len,
                           void *workspace, size_t workspace_bytes);

/* SnapKV prefill of an empty H2O layer ("Attention Sinks 与 KV Cache 淘汰策略"
 * section 4.3): the last `window` prompt tokens' queries vote for the earlier
 * positions, and only what they pick is kept.
 *   votes_gj  = sum over the window's queries i of query head g of
 *               softmax_j(q_gi . k_j / sqrt(d)) over j <= i;
 *   pooled_gj = max of votes_gj' over |j' - j| <= 3 within the prefix
 *               [0, prompt_len - window);
 *   each query head keeps its k_per_head prefix positions with the largest
 *   pooled vote (ties: the newer position); a KV head keeps the union over
 *   its G query heads plus the window.
 * The kept tokens fill slots 0, 1, ... in ascending position order, each with
 * the score (1/G) sum_g votes_gj (the attention it received from the window);
 * the other slots stay empty. The next decode steps of the layer put the new
 * token into each unit's lowest empty slot while it has one and evict by
 * score after that.
 *   Q_obs: device, [batch][n_q_heads][window][head_dim] bf16, the queries of
 *          prompt positions prompt_len - window .. prompt_len - 1;
 *   K, V:  device, [batch][n_kv_heads][prompt_len][head_dim] bf16;
 *   workspace: device, 256-byte aligned, at least
 *          kvevict_prefill_snapkv_workspace_bytes() bytes, owned by the caller.
 *          Layout: the window rows' normalisers, fp32 [batch * n_q_heads][Ps]
 *          (Ps: the window's tiles of 128 rows); then, at the next 256-byte
 *          boundary, the votes, fp32 [batch][n_q_heads][prompt_len]; then, at
 *          the next 256-byte boundary, 256 bytes of work counters that the call
 *          zeroes and the scoring kernels use.
 * INVALID_ARG unless the policy is H2O and the dtype bf16, for 1 <= window <
 * prompt_len <= 49152 not holding, for G * k_per_head + window above the
 * capacity (the union must fit), for null or misaligned pointers or a short
 * workspace; STATE if the layer already holds tokens or has decoded. */
int kvevict_prefill_snapkv_workspace_bytes(kvevict_t h, int prompt_len, int window, size_t *bytes);
int kvevict_prefill_snapkv(kvevict_t h, int layer, const void *Q_obs, const void *K, const void *V, int prompt_len,
                           int window, int k_per_head, void *workspace, size_t workspace_bytes);

/* kvevict_prefill_scored without caller memory. The pages have no
 * counterpart: this is for callers that cannot allocate device memory when
 * they prefill -- a serving framework that reserved the GPU's free memory for
 * its own pool at start-up, or a latency-bound path that cannot take the
 * device-wide synchronisation cudaMalloc and cudaFree may cause. It does what
 * kvevict_prefill_scored does (same arguments and results), but its scratch
 * is a fixed 16 MiB array inside the library that every GPU loading the
 * library holds until the process exits; it calls no allocator.
 *   - Errors: first every check of kvevict_prefill_scored except those on the
 *     workspace, with the same status; then INVALID_ARG (and a line on
 *     stderr) if the handle's device is not the current device; then
 *     CAPACITY (and a line on stderr) when the prompt needs more scratch than
 *     16 MiB (kvevict_prefill_scored_workspace_bytes tells how much): use
 *     kvevict_prefill_scored with a workspace then.
 *   - kvevict_create looks up the array's address on the handle's device for
 *     every handle that may call this (H2O, bf16, fp32 scores), so the call
 *     itself does no lookup and needs no warm-up call first.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (other streams, other handles) race and corrupt each other; order them.
 *     Nothing in it needs to start at zero. */
int kvevict_prefill_scored_static(kvevict_t h, int layer, const void *Q, const void *K, const void *V,
                                  int prompt_len);

/* One decode step of `layer` for every sequence (the four steps above).
 *   q:     device, [batch][n_q_heads][head_dim]; query heads g*G .. g*G+G-1
 *          share KV head g.
 *   k_new, v_new: device, [batch][n_kv_heads][head_dim], the new token.
 *   out:   device, [batch][n_q_heads][head_dim], attention output.
 * Steps of one layer must be issued in token order; layers are independent.
 * The new token's position is the layer's prompt length plus its decode
 * steps so far. One kernel launch; RANDOM adds a cut launch every r steps. */
int kvevict_decode_step(kvevict_t h, int layer, const void *q, const void *k_new, const void *v_new, void *out);

/* kvevict_decode_step with HOST buffers of the same layouts (pinned memory
 * for asynchronous copies). Copies the inputs in, runs the step and copies
 * out back on the handle's stream, then waits for the stream. */
int kvevict_decode_step_host(kvevict_t h, int layer, const void *q, const void *k_new, const void *v_new,
                             void *out);

/* kvevict_decode_step_host without waiting, for pipelining host-buffer steps.
 * Where all four buffers are pinned host memory mapped into the device's
 * address space (cudaPointerGetAttributes gives a device pointer; 16-byte
 * aligned), the step's kernel reads the inputs and writes the output in place
 * over the CPU-GPU link: no staging copies, and consecutive calls' launches
 * follow each other on the handle's stream as kvevict_decode_step's do.
 * Otherwise the inputs are copied in on an internal copy-in stream, into one
 * of two staging slots that alternate between calls; the step runs on the
 * handle's stream once they are in; the output is copied back on an internal
 * copy-out stream once the step is done. A call's copy-in overlaps the
 * previous call's step, and its copy-out the next call's. Either way the host
 * buffers must stay valid, and the inputs unchanged, until kvevict_sync
 * returns; the output holds the result only then. Steps run in call order on
 * the handle's stream. kvevict_decode_step_host waits for the pending calls
 * first. The copy streams and their events are created on the first call
 * that copies. */
int kvevict_decode_step_host_async(kvevict_t h, int layer, const void *q, const void *k_new, const void *v_new,
                                   void *out);

/* 1 if p is pinned host memory that kernels may address in place (the
 * in-place path of kvevict_decode_step_host_async), else 0 (also for null). */
int kvevict_host_buffer_mapped(const void *p);

/* Waits for every call queued on the handle: its stream and the copy streams
 * of kvevict_decode_step_host_async. Returns CUDA if any reported an error. */
int kvevict_sync(kvevict_t h);

/* Position held by every slot of `layer`, -1 for an empty slot:
 * dst [batch][n_kv_heads][C] int32, device (dst_is_device = 1, asynchronous)
 * or host (dst_is_device = 0, the call waits for the stream). */
int kvevict_slot_positions(kvevict_t h, int layer, int32_t *dst, int dst_is_device);

/* Cumulative H2O scores of every slot of `layer`, [batch][n_kv_heads][C]
 * fp32 (empty slots hold stale values; read them with the positions).
 * INVALID_ARG for policies that keep no scores. Same dst rules as above. */
int kvevict_scores(kvevict_t h, int layer, float *dst, int dst_is_device);

/* The H2O eviction decision alone, on scores the caller supplies (a test and
 * diagnostic entry point: it checks the decode step's selector against another
 * implementation's scores). For every unit of `layer`, among the slots whose
 * token is a candidate for the layer's next decode step -- n_sink <= pos <=
 * p - n_recent, p = the position that step appends (the layer's prompt length
 * plus its decode steps so far), empty slots never -- the one with the
 * smallest (score, position): the victim that step evicts when the cache is
 * full and its updated scores are `scores` ("h2o: heavy-hitter oracle"
 * summary, Algorithm 1: remove the token whose removal leaves the highest
 * cumulative score; ties to the older position). The kernel uses the decode
 * step's own candidate rule, key (fp32 score bits, then position) and
 * reductions, on the decode kernel's CTA shape.
 *   scores:  device, [batch][n_kv_heads][C] fp32, 16-byte aligned; values of
 *            empty slots are ignored. Scores are >= 0 (as the decode step's).
 *   victims: device, [batch][n_kv_heads] int32: the victim's slot, -1 where
 *            no slot is a candidate.
 * Reads the layer's slot positions, changes nothing in the handle; one launch
 * on the handle's stream. INVALID_ARG unless the policy is H2O, for null or
 * misaligned pointers; STATE for a layer out of range. */
int kvevict_select_victims(kvevict_t h, int layer, const float *scores, int32_t *victims);

/* Checkpoint and resume. A handle's state is the device buffer the caller
 * gave kvevict_create (caller-owned: the caller copies it) plus host-side
 * counters (per layer: prompt length, decode steps, tokens held, the Random,
 * fill, pool and block bookkeeping; the cumulative stats), which these calls
 * serialise as 64-bit fields with the configuration. Save: call
 * kvevict_checkpoint_save, then copy the state buffer once the handle's
 * stream has passed every queued call; the record describes the state after
 * the calls issued so far. Resume: kvevict_create with the same configuration
 * on a buffer of state_bytes, copy the saved bytes into it, then
 * kvevict_checkpoint_restore (it waits for the handle's queued calls first).
 * Eviction decisions (and the counter-based Random keys) then continue
 * exactly as in the run that was saved. kvevict_checkpoint_bytes gives the
 * record size; save returns CAPACITY if `bytes` is smaller; restore returns
 * INVALID_ARG if the record is not one of this format and configuration. A
 * trace set on the restoring handle is dropped. */
int kvevict_checkpoint_bytes(kvevict_t h, size_t *bytes);
int kvevict_checkpoint_save(kvevict_t h, void *dst, size_t bytes);
int kvevict_checkpoint_restore(kvevict_t h, const void *src, size_t bytes);

/* Failure detection, exercised without a fault: queues on the handle's stream
 * one kernel in which a thread waits, through the same bounded wait as the
 * decode pipeline, on a barrier that nothing completes. After the wait limit
 * (2 s of device time) the kernel records KVEVICT_DEV_WAIT_TIMEOUT in the
 * handle's error word and ends; kvevict_check then reports the bit and clears
 * it, and the handle and the CUDA context stay usable. Returns OK or CUDA
 * (launch failure). */
int kvevict_probe_wait_timeout(kvevict_t h);

/* Evicted-mass ledger of `layer` (policies with scores, else INVALID_ARG):
 * for every unit, the sum in fp64 of the stored cumulative scores of the
 * tokens that left it through decode steps -- the victim of an H2O step, a
 * released block (H2O_BLOCK), the token leaving the two pools (H2O_POOLS) --
 * since the handle was created. With exact scores (no moving average, fp32
 * storage) the retained scores plus this mass equal the mass the unit has
 * received: one per decode step (the G query heads' mean of a softmax), plus
 * what the prompt brought (kvevict_prefill_scored: the kept tokens' scores).
 * dst [batch][n_kv_heads] fp64; same dst rules as kvevict_slot_positions.
 * ("KV Cache 驱逐策略：从 LRU 到 H2O" names the evicted mass among the
 * quantities to watch.) */
int kvevict_evicted_mass(kvevict_t h, int layer, double *dst, int dst_is_device);

/* INT8 score storage only (else INVALID_ARG): every unit's scale for `layer`,
 * its largest score / 255 after the last step (0 before the first);
 * dst [batch][n_kv_heads] fp32. Same dst rules as kvevict_slot_positions. */
int kvevict_score_scales(kvevict_t h, int layer, float *dst, int dst_is_device);

/* Pool of every slot of `layer` (H2O_POOLS only, else INVALID_ARG): 0 the
 * recent pool, 1 the heavy-hitter pool, meaningful where the slot holds a
 * token; dst [batch][n_kv_heads][C] uint8. Same dst rules as above. */
int kvevict_slot_pools(kvevict_t h, int layer, uint8_t *dst, int dst_is_device);

/* Decode-step trace of `layer`: while set, decode step t (0-based, counted
 * from this call), for t < n_steps, writes for every unit four int32 into
 * dev_buf[t][batch][n_kv_heads][4] (device, 16-byte aligned): the slot the
 * new token took, the position that slot held before (-1 if it was empty:
 * otherwise the evicted token), the evicted token's cumulative score and the
 * new token's score (fp32 bit patterns; 0 for policies without scores).
 * H2O_POOLS: the slot is -1 when the new token itself left (the next two
 * words are then its position and score), and the fourth word records the
 * promotion: the slot of the token moved to the heavy-hitter pool, -2 when
 * the new token joined that pool, -1 when nothing was promoted.
 * dev_buf = NULL clears it. */
int kvevict_set_trace(kvevict_t h, int layer, int32_t *dev_buf, int n_steps);

/* Host-side counters of `layer`: prompt tokens appended, decode steps issued
 * and tokens held per unit (after the last issued step; H2O_POOLS: an upper
 * bound, a unit may hold fewer). Any pointer may be NULL. */
int kvevict_layer_state(kvevict_t h, int layer, int *prompt_len, int *steps, int *count);

/* CTAs per unit of the decode launch (1, 2, 4, 8 or 16; 0 = automatic).
 * A tuning knob: results do not depend on it beyond fp32 rounding order. */
int kvevict_set_split(kvevict_t h, int split);

/* Tail splitting of the decode launch (-1 automatic, the default; 0 off; 1
 * on; a tuning knob like kvevict_set_split, results do not depend on it beyond
 * fp32 rounding order). Automatic turns it on, at clusters of two, where one
 * CTA per SM holds a whole unit and the units do not divide evenly over the
 * SMs; setting it (0 or 1) keeps the current split.
 * On, a cluster of `split` CTAs gives each CTA an equal number of its units to
 * process alone and splits only the units left over (its unit count mod
 * split) across all its CTAs, so that every resident CTA gets work and the
 * grid's load differs by less than one unit between CTAs; only those
 * leftover units pay for the cluster exchange. The persistent grid is then
 * every cluster the GPU holds at once. A whole unit must fit one CTA's shared
 * memory: INVALID_ARG otherwise, with INT8 score storage, and for kernels run two
 * CTAs per SM (group sizes 1 and 2), which do not build it. */
int kvevict_set_tail_split(kvevict_t h, int on);

/* Validation mode for H2O (policy KVEVICT_H2O): 1 on, 0 off (the default).
 * On, every decode step that may evict is followed by a small kernel that
 * counts, per unit, the decisions whose runner-up candidate (the smallest
 * stored score among the candidates left, by the same candidate rule) lies
 * within 1e-5 relative of the evicted token's stored score (|a - b| <
 * 1e-5 max(a, b), equal scores included): the decisions that a different
 * rounding of the scores could have flipped. The counts accumulate per layer
 * on the device (kvevict_near_ties) and in kvevict_stats.near_ties. Costs one
 * extra launch per layer-step; results of the decode itself are unchanged.
 * The counters and a [B][Hkv][4] record area (used when no trace is set; with
 * a trace the step's trace records are read) are part of the state buffer of
 * every policy with scores, zeroed by kvevict_create. A step whose eviction
 * found no candidate (KVEVICT_DEV_NO_CANDIDATE) is not counted reliably.
 * INVALID_ARG outside 0..1, and for 1 with a policy other than KVEVICT_H2O. */
int kvevict_set_tie_audit(kvevict_t h, int on);

/* The near-tie count of one layer since the handle was created (validation
 * mode, kvevict_set_tie_audit; 0 if it was never on). Waits for the handle's
 * stream. STATE if the layer is out of range. */
int kvevict_near_ties(kvevict_t h, int layer, uint64_t *out);

/* Where the decode launch keeps its warps' partial outputs: -1 automatic
 * (the default), 0 in an area of their own, 1 over the unit's logits once the
 * score pass has read them, wherever they fit there (that frees shared memory
 * for more ring stages and costs one barrier per unit; automatic takes it
 * where it buys at least two stages). Kernels run two CTAs per SM (group sizes
 * 1 and 2) always use their own area. A tuning knob: results do not depend on
 * it. INVALID_ARG outside -1..1. */
int kvevict_set_partials_alias(kvevict_t h, int mode);

/* Decode arithmetic: 0 = automatic (tensor cores for bf16 caches, CUDA
 * cores for fp32), 1 = CUDA cores, 2 = tensor cores (bf16 only; mma.sync
 * m16n8k16 with 16 slots / 16 head_dim rows as M and the G query heads,
 * padded to 8, as N). A
 * tuning and test knob: both paths compute the same step, they differ in
 * rounding only (the tensor-core path rounds probabilities to bf16 for PV).
 * INVALID_ARG if the path is not available for the handle's dtype or its
 * shared memory would not fit. */
int kvevict_set_path(kvevict_t h, int path);

/* At most this many shared-memory ring stages (32-slot K or V tiles) per CTA
 * in the decode launch; 0 = as many as the shared-memory budget allows (the
 * default). Kernels that run two CTAs per SM switch to one CTA per SM (twice
 * the shared memory) when the request does not fit the two-CTA budget. A
 * tuning knob: results do not depend on it. INVALID_ARG outside 4..32. */
int kvevict_set_ring(kvevict_t h, int stages);

/* Number of clusters in the decode launch's persistent grid (each cluster
 * loops over units; 0 = automatic: as many as fit on the GPU at once, chosen
 * to divide the units evenly where possible). A tuning knob like
 * kvevict_set_split; results do not depend on it. */
int kvevict_set_clusters(kvevict_t h, int clusters);

/* The handle's counters. For policies with scores it reads the evicted-mass
 * ledgers from the device and so waits for the handle's stream. */
int kvevict_get_stats(kvevict_t h, kvevict_stats *out);

/* Waits for the stream, reads the device error word into *device_error (may
 * be NULL) and clears it. Returns DEVICE if any bit was set, CUDA if the
 * stream reported an error. */
int kvevict_check(kvevict_t h, uint32_t *device_error);

const char *kvevict_strerror(int code);

/* Releases the host handle. The caller still owns and frees `state`. */
void kvevict_destroy(kvevict_t h);

#ifdef __cplusplus
}
#endif

#endif /* KVEVICT_H */
