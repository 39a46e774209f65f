// api.cu -- host runtime of libkvevict.so: argument checks, the device state
// layout, per-layer step bookkeeping and the launches. See include/kvevict.h.
//
// Every per-layer quantity the kernels need besides the data (how many slots
// are occupied, where an insert goes before the cache is full, when Random
// cuts) depends only on the number of prompt tokens and decode steps so far,
// never on values, so it is tracked here on the host and passed by value.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "api_internal.h"
#include "aux_kernels.h"
#include "decode_dispatch.h"
#include "decode_kernel.cuh"
#include "kvevict.h"
#include "prompt_attn.h"

using namespace kvevict;

namespace {

// An NVTX range around a public call (visible in Nsight timelines; a no-op
// without a tool attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

}  // namespace

namespace {

constexpr size_t kAlign = 256;
constexpr int kSMs = 152;
constexpr float kNearTieRel = 1e-5f;  // two candidate scores closer than this (relative) are a near-tie

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Policies that keep cumulative attention scores.
bool scored(int policy)
{
    return policy == KVEVICT_H2O || policy == KVEVICT_H2O_BLOCK || policy == KVEVICT_H2O_POOLS;
}

struct Layout {
    int C = 0, G = 0, elem = 0;
    int Cs = 0;               // per-unit stride of pos/score (rows start on 16 bytes)
    int score_elem = 4;       // bytes per stored score
    size_t off_qscale = 0;    // INT8 scores: [L][B][Hkv] fp32 scale per unit
    int Ps = 0;               // per-unit stride of the pool flags (two-pool H2O; rows start on 16 bytes)
    size_t units = 0;         // B * Hkv
    size_t layer_slots = 0;   // units * C (K/V rows)
    size_t layer_pslots = 0;  // units * Cs (pos/score entries)
    size_t kv_layer_bytes = 0;
    size_t off_k = 0, off_v = 0, off_pos = 0, off_score = 0, off_pool = 0, off_free = 0, off_err = 0;
    size_t off_ledger = 0;  // [L][B][Hkv] fp64 evicted score mass (policies with scores)
    size_t off_tie = 0;     // validation mode (policies with scores): [L] u64 near-tie counts, then [B][Hkv][4] int32
                            // step records
    size_t tie_trace_off = 0;  // the step records' offset inside that region
    size_t off_sq[2] = {}, off_sk[2] = {}, off_sv[2] = {}, off_so[2] = {};  // host-path staging, two slots
    size_t total = 0;
    size_t q_bytes = 0, kvtok_bytes = 0;  // one layer-step's q/out and k_new/v_new
};

int validate(const kvevict_config *c)
{
    if (!c) return KVEVICT_ERR_INVALID_ARG;
    if (c->batch < 1 || c->batch > 65535 || c->n_layers < 1 || c->n_kv_heads < 1 || c->n_kv_heads > 65535 ||
        c->n_q_heads < 1)
        return KVEVICT_ERR_INVALID_ARG;
    if (c->n_q_heads % c->n_kv_heads) return KVEVICT_ERR_INVALID_ARG;
    const int G = c->n_q_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return KVEVICT_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128) return KVEVICT_ERR_INVALID_ARG;
    if (c->dtype != KVEVICT_F32 && c->dtype != KVEVICT_BF16) return KVEVICT_ERR_INVALID_ARG;
    if (c->budget < 1) return KVEVICT_ERR_INVALID_ARG;
    switch (c->policy) {
    case KVEVICT_H2O:
        if (c->n_sink < 0 || c->n_heavy < 0 || c->n_recent < 1 ||
            static_cast<long long>(c->n_sink) + c->n_heavy + c->n_recent != c->budget)
            return KVEVICT_ERR_INVALID_ARG;
        break;
    case KVEVICT_SINK_WINDOW:
        if (c->n_sink < 0 || c->n_heavy != 0 || c->n_recent < 1 ||
            static_cast<long long>(c->n_sink) + c->n_recent != c->budget)
            return KVEVICT_ERR_INVALID_ARG;
        break;
    case KVEVICT_H2O_BLOCK:
        if (c->n_sink < 0 || c->n_heavy < 0 || c->n_recent < 1 ||
            static_cast<long long>(c->n_sink) + c->n_heavy + c->n_recent != c->budget)
            return KVEVICT_ERR_INVALID_ARG;
        if (c->r < 1 || c->budget % c->r != 0) return KVEVICT_ERR_INVALID_ARG;
        {
            const long long nb = c->budget / c->r, nsb = (static_cast<long long>(c->n_sink) + c->r - 1) / c->r;
            if ((nb - nsb - 1) * c->r < c->n_recent) return KVEVICT_ERR_INVALID_ARG;
        }
        break;
    case KVEVICT_H2O_POOLS:
        if (c->n_sink != 0 || c->n_heavy < 0 || c->n_recent < 1 ||
            static_cast<long long>(c->n_heavy) + c->n_recent != c->budget || std::isnan(c->hh_threshold))
            return KVEVICT_ERR_INVALID_ARG;
        break;
    case KVEVICT_RANDOM:
        if (c->r < 1 || c->max_prompt < 0 || c->n_sink != 0 || c->n_heavy != 0 || c->n_recent != 0)
            return KVEVICT_ERR_INVALID_ARG;
        if (static_cast<long long>(c->budget) + c->r > kMaxRandomCandidates) return KVEVICT_ERR_INVALID_ARG;
        break;
    default:
        return KVEVICT_ERR_INVALID_ARG;
    }
    if (!(c->score_forget >= 0.f && c->score_forget < 1.f) || (c->score_half != 0 && c->score_half != 1))
        return KVEVICT_ERR_INVALID_ARG;
    if (c->score_forget != 0.f && !scored(c->policy)) return KVEVICT_ERR_INVALID_ARG;
    if (c->score_half && c->policy != KVEVICT_H2O && c->policy != KVEVICT_H2O_POOLS) return KVEVICT_ERR_INVALID_ARG;
    if (c->score_int8 != 0 && (c->score_int8 != 1 || c->policy != KVEVICT_H2O || c->score_half))
        return KVEVICT_ERR_INVALID_ARG;
    const long long C = c->policy == KVEVICT_RANDOM ? static_cast<long long>(c->max_prompt) + c->budget + c->r
                                                    : c->budget;
    if (C > (1 << 24)) return KVEVICT_ERR_INVALID_ARG;
    return KVEVICT_OK;
}

Layout make_layout(const kvevict_config *c)
{
    Layout L;
    L.G = c->n_q_heads / c->n_kv_heads;
    L.elem = c->dtype == KVEVICT_F32 ? 4 : 2;
    L.C = c->policy == KVEVICT_RANDOM ? c->max_prompt + c->budget + c->r : c->budget;
    // pos/score rows start on 16 bytes for the bulk copies: 4-byte entries need
    // a multiple of 4, binary16 scores a multiple of 8, 8-bit codes of 16
    L.Cs = c->score_int8 ? (L.C + 15) / 16 * 16 : c->score_half ? (L.C + 7) / 8 * 8 : (L.C + 3) / 4 * 4;
    L.score_elem = c->score_int8 ? 1 : c->score_half ? 2 : 4;
    L.Ps = c->policy == KVEVICT_H2O_POOLS ? (L.C + 15) / 16 * 16 : 0;
    L.units = static_cast<size_t>(c->batch) * c->n_kv_heads;
    L.layer_slots = L.units * L.C;
    L.layer_pslots = L.units * L.Cs;
    L.kv_layer_bytes = L.layer_slots * c->head_dim * L.elem;
    const size_t nl = c->n_layers;
    size_t off = 0;
    L.off_k = off; off = align_up(off + nl * L.kv_layer_bytes);
    L.off_v = off; off = align_up(off + nl * L.kv_layer_bytes);
    L.off_pos = off; off = align_up(off + nl * L.layer_pslots * 4);
    L.off_score = off; if (scored(c->policy)) off = align_up(off + nl * L.layer_pslots * L.score_elem);
    L.off_qscale = off; if (c->score_int8) off = align_up(off + nl * L.units * 4);
    L.off_ledger = off; if (scored(c->policy)) off = align_up(off + nl * L.units * 8);
    L.tie_trace_off = (nl * 8 + 15) / 16 * 16;
    L.off_tie = off; if (scored(c->policy)) off = align_up(off + L.tie_trace_off + L.units * 16);
    L.off_pool = off; off = align_up(off + nl * L.units * L.Ps);
    L.off_free = off;
    if (c->policy == KVEVICT_RANDOM || c->policy == KVEVICT_H2O_BLOCK) off = align_up(off + nl * L.units * c->r * 4);
    L.off_err = off; off = align_up(off + 16);
    L.q_bytes = static_cast<size_t>(c->batch) * c->n_q_heads * c->head_dim * L.elem;
    L.kvtok_bytes = L.units * c->head_dim * L.elem;
    for (int i = 0; i < 2; ++i) {
        L.off_sq[i] = off; off = align_up(off + L.q_bytes);
        L.off_sk[i] = off; off = align_up(off + L.kvtok_bytes);
        L.off_sv[i] = off; off = align_up(off + L.kvtok_bytes);
        L.off_so[i] = off; off = align_up(off + L.q_bytes);
    }
    L.total = off;
    return L;
}

struct LayerState {
    int prompt_len = 0;
    int t = 0;           // decode steps issued
    int count = 0;       // tokens held per unit (H2O, sink-window)
    int n_gen = 0;       // generated tokens held per unit (Random)
    bool cut_done = false;
    int fl_idx = 0;      // next free-list entry (Random after a cut)
    int32_t *trace = nullptr;
    int trace_len = 0, trace_t = 0;
    int fill_left = 0;   // H2O after a SnapKV prefill: steps left in which a unit may still have empty slots
    int n_rec = 0;       // H2O_POOLS: tokens in every unit's recent pool (count is then an upper bound)
    int blk_left = 0;    // H2O_BLOCK: slots of the open (released) block not yet refilled
    int blk_next = 0;    // H2O_BLOCK: next slot of the open block when every unit's is the same
    bool blk_uniform = false;  // H2O_BLOCK: the open block is the same slot range in every unit
};

}  // namespace

struct kvevict_handle {
    kvevict_config cfg;
    Layout L;
    uint8_t *state = nullptr;
    int device = -1;  // the CUDA device holding `state`
    cudaStream_t stream = nullptr;
    int split = 1;
    bool tail_split = false;  // clusters split only their leftover units (each CTA's others whole)
    int tail_req = -1;        // tail splitting requested: -1 automatic, 0 off, 1 on
    int clusters_req = 0;  // persistent grid size in clusters; 0 = automatic
    int last_layer = -1;   // layer of the last kernel this handle queued (-1: none, or unknown)
    int path_req = 0;      // 0 automatic, 1 CUDA cores, 2 tensor cores
    int ring_req = 0;      // ring stages requested (0 = fill the shared-memory budget)
    int alias_req = -1;    // warp partials over the logits: -1 automatic, 0 never, 1 where they fit
    bool use_mma = false;  // decode path in use
    // Validation mode: near-ties of the H2O decisions counted on the device
    // (per layer, in the state buffer), from each step's records (the caller's
    // trace, else the state buffer's record area).
    bool tie_audit = false;
    std::vector<CUtensorMap> tmk, tmv;  // per layer (bf16 caches)
    std::vector<LayerState> layers;
    kvevict_stats stats{};
    // host-buffer path without waiting: a stream for the copies in, one for the
    // copies out, and per staging slot the events "inputs are in", "the step is
    // done" and "the output is out" (created on first use)
    cudaStream_t in_stream = nullptr, out_stream = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_step[2] = {}, ev_out[2] = {};
    int async_calls = 0;
    bool async_pending = false;
    ~kvevict_handle()
    {
        if (in_stream) {
            cudaStreamSynchronize(in_stream);
            cudaStreamSynchronize(out_stream);
            for (int i = 0; i < 2; ++i) {
                cudaEventDestroy(ev_in[i]);
                cudaEventDestroy(ev_step[i]);
                cudaEventDestroy(ev_out[i]);
            }
            cudaStreamDestroy(in_stream);
            cudaStreamDestroy(out_stream);
        }
    }
    // decode kernel configured for (split, holes): function, shared memory, zcap
    struct Configured {
        int split = 0, clusters_req = -1, ring_req = -1, alias_req = -2;
        bool mma = false, tail_split = false, alias = false;
        DecodeKernelInfo ki{};
        size_t smem = 0;
        int zc = 0, nst = 0;
        int clusters = 0;  // persistent grid, in clusters
    } configured[2];
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return KVEVICT_OK;
    std::fprintf(stderr, "kvevict: CUDA error %s\n", cudaGetErrorString(e));
    return KVEVICT_ERR_CUDA;
}

int max_slots_per_cta(const Layout &L, int S)
{
    const int tiles = (L.C + kTile - 1) / kTile;
    return ((tiles + S - 1) / S) * kTile;
}

int n_aux_arrays(const kvevict_config &c, bool holes)
{
    if (c.policy == KVEVICT_H2O_POOLS) return 3;  // positions, scores, pool flags
    return scored(c.policy) ? 2 : (holes ? 1 : 0);
}

// Launches whose units may hold empty slots among the scanned ones (positions
// are then read before attention).
bool holes_policy(const kvevict_config &c) { return c.policy == KVEVICT_RANDOM || c.policy == KVEVICT_H2O_POOLS; }

constexpr size_t kMaxSmem = 227 * 1024;

// Ring stages filling the shared-memory budget of the kernel's target
// occupancy (two CTAs per SM when its registers allow, else one).
// A ring request above what the two-CTA budget holds selects the one-CTA
// budget (a deeper ring for one CTA per SM).
int ring_stages(const DecodeKernelInfo &ki, size_t fixed, int ring_req = 0)
{
    const size_t budget2 = 113 * 1024, budget1 = kMaxSmem;
    bool two = ki.ctas_per_sm >= 2 && fixed + kMinStages * ki.stage_bytes <= budget2;
    if (two && ring_req > 0 && fixed + static_cast<size_t>(ring_req) * ki.stage_bytes > budget2) two = false;
    const size_t budget = two ? budget2 : budget1;
    if (fixed + kMinStages * static_cast<size_t>(ki.stage_bytes) > budget) return 0;
    return static_cast<int>(std::min<size_t>(kMaxStages, (budget - fixed) / ki.stage_bytes));
}

// Shared memory of the decode launch with clusters of S CTAs; with tail
// splitting a CTA also holds whole units, so it is sized as at S = 1. The
// warps' partial outputs get an area of their own, or are written over the
// logits (alias): that costs one barrier per unit, and is taken automatically
// where it fits and buys at least two more ring stages.
size_t decode_smem(const kvevict_handle *h, int S, bool holes, int *nst_out = nullptr, bool tail = false,
                   bool *alias_out = nullptr)
{
    DecodeKernelInfo ki;
    if (!decode_kernel(h->cfg.dtype, h->cfg.head_dim, h->L.G, holes, h->use_mma, &ki)) return ~size_t(0);
    const int zc = ki.zcap(max_slots_per_cta(h->L, tail ? 1 : S));
    const int na = n_aux_arrays(h->cfg, holes);
    size_t best = ~size_t(0);
    int best_nst = 0;
    bool best_alias = false;
    const bool can_alias = ki.flex && ki.alias_fits(zc);
    for (int a = 0; a < 2; ++a) {
        const bool alias = a == 1;
        if (alias && (h->alias_req == 0 || !can_alias)) continue;
        if (!alias && h->alias_req == 1 && can_alias) continue;
        const size_t fixed = ki.fixed_bytes(zc, na, alias);
        int nst = ring_stages(ki, fixed, h->ring_req);
        if (h->ring_req > 0 && nst > 0) nst = std::min(nst, h->ring_req);
        if (nst == 0) continue;
        if (alias && h->alias_req < 0 && best_nst > 0 && nst < best_nst + 2) continue;
        best = fixed + static_cast<size_t>(nst) * ki.stage_bytes;
        best_nst = nst;
        best_alias = alias;
    }
    if (nst_out) *nst_out = best_nst;
    if (alias_out) *alias_out = best_alias;
    return best;
}

// CTAs per unit. The persistent kernel streams best with one CTA per unit: a
// cluster adds two barriers and a DSMEM exchange per unit. Split a unit over
// a cluster when its logits do not fit one CTA's shared memory, or when there
// are too few units to give every resident CTA (2 per SM) one while each CTA
// keeps >= 256 slots.
int auto_split(const kvevict_handle *h)
{
    const Layout &L = h->L;
    const bool holes = holes_policy(h->cfg);
    if (h->cfg.score_int8) return 1;  // INT8 scores need the unit's largest score in one CTA
    for (int S = 1; S <= kMaxSplit; S *= 2) {
        if (decode_smem(h, S, holes) > kMaxSmem) continue;
        if (S < 8 && static_cast<long long>(L.units) * S < 2LL * kSMs && L.C / (2 * S) >= 256) continue;
        return S;
    }
    return kMaxSplit;
}

// Tail splitting, automatically: where one CTA per SM holds a whole unit
// (the kernel's shared memory or registers allow no second CTA) and the
// whole-unit grid cannot give every SM the same number of units, clusters of
// two CTAs split the leftover units, so every SM streams until the end
// (measured on the GQA layer: 512 units on 152 SMs, 98 -> 93 us per launch).
// Kernels at two CTAs per SM do not gain (their SMs already overlap two CTAs).
void auto_tail(kvevict_handle *h)
{
    h->tail_split = false;
    if (h->tail_req == 0 || h->cfg.score_int8) return;
    const bool holes = holes_policy(h->cfg);
    if (h->tail_req == 1) {
        h->tail_split = decode_smem(h, h->split, holes, nullptr, true) <= kMaxSmem;
        return;
    }
    DecodeKernelInfo ki;
    if (h->split != 1 || !decode_kernel(h->cfg.dtype, h->cfg.head_dim, h->L.G, holes, h->use_mma, &ki) || !ki.flex)
        return;
    const size_t smem1 = decode_smem(h, 1, holes);
    const bool one_per_sm = ki.ctas_per_sm < 2 || smem1 > 113 * 1024;
    const long long units = static_cast<long long>(h->L.units);
    if (!one_per_sm || units <= kSMs || units % kSMs == 0) return;
    if (decode_smem(h, 2, holes, nullptr, true) > kMaxSmem) return;
    h->split = 2;
    h->tail_split = true;
}

int configure_kernel(const kvevict_handle *h, int S, bool holes, DecodeKernelInfo *ki, size_t *smem, int *zc, int *nst,
                     bool *alias)
{
    if (!decode_kernel(h->cfg.dtype, h->cfg.head_dim, h->L.G, holes, h->use_mma, ki)) return KVEVICT_ERR_INVALID_ARG;
    *zc = ki->zcap(max_slots_per_cta(h->L, h->tail_split ? 1 : S));
    *smem = decode_smem(h, S, holes, nst, h->tail_split, alias);
    if (*smem > kMaxSmem || *nst == 0) return KVEVICT_ERR_INVALID_ARG;
    cudaError_t e = cudaFuncSetAttribute(ki->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(*smem));
    if (e == cudaSuccess && S > 8) e = cudaFuncSetAttribute(ki->fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return cuda_status(e);
}

template <typename T> T *at(const kvevict_handle *h, size_t off) { return reinterpret_cast<T *>(h->state + off); }

// One layer's stored cumulative scores (fp32, or binary16 with score_half).
void *layer_scores(const kvevict_handle *h, int layer)
{
    return h->state + h->L.off_score + static_cast<size_t>(layer) * h->L.layer_pslots * h->L.score_elem;
}

// 2-D tensor map over rows of head_dim bf16 (a layer's K or V cache: rows =
// units * C; prompt Q or K: rows = heads * P); boxes of box_rows rows x 64
// elements, 128-byte swizzle.
int make_tensor_map(CUtensorMap *out, const void *base, uint64_t rows, int head_dim, int box_rows = kTile)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return KVEVICT_ERR_CUDA;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        std::fprintf(stderr, "kvevict: cuTensorMapEncodeTiled failed (%d)\n", static_cast<int>(r));
        return KVEVICT_ERR_CUDA;
    }
    return KVEVICT_OK;
}

bool mma_possible(const kvevict_config &c) { return c.dtype == KVEVICT_BF16; }
// Tensor cores for every bf16 cache: at G = 1 they still cut the issue
// count per slot about tenfold against the CUDA-core butterfly.
bool mma_auto(const kvevict_config &c) { return mma_possible(c); }

// Persistent grid size, in clusters: at most what the GPU holds at once.
// With few units per cluster, a count that divides the units evenly (every
// cluster then does the same number of units and none idles in the last
// round); with many, all of them.
int pick_clusters(const kvevict_handle *h, int S, const DecodeKernelInfo &ki, size_t smem, int *clusters)
{
    const int units = static_cast<int>(h->L.units);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(S, 1, 1);
    lc.blockDim = dim3(ki.threads, 1, 1);
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int maxc = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&maxc, ki.fn, &lc);
    if (e != cudaSuccess) return cuda_status(e);
    if (maxc < 1) return KVEVICT_ERR_INVALID_ARG;  // a cluster of this size does not fit
    if (h->clusters_req > 0) {
        *clusters = std::min(h->clusters_req, units);
        return KVEVICT_OK;
    }
    if (h->tail_split) {  // every resident cluster: the load differs by less than a unit between CTAs
        *clusters = std::min(maxc, units);
        return KVEVICT_OK;
    }
    if (units <= maxc) {
        *clusters = units;
        return KVEVICT_OK;
    }
    // Many units per cluster: the last round's imbalance is small and every
    // resident slot streaming beats an even split over fewer clusters.
    if ((units + maxc - 1) / maxc >= 5) {
        *clusters = maxc;
        return KVEVICT_OK;
    }
    int best = maxc;
    long long best_waste = -1;
    for (int n = maxc; n >= (3 * maxc + 3) / 4; --n) {
        const long long rounds = (units + n - 1) / n;
        const long long waste = rounds * n - units;
        if (best_waste < 0 || waste < best_waste) {
            best = n;
            best_waste = waste;
        }
        if (waste == 0) break;
    }
    *clusters = best;
    return KVEVICT_OK;
}

int launch_decode(kvevict_handle *h, int layer, const void *q, const void *kn, const void *vn, void *out)
{
    const kvevict_config &c = h->cfg;
    const Layout &L = h->L;
    LayerState &ls = h->layers[layer];

    DecodeParams P{};
    P.q = q; P.k_new = kn; P.v_new = vn; P.out = out;
    P.kc = h->state + L.off_k + layer * L.kv_layer_bytes;
    P.vc = h->state + L.off_v + layer * L.kv_layer_bytes;
    P.pos = at<int32_t>(h, L.off_pos) + layer * L.layer_pslots;
    P.score = scored(c.policy) ? layer_scores(h, layer) : nullptr;
    P.score_keep = 1.f - c.score_forget;
    P.score_half = c.score_half;
    P.score_int8 = c.score_int8;
    P.qscale = c.score_int8 ? at<float>(h, L.off_qscale) + static_cast<size_t>(layer) * L.units : nullptr;
    P.freelist = (c.policy == KVEVICT_RANDOM || c.policy == KVEVICT_H2O_BLOCK)
                     ? at<int32_t>(h, L.off_free) + layer * L.units * c.r
                     : nullptr;
    P.units = static_cast<int>(L.units);
    P.cstride = L.Cs;
    P.freelist_len = c.r;
    P.err = at<uint32_t>(h, L.off_err);
    P.ledger = scored(c.policy) ? at<double>(h, L.off_ledger) + static_cast<size_t>(layer) * L.units : nullptr;
    P.C = L.C;
    P.p = ls.prompt_len + ls.t;
    P.n_sink = c.n_sink;
    P.n_recent = c.n_recent;
    P.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c.head_dim)));
    P.trace = (ls.trace && ls.trace_t < ls.trace_len) ? ls.trace + static_cast<size_t>(ls.trace_t) * L.units * 4 : nullptr;
    const bool user_trace = P.trace != nullptr;

    bool holes = false;
    long long evicted = 0;
    bool released = false;  // H2O_BLOCK: a block was released for this token
    switch (c.policy) {
    case KVEVICT_H2O_BLOCK:
        if (ls.count < L.C) {  // the cache is still filling
            P.n_active = ls.count;
            P.mode = kInsertAt;
            P.dest_slot = ls.count;
        } else {
            P.n_active = L.C;
            holes = true;
            if (ls.blk_left == 0) {  // full: release a block before this token attends
                BlockReleaseParams bp{};
                bp.pos = P.pos;
                bp.score = static_cast<float *>(P.score);
                bp.freelist = const_cast<int32_t *>(P.freelist);
                bp.kc = P.kc;
                bp.vc = P.vc;
                bp.row_bytes = c.head_dim * L.elem;
                bp.C = L.C;
                bp.cstride = L.Cs;
                bp.bs = c.r;
                bp.n_sink = c.n_sink;
                bp.n_recent = c.n_recent;
                bp.p = P.p;
                bp.ledger = P.ledger;
                bp.err = P.err;
                int rc0 = cuda_status(launch_block_release(bp, static_cast<int>(L.units), h->stream));
                if (rc0) return rc0;
                h->last_layer = layer;  // the release wrote this layer: no early prefetch
                released = true;
                evicted = static_cast<long long>(L.units) * c.r;
                h->stats.cuts++;
                P.mode = kFromFreeList;
                P.freelist_idx = 0;
            } else if (ls.blk_uniform) {
                P.mode = kInsertAt;
                P.dest_slot = ls.blk_next;
            } else {
                P.mode = kFromFreeList;
                P.freelist_idx = c.r - ls.blk_left;
            }
        }
        break;
    case KVEVICT_H2O_POOLS:
        // ls.count bounds every unit's occupancy; a unit's tokens fill slots
        // 0, 1, ... (a slot is only freed for the token that takes it)
        P.n_active = ls.count;
        P.mode = kTwoPool;
        P.pool = at<uint8_t>(h, L.off_pool) + static_cast<size_t>(layer) * L.units * L.Ps;
        P.pstride = L.Ps;
        P.recent_full = ls.n_rec == c.n_recent ? 1 : 0;
        P.hh_threshold = c.hh_threshold;
        holes = true;
        if (P.recent_full) evicted = static_cast<long long>(L.units);
        break;
    case KVEVICT_SINK_WINDOW:
        P.n_active = ls.count;
        P.mode = kInsertAt;
        P.dest_slot = P.p < c.n_sink ? P.p : c.n_sink + (P.p - c.n_sink) % c.n_recent;
        if (ls.count == L.C) evicted = static_cast<long long>(L.units);
        break;
    case KVEVICT_H2O:
        P.n_active = ls.count;
        if (ls.fill_left > 0) {  // after a SnapKV prefill: per-unit empty slots
            P.mode = kH2OFill;
            holes = true;
        } else if (ls.count < L.C) {
            P.mode = kInsertAt;
            P.dest_slot = ls.count;
        } else {
            P.mode = kH2OEvict;
            evicted = static_cast<long long>(L.units);
        }
        break;
    default:  // Random
        if (!ls.cut_done) {
            P.n_active = ls.prompt_len + ls.n_gen;
            P.mode = kInsertAt;
            P.dest_slot = ls.prompt_len + ls.n_gen;
        } else {
            P.n_active = ls.prompt_len + c.budget + c.r;
            P.mode = kFromFreeList;
            P.freelist_idx = ls.fl_idx;
            holes = true;
        }
        break;
    }

    auto &cfgd = h->configured[holes ? 1 : 0];
    if (cfgd.split != h->split || cfgd.clusters_req != h->clusters_req || cfgd.mma != h->use_mma ||
        cfgd.ring_req != h->ring_req || cfgd.tail_split != h->tail_split || cfgd.alias_req != h->alias_req) {
        int rc0 = configure_kernel(h, h->split, holes, &cfgd.ki, &cfgd.smem, &cfgd.zc, &cfgd.nst, &cfgd.alias);
        if (rc0) return rc0;
        rc0 = pick_clusters(h, h->split, cfgd.ki, cfgd.smem, &cfgd.clusters);
        if (rc0) return rc0;
        cfgd.split = h->split;
        cfgd.clusters_req = h->clusters_req;
        cfgd.mma = h->use_mma;
        cfgd.ring_req = h->ring_req;
        cfgd.tail_split = h->tail_split;
        cfgd.alias_req = h->alias_req;
    }
    const DecodeKernelInfo &ki = cfgd.ki;
    const size_t smem = cfgd.smem;
    int rc = KVEVICT_OK;
    P.split = h->split;
    P.tail_split = h->tail_split ? 1 : 0;
    P.zcap = cfgd.zc;
    P.nst = cfgd.nst;
    P.part_alias = cfgd.alias ? 1 : 0;
    P.prefetch_early = (h->last_layer >= 0 && h->last_layer != layer) ? 1 : 0;
    if (h->use_mma) {
        static_assert(sizeof(CUtensorMap) == sizeof(TensorMapBytes), "tensor map size");
        std::memcpy(&P.tmk, &h->tmk[layer], sizeof(CUtensorMap));
        std::memcpy(&P.tmv, &h->tmv[layer], sizeof(CUtensorMap));
    }

    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(cfgd.clusters * h->split, 1, 1);
    lc.blockDim = dim3(ki.threads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = h->stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = h->split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 2;
    // validation mode: the step's records feed the near-tie count
    const bool audit = h->tie_audit && c.policy == KVEVICT_H2O && (P.mode == kH2OEvict || P.mode == kH2OFill);
    if (audit && !P.trace) P.trace = at<int32_t>(h, L.off_tie + L.tie_trace_off);
    void *args[] = {&P};
    rc = cuda_status(cudaLaunchKernelExC(&lc, ki.fn, args));
    if (rc) return rc;
    h->last_layer = layer;
    if (audit) {
        TieAuditParams tp{};
        tp.pos = P.pos;
        tp.score = P.score;
        tp.qscale = P.qscale;
        tp.trace = P.trace;
        tp.count = at<unsigned long long>(h, L.off_tie) + layer;
        tp.score_half = P.score_half;
        tp.score_int8 = P.score_int8;
        tp.n_active = P.n_active;
        tp.cstride = P.cstride;
        tp.p = P.p;
        tp.n_sink = P.n_sink;
        tp.n_recent = P.n_recent;
        tp.rel = kNearTieRel;
        rc = cuda_status(launch_tie_audit(tp, static_cast<int>(L.units), h->stream));
        if (rc) return rc;
    }

    // Bookkeeping of what the step did.
    if (user_trace) ls.trace_t++;
    h->stats.decode_steps++;
    h->stats.evictions += evicted;
    switch (c.policy) {
    case KVEVICT_SINK_WINDOW:
    case KVEVICT_H2O:
        ls.count = std::min(L.C, ls.count + 1);
        if (ls.fill_left > 0) ls.fill_left--;
        break;
    case KVEVICT_H2O_POOLS:
        ls.count = std::min(L.C, ls.count + 1);
        ls.n_rec = std::min(c.n_recent, ls.n_rec + 1);
        break;
    case KVEVICT_H2O_BLOCK:
        if (ls.count < L.C) {
            ls.count++;
        } else if (released) {
            ls.blk_left = c.r - 1;
            ls.blk_uniform = false;
        } else {
            ls.blk_left--;
            ls.blk_next++;
        }
        break;
    default:
        ls.n_gen++;
        if (ls.cut_done) ls.fl_idx++;
        if (ls.n_gen == c.budget + c.r) {
            CutParams cp{};
            cp.pos = P.pos;
            cp.freelist = const_cast<int32_t *>(P.freelist);
            cp.seed = c.seed;
            cp.layer = layer;
            cp.step = ls.t;
            cp.Hkv = c.n_kv_heads;
            cp.C = L.C;
            cp.cstride = L.Cs;
            cp.kc = P.kc;
            cp.vc = P.vc;
            cp.row_bytes = c.head_dim * L.elem;
            cp.first_slot = ls.prompt_len;
            cp.n_cand = c.budget + c.r;
            cp.n_pow2 = 1;
            while (cp.n_pow2 < cp.n_cand) cp.n_pow2 <<= 1;
            cp.r = c.r;
            rc = cuda_status(launch_random_cut(cp, c.batch, h->stream));
            if (rc) return rc;
            ls.n_gen = c.budget;
            ls.cut_done = true;
            ls.fl_idx = 0;
            h->stats.cuts++;
            h->stats.evictions += static_cast<long long>(L.units) * c.r;
        }
        break;
    }
    ls.t++;
    return KVEVICT_OK;
}

}  // namespace

extern "C" {

int kvevict_state_bytes(const kvevict_config *cfg, size_t *bytes)
{
    int rc = validate(cfg);
    if (rc) return rc;
    if (!bytes) return KVEVICT_ERR_INVALID_ARG;
    *bytes = make_layout(cfg).total;
    return KVEVICT_OK;
}

int kvevict_create(kvevict_t *out, const kvevict_config *cfg, void *state, size_t state_bytes, void *cuda_stream)
{
    NvtxRange nvtx("kvevict_create");
    if (!out) return KVEVICT_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = validate(cfg);
    if (rc) return rc;
    Layout L = make_layout(cfg);
    if (!state || (reinterpret_cast<uintptr_t>(state) & (kAlign - 1))) return KVEVICT_ERR_INVALID_ARG;
    if (state_bytes < L.total) return KVEVICT_ERR_CAPACITY;
    cudaPointerAttributes pa{};
    if (cudaPointerGetAttributes(&pa, state) != cudaSuccess || pa.type != cudaMemoryTypeDevice) {
        cudaGetLastError();  // clear the sticky-free error of a failed query
        return KVEVICT_ERR_INVALID_ARG;
    }
    kvevict_handle *h = new (std::nothrow) kvevict_handle();
    if (!h) return KVEVICT_ERR_CAPACITY;
    h->device = pa.device;
    h->cfg = *cfg;
    h->L = L;
    h->state = static_cast<uint8_t *>(state);
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    h->layers.resize(cfg->n_layers);
    h->use_mma = mma_auto(*cfg);
    if (mma_possible(*cfg)) {
        h->tmk.resize(cfg->n_layers);
        h->tmv.resize(cfg->n_layers);
        for (int l = 0; l < cfg->n_layers; ++l) {
            int rc0 = make_tensor_map(&h->tmk[l], h->state + L.off_k + l * L.kv_layer_bytes, L.layer_slots, cfg->head_dim);
            if (!rc0) rc0 = make_tensor_map(&h->tmv[l], h->state + L.off_v + l * L.kv_layer_bytes, L.layer_slots, cfg->head_dim);
            if (rc0) {
                delete h;
                return rc0;
            }
        }
    }
    h->split = auto_split(h);
    auto_tail(h);
    h->stats.tail_split = h->tail_split ? 1 : 0;
    // INT8 scores need one CTA per unit: a unit must fit one CTA's shared memory
    if (cfg->score_int8 && decode_smem(h, 1, holes_policy(*cfg)) > kMaxSmem) {
        delete h;
        return KVEVICT_ERR_INVALID_ARG;
    }
    // A handle that may call kvevict_prefill_scored_static: look up the fixed
    // scratch array's address on this device now, so that call does no lookup
    // of its own (and can be captured in a stream like the other calls).
    if (cfg->policy == KVEVICT_H2O && cfg->dtype == KVEVICT_BF16 && !cfg->score_half && !cfg->score_int8) {
        void *scratch = nullptr;
        int rc0 = kvevict_static_scratch_address(h->device, &scratch);
        if (rc0) {
            delete h;
            return rc0;
        }
    }
    // Empty cache: K/V zero (every row a tile may touch is finite), every
    // position -1, every score 0, no error bits.
    cudaError_t e = cudaMemsetAsync(h->state + L.off_k, 0, L.off_pos - L.off_k, h->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->state + L.off_pos, 0xFF, cfg->n_layers * L.layer_pslots * 4, h->stream);
    if (e == cudaSuccess && scored(cfg->policy))
        e = cudaMemsetAsync(h->state + L.off_score, 0, cfg->n_layers * L.layer_pslots * L.score_elem, h->stream);
    if (e == cudaSuccess && cfg->score_int8)
        e = cudaMemsetAsync(h->state + L.off_qscale, 0, cfg->n_layers * L.units * 4, h->stream);
    if (e == cudaSuccess && scored(cfg->policy))
        e = cudaMemsetAsync(h->state + L.off_ledger, 0, cfg->n_layers * L.units * 8, h->stream);
    if (e == cudaSuccess && scored(cfg->policy))
        e = cudaMemsetAsync(h->state + L.off_tie, 0, L.tie_trace_off + L.units * 16, h->stream);
    if (e == cudaSuccess && L.Ps > 0)
        e = cudaMemsetAsync(h->state + L.off_pool, 0, cfg->n_layers * L.units * L.Ps, h->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->state + L.off_err, 0, 16, h->stream);
    if (e != cudaSuccess) {
        delete h;
        return cuda_status(e);
    }
    h->stats.split = h->split;
    h->stats.capacity = L.C;
    *out = h;
    return KVEVICT_OK;
}

int kvevict_prefill(kvevict_t h, int layer, const void *K, const void *V, int n_tokens)
{
    NvtxRange nvtx("kvevict_prefill");
    if (!h || layer < 0 || layer >= h->cfg.n_layers) return h ? KVEVICT_ERR_STATE : KVEVICT_ERR_INVALID_ARG;
    if (n_tokens < 0 || (n_tokens > 0 && (!K || !V || !aligned16(K) || !aligned16(V)))) return KVEVICT_ERR_INVALID_ARG;
    LayerState &ls = h->layers[layer];
    if (ls.t > 0) return KVEVICT_ERR_STATE;
    const kvevict_config &c = h->cfg;
    const Layout &L = h->L;
    if (c.policy == KVEVICT_RANDOM && static_cast<long long>(ls.prompt_len) + n_tokens > c.max_prompt)
        return KVEVICT_ERR_CAPACITY;
    if (static_cast<long long>(ls.prompt_len) + n_tokens > (1LL << 30)) return KVEVICT_ERR_INVALID_ARG;
    if (n_tokens == 0) return KVEVICT_OK;

    PrefillParams P{};
    P.K = K; P.V = V;
    P.kc = h->state + L.off_k + layer * L.kv_layer_bytes;
    P.vc = h->state + L.off_v + layer * L.kv_layer_bytes;
    P.pos = at<int32_t>(h, L.off_pos) + layer * L.layer_pslots;
    P.score = scored(c.policy) ? layer_scores(h, layer) : nullptr;
    P.score_half = c.score_half;
    P.score_int8 = c.score_int8;
    P.n_tok = n_tokens;
    P.p0 = ls.prompt_len;
    P.C = L.C;
    P.cstride = L.Cs;
    P.Hkv = c.n_kv_heads;
    P.head_dim = c.head_dim;
    P.elem_bytes = L.elem;
    if (c.policy == KVEVICT_RANDOM) {
        P.n_sink = 0;
        P.ring_len = 0;
        P.a0 = 0; P.a1 = n_tokens;
        P.b0 = P.b1 = 0;
    } else {
        P.n_sink = c.n_sink;
        P.ring_len = L.C - c.n_sink;
        if (c.policy == KVEVICT_H2O_POOLS) {
            // every prompt score is 0, so the recent pool's oldest member leaves each
            // time: dropped (threshold >= 0: the last n_recent stay, a ring of
            // n_recent slots) or promoted (threshold < 0: the last C stay, a ring of
            // C slots, the ones before the last n_recent in the heavy-hitter pool)
            if (ls.prompt_len != 0) return KVEVICT_ERR_STATE;  // the whole prompt in one call
            P.ring_len = c.hh_threshold >= 0.f ? c.n_recent : L.C;
            P.pool = at<uint8_t>(h, L.off_pool) + static_cast<size_t>(layer) * L.units * L.Ps;
            P.pstride = L.Ps;
            P.hh_below = n_tokens - c.n_recent;
        }
        P.a0 = 0;
        P.a1 = std::min(n_tokens, std::max(0, c.n_sink - P.p0));
        P.b0 = std::max({0, c.n_sink - P.p0, n_tokens - P.ring_len});
        P.b1 = n_tokens;
        if (P.b0 > P.b1) P.b0 = P.b1;
    }
    if (c.policy == KVEVICT_H2O_BLOCK) {
        // the whole prompt in one call: the closed-form layout covers it
        if (ls.prompt_len != 0) return KVEVICT_ERR_STATE;
        BlockPrefillParams bp{};
        bp.K = K;
        bp.V = V;
        bp.kc = P.kc;
        bp.vc = P.vc;
        bp.pos = P.pos;
        bp.score = static_cast<float *>(P.score);
        bp.n_tok = n_tokens;
        bp.C = L.C;
        bp.cstride = L.Cs;
        bp.Hkv = c.n_kv_heads;
        bp.row_bytes = c.head_dim * L.elem;
        bp.bs = c.r;
        bp.nsb = (c.n_sink + c.r - 1) / c.r;
        launch_block_prefill(bp, c.batch, h->stream);
        int rc = cuda_status(cudaGetLastError());
        if (rc) return rc;
        h->last_layer = layer;
        ls.prompt_len = n_tokens;
        ls.count = std::min(L.C, n_tokens);
        ls.blk_left = 0;
        if (n_tokens > L.C && (n_tokens - L.C) % c.r) {  // the last released block is partly refilled
            const int nb = L.C / c.r, released = (n_tokens - L.C + c.r - 1) / c.r;
            const int blk = bp.nsb + (released - 1) % (nb - bp.nsb);
            ls.blk_next = blk * c.r + (n_tokens - L.C) % c.r;
            ls.blk_left = c.r - (n_tokens - L.C) % c.r;
            ls.blk_uniform = true;
        }
        h->stats.prefill_tokens += n_tokens;
        return KVEVICT_OK;
    }
    launch_prefill(P, (P.a1 - P.a0) + (P.b1 - P.b0), c.batch, h->stream);
    int rc = cuda_status(cudaGetLastError());
    if (rc) return rc;
    h->last_layer = layer;
    ls.prompt_len += n_tokens;
    ls.count = c.policy == KVEVICT_RANDOM ? ls.prompt_len : std::min(L.C, ls.prompt_len);
    if (c.policy == KVEVICT_H2O_POOLS) {
        ls.count = std::min(P.ring_len, n_tokens);
        ls.n_rec = std::min(c.n_recent, n_tokens);
    }
    h->stats.prefill_tokens += n_tokens;
    return KVEVICT_OK;
}

namespace {

// Workspace of the Q-seeded prefill: per query row its log-normaliser
// ([B * Hq][Ps], Ps = P rounded up to a tile, so each tile's 128 entries are
// addressable), then per key its score ([B * Hkv][P]).
struct ScoredWorkspace {
    size_t stats_off = 0, score_off = 0, work_off = 0, bytes = 0;
    int Ps = 0;
};

ScoredWorkspace scored_workspace(const kvevict_config &c, int P)
{
    ScoredWorkspace w;
    w.Ps = (P + kPromptTile - 1) / kPromptTile * kPromptTile;
    w.stats_off = 0;
    w.score_off = align_up(static_cast<size_t>(c.batch) * c.n_q_heads * w.Ps * 4);
    w.work_off = w.score_off + align_up(static_cast<size_t>(c.batch) * c.n_kv_heads * P * 4);
    w.bytes = w.work_off + kAlign;  // the scoring passes' work counters
    return w;
}

}  // namespace

int kvevict_handle_device(kvevict_t h) { return h ? h->device : -1; }

int kvevict_prefill_scored_check(kvevict_t h, int layer, const void *Q, const void *K, const void *V, int prompt_len)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const kvevict_config &c = h->cfg;
    const int P = prompt_len;
    if (c.policy != KVEVICT_H2O || c.dtype != KVEVICT_BF16 || c.score_half || c.score_int8)
        return KVEVICT_ERR_INVALID_ARG;
    if (P < 1 || P > kPromptMaxLen) return KVEVICT_ERR_INVALID_ARG;
    if (!Q || !K || !V || !aligned16(Q) || !aligned16(K) || !aligned16(V)) return KVEVICT_ERR_INVALID_ARG;
    const long long q_rows = static_cast<long long>(c.batch) * c.n_q_heads * P;
    if (q_rows >= (1LL << 31)) return KVEVICT_ERR_INVALID_ARG;  // tensor-map row coordinates are int32
    if (static_cast<long long>(c.batch) * c.n_q_heads > 65535) return KVEVICT_ERR_INVALID_ARG;  // grid height
    const LayerState &ls = h->layers[layer];
    if (ls.prompt_len != 0 || ls.t != 0) return KVEVICT_ERR_STATE;
    return KVEVICT_OK;
}

int kvevict_prefill_scored_workspace_bytes(kvevict_t h, int prompt_len, size_t *bytes)
{
    if (!h || !bytes || prompt_len < 1 || prompt_len > kPromptMaxLen) return KVEVICT_ERR_INVALID_ARG;
    *bytes = scored_workspace(h->cfg, prompt_len).bytes;
    return KVEVICT_OK;
}

int kvevict_prefill_scored(kvevict_t h, int layer, const void *Q, const void *K, const void *V, int prompt_len,
                           void *workspace, size_t workspace_bytes)
{
    NvtxRange nvtx("kvevict_prefill_scored");
    int rc = kvevict_prefill_scored_check(h, layer, Q, K, V, prompt_len);
    if (rc) return rc;
    const kvevict_config &c = h->cfg;
    const Layout &L = h->L;
    const int P = prompt_len;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return KVEVICT_ERR_INVALID_ARG;
    const ScoredWorkspace ws = scored_workspace(c, P);
    if (workspace_bytes < ws.bytes) return KVEVICT_ERR_INVALID_ARG;
    const long long q_rows = static_cast<long long>(c.batch) * c.n_q_heads * P;
    LayerState &ls = h->layers[layer];

    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    PromptAttnParams ap{};
    CUtensorMap tq, tk;
    rc = make_tensor_map(&tq, Q, static_cast<uint64_t>(q_rows), c.head_dim, kPromptTile);
    if (rc == KVEVICT_OK)
        rc = make_tensor_map(&tk, K, static_cast<uint64_t>(c.batch) * c.n_kv_heads * P, c.head_dim, kPromptTile);
    if (rc) return rc;
    static_assert(sizeof(CUtensorMap) == sizeof(PromptTmap), "tensor map size");
    ap.stats = reinterpret_cast<float *>(wsb + ws.stats_off);
    ap.score = reinterpret_cast<float *>(wsb + ws.score_off);
    ap.P = P;
    ap.Ps = ws.Ps;
    ap.G = L.G;
    ap.Hq = c.n_q_heads;
    ap.Hkv = c.n_kv_heads;
    ap.q_lo = 0;
    ap.q_stride = P;
    ap.q_first = 0;
    ap.per_head = 0;
    ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c.head_dim)));
    ap.err = at<uint32_t>(h, L.off_err);
    int *work = reinterpret_cast<int *>(wsb + ws.work_off);  // [0]: pass 1, [1]: pass 2
    // pass 1: A = query tiles, B = key tiles; pass 2: A = key tiles, B = query tiles
    std::memcpy(&ap.tma, &tq, sizeof tq);
    std::memcpy(&ap.tmb, &tk, sizeof tk);
    ap.work = work;
    cudaError_t e = cudaMemsetAsync(work, 0, 2 * sizeof(int), h->stream);
    if (e == cudaSuccess) e = launch_prompt_rowstats(ap, c.head_dim, c.batch, h->stream);
    if (e == cudaSuccess) {
        std::memcpy(&ap.tma, &tk, sizeof tk);
        std::memcpy(&ap.tmb, &tq, sizeof tq);
        ap.work = work + 1;
        e = launch_prompt_colsum(ap, c.head_dim, c.batch, h->stream);
    }
    if (e == cudaSuccess) {
        PromptSelectParams sp{};
        sp.score = ap.score;
        sp.K = K;
        sp.V = V;
        sp.kc = h->state + L.off_k + layer * L.kv_layer_bytes;
        sp.vc = h->state + L.off_v + layer * L.kv_layer_bytes;
        sp.pos = at<int32_t>(h, L.off_pos) + layer * L.layer_pslots;
        sp.cscore = static_cast<float *>(layer_scores(h, layer));
        sp.P = P;
        sp.C = L.C;
        sp.cstride = L.Cs;
        sp.row_bytes = c.head_dim * L.elem;
        sp.budget = c.budget;
        sp.n_sink = c.n_sink;
        sp.n_recent = c.n_recent;
        sp.err = ap.err;
        e = launch_prompt_select(sp, static_cast<int>(L.units), h->stream);
    }
    if (e != cudaSuccess) return cuda_status(e);
    h->last_layer = layer;
    ls.prompt_len = P;
    ls.count = std::min(L.C, P);
    h->stats.prefill_tokens += P;
    return KVEVICT_OK;
}

namespace {

// Workspace of the SnapKV prefill: the normalisers of the window's query rows
// ([B * Hq][Ps], from the window's first tile on), then the votes of every
// query head on every prompt key ([B * Hq][P]).
struct SnapWorkspace {
    size_t stats_off = 0, votes_off = 0, work_off = 0, bytes = 0;
    int Ps = 0, qs0 = 0;
};

SnapWorkspace snap_workspace(const kvevict_config &c, int P, int window)
{
    SnapWorkspace w;
    w.qs0 = (P - window) / kPromptTile * kPromptTile;
    w.Ps = (P - w.qs0 + kPromptTile - 1) / kPromptTile * kPromptTile;
    w.stats_off = 0;
    w.votes_off = align_up(static_cast<size_t>(c.batch) * c.n_q_heads * w.Ps * 4);
    w.work_off = w.votes_off + align_up(static_cast<size_t>(c.batch) * c.n_q_heads * P * 4);
    w.bytes = w.work_off + kAlign;  // the scoring passes' work counters
    return w;
}

}  // namespace

int kvevict_prefill_snapkv_workspace_bytes(kvevict_t h, int prompt_len, int window, size_t *bytes)
{
    if (!h || !bytes || prompt_len < 2 || prompt_len > kPromptMaxLen || window < 1 || window >= prompt_len)
        return KVEVICT_ERR_INVALID_ARG;
    *bytes = snap_workspace(h->cfg, prompt_len, window).bytes;
    return KVEVICT_OK;
}

int kvevict_prefill_snapkv(kvevict_t h, int layer, const void *Q_obs, const void *K, const void *V, int prompt_len,
                           int window, int k_per_head, void *workspace, size_t workspace_bytes)
{
    NvtxRange nvtx("kvevict_prefill_snapkv");
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const kvevict_config &c = h->cfg;
    const Layout &L = h->L;
    const int P = prompt_len;
    if (c.policy != KVEVICT_H2O || c.dtype != KVEVICT_BF16 || c.score_half || c.score_int8)
        return KVEVICT_ERR_INVALID_ARG;
    if (P < 2 || P > kPromptMaxLen || window < 1 || window >= P || k_per_head < 0) return KVEVICT_ERR_INVALID_ARG;
    // the union of the G heads' top-k lists plus the window must fit the unit
    if (static_cast<long long>(L.G) * k_per_head + window > L.C) return KVEVICT_ERR_INVALID_ARG;
    if (!Q_obs || !K || !V || !workspace || !aligned16(Q_obs) || !aligned16(K) || !aligned16(V) ||
        (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)))
        return KVEVICT_ERR_INVALID_ARG;
    const SnapWorkspace ws = snap_workspace(c, P, window);
    if (workspace_bytes < ws.bytes) return KVEVICT_ERR_INVALID_ARG;
    if (static_cast<long long>(c.batch) * c.n_q_heads > 65535 ||
        static_cast<long long>(c.batch) * c.n_kv_heads * P >= (1LL << 31))
        return KVEVICT_ERR_INVALID_ARG;
    LayerState &ls = h->layers[layer];
    if (ls.prompt_len != 0 || ls.t != 0) return KVEVICT_ERR_STATE;

    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    CUtensorMap tq, tk;
    int rc = make_tensor_map(&tq, Q_obs, static_cast<uint64_t>(c.batch) * c.n_q_heads * window, c.head_dim,
                             kPromptTile);
    if (rc == KVEVICT_OK)
        rc = make_tensor_map(&tk, K, static_cast<uint64_t>(c.batch) * c.n_kv_heads * P, c.head_dim, kPromptTile);
    if (rc) return rc;
    PromptAttnParams ap{};
    ap.stats = reinterpret_cast<float *>(wsb + ws.stats_off);
    ap.score = reinterpret_cast<float *>(wsb + ws.votes_off);
    ap.P = P;
    ap.Ps = ws.Ps;
    ap.G = L.G;
    ap.Hq = c.n_q_heads;
    ap.Hkv = c.n_kv_heads;
    ap.q_lo = P - window;
    ap.q_stride = window;
    ap.q_first = P - window;
    ap.per_head = 1;
    // stack the G heads' window rows into shared tiles when every 32-row chunk belongs to one head
    ap.stacked = window % 32 == 0;
    if (ap.stacked) ap.Ps = (L.G * window + kPromptTile - 1) / kPromptTile * kPromptTile;
    ap.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c.head_dim)));
    ap.err = at<uint32_t>(h, L.off_err);
    std::memcpy(&ap.tma, &tq, sizeof tq);
    std::memcpy(&ap.tmb, &tk, sizeof tk);
    int *work = reinterpret_cast<int *>(wsb + ws.work_off);  // [0]: pass 1, [1]: pass 2
    ap.work = work;
    cudaError_t e = cudaMemsetAsync(work, 0, 2 * sizeof(int), h->stream);
    if (e == cudaSuccess) e = launch_prompt_rowstats(ap, c.head_dim, c.batch, h->stream);
    const int Lq = L.G * window;
    if (e == cudaSuccess && ap.stacked && Lq <= kSnapVotesMaxRows) {
        // the votes streamed: the unit's stacked window rows stay resident, key tiles stream
        CUtensorMap tqn;
        rc = make_tensor_map(&tqn, Q_obs, static_cast<uint64_t>(c.batch) * c.n_q_heads * window, c.head_dim, Lq);
        if (rc) return rc;
        SnapVotesParams vp{};
        std::memcpy(&vp.tmk, &tk, sizeof tk);
        std::memcpy(&vp.tmq, &tqn, sizeof tqn);
        vp.stats = ap.stats;
        vp.votes = ap.score;
        vp.P = P;
        vp.Ps = ap.Ps;
        vp.w = window;
        vp.G = L.G;
        vp.Hq = c.n_q_heads;
        vp.Hkv = c.n_kv_heads;
        vp.Lq = Lq;
        vp.units = static_cast<int>(L.units);
        vp.scale_log2 = ap.scale_log2;
        vp.err = ap.err;
        int dev = 0, sms = kSMs;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        e = launch_snapkv_votes(vp, c.head_dim, sms, h->stream);
    } else if (e == cudaSuccess) {
        std::memcpy(&ap.tma, &tk, sizeof tk);
        std::memcpy(&ap.tmb, &tq, sizeof tq);
        ap.work = work + 1;
        e = launch_prompt_colsum(ap, c.head_dim, c.batch, h->stream);
    }
    if (e == cudaSuccess) {
        SnapSelectParams sp{};
        sp.votes = ap.score;
        sp.K = K;
        sp.V = V;
        sp.kc = h->state + L.off_k + layer * L.kv_layer_bytes;
        sp.vc = h->state + L.off_v + layer * L.kv_layer_bytes;
        sp.pos = at<int32_t>(h, L.off_pos) + layer * L.layer_pslots;
        sp.cscore = static_cast<float *>(layer_scores(h, layer));
        sp.P = P;
        sp.C = L.C;
        sp.cstride = L.Cs;
        sp.row_bytes = c.head_dim * L.elem;
        sp.G = L.G;
        sp.Hq = c.n_q_heads;
        sp.Hkv = c.n_kv_heads;
        sp.window = window;
        sp.topk = k_per_head;
        sp.err = ap.err;
        e = launch_snapkv_select(sp, static_cast<int>(L.units), h->stream);
    }
    if (e != cudaSuccess) return cuda_status(e);
    h->last_layer = layer;
    ls.prompt_len = P;
    // Every unit keeps between min(k, P - window) + window and the capacity
    // tokens, in slots from 0 on; the rest of its slots are empty. Decode
    // steps fill each unit's lowest empty slot until every unit is surely
    // full, then evict as usual.
    ls.count = L.C;
    ls.fill_left = L.C - (std::min(k_per_head, P - window) + window);
    h->stats.prefill_tokens += P;
    return KVEVICT_OK;
}

int kvevict_decode_step(kvevict_t h, int layer, const void *q, const void *k_new, const void *v_new, void *out)
{
    NvtxRange nvtx("kvevict_decode_step");
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    if (!q || !k_new || !v_new || !out) return KVEVICT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out)) return KVEVICT_ERR_INVALID_ARG;
    if (h->layers[layer].prompt_len + static_cast<long long>(h->layers[layer].t) >= (1LL << 31) - 1)
        return KVEVICT_ERR_STATE;
    return launch_decode(h, layer, q, k_new, v_new, out);
}

int kvevict_sync(kvevict_t h)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    cudaError_t e = cudaSuccess;
    if (h->in_stream) {
        e = cudaStreamSynchronize(h->in_stream);
        cudaError_t e1 = cudaStreamSynchronize(h->out_stream);
        if (e == cudaSuccess) e = e1;
    }
    cudaError_t e2 = cudaStreamSynchronize(h->stream);
    h->async_pending = false;
    return cuda_status(e != cudaSuccess ? e : e2);
}

// The device address of a pinned host buffer that kernels may read and write in
// place (mapped into the device's address space), or null (any other memory).
static void *mapped_host(const void *p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the error of a failed query
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int kvevict_host_buffer_mapped(const void *p) { return p && mapped_host(p) ? 1 : 0; }

int kvevict_decode_step_host_async(kvevict_t h, int layer, const void *q, const void *k_new, const void *v_new,
                                   void *out)
{
    NvtxRange nvtx("kvevict_decode_step_host_async");
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    if (!q || !k_new || !v_new || !out) return KVEVICT_ERR_INVALID_ARG;
    if (h->layers[layer].prompt_len + static_cast<long long>(h->layers[layer].t) >= (1LL << 31) - 1)
        return KVEVICT_ERR_STATE;
    // Pinned buffers the GPU can address (over the CPU-GPU link): the kernel reads
    // the inputs and writes the output in place, with no staging copies and no
    // event waits between the launches of consecutive calls.
    void *mq = mapped_host(q), *mk = mapped_host(k_new), *mv = mapped_host(v_new), *mo = mapped_host(out);
    if (mq && mk && mv && mo && aligned16(mq) && aligned16(mk) && aligned16(mv) && aligned16(mo)) {
        const int rc = launch_decode(h, layer, mq, mk, mv, mo);
        if (rc) return rc;
        h->async_calls++;
        h->async_pending = true;
        return KVEVICT_OK;
    }
    cudaError_t e = cudaSuccess;
    if (!h->in_stream) {
        e = cudaStreamCreateWithFlags(&h->in_stream, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->out_stream, cudaStreamNonBlocking);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_step[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return cuda_status(e);
    }
    const Layout &L = h->L;
    const int sl = h->async_calls & 1;
    void *dq = h->state + L.off_sq[sl], *dk = h->state + L.off_sk[sl], *dv = h->state + L.off_sv[sl];
    void *dout = h->state + L.off_so[sl];
    // Inputs in on the copy-in stream, once the step two calls back (same slot)
    // has read them; a wait on an event never recorded passes at once.
    e = cudaStreamWaitEvent(h->in_stream, h->ev_step[sl], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dq, q, L.q_bytes, cudaMemcpyHostToDevice, h->in_stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, k_new, L.kvtok_bytes, cudaMemcpyHostToDevice, h->in_stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, v_new, L.kvtok_bytes, cudaMemcpyHostToDevice, h->in_stream);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_in[sl], h->in_stream);
    // the step on the handle's stream once the inputs are in and the copy-out two
    // calls back has drained this slot's output
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, h->ev_in[sl], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, h->ev_out[sl], 0);
    if (e != cudaSuccess) return cuda_status(e);
    h->last_layer = -1;  // the launch follows event waits, not a kernel of this handle
    int rc = launch_decode(h, layer, dq, dk, dv, dout);
    if (rc) return rc;
    // the output back on the copy-out stream once the step (and a Random cut) is done
    e = cudaEventRecord(h->ev_step[sl], h->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(h->out_stream, h->ev_step[sl], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out, dout, L.q_bytes, cudaMemcpyDeviceToHost, h->out_stream);
    if (e == cudaSuccess) e = cudaEventRecord(h->ev_out[sl], h->out_stream);
    if (e != cudaSuccess) return cuda_status(e);
    h->async_calls++;
    h->async_pending = true;
    return KVEVICT_OK;
}

int kvevict_decode_step_host(kvevict_t h, int layer, const void *q, const void *k_new, const void *v_new, void *out)
{
    NvtxRange nvtx("kvevict_decode_step_host");
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    if (!q || !k_new || !v_new || !out) return KVEVICT_ERR_INVALID_ARG;
    if (h->async_pending) {  // calls without waiting may still use the staging slots
        int rc0 = kvevict_sync(h);
        if (rc0) return rc0;
    }
    // pinned buffers the GPU can address: read and written in place, as in the call without waiting
    void *mq = mapped_host(q), *mk = mapped_host(k_new), *mv = mapped_host(v_new), *mo = mapped_host(out);
    if (mq && mk && mv && mo && aligned16(mq) && aligned16(mk) && aligned16(mv) && aligned16(mo)) {
        const int rc = launch_decode(h, layer, mq, mk, mv, mo);
        if (rc) return rc;
        return cuda_status(cudaStreamSynchronize(h->stream));
    }
    const Layout &L = h->L;
    void *dq = h->state + L.off_sq[0], *dk = h->state + L.off_sk[0], *dv = h->state + L.off_sv[0];
    void *dout = h->state + L.off_so[0];
    h->last_layer = -1;  // the launch follows copies, not a kernel of this handle
    cudaError_t e = cudaMemcpyAsync(dq, q, L.q_bytes, cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dk, k_new, L.kvtok_bytes, cudaMemcpyHostToDevice, h->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dv, v_new, L.kvtok_bytes, cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_status(e);
    int rc = launch_decode(h, layer, dq, dk, dv, dout);
    if (rc) return rc;
    e = cudaMemcpyAsync(out, dout, L.q_bytes, cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    return cuda_status(e);
}

int kvevict_slot_positions(kvevict_t h, int layer, int32_t *dst, int dst_is_device)
{
    if (!h || !dst) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const Layout &L = h->L;
    const void *src = at<int32_t>(h, L.off_pos) + layer * L.layer_pslots;
    cudaError_t e = cudaMemcpy2DAsync(dst, L.C * 4, src, L.Cs * 4, L.C * 4, L.units,
                                      dst_is_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess && !dst_is_device) e = cudaStreamSynchronize(h->stream);
    return cuda_status(e);
}

int kvevict_scores(kvevict_t h, int layer, float *dst, int dst_is_device)
{
    if (!h || !dst) return KVEVICT_ERR_INVALID_ARG;
    if (!scored(h->cfg.policy)) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const Layout &L = h->L;
    const void *src = layer_scores(h, layer);
    if (L.score_elem == 1) {  // INT8 codes times each unit's scale, returned as fp32
        const float *scl = at<float>(h, L.off_qscale) + static_cast<size_t>(layer) * L.units;
        if (dst_is_device)
            return cuda_status(launch_scores_int8_to_f32(dst, src, scl, L.C, L.Cs, L.units, h->stream));
        std::vector<uint8_t> codes(static_cast<size_t>(L.units) * L.C);
        std::vector<float> scales(L.units);
        cudaError_t e = cudaMemcpy2DAsync(codes.data(), L.C, src, L.Cs, L.C, L.units, cudaMemcpyDeviceToHost,
                                          h->stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(scales.data(), scl, L.units * 4, cudaMemcpyDeviceToHost, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e != cudaSuccess) return cuda_status(e);
        for (size_t i = 0; i < codes.size(); ++i) dst[i] = static_cast<float>(codes[i]) * scales[i / L.C];
        return KVEVICT_OK;
    }
    if (L.score_elem == 2) {  // binary16 storage, returned as fp32
        if (dst_is_device) return cuda_status(launch_scores_to_f32(dst, src, L.C, L.Cs, L.units, h->stream));
        std::vector<__half> tmp(static_cast<size_t>(L.units) * L.C);
        cudaError_t e = cudaMemcpy2DAsync(tmp.data(), L.C * 2, src, L.Cs * 2, L.C * 2, L.units,
                                          cudaMemcpyDeviceToHost, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e != cudaSuccess) return cuda_status(e);
        for (size_t i = 0; i < tmp.size(); ++i) dst[i] = __half2float(tmp[i]);
        return KVEVICT_OK;
    }
    cudaError_t e = cudaMemcpy2DAsync(dst, L.C * 4, src, L.Cs * 4, L.C * 4, L.units,
                                      dst_is_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess && !dst_is_device) e = cudaStreamSynchronize(h->stream);
    return cuda_status(e);
}

namespace {

constexpr int64_t kCkptMagic = 0x31504b4356454b56ll;  // "VKEVCKP1" little-endian
constexpr int64_t kCkptVersion = 1;

int64_t f32_bits(float f)
{
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return static_cast<int64_t>(u);
}

// The handle's host-side state as 64-bit fields: magic, version, the config,
// the counters of every layer, the cumulative stats.
std::vector<int64_t> checkpoint_record(const kvevict_handle *h)
{
    const kvevict_config &c = h->cfg;
    std::vector<int64_t> r = {kCkptMagic, kCkptVersion, c.policy, c.n_sink, c.n_heavy, c.n_recent, c.budget, c.r,
                              static_cast<int64_t>(c.seed), c.batch, c.n_layers, c.n_q_heads, c.n_kv_heads,
                              c.head_dim, c.dtype, c.max_prompt, f32_bits(c.score_forget), c.score_half,
                              f32_bits(c.hh_threshold), c.score_int8};
    for (const LayerState &ls : h->layers) {
        const int64_t f[] = {ls.prompt_len, ls.t,         ls.count,    ls.n_gen,    ls.cut_done ? 1 : 0,
                             ls.fl_idx,     ls.fill_left, ls.n_rec,    ls.blk_left, ls.blk_next,
                             ls.blk_uniform ? 1 : 0};
        r.insert(r.end(), std::begin(f), std::end(f));
    }
    const int64_t s[] = {h->stats.decode_steps, h->stats.prefill_tokens, h->stats.evictions, h->stats.cuts};
    r.insert(r.end(), std::begin(s), std::end(s));
    return r;
}

constexpr size_t kCkptHead = 20;   // magic, version, 18 config fields
constexpr size_t kCkptLayer = 11;  // fields per layer

}  // namespace

int kvevict_checkpoint_bytes(kvevict_t h, size_t *bytes)
{
    if (!h || !bytes) return KVEVICT_ERR_INVALID_ARG;
    *bytes = checkpoint_record(h).size() * sizeof(int64_t);
    return KVEVICT_OK;
}

int kvevict_checkpoint_save(kvevict_t h, void *dst, size_t bytes)
{
    NvtxRange nvtx("kvevict_checkpoint_save");
    if (!h || !dst) return KVEVICT_ERR_INVALID_ARG;
    const std::vector<int64_t> r = checkpoint_record(h);
    if (bytes < r.size() * sizeof(int64_t)) return KVEVICT_ERR_CAPACITY;
    std::memcpy(dst, r.data(), r.size() * sizeof(int64_t));
    return KVEVICT_OK;
}

int kvevict_checkpoint_restore(kvevict_t h, const void *src, size_t bytes)
{
    NvtxRange nvtx("kvevict_checkpoint_restore");
    if (!h || !src) return KVEVICT_ERR_INVALID_ARG;
    const std::vector<int64_t> mine = checkpoint_record(h);
    if (bytes != mine.size() * sizeof(int64_t)) return KVEVICT_ERR_INVALID_ARG;
    std::vector<int64_t> r(mine.size());
    std::memcpy(r.data(), src, bytes);
    // same format and the same configuration, field by field
    if (!std::equal(r.begin(), r.begin() + kCkptHead, mine.begin())) return KVEVICT_ERR_INVALID_ARG;
    const int rc = kvevict_sync(h);  // no call of this handle in flight while its counters change
    if (rc) return rc;
    const int64_t *f = r.data() + kCkptHead;
    for (LayerState &ls : h->layers) {
        ls = LayerState{};  // (a trace set on this handle is dropped)
        ls.prompt_len = static_cast<int>(f[0]);
        ls.t = static_cast<int>(f[1]);
        ls.count = static_cast<int>(f[2]);
        ls.n_gen = static_cast<int>(f[3]);
        ls.cut_done = f[4] != 0;
        ls.fl_idx = static_cast<int>(f[5]);
        ls.fill_left = static_cast<int>(f[6]);
        ls.n_rec = static_cast<int>(f[7]);
        ls.blk_left = static_cast<int>(f[8]);
        ls.blk_next = static_cast<int>(f[9]);
        ls.blk_uniform = f[10] != 0;
        f += kCkptLayer;
    }
    h->stats.decode_steps = f[0];
    h->stats.prefill_tokens = f[1];
    h->stats.evictions = f[2];
    h->stats.cuts = f[3];
    h->last_layer = -1;  // the state buffer was just written by the caller: no early prefetch
    return KVEVICT_OK;
}

int kvevict_select_victims(kvevict_t h, int layer, const float *scores, int32_t *victims)
{
    NvtxRange nvtx("kvevict_select_victims");
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    if (h->cfg.policy != KVEVICT_H2O) return KVEVICT_ERR_INVALID_ARG;
    if (!scores || !victims || !aligned16(scores) || (reinterpret_cast<uintptr_t>(victims) & 3u))
        return KVEVICT_ERR_INVALID_ARG;
    const LayerState &ls = h->layers[layer];
    SelectParams sp{};
    sp.score = scores;
    sp.pos = at<int32_t>(h, h->L.off_pos) + static_cast<size_t>(layer) * h->L.layer_pslots;
    sp.victim = victims;
    sp.C = h->L.C;
    sp.cstride = h->L.Cs;
    sp.n_active = h->L.C;  // empty slots hold position -1: never a candidate
    sp.n_sink = h->cfg.n_sink;
    sp.n_recent = h->cfg.n_recent;
    sp.p = ls.prompt_len + ls.t;
    int rc = cuda_status(launch_h2o_select(sp, static_cast<int>(h->L.units), h->stream));
    if (rc) return rc;
    h->last_layer = -1;  // a launch that is not a decode step of any layer came last
    return KVEVICT_OK;
}

int kvevict_probe_wait_timeout(kvevict_t h)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    return cuda_status(launch_wait_timeout_probe(at<uint32_t>(h, h->L.off_err), h->stream));
}

int kvevict_evicted_mass(kvevict_t h, int layer, double *dst, int dst_is_device)
{
    if (!h || !dst) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    if (!scored(h->cfg.policy)) return KVEVICT_ERR_INVALID_ARG;
    const size_t n = h->L.units;
    cudaError_t e = cudaMemcpyAsync(dst, at<double>(h, h->L.off_ledger) + static_cast<size_t>(layer) * n, n * 8,
                                    dst_is_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess && !dst_is_device) e = cudaStreamSynchronize(h->stream);
    return cuda_status(e);
}

int kvevict_score_scales(kvevict_t h, int layer, float *dst, int dst_is_device)
{
    if (!h || !dst) return KVEVICT_ERR_INVALID_ARG;
    if (!h->cfg.score_int8) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const Layout &L = h->L;
    const float *src = at<float>(h, L.off_qscale) + static_cast<size_t>(layer) * L.units;
    cudaError_t e = cudaMemcpyAsync(dst, src, L.units * 4,
                                    dst_is_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess && !dst_is_device) e = cudaStreamSynchronize(h->stream);
    return cuda_status(e);
}

int kvevict_slot_pools(kvevict_t h, int layer, uint8_t *dst, int dst_is_device)
{
    if (!h || !dst) return KVEVICT_ERR_INVALID_ARG;
    if (h->cfg.policy != KVEVICT_H2O_POOLS) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const Layout &L = h->L;
    const void *src = at<uint8_t>(h, L.off_pool) + static_cast<size_t>(layer) * L.units * L.Ps;
    cudaError_t e = cudaMemcpy2DAsync(dst, L.C, src, L.Ps, L.C, L.units,
                                      dst_is_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess && !dst_is_device) e = cudaStreamSynchronize(h->stream);
    return cuda_status(e);
}

int kvevict_set_trace(kvevict_t h, int layer, int32_t *dev_buf, int n_steps)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    if (dev_buf && (n_steps < 0 || !aligned16(dev_buf))) return KVEVICT_ERR_INVALID_ARG;
    LayerState &ls = h->layers[layer];
    ls.trace = dev_buf;
    ls.trace_len = dev_buf ? n_steps : 0;
    ls.trace_t = 0;
    return KVEVICT_OK;
}

int kvevict_layer_state(kvevict_t h, int layer, int *prompt_len, int *steps, int *count)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    const LayerState &ls = h->layers[layer];
    if (prompt_len) *prompt_len = ls.prompt_len;
    if (steps) *steps = ls.t;
    if (count) *count = h->cfg.policy == KVEVICT_RANDOM ? ls.prompt_len + ls.n_gen : ls.count;
    return KVEVICT_OK;
}

int kvevict_set_split(kvevict_t h, int split)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (split == 0) {
        h->split = auto_split(h);
        auto_tail(h);
        h->stats.tail_split = h->tail_split ? 1 : 0;
    } else {
        if (split < 1 || split > kMaxSplit || (split & (split - 1))) return KVEVICT_ERR_INVALID_ARG;
        if (split > 1 && h->cfg.score_int8) return KVEVICT_ERR_INVALID_ARG;  // one CTA per unit
        // an explicit split keeps tail splitting only where it was asked for
        const bool tail = h->tail_req == 1;
        if (decode_smem(h, split, holes_policy(h->cfg), nullptr, tail) > kMaxSmem) return KVEVICT_ERR_INVALID_ARG;
        h->split = split;
        h->tail_split = tail;
        h->stats.tail_split = tail ? 1 : 0;
    }
    h->stats.split = h->split;
    return KVEVICT_OK;
}

int kvevict_set_partials_alias(kvevict_t h, int mode)
{
    if (!h || mode < -1 || mode > 1) return KVEVICT_ERR_INVALID_ARG;
    h->alias_req = mode;
    return KVEVICT_OK;
}

int kvevict_set_tie_audit(kvevict_t h, int on)
{
    if (!h || on < 0 || on > 1) return KVEVICT_ERR_INVALID_ARG;
    if (on && h->cfg.policy != KVEVICT_H2O) return KVEVICT_ERR_INVALID_ARG;
    h->tie_audit = on == 1;
    return KVEVICT_OK;
}

int kvevict_near_ties(kvevict_t h, int layer, uint64_t *out)
{
    if (!h || !out) return KVEVICT_ERR_INVALID_ARG;
    if (layer < 0 || layer >= h->cfg.n_layers) return KVEVICT_ERR_STATE;
    *out = 0;
    if (!scored(h->cfg.policy)) return KVEVICT_OK;
    unsigned long long v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, at<unsigned long long>(h, h->L.off_tie) + layer, sizeof v,
                                    cudaMemcpyDeviceToHost, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_status(e);
    *out = v;
    return KVEVICT_OK;
}

int kvevict_set_tail_split(kvevict_t h, int on)
{
    if (!h || on < -1 || on > 1) return KVEVICT_ERR_INVALID_ARG;
    if (on == 1) {
        if (h->cfg.score_int8) return KVEVICT_ERR_INVALID_ARG;  // INT8 scores: one CTA per unit
        DecodeKernelInfo ki;
        if (!decode_kernel(h->cfg.dtype, h->cfg.head_dim, h->L.G, holes_policy(h->cfg), h->use_mma, &ki) || !ki.flex)
            return KVEVICT_ERR_INVALID_ARG;  // built into the one-CTA-per-SM kernels only
        if (decode_smem(h, h->split, holes_policy(h->cfg), nullptr, true) > kMaxSmem)
            return KVEVICT_ERR_INVALID_ARG;  // a whole unit does not fit one CTA
    }
    h->tail_req = on;
    if (on >= 0) {
        h->tail_split = on == 1;
    } else {  // automatic: from the automatic split
        h->split = auto_split(h);
        auto_tail(h);
        h->stats.split = h->split;
    }
    h->stats.tail_split = h->tail_split ? 1 : 0;
    return KVEVICT_OK;
}

int kvevict_set_path(kvevict_t h, int path)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (path < 0 || path > 2) return KVEVICT_ERR_INVALID_ARG;
    if (path == 2 && !mma_possible(h->cfg)) return KVEVICT_ERR_INVALID_ARG;
    const bool mma = path == 0 ? mma_auto(h->cfg) : path == 2;
    const bool old = h->use_mma;
    h->use_mma = mma;
    if (decode_smem(h, h->split, h->cfg.policy == KVEVICT_RANDOM) > kMaxSmem) {
        h->use_mma = old;
        return KVEVICT_ERR_INVALID_ARG;
    }
    h->path_req = path;
    return KVEVICT_OK;
}

int kvevict_set_ring(kvevict_t h, int stages)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (stages != 0 && (stages < kMinStages || stages > kMaxStages)) return KVEVICT_ERR_INVALID_ARG;
    h->ring_req = stages;
    return KVEVICT_OK;
}

int kvevict_set_clusters(kvevict_t h, int clusters)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    if (clusters < 0) return KVEVICT_ERR_INVALID_ARG;
    h->clusters_req = clusters;
    return KVEVICT_OK;
}

int kvevict_get_stats(kvevict_t h, kvevict_stats *out)
{
    if (!h || !out) return KVEVICT_ERR_INVALID_ARG;
    *out = h->stats;
    out->evicted_mass = 0.0;
    if (scored(h->cfg.policy)) {  // the ledger of every layer and unit, summed on the host in fp64
        std::vector<double> led(static_cast<size_t>(h->cfg.n_layers) * h->L.units);
        cudaError_t e = cudaMemcpyAsync(led.data(), h->state + h->L.off_ledger, led.size() * 8,
                                        cudaMemcpyDeviceToHost, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e != cudaSuccess) return cuda_status(e);
        for (double v : led) out->evicted_mass += v;
    }
    out->clusters = h->configured[0].clusters ? h->configured[0].clusters : h->configured[1].clusters;
    out->tensor_cores = h->use_mma ? 1 : 0;
    out->ring_stages = h->configured[0].nst ? h->configured[0].nst : h->configured[1].nst;
    out->partials_alias = (h->configured[0].nst ? h->configured[0].alias : h->configured[1].alias) ? 1 : 0;
    out->near_ties = 0;
    if (scored(h->cfg.policy)) {
        std::vector<unsigned long long> cnt(h->cfg.n_layers);
        cudaError_t e = cudaMemcpyAsync(cnt.data(), at<unsigned long long>(h, h->L.off_tie),
                                        cnt.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost, h->stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
        if (e != cudaSuccess) return cuda_status(e);
        for (unsigned long long v : cnt) out->near_ties += static_cast<int64_t>(v);
    }
    return KVEVICT_OK;
}

int kvevict_check(kvevict_t h, uint32_t *device_error)
{
    NvtxRange nvtx("kvevict_check");
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_status(e);
    uint32_t w = 0;
    e = cudaMemcpy(&w, h->state + h->L.off_err, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->state + h->L.off_err, 0, 4, h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_status(e);
    if (device_error) *device_error = w;
    return w ? KVEVICT_ERR_DEVICE : KVEVICT_OK;
}

const char *kvevict_strerror(int code)
{
    switch (code) {
    case KVEVICT_OK: return "ok";
    case KVEVICT_ERR_INVALID_ARG: return "invalid argument";
    case KVEVICT_ERR_CAPACITY: return "capacity exceeded";
    case KVEVICT_ERR_STATE: return "call out of order or layer out of range";
    case KVEVICT_ERR_CUDA: return "CUDA runtime error";
    case KVEVICT_ERR_DEVICE: return "device error bits set";
    default: return "unknown status";
    }
}

void kvevict_destroy(kvevict_t h) { delete h; }

}  // extern "C"
