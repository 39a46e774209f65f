// aux_kernels.cu -- prompt prefill and the Random Attention periodic cut.
#include <algorithm>
#include <climits>

#include <cuda_fp16.h>

#include "aux_kernels.h"
#include "device_common.cuh"

namespace kvevict {

// ---------------------------------------------------------------- prefill
// Prompt tokens enter with score 0 and no attention. For H2O (all scores
// equal, ties to the older position) and StreamingLLM that keeps the first
// n_sink positions in slots 0..n_sink-1 and the newest C - n_sink in ring
// order: slot(p) = n_sink + (p - n_sink) mod (C - n_sink). Two-pool H2O is a
// ring without sinks, of n_recent or C slots, its older part flagged as heavy
// hitters. Random keeps every prompt token: slot(p) = p. Rows of this chunk: range A = [a0, a1) (sinks or,
// for Random, everything), range B = [b0, b1) (kept ring rows). One warp per
// row, 16-byte vector copies.
__global__ void __launch_bounds__(256) prefill_kernel(const PrefillParams P)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int idx = blockIdx.x * 8 + warp;
    const int na = P.a1 - P.a0;
    int i;
    if (idx < na) i = P.a0 + idx;
    else if (idx - na < P.b1 - P.b0) i = P.b0 + (idx - na);
    else return;
    const int p = P.p0 + i;
    const int slot = (P.ring_len > 0 && p >= P.n_sink) ? P.n_sink + (p - P.n_sink) % P.ring_len : p;
    const size_t unit = static_cast<size_t>(blockIdx.z) * P.Hkv + blockIdx.y;
    const size_t row_bytes = static_cast<size_t>(P.head_dim) * P.elem_bytes;
    const int vecs = static_cast<int>(row_bytes / 16);
    const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.K) +
                                                      (unit * P.n_tok + i) * row_bytes);
    const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.V) +
                                                      (unit * P.n_tok + i) * row_bytes);
    uint4 *kd = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.kc) + (unit * P.C + slot) * row_bytes);
    uint4 *vd = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.vc) + (unit * P.C + slot) * row_bytes);
    for (int v = lane; v < vecs; v += 32) {
        kd[v] = ks[v];
        vd[v] = vs[v];
    }
    if (lane == 0) {
        P.pos[unit * P.cstride + slot] = p;
        if (P.pool) P.pool[unit * P.pstride + slot] = p < P.hh_below ? 1 : 0;
        if (P.score) {
            if (P.score_int8) static_cast<uint8_t *>(P.score)[unit * P.cstride + slot] = 0;  // code 0
            else if (P.score_half) static_cast<uint16_t *>(P.score)[unit * P.cstride + slot] = 0;  // +0 in binary16
            else static_cast<float *>(P.score)[unit * P.cstride + slot] = 0.f;
        }
    }
}

// ------------------------------------------------------------ random cut
// Random Attention ("Random Attention" summary, 方法): the prompt is kept;
// when a unit holds K + r generated tokens, each unit independently evicts r
// of them uniformly at random. Every generated token gets a fresh 64-bit
// Philox key for this step; the r smallest (key, position) leave. One CTA per
// unit: keys into shared memory, bitonic sort of (key, position << 32 | slot),
// then the r freed slots are written to the unit's free list in ascending
// slot order (the next r decode steps fill them lowest first).
__global__ void __launch_bounds__(kCutThreads) random_cut_kernel(const CutParams P)
{
    extern __shared__ __align__(16) uint64_t cut_smem[];
    uint64_t *key = cut_smem;
    uint64_t *aux = cut_smem + P.n_pow2;
    int32_t *freed = reinterpret_cast<int32_t *>(cut_smem + 2 * static_cast<size_t>(P.n_pow2));
    const int tid = threadIdx.x;
    const int h = blockIdx.x, b = blockIdx.y;
    const size_t unit = static_cast<size_t>(b) * P.Hkv + h;
    int32_t *pos = P.pos + unit * P.cstride;

    grid_dependency_wait();

    for (int i = tid; i < P.n_pow2; i += blockDim.x) {
        if (i < P.n_cand) {
            const int slot = P.first_slot + i;
            const int32_t ps = pos[slot];
            key[i] = random_evict_key(P.seed, static_cast<uint32_t>(b), static_cast<uint32_t>(P.layer),
                                      static_cast<uint32_t>(h), static_cast<uint32_t>(P.step),
                                      static_cast<uint32_t>(ps));
            aux[i] = (static_cast<uint64_t>(static_cast<uint32_t>(ps)) << 32) | static_cast<uint32_t>(slot);
        } else {
            key[i] = ~0ull;
            aux[i] = ~0ull;
        }
    }
    __syncthreads();
    // Bitonic sort, ascending by (key, aux).
    for (int k = 2; k <= P.n_pow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P.n_pow2; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const bool up = (i & k) == 0;
                    const uint64_t ka = key[i], kb = key[ixj], xa = aux[i], xb = aux[ixj];
                    const bool a_gt_b = ka > kb || (ka == kb && xa > xb);
                    if (a_gt_b == up) {
                        key[i] = kb; key[ixj] = ka;
                        aux[i] = xb; aux[ixj] = xa;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < P.r; i += blockDim.x) freed[i] = static_cast<int32_t>(aux[i] & 0xFFFFFFFFu);
    __syncthreads();
    // Ascending slot order by rank counting (slots are distinct).
    for (int i = tid; i < P.r; i += blockDim.x) {
        const int32_t s = freed[i];
        int rnk = 0;
        for (int j = 0; j < P.r; ++j) rnk += freed[j] < s;
        P.freelist[unit * P.r + rnk] = s;
        pos[s] = -1;
    }
    // Zero the freed rows: until refilled they are masked out, and a zero
    // row is finite whatever value the evicted token held.
    const int vecs = P.row_bytes / 16;
    for (int i = tid; i < P.r * vecs; i += blockDim.x) {
        const size_t row = unit * P.C + freed[i / vecs];
        reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.kc) + row * P.row_bytes)[i % vecs] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.vc) + row * P.row_bytes)[i % vecs] = make_uint4(0, 0, 0, 0);
    }
}

// ------------------------------------------------- block-granular H2O
// Prompt admission for block-granular H2O ("Attention Sinks 与 KV Cache 淘汰
// 策略" section 5: whole blocks are released). Every prompt token enters with
// score 0, so when the cache is full the released block is the eligible one
// holding the oldest token: the blocks holding sinks never leave and the
// others are released round robin, each refilled by the next bs positions.
// Slot-centric: one warp per slot works out which position the slot holds
// at the end of the prompt (or none: the unfilled rest of the block released
// last) and copies its row.
__global__ void __launch_bounds__(256) prefill_block_kernel(const BlockPrefillParams P)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.x * 8 + warp;
    if (s >= P.C) return;
    const size_t unit = static_cast<size_t>(blockIdx.z) * P.Hkv + blockIdx.y;
    const int b = s / P.bs, o = s - b * P.bs, nb = P.C / P.bs;
    int src;
    if (P.n_tok <= P.C || b < P.nsb) {
        src = s < P.n_tok ? s : -1;
    } else {
        const int released = (P.n_tok - P.C + P.bs - 1) / P.bs;  // releases so far
        const int nr = nb - P.nsb, idx = b - P.nsb;
        if (released - 1 < idx) {
            src = s;  // never released: the original prompt position
        } else {
            const int last = idx + nr * ((released - 1 - idx) / nr);  // its last release (0-based)
            src = P.C + last * P.bs + o;
            if (src >= P.n_tok) src = -1;
        }
    }
    const int vecs = P.row_bytes / 16;
    uint4 *kd = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.kc) + (unit * P.C + s) * P.row_bytes);
    uint4 *vd = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.vc) + (unit * P.C + s) * P.row_bytes);
    const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.K) +
                                                      (unit * P.n_tok + (src < 0 ? 0 : src)) * P.row_bytes);
    const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(P.V) +
                                                      (unit * P.n_tok + (src < 0 ? 0 : src)) * P.row_bytes);
    for (int v = lane; v < vecs; v += 32) {
        kd[v] = src < 0 ? make_uint4(0, 0, 0, 0) : ks[v];
        vd[v] = src < 0 ? make_uint4(0, 0, 0, 0) : vs[v];
    }
    if (lane == 0) {
        P.pos[unit * P.cstride + s] = src;
        P.score[unit * P.cstride + s] = 0.f;
    }
}

// The release: among the blocks of bs consecutive slots whose tokens all lie
// outside the sinks and the recent window (n_sink <= pos <= p - n_recent), the
// one with the smallest (sum of scores, oldest position) leaves -- the block
// whose removal keeps the highest remaining cumulative score. Its slots are
// emptied (position -1, score 0, K/V rows zeroed so that every row a tile may
// touch is finite) and listed, ascending, in the unit's free list, which the
// next bs decode steps fill. One CTA per unit.
__global__ void __launch_bounds__(256) block_release_kernel(const BlockReleaseParams P)
{
    __shared__ uint64_t wkey[8];
    __shared__ int32_t wblk[8];
    __shared__ int32_t chosen;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t unit = blockIdx.x;
    const int32_t *pos = P.pos + unit * P.cstride;
    const float *sc = P.score + unit * P.cstride;
    const int nb = P.C / P.bs;
    uint64_t best = ~0ull;
    int32_t bblk = -1;
    for (int b = tid; b < nb; b += blockDim.x) {
        float sum = 0.f;
        int32_t mn = INT_MAX, mx = -1;
        bool full = true;
        for (int o = 0; o < P.bs; ++o) {
            const int32_t ps = pos[b * P.bs + o];
            if (ps < 0) {
                full = false;
                break;
            }
            sum += sc[b * P.bs + o];
            mn = min(mn, ps);
            mx = max(mx, ps);
        }
        if (!full || mn < P.n_sink || mx > P.p - P.n_recent) continue;
        const uint64_t key = (static_cast<uint64_t>(__float_as_uint(sum)) << 32) | static_cast<uint32_t>(mn);
        if (key < best) {
            best = key;
            bblk = b;
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const uint64_t ok = __shfl_xor_sync(0xffffffffu, best, off);
        const int32_t ob = __shfl_xor_sync(0xffffffffu, bblk, off);
        if (ok < best) {
            best = ok;
            bblk = ob;
        }
    }
    if (lane == 0) {
        wkey[warp] = best;
        wblk[warp] = bblk;
    }
    __syncthreads();
    if (tid == 0) {
        uint64_t k = ~0ull;
        int32_t bk = -1;
        for (int w = 0; w < static_cast<int>(blockDim.x / 32); ++w)
            if (wkey[w] < k) {
                k = wkey[w];
                bk = wblk[w];
            }
        chosen = bk;
        if (bk < 0) atomicOr(P.err, KVEVICT_DEV_NO_CANDIDATE);
    }
    __syncthreads();
    const int blk = chosen;
    if (blk >= 0 && tid == 0 && P.ledger) {  // the released tokens' scores leave the cache
        double m = 0.0;
        for (int o = 0; o < P.bs; ++o) m += static_cast<double>(sc[blk * P.bs + o]);
        P.ledger[unit] += m;
    }
    __syncthreads();  // the scores are read before they are cleared
    int32_t *posw = P.pos + unit * P.cstride;
    for (int o = tid; o < P.bs; o += blockDim.x) {
        P.freelist[unit * P.bs + o] = blk < 0 ? -1 : blk * P.bs + o;  // -1: the decode step drops its token
        if (blk >= 0) {
            posw[blk * P.bs + o] = -1;
            P.score[unit * P.cstride + blk * P.bs + o] = 0.f;
        }
    }
    if (blk < 0) return;
    const int vecs = P.row_bytes / 16;
    for (int i = tid; i < P.bs * vecs; i += blockDim.x) {
        const size_t row = unit * P.C + blk * P.bs + i / vecs;
        reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.kc) + row * P.row_bytes)[i % vecs] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(static_cast<uint8_t *>(P.vc) + row * P.row_bytes)[i % vecs] = make_uint4(0, 0, 0, 0);
    }
}

// Near-ties of one H2O step ("h2o: heavy-hitter oracle" summary, Algorithm 1:
// the greedy removal of the lowest-score candidate). For every unit whose
// step evicted a token: the smallest stored score among the candidates left
// (the step's candidate rule at position p: a token at ps >= n_sink and
// <= p - n_recent; the new token is never one) is the runner-up of the
// decision, since the step changes no other slot after its score pass. A
// unit counts when the runner-up's score is within `rel` of the evicted one's
// (|a - b| < rel max(a, b), equal scores included): there a different
// rounding of the scores could have chosen the other token. One CTA per unit.
__global__ void __launch_bounds__(256) tie_audit_kernel(const TieAuditParams P)
{
    __shared__ float wmin[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t unit = blockIdx.x;
    const int32_t *tr = P.trace + unit * 4;
    const int dest = tr[0], old_pos = tr[1];
    if (old_pos < 0) return;  // an empty slot took the token: no decision between tokens
    const float s1 = __int_as_float(tr[2]);
    const int32_t *pos = P.pos + unit * P.cstride;
    const float scl = P.score_int8 ? P.qscale[unit] : 0.f;
    float mn = INFINITY;
    for (int j = tid; j < P.n_active; j += blockDim.x) {
        const int32_t ps = pos[j];
        if (j == dest || ps < P.n_sink || ps > P.p - P.n_recent) continue;
        const size_t i = unit * P.cstride + j;
        const float s = P.score_int8   ? static_cast<float>(static_cast<const uint8_t *>(P.score)[i]) * scl
                        : P.score_half ? __half2float(static_cast<const __half *>(P.score)[i])
                                       : static_cast<const float *>(P.score)[i];
        mn = fminf(mn, s);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    if (lane == 0) wmin[warp] = mn;
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < static_cast<int>(blockDim.x / 32); ++w) mn = fminf(mn, wmin[w]);
        mn = fminf(mn, wmin[0]);
        if (mn != INFINITY && (mn == s1 || fabsf(mn - s1) < P.rel * fmaxf(mn, s1))) atomicAdd(P.count, 1ull);
    }
}

cudaError_t launch_tie_audit(const TieAuditParams &p, int units, cudaStream_t st)
{
    tie_audit_kernel<<<units, 256, 0, st>>>(p);
    return cudaGetLastError();
}

void launch_block_prefill(const BlockPrefillParams &p, int B, cudaStream_t st)
{
    dim3 grid((p.C + 7) / 8, p.Hkv, B);
    prefill_block_kernel<<<grid, 256, 0, st>>>(p);
}

cudaError_t launch_block_release(const BlockReleaseParams &p, int units, cudaStream_t st)
{
    block_release_kernel<<<units, 256, 0, st>>>(p);
    return cudaGetLastError();
}

__global__ void scores_to_f32_kernel(float *dst, const __half *src, int C, int cstride, size_t n)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t u = i / C, j = i - u * C;
        dst[i] = __half2float(src[u * cstride + j]);
    }
}

cudaError_t launch_scores_to_f32(float *dst, const void *src, int C, int cstride, size_t units, cudaStream_t st)
{
    const size_t n = units * C;
    const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
    scores_to_f32_kernel<<<blocks, 256, 0, st>>>(dst, static_cast<const __half *>(src), C, cstride, n);
    return cudaGetLastError();
}

__global__ void scores_int8_to_f32_kernel(float *dst, const uint8_t *src, const float *scale, int C, int cstride,
                                          size_t n)
{
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t u = i / C, j = i - u * C;
        dst[i] = static_cast<float>(src[u * cstride + j]) * scale[u];
    }
}

cudaError_t launch_scores_int8_to_f32(float *dst, const void *src, const float *scale, int C, int cstride,
                                      size_t units, cudaStream_t st)
{
    const size_t n = units * C;
    if (n == 0) return cudaSuccess;
    const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 4096));
    scores_int8_to_f32_kernel<<<blocks, 256, 0, st>>>(dst, static_cast<const uint8_t *>(src), scale, C, cstride, n);
    return cudaGetLastError();
}

// Failure detection, exercised without a fault: one thread waits through the
// pipelines' bounded wait on an mbarrier that nothing arrives at. The wait
// gives up after its limit; the kernel records KVEVICT_DEV_WAIT_TIMEOUT and
// ends normally, so the context stays usable.
__global__ void wait_timeout_probe_kernel(uint32_t *err)
{
    __shared__ alignas(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    mbar_fence_init();
    if (!mbar_wait(&bar, 0)) atomicOr(err, KVEVICT_DEV_WAIT_TIMEOUT);
}

cudaError_t launch_wait_timeout_probe(uint32_t *err, cudaStream_t st)
{
    wait_timeout_probe_kernel<<<1, 32, 0, st>>>(err);
    return cudaGetLastError();
}

void launch_prefill(const PrefillParams &p, int rows, int B, cudaStream_t st)
{
    if (rows <= 0) return;
    dim3 grid((rows + 7) / 8, p.Hkv, B);
    prefill_kernel<<<grid, 256, 0, st>>>(p);
}

size_t cut_smem_bytes(int n_pow2, int r)
{
    return 2 * sizeof(uint64_t) * static_cast<size_t>(n_pow2) + sizeof(int32_t) * static_cast<size_t>(r);
}

cudaError_t launch_random_cut(const CutParams &p, int B, cudaStream_t st)
{
    const size_t smem = cut_smem_bytes(p.n_pow2, p.r);
    cudaError_t e = cudaFuncSetAttribute(random_cut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.Hkv, B, 1);
    cfg.blockDim = dim3(kCutThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, random_cut_kernel, p);
}

}  // namespace kvevict
