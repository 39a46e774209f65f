// api_static.cu -- kvevict_prefill_scored_static: the Q-seeded prefill with
// its scratch in a fixed device array instead of caller-provided memory.
//
// Why: some callers cannot allocate device memory when they prefill. A
// serving framework that reserved the GPU's free memory for its own pool at
// start-up leaves nothing for a cudaMalloc, and a caller on a latency-bound
// path cannot afford the device-wide synchronisation that cudaMalloc and
// cudaFree may cause. This entry point needs no allocation: its scratch (the
// per-query softmax normalisers and the per-key scores of the prompt) lives in
// the array below, which every GPU that loads the library holds until the
// process exits.
#include <cstdio>
#include <mutex>

#include "kvevict.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB

// In host code this name stands for the array but is not its device address:
// a kernel given it would fault or, where the GPU can reach host memory,
// silently use the wrong memory. Host code passes the address that
// cudaGetSymbolAddress returns for the current device instead.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// The scratch array's device address on the current device; resolved once per
// device, on the first call made with that device current.
int scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        std::fprintf(stderr, "kvevict: prefill_scored_static: no usable current device (%s)\n",
                     cudaGetErrorString(e));
        return KVEVICT_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p) {
            std::fprintf(stderr, "kvevict: prefill_scored_static: cudaGetSymbolAddress failed (%s)\n",
                         cudaGetErrorString(e));
            return KVEVICT_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KVEVICT_OK;
}

}  // namespace

extern "C" int kvevict_prefill_scored_static(kvevict_t h, int layer, const void *Q, const void *K, const void *V,
                                             int prompt_len)
{
    if (!h) return KVEVICT_ERR_INVALID_ARG;
    size_t need = 0;
    int rc = kvevict_prefill_scored_workspace_bytes(h, prompt_len, &need);
    if (rc) return rc;
    if (need > kStaticScratchBytes) {
        std::fprintf(stderr,
                     "kvevict: prefill_scored_static: this prompt needs %zu bytes of scratch, the static area "
                     "holds %zu; use kvevict_prefill_scored with a workspace instead\n",
                     need, kStaticScratchBytes);
        return KVEVICT_ERR_CAPACITY;
    }
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc) return rc;
    // Nothing in the scratch needs to start at zero: every entry whose value is
    // used is written by the same call before it is read (stale entries past
    // the prompt's end are read only under a mask).
    return kvevict_prefill_scored(h, layer, Q, K, V, prompt_len, scratch, kStaticScratchBytes);
}
