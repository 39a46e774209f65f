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

#include "api_internal.h"
#include "kvevict.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB

// In host code this name stands for the array but is not its device address:
// a kernel given it would fault or, where the GPU can reach host memory,
// silently use the wrong memory. Host code passes the address that
// cudaGetSymbolAddress returns for the handle's device instead.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" int kvevict_static_scratch_address(int device, void **out)
{
    if (device < 0 || device >= kMaxDevices || !out) return KVEVICT_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[device]) {
        int cur = -1;
        cudaError_t e = cudaGetDevice(&cur);
        if (e == cudaSuccess && cur != device) e = cudaSetDevice(device);
        void *p = nullptr;
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_scratch);
        if (cur >= 0 && cur != device) {
            const cudaError_t e2 = cudaSetDevice(cur);  // the caller's device, whatever happened
            if (e == cudaSuccess) e = e2;
        }
        if (e != cudaSuccess || !p) {
            std::fprintf(stderr, "kvevict: static scratch: address lookup on device %d failed (%s)\n", device,
                         cudaGetErrorString(e));
            return KVEVICT_ERR_CUDA;
        }
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return KVEVICT_OK;
}

extern "C" int kvevict_prefill_scored_static(kvevict_t h, int layer, const void *Q, const void *K, const void *V,
                                             int prompt_len)
{
    // the same argument and state checks as kvevict_prefill_scored, first
    int rc = kvevict_prefill_scored_check(h, layer, Q, K, V, prompt_len);
    if (rc) return rc;
    // the scratch array is per device: the handle's device must be the current one
    const int dev = kvevict_handle_device(h);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != dev) {
        std::fprintf(stderr,
                     "kvevict: prefill_scored_static: the handle's state is on device %d but device %d is "
                     "current; make the handle's device current first\n",
                     dev, cur);
        return KVEVICT_ERR_INVALID_ARG;
    }
    size_t need = 0;
    rc = kvevict_prefill_scored_workspace_bytes(h, prompt_len, &need);
    if (rc) return rc;
    if (need > kStaticScratchBytes) {
        std::fprintf(stderr,
                     "kvevict: prefill_scored_static: this prompt needs %zu bytes of scratch, the static area "
                     "holds %zu; use kvevict_prefill_scored with a workspace instead\n",
                     need, kStaticScratchBytes);
        return KVEVICT_ERR_CAPACITY;
    }
    // resolved when the handle was created; this only reads the cached address
    void *scratch = nullptr;
    rc = kvevict_static_scratch_address(dev, &scratch);
    if (rc) return rc;
    // Nothing in the scratch needs to start at zero: every entry whose value is
    // used is written by the same call before it is read (stale entries past
    // the prompt's end are read only under a mask), and the work counters at
    // its end are zeroed by kvevict_prefill_scored on the stream.
    return kvevict_prefill_scored(h, layer, Q, K, V, prompt_len, scratch, kStaticScratchBytes);
}
