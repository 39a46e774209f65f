// decode_f32.cu -- decode-step kernel instantiations for float caches.
#include "decode_dispatch.h"
#include "decode_kernel.cuh"

namespace kvevict {
namespace {

template <int D, int G, bool H, bool MMA> DecodeKernelInfo info()
{
    using L = DecodeLayout<float, D, G, MMA>;
    return DecodeKernelInfo{reinterpret_cast<const void *>(&decode_step_kernel<float, D, G, H, MMA>),
                            [](int zc, int n_aux, bool alias) { return L::fixed_bytes(zc, n_aux, alias); },
                            [](int zc) { return L::alias_fits(zc); }, [](int n) { return L::zcap(n); },
                            L::kStageBytes, min_blocks<G, MMA>(), L::kThreads, flex_layout<G, MMA>()};
}

template <int D, bool H, bool MMA> bool pick_g(int G, DecodeKernelInfo *out)
{
    switch (G) {
    case 1: *out = info<D, 1, H, MMA>(); return true;
    case 2: *out = info<D, 2, H, MMA>(); return true;
    case 4: *out = info<D, 4, H, MMA>(); return true;
    case 8: *out = info<D, 8, H, MMA>(); return true;
    default: return false;
    }
}

}  // namespace

cudaError_t launch_h2o_select(const SelectParams &p, int units, cudaStream_t stream)
{
    constexpr int kWarps = warps_for<1, false>();  // the decode kernel's warps per CTA
    if (units < 1) return cudaSuccess;
    h2o_select_kernel<kWarps><<<units, kWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

bool decode_kernel_f32(int head_dim, int G, bool holes, DecodeKernelInfo *out)
{
    if (head_dim == 64) return holes ? pick_g<64, true, false>(G, out) : pick_g<64, false, false>(G, out);
    if (head_dim == 128) return holes ? pick_g<128, true, false>(G, out) : pick_g<128, false, false>(G, out);
    return false;
}

}  // namespace kvevict
