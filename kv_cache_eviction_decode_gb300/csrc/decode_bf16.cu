// decode_bf16.cu -- decode-step kernel instantiations for __nv_bfloat16 caches.
#include "decode_dispatch.h"
#include "decode_kernel.cuh"

namespace kvevict {
namespace {

template <int D, int G, bool H, bool MMA> DecodeKernelInfo info()
{
    using L = DecodeLayout<__nv_bfloat16, D, G, MMA>;
    return DecodeKernelInfo{reinterpret_cast<const void *>(&decode_step_kernel<__nv_bfloat16, D, G, H, MMA>),
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

bool decode_kernel_bf16(int head_dim, int G, bool holes, bool mma, DecodeKernelInfo *out)
{
    if (head_dim == 64) {
        if (mma) return holes ? pick_g<64, true, true>(G, out) : pick_g<64, false, true>(G, out);
        return holes ? pick_g<64, true, false>(G, out) : pick_g<64, false, false>(G, out);
    }
    if (head_dim == 128) {
        if (mma) return holes ? pick_g<128, true, true>(G, out) : pick_g<128, false, true>(G, out);
        return holes ? pick_g<128, true, false>(G, out) : pick_g<128, false, false>(G, out);
    }
    return false;
}

}  // namespace kvevict
