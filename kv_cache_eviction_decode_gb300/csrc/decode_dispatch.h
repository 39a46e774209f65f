// decode_dispatch.h -- lookup of the decode-step kernel instantiation for a
// (dtype, head_dim, group size, holes) combination.
#pragma once

#include <cstddef>

#include <cuda_runtime.h>

namespace kvevict {

struct DecodeKernelInfo {
    const void *fn;                    // __global__ decode_step_kernel<...>
    size_t (*fixed_bytes)(int zcap, int n_aux, bool alias);  // dynamic shared memory besides the ring (n_aux: 0..3;
                                                             // alias: warp partials over the logits)
    bool (*alias_fits)(int zcap);      // the warp partials fit in the logit area
    int (*zcap)(int max_slots_per_cta);
    int stage_bytes;   // one ring stage
    int ctas_per_sm;   // register-limited target occupancy (1 or 2)
    int threads;       // CTA size
    bool flex;         // tail splitting and partials over the logits are built in
};

// dtype: 0 fp32, 1 bf16; mma: the tensor-core path (bf16 only). Returns
// false if the combination is not built.
bool decode_kernel_f32(int head_dim, int G, bool holes, DecodeKernelInfo *out);
bool decode_kernel_bf16(int head_dim, int G, bool holes, bool mma, DecodeKernelInfo *out);

struct SelectParams;
// The H2O selector alone (one CTA per unit), on the decode kernel's CTA shape.
cudaError_t launch_h2o_select(const SelectParams &p, int units, cudaStream_t stream);

inline bool decode_kernel(int dtype, int head_dim, int G, bool holes, bool mma, DecodeKernelInfo *out)
{
    if (dtype == 0) return !mma && decode_kernel_f32(head_dim, G, holes, out);
    return decode_kernel_bf16(head_dim, G, holes, mma, out);
}

}  // namespace kvevict
