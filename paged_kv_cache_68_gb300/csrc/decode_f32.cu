// Decode kernels for f32 pools (one translation unit per element type so the
// instantiations compile in parallel).
#include "decode_kernel.cuh"

namespace pagedkv {

cudaError_t decode_dispatch_f32(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                               cudaStream_t stream) {
    return dec::dispatch<float>(pool, call, plan, stream);
}

cudaError_t decode_attrs_f32(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm) {
    return dec::attrs<float>(pool, group, smem, ctas_per_sm);
}

}  // namespace pagedkv
