// Decode kernels for f16 pools (one translation unit per element type so the
// instantiations compile in parallel).
#include "decode_kernel.cuh"

namespace pagedkv {

cudaError_t decode_dispatch_f16(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                               cudaStream_t stream) {
    return dec::dispatch<__half>(pool, call, plan, stream);
}

cudaError_t decode_attrs_f16(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm) {
    return dec::attrs<__half>(pool, group, smem, ctas_per_sm);
}

}  // namespace pagedkv
