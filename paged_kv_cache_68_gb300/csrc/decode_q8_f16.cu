// Decode kernels for 8-bit pools (FP8 E4M3 / INT8 codes) with f16 queries and
// outputs (one translation unit per query type).
#include "decode_kernel.cuh"

namespace pagedkv {

cudaError_t decode_dispatch_q8_f16(const kv_pool& pool, const DecodeCall& call,
                                  const DecodePlan& plan, cudaStream_t stream) {
    return dec::dispatch_q8<__half>(pool, call, plan, stream);
}

cudaError_t decode_attrs_q8_f16(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm) {
    return dec::attrs_q8<__half>(pool, group, smem, ctas_per_sm);
}

}  // namespace pagedkv
