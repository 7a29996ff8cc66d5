// Cascade decode's shared-prefix pass for 8-bit pools (FP8 E4M3 / INT8
// codes) with f16 queries (one translation unit per query type).
#include "decode_prefix.cuh"

namespace pagedkv {

cudaError_t prefix_q8_attrs_f16(const kv_pool& pool, int group, size_t smem, int* occ) {
    return dec::by_q8_shape<__half>(pool, group, [&]<typename T, int G, int BS, class Pol>() {
        return dec::prefix_attrs<T, G, BS, Pol>(smem, occ);
    });
}

cudaError_t prefix_q8_launch_f16(const kv_pool& pool, int group, const dec::PParams& p,
                                  size_t smem, int grid, cudaStream_t stream) {
    return dec::by_q8_shape<__half>(pool, group, [&]<typename T, int G, int BS, class Pol>() {
        return dec::prefix_launch<T, G, BS, Pol>(pool.tmap_k_swz, pool.tmap_v_swz, p, smem, grid,
                                                 stream);
    });
}

}  // namespace pagedkv
