// Paged (chunked) prefill: host-side checks, the per-call query tensor map and
// the launch of the tcgen05 kernel (prefill_kernel.cuh).
#include <cstdint>

#include "prefill_kernel.cuh"

namespace pagedkv {
namespace pf {

// FMT: -1 for 16-bit pools, else the 8-bit pool's code format.
template <typename T, int G, int FMT>
cudaError_t launch_typed(const kv_pool& pool, const PrefillCall& c, cudaStream_t stream) {
    constexpr bool Q8 = FMT >= 0;
    constexpr int QT = BM / G;
    // q viewed as [T rows][Hq][D]; one box = QT rows x the group's G heads x
    // 64 dims (128 bytes, swizzled), so the tile lands as row = query * G + head
    CUtensorMap tmap_q;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)c.num_q_heads,
                                (cuuint64_t)c.num_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2u, (cuuint64_t)c.num_q_heads * D * 2u};
    const cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)QT};
    if (!encode_tiled_map(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(c.q), dims,
                          strides, box, true))
        return cudaErrorInvalidValue;
    // K/V boxes of min(bs, BN) rows: the pool's swizzled maps (box = one
    // block; 8-bit pools: 128 code bytes = all dims) when a block fits a KV
    // tile, else maps with BN-row boxes
    const CUtensorMap* mk = &pool.tmap_k_swz;
    const CUtensorMap* mv = &pool.tmap_v_swz;
    CUtensorMap tk, tv;
    if (pool.block_size > BN) {
        const cuuint64_t elt = Q8 ? 1u : 2u;
        const cuuint64_t kdims[3] = {(cuuint64_t)D, (cuuint64_t)pool.num_kv_heads,
                                     (cuuint64_t)pool.num_blocks * (cuuint64_t)pool.block_size};
        const cuuint64_t kstr[2] = {(cuuint64_t)D * elt, (cuuint64_t)pool.num_kv_heads * D * elt};
        const cuuint32_t kbox[3] = {Q8 ? 128u : 64u, 1u, (cuuint32_t)BN};
        const CUtensorMapDataType dt = Q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
        if (!encode_tiled_map(&tk, dt, 3, pool.k, kdims, kstr, kbox, true) ||
            !encode_tiled_map(&tv, dt, 3, pool.v, kdims, kstr, kbox, true))
            return cudaErrorInvalidValue;
        mk = &tk;
        mv = &tv;
    }
    auto kern = paged_prefill<T, G, FMT>;
    constexpr uint32_t smem_bytes = Lay<Q8>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes);
    if (e != cudaSuccess) return e;
    Params p;
    p.q = c.q;
    p.out = c.out;
    p.cu_seqlens = c.cu_seqlens;
    p.block_tables = c.block_tables;
    p.seq_lens = c.seq_lens;
    p.err = pool.d_err;
    p.num_tokens = c.num_tokens;
    p.max_blocks = c.max_blocks;
    p.batch = c.batch;
    p.num_q_heads = c.num_q_heads;
    p.num_blocks = pool.num_blocks;
    p.bs = pool.block_size;
    p.max_q = c.max_query_len;
    p.box_rows = pool.block_size < BN ? pool.block_size : BN;
    // FP8: the K scale multiplies every score, the V scale the output
    const bool fp8 = pool.cache_dtype == KV_FP8_E4M3;
    p.qscale = c.scale * 1.4426950408889634f * (fp8 ? pool.fp8_k_scale : 1.f);
    p.vscale = fp8 ? pool.fp8_v_scale : 1.f;
    p.k_scales = pool.k_scales;
    p.v_scales = pool.v_scales;
    p.num_kv_heads = pool.num_kv_heads;
    p.wait_ns = pool.wait_ns;
    cudaLaunchConfig_t cfg = {};
    // one CTA per pair of query tiles
    cfg.gridDim = dim3((unsigned)((c.max_query_len + 2 * QT - 1) / (2 * QT)),
                       (unsigned)pool.num_kv_heads, (unsigned)c.batch);
    cfg.blockDim = dim3(FMT >= 0 ? NTHREADS_Q8 : NTHREADS);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmap_q, *mk, *mv, p);
}

template <typename T, int FMT>
cudaError_t launch_group(const kv_pool& pool, const PrefillCall& c, cudaStream_t stream) {
    switch (c.num_q_heads / pool.num_kv_heads) {
        case 1: return launch_typed<T, 1, FMT>(pool, c, stream);
        case 2: return launch_typed<T, 2, FMT>(pool, c, stream);
        case 4: return launch_typed<T, 4, FMT>(pool, c, stream);
        case 8: return launch_typed<T, 8, FMT>(pool, c, stream);
    }
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t launch_format(const kv_pool& pool, const PrefillCall& c, cudaStream_t stream) {
    if (pool.cache_dtype == KV_FP8_E4M3) return launch_group<T, dec::kFmtE4M3>(pool, c, stream);
    if (pool.cache_dtype == KV_INT8) return launch_group<T, dec::kFmtInt8>(pool, c, stream);
    return launch_group<T, -1>(pool, c, stream);
}

}  // namespace pf

cudaError_t launch_prefill(const kv_pool& pool, const PrefillCall& c, cudaStream_t stream) {
    if (pool.dtype == KV_BF16) return pf::launch_format<__nv_bfloat16>(pool, c, stream);
    if (pool.dtype == KV_F16) return pf::launch_format<__half>(pool, c, stream);
    return cudaErrorNotSupported;
}

}  // namespace pagedkv

extern "C" {

kv_status paged_attention_prefill(kv_pool_t pool, const void* q, void* out,
                                  const int32_t* cu_seqlens, int num_tokens, int max_query_len,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* seq_lens, int batch, int num_q_heads,
                                  float scale, int num_kv_heads, void* stream) {
    const pagedkv::NvtxRange range("paged_attention_prefill");
    if (!pool || batch < 1 || num_q_heads < 1 || num_tokens < 0) return KV_EINVAL;
    if (num_kv_heads != pool->num_kv_heads || num_q_heads % num_kv_heads) return KV_EINVAL;
    const int g = num_q_heads / num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return KV_EUNSUPPORTED;
    if ((pool->dtype != KV_BF16 && pool->dtype != KV_F16) || pool->head_dim != 128 ||
        !pool->has_swizzled_maps)
        return KV_EUNSUPPORTED;
    const int bs = pool->block_size;
    if (bs < 8 || bs > 128 || (bs & (bs - 1))) return KV_EUNSUPPORTED;
    if (pagedkv::is_q8(*pool) && bs < 16) return KV_EUNSUPPORTED;
    if (batch > 65535 || num_kv_heads > 65535) return KV_EUNSUPPORTED;
    if (num_tokens == 0) return KV_OK;
    if (max_query_len < 1 || max_query_len > num_tokens) return KV_EINVAL;
    if (!q || !out || !cu_seqlens || !block_tables || !seq_lens) return KV_EINVAL;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (!a16(q) || !a16(out) || !a4(cu_seqlens) || !a4(block_tables) || !a4(seq_lens))
        return KV_EINVAL;
    if (max_blocks_per_seq < 1 ||
        (long long)batch * max_blocks_per_seq >= (1ll << 31) ||
        (long long)max_blocks_per_seq * bs >= (1ll << 31))
        return KV_EINVAL;
    if ((long long)num_tokens * num_q_heads * 128 >= (1ll << 40)) return KV_EINVAL;
    if (!(scale > 0.f) || !(scale < 3.4e38f)) return KV_EINVAL;
    pagedkv::PrefillCall call{q,            out,
                              cu_seqlens,   num_tokens,
                              max_query_len, block_tables,
                              max_blocks_per_seq, seq_lens,
                              batch,        num_q_heads,
                              scale};
    cudaError_t e = pagedkv::launch_prefill(*pool, call, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return KV_EUNSUPPORTED;
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "paged_attention_prefill");
}

}  // extern "C"
