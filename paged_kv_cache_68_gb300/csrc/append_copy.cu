// Slot-mapped append (reshape-and-cache) and batched copy-on-write block copy.
//
// Both are pure data movement, bound by HBM: 16-byte vector loads and stores,
// each warp moving whole rows (append) or each CTA moving one whole block of
// one pool (copy).  Sources: "Part 3: single node" (random-liu.github.io),
// ch. 13 sec. 1 -- the GPU only executes kv_cache[slot_mapping[i]] = new_kv;
// "Lecture 3" (semidirectx.com, CS349D notes), sec. 3.2 -- the write by block
// table is one fused kernel and the many small copy-on-write copies are merged
// into one launch; sec. 4.1 -- copy-on-write copies the whole block.
#include "pagedkv_internal.cuh"

namespace pagedkv {
namespace {

__device__ __forceinline__ uint4 ldg_nc16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Programmatic dependent launch (no-ops without a programmatic dependency):
// let the next kernel start launching, and wait for the previous one.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void stg16(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// One warp per (token, K-or-V) row.  row16 = row bytes / 16.
__global__ void __launch_bounds__(256) append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slots, int num_tokens, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, long long num_rows, int row16, int* __restrict__ err) {
    pdl_launch_dependents();
    pdl_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= 2 * num_tokens) return;
    const int tok = warp >> 1;
    const bool is_v = warp & 1;
    const int64_t slot = slots[tok];
    if (slot < 0) return;                        // padding
    if (slot >= num_rows) {                      // outside the pool
        if (lane == 0 && !is_v) atomicOr(err, KV_DEVERR_SLOT_RANGE);
        return;
    }
    const uint4* src = (is_v ? v_new : k_new) + (size_t)tok * row16;
    uint4* dst = (is_v ? v_pool : k_pool) + (size_t)slot * row16;
    for (int i = lane; i < row16; i += 32) stg16(dst + i, ldg_nc16(src + i));
}

// One CTA per (pair, K-or-V): a whole block, blk16 = block bytes / 16.
__global__ void __launch_bounds__(256) copy_blocks_kernel(
    const int32_t* __restrict__ pairs, int num_pairs, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, int num_blocks, int blk16, int* __restrict__ err) {
    pdl_launch_dependents();
    pdl_wait();
    const int pair = blockIdx.x >> 1;
    const bool is_v = blockIdx.x & 1;
    if (pair >= num_pairs) return;
    const int src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && !is_v) atomicOr(err, KV_DEVERR_PAIR_RANGE);
        return;
    }
    uint4* base = is_v ? v_pool : k_pool;
    const uint4* s = base + (size_t)src * blk16;
    uint4* d = base + (size_t)dst * blk16;
    // Four independent 16-byte loads in flight per thread before the stores.
    int i = threadIdx.x;
    for (; i + 3 * 256 < blk16; i += 4 * 256) {
        uint4 a = s[i], b = s[i + 256], c = s[i + 512], e = s[i + 768];
        stg16(d + i, a);
        stg16(d + i + 256, b);
        stg16(d + i + 512, c);
        stg16(d + i + 768, e);
    }
    for (; i < blk16; i += 256) stg16(d + i, s[i]);
}

cudaLaunchConfig_t pdl_config(int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    return cfg;
}

// The launch may overlap the previous kernel of the stream (each kernel waits
// with griddepcontrol.wait before touching memory).
void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute& attr) {
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
}

}  // namespace

cudaError_t launch_append(const kv_pool& pool, const void* k_new, const void* v_new,
                          const int64_t* slots, int num_tokens, cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    const int row16 = pool.num_kv_heads * pool.head_dim * pool.elem_bytes / 16;
    const long long warps = 2ll * num_tokens;
    const int grid = (int)((warps * 32 + 255) / 256);
    cudaLaunchConfig_t cfg = pdl_config(grid, stream);
    cudaLaunchAttribute attr;
    pdl_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, append_kernel, static_cast<const uint4*>(k_new),
                              static_cast<const uint4*>(v_new), slots, num_tokens,
                              static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v),
                              (long long)pool.num_blocks * pool.block_size, row16, pool.d_err);
}

cudaError_t launch_copy_blocks(const kv_pool& pool, const int32_t* pairs, int num_pairs,
                               cudaStream_t stream) {
    if (num_pairs <= 0) return cudaSuccess;
    const int blk16 = pool.block_size * pool.num_kv_heads * pool.head_dim * pool.elem_bytes / 16;
    cudaLaunchConfig_t cfg = pdl_config(2 * num_pairs, stream);
    cudaLaunchAttribute attr;
    pdl_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, pairs, num_pairs,
                              static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v),
                              pool.num_blocks, blk16, pool.d_err);
}

}  // namespace pagedkv
