// Slot-mapped append (reshape-and-cache) and batched copy-on-write block copy.
//
// Both are pure data movement, bound by HBM: 16-byte vector loads and stores,
// each warp moving whole rows (append) or each CTA moving one whole block of
// one pool (copy).  Sources: "Part 3: single node" (random-liu.github.io),
// ch. 13 sec. 1 -- the GPU only executes kv_cache[slot_mapping[i]] = new_kv;
// "Lecture 3" (semidirectx.com, CS349D notes), sec. 3.2 -- the write by block
// table is one fused kernel and the many small copy-on-write copies are merged
// into one launch; sec. 4.1 -- copy-on-write copies the whole block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

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

// Quantising append for 8-bit pools: one warp per (token, K-or-V) row of
// Hkv x D 16-bit values; a head's D = 128 values are spread over 16 lanes (8
// each), so a warp step covers two heads.  FP8 E4M3: code = E4M3(x / scale),
// the division in fp32, nearest-even rounding with saturation.  INT8: amax of
// the head's row, inv = 127 / amax and scale = amax / 127 in fp32, code =
// rint(x * inv) clipped to [-127, 127]; an all-zero row gets scale 0 and a row
// holding NaN or an infinity scale NaN and codes 0.  ("Part 3: single node",
// random-liu.github.io, ch. 10 sec. 1 and 3: K and V are scaled and rounded to
// 8 bits when written; INT8 with a per-token scale.)
template <typename T> __device__ __forceinline__ float2 to_f2(uint32_t w);
template <> __device__ __forceinline__ float2 to_f2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <> __device__ __forceinline__ float2 to_f2<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

template <typename T, bool INT8>
__global__ void __launch_bounds__(256) append_q8_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slots, int num_tokens, unsigned char* __restrict__ k_pool,
    unsigned char* __restrict__ v_pool, float* __restrict__ k_scales, float* __restrict__ v_scales,
    float k_div, float v_div, long long num_rows, int bs, int hkv, int* __restrict__ err) {
    constexpr int D = 128;
    pdl_launch_dependents();
    pdl_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= 2 * num_tokens) return;
    const int tok = warp >> 1;
    const bool is_v = warp & 1;
    const int64_t slot = slots[tok];
    if (slot < 0) return;
    if (slot >= num_rows) {
        if (lane == 0 && !is_v) atomicOr(err, KV_DEVERR_SLOT_RANGE);
        return;
    }
    const uint4* src = (is_v ? v_new : k_new) + (size_t)tok * hkv * (D / 8);
    unsigned char* dst = (is_v ? v_pool : k_pool) + (size_t)slot * hkv * D;
    float* scales = is_v ? v_scales : k_scales;
    const float div = is_v ? v_div : k_div;
    const long long blk = slot / bs, off = slot % bs;
    const int half = lane >> 4, hl = lane & 15;       // head of the pair, lane in the head
    for (int h0 = 0; h0 < hkv; h0 += 2) {
        const int h = h0 + half;
        const bool act = h < hkv;
        float x[8];
        if (act) {
            const uint4 w = ldg_nc16(src + (size_t)h * (D / 8) + hl);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = to_f2<T>(ws[i]);
                x[2 * i] = f.x;
                x[2 * i + 1] = f.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = 0.f;
        }
        uint2 codes;
        if constexpr (INT8) {
            float amax = 0.f;
            bool finite = true;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                finite = finite && isfinite(x[i]);
                amax = fmaxf(amax, fabsf(x[i]));
            }
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) {
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                finite = __shfl_xor_sync(0xffffffffu, (int)finite, o) && finite;
            }
            float scale = 0.f;
            uint32_t b[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (!finite) {
                scale = __int_as_float(0x7fc00000);
            } else if (amax > 0.f) {
                const float inv = __fdiv_rn(127.f, amax);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = min(127, max(-127, __float2int_rn(__fmul_rn(x[i], inv))));
                    b[i] = (uint32_t)c & 0xffu;
                }
                scale = __fdiv_rn(amax, 127.f);
            }
            codes.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
            codes.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
            if (act && hl == 0) scales[((size_t)blk * hkv + h) * bs + off] = scale;
        } else {
            uint32_t pr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                pr[i] = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(x[2 * i], div), __fdiv_rn(x[2 * i + 1], div)),
                    __NV_SATFINITE, __NV_E4M3);
            codes.x = pr[0] | (pr[1] << 16);
            codes.y = pr[2] | (pr[3] << 16);
        }
        if (act) *reinterpret_cast<uint2*>(dst + (size_t)h * D + hl * 8) = codes;
    }
}

// One CTA per (pair, array): a whole block of one of the pool's arrays (K, V
// and, for INT8 pools, the K and V scales), blk16[a] = its block bytes / 16.
struct CopyArrays {
    uint4* base[4];
    int blk16[4];
    int n;
};

__global__ void __launch_bounds__(256) copy_blocks_kernel(
    const int32_t* __restrict__ pairs, int num_pairs, CopyArrays arrays, int num_blocks,
    int* __restrict__ err) {
    pdl_launch_dependents();
    pdl_wait();
    const int pair = blockIdx.x / arrays.n;
    const int a = blockIdx.x % arrays.n;
    if (pair >= num_pairs) return;
    const int src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && a == 0) atomicOr(err, KV_DEVERR_PAIR_RANGE);
        return;
    }
    const int blk16 = arrays.blk16[a];
    uint4* base = arrays.base[a];
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

// Swap to host and back ("Lecture 3", semidirectx.com CS349D notes, sec. 5.2:
// a preempted request's blocks go to CPU memory and return when it resumes):
// one CTA per (pair, array), whole blocks with 16-byte accesses, the host side
// addressed directly in pinned host memory (NVLink-C2C on Grace; no per-block
// copy call).  out: host[h] <- gpu[g]; in: gpu[g] <- host[h].
struct SwapArrays {
    uint4* gpu[4];
    uint4* host[4];
    int blk16[4];
    int n;
};

__global__ void __launch_bounds__(256) swap_blocks_kernel(
    const int32_t* __restrict__ pairs, int num_pairs, SwapArrays arrays, int num_gpu_blocks,
    int num_host_blocks, int to_host, int* __restrict__ err) {
    pdl_launch_dependents();
    pdl_wait();
    const int pair = blockIdx.x / arrays.n;
    const int a = blockIdx.x % arrays.n;
    if (pair >= num_pairs) return;
    const int g = pairs[2 * pair], h = pairs[2 * pair + 1];
    if (g < 0 || g >= num_gpu_blocks || h < 0 || h >= num_host_blocks) {
        if (threadIdx.x == 0 && a == 0) atomicOr(err, KV_DEVERR_PAIR_RANGE);
        return;
    }
    const int blk16 = arrays.blk16[a];
    uint4* gp = arrays.gpu[a] + (size_t)g * blk16;
    uint4* hp = arrays.host[a] + (size_t)h * blk16;
    const uint4* s = to_host ? gp : hp;
    uint4* d = to_host ? hp : gp;
    int i = threadIdx.x;
    for (; i + 3 * 256 < blk16; i += 4 * 256) {
        const uint4 x0 = ldg_nc16(s + i), x1 = ldg_nc16(s + i + 256);
        const uint4 x2 = ldg_nc16(s + i + 512), x3 = ldg_nc16(s + i + 768);
        stg16(d + i, x0);
        stg16(d + i + 256, x1);
        stg16(d + i + 512, x2);
        stg16(d + i + 768, x3);
    }
    for (; i < blk16; i += 256) stg16(d + i, ldg_nc16(s + i));
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
    if (is_q8(pool)) {
        const long long warps = 2ll * num_tokens;
        const int grid = (int)((warps * 32 + 255) / 256);
        cudaLaunchConfig_t cfg = pdl_config(grid, stream);
        cudaLaunchAttribute attr;
        pdl_attr(cfg, attr);
        const bool i8 = pool.cache_dtype == KV_INT8, bf = pool.dtype == KV_BF16;
        auto kern = i8 ? (bf ? append_q8_kernel<__nv_bfloat16, true> : append_q8_kernel<__half, true>)
                       : (bf ? append_q8_kernel<__nv_bfloat16, false> : append_q8_kernel<__half, false>);
        return cudaLaunchKernelEx(&cfg, kern, static_cast<const uint4*>(k_new),
                                  static_cast<const uint4*>(v_new), slots, num_tokens,
                                  static_cast<unsigned char*>(pool.k),
                                  static_cast<unsigned char*>(pool.v), pool.k_scales,
                                  pool.v_scales, pool.fp8_k_scale, pool.fp8_v_scale,
                                  (long long)pool.num_blocks * pool.block_size, pool.block_size,
                                  pool.num_kv_heads, pool.d_err);
    }
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
    CopyArrays arr = {};
    const int blk16 = pool.block_size * pool.num_kv_heads * pool.head_dim * pool.elem_bytes / 16;
    arr.base[0] = static_cast<uint4*>(pool.k);
    arr.base[1] = static_cast<uint4*>(pool.v);
    arr.blk16[0] = arr.blk16[1] = blk16;
    arr.n = 2;
    if (pool.cache_dtype == KV_INT8) {
        arr.base[2] = reinterpret_cast<uint4*>(pool.k_scales);
        arr.base[3] = reinterpret_cast<uint4*>(pool.v_scales);
        arr.blk16[2] = arr.blk16[3] = pool.block_size * pool.num_kv_heads * 4 / 16;
        arr.n = 4;
    }
    if ((long long)arr.n * num_pairs > 0x7fffffffll) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = pdl_config(arr.n * num_pairs, stream);
    cudaLaunchAttribute attr;
    pdl_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, pairs, num_pairs, arr, pool.num_blocks,
                              pool.d_err);
}

cudaError_t launch_swap_blocks(const kv_pool& pool, void* host_k, void* host_v,
                               float* host_k_scales, float* host_v_scales, int num_host_blocks,
                               const int32_t* pairs, int num_pairs, bool to_host,
                               cudaStream_t stream) {
    if (num_pairs <= 0) return cudaSuccess;
    SwapArrays arr = {};
    const int blk16 = pool.block_size * pool.num_kv_heads * pool.head_dim * pool.elem_bytes / 16;
    arr.gpu[0] = static_cast<uint4*>(pool.k);
    arr.gpu[1] = static_cast<uint4*>(pool.v);
    arr.host[0] = static_cast<uint4*>(host_k);
    arr.host[1] = static_cast<uint4*>(host_v);
    arr.blk16[0] = arr.blk16[1] = blk16;
    arr.n = 2;
    if (pool.cache_dtype == KV_INT8) {
        arr.gpu[2] = reinterpret_cast<uint4*>(pool.k_scales);
        arr.gpu[3] = reinterpret_cast<uint4*>(pool.v_scales);
        arr.host[2] = reinterpret_cast<uint4*>(host_k_scales);
        arr.host[3] = reinterpret_cast<uint4*>(host_v_scales);
        arr.blk16[2] = arr.blk16[3] = pool.block_size * pool.num_kv_heads * 4 / 16;
        arr.n = 4;
    }
    if ((long long)arr.n * num_pairs > 0x7fffffffll) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = pdl_config(arr.n * num_pairs, stream);
    cudaLaunchAttribute attr;
    pdl_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, swap_blocks_kernel, pairs, num_pairs, arr, pool.num_blocks,
                              num_host_blocks, to_host ? 1 : 0, pool.d_err);
}

}  // namespace pagedkv
