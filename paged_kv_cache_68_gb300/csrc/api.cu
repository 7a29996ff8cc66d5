// C-ABI front end: argument checks, pool descriptors (TMA tensor maps), launch
// planning and dispatch.  Every entry point validates on the host, enqueues on
// the caller's stream and returns; see pagedkv.h for the contract.
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cstdio>
#include <random>
#include <cstring>
#include <mutex>
#include <new>

#include "decode_kernel.cuh"
#include "pagedkv_internal.cuh"

namespace {

thread_local char g_last_cuda_error[256] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(kv_dtype d) { return d == KV_F32 ? 4 : 2; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// The pool viewed as [N*bs rows][Hkv][D]; one box = the bs rows of one block
// for one KV head: {D, 1, bs} unswizzled, or {128 bytes of dims, 1, bs} with
// the 128-byte swizzle (one box per half row of a head_dim-128 16-bit pool).
bool encode_pool_map(CUtensorMap* map, void* base, const kv_pool& p, bool swizzled) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t elt = (cuuint64_t)p.elem_bytes;
    cuuint64_t dims[3] = {(cuuint64_t)p.head_dim, (cuuint64_t)p.num_kv_heads,
                          (cuuint64_t)p.num_blocks * (cuuint64_t)p.block_size};
    cuuint64_t strides[2] = {(cuuint64_t)p.head_dim * elt,
                             (cuuint64_t)p.num_kv_heads * p.head_dim * elt};
    const cuuint32_t inner = swizzled ? (cuuint32_t)(128 / elt) : (cuuint32_t)p.head_dim;
    cuuint32_t box[3] = {inner, 1u, (cuuint32_t)p.block_size};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapDataType dt = p.elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : p.elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    // L2 fills of 256 B match a 16-bit head row (or a 128-byte half of it); an
    // 8-bit head row is 128 B and a 256-byte fill would drag in the next head's row
    const CUtensorMapL2promotion l2 = p.elem_bytes == 1 && p.head_dim * elt <= 128
                                          ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                          : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    return enc(map, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, l2,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 16-bit head_dim-128 pool viewed as [heads][2 halves][N*bs rows][64 dims]
// (dimension order 64 dims, rows, halves, heads): one box {64, bs, 2, 1} is a
// block's rows for one KV head, 128-byte swizzled, the first half's bs rows
// then the second half's -- the layout of two {64, 1, bs} boxes, in one copy.
bool encode_pool_map_h2(CUtensorMap* map, void* base, const kv_pool& p) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t row = (cuuint64_t)p.num_kv_heads * 256u;       // bytes per token row
    cuuint64_t dims[4] = {64u, (cuuint64_t)p.num_blocks * (cuuint64_t)p.block_size, 2u,
                          (cuuint64_t)p.num_kv_heads};
    cuuint64_t strides[3] = {row, 128u, 256u};
    cuuint32_t box[4] = {64u, (cuuint32_t)p.block_size, 2u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t kMaxRingBytes = 128 * 1024;   // shared-memory ring per CTA, at most
constexpr size_t kMaxSmem = 227 * 1024;

}  // namespace

namespace pagedkv {

bool encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                      bool swizzle128) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
    return enc(map, dt, (cuuint32_t)rank, base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned long long new_counter_tag() {
    static std::atomic<unsigned long long> next{0};
    static const unsigned long long key = [] {
        std::random_device rd;
        const unsigned long long t = (unsigned long long)
            std::chrono::high_resolution_clock::now().time_since_epoch().count();
        return ((unsigned long long)rd() << 32) ^ rd() ^ (t * 0x9e3779b97f4a7c15ull);
    }();
    while (true) {
        // splitmix64's finaliser: a bijection, so distinct counters give distinct tags
        unsigned long long z = key + next.fetch_add(1) * 0x9e3779b97f4a7c15ull;
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        z ^= z >> 31;
        if (z != 0 && z != ~0ull) return z;
    }
}

kv_status cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", where,
                  cudaGetErrorString(e));
    return KV_ECUDA;
}

cudaError_t plan_decode(kv_pool& pool, int batch, int num_q_heads, int num_groups,
                        DecodePlan* plan) {
    {
        std::lock_guard<std::mutex> lock(pool.plan_mu);
        if (pool.plan_batch == batch && pool.plan_hq == num_q_heads &&
            pool.plan_groups == num_groups) {
            *plan = pool.plan;
            return cudaSuccess;
        }
    }
    const int G = num_q_heads / pool.num_kv_heads;
    const int D = pool.head_dim, elt = pool.elem_bytes;
    const bool q8 = is_q8(pool);
    // tokens per work unit: block size 8 on the tensor cores, and 8-bit pools
    // of block size 16 with groups of 4 or 8, pair two blocks (TcPolicy8x2,
    // Tc8Policy2); the kernel lays out its ring for the same unit size
    const bool pairs = q8 ? dec::q8_pairs_blocks(pool, G)
                          : pool.block_size == 8 && dec::use_tensor_cores(pool, G);
    const int bs = pool.block_size * (pairs ? 2 : 1);
    const int sb = pool.cache_dtype == KV_INT8 ? 4 : 0;     // scale bytes per tile row
    const size_t stage = 2ull * bs * D * elt + 2ull * bs * sb;
    // Ring depth S is a multiple of the consumer-warp count (each stage has a
    // fixed consumer).  Pick the S with the most (resident CTAs x stages per
    // warp, the latter counted up to max_per_warp), then the deepest ring.
    const int ncw = dec::NCW;
    // INT8 warps spend the longest on a unit (codes and per-token scales), so
    // a third stage per warp pays even at one CTA fewer per SM (Llama-3-8B
    // step 0.2036 -> 0.1932 ms); 16-bit and FP8 pools run faster with three
    // CTAs of two stages per warp (0.1854 -> 0.1898 ms FP8, 0.2844 -> 0.2879 bf16).
    const int max_per_warp = pool.cache_dtype == KV_INT8 ? 3 : 2;
    int best_s = 0, best_occ = 0, best_score = -1;
    size_t best_smem = 0;
    for (int S = ncw; S <= 8 * ncw; S += ncw) {
        if (S > ncw && (size_t)S * stage > kMaxRingBytes) break;
        // + 1 KB: the kernel rounds its shared-memory base up to 1 KB
        const size_t smem = dec::Layout(S, batch, bs, G, D, elt, num_groups, sb).total + 1024;
        if (smem > kMaxSmem) break;
        int occ = 0;
        cudaError_t e = cudaErrorNotSupported;
        if (q8) {
            if (pool.dtype == KV_F16) e = decode_attrs_q8_f16(pool, G, smem, &occ);
            if (pool.dtype == KV_BF16) e = decode_attrs_q8_bf16(pool, G, smem, &occ);
        } else {
            if (pool.dtype == KV_F32) e = decode_attrs_f32(pool, G, smem, &occ);
            if (pool.dtype == KV_F16) e = decode_attrs_f16(pool, G, smem, &occ);
            if (pool.dtype == KV_BF16) e = decode_attrs_bf16(pool, G, smem, &occ);
        }
        if (e != cudaSuccess) return e;
        const int per_warp = S / ncw > max_per_warp ? max_per_warp : S / ncw;
        const int score = occ * per_warp;
        if (occ >= 1 && score >= best_score) {
            best_s = S;
            best_occ = occ;
            best_score = score;
            best_smem = smem;
        }
    }
    if (best_s == 0 || best_occ < 1) return cudaErrorNotSupported;
    DecodePlan pl;
    pl.group = G;
    pl.stages = best_s;
    pl.smem_bytes = best_smem;
    pl.num_ctas = pool.num_sms * best_occ;
    size_t off = 0;
    pl.ws_counter_off = off;                 // piece counters {tag, count}, one per (b, g)
    off = align_up(off + 16ull * batch * pool.num_kv_heads, 256);
    // two partial slots per worker (one worker per warp of the grid)
    const size_t workers = (size_t)pl.num_ctas * dec::NCW;
    pl.ws_part_o_off = off;
    off = align_up(off + 4ull * workers * 2 * G * D, 256);
    pl.ws_part_lse_off = off;
    off = align_up(off + 4ull * workers * 2 * G, 256);
    pl.ws_bytes = off;
    {
        std::lock_guard<std::mutex> lock(pool.plan_mu);
        pool.plan = pl;
        pool.plan_batch = batch;
        pool.plan_hq = num_q_heads;
        pool.plan_groups = num_groups;
    }
    *plan = pl;
    return cudaSuccess;
}

cudaError_t launch_decode(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                          cudaStream_t stream) {
    if (is_q8(pool)) {
        if (pool.dtype == KV_F16) return decode_dispatch_q8_f16(pool, call, plan, stream);
        if (pool.dtype == KV_BF16) return decode_dispatch_q8_bf16(pool, call, plan, stream);
        return cudaErrorNotSupported;
    }
    switch (pool.dtype) {
        case KV_F32: return decode_dispatch_f32(pool, call, plan, stream);
        case KV_F16: return decode_dispatch_f16(pool, call, plan, stream);
        case KV_BF16: return decode_dispatch_bf16(pool, call, plan, stream);
    }
    return cudaErrorNotSupported;
}

}  // namespace pagedkv

extern "C" {

// Geometry checks shared by both pool constructors.
static kv_status check_geometry(int num_blocks, int block_size, int num_kv_heads, void* k_pool,
                                void* v_pool) {
    if (num_blocks < 1 || block_size < 1 || block_size > 256 || num_kv_heads < 1 ||
        num_kv_heads > 1024)
        return KV_EINVAL;
    if ((long long)num_blocks * block_size >= (1ll << 31)) return KV_EINVAL;
    if (!k_pool || !v_pool || !aligned16(k_pool) || !aligned16(v_pool)) return KV_EINVAL;
    return KV_OK;
}

static kv_status finish_pool(kv_pool* p, kv_pool_t* out);

kv_status kv_pool_create(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                         kv_dtype dtype, void* k_pool, void* v_pool, kv_pool_t* out) {
    if (!out) return KV_EINVAL;
    *out = nullptr;
    if (dtype != KV_F32 && dtype != KV_F16 && dtype != KV_BF16) return KV_EUNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return KV_EUNSUPPORTED;
    kv_status st = check_geometry(num_blocks, block_size, num_kv_heads, k_pool, v_pool);
    if (st != KV_OK) return st;
    kv_pool* p = new (std::nothrow) kv_pool();
    if (!p) return KV_EINVAL;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->num_kv_heads = num_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    p->cache_dtype = dtype;
    p->elem_bytes = elem_bytes(dtype);
    p->k = k_pool;
    p->v = v_pool;
    return finish_pool(p, out);
}

kv_status kv_pool_create_quantized(int num_blocks, int block_size, int num_kv_heads,
                                   int head_dim, kv_dtype cache_dtype, kv_dtype dtype,
                                   void* k_pool, void* v_pool, float* k_scales, float* v_scales,
                                   float k_scale, float v_scale, kv_pool_t* out) {
    if (!out) return KV_EINVAL;
    *out = nullptr;
    if (cache_dtype != KV_FP8_E4M3 && cache_dtype != KV_INT8) return KV_EUNSUPPORTED;
    if (dtype != KV_F16 && dtype != KV_BF16) return KV_EUNSUPPORTED;
    if (head_dim != 128 || block_size % 16 != 0) return KV_EUNSUPPORTED;
    kv_status st = check_geometry(num_blocks, block_size, num_kv_heads, k_pool, v_pool);
    if (st != KV_OK) return st;
    if (cache_dtype == KV_INT8) {
        if (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales))
            return KV_EINVAL;
    } else {
        if (k_scales || v_scales) return KV_EINVAL;
        if (!(k_scale > 0.f && k_scale <= 3.4e38f) || !(v_scale > 0.f && v_scale <= 3.4e38f))
            return KV_EINVAL;
    }
    kv_pool* p = new (std::nothrow) kv_pool();
    if (!p) return KV_EINVAL;
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->num_kv_heads = num_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    p->cache_dtype = cache_dtype;
    p->elem_bytes = 1;
    p->k = k_pool;
    p->v = v_pool;
    if (cache_dtype == KV_INT8) {
        p->k_scales = k_scales;
        p->v_scales = v_scales;
    } else {
        p->fp8_k_scale = k_scale;
        p->fp8_v_scale = v_scale;
    }
    return finish_pool(p, out);
}

// Device, error word and tensor maps of a filled-in pool; frees it on failure.
static kv_status finish_pool(kv_pool* p, kv_pool_t* out) {
    const int head_dim = p->head_dim, block_size = p->block_size;
    void* k_pool = p->k;
    void* v_pool = p->v;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) e = cudaMalloc(&p->d_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(int));
    if (e != cudaSuccess) {
        if (p->d_err) cudaFree(p->d_err);
        delete p;
        return pagedkv::cuda_fail(e, "kv_pool_create");
    }
    // 128-byte-swizzled boxes: 16-bit pools (two per row of head_dim 128) and
    // 8-bit pools (one per row)
    p->has_swizzled_maps = (p->elem_bytes == 2 || p->elem_bytes == 1) && head_dim == 128 &&
                           block_size <= 256;
    bool maps_ok = encode_pool_map(&p->tmap_k, k_pool, *p, false) &&
                   encode_pool_map(&p->tmap_v, v_pool, *p, false);
    if (maps_ok && p->has_swizzled_maps)
        maps_ok = encode_pool_map(&p->tmap_k_swz, k_pool, *p, true) &&
                  encode_pool_map(&p->tmap_v_swz, v_pool, *p, true);
    // one-copy boxes for the tensor-core decode (without them it runs on the
    // CUDA cores)
    if (maps_ok && p->has_swizzled_maps && p->elem_bytes == 2)
        p->has_h2_maps = encode_pool_map_h2(&p->tmap_k_h2, k_pool, *p) &&
                         encode_pool_map_h2(&p->tmap_v_h2, v_pool, *p);
    if (!maps_ok) {
        cudaFree(p->d_err);
        delete p;
        std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error,
                      "kv_pool_create: cuTensorMapEncodeTiled failed");
        return KV_ECUDA;
    }
    *out = p;
    return KV_OK;
}

kv_status kv_pool_destroy(kv_pool_t pool) {
    if (!pool) return KV_OK;
    cudaError_t e = cudaFree(pool->d_err);
    delete pool;
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "kv_pool_destroy");
}

kv_status kv_append(kv_pool_t pool, const void* k_new, const void* v_new,
                    const int64_t* slot_mapping, int num_tokens, void* stream) {
    const pagedkv::NvtxRange range("kv_append");
    if (!pool || num_tokens < 0) return KV_EINVAL;
    if (num_tokens == 0) return KV_OK;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return KV_EINVAL;
    cudaError_t e = pagedkv::launch_append(*pool, k_new, v_new, slot_mapping, num_tokens,
                                           static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "kv_append");
}

kv_status copy_blocks(kv_pool_t pool, const int32_t* pairs, int num_pairs, void* stream) {
    const pagedkv::NvtxRange range("copy_blocks");
    if (!pool || num_pairs < 0 || num_pairs > (1 << 30)) return KV_EINVAL;
    if (num_pairs == 0) return KV_OK;
    if (!pairs || (reinterpret_cast<uintptr_t>(pairs) & 7u)) return KV_EINVAL;
    cudaError_t e = pagedkv::launch_copy_blocks(*pool, pairs, num_pairs,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "copy_blocks");
}

// Memory the device can address: device memory, or host memory that is
// pinned (page-locked, mapped into the unified address space) or managed.
static bool device_accessible(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
           (a.type == cudaMemoryTypeHost && a.devicePointer == p);
}

kv_status kv_swap_blocks(kv_pool_t pool, void* host_k, void* host_v, float* host_k_scales,
                         float* host_v_scales, int num_host_blocks, const int32_t* pairs,
                         int num_pairs, int direction, void* stream) {
    const pagedkv::NvtxRange range("kv_swap_blocks");
    if (!pool || num_pairs < 0 || num_pairs > (1 << 28) || num_host_blocks < 1) return KV_EINVAL;
    if (direction != KV_SWAP_OUT && direction != KV_SWAP_IN) return KV_EINVAL;
    if (num_pairs == 0) return KV_OK;
    if (!pairs || (reinterpret_cast<uintptr_t>(pairs) & 7u) || !device_accessible(pairs))
        return KV_EINVAL;
    if (!host_k || !host_v || !aligned16(host_k) || !aligned16(host_v) ||
        !device_accessible(host_k) || !device_accessible(host_v))
        return KV_EINVAL;
    if ((long long)num_host_blocks * pool->block_size >= (1ll << 31)) return KV_EINVAL;
    if (pool->cache_dtype == KV_INT8) {
        if (!host_k_scales || !host_v_scales || !aligned16(host_k_scales) ||
            !aligned16(host_v_scales) || !device_accessible(host_k_scales) ||
            !device_accessible(host_v_scales))
            return KV_EINVAL;
    } else if (host_k_scales || host_v_scales) {
        return KV_EINVAL;
    }
    cudaError_t e = pagedkv::launch_swap_blocks(*pool, host_k, host_v, host_k_scales,
                                                host_v_scales, num_host_blocks, pairs, num_pairs,
                                                direction == KV_SWAP_OUT,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "kv_swap_blocks");
}

static kv_status check_decode_shape(kv_pool_t pool, int batch, int num_q_heads) {
    if (!pool || batch < 1 || num_q_heads < 1) return KV_EINVAL;
    if (batch > pagedkv::kMaxBatch) return KV_EUNSUPPORTED;
    if (num_q_heads % pool->num_kv_heads) return KV_EINVAL;
    const int g = num_q_heads / pool->num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return KV_EUNSUPPORTED;
    return KV_OK;
}

kv_status paged_attention_workspace_size(kv_pool_t pool, int batch, int num_q_heads,
                                         size_t* bytes) {
    if (!bytes) return KV_EINVAL;
    kv_status st = check_decode_shape(pool, batch, num_q_heads);
    if (st != KV_OK) return st;
    pagedkv::DecodePlan plan;
    cudaError_t e = pagedkv::plan_decode(*pool, batch, num_q_heads, 0, &plan);
    if (e == cudaErrorNotSupported) return KV_EUNSUPPORTED;
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_workspace_size");
    *bytes = plan.ws_bytes;
    return KV_OK;
}

kv_status paged_attention_decode_launches(kv_pool_t pool, int batch, int num_q_heads,
                                          int* launches) {
    if (!launches) return KV_EINVAL;
    kv_status st = check_decode_shape(pool, batch, num_q_heads);
    if (st != KV_OK) return st;
    pagedkv::DecodePlan plan;
    cudaError_t e = pagedkv::plan_decode(*pool, batch, num_q_heads, 0, &plan);
    if (e == cudaErrorNotSupported) return KV_EUNSUPPORTED;
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_decode_launches");
    *launches = 1 + (pagedkv::merge_warps_per_pair(plan.num_ctas * pagedkv::dec::NCW,
                                                    batch * pool->num_kv_heads) > 0);
    return KV_OK;
}

static kv_status decode_impl(kv_pool_t pool, const void* q, void* out,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* seq_lens, int batch, int num_q_heads, float scale,
                             int num_kv_heads, void* workspace, size_t workspace_bytes,
                             const int32_t* g_first, const int32_t* g_size,
                             const int32_t* g_blocks, int num_groups, const float* pst_o,
                             const float* pst_lse, unsigned long long tag, void* stream) {
    kv_status st = check_decode_shape(pool, batch, num_q_heads);
    if (st != KV_OK) return st;
    if (num_kv_heads != pool->num_kv_heads) return KV_EINVAL;
    if (!q || !out || !block_tables || !seq_lens || !workspace) return KV_EINVAL;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return KV_EINVAL;
    if (max_blocks_per_seq < 1) return KV_EINVAL;
    if ((long long)batch * max_blocks_per_seq * pool->num_kv_heads >= (1ll << 31))
        return KV_EUNSUPPORTED;
    if (!(scale == scale)) return KV_EINVAL;
    pagedkv::DecodePlan plan;
    cudaError_t e = pagedkv::plan_decode(*pool, batch, num_q_heads, num_groups, &plan);
    if (e == cudaErrorNotSupported) return KV_EUNSUPPORTED;
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_decode(plan)");
    if (workspace_bytes < plan.ws_bytes) return KV_ENOWORKSPACE;
    pagedkv::DecodeCall call{q,     out,   block_tables, max_blocks_per_seq, seq_lens, batch,
                             num_q_heads, scale, workspace, workspace_bytes};
    call.tag = tag ? tag : pagedkv::new_counter_tag();
    call.g_first = g_first;
    call.g_size = g_size;
    call.g_blocks = g_blocks;
    call.num_groups = num_groups;
    call.pst_o = pst_o;
    call.pst_lse = pst_lse;
    e = pagedkv::launch_decode(*pool, call, plan, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "paged_attention_decode");
}

kv_status paged_attention_decode(kv_pool_t pool, const void* q, void* out,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int batch, int num_q_heads, float scale,
                                 int num_kv_heads, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    const pagedkv::NvtxRange range("paged_attention_decode");
    return decode_impl(pool, q, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                       num_q_heads, scale, num_kv_heads, workspace, workspace_bytes, nullptr,
                       nullptr, nullptr, 0, nullptr, nullptr, 0, stream);
}

kv_status kv_pool_set_wait_limit(kv_pool_t pool, unsigned long long limit_ns) {
    if (!pool) return KV_EINVAL;
    pool->wait_ns = limit_ns < pagedkv::kWaitLimitNs ? limit_ns : pagedkv::kWaitLimitNs;
    return KV_OK;
}

kv_status kv_pool_get_error(kv_pool_t pool, int* device_error_bits) {
    if (!pool || !device_error_bits) return KV_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess)
        e = cudaMemcpy(device_error_bits, pool->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "kv_pool_get_error");
    return *device_error_bits ? KV_ERANGE : KV_OK;
}

kv_status kv_pool_clear_error(kv_pool_t pool) {
    if (!pool) return KV_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemset(pool->d_err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return e == cudaSuccess ? KV_OK : pagedkv::cuda_fail(e, "kv_pool_clear_error");
}

const char* kv_strerror(kv_status status) {
    switch (status) {
        case KV_OK: return "ok";
        case KV_EINVAL: return "invalid argument";
        case KV_EUNSUPPORTED: return "unsupported shape or type";
        case KV_ECUDA: return "CUDA error";
        case KV_ERANGE: return "device error word set (out-of-range slot, block, pair or length)";
        case KV_ENOWORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

const char* kv_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"

namespace pagedkv {

kv_status decode_after_prefix(kv_pool* pool, const void* q, void* out, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                              int num_q_heads, float scale, void* workspace,
                              size_t plain_ws_bytes, const int32_t* g_first, const int32_t* g_size,
                              const int32_t* g_blocks, int num_groups, const float* pst_o,
                              const float* pst_lse, cudaStream_t stream) {
    return decode_impl(pool, q, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                       num_q_heads, scale, pool->num_kv_heads, workspace, plain_ws_bytes, g_first,
                       g_size, g_blocks, num_groups, pst_o, pst_lse, 0, stream);
}

kv_status decode_with_workspace(kv_pool* pool, const void* q, void* out,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* seq_lens, int batch, int num_q_heads, float scale,
                                int num_kv_heads, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
    return decode_impl(pool, q, out, block_tables, max_blocks_per_seq, seq_lens, batch,
                       num_q_heads, scale, num_kv_heads, workspace, workspace_bytes, nullptr,
                       nullptr, nullptr, 0, nullptr, nullptr, 0, stream);
}

}  // namespace pagedkv
