// Internal declarations shared by the C-ABI front end and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "pagedkv.h"

namespace pagedkv {
// Bounded waits: a pipeline wait gives up after this many nanoseconds (by
// default; kv_pool_set_wait_limit lowers it for the decode kernels), sets
// KV_DEVERR_TIMEOUT and lets the kernel finish without the missing data.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Launch plan of one decode: grid size, ring depth, shared memory, workspace.
struct DecodePlan {
    int group;
    int stages;
    int num_ctas;
    size_t smem_bytes;
    size_t ws_bytes;
    size_t ws_counter_off, ws_part_o_off, ws_part_lse_off;
};
}  // namespace pagedkv

struct kv_pool {
    int num_blocks;
    int block_size;
    int num_kv_heads;
    int head_dim;
    kv_dtype dtype;         // q, out and new K/V rows
    kv_dtype cache_dtype;   // the pool's elements: dtype, or KV_FP8_E4M3 / KV_INT8
    int elem_bytes;         // bytes per pool element
    void* k;
    void* v;
    float* k_scales = nullptr;   // KV_INT8: [num_blocks][num_kv_heads][block_size]
    float* v_scales = nullptr;
    float fp8_k_scale = 1.f;     // KV_FP8_E4M3: per-pool scales
    float fp8_v_scale = 1.f;
    int* d_err;             // device error word (KV_DEVERR_* bits)
    CUtensorMap tmap_k;     // 3-D {head_dim, num_kv_heads, num_blocks*block_size},
    CUtensorMap tmap_v;     //   box {head_dim, 1, block_size}, no swizzle
    CUtensorMap tmap_k_swz; // same view, box {128 bytes of dims, 1, block_size},
    CUtensorMap tmap_v_swz; //   128-byte swizzle (16-bit pools, head_dim 128)
    bool has_swizzled_maps;
    CUtensorMap tmap_k_h2;  // 16-bit pools, head_dim 128: 4-D {64 dims, rows, 2 halves,
    CUtensorMap tmap_v_h2;  //   heads}, box {64, block_size, 2, 1}, 128-byte swizzle: one
    bool has_h2_maps = false;   // copy puts both 128-byte halves of a block's rows,
                                // one after the other, in shared memory
    int device;
    int num_sms;
    // limit of one pipeline wait in the decode kernels (kv_pool_set_wait_limit)
    unsigned long long wait_ns = pagedkv::kWaitLimitNs;
    // last decode plan, keyed by (batch, num_q_heads)
    std::mutex plan_mu;
    int plan_batch = -1;
    int plan_hq = -1;
    int plan_groups = -1;
    pagedkv::DecodePlan plan;
};

namespace pagedkv {

// Where the decode merges the partials of a (b, g) cut across warp ranges
// (warps = the split grid's warps, pairs = batch x KV heads): 0 = in the
// split kernel, by the warp that finishes last (a cut (b, g) has two or three
// partials); > 0 = in the merge kernel, that many warps per (b, g) (long
// contexts: dozens of partials each).
inline int merge_warps_per_pair(int warps, int pairs) {
    return warps < 2 * pairs ? 0 : (pairs <= 512 ? 4 : 1);
}

// A named range in the "pagedkv" NVTX domain around one C-ABI call, so a
// profiler's timeline (Nsight Systems, `ncu --nvtx`) shows each call with the
// kernels it launched.  Without an attached tool a push or pop tests one
// function pointer and returns.
inline nvtxDomainHandle_t nvtx_domain() {
    static const nvtxDomainHandle_t d = nvtxDomainCreateA("pagedkv");
    return d;
}
class NvtxRange {
public:
    explicit NvtxRange(const char* name) {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(nvtx_domain(), &a);
    }
    ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kMaxBatch = 4096;
constexpr int kMaxGroups = 1024;   // cascade decode: groups per call

// Record the text of a failed CUDA call for kv_last_cuda_error; returns KV_ECUDA.
kv_status cuda_fail(cudaError_t e, const char* where);

// cuTensorMapEncodeTiled through the runtime's driver entry point (element
// strides 1, no interleave, optional 128-byte swizzle, 256-byte L2 fills).
bool encode_tiled_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                      bool swizzle128);

// Paged prefill: the tcgen05 kernel's launcher (one per query type).
struct PrefillCall {
    const void* q;
    void* out;
    const int32_t* cu_seqlens;
    int num_tokens;
    int max_query_len;
    const int32_t* block_tables;
    int max_blocks;
    const int32_t* seq_lens;
    int batch;
    int num_q_heads;
    float scale;
};
cudaError_t launch_prefill(const kv_pool& pool, const PrefillCall& call, cudaStream_t stream);

// The split decode after a cascade prefix pass: the groups, and that pass's
// states in the workspace; `plain_ws_bytes` is the part of the workspace the
// split kernel itself uses (at its start).
kv_status decode_after_prefix(kv_pool* pool, const void* q, void* out, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                              int num_q_heads, float scale, void* workspace,
                              size_t plain_ws_bytes, const int32_t* g_first, const int32_t* g_size,
                              const int32_t* g_blocks, int num_groups, const float* pst_o,
                              const float* pst_lse, cudaStream_t stream);

// paged_attention_decode without its NVTX range (for the entry points built
// on it, which open their own).
kv_status decode_with_workspace(kv_pool* pool, const void* q, void* out,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* seq_lens, int batch, int num_q_heads, float scale,
                                int num_kv_heads, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

// A fresh random 64-bit tag for one call's piece counters (never 0): a
// process-wide counter through the splitmix64 finaliser, keyed once per
// process from the clock and a random device.
unsigned long long new_counter_tag();

cudaError_t launch_append(const kv_pool& pool, const void* k_new, const void* v_new,
                          const int64_t* slots, int num_tokens, cudaStream_t stream);

cudaError_t launch_copy_blocks(const kv_pool& pool, const int32_t* pairs, int num_pairs,
                               cudaStream_t stream);

cudaError_t launch_swap_blocks(const kv_pool& pool, void* host_k, void* host_v,
                               float* host_k_scales, float* host_v_scales, int num_host_blocks,
                               const int32_t* pairs, int num_pairs, bool to_host,
                               cudaStream_t stream);

struct DecodeCall {
    const void* q;
    void* out;
    const int32_t* block_tables;
    int max_blocks;
    const int32_t* seq_lens;
    int batch;
    int num_q_heads;
    float scale;
    void* workspace;
    size_t workspace_bytes;
    unsigned long long tag = 0;      // random per-call tag of the piece counters
    // cascade decode: the groups and the shared-prefix pass's states
    const int32_t* g_first = nullptr;
    const int32_t* g_size = nullptr;
    const int32_t* g_blocks = nullptr;
    int num_groups = 0;
    const float* pst_o = nullptr;
    const float* pst_lse = nullptr;
};

// Fill `plan` for this pool / batch / head count on the current device
// (cached per pool).  Returns cudaErrorNotSupported for shapes with no
// compiled kernel.
cudaError_t plan_decode(kv_pool& pool, int batch, int num_q_heads, int num_groups,
                        DecodePlan* plan);

cudaError_t launch_decode(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                          cudaStream_t stream);

// Per-dtype entry points (one translation unit each).
cudaError_t decode_dispatch_f32(const kv_pool&, const DecodeCall&, const DecodePlan&, cudaStream_t);
cudaError_t decode_dispatch_f16(const kv_pool&, const DecodeCall&, const DecodePlan&, cudaStream_t);
cudaError_t decode_dispatch_bf16(const kv_pool&, const DecodeCall&, const DecodePlan&, cudaStream_t);
cudaError_t decode_attrs_f32(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm);
cudaError_t decode_attrs_f16(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm);
cudaError_t decode_attrs_bf16(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm);
// 8-bit pools, by query type
cudaError_t decode_dispatch_q8_f16(const kv_pool&, const DecodeCall&, const DecodePlan&, cudaStream_t);
cudaError_t decode_dispatch_q8_bf16(const kv_pool&, const DecodeCall&, const DecodePlan&, cudaStream_t);
cudaError_t decode_attrs_q8_f16(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm);
cudaError_t decode_attrs_q8_bf16(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm);

inline bool is_q8(const kv_pool& pool) {
    return pool.cache_dtype == KV_FP8_E4M3 || pool.cache_dtype == KV_INT8;
}

}  // namespace pagedkv
