// Cascade (shared-prefix) decode: planning, launch and the C-ABI entry points.
//
// Two launches on the caller's stream: the shared-prefix pass
// (paged_decode_prefix) leaves per-(sequence, head) prefix states in the
// workspace, then the split kernel attends each sequence's remaining blocks
// and folds the prefix state into its log-sum-exp merge.  Shapes without a
// prefix kernel (fp32 pools, head_dim 64, block sizes other than 16 and 32)
// and calls with no groups run the plain decode, which gives the same result.
// 16-bit and 8-bit (FP8 E4M3, INT8) pools alike.
#include <atomic>
#include <cstdio>
#include <mutex>

#include "decode_prefix_tc.cuh"
#include "pagedkv_internal.cuh"

namespace pagedkv {
namespace {

constexpr size_t kMaxSmemP = 227 * 1024;
constexpr size_t kMaxRingBytesP = 128 * 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct PrefixPlan {
    int stages;
    int num_ctas;
    size_t smem_bytes;
    // workspace, after the plain decode's part
    size_t off_pst_o, off_pst_lse, off_ctr, off_part_o, off_part_lse, end;
};

// The split kernel's part at the start of a cascade workspace: as large as
// both its plans need (with and without the groups' shared-memory tables;
// the grids can differ), given the plain plan's need in *bytes.
kv_status split_part(kv_pool* pool, int batch, int num_q_heads, int num_groups, size_t* bytes) {
    DecodePlan dp;
    cudaError_t e = plan_decode(*pool, batch, num_q_heads, num_groups, &dp);
    if (e == cudaErrorNotSupported) return KV_EUNSUPPORTED;
    if (e != cudaSuccess) return cuda_fail(e, "paged_attention_decode_cascade(plan)");
    if (dp.ws_bytes > *bytes) *bytes = dp.ws_bytes;
    return KV_OK;
}

// The shapes with a prefix kernel: head_dim 128, groups of 1, 2, 4 or 8, block
// size 16 or 32, a pool with 128-byte-swizzled tensor maps; 16-bit pools, and
// 8-bit pools with 16-bit queries.
bool cascade_shape(const kv_pool& pool, int group) {
    if (pool.head_dim != 128 || !(group == 1 || group == 2 || group == 4 || group == 8) ||
        !(pool.block_size == 16 || pool.block_size == 32) || !pool.has_swizzled_maps)
        return false;
    if (is_q8(pool)) return pool.dtype == KV_BF16 || pool.dtype == KV_F16;
    return pool.elem_bytes == 2;
}

// The 16-bit pools' prefix pass runs on tcgen05 (one CTA per SM), the 8-bit
// pools' on mma.sync (decode_prefix.cuh; codes convert in registers).
bool tc_prefix(const kv_pool& pool) { return !is_q8(pool); }

cudaError_t prefix_attrs_any(const kv_pool& pool, int group, size_t smem, int* occ) {
    if (is_q8(pool))
        return pool.dtype == KV_BF16 ? prefix_q8_attrs_bf16(pool, group, smem, occ)
                                     : prefix_q8_attrs_f16(pool, group, smem, occ);
    return ptc::by_tc_shape(pool, group, [&]<typename T, int GG, int BB>() {
        return ptc::prefix_tc_attrs<T, GG, BB>(smem, occ);
    });
}

cudaError_t prefix_launch_any(const kv_pool& pool, int group, const dec::PParams& p, size_t smem,
                              int grid, cudaStream_t stream) {
    if (is_q8(pool))
        return pool.dtype == KV_BF16 ? prefix_q8_launch_bf16(pool, group, p, smem, grid, stream)
                                     : prefix_q8_launch_f16(pool, group, p, smem, grid, stream);
    return ptc::by_tc_shape(pool, group, [&]<typename T, int GG, int BB>() {
        return ptc::prefix_tc_launch<T, GG, BB>(pool.tmap_k_swz, pool.tmap_v_swz, p, smem, grid,
                                                stream);
    });
}

// Shared memory and grid of the prefix pass.  tcgen05 (16-bit pools): one CTA
// per SM with the deepest K and V rings that fit (three tiles each, else
// two).  mma.sync (8-bit pools): the ring depth with the most resident CTAs
// x stages per consumer warp (counted up to 2), then the deepest.
cudaError_t plan_prefix(const kv_pool& pool, int batch, int num_q_heads, int num_groups,
                        size_t base, PrefixPlan* pp) {
    const int G = num_q_heads / pool.num_kv_heads;
    const int D = pool.head_dim;
    int best_s = 0, best_occ = 0, best_score = -1;
    size_t best_smem = 0;
    if (tc_prefix(pool)) {
        for (int S = 3; S >= 2 && best_s == 0; --S) {
            const size_t smem = ptc::TLayout(S, S, num_groups).total + 1024;
            if (smem > kMaxSmemP) continue;
            int occ = 0;
            cudaError_t e = prefix_attrs_any(pool, G, smem, &occ);
            if (e != cudaSuccess) return e;
            if (occ >= 1) {
                best_s = S;
                best_occ = 1;
                best_smem = smem;
            }
        }
    } else {
        // 32-row units of 128-byte code rows; INT8 adds the rows' scales
        constexpr int rows = 32;
        const bool scales = pool.cache_dtype == KV_INT8;
        const size_t stage = 2ull * rows * D;
        for (int S = dec::NCW; S <= 8 * dec::NCW; S += dec::NCW) {
            if (S > dec::NCW && (size_t)S * stage > kMaxRingBytesP) break;
            const size_t smem = dec::PLayout(S, num_groups, rows, D, 1, scales).total + 1024;
            if (smem > kMaxSmemP) break;
            int occ = 0;
            cudaError_t e = prefix_attrs_any(pool, G, smem, &occ);
            if (e != cudaSuccess) return e;
            const int per_warp = S / dec::NCW > 2 ? 2 : S / dec::NCW;
            if (occ >= 1 && occ * per_warp >= best_score) {
                best_s = S;
                best_occ = occ;
                best_score = occ * per_warp;
                best_smem = smem;
            }
        }
    }
    if (best_s == 0) return cudaErrorNotSupported;
    pp->stages = best_s;
    pp->smem_bytes = best_smem;
    pp->num_ctas = pool.num_sms * best_occ;
    size_t off = align_up(base, 256);
    pp->off_pst_o = off;     off = align_up(off + 4ull * batch * num_q_heads * D, 256);
    pp->off_pst_lse = off;   off = align_up(off + 4ull * batch * num_q_heads, 256);
    pp->off_ctr = off;       off = align_up(off + 16ull * batch * pool.num_kv_heads, 256);
    pp->off_part_o = off;    off = align_up(off + 4ull * pp->num_ctas * 2 * dec::kRows * D, 256);
    pp->off_part_lse = off;  off = align_up(off + 4ull * pp->num_ctas * 2 * dec::kRows, 256);
    pp->end = off;
    return cudaSuccess;
}

}  // namespace
}  // namespace pagedkv

extern "C" {

kv_status paged_attention_cascade_workspace_size(kv_pool_t pool, int batch, int num_q_heads,
                                                 int num_groups, size_t* bytes) {
    if (!bytes || num_groups < 0 || num_groups > pagedkv::kMaxGroups) return KV_EINVAL;
    size_t plain = 0;
    kv_status st = paged_attention_workspace_size(pool, batch, num_q_heads, &plain);
    if (st != KV_OK) return st;
    const int G = num_q_heads / pool->num_kv_heads;
    if (num_groups == 0 || !pagedkv::cascade_shape(*pool, G)) {
        *bytes = plain;
        return KV_OK;
    }
    st = pagedkv::split_part(pool, batch, num_q_heads, num_groups, &plain);
    if (st != KV_OK) return st;
    pagedkv::PrefixPlan pp;
    cudaError_t e = pagedkv::plan_prefix(*pool, batch, num_q_heads, num_groups, plain, &pp);
    if (e == cudaErrorNotSupported) {
        *bytes = plain;
        return KV_OK;
    }
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_cascade_workspace_size");
    *bytes = pp.end;
    return KV_OK;
}

kv_status paged_attention_decode_cascade(kv_pool_t pool, const void* q, void* out,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* seq_lens, int batch, int num_q_heads,
                                         float scale, int num_kv_heads, const int32_t* group_first,
                                         const int32_t* group_size,
                                         const int32_t* group_shared_blocks, int num_groups,
                                         void* workspace, size_t workspace_bytes, void* stream) {
    const pagedkv::NvtxRange range("paged_attention_decode_cascade");
    if (num_groups < 0 || num_groups > pagedkv::kMaxGroups) return KV_EINVAL;
    if (num_groups > 0 && (!group_first || !group_size || !group_shared_blocks ||
                           (reinterpret_cast<uintptr_t>(group_first) & 3u) ||
                           (reinterpret_cast<uintptr_t>(group_size) & 3u) ||
                           (reinterpret_cast<uintptr_t>(group_shared_blocks) & 3u)))
        return KV_EINVAL;
    if (!pool || num_kv_heads != pool->num_kv_heads || num_q_heads < 1 ||
        num_q_heads % num_kv_heads)
        return KV_EINVAL;
    const int G = num_q_heads / num_kv_heads;
    if (num_groups == 0 || !pagedkv::cascade_shape(*pool, G))
        return pagedkv::decode_with_workspace(pool, q, out, block_tables, max_blocks_per_seq,
                                              seq_lens, batch, num_q_heads, scale, num_kv_heads,
                                              workspace, workspace_bytes,
                                              static_cast<cudaStream_t>(stream));
    size_t plain = 0;
    kv_status st = paged_attention_workspace_size(pool, batch, num_q_heads, &plain);
    if (st != KV_OK) return st;
    st = pagedkv::split_part(pool, batch, num_q_heads, num_groups, &plain);
    if (st != KV_OK) return st;
    pagedkv::PrefixPlan pp;
    cudaError_t e = pagedkv::plan_prefix(*pool, batch, num_q_heads, num_groups, plain, &pp);
    if (e == cudaErrorNotSupported)
        return pagedkv::decode_with_workspace(pool, q, out, block_tables, max_blocks_per_seq,
                                              seq_lens, batch, num_q_heads, scale, num_kv_heads,
                                              workspace, workspace_bytes,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_decode_cascade(plan)");
    if (!workspace || workspace_bytes < pp.end) return KV_ENOWORKSPACE;
    // the plain decode checks the remaining arguments before anything is enqueued
    if (!q || !out || !block_tables || !seq_lens) return KV_EINVAL;

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    pagedkv::dec::PParams p;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.g_first = group_first;
    p.g_size = group_size;
    p.g_blocks = group_shared_blocks;
    p.err = pool->d_err;
    p.pst_o = reinterpret_cast<float*>(ws + pp.off_pst_o);
    p.pst_lse = reinterpret_cast<float*>(ws + pp.off_pst_lse);
    p.counters = reinterpret_cast<unsigned long long*>(ws + pp.off_ctr);
    p.tag = pagedkv::new_counter_tag();
    p.part_o = reinterpret_cast<float*>(ws + pp.off_part_o);
    p.part_lse = reinterpret_cast<float*>(ws + pp.off_part_lse);
    p.num_groups = num_groups;
    p.max_blocks = max_blocks_per_seq;
    p.batch = batch;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = pool->num_blocks;
    p.bs = pool->block_size;
    p.stages = pp.stages;
    p.num_ctas = pp.num_ctas;
    p.k_scales = pool->k_scales;
    p.v_scales = pool->v_scales;
    // FP8 pools: the K scale multiplies every score, the V scale the output
    const bool fp8 = pool->cache_dtype == KV_FP8_E4M3;
    p.qscale = scale * 1.4426950408889634f * (fp8 ? pool->fp8_k_scale : 1.f);
    p.vscale = fp8 ? pool->fp8_v_scale : 1.f;
    p.wait_ns = pool->wait_ns;
    // argument checks of the second pass first, so nothing is enqueued on error
    if (batch < 1 || batch > pagedkv::kMaxBatch || max_blocks_per_seq < 1 ||
        (long long)batch * max_blocks_per_seq * num_kv_heads >= (1ll << 31) ||
        (reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
        (reinterpret_cast<uintptr_t>(workspace) & 15u) || !(scale == scale))
        return KV_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = pagedkv::prefix_launch_any(*pool, G, p, pp.smem_bytes, pp.num_ctas, s);
    if (e != cudaSuccess) return pagedkv::cuda_fail(e, "paged_attention_decode_cascade(prefix)");
    return pagedkv::decode_after_prefix(pool, q, out, block_tables, max_blocks_per_seq, seq_lens,
                                        batch, num_q_heads, scale, workspace, plain,
                                        group_first, group_size, group_shared_blocks, num_groups,
                                        p.pst_o, p.pst_lse, s);
}

}  // extern "C"
