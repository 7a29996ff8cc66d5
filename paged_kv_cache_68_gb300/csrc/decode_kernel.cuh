// PagedAttention decode for sm_103a: one persistent, token-balanced kernel fed
// by TMA, with a log-sum-exp merge of the pieces cut across warps.
//
// What is computed ("Lecture 3", semidirectx.com CS349D notes, sec. 3.2; S06
// "Implementation", llminference.xinbetween.com): for each sequence b and
// query head h, softmax(scale * q K^T) V over the sequence's L tokens, K and V
// read through the block table inside the kernel.  Block-wise partial
// softmaxes are merged with a running maximum and sum ("Lecture 24",
// semidirectx.com CMU 11-868 notes, sec. 3.2 -- the FlashAttention /
// Flash-Decoding trick); partial results of one sequence computed on
// different warps are merged by log-sum-exp.
//
// Work decomposition.  A unit is one (sequence b, KV head g, logical block j).
// Units are ordered b-major, then g, then j, and the U units are cut into
// equal contiguous ranges, one per warp of a persistent grid (#SMs x resident
// CTAs x NCW warps), so every warp streams the same number of KV blocks
// whatever the length mix.  Every CTA derives the cut itself from seq_lens (a
// prefix sum in shared memory): no host synchronisation, no atomics for
// scheduling, no extra launch.  The run of units of one (b, g) inside a
// warp's range is a "piece".  A piece that is a whole (b, g) is finished by
// the warp and written to `out`; a piece cut by a range boundary is written
// as a partial (normalised o, log2-sum-exp) to one of two workspace slots of
// its warp -- slot 0 for the warp's first piece, slot 1 for its last -- and
// counted in a per-(b, g) counter tagged with a random per-call value (a
// counter of another tag counts as zero); the warp that completes the count
// merges the partials by log-sum-exp (no second kernel).
//
// Each warp loads its own units: it owns S / NCW stages of the CTA's
// shared-memory ring (one full mbarrier each), looks the block ids of its
// next 32 units up in the block table (one lane each), and after attending a
// unit issues the TMA tile loads of the unit S / NCW further on (the K and V
// rows of that block for KV head g: boxes of the pool viewed as
// [N*bs, Hkv, D]) into the stage it just read.  No warp waits on another.
// The K/V of a block is loaded once for the whole GQA group of G query heads.
// Two compute policies share this frame:
//   CorePolicy (CUDA cores; fp32 pools, groups of 1-2, odd block sizes):
//     QK with TPT lanes per token holding D/TPT dims of all G pre-scaled query
//     rows, a transposing shuffle reduction, packed fp32x2 FMAs; PV with each
//     lane owning 4 dims of the G output rows.
//   TcPolicy (tensor cores, mma.sync m16n8k16; 16-bit pools, groups of 4 or
//     8, block sizes 16 and 32): S^T[tokens x heads] = K_blk Q^T and
//     O^T[dims x heads] += V_blk^T P^T, the group's heads filling N = 8.
//     K/V tiles arrive 128-byte-swizzled so ldmatrix is conflict-free; P^T is
//     transposed in registers with movmatrix and fed as bf16/f16 hi + lo
//     halves, so its rounding stays below 2^-17 relative.
// Softmax state is per block, per head, fp32, base 2.  Rows past the sequence
// end never contribute.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include <algorithm>
#include <type_traits>

#include "pagedkv_internal.cuh"

namespace pagedkv {
namespace dec {

constexpr int NCW = 4;                       // attending warps per CTA
constexpr int NTHREADS = (NCW + 1) * 32;     // + one producer warp (prefix pass)
constexpr int SPLIT_THREADS = NCW * 32;      // split kernel: the consumer warps load too
constexpr unsigned FULL = 0xffffffffu;
constexpr int kMinChunk = 8;                 // fewest units a CTA is given

struct Params {
    const void* q;
    void* out;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    int* err;
    unsigned long long* counters;  // [batch][num_kv_heads][2]: {tag, pieces done}
    unsigned long long tag;        // this call's random counter tag
    float* part_o;         // [num_ctas][2][G][D]
    float* part_lse;       // [num_ctas][2][G]
    int max_blocks;
    int batch;
    int num_q_heads;
    int num_kv_heads;
    int num_blocks;
    int bs;
    int stages;
    int num_ctas;
    float qscale;          // scale * log2(e)
    unsigned long long wait_ns;   // limit of one wait for a tile (the pool's setting)
    // Cascade decode (num_groups > 0): the groups of sequences sharing leading
    // blocks, and the shared-prefix pass's states for their members; this pass
    // then covers only each member's remaining blocks.
    const int32_t* g_first;
    const int32_t* g_size;
    const int32_t* g_blocks;
    int num_groups;
    const float* pst_o;    // [batch][num_q_heads][D], normalised
    const float* pst_lse;  // [batch][num_q_heads], log2-sum-exp
    // 8-bit pools: INT8 scales per (block, KV head, token), FP8 scales per pool
    const float* k_scales; // [num_blocks][num_kv_heads][bs]
    const float* v_scales;
    float fp8_k_scale, fp8_v_scale;
    // Partials of a (b, g) cut across warps: 0 = counted and merged in the
    // split kernel by the warp that finishes last; > 0 = merged by
    // paged_decode_merge, that many warps per (b, g) (they split its partials)
    int merge_wpp;
};

// ---------------------------------------------------------------- layout ---
struct Layout {
    uint32_t full, valid, misc, prefix, groups, skip, pst, pbuf, abuf, sring, ring;
    uint32_t pst_bytes, tx_bytes, stage_bytes, total;
    // elt: bytes per pool element; K: cascade groups (0 for plain decode);
    // sb: scale bytes per token row of a tile (INT8 pools: 4)
    __host__ __device__ Layout(int S, int B, int bs, int G, int D, int elt, int K = 0, int sb = 0) {
        uint32_t off = 0;
        full = off;   off += 8u * S;
        valid = off;  off += 4u * S;
        misc = off;   off += 4u * 40;            // abort flag + warp totals
        prefix = off; off += 4u * (B + 1);
        groups = off; off += K > 0 ? 4u * 3u * K : 0u;   // used groups: first, size, blocks
        skip = off;   off += K > 0 ? 4u * B : 0u;        // leading blocks each sequence skips
        off = (off + 15u) & ~15u;
        pst_bytes = K > 0 ? (4u * G * D + 4u * G + 15u) & ~15u : 0u;
        pst = off;    off += NCW * pst_bytes;    // prefix state, one per warp
        pbuf = off;   off += 8u * NCW * bs * G;
        abuf = off;   off += 8u * NCW * G;
        off = (off + 15u) & ~15u;
        sring = off;  off += (uint32_t)S * 2u * bs * sb;  // per stage: K then V scales
        off = (off + 1023u) & ~1023u;              // swizzle atoms are 1 KB
        ring = off;
        stage_bytes = (2u * bs * D * elt + 127u) & ~127u;   // K tile then V tile
        tx_bytes = 2u * bs * D * elt + 2u * bs * sb;
        off += stage_bytes * S;
        total = off;
    }
};

// ------------------------------------------------------------- PTX helpers --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// The dynamic shared-memory base rounded up to 1 KB (the swizzle atom) by
// pointer arithmetic on the shared array itself: pointers derived from it stay
// known to address shared memory, so their accesses compile to shared-memory
// loads and stores rather than generic ones.
__device__ __forceinline__ unsigned char* smem_align_1k(unsigned char* raw) {
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// As mbar_try, but a thread whose phase is not complete may stay suspended for
// up to `ns` nanoseconds; the hardware wakes it as soon as the phase
// completes, so a waiting warp takes no issue slots from the warps working
// beside it.
__device__ __forceinline__ bool mbar_try_for(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Whether the phase of `bar` with `parity` has completed, without waiting
// (try_wait may wait for a while before it answers no; test_wait does not).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase of `bar` with `parity` to complete; give up after
// `limit_ns` nanoseconds and return false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (limit_ns == 0) return mbar_test(bar, parity);
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}
// mbar_wait with suspended (not spinning) retries; same limit and result.  A
// retry is never suspended for longer than the limit itself, and a limit of
// 0 gives up as soon as the phase is found incomplete.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                unsigned long long limit_ns = kWaitLimitNs) {
    if (limit_ns == 0) return mbar_test(bar, parity);
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    const uint32_t hint = limit_ns < 200000ull ? (uint32_t)limit_ns : 200000u;
    while (!mbar_try_for(bar, parity, hint)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}
// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completing on the mbarrier like a tile load.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// Named barriers among the NCW attending warps (id 0 is __syncthreads; the
// prefix pass's warps merge through them).
__device__ __forceinline__ void named_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(NCW * 32) : "memory");
}
__device__ __forceinline__ void named_arrive(int id) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "n"(NCW * 32) : "memory");
}
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// -- tensor-core helpers (16-bit operands, fp32 accumulate) --
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
    __device__ static __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // (lo, hi) -> packed pair, element `lo` in the low half
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    __device__ static __forceinline__ float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};
template <> struct Mma<__half> {
    __device__ static __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    __device__ static __forceinline__ float2 unpack(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    }
};
// Programmatic dependent launch: let the next kernel in the stream start its
// launch now / wait until the previous kernel's results are visible.  Both
// are no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Asynchronous global -> shared copies (LDGSTS): 16 bytes through L2 only,
// or 4 bytes; wait_all blocks until this thread's copies have landed.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// ------------------------------------------------------------ element I/O --
template <typename T> struct Elt;
template <> struct Elt<float> {
    // 16 bytes -> 4 values
    __device__ static __forceinline__ void chunk(uint4 r, float* f) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
    // 4 values starting at p (16 bytes)
    __device__ static __forceinline__ void four(const unsigned char* p, float* f) {
        chunk(*reinterpret_cast<const uint4*>(p), f);
    }
    // the same as consecutive pairs (element 2i in .x, 2i+1 in .y)
    __device__ static __forceinline__ void chunk2(uint4 r, float2* f) {
        f[0] = make_float2(__uint_as_float(r.x), __uint_as_float(r.y));
        f[1] = make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
    __device__ static __forceinline__ void four2(const unsigned char* p, float2* f) {
        chunk2(*reinterpret_cast<const uint4*>(p), f);
    }
    __device__ static __forceinline__ float store(float x) { return x; }
};
template <> struct Elt<__half> {
    __device__ static __forceinline__ void pair(uint32_t w, float* f) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w));
        f[0] = v.x; f[1] = v.y;
    }
    __device__ static __forceinline__ void chunk(uint4 r, float* f) {
        pair(r.x, f); pair(r.y, f + 2); pair(r.z, f + 4); pair(r.w, f + 6);
    }
    __device__ static __forceinline__ void four(const unsigned char* p, float* f) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        pair(r.x, f); pair(r.y, f + 2);
    }
    __device__ static __forceinline__ float2 pair2(uint32_t w) {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    }
    __device__ static __forceinline__ void chunk2(uint4 r, float2* f) {
        f[0] = pair2(r.x); f[1] = pair2(r.y); f[2] = pair2(r.z); f[3] = pair2(r.w);
    }
    __device__ static __forceinline__ void four2(const unsigned char* p, float2* f) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        f[0] = pair2(r.x); f[1] = pair2(r.y);
    }
    __device__ static __forceinline__ __half store(float x) { return __float2half_rn(x); }
};
template <> struct Elt<__nv_bfloat16> {
    // bf16 is the top half of an fp32: widening is a shift / mask.
    __device__ static __forceinline__ void pair(uint32_t w, float* f) {
        f[0] = __uint_as_float(w << 16);
        f[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ static __forceinline__ void chunk(uint4 r, float* f) {
        pair(r.x, f); pair(r.y, f + 2); pair(r.z, f + 4); pair(r.w, f + 6);
    }
    __device__ static __forceinline__ void four(const unsigned char* p, float* f) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        pair(r.x, f); pair(r.y, f + 2);
    }
    __device__ static __forceinline__ float2 pair2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ static __forceinline__ void chunk2(uint4 r, float2* f) {
        f[0] = pair2(r.x); f[1] = pair2(r.y); f[2] = pair2(r.z); f[3] = pair2(r.w);
    }
    __device__ static __forceinline__ void four2(const unsigned char* p, float2* f) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        f[0] = pair2(r.x); f[1] = pair2(r.y);
    }
    __device__ static __forceinline__ __nv_bfloat16 store(float x) { return __float2bfloat16_rn(x); }
};

template <int X> struct Log2 { static constexpr int v = 1 + Log2<X / 2>::v; };
template <> struct Log2<1> { static constexpr int v = 0; };

template <typename T, int D, int G>
struct Cfg {
    static constexpr int ELT = sizeof(T);
    static constexpr int VE = 16 / ELT;                          // values per 16 B chunk
    static constexpr int CHUNKS = D * ELT / 16;                  // chunks per row
    static constexpr int TPT = (G * D / 64 > 8) ? G * D / 64 : 8;  // QK lanes per token
    static constexpr int TPS = 32 / TPT;                         // tokens per QK step
    static constexpr int NCH = CHUNKS / TPT;                     // chunks per lane
    static constexpr int QE = NCH * VE;                          // q values per lane per head
    static constexpr int HSHIFT = Log2<TPT>::v - Log2<G>::v;     // head of a lane after reduce
    static constexpr int LPV = D / 4;                            // PV lanes per token
    static constexpr int TPSV = 32 / LPV;                        // tokens per PV step
    static_assert(CHUNKS % TPT == 0 && NCH >= 1, "row does not split over the QK lanes");
    static_assert(G <= TPT && (G & (G - 1)) == 0, "group size must be a power of two <= TPT");
    static_assert(LPV <= 32 && 32 % LPV == 0, "head_dim must be 64 or 128");
};

// Transposing reduction of N partial sums over the lanes differing in bits
// O, O/2, ..., 1: each split step halves the values a lane carries; when one
// value is left the remaining steps are plain butterflies.  Afterwards lane j
// holds the full sum of value ((j >> log2(TPT/G)) & (G-1)).
template <int N, int O> struct TReduce {
    __device__ static __forceinline__ void run(float* v, int lane) {
        const bool up = (lane & O) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float send = up ? v[i] : v[i + N / 2];
            const float keep = up ? v[i + N / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL, send, O);
        }
        TReduce<N / 2, O / 2>::run(v, lane);
    }
};
template <int O> struct TReduce<1, O> {
    __device__ static __forceinline__ void run(float* v, int lane) {
        v[0] += __shfl_xor_sync(FULL, v[0], O);
        TReduce<1, O / 2>::run(v, lane);
    }
};
template <> struct TReduce<1, 0> {
    __device__ static __forceinline__ void run(float*, int) {}
};

// Largest b in [0, B) with prefix[b] * H <= u (prefix[0] = 0 <= u < prefix[B] * H).
__device__ __forceinline__ int find_seq(const int* prefix, int B, int u, int H) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] * H <= u) lo = mid; else hi = mid;
    }
    return lo;
}

__host__ __device__ __forceinline__ int unit_chunk(int U, int num_ctas) {
    const int c = (U + num_ctas - 1) / num_ctas;
    return c < kMinChunk ? kMinChunk : c;
}

// How the split kernel cuts the units into one range per warp.  A piece of a
// (b, g) costs a warp more than its units -- loading the query rows,
// finishing the softmax, writing the result -- so the ranges are equal in
// cost, not in units: each (b, g) segment s (s = b H + g, its nb units
// starting at unit first) counts kPieceCost units more, placed before its
// first unit, and unit u of segment s sits at cost u + kPieceCost (s + 1).
// Warp c's range is the units whose cost falls in [c chunk, (c + 1) chunk).
constexpr int kPieceCost = 2;
struct WorkCut {
    const int* prefix;     // [B + 1] units of KV head 0 before each sequence
    int B, H, chunk;
    __host__ __device__ __forceinline__ WorkCut(const int* pre, int B_, int H_, int W)
        : prefix(pre), B(B_), H(H_) {
        chunk = unit_chunk(pre[B_] * H_ + kPieceCost * B_ * H_, W);
    }
    // the range holding unit u of segment s
    __host__ __device__ __forceinline__ int range_of(int u, int s) const {
        return (u + kPieceCost * (s + 1)) / chunk;
    }
    // the first unit of range c (the total U when the range is empty at the end)
    __host__ __device__ __forceinline__ int start_unit(int c) const {
        const long long x = (long long)c * chunk;          // cost position
        const long long total = (long long)prefix[B] * H + (long long)kPieceCost * B * H;
        if (x >= total) return prefix[B] * H;
        // the sequence b whose cost interval holds x: prefix[b] H + kPieceCost H b
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((long long)prefix[mid] * H + (long long)kPieceCost * H * mid <= x) lo = mid; else hi = mid;
        }
        const int nb = prefix[lo + 1] - prefix[lo];
        const long long rel = x - ((long long)prefix[lo] * H + (long long)kPieceCost * H * lo);
        const int g = (int)(rel / (nb + kPieceCost));
        const int o = (int)(rel - (long long)g * (nb + kPieceCost));
        // a position in a segment's extra cost starts the range at its first unit
        return prefix[lo] * H + g * nb + (o > kPieceCost ? o - kPieceCost : 0);
    }
};

// ------------------------------------------------------- compute policies --
// Both policies keep one warp's running softmax state for one (b, g) piece and
// expose: begin (load the group's query rows), block (fold one KV block in),
// fold (finish cross-lane sums) and merge_store (normalise the state and
// write the output or the partial).

// Where a warp writes a finished piece.
struct PieceOut {
    bool complete;        // whole (b, g): write `out`; else a partial slot
    void* out;            // &out[b, g*G, 0] (element type of the pool)
    float* part_o;        // &part_o[slot][0][0]
    float* part_lse;      // &part_lse[slot][0]
    const float* pst_o;   // cascade: &pst_o[b, g*G, 0] to fold into a complete piece, or null
    const float* pst_lse; // cascade: &pst_lse[b, g*G]
};

// Fold a normalised state (o_p, lse_p) into an unnormalised one (num, den at
// base M): returns the new base and rescales num/den in place.
__device__ __forceinline__ float fold_state(float M, float& den, float lse_p, float& cs, float& cp) {
    const float M2 = fmaxf(M, lse_p);
    cs = (M2 == -CUDART_INF_F || M == -CUDART_INF_F) ? 0.f : fast_exp2(M - M2);
    cp = (M2 == -CUDART_INF_F || lse_p == -CUDART_INF_F) ? 0.f : fast_exp2(lse_p - M2);
    den = den * cs + cp;
    return M2;
}

template <typename T, int D, int G, int BSC>
struct CorePolicy {
    using C = Cfg<T, D, G>;
    static constexpr bool kSwizzled = false;
    static constexpr bool kH2 = false;        // tiles by the 3-D maps
    static constexpr int kMinBlocks = G >= 8 ? 2 : (G >= 4 ? 3 : 4);
    static constexpr int kKvBytes = sizeof(T);   // pool element
    static constexpr int kScaleBytes = 0;
    static constexpr int kUnitBlocks = 1;        // pool blocks per work unit

    float2* pb;                   // this warp's (score | p, p) [bs][G]
    float2* ab;                   // this warp's (alpha, alpha) [G]
    float2 qf[G][C::QE / 2];      // scaled query rows, pairs of consecutive dims
    float2 o[G][2];               // dims dl*4 .. dl*4+3 of each head
    float m_run, l_run;           // for head lane % G

    __device__ __forceinline__ CorePolicy(float2* pbuf, float2* abuf) : pb(pbuf), ab(abuf) {}
    __device__ __forceinline__ void setup(const Params&) {}

    __device__ __forceinline__ void begin(const T* qp, float qscale, int lane) {
        const int jl = lane % C::TPT;
        const float2 sc2 = make_float2(qscale, qscale);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int i = 0; i < C::NCH; ++i) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
                    qp + (size_t)h * D + (jl + C::TPT * i) * C::VE));
                float2 f[C::VE / 2];
                Elt<T>::chunk2(raw, f);
#pragma unroll
                for (int e = 0; e < C::VE / 2; ++e) qf[h][i * C::VE / 2 + e] = __fmul2_rn(f[e], sc2);
            }
        m_run = -CUDART_INF_F;
        l_run = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h) o[h][0] = o[h][1] = make_float2(0.f, 0.f);
    }

    __device__ __forceinline__ void block(const unsigned char* Ks, const unsigned char* Vs,
                                          const float*, int n_valid, int bs_rt, float, int lane) {
        const int bs = BSC > 0 ? BSC : bs_rt;
        const int tg = lane / C::TPT, jl = lane % C::TPT;
        const int hsel = (jl >> C::HSHIFT) & (G - 1);
        const bool leader = (jl & ((1 << C::HSHIFT) - 1)) == 0;
        const int hh = lane % G;
        const int tv = lane / C::LPV, dl = lane % C::LPV;
        // -- scores --------------------------------------------------------
#pragma unroll 1
        for (int t0 = 0; t0 < bs; t0 += C::TPS) {
            const int t = t0 + tg;
            float2 acc2[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc2[h] = make_float2(0.f, 0.f);
            if (t < n_valid) {
#pragma unroll
                for (int i = 0; i < C::NCH; ++i) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(
                        Ks + (uint32_t)(t * C::CHUNKS + jl + C::TPT * i) * 16u);
                    float2 kf[C::VE / 2];
                    Elt<T>::chunk2(raw, kf);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < C::VE / 2; ++e)
                            acc2[h] = __ffma2_rn(qf[h][i * C::VE / 2 + e], kf[e], acc2[h]);
                }
            }
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = acc2[h].x + acc2[h].y;
            TReduce<G, C::TPT / 2>::run(acc, lane);
            if (leader && t < bs) pb[t * G + hsel].x = (t < n_valid) ? acc[0] : -CUDART_INF_F;
        }
        __syncwarp();
        // -- online softmax, per head ---------------------------------------
        float mloc = -CUDART_INF_F;
#pragma unroll
        for (int t = lane / G; t < bs; t += 32 / G) mloc = fmaxf(mloc, pb[t * G + hh].x);
#pragma unroll
        for (int off = 16; off >= G; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(FULL, mloc, off));
        const float m_new = fmaxf(m_run, mloc);
        float alpha = 1.f, lsum = 0.f;
        if (m_new != -CUDART_INF_F) {
            alpha = fast_exp2(m_run - m_new);
            for (int t = lane / G; t < bs; t += 32 / G) {
                const float pe = fast_exp2(pb[t * G + hh].x - m_new);
                pb[t * G + hh] = make_float2(pe, pe);
                lsum += pe;
            }
        } else {
            for (int t = lane / G; t < bs; t += 32 / G) pb[t * G + hh] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int off = 16; off >= G; off >>= 1) lsum += __shfl_xor_sync(FULL, lsum, off);
        l_run = l_run * alpha + lsum;
        m_run = m_new;
        if (lane < G) ab[lane] = make_float2(alpha, alpha);
        __syncwarp();
        // -- weighted sum of V ------------------------------------------------
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float2 a = ab[h];
            o[h][0] = __fmul2_rn(o[h][0], a);
            o[h][1] = __fmul2_rn(o[h][1], a);
        }
#pragma unroll 4
        for (int tt = 0; tt < bs; tt += C::TPSV) {
            const int t = tt + tv;
            if (t < n_valid) {
                float2 vf[2];
                Elt<T>::four2(Vs + (uint32_t)(t * D + dl * 4) * C::ELT, vf);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float2 pr = pb[t * G + h];
                    o[h][0] = __ffma2_rn(pr, vf[0], o[h][0]);
                    o[h][1] = __ffma2_rn(pr, vf[1], o[h][1]);
                }
            }
        }
    }

    __device__ __forceinline__ void fold(int) {
#pragma unroll
        for (int off = C::LPV; off < 32; off <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    o[h][e].x += __shfl_xor_sync(FULL, o[h][e].x, off);
                    o[h][e].y += __shfl_xor_sync(FULL, o[h][e].y, off);
                }
    }

    // Normalise the warp's state and write `out` or the partial slot.
    __device__ __forceinline__ void merge_store(int lane, const PieceOut& po) const {
        const int dl = lane % C::LPV;
        // every load of the merge before the first store: the compiler
        // cannot move a load above a store it might alias
        float4 res[G];
        float lse[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float M = __shfl_sync(FULL, m_run, h);
            const float l0 = __shfl_sync(FULL, l_run, h);
            float den = 0.f;
            float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != -CUDART_INF_F) {
                den = l0;
                num = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
            }
            if (po.complete && po.pst_lse != nullptr) {
                float cs, cp;
                M = fold_state(M, den, po.pst_lse[h], cs, cp);
                const float4 op4 = *reinterpret_cast<const float4*>(po.pst_o + h * D + dl * 4);
                num.x = num.x * cs + op4.x * cp; num.y = num.y * cs + op4.y * cp;
                num.z = num.z * cs + op4.z * cp; num.w = num.w * cs + op4.w * cp;
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
            res[h] = make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
            lse[h] = den > 0.f ? M + fast_log2(den) : -CUDART_INF_F;
        }
        if (lane < C::LPV) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                if (po.complete) {
                    T* op = static_cast<T*>(po.out) + h * D + dl * 4;
                    op[0] = Elt<T>::store(res[h].x);
                    op[1] = Elt<T>::store(res[h].y);
                    op[2] = Elt<T>::store(res[h].z);
                    op[3] = Elt<T>::store(res[h].w);
                } else {
                    *reinterpret_cast<float4*>(po.part_o + h * D + dl * 4) = res[h];
                    if (lane == 0) po.part_lse[h] = lse[h];
                }
            }
        }
    }
};

// Tensor-core policy.  Lane roles in the m16n8k16 fragments: gid = lane / 4,
// tig = lane % 4.  S^T (tokens x heads): the lane holds tokens gid, gid + 8 of
// each 16-token tile for heads 2 tig, 2 tig + 1.  O^T (dims x heads): the lane
// holds dims 16 mt + gid, 16 mt + gid + 8 for the same two heads.  Heads >= G
// are padding (zero query rows) and are never written out.
// kPermV: the MMA's output rows (m-slots) 16 mt + gid + 8 hf hold dims
// 16 gid + 2 mt + hf instead of 16 mt + gid + 8 hf (the 8-bit policy loads V
// that way); merge_store writes every value to its own dim.
// kPair: the tile holds two 8-row blocks, block i at byte 2048 i, each as
// [half][8 rows][128 bytes] (block size 8, two blocks per work unit).
template <typename T, int D, int G, int BSC, bool kPermV = false, bool kPair = false>
struct TcPolicy {
    static_assert(sizeof(T) == 2, "tensor-core path takes 16-bit pools");
    static_assert(BSC % 16 == 0 && BSC > 0, "tensor-core path needs a block size of 16k");
    static_assert(G >= 1 && G <= 8, "the group's heads fill N = 8");
    static constexpr bool kSwizzled = true;
    // 16-bit tiles come by the 4-D maps: one copy per block for both halves
    static constexpr bool kH2 = sizeof(T) == 2 && D == 128;
    // (the ring of a head_dim-128 16-bit tile allows three CTAs per SM at
    // most, so the register cap is that of three)
    static constexpr int kMinBlocks = 3;
    static constexpr int kKvBytes = sizeof(T);
    static constexpr int kScaleBytes = 0;
    static constexpr int kUnitBlocks = 1;  // pool blocks per work unit
    static constexpr int KS = D / 16;      // QK k-steps (16 dims each)
    static constexpr int MT = D / 16;      // PV m-tiles (16 dims each)
    static constexpr int TT = BSC / 16;    // 16-token tiles per block
    // Groups of up to 4 heads leave half of the MMA's N = 8 columns free:
    // columns 4..7 repeat the query heads of columns 0..3, so their scores,
    // maxima and weights are bit-identical, and the PV product takes the hi
    // halves of P in columns 0..3 and the lo halves in 4..7 -- one MMA per
    // m-tile instead of two.  fold() adds the two halves.
    static constexpr bool kPairHL = G <= 4;

    uint32_t qb[KS][2];                    // Q^T fragments (raw 16-bit query)
    float oacc[MT][4];                     // O^T accumulators
    float m_run[2], l_run[2];              // heads 2 tig, 2 tig + 1

    __device__ __forceinline__ TcPolicy(float2*, float2*) {}
    __device__ __forceinline__ void setup(const Params&) {}

    __device__ static __forceinline__ int dim(int mt, int gid, int hf) {
        return kPermV ? 16 * gid + 2 * mt + hf : mt * 16 + gid + 8 * hf;
    }

    // Byte offset of the 128-byte line holding half hf of row r: the halves
    // are BSC rows apart (kPair: 8 rows apart within each 2 KB block).
    __device__ static __forceinline__ int line(int r, int hf) {
        return kPair ? (r >> 3) * 2048 + hf * 1024 + (r & 7) * 128 : hf * BSC * 128 + r * 128;
    }
    // Shared address of 16-byte chunk c of row r in a 128-byte-swizzled tile
    // (chunks 0-7 in the first 128-byte half, 8-15 in the second).
    __device__ static __forceinline__ uint32_t swz(uint32_t tile, int r, int c) {
        return tile + (uint32_t)(line(r, c >> 3) + (((c & 7) ^ (r & 7)) << 4));
    }

    // query head of MMA column n (-1: a padding column)
    __device__ static __forceinline__ int col_head(int n) {
        const int h = kPairHL ? (n & 3) : n;
        return h < G ? h : -1;
    }

    __device__ __forceinline__ void begin(const T* qp, float, int lane) {
        const int gid = lane >> 2, tig = lane & 3, hq = col_head(gid);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int j = 0; j < 2; ++j)
                qb[ks][j] = hq >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(
                                          qp + hq * D + ks * 16 + j * 8 + tig * 2))
                                    : 0u;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
        m_run[0] = m_run[1] = -CUDART_INF_F;
        l_run[0] = l_run[1] = 0.f;
    }

    __device__ __forceinline__ void block(const unsigned char* Ks, const unsigned char* Vs,
                                          const float*, int n_valid, int, float qscale, int lane) {
        const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, r8 = lane & 7;
        const uint32_t kbase = smem_u32(Ks), vbase = smem_u32(Vs);
        if (n_valid < BSC) {
            // rows past the sequence end may hold anything; P is 0 there, and
            // 0 * NaN would still poison the MMA, so clear those V rows
            unsigned char* V = const_cast<unsigned char*>(Vs);
            for (int i = lane; i < (BSC - n_valid) * 8; i += 32) {
                const int r = n_valid + (i >> 3);
#pragma unroll
                for (int hf = 0; hf < D / 64; ++hf)
                    *reinterpret_cast<uint4*>(V + line(r, hf) + (i & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async();
            __syncwarp();
        }
        // -- S^T = K_blk Q^T, scaled to base 2, masked past the end ----------
        float s[TT][4];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(a, swz(kbase, tt * 16 + (mi & 1) * 8 + r8, ks * 2 + (mi >> 1)));
                Mma<T>::run(acc, a, qb[ks][0], qb[ks][1]);
            }
            const bool v0 = tt * 16 + gid < n_valid, v1 = tt * 16 + gid + 8 < n_valid;
            s[tt][0] = v0 ? acc[0] * qscale : -CUDART_INF_F;
            s[tt][1] = v0 ? acc[1] * qscale : -CUDART_INF_F;
            s[tt][2] = v1 ? acc[2] * qscale : -CUDART_INF_F;
            s[tt][3] = v1 ? acc[3] * qscale : -CUDART_INF_F;
        }
        // -- online softmax for heads 2 tig (j = 0) and 2 tig + 1 (j = 1) -----
        float mloc[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mloc[j] = -CUDART_INF_F;
#pragma unroll
            for (int tt = 0; tt < TT; ++tt) mloc[j] = fmaxf(mloc[j], fmaxf(s[tt][j], s[tt][j + 2]));
        }
        online_max(mloc, lane);
        softmax_weights<TT>(s);
        pv<TT>(s, vbase, lane);
    }

    // Raise the running maxima to cover this tile's scores (mloc: this
    // lane's maxima).  When no lane's score passes its head's running
    // maximum, nothing moves and the shuffles are skipped; otherwise the
    // maxima are reduced over the tile's token lanes and the accumulators and
    // lane sums rescaled.
    __device__ __forceinline__ void online_max(float (&mloc)[2], int) {
        if (!__any_sync(FULL, mloc[0] > m_run[0] || mloc[1] > m_run[1])) return;
        float alpha[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = mloc[j];
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
            const float mnew = fmaxf(m_run[j], mx);
            alpha[j] = mnew == -CUDART_INF_F ? 1.f : fast_exp2(m_run[j] - mnew);
            m_run[j] = mnew;
            l_run[j] *= alpha[j];
        }
        rescale(alpha[0], alpha[1]);
    }

    __device__ __forceinline__ void rescale(float a0, float a1) {
        if (__all_sync(FULL, a0 == 1.f && a1 == 1.f)) return;
        const float2 a2 = make_float2(a0, a1);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            float2 lo = __fmul2_rn(make_float2(oacc[mt][0], oacc[mt][1]), a2);
            float2 hi = __fmul2_rn(make_float2(oacc[mt][2], oacc[mt][3]), a2);
            oacc[mt][0] = lo.x; oacc[mt][1] = lo.y; oacc[mt][2] = hi.x; oacc[mt][3] = hi.y;
        }
    }

    // scores -> weights exp2(s - m) in place; the lane's own sums go into
    // l_run (the token lanes' sums are added in fold())
    template <int NT>
    __device__ __forceinline__ void softmax_weights(float (&s)[NT][4]) {
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = e & 1;
                const float pe = m_run[j] == -CUDART_INF_F ? 0.f : fast_exp2(s[tt][e] - m_run[j]);
                s[tt][e] = pe;
                l_run[j] += pe;
            }
    }

    // P^T operands of 16-token tile: hi + lo 16-bit halves of the weights
    // (paired groups: one operand, hi in columns 0..3 and lo in 4..7)
    template <typename M>
    __device__ __forceinline__ void p_operands(const float (&p)[4], int lane, uint32_t (&bh)[2],
                                               uint32_t (&bl)[2]) const {
        const uint32_t h01 = M::pack(p[0], p[1]);
        const uint32_t h23 = M::pack(p[2], p[3]);
        const float2 f01 = M::unpack(h01), f23 = M::unpack(h23);
        const uint32_t l01 = M::pack(p[0] - f01.x, p[1] - f01.y);
        const uint32_t l23 = M::pack(p[2] - f23.x, p[3] - f23.y);
        if constexpr (kPairHL) {
            const bool lo = (lane & 3) >= 2;       // columns 4..7
            bh[0] = movm_t(lo ? l01 : h01);
            bh[1] = movm_t(lo ? l23 : h23);
        } else {
            bh[0] = movm_t(h01); bh[1] = movm_t(h23);
            bl[0] = movm_t(l01); bl[1] = movm_t(l23);
        }
    }

    // -- O^T += V_blk^T P^T ----------------------------------------------------
    template <int NT>
    __device__ __forceinline__ void pv(const float (&s)[NT][4], uint32_t vbase, int lane) {
        const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            uint32_t bh[2], bl[2];
            p_operands<Mma<T>>(s[tt], lane, bh, bl);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                ldsm_x4_t(a, swz(vbase, tt * 16 + (mi >> 1) * 8 + r8, mt * 2 + (mi & 1)));
                Mma<T>::run(oacc[mt], a, bh[0], bh[1]);
                if constexpr (!kPairHL) Mma<T>::run(oacc[mt], a, bl[0], bl[1]);
            }
        }
    }

    // End of a piece: the lo-column accumulators join the hi ones (paired
    // groups) and the token lanes' sums are added up.
    __device__ __forceinline__ void fold(int) {
        if constexpr (kPairHL) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int c = 0; c < 4; ++c) oacc[mt][c] += __shfl_xor_sync(FULL, oacc[mt][c], 2);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[j] += __shfl_xor_sync(FULL, l_run[j], 4);
            l_run[j] += __shfl_xor_sync(FULL, l_run[j], 8);
            l_run[j] += __shfl_xor_sync(FULL, l_run[j], 16);
        }
    }

    // Normalise the warp's state and write `out` or the partial slot.
    __device__ __forceinline__ void merge_store(int lane, const PieceOut& po) const {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int h = 2 * tig + j;
            if (h >= G) continue;
            float M = m_run[j];
            const float c0 = M == -CUDART_INF_F ? 0.f : 1.f;   // an empty state counts zero
            float den = c0 * l_run[j];
            float fs = 1.f, fp = 0.f;                 // cascade: fold the prefix state
            if (po.complete && po.pst_lse != nullptr) M = fold_state(M, den, po.pst_lse[h], fs, fp);
            const float inv = den > 0.f ? 1.f / den : 0.f;
            // every load of the merge before the first store: the compiler
            // cannot move a load above a store it might alias
            float v[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int d = dim(mt, gid, hf);
                    float num = c0 * oacc[mt][j + 2 * hf];
                    if (po.complete && po.pst_lse != nullptr) num = num * fs + po.pst_o[h * D + d] * fp;
                    v[mt][hf] = num * inv;
                }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int d = dim(mt, gid, hf);
                    if (po.complete)
                        static_cast<T*>(po.out)[h * D + d] = Elt<T>::store(v[mt][hf]);
                    else
                        po.part_o[h * D + d] = v[mt][hf];
                }
            if (!po.complete && gid == 0)
                po.part_lse[h] = den > 0.f ? M + fast_log2(den) : -CUDART_INF_F;
        }
    }
};

// Block size 8 on the tensor cores: a work unit is two consecutive logical
// blocks, loaded into one 16-row tile (block i of the unit is rows
// 8 i .. 8 i + 7, the 2 KB at byte 2048 i: its first 64-dim half, then its
// second, the same 128-byte swizzle pattern), and attended exactly like a
// 16-token block.
template <typename T, int D, int G>
struct TcPolicy8x2 : TcPolicy<T, D, G, 16, false, true> {
    static constexpr int kUnitBlocks = 2;
    __device__ __forceinline__ TcPolicy8x2(float2* a, float2* b)
        : TcPolicy<T, D, G, 16, false, true>(a, b) {}
};

// ---------------------------------------------------- 8-bit pools on MMA --
// K/V stored as 8-bit codes ("Part 3: single node", random-liu.github.io,
// ch. 10: a token's K and V are scaled and rounded to 8 bits when written and
// turned back into wider numbers when read): FP8 E4M3 with one scale per pool,
// or INT8 with one fp32 scale per (block, KV head, token row).  The tiles
// arrive by TMA with the 128-byte swizzle (one 128-byte row per token); INT8
// scales come by bulk copy into a small ring beside them.  The warp builds
// the f16 MMA fragments straight from the codes in registers -- every E4M3
// value and every integer in [-128, 127] is an f16, so the conversion is
// exact -- with no shared-memory round trip:
//   * QK (A = K rows): MMA k-slot 2 tig + {0, 1, 8, 9} of k-step ks stands for
//     dim 32 tig + 4 ks + {0, 1, 2, 3} (a relabelling of the dot product's
//     terms, applied to Q too), so a lane's K codes for all k-steps are two
//     16-byte chunks per row;
//   * PV (A = V^T): output row (m-slot) 16 mt + gid + 8 hf stands for dim
//     16 gid + 2 mt + hf, so a lane's V codes are one 16-byte chunk of each of
//     its four token rows; the merge writes every value to its own dim.
// Both read patterns are bank-conflict-free under the swizzle.  The scales
// never pass through f16: Q is held as f16 * 2^e (a power of two per piece
// keeps the group's largest |q| below 2^15; bf16 and f16 queries convert
// exactly) and a score is acc * scale * log2(e) * 2^-e * kscale_t in fp32; P
// is multiplied by vscale_t / vref (vref the tile's largest V scale) before
// its hi + lo f16 split, and the accumulator is kept as O / R with R the last
// vref (a change of R rescales it with the softmax alpha).
constexpr int kFmtE4M3 = 0;
constexpr int kFmtInt8 = 1;

// Four codes (bytes 0..3 of w) -> f16x2 of bytes (0, 1) and of bytes (2, 3).
template <int FMT>
__device__ __forceinline__ void cvt4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if constexpr (FMT == kFmtE4M3) {
        // the two 16-bit halves of w, each a pair of codes, straight into the
        // conversion (E4M3 -> f16 is exact)
        asm("{ .reg .b16 l, h;\n"
            "  mov.b32 {l, h}, %2;\n"
            "  cvt.rn.f16x2.e4m3x2 %0, l;\n"
            "  cvt.rn.f16x2.e4m3x2 %1, h; }"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    } else {
        // two's complement byte b -> f16 (1024 + (b ^ 0x80)) - 1152 = b
        const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        const uint32_t x = w ^ 0x80808080u;
        const uint32_t l = __byte_perm(x, 0x64646464u, 0x7150);
        const uint32_t h = __byte_perm(x, 0x64646464u, 0x7352);
        const __half2 lh = __hsub2(*reinterpret_cast<const __half2*>(&l), bias);
        const __half2 hh = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
        lo = *reinterpret_cast<const uint32_t*>(&lh);
        hi = *reinterpret_cast<const uint32_t*>(&hh);
    }
}

template <typename T, int D, int G, int FMT>
struct Tc8Policy : TcPolicy<T, D, G, 16, true> {
    using Base = TcPolicy<T, D, G, 16, true>;
    static_assert(D == 128, "one 128-byte code row per token");
    static constexpr int KS = Base::KS;
    static constexpr int MT = Base::MT;
    static constexpr bool kSwizzled = true;
    static constexpr bool kH2 = false;           // one 128-byte code row: 3-D maps
    // A ring of two 8 KB stages per warp (32 code rows of K and V) leaves room
    // for 3 CTAs per SM, and so do larger blocks: up to 168 registers a
    // thread cost no occupancy (the two-tile step needs about 160).
    static constexpr int kMinBlocks = 3;
    static constexpr int kKvBytes = 1;
    static constexpr int kScaleBytes = FMT == kFmtInt8 ? 4 : 0;

    float qs;             // scale * log2(e) * 2^-e (* the FP8 K scale)
    float vq;             // FP8: the V scale; INT8: 1
    float kq;             // FP8: the K scale; INT8: 1
    float R;              // the accumulators hold O / R
    float Rinv;           // INT8: 1 / R (0 while R is 0)

    __device__ __forceinline__ Tc8Policy(float2* a, float2* b) : Base(a, b) {}

    __device__ __forceinline__ void setup(const Params& p) {
        kq = FMT == kFmtE4M3 ? p.fp8_k_scale : 1.f;
        vq = FMT == kFmtE4M3 ? p.fp8_v_scale : 1.f;
    }

    // 16-byte chunk c of row r of a 128-byte-swizzled tile (1 KB-aligned base)
    __device__ static __forceinline__ uint4 chunk(const unsigned char* tile, int r, int c) {
        return *reinterpret_cast<const uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4));
    }

    __device__ __forceinline__ void begin(const T* qp, float qscale, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        float2 qf[KS][2];
        float amax = 0.f;
        const int hq = Base::col_head(gid);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint2 raw = make_uint2(0u, 0u);
            if (hq >= 0) raw = __ldg(reinterpret_cast<const uint2*>(qp + hq * D + 32 * tig + 4 * ks));
            qf[ks][0] = Mma<T>::unpack(raw.x);
            qf[ks][1] = Mma<T>::unpack(raw.y);
#pragma unroll
            for (int j = 0; j < 2; ++j)
                amax = fmaxf(amax, fmaxf(fabsf(qf[ks][j].x), fabsf(qf[ks][j].y)));
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, off));
        // 2^e with amax * 2^e in [2^14, 2^15): exponent field of amax, clamped
        int e = 0;
        if (amax > 0.f && amax <= 3.0e38f) {
            const int ex = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 126;   // amax < 2^ex
            e = min(max(15 - ex, -120), 120);
        }
        const float up = __uint_as_float((uint32_t)(e + 127) << 23);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const __half2 h = __floats2half2_rn(qf[ks][j].x * up, qf[ks][j].y * up);
                this->qb[ks][j] = *reinterpret_cast<const uint32_t*>(&h);
            }
        qs = qscale * kq * __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            this->oacc[mt][0] = this->oacc[mt][1] = this->oacc[mt][2] = this->oacc[mt][3] = 0.f;
        this->m_run[0] = this->m_run[1] = -CUDART_INF_F;
        this->l_run[0] = this->l_run[1] = 0.f;
        // INT8: R is the largest V scale met so far in the piece (raised, with
        // a rescale, when a tile brings a larger one); FP8: the pool's V scale
        R = FMT == kFmtInt8 ? 0.f : vq;
        Rinv = 0.f;
    }

    // Two 16-token tiles per step (rows t0 .. t0 + 31): both tiles' QK
    // products are issued together, one max vote covers the 32 tokens, then
    // both tiles' PV products.  When the rows end inside the first tile the
    // second tile's scores are masked and its V rows read as zeros; its K
    // reads stay inside the stage (a K tile is followed by its V tile).
    __device__ __forceinline__ void block(const unsigned char* Ks, const unsigned char* Vs,
                                          const float* sc, int n_valid, int bs, float, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        for (int t0 = 0; t0 < n_valid; t0 += 32) {
            // -- S^T of the two tiles: 16 tokens x the group's heads each ------
            float acc[2][2][4];
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
                for (int c = 0; c < 2; ++c) acc[x][c][0] = acc[x][c][1] = acc[x][c][2] = acc[x][c][3] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t wa[2][4], wb[2][4];
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const unsigned char* Kt = Ks + (t0 + 16 * x) * 128;
                    const uint4 ra = chunk(Kt, gid, 2 * tig + h), rb = chunk(Kt, gid + 8, 2 * tig + h);
                    wa[x][0] = ra.x; wa[x][1] = ra.y; wa[x][2] = ra.z; wa[x][3] = ra.w;
                    wb[x][0] = rb.x; wb[x][1] = rb.y; wb[x][2] = rb.z; wb[x][3] = rb.w;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        uint32_t a[4];
                        cvt4<FMT>(wa[x][q], a[0], a[2]);
                        cvt4<FMT>(wb[x][q], a[1], a[3]);
                        Mma<__half>::run(acc[x][q & 1], a, this->qb[4 * h + q][0],
                                         this->qb[4 * h + q][1]);
                    }
            }
            float s[2][4];
            float sv[2][2];                         // INT8: the V scales of the lane's rows
            float smax = 0.f;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int ta = t0 + 16 * x + gid, tb = ta + 8;
                const bool v0 = ta < n_valid, v1 = tb < n_valid;
                float fa = qs, fb = qs;
                sv[x][0] = sv[x][1] = 0.f;
                if constexpr (FMT == kFmtInt8) {
                    fa *= v0 ? sc[ta] : 0.f;
                    fb *= v1 ? sc[tb] : 0.f;
                    sv[x][0] = v0 ? sc[bs + ta] : 0.f;
                    sv[x][1] = v1 ? sc[bs + tb] : 0.f;
                    smax = fmaxf(smax, fmaxf(sv[x][0], sv[x][1]));
                }
                s[x][0] = v0 ? (acc[x][0][0] + acc[x][1][0]) * fa : -CUDART_INF_F;
                s[x][1] = v0 ? (acc[x][0][1] + acc[x][1][1]) * fa : -CUDART_INF_F;
                s[x][2] = v1 ? (acc[x][0][2] + acc[x][1][2]) * fb : -CUDART_INF_F;
                s[x][3] = v1 ? (acc[x][0][3] + acc[x][1][3]) * fb : -CUDART_INF_F;
            }
            // -- online softmax, heads 2 tig (j = 0) and 2 tig + 1 (j = 1); INT8:
            // the running largest V scale R moves with the maxima ----------------
            const float mloc[2] = {fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2])),
                                   fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]))};
            if (__any_sync(FULL, mloc[0] > this->m_run[0] || mloc[1] > this->m_run[1] ||
                                     (FMT == kFmtInt8 && smax > R))) {
                float alpha[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float mx = mloc[j];
                    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
                    const float mnew = fmaxf(this->m_run[j], mx);
                    alpha[j] = mnew == -CUDART_INF_F ? 1.f : fast_exp2(this->m_run[j] - mnew);
                    this->m_run[j] = mnew;
                    this->l_run[j] *= alpha[j];
                }
                float rf = 1.f;
                if constexpr (FMT == kFmtInt8) {
                    float mx = smax;
#pragma unroll
                    for (int off = 16; off >= 4; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
                    if (mx > R) {                     // (uniform: every lane sees all token rows)
                        Rinv = __frcp_rn(mx);
                        rf = R * Rinv;
                        R = mx;
                    }
                }
                this->rescale(alpha[0] * rf, alpha[1] * rf);
            }
            this->template softmax_weights<2>(s);
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                // V scales: P' = P * vscale_t / R
                if constexpr (FMT == kFmtInt8) {
                    const float wa = sv[x][0] * Rinv, wb = sv[x][1] * Rinv;
                    s[x][0] *= wa; s[x][1] *= wa; s[x][2] *= wb; s[x][3] *= wb;
                }
                uint32_t bh[2], bl[2];
                this->template p_operands<Mma<__half>>(s[x], lane, bh, bl);
                // -- O^T += V_tile^T P'^T: token rows 2 tig, 2 tig + 1, + 8, + 9 --
                // (rows past the sequence end read as zero codes: P' is 0 there,
                // but an E4M3 NaN code would still poison the MMA)
                const int tv = t0 + 16 * x;
                const unsigned char* Vt = Vs + tv * 128;
                uint32_t vw[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 2 * tig + (i & 1) + 8 * (i >> 1);
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (tv + r < n_valid) v = chunk(Vt, r, gid);
                    vw[i][0] = v.x; vw[i][1] = v.y; vw[i][2] = v.z; vw[i][3] = v.w;
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    // dims 16 gid + 2 mt (+1): bytes 2 mt, 2 mt + 1 of each row's chunk
                    const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                    const uint32_t x01 = __byte_perm(vw[0][mt >> 1], vw[1][mt >> 1], sel);
                    const uint32_t x23 = __byte_perm(vw[2][mt >> 1], vw[3][mt >> 1], sel);
                    uint32_t a[4];
                    cvt4<FMT>(x01, a[0], a[1]);
                    cvt4<FMT>(x23, a[2], a[3]);
                    Mma<__half>::run(this->oacc[mt], a, bh[0], bh[1]);
                    if constexpr (!Base::kPairHL) Mma<__half>::run(this->oacc[mt], a, bl[0], bl[1]);
                }
            }
        }
    }

    // Before the warp merge: the accumulators become O itself.
    __device__ __forceinline__ void fold(int lane) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) this->oacc[mt][i] *= R;
        R = 1.f;
        Base::fold(lane);
    }
};

// Two consecutive 16-row blocks per work unit (the kernel puts the second
// block's code rows, and its INT8 scales, right after the first's).
template <typename T, int D, int G, int FMT>
struct Tc8Policy2 : Tc8Policy<T, D, G, FMT> {
    static constexpr int kUnitBlocks = 2;
    __device__ __forceinline__ Tc8Policy2(float2* a, float2* b) : Tc8Policy<T, D, G, FMT>(a, b) {}
};

// ---------------------------------------------- cross-range partial merge --
// Pieces of one (b, g) cut across work ranges (a warp's in the split kernel,
// a CTA's in the prefix pass): range c holds its piece in slot (c, 0) when
// the piece is its first, else (c, 1).  Each cut piece is counted in the
// (b, g)'s 16-byte counter {tag, count}: `tag` is a 64-bit value drawn at
// random for every call, and a counter whose tag is not the call's counts as
// zero -- so the workspace needs no clearing: a stale counter of an earlier
// call has that call's tag, and leftover data holds the call's tag only with
// probability 2^-64.  Counting is a 128-bit compare-and-swap; the worker
// whose count completes the set merges.
__device__ __forceinline__ void cas128(unsigned long long* p, unsigned long long& lo,
                                       unsigned long long& hi, unsigned long long nlo,
                                       unsigned long long nhi) {
    asm volatile(
        "{ .reg .b128 d, b, c; mov.b128 b, {%0, %1}; mov.b128 c, {%2, %3};"
        " atom.relaxed.gpu.global.cas.b128 d, [%4], b, c; mov.b128 {%0, %1}, d; }"
        : "+l"(lo), "+l"(hi)
        : "l"(nlo), "l"(nhi), "l"(p)
        : "memory");
}
__device__ __forceinline__ bool count_piece(unsigned long long* ctr, unsigned long long tag,
                                            int pieces) {
    unsigned long long lo = tag, hi = 0;           // a first guess: this call's, none counted
    while (true) {
        const unsigned long long elo = lo, ehi = hi;
        const unsigned long long next = (lo == tag ? hi : 0ull) + 1ull;
        cas128(ctr, lo, hi, tag, next);            // lo, hi: the value found
        if (lo == elo && hi == ehi) return next == (unsigned long long)pieces;
    }
}

// Fold one normalised state (log2-sum-exp l, output o[0..N)) into a running
// (base M, denominator den, numerator acc).
template <int N>
__device__ __forceinline__ void lse_add(float& M, float& den, float* acc, float l, const float* o) {
    const float M2 = fmaxf(M, l);
    if (M2 == -CUDART_INF_F) return;
    const float a = M == -CUDART_INF_F ? 0.f : fast_exp2(M - M2);
    const float w = l == -CUDART_INF_F ? 0.f : fast_exp2(l - M2);
    den = den * a + w;
#pragma unroll
    for (int k = 0; k < N; ++k) acc[k] = acc[k] * a + w * o[k];
    M = M2;
}

template <int N>
__device__ __forceinline__ void load_row(float* v, const float* src, bool cached_l2_only) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int k = 0; k < N; k += 4) {
            const float4 x = cached_l2_only ? __ldcg(reinterpret_cast<const float4*>(src + k))
                                            : *reinterpret_cast<const float4*>(src + k);
            v[k] = x.x; v[k + 1] = x.y; v[k + 2] = x.z; v[k + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < N; ++k) v[k] = cached_l2_only ? __ldcg(src + k) : src[k];
    }
}

// One warp merges the partial states that a segment cut across ranges c0..c1
// left in their slots (range c0's piece in slot slot0 of c0, every later
// range's in slot 0), plus an optional extra state (x_o, x_lse; null for none).  Each
// is a normalised output [R][D] with its log2-sum-exp [R]:
//   out[r, d] = sum_i 2^(lse_i[r] - M) o_i[r, d] / sum_i 2^(lse_i[r] - M).
// A lane owns EPL consecutive dims of one row; the slots are read
// kMergeBatch at a time so that their loads are in flight together.  store(r, d0, vals, lse)
// takes row r's merge_epl<R, D>() results from dim d0 and the row's merged
// log2-sum-exp.
constexpr int kMergeBatch = 2;   // slots whose loads merge_cut issues together

template <int R, int D>
__host__ __device__ constexpr int merge_epl() {
    return ((R * D) % 256 == 0 && D % 8 == 0) ? 8 : ((R * D) % 128 == 0 && D % 4 == 0) ? 4
         : ((R * D) % 64 == 0 && D % 2 == 0) ? 2 : 1;
}

// merge_cut over the element passes pass0, pass0 + pstep, ... (one warp each
// when several warps share a segment), BATCH slots in flight at a time.
template <int R, int D, int BATCH, class Store>
__device__ __forceinline__ void merge_slots(const float* part_o, const float* part_lse, int c0,
                                            int c1, int slot0, const float* x_o,
                                            const float* x_lse, int lane, int pass0, int pstep,
                                            Store&& store) {
    constexpr int E = R * D;
    constexpr int EPL = merge_epl<R, D>();
    static_assert(E % (32 * EPL) == 0, "rows x dims must be whole warps of lanes");
#pragma unroll 1
    for (int pass = pass0; pass < E / (32 * EPL); pass += pstep) {
        const int e0 = (pass * 32 + lane) * EPL;
        const int r = e0 / D, d0 = e0 % D;
        float M = -CUDART_INF_F, den = 0.f, acc[EPL];
#pragma unroll
        for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
        for (int c = c0; c <= c1; c += BATCH) {
            float ls[BATCH], ov[BATCH][EPL];
#pragma unroll
            for (int t = 0; t < BATCH; ++t) {
                const int cc = c + t;
                const size_t slot = (size_t)cc * 2 + (cc == c0 ? slot0 : 0);
                ls[t] = -CUDART_INF_F;
                if (cc <= c1) {
                    ls[t] = __ldcg(part_lse + slot * R + r);
                    load_row<EPL>(ov[t], part_o + (slot * R + r) * D + d0, true);
                }
            }
#pragma unroll
            for (int t = 0; t < BATCH; ++t)
                if (c + t <= c1) lse_add<EPL>(M, den, acc, ls[t], ov[t]);
        }
        if (x_lse != nullptr) {
            float xv[EPL];
            load_row<EPL>(xv, x_o + r * D + d0, false);
            lse_add<EPL>(M, den, acc, x_lse[r], xv);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
        for (int k = 0; k < EPL; ++k) acc[k] *= inv;
        store(r, d0, acc, den > 0.f ? M + fast_log2(den) : -CUDART_INF_F);
    }
}

template <int R, int D, class Store>
__device__ __forceinline__ void merge_cut(const float* part_o, const float* part_lse, int c0,
                                          int c1, int slot0, const float* x_o, const float* x_lse,
                                          int lane, Store&& store) {
    merge_slots<R, D, kMergeBatch>(part_o, part_lse, c0, c1, slot0, x_o, x_lse, lane, 0, 1,
                                   static_cast<Store&&>(store));
}

// ------------------------------------------------- block-wide scans --
// One int per thread, every thread of the CTA calls; `scratch` holds a word
// per warp.  Exclusive sum (and the total), exclusive max of non-negatives.
__device__ __forceinline__ int block_excl_sum(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        if (w < warp) off += scratch[w];
        tot += scratch[w];
    }
    __syncthreads();
    if (total) *total = tot;
    return off + x - v;
}
__device__ __forceinline__ int block_excl_max(int v, int* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x = max(x, y);
    }
    const int up = __shfl_up_sync(FULL, x, 1);
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    int off = lane > 0 ? up : 0;
    for (int w = 0; w < warp; ++w) off = max(off, scratch[w]);
    __syncthreads();
    return off;
}

// ------------------------------------------- cascade groups (both passes) --
// A group (first member, members, shared leading blocks) is used when it lies
// inside the batch, starts at or after the end of every earlier group, and at
// least one work unit is shared (the block count is clamped to each member's
// count of full blocks -- blocks whose every row holds one of its tokens --
// then counted in whole units of `ub` blocks: both passes must use the same
// unit).  Both passes compact the used groups, in order,
// into shared memory (vg: first[n], size[n], shared units[n]) and return n;
// unused groups set KV_DEVERR_GROUP_RANGE when malformed.  Every thread of
// the CTA calls.
__device__ __forceinline__ int load_groups(const int32_t* g_first, const int32_t* g_size,
                                           const int32_t* g_blocks, int K, const int32_t* seq_lens,
                                           int B, int bs, int cap, int ub, int* vg, int* scratch,
                                           int* err) {
    const int per = (K + (int)blockDim.x - 1) / (int)blockDim.x;
    const int k0 = min(K, (int)threadIdx.x * per), k1 = min(K, k0 + per);
    auto raw_end = [&](int k) {
        const long long e = (long long)g_first[k] + (long long)max(g_size[k], 0);
        return (int)min(max(e, 0ll), 2147483647ll);
    };
    auto shared_blocks = [&](int k, int before, bool& ok) {
        const int first = g_first[k], size = g_size[k];
        int blocks = g_blocks[k];
        ok = first >= 0 && size >= 1 && (long long)first + size <= B && blocks >= 0 &&
             first >= before;
        if (!ok) return 0;
        for (int m = 0; m < size; ++m)
            blocks = min(blocks, min(max(seq_lens[first + m], 0), cap) / bs);
        return blocks / ub;
    };
    int cmax = 0;
    for (int k = k0; k < k1; ++k) cmax = max(cmax, raw_end(k));
    const int before0 = block_excl_max(cmax, scratch);
    int before = before0, keep = 0;
    bool bad = false;
    for (int k = k0; k < k1; ++k) {
        bool ok;
        keep += shared_blocks(k, before, ok) > 0;
        bad |= !ok;
        before = max(before, raw_end(k));
    }
    if (bad && blockIdx.x == 0) atomicOr(err, KV_DEVERR_GROUP_RANGE);
    int n = 0;
    int idx = block_excl_sum(keep, scratch, &n);
    before = before0;
    for (int k = k0; k < k1; ++k) {
        bool ok;
        const int blocks = shared_blocks(k, before, ok);
        before = max(before, raw_end(k));
        if (blocks > 0) {
            vg[idx] = g_first[k];
            vg[K + idx] = g_size[k];
            vg[2 * K + idx] = blocks;
            ++idx;
        }
    }
    __syncthreads();
    return n;
}

// Shared leading units of sequence b (0 outside every used group).
__device__ __forceinline__ int group_skip(const int* vg, int K, int n, int b) {
    if (n == 0 || b < vg[0]) return 0;
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (vg[mid] <= b) lo = mid; else hi = mid;
    }
    return b < vg[lo] + vg[K + lo] ? vg[2 * K + lo] : 0;
}

// -- the units of a call ------------------------------------------------------
// prefix[b] (shared memory) = the units of KV head 0 in sequences before b:
// each sequence contributes its blocks (clamped to the table's capacity, in
// units of bsu tokens) less, for cascade decode, the leading units the
// shared-prefix pass attended (skip_s[b]).  prefix[B] is the total.  Every
// thread of the CTA calls; `report` flags contexts longer than the table.
__device__ __forceinline__ void unit_prefix(const Params& p, unsigned char* smem, const Layout& lay,
                                            int bsu, bool cascade, bool report) {
    const int B = p.batch, tid = threadIdx.x, nthreads = blockDim.x;
    const int cap = p.max_blocks * p.bs;
    int* warp_tot = reinterpret_cast<int*>(smem + lay.misc) + 8;
    int* prefix = reinterpret_cast<int*>(smem + lay.prefix);
    int* skip_s = reinterpret_cast<int*>(smem + lay.skip);
    // cascade: the leading units the shared-prefix pass attended
    int* vg = reinterpret_cast<int*>(smem + lay.groups);
    const int nvg = cascade ? load_groups(p.g_first, p.g_size, p.g_blocks, p.num_groups,
                                          p.seq_lens, B, p.bs, cap, bsu / p.bs, vg, warp_tot,
                                          p.err)
                            : 0;
    const int per = (B + nthreads - 1) / nthreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int local = 0;
    bool over = false;
    for (int b = b0; b < b1; ++b) {
        const int L = p.seq_lens[b];
        over |= L > cap;
        const int nb = (min(max(L, 0), cap) + bsu - 1) / bsu;
        const int skip = cascade ? min(group_skip(vg, p.num_groups, nvg, b), nb) : 0;
        if (cascade) skip_s[b] = skip;
        local += nb - skip;
    }
    if (over && report) atomicOr(p.err, KV_DEVERR_SEQ_RANGE);
    int total = 0;
    int run = block_excl_sum(local, warp_tot, &total);
    for (int b = b0; b < b1; ++b) {
        prefix[b] = run;
        const int nb = (min(max(p.seq_lens[b], 0), cap) + bsu - 1) / bsu;
        run += nb - (cascade ? skip_s[b] : 0);
    }
    if (tid == 0) prefix[B] = total;
}

// ------------------------------------------------------------ split kernel --
template <typename T, int D, int G, class Pol>
__global__ void __launch_bounds__(SPLIT_THREADS, Pol::kMinBlocks) paged_decode_split(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const Params p) {
    constexpr int ELT = Pol::kKvBytes;             // bytes per pool element
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_align_1k(smem_raw);
    const int B = p.batch, S = p.stages, H = p.num_kv_heads, bs = p.bs;
    constexpr int UB = Pol::kUnitBlocks;           // pool blocks per work unit
    const int bsu = bs * UB;                       // tokens per work unit
    const Layout lay(S, B, bsu, G, D, ELT, p.num_groups, Pol::kScaleBytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.full);
    volatile int* valid = reinterpret_cast<volatile int*>(smem + lay.valid);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc);
    const int* prefix = reinterpret_cast<const int*>(smem + lay.prefix);
    const int* skip_s = reinterpret_cast<const int*>(smem + lay.skip);
    unsigned char* ring = smem + lay.ring;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cap = p.max_blocks * bs;              // longest context a table can hold
    // cascade: the groups' shared prefix is counted in whole units of UB
    // blocks (load_groups), so paired-block units skip it like single ones
    const bool cascade = p.num_groups > 0;

    // -- 1. the blocks-per-sequence prefix of the clamped lengths -----------
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(smem_u32(&full[s]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_launch_dependents();
    // A plain decode waits here for the kernels before it (the append writes
    // K/V rows).  A cascade decode's prefix pass lets this kernel in only
    // after its own wait, so the pool is complete: this kernel streams its
    // blocks at once and waits for the prefix pass just before it first
    // reads the prefix states (and, at the latest, before each warp exits,
    // so that this grid never ends before the prefix pass).
    if (!cascade) pdl_wait();
    unit_prefix(p, smem, lay, bsu, cascade, blockIdx.x == 0);
    __syncthreads();
    // sequences no unit covers: zeros, or (cascade) the prefix state alone
    for (int b = blockIdx.x; b < B; b += gridDim.x)
        if (prefix[b + 1] == prefix[b]) {
            T* ob = static_cast<T*>(p.out) + (size_t)b * p.num_q_heads * D;
            const bool has = cascade && skip_s[b] > 0;
            if (has) pdl_wait();                   // b's prefix state is written
            for (int i = tid; i < p.num_q_heads * D; i += SPLIT_THREADS) {
                const size_t row = (size_t)b * p.num_q_heads + i / D;
                ob[i] = Elt<T>::store(has ? p.pst_o[row * D + i % D] : 0.f);
            }
        }

    // -- 2. this warp's range of units -------------------------------------
    // Every warp is a worker of its own: the units (b, g, j) are cut into
    // equal contiguous ranges, one per warp of the grid, so no warp waits on
    // another of its CTA from here on.
    const int U = prefix[B] * H;
    const int worker = blockIdx.x * NCW + warp;
    const WorkCut cut(prefix, B, H, p.num_ctas * NCW);
    const int start = cut.start_unit(worker);
    const int end = cut.start_unit(worker + 1);
    if (start >= end) {
        if (cascade) pdl_wait();
        return;
    }

    // ------------------------------------------------------ the warp's work --
    const int w = warp;
    float2* pb = reinterpret_cast<float2*>(smem + lay.pbuf) + w * bs * G;
    float2* ab = reinterpret_cast<float2*>(smem + lay.abuf) + w * G;
    // cascade: this warp's copy of the prefix state, [G][D] then [G]
    float* pst_s = reinterpret_cast<float*>(smem + lay.pst + w * lay.pst_bytes);
    const T* qbase = static_cast<const T*>(p.q);
    T* obase = static_cast<T*>(p.out);
    Pol pol(pb, ab);
    pol.setup(p);

    // -- 3. loads: each warp issues the TMA copies of its own units ---------
    // Warp w owns stages w + NCW j (j < S / NCW); unit k = uu - start goes to
    // j = k % (S / NCW).  After attending unit k the warp loads unit
    // k + S / NCW into the same stage.  A box is one
    // block's rows of one 128-byte half (swizzled) or of the whole row; the
    // halves of a unit's tile are bsu rows apart.
    constexpr int kBoxes = Pol::kSwizzled ? D * ELT / 128 : 1;
    const uint32_t box_bytes = (uint32_t)bs * (Pol::kSwizzled ? 128u : (uint32_t)(D * ELT));
    const uint32_t half_bytes = (uint32_t)bsu * (Pol::kSwizzled ? 128u : (uint32_t)(D * ELT));
    const int per_warp = S / NCW;                  // stages this warp owns
    // block ids of this warp's issue i (unit start + i): the first and
    // (UB = 2) the second, -2 when the sequence ends inside the first; -1: none
    auto fetch = [&](int i, int& id, int& id2, int& gg) {
        id = -1;
        id2 = -2;
        gg = 0;
        const int uu = start + i;
        if (uu < end) {
            const int b = find_seq(prefix, B, uu, H);
            const int nb = prefix[b + 1] - prefix[b];
            const int r = uu - prefix[b] * H;
            gg = r / nb;
            const int lb = ((cascade ? skip_s[b] : 0) + (r - gg * nb)) * UB;
            const int32_t* row = p.block_tables + (size_t)b * p.max_blocks;
            id = __ldg(row + lb);
            if (UB == 2 && (lb + 1) * bs < min(max(p.seq_lens[b], 0), cap))
                id2 = __ldg(row + lb + 1);
        }
    };
    int nx = 0;                                    // issues made (= unit nx)
    int na = 0;                                    // lane 0: issues that reached the barrier
    int ib = 0;                                    // first issue of the fetched batch
    int is = w;                                    // stage of issue nx
    // lane l holds issue ib + l and, one batch ahead (its table loads in
    // flight meanwhile), issue ib + 32 + l
    int id_b, id2_b, g_b, id_n, id2_n, g_n;
    fetch(lane, id_b, id2_b, g_b);
    fetch(32 + lane, id_n, id2_n, g_n);
    const int n_issue = end - start;
    auto issue_next = [&]() {
        if (nx >= n_issue) return;
        if (nx - ib == 32) {                       // (warp-uniform)
            ib += 32;
            id_b = id_n; id2_b = id2_n; g_b = g_n;
            fetch(ib + 32 + lane, id_n, id2_n, g_n);
        }
        const int i = nx - ib;
        const int id = __shfl_sync(FULL, id_b, i);
        const int id2 = __shfl_sync(FULL, id2_b, i);
        const int gg = __shfl_sync(FULL, g_b, i);
        const int st = is;
        ++nx;
        is += NCW;
        if (is >= S) is -= S;
        // After an abort a stage's barrier is not touched again: its last
        // phase may still be waiting for bytes, and an arrival on it would
        // be one too many.  The issues before that are drained at the end.
        if (lane == 0 && *abort_flag == 0) {
            const uint32_t fb = smem_u32(&full[st]);
            const bool second = UB == 2 && id2 != -2;   // the unit's second block
            ++na;
            if (id >= 0 && id < p.num_blocks && (!second || (id2 >= 0 && id2 < p.num_blocks))) {
                valid[st] = 1;
                // No proxy fence: every read of the stage fed an MMA or FMA that
                // the warp issued before this point, so the reads are complete;
                // a policy that writes into a stage fences those writes itself.
                mbar_arrive_tx(fb, second ? lay.tx_bytes : lay.tx_bytes / UB);
                const uint32_t dst = smem_u32(ring + (size_t)st * lay.stage_bytes);
                const uint32_t vdst = dst + (uint32_t)(bsu * D * ELT);
                if constexpr (Pol::kH2) {
                    // one copy per block: both halves, [half][bs rows][128 B]
                    const uint32_t blk = 2u * (uint32_t)bs * 128u;
                    tma_load_4d(dst, &tmap_k, 0, id * bs, 0, gg, fb);
                    tma_load_4d(vdst, &tmap_v, 0, id * bs, 0, gg, fb);
                    if (second) {
                        tma_load_4d(dst + blk, &tmap_k, 0, id2 * bs, 0, gg, fb);
                        tma_load_4d(vdst + blk, &tmap_v, 0, id2 * bs, 0, gg, fb);
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < kBoxes; ++x) {
                        const int col = x * (int)(128 / ELT);
                        tma_load_3d(dst + x * half_bytes, &tmap_k, col, gg, id * bs, fb);
                        tma_load_3d(vdst + x * half_bytes, &tmap_v, col, gg, id * bs, fb);
                        if (second) {
                            tma_load_3d(dst + x * half_bytes + box_bytes, &tmap_k, col, gg,
                                        id2 * bs, fb);
                            tma_load_3d(vdst + x * half_bytes + box_bytes, &tmap_v, col, gg,
                                        id2 * bs, fb);
                        }
                    }
                }
                if constexpr (Pol::kScaleBytes > 0) {
                    // per stage: the unit's K scales [bsu], then its V scales [bsu]
                    const size_t srow = ((size_t)id * H + gg) * bs;
                    const uint32_t sdst = smem_u32(smem + lay.sring) + (uint32_t)(st * 2 * bsu * 4);
                    bulk_load(sdst, p.k_scales + srow, (uint32_t)bs * 4u, fb);
                    bulk_load(sdst + (uint32_t)bsu * 4u, p.v_scales + srow, (uint32_t)bs * 4u, fb);
                    if (second) {
                        const size_t srow2 = ((size_t)id2 * H + gg) * bs;
                        bulk_load(sdst + (uint32_t)bs * 4u, p.k_scales + srow2, (uint32_t)bs * 4u, fb);
                        bulk_load(sdst + (uint32_t)(bsu + bs) * 4u, p.v_scales + srow2,
                                  (uint32_t)bs * 4u, fb);
                    }
                }
            } else {
                valid[st] = 0;
                atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                mbar_arrive(fb);
            }
        }
    };
    for (int i = 0; i < per_warp; ++i) issue_next();

    // stage and pass parity of this warp's next unit
    int cs = w, cpar = 0;
    for (int u = start; u < end;) {
        const int b = find_seq(prefix, B, u, H);
        const int nb = prefix[b + 1] - prefix[b];
        const int r = u - prefix[b] * H;
        const int g = r / nb;
        const int j0 = r - g * nb;
        const int seg_start = prefix[b] * H + g * nb;
        const int piece_end = min(end, seg_start + nb);
        const int Lb = min(max(p.seq_lens[b], 0), cap);
        const int skip = cascade ? skip_s[b] : 0;
        const size_t head0 = (size_t)b * p.num_q_heads + (size_t)g * G;
        // cascade: stage this (b, g)'s prefix state in shared memory while
        // the piece's blocks are attended
        if (skip > 0) {
            pdl_wait();                            // the prefix pass's states are written
            __syncwarp();                          // the last piece's reads are done
            for (int i = lane; i < G * D / 4; i += 32)
                cp_async16(pst_s + 4 * i, p.pst_o + head0 * D + 4 * i);
            if (lane < G) cp_async4(pst_s + G * D + lane, p.pst_lse + head0 + lane);
        }

        pol.begin(qbase + head0 * D, p.qscale, lane);

        for (int uu = u; uu < piece_end; ++uu) {
            const int s = cs;
            cs += NCW;
            const uint32_t par = cpar;
            if (cs >= S) {
                cs -= S;
                cpar ^= 1;
            }
            bool ok = *abort_flag == 0;
            if (ok && !mbar_wait_sleep(smem_u32(&full[s]), par, p.wait_ns)) {
                *abort_flag = 1;
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(FULL, ok);
            if (ok && valid[s]) {
                const int j = skip + j0 + (uu - u);
                const unsigned char* Ks = ring + (size_t)s * lay.stage_bytes;
                const float* sc = Pol::kScaleBytes > 0
                                      ? reinterpret_cast<const float*>(smem + lay.sring) + s * 2 * bsu
                                      : nullptr;
                pol.block(Ks, Ks + bsu * D * ELT, sc, min(bsu, Lb - j * bsu), bsu, p.qscale, lane);
            }
            __syncwarp();                          // every lane is done with stage s
            issue_next();                          // unit k + S into stage s
        }

        // -- the piece's result: out, or a partial for the cross-warp merge ---
        pol.fold(lane);
        {
            const size_t ps = (size_t)worker * 2 + ((u == start) ? 0 : 1);
            PieceOut po;
            po.complete = seg_start >= start && seg_start + nb <= end;
            po.out = obase + head0 * D;
            po.part_o = p.part_o + ps * G * D;
            po.part_lse = p.part_lse + ps * G;
            po.pst_o = skip > 0 ? pst_s : nullptr;
            po.pst_lse = skip > 0 ? pst_s + G * D : nullptr;
            if (skip > 0) {
                cp_async_wait_all();
                __syncwarp();
            }
            pol.merge_store(lane, po);
            if (!po.complete && p.merge_wpp == 0) {
                // Count the finished pieces of (b, g); the warp that finishes
                // the last one merges all their partials into `out`.  (With
                // merge_wpp > 0 the partials wait for paged_decode_merge.)
                __threadfence();
                __syncwarp();
                const int c0 = cut.range_of(seg_start, b * H + g);
                const int c1 = cut.range_of(seg_start + nb - 1, b * H + g);
                int last = 0;
                if (lane == 0)
                    last = count_piece(p.counters + 2 * ((size_t)b * H + g), p.tag, c1 - c0 + 1);
                if (__shfl_sync(FULL, last, 0)) {
                    __threadfence();
                    T* ob = obase + head0 * D;
                    merge_cut<G, D>(p.part_o, p.part_lse, c0, c1,
                                    seg_start == cut.start_unit(c0) ? 0 : 1, po.pst_o, po.pst_lse, lane,
                                    [&](int r, int d0, const float* v, float) {
#pragma unroll
                                        for (int k = 0; k < merge_epl<G, D>(); ++k)
                                            ob[r * D + d0 + k] = Elt<T>::store(v[k]);
                                    });
                }
            }
        }
        u = piece_end;
    }
    if (cascade) pdl_wait();
    // Drain: no copy may still be landing in shared memory at exit (after a
    // timeout the waits above were skipped).  The issues that reached a
    // barrier are the first na; their last per_warp hold distinct stages,
    // each with at most that one phase outstanding (a stage is refilled only
    // after its previous phase was waited on), and a phase already waited on
    // passes at once.  These waits take the full limit whatever the pool's
    // setting, so every copy in flight lands before the CTA exits.
    if (lane == 0)
        for (int i = max(0, na - per_warp); i < na; ++i) {
            if (!mbar_wait_sleep(smem_u32(&full[w + NCW * (i % per_warp)]), (i / per_warp) & 1,
                                 kWaitLimitNs))
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
        }
}

// Shared memory the merge kernel's warps exchange their states through: per
// warp, element pass and lane, the running (M, den) and EPL numerators.
template <int G, int D>
__host__ __device__ constexpr int merge_red_bytes() {
    return NCW * (G * D / (32 * merge_epl<G, D>())) * 32 * (merge_epl<G, D>() + 2) * 4;
}

// One warp's share of a cut segment: the unnormalised log-sum-exp state
// (base M, denominator den, numerators acc) of the partials in slots of
// ranges lo..hi (range c0's piece in slot slot0 of c0, every later range's in
// slot 0) for element pass `pass`, BATCH slots' loads in flight together.
template <int R, int D, int BATCH>
__device__ __forceinline__ void lse_range(const float* part_o, const float* part_lse, int lo,
                                          int hi, int c0, int slot0, int pass, int lane,
                                          float& M, float& den, float* acc) {
    constexpr int EPL = merge_epl<R, D>();
    const int e0 = (pass * 32 + lane) * EPL;
    const int r = e0 / D, d0 = e0 % D;
    M = -CUDART_INF_F;
    den = 0.f;
#pragma unroll
    for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
    for (int c = lo; c <= hi; c += BATCH) {
        float ls[BATCH], ov[BATCH][EPL];
#pragma unroll
        for (int t = 0; t < BATCH; ++t) {
            const int cc = c + t;
            const size_t slot = (size_t)cc * 2 + (cc == c0 ? slot0 : 0);
            ls[t] = -CUDART_INF_F;
            if (cc <= hi) {
                ls[t] = __ldcg(part_lse + slot * R + r);
                load_row<EPL>(ov[t], part_o + (slot * R + r) * D + d0, true);
            }
        }
#pragma unroll
        for (int t = 0; t < BATCH; ++t)
            if (c + t <= hi) lse_add<EPL>(M, den, acc, ls[t], ov[t]);
    }
}

// ------------------------------------------------------------ merge kernel --
// After the split kernel (programmatic dependent launch): the (sequence b,
// KV head g) pairs whose units fall in more than one warp's range were left
// as partials in those warps' slots (the first warp's slot 0 or 1, every later
// warp's slot 0); they are merged by log-sum-exp (with the cascade prefix
// state, if any) into `out`.  merge_wpp = NCW: a CTA takes one pair at a time
// and its warps split the pair's partials, then combine their states through
// shared memory (long contexts: dozens of partials per pair); merge_wpp = 1:
// a warp per pair.  The split kernel's cut is recomputed here from the same
// seq_lens and grid.
template <typename T, int D, int G, int UB>
__global__ void __launch_bounds__(SPLIT_THREADS) paged_decode_merge(const Params p) {
    constexpr int EPL = merge_epl<G, D>();
    constexpr int NP = G * D / (32 * EPL);         // element passes of a warp
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_align_1k(smem_raw);
    const int B = p.batch, H = p.num_kv_heads;
    const int bsu = p.bs * UB;
    const Layout lay(0, B, bsu, G, D, 2, p.num_groups, 0);
    const int* prefix = reinterpret_cast<const int*>(smem + lay.prefix);
    const int* skip_s = reinterpret_cast<const int*>(smem + lay.skip);
    float* red = reinterpret_cast<float*>(smem + lay.pst);   // [NCW][NP][32][EPL + 2]
    const bool cascade = p.num_groups > 0;
    pdl_wait();                                    // the split kernel's partials are visible
    unit_prefix(p, smem, lay, bsu, cascade, false);
    __syncthreads();
    const WorkCut cut(prefix, B, H, p.num_ctas * NCW);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    T* obase = static_cast<T*>(p.out);
    auto store = [&](T* ob, int r, int d0, const float* v) {
#pragma unroll
        for (int k = 0; k < EPL; ++k) ob[r * D + d0 + k] = Elt<T>::store(v[k]);
    };
    if (p.merge_wpp == NCW) {
        for (int pair = blockIdx.x; pair < B * H; pair += gridDim.x) {   // CTA-uniform
            const int b = pair / H, g = pair - b * H;
            const int nb = prefix[b + 1] - prefix[b];
            if (nb == 0) continue;
            const int seg_start = prefix[b] * H + g * nb;
            const int c0 = cut.range_of(seg_start, pair), c1 = cut.range_of(seg_start + nb - 1, pair);
            if (c0 == c1) continue;                // one warp's: written by the split kernel
            const int slot0 = seg_start == cut.start_unit(c0) ? 0 : 1;
            const int per = (c1 - c0 + NCW) / NCW;
            const int lo = c0 + warp * per, hi = min(c1, lo + per - 1);
#pragma unroll
            for (int pass = 0; pass < NP; ++pass) {
                float M, den, acc[EPL];
                lse_range<G, D, 8>(p.part_o, p.part_lse, lo, hi, c0, slot0, pass, lane, M, den, acc);
                float* st = red + ((warp * NP + pass) * 32 + lane) * (EPL + 2);
                st[0] = M;
                st[1] = den;
#pragma unroll
                for (int k = 0; k < EPL; ++k) st[2 + k] = acc[k];
            }
            __syncthreads();
            const size_t head0 = (size_t)b * p.num_q_heads + (size_t)g * G;
            const bool pst = cascade && skip_s[b] > 0;
            for (int pass = warp; pass < NP; pass += NCW) {
                float M = -CUDART_INF_F;
#pragma unroll
                for (int w2 = 0; w2 < NCW; ++w2) M = fmaxf(M, red[((w2 * NP + pass) * 32 + lane) * (EPL + 2)]);
                float den = 0.f, acc[EPL];
#pragma unroll
                for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
                if (M != -CUDART_INF_F) {
#pragma unroll
                    for (int w2 = 0; w2 < NCW; ++w2) {
                        const float* st = red + ((w2 * NP + pass) * 32 + lane) * (EPL + 2);
                        const float c = st[0] == -CUDART_INF_F ? 0.f : fast_exp2(st[0] - M);
                        den += c * st[1];
#pragma unroll
                        for (int k = 0; k < EPL; ++k) acc[k] += c * st[2 + k];
                    }
                }
                const int e0 = (pass * 32 + lane) * EPL;
                const int r = e0 / D, d0 = e0 % D;
                if (pst) {                          // the cascade prefix state, normalised
                    float xv[EPL];
                    load_row<EPL>(xv, p.pst_o + head0 * D + r * D + d0, false);
                    lse_add<EPL>(M, den, acc, p.pst_lse[head0 + r], xv);
                }
                const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
                for (int k = 0; k < EPL; ++k) acc[k] *= inv;
                store(obase + head0 * D, r, d0, acc);
            }
            __syncthreads();                       // red is read before the next pair's writes
        }
        return;
    }
    for (int pair = blockIdx.x * NCW + warp; pair < B * H; pair += gridDim.x * NCW) {
        const int b = pair / H, g = pair - b * H;
        const int nb = prefix[b + 1] - prefix[b];
        if (nb == 0) continue;
        const int seg_start = prefix[b] * H + g * nb;
        const int c0 = cut.range_of(seg_start, pair), c1 = cut.range_of(seg_start + nb - 1, pair);
        if (c0 == c1) continue;                    // one warp's: written by the split kernel
        const size_t head0 = (size_t)b * p.num_q_heads + (size_t)g * G;
        const bool pst = cascade && skip_s[b] > 0;
        T* ob = obase + head0 * D;
        merge_slots<G, D, 4>(p.part_o, p.part_lse, c0, c1, seg_start == cut.start_unit(c0) ? 0 : 1,
                             pst ? p.pst_o + head0 * D : nullptr, pst ? p.pst_lse + head0 : nullptr,
                             lane, 0, 1, [&](int r, int d0, const float* v, float) {
                                 store(ob, r, d0, v);
                             });
    }
}

// ------------------------------------------------------------- host side --
template <typename T, int D, int G, class Pol>
cudaError_t launch_typed(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                         cudaStream_t stream) {
    auto split = paged_decode_split<T, D, G, Pol>;
    cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan.smem_bytes);
    if (e != cudaSuccess) return e;
    Params p;
    p.q = call.q;
    p.out = call.out;
    p.block_tables = call.block_tables;
    p.seq_lens = call.seq_lens;
    p.err = pool.d_err;
    unsigned char* ws = static_cast<unsigned char*>(call.workspace);
    p.counters = reinterpret_cast<unsigned long long*>(ws + plan.ws_counter_off);
    p.tag = call.tag;
    p.part_o = reinterpret_cast<float*>(ws + plan.ws_part_o_off);
    p.part_lse = reinterpret_cast<float*>(ws + plan.ws_part_lse_off);
    p.max_blocks = call.max_blocks;
    p.batch = call.batch;
    p.num_q_heads = call.num_q_heads;
    p.num_kv_heads = pool.num_kv_heads;
    p.num_blocks = pool.num_blocks;
    p.bs = pool.block_size;
    p.stages = plan.stages;
    p.num_ctas = plan.num_ctas;
    p.qscale = call.scale * 1.4426950408889634f;
    p.wait_ns = pool.wait_ns;
    p.g_first = call.g_first;
    p.g_size = call.g_size;
    p.g_blocks = call.g_blocks;
    p.num_groups = call.num_groups;
    p.pst_o = call.pst_o;
    p.pst_lse = call.pst_lse;
    p.k_scales = pool.k_scales;
    p.v_scales = pool.v_scales;
    p.fp8_k_scale = pool.fp8_k_scale;
    p.fp8_v_scale = pool.fp8_v_scale;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.num_ctas);
    cfg.blockDim = dim3(SPLIT_THREADS);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // where the partials of cut (b, g) merge: in this kernel or a second one
    const int pairs = call.batch * pool.num_kv_heads;
    p.merge_wpp = merge_warps_per_pair(plan.num_ctas * NCW, pairs);
    if (Pol::kH2)
        e = cudaLaunchKernelEx(&cfg, split, pool.tmap_k_h2, pool.tmap_v_h2, p);
    else if (Pol::kSwizzled)
        e = cudaLaunchKernelEx(&cfg, split, pool.tmap_k_swz, pool.tmap_v_swz, p);
    else
        e = cudaLaunchKernelEx(&cfg, split, pool.tmap_k, pool.tmap_v, p);
    if (e != cudaSuccess || p.merge_wpp == 0) return e;
    // the partials of (b, g) cut across warps, merged behind the split kernel
    auto merge = paged_decode_merge<T, D, G, Pol::kUnitBlocks>;
    const Layout ml(0, call.batch, pool.block_size * Pol::kUnitBlocks, G, D, 2, call.num_groups, 0);
    const size_t merge_smem = ml.pst + merge_red_bytes<G, D>() + 1024;
    cfg.gridDim = dim3((unsigned)std::max(1, std::min((pairs * p.merge_wpp + NCW - 1) / NCW,
                                                      pool.num_sms * 4)));
    cfg.dynamicSmemBytes = merge_smem;
    if (merge_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)merge_smem);
        if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, merge, p);
}

template <typename T, int D, int G, class Pol>
cudaError_t attrs_typed(size_t smem, int* ctas_per_sm) {
    auto split = paged_decode_split<T, D, G, Pol>;
    cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, split, SPLIT_THREADS, smem);
}

// Which compute policy runs a shape.  Tensor cores: 16-bit pools, head_dim
// 128, groups of 1, 2, 4 or 8 (groups of up to 4 fill the free MMA columns
// with the lo halves of P), block size 8 (two blocks per unit), 16 or 32, a
// pool with one-copy (4-D) tensor maps.  CUDA cores otherwise (fp32 pools,
// head_dim 64, other block sizes), with the token loops unrolled for block
// size 16 (and 8 / 32 on bf16 head_dim 128); other block sizes take the
// generic instance.
template <typename T, int D>
constexpr bool kExtraBlockSizes = std::is_same<T, __nv_bfloat16>::value && D == 128;
template <typename T, int D, int G>
constexpr bool kTensorCores = sizeof(T) == 2 && D == 128 && (G == 1 || G == 2 || G == 4 || G == 8);

inline bool use_tensor_cores(const kv_pool& pool, int G) {
    return pool.elem_bytes == 2 && pool.head_dim == 128 && (G == 1 || G == 2 || G == 4 || G == 8) &&
           (pool.block_size == 8 || pool.block_size == 16 || pool.block_size == 32) &&
           pool.has_h2_maps;
}

template <typename T, int D, int G, template <typename, int, int, class> class Fn, typename... A>
cudaError_t with_policy(int bs, bool tc, A... args) {
    if constexpr (kTensorCores<T, D, G>) {
        if (tc && bs == 8) return Fn<T, D, G, TcPolicy8x2<T, D, G>>::run(args...);
        if (tc && bs == 16) return Fn<T, D, G, TcPolicy<T, D, G, 16>>::run(args...);
        if (tc && bs == 32) return Fn<T, D, G, TcPolicy<T, D, G, 32>>::run(args...);
    }
    if (bs == 16) return Fn<T, D, G, CorePolicy<T, D, G, 16>>::run(args...);
    if constexpr (kExtraBlockSizes<T, D>) {
        if (bs == 8) return Fn<T, D, G, CorePolicy<T, D, G, 8>>::run(args...);
        if (bs == 32) return Fn<T, D, G, CorePolicy<T, D, G, 32>>::run(args...);
    }
    return Fn<T, D, G, CorePolicy<T, D, G, 0>>::run(args...);
}

template <typename T, int D, int G, class Pol> struct LaunchFn {
    static cudaError_t run(const kv_pool* pool, const DecodeCall* call, const DecodePlan* plan,
                           cudaStream_t stream) {
        return launch_typed<T, D, G, Pol>(*pool, *call, *plan, stream);
    }
};
template <typename T, int D, int G, class Pol> struct AttrsFn {
    static cudaError_t run(size_t smem, int* ctas_per_sm) {
        return attrs_typed<T, D, G, Pol>(smem, ctas_per_sm);
    }
};

template <typename T>
cudaError_t dispatch(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                     cudaStream_t stream) {
    const bool tc = use_tensor_cores(pool, plan.group);
#define PKV_CASE(DD, GG)                                                                 \
    if (pool.head_dim == DD && plan.group == GG)                                         \
        return with_policy<T, DD, GG, LaunchFn>(pool.block_size, tc, &pool, &call, &plan, \
                                                stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t attrs(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm) {
    const bool tc = use_tensor_cores(pool, group);
#define PKV_CASE(DD, GG)                                                                        \
    if (pool.head_dim == DD && group == GG)                                                     \
        return with_policy<T, DD, GG, AttrsFn>(pool.block_size, tc, smem, ctas_per_sm);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
    return cudaErrorNotSupported;
}

// 8-bit pools: Tc8Policy for head_dim 128, block sizes that are multiples of
// 16, groups of 1, 2, 4 or 8 (T = the query / output type).
inline bool q8_shape_ok(const kv_pool& pool) {
    return pool.head_dim == 128 && pool.block_size % 16 == 0 && pool.block_size <= 256;
}

// Block size 16: a work unit is two consecutive blocks (a 32-row tile, the
// second block's rows after the first's), which halves the per-unit costs
// (loads issued, barrier waits) per token.
inline bool q8_pairs_blocks(const kv_pool& pool, int G) {
    return pool.block_size == 16 && (G == 1 || G == 2 || G == 4 || G == 8);
}

template <typename T, int FMT, template <typename, int, int, class> class Fn, typename... A>
cudaError_t with_q8_policy(int G, bool pairs, A... args) {
    if (pairs && G == 1) return Fn<T, 128, 1, Tc8Policy2<T, 128, 1, FMT>>::run(args...);
    if (pairs && G == 2) return Fn<T, 128, 2, Tc8Policy2<T, 128, 2, FMT>>::run(args...);
    if (pairs && G == 4) return Fn<T, 128, 4, Tc8Policy2<T, 128, 4, FMT>>::run(args...);
    if (pairs && G == 8) return Fn<T, 128, 8, Tc8Policy2<T, 128, 8, FMT>>::run(args...);
    if (G == 1) return Fn<T, 128, 1, Tc8Policy<T, 128, 1, FMT>>::run(args...);
    if (G == 2) return Fn<T, 128, 2, Tc8Policy<T, 128, 2, FMT>>::run(args...);
    if (G == 4) return Fn<T, 128, 4, Tc8Policy<T, 128, 4, FMT>>::run(args...);
    if (G == 8) return Fn<T, 128, 8, Tc8Policy<T, 128, 8, FMT>>::run(args...);
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t dispatch_q8(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                        cudaStream_t stream) {
    if (!q8_shape_ok(pool)) return cudaErrorNotSupported;
    const bool pairs = q8_pairs_blocks(pool, plan.group);
    if (pool.cache_dtype == KV_FP8_E4M3)
        return with_q8_policy<T, kFmtE4M3, LaunchFn>(plan.group, pairs, &pool, &call, &plan, stream);
    if (pool.cache_dtype == KV_INT8)
        return with_q8_policy<T, kFmtInt8, LaunchFn>(plan.group, pairs, &pool, &call, &plan, stream);
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t attrs_q8(const kv_pool& pool, int group, size_t smem, int* ctas_per_sm) {
    if (!q8_shape_ok(pool)) return cudaErrorNotSupported;
    const bool pairs = q8_pairs_blocks(pool, group);
    if (pool.cache_dtype == KV_FP8_E4M3)
        return with_q8_policy<T, kFmtE4M3, AttrsFn>(group, pairs, smem, ctas_per_sm);
    if (pool.cache_dtype == KV_INT8)
        return with_q8_policy<T, kFmtInt8, AttrsFn>(group, pairs, smem, ctas_per_sm);
    return cudaErrorNotSupported;
}

}  // namespace dec
}  // namespace pagedkv
