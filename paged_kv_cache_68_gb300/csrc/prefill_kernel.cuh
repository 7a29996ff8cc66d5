// Paged (chunked) prefill attention for sm_103a on the 5th-generation tensor
// cores: tcgen05.mma with operands staged by TMA in shared memory and the
// score / output accumulators in tensor memory (TMEM).
//
// What is computed ("Part 3: single node", random-liu.github.io, ch. 13
// sec. 1-2: the new tokens of a batch are flattened into one stream with
// request boundaries cu_seqlens; a long prompt is processed one chunk per
// iteration, and a chunk's attention reads the cached earlier part of the
// prompt through the block table, like decode).  Request b has
// C_b = cu_seqlens[b+1] - cu_seqlens[b] queries, its last C_b positions
// L_b - C_b .. L_b - 1 (L_b = seq_lens[b], counted after the chunk's own K/V
// were appended); query i attends causally to positions 0 .. L_b - C_b + i.
// C_b = 1 is a decode request.  Softmax is computed block-wise with a running
// maximum and sum ("Lecture 24", semidirectx.com CMU 11-868 notes, sec. 3.2).
//
// Tiling.  One CTA computes one tile of BM = 128 rows: QT = 128 / G
// consecutive queries of one request times the G query heads that share one
// KV head (row = query * G + head), so each K/V tile is read once for the
// whole GQA group.  The CTA walks the request's tokens in KV tiles of BN = 128
// (BN / bs pool blocks, each fetched by TMA through the block table), up to
// the last position its queries can see.
//   S  = Q K^T      tcgen05.mma, A = Q (smem), B = K tile (smem), D = TMEM
//   P  = exp2(S * scale * log2 e - m)            (softmax warps, fp32)
//   O += P V        tcgen05.mma, A = P (TMEM), B = V tile (smem), D = TMEM
// P overwrites S in TMEM as 16-bit hi + lo halves (P = hi + lo to 2^-16
// relative) and is multiplied twice, so the result keeps fp32-level accuracy.
// The running maximum is updated lazily: O and the sum are rescaled only when
// a row's maximum grows by more than 2^8, so P stays below 256.
//
// Two CTAs share an SM (96 KB of shared memory and 256 TMEM columns each):
// one CTA's softmax runs while the other's products occupy the tensor pipe,
// which hides the serial S -> softmax -> PV chain of each tile.
//
// Warp roles (192 threads):
//   warps 0-3  softmax and epilogue; thread r owns row r (TMEM lane r);
//   warp 4     TMA producer: Q once, then the K and V tiles (one buffer each:
//              K_{j+1} lands while tile j's softmax and PV run, V_{j+1} while
//              S_{j+1} and its softmax run);
//   warp 5     TMEM allocation and the single MMA-issuing thread.
// Every mbarrier wait is bounded; a wait that gives up sets KV_DEVERR_TIMEOUT,
// raises the CTA's abort flag, and the CTA drains its copies and MMAs, frees
// TMEM and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_kernel.cuh"
#include "pagedkv_internal.cuh"

namespace pagedkv {
namespace pf {

using dec::FULL;

constexpr int D = 128;            // head_dim
constexpr int BM = 128;           // rows of a tile
constexpr int BN = 128;           // tokens of a KV tile
constexpr int NSOFT = 4;          // softmax warps = TMEM lane quadrants
constexpr int WARP_TMA = 4, WARP_MMA = 5;
constexpr int NTHREADS = 6 * 32;
constexpr int CTAS_PER_SM = 2;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t COL_S = 0, COL_O = 128;    // P (hi, then lo) overwrites S
constexpr uint32_t COL_PH = COL_S, COL_PL = COL_S + 64;
constexpr float kRescaleLog2 = 8.f;   // lazy rescale threshold (log2 units)

constexpr uint32_t HALF_BYTES = 128u * 128u;    // 128 rows x 128 B (64 dims)
constexpr uint32_t TILE_BYTES = 2u * HALF_BYTES;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = TILE_BYTES;
constexpr uint32_t OFF_V = 2u * TILE_BYTES;
constexpr uint32_t OFF_BAR = 3u * TILE_BYTES;
// barriers (8 B each), then the TMEM address and the abort flag
constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = 2, BAR_VF = 3, BAR_VE = 4, BAR_SF = 5,
              BAR_PF = 6, BAR_OF = 7, BAR_DR = 8, NBARS = 9;
constexpr uint32_t OFF_TMEM = OFF_BAR + 8u * NBARS;
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4u;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4u + 1024u;   // + slack to align the base to 1 KB

struct Params {
    const void* q;                // [T, Hq, D]
    void* out;                    // [T, Hq, D]
    const int32_t* cu_seqlens;    // [batch + 1]
    const int32_t* block_tables;  // [batch, max_blocks]
    const int32_t* seq_lens;      // [batch]
    int* err;
    int num_tokens;
    int max_blocks;
    int batch;
    int num_q_heads;
    int num_blocks;
    int bs;
    int max_q;                    // the largest C_b the grid covers
    float qscale;                 // scale * log2(e), > 0
};

// ------------------------------------------------------------ tcgen05 PTX --
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family format:
// start >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride byte
// offset >> 4 in 32-45, version 1 in bits 46-47, layout 2 = SWIZZLE_128B in
// bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (fmt 0 = f16, 1 = bf16), A K-major, B K- or MN-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t fmt, uint32_t b_mn_major, uint32_t M,
                                                 uint32_t N) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn_major << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                       uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

#define PKV_R8(i) "=r"(v[i]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), \
                  "=r"(v[i + 4]), "=r"(v[i + 5]), "=r"(v[i + 6]), "=r"(v[i + 7])
#define PKV_W8(i) "r"(v[i]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), \
                  "r"(v[i + 4]), "r"(v[i + 5]), "r"(v[i + 6]), "r"(v[i + 7])

// 32 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 PKV_W8(0)
                 : "memory");
}
#undef PKV_R8
#undef PKV_W8
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16-bit element helpers: round a pair to the type (element `lo` in the low
// half) and widen the low / high half back to fp32.
template <typename T> struct H16;
template <> struct H16<__nv_bfloat16> {
    static constexpr uint32_t kFmt = 1;
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    __device__ static __forceinline__ float low(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ static __forceinline__ float high(uint32_t w) {
        return __uint_as_float(w & 0xffff0000u);
    }
    // p = hi + lo: hi keeps the top 16 bits of each fp32 (truncation, exact
    // remainder), lo is the remainder rounded to bf16 (|error| <= 2^-16 p)
    __device__ static __forceinline__ void split(float p0, float p1, uint32_t& hi, uint32_t& lo) {
        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
        hi = __byte_perm(b0, b1, 0x7632);
        const float2 r = __ffma2_rn(make_float2(__uint_as_float(b0 & 0xffff0000u),
                                                __uint_as_float(b1 & 0xffff0000u)),
                                    make_float2(-1.f, -1.f), make_float2(p0, p1));
        lo = pack(r.x, r.y);
    }
};
template <> struct H16<__half> {
    static constexpr uint32_t kFmt = 0;
    __device__ static __forceinline__ uint32_t pack(float lo, float hi) {
        uint32_t r;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
        return r;
    }
    __device__ static __forceinline__ float low(uint32_t w) {
        return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
    }
    __device__ static __forceinline__ float high(uint32_t w) {
        return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    }
    // p = hi + lo: hi rounded to f16, lo the remainder rounded to f16
    __device__ static __forceinline__ void split(float p0, float p1, uint32_t& hi, uint32_t& lo) {
        hi = pack(p0, p1);
        lo = pack(p0 - low(hi), p1 - high(hi));
    }
};

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Bounded wait; on expiry (or when another role already gave up) raise the
// abort flag and return false.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int* err) {
    if (dec::mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (dec::mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    atomicOr(err, KV_DEVERR_TIMEOUT);
    return false;
}

template <typename T, int G>
__global__ void __launch_bounds__(NTHREADS, CTAS_PER_SM)
    paged_prefill(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const Params p) {
    constexpr int QT = BM / G;                    // queries per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = dec::smem_u32(smem);
    auto bar = [&](int i) { return sbase + OFF_BAR + 8u * (uint32_t)i; };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, g = blockIdx.y;
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;   // later query tiles (more work) first
    const int bs = p.bs;

    dec::pdl_launch_dependents();
    dec::pdl_wait();                              // inputs of earlier kernels are visible

    // -- the tile's queries and the tokens they see --------------------------
    int cu0 = p.cu_seqlens[b], cu1 = p.cu_seqlens[b + 1];
    int L = p.seq_lens[b];
    int C = cu1 - cu0;
    const bool bad_q = cu0 < 0 || cu1 < cu0 || cu1 > p.num_tokens;
    if (bad_q) C = 0;
    const int cap = p.max_blocks * bs;
    const bool bad_len = L > cap;
    L = max(0, min(L, cap));
    if (tid == 0 && qt == 0 && (bad_q || C > p.max_q)) atomicOr(p.err, KV_DEVERR_QUERY_RANGE);
    if (tid == 0 && qt == 0 && g == 0 && bad_len) atomicOr(p.err, KV_DEVERR_SEQ_RANGE);
    const int q0 = qt * QT;
    const int nq = min(QT, min(C, p.max_q) - q0);  // valid queries of this tile
    if (nq <= 0) return;                           // whole CTA, before any barrier
    const int P0 = L - C + q0;                     // position of the tile's first query
    const int Pmax = P0 + nq - 1;                  // and of its last (<= L - 1)
    const int ntiles = Pmax >= 0 ? Pmax / BN + 1 : 0;

    // -- set-up: barriers, TMEM ----------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < NBARS; ++i) dec::mbar_init(bar(i), i == BAR_PF ? NSOFT : 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == WARP_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + OFF_TMEM),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_TMA) {
        // ------------------------------------------------------ producer ----
        const int nb_tile = BN / bs;               // pool blocks per KV tile (<= 16)
        const uint32_t blk_bytes = (uint32_t)bs * 128u;   // one block, one 64-dim half
        int issued_k = 0, issued_v = 0;
        if (ntiles > 0) {
            if (lane == 0) {
                dec::mbar_arrive_tx(bar(BAR_Q), TILE_BYTES);
                dec::tma_load_3d(sbase + OFF_Q, &tmap_q, 0, g * G, cu0 + q0, bar(BAR_Q));
                dec::tma_load_3d(sbase + OFF_Q + HALF_BYTES, &tmap_q, 64, g * G, cu0 + q0,
                                 bar(BAR_Q));
            }
            const int32_t* table = p.block_tables + (size_t)b * p.max_blocks;
            // one KV tile into one buffer: the lanes' blocks, bytes counted first
            auto load_tile = [&](int j, int full, uint32_t dst, const CUtensorMap* map) {
                const int lb = j * nb_tile + lane;  // logical block of this lane
                int id = -1;
                bool load = false;
                if (lane < nb_tile && lb * bs < L) {
                    id = table[lb];
                    load = id >= 0 && id < p.num_blocks;
                    if (!load && map == &tmap_k) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                }
                const unsigned mask = __ballot_sync(FULL, load);
                if (lane == 0) dec::mbar_arrive_tx(bar(full), (uint32_t)__popc(mask) * 2u * blk_bytes);
                __syncwarp();
                if (load) {
                    const uint32_t d = dst + (uint32_t)lane * blk_bytes;
                    dec::tma_load_3d(d, map, 0, g, id * bs, bar(full));
                    dec::tma_load_3d(d + HALF_BYTES, map, 64, g, id * bs, bar(full));
                }
            };
            // K_j needs S_{j-1} done (k_empty), V_j needs PV_{j-1} done (v_empty);
            // K runs one tile ahead of V
            for (int j = 0; j < ntiles; ++j) {
                bool ok = true;
                if (lane == 0 && j > 0)
                    ok = wait_or_abort(bar(BAR_KE), (j - 1) & 1, abort_flag, p.err);
                if (!__shfl_sync(FULL, ok ? 1 : 0, 0)) break;
                load_tile(j, BAR_KF, sbase + OFF_K, &tmap_k);
                issued_k = j + 1;
                if (lane == 0 && j > 0)
                    ok = wait_or_abort(bar(BAR_VE), (j - 1) & 1, abort_flag, p.err);
                if (!__shfl_sync(FULL, ok ? 1 : 0, 0)) break;
                load_tile(j, BAR_VF, sbase + OFF_V, &tmap_v);
                issued_v = j + 1;
            }
            // Drain: no copy may still be landing in shared memory at exit.
            if (lane == 0) {
                bool ok = dec::mbar_wait(bar(BAR_Q), 0);
                if (issued_k > 0) ok &= dec::mbar_wait(bar(BAR_KF), (issued_k - 1) & 1);
                if (issued_v > 0) ok &= dec::mbar_wait(bar(BAR_VF), (issued_v - 1) & 1);
                if (!ok) atomicOr(p.err, KV_DEVERR_TIMEOUT);
            }
        }
    } else if (warp == WARP_MMA) {
        // ----------------------------------------------------------- MMA ----
        if (ntiles > 0 && lane == 0) {
            constexpr uint32_t fmt = H16<T>::kFmt;
            constexpr uint32_t id_s = idesc_f16(fmt, 0, BM, BN);   // S = Q K^T
            constexpr uint32_t id_pv = idesc_f16(fmt, 1, BM, D);   // O += P V (V MN-major)
            const uint32_t q_addr = sbase + OFF_Q, k_addr = sbase + OFF_K, v_addr = sbase + OFF_V;
            bool ok = wait_or_abort(bar(BAR_Q), 0, abort_flag, p.err);
            for (int j = 0; ok && j < ntiles; ++j) {
                const uint32_t par = j & 1;
                // S_j overwrites P_{j-1}: PV_{j-1} must have finished reading it
                if (j > 0 && !wait_or_abort(bar(BAR_OF), par ^ 1u, abort_flag, p.err)) break;
                if (!wait_or_abort(bar(BAR_KF), par, abort_flag, p.err)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // 16 dims = 32 bytes inside a 128-byte swizzled row
                    const uint32_t off = (uint32_t)(kk >> 2) * HALF_BYTES + (uint32_t)(kk & 3) * 32u;
                    mma_ss(tmem + COL_S, sdesc_sw128(q_addr + off, 16u, 1024u),
                           sdesc_sw128(k_addr + off, 16u, 1024u), id_s, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(BAR_KE));
                mma_commit(bar(BAR_SF));
                if (!wait_or_abort(bar(BAR_PF), par, abort_flag, p.err)) break;
                if (!wait_or_abort(bar(BAR_VF), par, abort_flag, p.err)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    // 16 tokens = two 8-row swizzle atoms; the two 64-dim halves
                    // are HALF_BYTES apart (leading byte offset)
                    const uint64_t vdesc = sdesc_sw128(v_addr + (uint32_t)kk * 2048u, HALF_BYTES, 1024u);
                    mma_ts(tmem + COL_O, tmem + COL_PH + (uint32_t)kk * 8u, vdesc, id_pv,
                           (j > 0 || kk > 0) ? 1u : 0u);
                    mma_ts(tmem + COL_O, tmem + COL_PL + (uint32_t)kk * 8u, vdesc, id_pv, 1u);
                }
                mma_commit(bar(BAR_VE));
                mma_commit(bar(BAR_OF));
            }
            // Drain: every MMA issued has completed before TMEM is freed.
            mma_commit(bar(BAR_DR));
            if (!dec::mbar_wait(bar(BAR_DR), 0)) atomicOr(p.err, KV_DEVERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- softmax, epilogue ----
        const int r = tid;                         // row = TMEM lane
        const int qi = r / G, hh = r % G;
        const bool valid = qi < nq;
        const int lim = valid ? P0 + qi : -1;      // last visible position
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float qs = p.qscale;
        float m = -CUDART_INF_F;
        float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // partial row sums
        bool ok = true;
        // tcgen05.ld / st are warp-collective: every wait's outcome is made
        // uniform across the warp
        auto wait_warp = [&](uint32_t bb, uint32_t parity) {
            return __all_sync(FULL, wait_or_abort(bb, parity, abort_flag, p.err));
        };
        for (int j = 0; j < ntiles; ++j) {
            const int t0 = j * BN;
            // S_j complete (and with it PV_{j-1}: the commit covers every
            // earlier product)
            if (!wait_warp(bar(BAR_SF), j & 1)) { ok = false; break; }
            tc_fence_after();
            uint32_t sv[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(trow + COL_S + 32u * c, sv[c]);
            tmem_wait_ld();
            // causal / length mask: tokens past `lim` do not exist for this row
            if (t0 + BN - 1 > lim) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (t0 + 32 * c + e > lim) sv[c][e] = __float_as_uint(-CUDART_INF_F);
            }
            // row maximum: four independent chains of three-input maxima
            float mx4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                mx4[i] = fmaxf(__uint_as_float(sv[i][0]), __uint_as_float(sv[i][1]));
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 2; e < 32; e += 2)
                    mx4[i] = max3(mx4[i], __uint_as_float(sv[i][e]), __uint_as_float(sv[i][e + 1]));
            const float mx = max3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
            const float m_new = fmaxf(m, mx * qs);
            float alpha = 1.f;
            const bool grow = m_new > m + kRescaleLog2;   // false while both are -inf
            if (grow) {
                alpha = dec::fast_exp2(m - m_new);       // 0 when m was -inf
                m = m_new;
            }
            const float mu = m == -CUDART_INF_F ? 0.f : m;
            l2[0] = __fmul2_rn(l2[0], make_float2(alpha, alpha));
            l2[1] = __fmul2_rn(l2[1], make_float2(alpha, alpha));
            // P = hi + lo over S's columns (S was read in full above), 16
            // tokens at a time
            const float2 qs2 = make_float2(qs, qs), nmu2 = make_float2(-mu, -mu);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t ph[8], pl[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const uint32_t* sc = sv[c >> 1] + 16 * (c & 1);
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(sc[e]), __uint_as_float(sc[e + 1])), qs2, nmu2);
                    const float2 pp = make_float2(dec::fast_exp2(x.x), dec::fast_exp2(x.y));
                    l2[(e >> 1) & 1] = __fadd2_rn(l2[(e >> 1) & 1], pp);
                    H16<T>::split(pp.x, pp.y, ph[e / 2], pl[e / 2]);
                }
                tmem_st8(trow + COL_PH + 8u * c, ph);
                tmem_st8(trow + COL_PL + 8u * c, pl);
            }
            // O was last written by PV_{j-1}; rescale it when any row's maximum grew
            // (after P, so S's registers are free)
            if (j > 0 && __any_sync(FULL, grow)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(trow + COL_O + 32u * c, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                    tmem_st32(trow + COL_O + 32u * c, ov);
                }
            }
            // the last tile: zero V rows past the sequence end (P is 0 there,
            // but 0 x NaN from an unwritten row would poison the product)
            if (t0 + BN > L) {
                if (!wait_warp(bar(BAR_VF), j & 1)) { ok = false; break; }
                const int r0 = max(L - t0, 0);
                unsigned char* vt = smem + OFF_V;
                const int nchunks = (BN - r0) * 16;     // 16-byte chunks in both halves
                for (int i = tid; i < nchunks; i += NSOFT * 32) {
                    const int row = r0 + (i >> 4), ch = i & 15;
                    *reinterpret_cast<uint4*>(vt + (ch >> 3) * HALF_BYTES + row * 128 + (ch & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                dec::fence_proxy_async();
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) dec::mbar_arrive(bar(BAR_PF));
        }
        // -- epilogue: out = O / l, rounded once to the output type ----------
        ok = __all_sync(FULL, ok);
        const bool have_o = ok && ntiles > 0 && wait_warp(bar(BAR_OF), (ntiles - 1) & 1);
        if (ntiles > 0) tc_fence_after();
        const float l = (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* orow = static_cast<T*>(p.out) +
                  ((size_t)(cu0 + q0 + qi) * p.num_q_heads + (size_t)g * G + hh) * D;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            if (have_o) {
                tmem_ld32(trow + COL_O + 32u * c, ov);
                tmem_wait_ld();
            }
            if (valid && (have_o || (ok && ntiles == 0))) {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = have_o ? H16<T>::pack(__uint_as_float(ov[2 * e]) * inv,
                                                 __uint_as_float(ov[2 * e + 1]) * inv)
                                  : 0u;
                uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
            }
        }
    }

    // -- teardown: free TMEM once every role is done with it ------------------
    tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace pf
}  // namespace pagedkv
