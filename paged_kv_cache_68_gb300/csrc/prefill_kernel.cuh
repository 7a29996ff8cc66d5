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
// Tiling.  A query tile is BM = 128 rows: QT = 128 / G consecutive queries
// of one request times the G query heads that share one KV head (row =
// query * G + head), so each K/V tile is read once for the whole GQA group.
// One CTA runs two query tiles of the same request and KV head ("streams" A
// and B: query tiles 2t and 2t+1) over shared K/V tiles of BN = 64 tokens
// (BN / bs pool blocks, or half a block for bs = 128, fetched by TMA through
// the block table), up to the last position the later tile can see.  Per
// stream and KV tile:
//   S  = Q K^T      tcgen05.mma, A = Q (smem), B = K tile (smem), D = TMEM
//   P  = exp2(S * scale * log2 e - m)            (softmax warps, fp32)
//   O += P V        tcgen05.mma, A = P (TMEM), B = V tile (smem), D = TMEM
// P is stored in TMEM as 16-bit hi + lo halves (P = hi + lo to 2^-16
// relative) and multiplied twice, so the result keeps fp32-level accuracy.
// The running maximum is updated lazily: O and the sum are rescaled only when
// a row's maximum grows by more than 2^8, so P stays below 256.
//
// Overlap.  Each stream has its own S (64 TMEM columns), P (64) and O (128):
// S_{j+1} is computed while tile j's softmax runs, and tile j+1's softmax
// while PV_j runs.  The two streams' softmax warps share every SM
// sub-partition (a warp may only read the TMEM lanes of its own
// sub-partition, so all warps there work on the same 32 rows of a tile); with
// two streams, one stream's exponentials (the ex2 unit is the softmax's
// floor) overlap the other's loads, reductions and stores.
//
// Warp roles (384 threads, one CTA per SM):
//   warps 0-7  softmax and epilogue, warps 4X..4X+3 for stream X: thread
//              (w, lane) owns row 32 (w % 4) + lane of its stream's tile (its
//              TMEM lane), all 64 columns of each KV tile;
//   warp 8     TMA producer of the two Q tiles (once) and the K tiles
//              (4-stage ring, released when both streams' S are done);
//   warp 9     TMA producer of the V tiles (3-stage ring, released when both
//              streams' PV are done);
//   warps 10, 11 the MMA issue of stream A and of stream B (one elected
//              lane each; warp 10 also allocates and frees TMEM).
// Every mbarrier wait is bounded; a wait that gives up sets KV_DEVERR_TIMEOUT,
// raises the CTA's abort flag, and the CTA drains its copies and MMAs, frees
// TMEM and exits.
//
// 8-bit pools (FMT >= 0: FP8 E4M3 with one K and one V scale per pool, INT8
// with a scale per token and head).  The producers land a tile's code rows
// (128 bytes each) in a ring of their own and turn them into the query type
// in the K / V ring as f16 (E4M3 and INT8 codes convert to f16 exactly), and
// the MMAs run on f16.  bf16 query tiles are turned into f16 in place, each
// row times a power of two 2^e of its own (its largest |q| in [2^14, 2^15):
// the conversion is exact), and the row's scores are multiplied by 2^-e.
// FP8: the K scale multiplies the scores (with the softmax scale), the V
// scale the output.  INT8: the producers also copy the tile's
// token scales to a ring the softmax reads: K scales multiply the scores'
// columns, V scales P's columns before the hi / lo split.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_kernel.cuh"
#include "pagedkv_internal.cuh"

namespace pagedkv {
namespace pf {

using dec::FULL;

constexpr int D = 128;            // head_dim
constexpr int BM = 128;           // rows of a query tile
constexpr int BN = 64;            // tokens of a KV tile
constexpr int KST = 4, VST = 3;   // K and V ring depths
constexpr int NSOFT = 4;          // softmax warps per stream: one per TMEM lane quadrant
constexpr int WARP_TMAK = 2 * NSOFT, WARP_TMAV = WARP_TMAK + 1, WARP_MMA = WARP_TMAK + 2;
constexpr int NTHREADS = (2 * NSOFT + 4) * 32;
// 8-bit pools: a second converter warp per side turns half of each tile's
// code rows into 16-bit values beside the producer.  The helpers take warps
// 10 and 11 (SM sub-partitions 2 and 3, the ones no producer issues from)
// and the MMA warps move to 12 and 13.
constexpr int WARP_CVK = WARP_TMAK + 2, WARP_CVV = WARP_CVK + 1, WARP_MMA_Q8 = WARP_TMAK + 4;
constexpr int NTHREADS_Q8 = NTHREADS + 2 * 32;
constexpr uint32_t TMEM_COLS = 512;
// per stream X: base 256 X; S, then P hi, P lo, then O
constexpr uint32_t COL_S = 0, COL_PH = 64, COL_PL = 96, COL_O = 128, COL_STREAM = 256;
constexpr float kRescaleLog2 = 8.f;   // lazy rescale threshold (log2 units)

constexpr uint32_t QHALF = 128u * 128u;          // Q: 128 rows x 128 B (64 dims)
constexpr uint32_t QTILE = 2u * QHALF;
constexpr uint32_t KVHALF = (uint32_t)BN * 128u; // K/V: 64 rows x 128 B
constexpr uint32_t KVTILE = 2u * KVHALF;
constexpr uint32_t OFF_Q = 0;                    // two query tiles
constexpr uint32_t OFF_K = 2u * QTILE;
constexpr uint32_t OFF_V = OFF_K + KST * KVTILE;
constexpr uint32_t OFF_BAR = OFF_V + VST * KVTILE;
// barriers (8 B each): q_full, k_full[KST], k_empty[KST], v_full[VST],
// v_empty[VST], then per stream: s_full, s_free, p_full, o_full, drain
constexpr int BAR_Q = 0, BAR_KF = 1, BAR_KE = BAR_KF + KST, BAR_VF = BAR_KE + KST,
              BAR_VE = BAR_VF + VST, BAR_STREAM = BAR_VE + VST;
constexpr int SB_SF = 0, SB_SR = 1, SB_PF = 2, SB_OF = 3, SB_DR = 4, SB_N = 5;
constexpr int NBARS = BAR_STREAM + 2 * SB_N;
// 8-bit pools: then the K and V code rings' full barriers, the INT8 scale
// ring's full / empty barriers, the converted-query barrier and, per side and
// code stage, the helper converter's done-reading barrier
constexpr int CST = 2;                            // code tiles per ring
constexpr uint32_t CTILE = (uint32_t)BN * 128u;   // a tile's code rows: 64 x 128 B
constexpr int SCS = 4;                            // INT8 scale ring depth
constexpr int BAR_CK = NBARS, BAR_CV = BAR_CK + CST, BAR_SCF = BAR_CV + CST,
              BAR_SCE = BAR_SCF + SCS, BAR_QC = BAR_SCE + SCS, BAR_HK = BAR_QC + 1,
              BAR_HV = BAR_HK + CST, NBARS_Q8 = BAR_HV + CST;
// launch order: the requests' costs (up to kMaxRanked of them) and the
// request this CTA takes
constexpr int kMaxRanked = 256;
constexpr uint32_t OFF_ORDER = OFF_BAR + 8u * NBARS;
constexpr uint32_t OFF_TMEM = OFF_ORDER + 4u * (kMaxRanked + 4);
constexpr uint32_t OFF_ABORT = OFF_TMEM + 4u;
constexpr uint32_t SMEM_BYTES = OFF_ABORT + 4u + 1024u;   // + slack to align the base to 1 KB

// The layout of one CTA's shared memory: as above for 16-bit pools; 8-bit
// pools add the code rings (and the INT8 scale ring: K then V scales of a
// tile, 64 each) after the V ring.
template <bool Q8>
struct Lay {
    static constexpr uint32_t ck = OFF_V + VST * KVTILE;
    static constexpr uint32_t cv = ck + (Q8 ? CST * CTILE : 0u);
    static constexpr uint32_t sc = cv + (Q8 ? CST * CTILE : 0u);       // [SCS][K, V][BN]
    static constexpr uint32_t csc = sc + (Q8 ? SCS * 2u * BN * 4u : 0u); // [K, V][CST][BN]
    static constexpr uint32_t qinv = csc + (Q8 ? 2u * CST * BN * 4u : 0u); // [stream][BM] 2^-e
    static constexpr uint32_t bar = qinv + (Q8 ? 2u * BM * 4u : 0u);
    static constexpr int nbars = Q8 ? NBARS_Q8 : NBARS;
    static constexpr uint32_t order = bar + 8u * nbars;
    static constexpr uint32_t tmem = order + 4u * (kMaxRanked + 4);
    static constexpr uint32_t abort_flag = tmem + 4u;
    static constexpr uint32_t bytes = abort_flag + 4u + 1024u;
};
static_assert(Lay<false>::bytes == SMEM_BYTES, "16-bit layout");
static_assert(Lay<true>::bytes <= 227u * 1024u, "8-bit layout fits");

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
    int box_rows;                 // rows of one K/V box: min(bs, BN)
    float qscale;                 // scale * log2(e) (* the FP8 K scale), > 0
    float vscale;                 // FP8: the pool's V scale; 1 otherwise
    const float* k_scales;        // INT8: [num_blocks][num_kv_heads][bs]
    const float* v_scales;
    int num_kv_heads;
    unsigned long long wait_ns;   // limit of one pipeline wait (the pool's setting)
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
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        PKV_W8(0), PKV_W8(8)
        : "memory");
}
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

// One lane of the (fully active) warp is elected.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile("{ .reg .pred p; elect.sync _|p, 0xffffffff; selp.u32 %0, 1, 0, p; }" : "=r"(pred));
    return pred != 0;
}


// 16 codes (one 16-byte chunk, FMT a dec:: code format) -> 16 values of T
// (two 16-byte chunks): E4M3 and INT8 codes convert to f16 exactly, and an
// f16 of at most 8 significant bits converts to bf16 exactly.
template <typename T, int FMT>
__device__ __forceinline__ void codes_to(uint4 c, uint4& lo, uint4& hi) {
    uint32_t o[8];
    dec::cvt4<FMT>(c.x, o[0], o[1]);
    dec::cvt4<FMT>(c.y, o[2], o[3]);
    dec::cvt4<FMT>(c.z, o[4], o[5]);
    dec::cvt4<FMT>(c.w, o[6], o[7]);
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&o[i]));
            o[i] = H16<__nv_bfloat16>::pack(f.x, f.y);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Code row r of a tile (a code stage: 64 rows x 128 B, 128-byte swizzled) ->
// row r of a 16-bit ring slot (two 64-dim halves of 64 rows x 128 B, each
// 128-byte swizzled): code chunk c (dims 16 c ..) becomes 16-byte chunks
// 2 (c % 4) and 2 (c % 4) + 1 of half c / 4.
template <typename MT, int FMT>
__device__ __forceinline__ void convert_row(const unsigned char* crows, unsigned char* orows, int r) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(crows + r * 128 + ((c ^ (r & 7)) << 4));
        uint4 lo, hi;
        codes_to<MT, FMT>(w, lo, hi);
        unsigned char* h = orows + (c >> 2) * KVHALF + r * 128;
        const int c0 = 2 * (c & 3);
        *reinterpret_cast<uint4*>(h + ((c0 ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(h + (((c0 + 1) ^ (r & 7)) << 4)) = hi;
    }
}

// Bounded wait (limit_ns); on expiry (or when another role already gave up)
// raise the abort flag and return false.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int* err,
                                              unsigned long long limit_ns) {
    if (limit_ns == 0 ? dec::mbar_test(bar, parity) : dec::mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (limit_ns > 0 && dec::mbar_wait(bar, parity, limit_ns)) return true;
    *abort_flag = 1;
    atomicOr(err, KV_DEVERR_TIMEOUT);
    return false;
}

// FMT: -1 for 16-bit pools (of type T), else the 8-bit pool's code format
// (T is then the queries' type); the K / V maps address code rows.
template <typename T, int G, int FMT = -1>
__global__ void __launch_bounds__(FMT >= 0 ? NTHREADS_Q8 : NTHREADS, 1)
    paged_prefill(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const Params p) {
    constexpr bool Q8 = FMT >= 0;
    constexpr bool SCALES = FMT == dec::kFmtInt8;
    // 8-bit pools: the products run on f16 (bf16 queries are converted)
    using MT = typename std::conditional<Q8, __half, T>::type;
    constexpr bool QCONV = Q8 && !std::is_same<T, __half>::value;
    using LY = Lay<Q8>;
    constexpr int WMMA = Q8 ? WARP_MMA_Q8 : WARP_MMA;   // the first MMA warp
    constexpr int QT = BM / G;                    // queries per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = dec::smem_align_1k(smem_raw);
    const uint32_t sbase = dec::smem_u32(smem);
    auto bar = [&](int i) { return sbase + LY::bar + 8u * (uint32_t)i; };
    auto sbar = [&](int x, int i) { return bar(BAR_STREAM + x * SB_N + i); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::abort_flag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::tmem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bs = p.bs;

    dec::pdl_launch_dependents();
    dec::pdl_wait();                              // inputs of earlier kernels are visible

    // -- which (request, KV head, tile pair) this CTA takes -------------------
    // CTAs start in launch order (x fastest).  Requests are taken longest
    // first (the KV tiles their last queries walk), then their tile pairs from
    // the last (which sees the most tokens), so the long work starts early and
    // short work fills the tail.  Batches of more than kMaxRanked requests
    // keep the grid's own order.
    int b = blockIdx.z, g = blockIdx.y;
    int pt = (int)gridDim.x - 1 - (int)blockIdx.x;
    if (p.batch <= kMaxRanked) {
        int* cost = reinterpret_cast<int*>(smem + LY::order);
        int* pick = cost + kMaxRanked;
        const int k = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
        const int per_req = (int)(gridDim.x * gridDim.y);
        const int rank = k / per_req, rem = k % per_req;
        for (int i = tid; i < p.batch; i += (int)blockDim.x) {
            const int c0 = p.cu_seqlens[i], c1 = p.cu_seqlens[i + 1];
            const int Li = min(p.seq_lens[i], p.max_blocks * bs);
            cost[i] = (c1 > c0 && Li > 0) ? (Li + BN - 1) / BN : 0;
        }
        __syncthreads();
        for (int i = tid; i < p.batch; i += (int)blockDim.x) {
            const int ci = cost[i];
            int above = 0;                         // requests ordered before i
            for (int o = 0; o < p.batch; ++o) above += cost[o] > ci || (cost[o] == ci && o < i);
            if (above == rank) *pick = i;
        }
        __syncthreads();
        b = *pick;
        g = rem % (int)gridDim.y;
        pt = (int)gridDim.x - 1 - rem / (int)gridDim.y;
        __syncthreads();                           // every thread has read the pick
    }

    // -- the two tiles' queries and the tokens they see ----------------------
    int cu0 = p.cu_seqlens[b], cu1 = p.cu_seqlens[b + 1];
    int L = p.seq_lens[b];
    int C = cu1 - cu0;
    const bool bad_q = cu0 < 0 || cu1 < cu0 || cu1 > p.num_tokens;
    if (bad_q) C = 0;
    const int cap = p.max_blocks * bs;
    const bool bad_len = L > cap;
    L = max(0, min(L, cap));
    if (tid == 0 && pt == 0 && (bad_q || C > p.max_q)) atomicOr(p.err, KV_DEVERR_QUERY_RANGE);
    if (tid == 0 && pt == 0 && g == 0 && bad_len) atomicOr(p.err, KV_DEVERR_SEQ_RANGE);
    const int Cq = min(C, p.max_q);
    const int q0 = 2 * pt * QT;                    // first query of stream A
    const int nqa = min(QT, Cq - q0), nqb = min(QT, Cq - q0 - QT);
    if (nqa <= 0) return;                          // whole CTA, before any barrier
    const int nstreams = nqb > 0 ? 2 : 1;
    const int P0 = L - C + q0;                     // position of stream A's first query
    const int Pmax = P0 + (nstreams == 2 ? QT + nqb : nqa) - 1;   // the last query's (<= L - 1)
    // every active stream walks all tiles (rows past their own limit are
    // masked), so each K/V tile has exactly `nstreams` consumers
    const int ntiles = Pmax >= 0 ? Pmax / BN + 1 : 0;

    // -- set-up: barriers, TMEM ----------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < LY::nbars; ++i) {
            uint32_t count = 1;
            if ((i >= BAR_KE && i < BAR_KE + KST) || (i >= BAR_VE && i < BAR_VE + VST))
                count = (uint32_t)nstreams;
            // 8-bit pools: a ring slot is full when both converters of its side
            // have written their rows
            if (Q8 && ((i >= BAR_KF && i < BAR_KF + KST) || (i >= BAR_VF && i < BAR_VF + VST)))
                count = 2;
            if (i >= BAR_STREAM && i < NBARS &&
                ((i - BAR_STREAM) % SB_N == SB_SR || (i - BAR_STREAM) % SB_N == SB_PF))
                count = NSOFT;
            // INT8 scale ring: written by both producers, read by every softmax warp
            if (i >= BAR_SCF && i < BAR_SCF + SCS) count = 2;
            if (i >= BAR_SCE && i < BAR_SCE + SCS) count = (uint32_t)(NSOFT * nstreams);
            if (i == BAR_QC) count = (uint32_t)nstreams;   // one producer per query tile
            dec::mbar_init(bar(i), count);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == WMMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + LY::tmem),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_TMAK || warp == WARP_TMAV) {
        // ----------------------------------------------------- producers ----
        const bool is_k = warp == WARP_TMAK;
        const int nst = is_k ? KST : VST;
        const int full0 = is_k ? BAR_KF : BAR_VF, empty0 = is_k ? BAR_KE : BAR_VE;
        const uint32_t buf0 = sbase + (is_k ? OFF_K : OFF_V);
        const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
        const int R = p.box_rows;                  // rows per box: min(bs, BN)
        const int nbox = BN / R;                   // boxes per KV tile (<= 8)
        const uint32_t box_bytes = (uint32_t)R * 128u;   // one box, one 64-dim half
        if (ntiles > 0) {
            if (is_k && lane == 0) {
                dec::mbar_arrive_tx(bar(BAR_Q), (uint32_t)nstreams * QTILE);
                for (int x = 0; x < nstreams; ++x) {
                    const uint32_t d = sbase + OFF_Q + (uint32_t)x * QTILE;
                    dec::tma_load_3d(d, &tmap_q, 0, g * G, cu0 + q0 + x * QT, bar(BAR_Q));
                    dec::tma_load_3d(d + QHALF, &tmap_q, 64, g * G, cu0 + q0 + x * QT, bar(BAR_Q));
                }
            }
            const int32_t* table = p.block_tables + (size_t)b * p.max_blocks;
            if constexpr (Q8) {
                // Tile jj's code rows land in code stage jj % CST (INT8: its
                // token scales beside them); tile j is converted into ring
                // slot j % nst, which then counts as full.
                const uint32_t code0 = sbase + (is_k ? LY::ck : LY::cv);
                const int cfull0 = is_k ? BAR_CK : BAR_CV;
                float* csc = reinterpret_cast<float*>(smem + LY::csc) + (is_k ? 0 : CST * BN);
                const float* gsc = is_k ? p.k_scales : p.v_scales;
                int codes_issued = 0;
                auto issue_codes = [&](int jj) {
                    const int t = jj * BN + lane * R;   // first token of this lane's box
                    int row = -1, id = -1;
                    bool load = false;
                    if (lane < nbox && t < L) {
                        id = table[t / bs];
                        load = id >= 0 && id < p.num_blocks;
                        if (!load && is_k) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                        row = id * bs + t % bs;
                    }
                    const unsigned mask = __ballot_sync(FULL, load);
                    const uint32_t cb = bar(cfull0 + jj % CST);
                    const uint32_t per_box = (uint32_t)R * 128u + (SCALES ? (uint32_t)R * 4u : 0u);
                    if (lane == 0) dec::mbar_arrive_tx(cb, (uint32_t)__popc(mask) * per_box);
                    __syncwarp();
                    if (load) {
                        dec::tma_load_3d(code0 + (uint32_t)(jj % CST) * CTILE + (uint32_t)lane * R * 128u,
                                         map, 0, g, row, cb);
                        if constexpr (SCALES) {
                            const size_t srow = ((size_t)id * p.num_kv_heads + g) * bs + t % bs;
                            dec::bulk_load(dec::smem_u32(csc + (jj % CST) * BN + lane * R), gsc + srow,
                                           (uint32_t)R * 4u, cb);
                        }
                    }
                    codes_issued = jj + 1;
                };
                for (int jj = 0; jj < min(CST, ntiles); ++jj) issue_codes(jj);
                if constexpr (QCONV) {
                    // query tile x (the K producer stream A's, the V producer
                    // B's) into f16 in place: lane takes rows lane + 32 k
                    const int x = is_k ? 0 : 1;
                    if (x < nstreams) {
                        bool ok = true;
                        if (lane == 0) ok = wait_or_abort(bar(BAR_Q), 0, abort_flag, p.err, p.wait_ns);
                        if (__shfl_sync(FULL, ok ? 1 : 0, 0)) {
                            unsigned char* qt = smem + OFF_Q + (uint32_t)x * QTILE;
                            float* qinv = reinterpret_cast<float*>(smem + LY::qinv) + x * BM;
#pragma unroll 1
                            for (int k = 0; k < BM / 32; ++k) {
                                const int r = lane + 32 * k;
                                // the row's 16-byte chunk c: 64-dim half c / 8, chunk c % 8
                                auto chunk = [&](int c) {
                                    return reinterpret_cast<uint4*>(qt + (c >> 3) * QHALF + r * 128 +
                                                                    (((c & 7) ^ (r & 7)) << 4));
                                };
                                float amax = 0.f;
#pragma unroll 4
                                for (int c = 0; c < 16; ++c) {
                                    const uint4 w = *chunk(c);
                                    const uint32_t e4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        amax = fmaxf(amax, fmaxf(fabsf(H16<T>::low(e4[e])),
                                                                 fabsf(H16<T>::high(e4[e]))));
                                }
                                // 2^e with amax * 2^e in [2^14, 2^15): the exponent field of amax
                                int ex2 = 0;
                                if (amax > 0.f && amax <= 3.0e38f) {
                                    const int ex = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 126;
                                    ex2 = min(max(15 - ex, -120), 120);
                                }
                                const float up = __uint_as_float((uint32_t)(ex2 + 127) << 23);
                                qinv[r] = __uint_as_float((uint32_t)(127 - ex2) << 23);
#pragma unroll 4
                                for (int c = 0; c < 16; ++c) {
                                    const uint4 w = *chunk(c);
                                    uint32_t e4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        e4[e] = H16<__half>::pack(H16<T>::low(e4[e]) * up,
                                                                  H16<T>::high(e4[e]) * up);
                                    *chunk(c) = make_uint4(e4[0], e4[1], e4[2], e4[3]);
                                }
                            }
                            dec::fence_proxy_async();
                            __syncwarp();
                            if (lane == 0) dec::mbar_arrive(bar(BAR_QC));
                        }
                    }
                }
                for (int j = 0; j < ntiles; ++j) {
                    const int slot = j % nst, cs = j % CST;
                    bool ok = true;
                    if (lane == 0 && j >= nst)
                        ok = wait_or_abort(bar(empty0 + slot), (j / nst - 1) & 1, abort_flag, p.err,
                                           p.wait_ns);
                    if (lane == 0 && ok)
                        ok = wait_or_abort(bar(cfull0 + cs), (j / CST) & 1, abort_flag, p.err, p.wait_ns);
                    if (SCALES && lane == 0 && ok && j >= SCS)
                        ok = wait_or_abort(bar(BAR_SCE + j % SCS), (j / SCS - 1) & 1, abort_flag, p.err,
                                           p.wait_ns);
                    if (!__shfl_sync(FULL, ok ? 1 : 0, 0)) break;
                    // token rows 0..31 (the helper converter takes 32..63)
                    convert_row<MT, FMT>(smem + (is_k ? LY::ck : LY::cv) + (uint32_t)cs * CTILE,
                                         smem + (is_k ? OFF_K : OFF_V) + (uint32_t)slot * KVTILE, lane);
                    if constexpr (SCALES) {
                        float* ring = reinterpret_cast<float*>(smem + LY::sc) + (j % SCS) * 2 * BN +
                                      (is_k ? 0 : BN);
                        ring[lane] = csc[cs * BN + lane];
                        ring[lane + 32] = csc[cs * BN + lane + 32];
                    }
                    dec::fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) {
                        dec::mbar_arrive(bar(full0 + slot));
                        if constexpr (SCALES) dec::mbar_arrive(bar(BAR_SCF + j % SCS));
                    }
                    // the code stage is free once the helper has read its rows
                    // too: tile j + CST's codes into it
                    if (j + CST < ntiles) {
                        bool hok = true;
                        if (lane == 0)
                            hok = wait_or_abort(bar((is_k ? BAR_HK : BAR_HV) + cs), (j / CST) & 1,
                                                abort_flag, p.err, p.wait_ns);
                        if (!__shfl_sync(FULL, hok ? 1 : 0, 0)) break;
                        issue_codes(j + CST);
                    }
                }
                // Drain: no copy may still be landing in shared memory at exit.
                if (lane == 0) {
                    bool ok = !is_k || dec::mbar_wait(bar(BAR_Q), 0);
                    for (int jj = max(0, codes_issued - CST); jj < codes_issued; ++jj)
                        ok &= dec::mbar_wait(bar(cfull0 + jj % CST), (jj / CST) & 1);
                    if (!ok) atomicOr(p.err, KV_DEVERR_TIMEOUT);
                }
            } else {
                int issued = 0;
                for (int j = 0; j < ntiles; ++j) {
                    const int slot = j % nst;
                    bool ok = true;
                    // tile j reuses the buffer of tile j - nst: freed when every
                    // stream's S (K) or PV (V) of that tile is done
                    if (lane == 0 && j >= nst)
                        ok = wait_or_abort(bar(empty0 + slot), (j / nst - 1) & 1, abort_flag, p.err,
                                           p.wait_ns);
                    if (!__shfl_sync(FULL, ok ? 1 : 0, 0)) break;
                    const int t = j * BN + lane * R;   // first token of this lane's box
                    int row = -1;
                    bool load = false;
                    if (lane < nbox && t < L) {
                        const int id = table[t / bs];
                        load = id >= 0 && id < p.num_blocks;
                        if (!load && is_k) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                        row = id * bs + t % bs;
                    }
                    const unsigned mask = __ballot_sync(FULL, load);
                    if (lane == 0)
                        dec::mbar_arrive_tx(bar(full0 + slot), (uint32_t)__popc(mask) * 2u * box_bytes);
                    __syncwarp();
                    if (load) {
                        const uint32_t d = buf0 + (uint32_t)slot * KVTILE + (uint32_t)lane * box_bytes;
                        dec::tma_load_3d(d, map, 0, g, row, bar(full0 + slot));
                        dec::tma_load_3d(d + KVHALF, map, 64, g, row, bar(full0 + slot));
                    }
                    issued = j + 1;
                }
                // Drain: no copy may still be landing in shared memory at exit.
                if (lane == 0) {
                    bool ok = !is_k || dec::mbar_wait(bar(BAR_Q), 0);
                    for (int j = max(0, issued - nst); j < issued; ++j)
                        ok &= dec::mbar_wait(bar(full0 + j % nst), (j / nst) & 1);
                    if (!ok) atomicOr(p.err, KV_DEVERR_TIMEOUT);
                }
            }
        }
    } else if (Q8 && (warp == WARP_CVK || warp == WARP_CVV)) {
      if constexpr (Q8) {
        // ------------------------------------- helper converters (8-bit) ----
        // Token rows 32..63 of every tile of its side, from the code stage the
        // producer loaded into the ring slot the producer fills too; the slot
        // counts as full after both have arrived, and the code stage is
        // refilled only after this warp has said it is done reading.
        const bool is_k = warp == WARP_CVK;
        const int nst = is_k ? KST : VST;
        const int full0 = is_k ? BAR_KF : BAR_VF, empty0 = is_k ? BAR_KE : BAR_VE;
        const int cfull0 = is_k ? BAR_CK : BAR_CV, hdone0 = is_k ? BAR_HK : BAR_HV;
        for (int j = 0; j < ntiles; ++j) {
            const int slot = j % nst, cs = j % CST;
            bool ok = true;
            if (lane == 0 && j >= nst)
                ok = wait_or_abort(bar(empty0 + slot), (j / nst - 1) & 1, abort_flag, p.err,
                                   p.wait_ns);
            if (lane == 0 && ok)
                ok = wait_or_abort(bar(cfull0 + cs), (j / CST) & 1, abort_flag, p.err, p.wait_ns);
            if (!__shfl_sync(FULL, ok ? 1 : 0, 0)) break;
            convert_row<MT, FMT>(smem + (is_k ? LY::ck : LY::cv) + (uint32_t)cs * CTILE,
                                 smem + (is_k ? OFF_K : OFF_V) + (uint32_t)slot * KVTILE, lane + 32);
            dec::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                dec::mbar_arrive(bar(full0 + slot));
                dec::mbar_arrive(bar(hdone0 + cs));
            }
        }
      }
    } else if (warp >= WMMA) {
        // ----------------------------------------------------------- MMA ----
        // One warp per stream runs the loop (waits included) so every operand
        // is warp-uniform; one elected lane issues each tcgen05 instruction.
        const int x = warp - WMMA;
        if (ntiles > 0 && x < nstreams) {
            constexpr uint32_t fmt = H16<MT>::kFmt;
            constexpr uint32_t id_s = idesc_f16(fmt, 0, BM, BN);   // S = Q K^T
            constexpr uint32_t id_pv = idesc_f16(fmt, 1, BM, D);   // O += P V (V MN-major)
            const uint32_t tm = __shfl_sync(FULL, tmem, 0) + (uint32_t)x * COL_STREAM;
            // base descriptors; a K step adds (byte offset >> 4) to the start field
            const uint64_t dq = sdesc_sw128(sbase + OFF_Q + (uint32_t)x * QTILE, 16u, 1024u);
            const uint64_t dk = sdesc_sw128(sbase + OFF_K, 16u, 1024u);
            const uint64_t dv = sdesc_sw128(sbase + OFF_V, KVHALF, 1024u);
            auto wait_all = [&](uint32_t bb, uint32_t parity) {
                return __all_sync(FULL, wait_or_abort(bb, parity, abort_flag, p.err, p.wait_ns));
            };
            bool ok = wait_all(bar(QCONV ? BAR_QC : BAR_Q), 0);
            int done_pv = 0;                       // PV products issued
            auto pv = [&](int jj) -> bool {
                const int s = jj % VST;
                if (!wait_all(sbar(x, SB_PF), jj & 1)) return false;
                if (!wait_all(bar(BAR_VF + s), (jj / VST) & 1)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // 16 tokens = two 8-row swizzle atoms (2 KB); the two
                        // 64-dim halves are KVHALF apart (leading byte offset)
                        const uint64_t vdesc = dv + (uint64_t)(((uint32_t)s * KVTILE + (uint32_t)kk * 2048u) >> 4);
                        mma_ts(tm + COL_O, tm + COL_PH + (uint32_t)kk * 8u, vdesc, id_pv,
                               (jj > 0 || kk > 0) ? 1u : 0u);
                        mma_ts(tm + COL_O, tm + COL_PL + (uint32_t)kk * 8u, vdesc, id_pv, 1u);
                    }
                    mma_commit(bar(BAR_VE + s));
                    mma_commit(sbar(x, SB_OF));
                }
                __syncwarp();
                done_pv = jj + 1;
                return true;
            };
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j % KST;
                if (!wait_all(bar(BAR_KF + s), (j / KST) & 1)) break;
                // S_j overwrites S_{j-1}: the softmax must have read it
                if (j > 0 && !wait_all(sbar(x, SB_SR), (j - 1) & 1)) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        // 16 dims = 32 bytes inside a 128-byte swizzled row
                        const uint32_t qo = ((uint32_t)(kk >> 2) * QHALF + (uint32_t)(kk & 3) * 32u) >> 4;
                        const uint32_t ko = ((uint32_t)s * KVTILE + (uint32_t)(kk >> 2) * KVHALF +
                                             (uint32_t)(kk & 3) * 32u) >> 4;
                        mma_ss(tm + COL_S, dq + qo, dk + ko, id_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(BAR_KE + s));
                    mma_commit(sbar(x, SB_SF));
                }
                __syncwarp();
                if (j > 0 && !pv(j - 1)) break;
            }
            if (ok && *abort_flag == 0 && done_pv == ntiles - 1) pv(ntiles - 1);
            // Drain: every MMA issued has completed before TMEM is freed --
            // after an abort too, so this wait takes the full limit and does
            // not give up because another role did.
            if (elect_one()) mma_commit(sbar(x, SB_DR));
            __syncwarp();
            if (!__all_sync(FULL, dec::mbar_wait(sbar(x, SB_DR), 0, kWaitLimitNs)))
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp / NSOFT < nstreams) {
        // ---------------------------------------------- softmax, epilogue ----
        const int x = warp / NSOFT, qd = warp % NSOFT;
        const int r = 32 * qd + lane;              // row = TMEM lane
        const int qi = r / G, hh = r % G;
        const int nq = x == 0 ? nqa : nqb;
        const bool valid = qi < nq;
        const int lim = valid ? P0 + x * QT + qi : -1;   // last visible position
        const uint32_t trow = tmem + (uint32_t)x * COL_STREAM + ((uint32_t)(32 * qd) << 16);
        const int stid = tid - x * NSOFT * 32;     // thread index within the stream
        float qs = p.qscale;
        float m = -CUDART_INF_F;
        float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // partial row sums
        bool ok = true;
        // tcgen05.ld / st are warp-collective: every wait's outcome is made
        // uniform across the warp; after a failed wait the warp touches
        // neither TMEM nor the pipeline barriers again.
        auto wait_warp = [&](uint32_t bb, uint32_t parity) {
            return __all_sync(FULL, wait_or_abort(bb, parity, abort_flag, p.err, p.wait_ns));
        };
        if constexpr (QCONV) {
            // the row's 2^-e, written with the converted query tile
            if (ntiles > 0) {
                ok = wait_warp(bar(BAR_QC), 0);
                if (ok) qs *= reinterpret_cast<const float*>(smem + LY::qinv)[x * BM + r];
            }
        }
        for (int j = 0; ok && j < ntiles; ++j) {
            const int t0 = j * BN;
            uint32_t sv[2][32];
            ok = wait_warp(sbar(x, SB_SF), j & 1);
            if (!ok) break;
            tc_fence_after();
            tmem_ld32(trow + COL_S, sv[0]);
            tmem_ld32(trow + COL_S + 32u, sv[1]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) dec::mbar_arrive(sbar(x, SB_SR));   // S may be overwritten
            // INT8: the tile's token scales (K, then V), released once P is built
            const float* tsc = reinterpret_cast<const float*>(smem + LY::sc) + (j % SCS) * 2 * BN;
            if constexpr (SCALES) {
                ok = wait_warp(bar(BAR_SCF + j % SCS), (j / SCS) & 1);
                if (!ok) break;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        sv[c][e] = __float_as_uint(__uint_as_float(sv[c][e]) * tsc[32 * c + e]);
            }
            // causal / length mask: tokens past `lim` do not exist for this row
            if (t0 + BN - 1 > lim) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (t0 + 32 * c + e > lim) sv[c][e] = __float_as_uint(-CUDART_INF_F);
            }
            float mx2[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                mx2[c] = fmaxf(__uint_as_float(sv[c][0]), __uint_as_float(sv[c][1]));
#pragma unroll
                for (int e = 2; e < 32; e += 2)
                    mx2[c] = max3(mx2[c], __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
            }
            const float m_new = fmaxf(m, fmaxf(mx2[0], mx2[1]) * qs);
            float alpha = 1.f;
            const bool grow = m_new > m + kRescaleLog2;   // false while both are -inf
            if (grow) {
                alpha = dec::fast_exp2(m - m_new);       // 0 when m was -inf
                m = m_new;
            }
            const float mu = m == -CUDART_INF_F ? 0.f : m;
            l2[0] = __fmul2_rn(l2[0], make_float2(alpha, alpha));
            l2[1] = __fmul2_rn(l2[1], make_float2(alpha, alpha));
            // P = hi + lo of the tile's 64 tokens, in registers until PV_{j-1}
            // has finished with the P columns
            const float2 qs2 = make_float2(qs, qs), nmu2 = make_float2(-mu, -mu);
            uint32_t ph[32], pl[32];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 xx = __ffma2_rn(
                        make_float2(__uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1])), qs2,
                        nmu2);
                    const float2 pp = make_float2(dec::fast_exp2(xx.x), dec::fast_exp2(xx.y));
                    l2[(e >> 1) & 1] = __fadd2_rn(l2[(e >> 1) & 1], pp);
                    float2 pv = pp;
                    if constexpr (SCALES) {
                        // P times the token's V scale (0 where P is: masked
                        // tokens' scales may be anything)
                        const float v0 = tsc[BN + 32 * c + e], v1 = tsc[BN + 32 * c + e + 1];
                        pv = make_float2(pp.x > 0.f ? pp.x * v0 : 0.f, pp.y > 0.f ? pp.y * v1 : 0.f);
                    }
                    H16<MT>::split(pv.x, pv.y, ph[16 * c + e / 2], pl[16 * c + e / 2]);
                }
            if constexpr (SCALES) {
                __syncwarp();                     // every lane has read the tile's scales
                if (lane == 0) dec::mbar_arrive(bar(BAR_SCE + j % SCS));
            }
            // the last tile: zero V rows past the sequence end (P is 0 there,
            // but 0 x NaN from an unwritten row would poison the product);
            // each stream zeroes before its own PV (both write the same zeros)
            if (j * BN + BN > L) {
                ok = wait_warp(bar(BAR_VF + j % VST), (j / VST) & 1);
                if (!ok) break;
                const int r0 = max(L - j * BN, 0);
                unsigned char* vt = smem + OFF_V + (uint32_t)(j % VST) * KVTILE;
                const int nchunks = (BN - r0) * 16;     // 16-byte chunks in both halves
                for (int i = stid; i < nchunks; i += NSOFT * 32) {
                    const int row = r0 + (i >> 4), ch = i & 15;
                    *reinterpret_cast<uint4*>(vt + (ch >> 3) * KVHALF + row * 128 + (ch & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                dec::fence_proxy_async();
            }
            // PV_{j-1} done: the P columns are free and O holds tile j-1's sum;
            // rescale O when any row's maximum grew
            if (j > 0) {
                ok = wait_warp(sbar(x, SB_OF), (j - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(FULL, grow)) {
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
            }
            tmem_st32(trow + COL_PH, ph);
            tmem_st32(trow + COL_PL, pl);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) dec::mbar_arrive(sbar(x, SB_PF));
        }
        // -- epilogue: out = O / l, rounded once to the output type ----------
        const bool have_o = ok && ntiles > 0 && wait_warp(sbar(x, SB_OF), (ntiles - 1) & 1);
        if (have_o) tc_fence_after();
        const float l = (l2[0].x + l2[0].y) + (l2[1].x + l2[1].y);
        const bool done = have_o || (ok && ntiles == 0);
        const float inv = l > 0.f ? p.vscale / l : 0.f;   // FP8: the pool's V scale
        T* orow = static_cast<T*>(p.out) +
                  ((size_t)(cu0 + q0 + x * QT + qi) * p.num_q_heads + (size_t)g * G + hh) * D;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            if (have_o) {
                tmem_ld32(trow + COL_O + 32u * c, ov);
                tmem_wait_ld();
            }
            if (valid && done) {
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
    if (warp == WMMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

}  // namespace pf
}  // namespace pagedkv
