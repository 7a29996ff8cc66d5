// Cascade (shared-prefix) decode, first pass, on the 5th-generation tensor
// cores: tcgen05.mma with the K/V tiles staged by TMA in shared memory and
// the score and output accumulators in tensor memory (TMEM).
//
// What is computed is the prefix pass of decode_prefix.cuh: for a sub-group
// of a group's members (16 query rows = members x the G heads of one KV
// head) and the blocks all of them share, a normalised partial output and
// its log2-sum-exp per row ("prefix state"), which the split kernel folds
// into each sequence's log-sum-exp merge ("Lecture 24", semidirectx.com CMU
// 11-868 notes, sec. 3.2; the S06 page, llminference.xinbetween.com, "In
// production", names this cascade split for shared prompts).
//
// Orientation.  With only 16 query rows per KV tile, the products are taken
// transposed so that no MMA row is padding: a unit is a tile of 128 shared
// tokens (8 blocks of 16 or 4 of 32; fewer in a segment's last tile), and
//   S^T  = K_tile Q^T     M = 128 tokens, N = 16 rows, K = 128 dims
//   P^T  = exp2(S^T * scale * log2 e - m)     (softmax warps, fp32)
//   O^T += V_tile^T P^T   M = 128 dims,   N = 16 rows, K = the tile's tokens
// K_tile is a K-major A operand, V_tile^T an MN-major one (the tile as TMA
// leaves it, 128-byte swizzled, serves both), Q and P^T K-major B operands.
// P^T is stored as 16-bit hi + lo halves (P = hi + lo to 2^-16 relative):
// one B operand of 32 rows (hi, then lo), so one N = 32 product accumulates
// O_hi^T and O_lo^T side by side and the epilogue adds them -- the result
// keeps fp32-level accuracy for half the MMA instructions.  The running
// maximum is updated lazily: O^T and the sums are rescaled only when a row's
// maximum grows by more than 2^8, so P stays below 256.
//
// Thread (warp w < 4, lane) of the softmax warps owns TMEM lane 32 w + lane:
// token t of a tile's S^T (its 16 scores, one per row) and dim d of O^T.  A
// row's maximum over the tile is a transposed butterfly in the warp and a
// 4-warp exchange in shared memory; a row's sum stays a per-thread partial
// until the piece ends.
//
// Pools: 16-bit, head_dim 128, block size 16 or 32 (8-bit pools take the
// mma.sync pass of decode_prefix.cuh, which converts codes in registers).
// The K and V tiles have rings of their own, each fed by its own producer
// warp: a K tile is consumed by S^T early and its stage refilled at once,
// while a V tile stays until its O^T product.
//
// The prefix covers only blocks that are full for every member, so no token
// of a tile is masked for some rows and not for others, and a tile's valid
// tokens are a multiple of 16.  Work split, partial slots and tagged piece
// counters are the mma.sync pass's: a persistent grid cut into equal unit
// ranges, and the CTA finishing the last piece of a cut segment merges.
#pragma once

#include "decode_prefix.cuh"
#include "prefill_kernel.cuh"

namespace pagedkv {
namespace ptc {

using dec::FULL;
using dec::PParams;

constexpr int D = 128;
constexpr int TOK = 128;                  // tokens per unit tile
constexpr int NR = dec::kRows;            // query rows (MMA N)
constexpr int NSOFT = 4;                  // softmax warps: TMEM lanes 0-127
// producers of K (and Q) and of V; S^T issue (and TMEM allocation); O^T issue
constexpr int WARP_PK = NSOFT, WARP_PV_LOAD = NSOFT + 1, WARP_MMA = NSOFT + 2, WARP_PV = NSOFT + 3;
constexpr int NTHREADS = (NSOFT + 4) * 32;

constexpr uint32_t KVHALF = TOK * 128u;   // 128 rows x 128 B: one 64-dim half of a 16-bit tile
constexpr uint32_t KVTILE = 2u * KVHALF;  // a K or V tile, 32 KB
constexpr uint32_t QHALF = NR * 128u;     // 16 rows x 128 B
constexpr uint32_t QBUF = 2u * QHALF;     // 4 KB
constexpr uint32_t PHALF = 2u * NR * 128u;  // 32 rows (hi, lo) x 64 tokens
constexpr uint32_t PBUF = 2u * PHALF;       // 8 KB: P^T hi and lo of one tile
constexpr uint32_t TMEM_COLS = 64;
constexpr uint32_t COL_S = 0, COL_O = 32; // S^T: two buffers of 16 columns; O^T: 32 (hi, lo)
constexpr float kRescaleLog2 = 8.f;

// barriers after the rings' (pairs are per buffer: Q by piece, S^T and P^T
// by unit parity; the drain one per MMA warp)
enum { B_QFULL = 0, B_QEMPTY = 2, B_SFULL = 4, B_SFREE = 6, B_PFULL = 8, B_PVDONE = 10,
       B_DRAIN = 12, B_N = 14 };

// Shared memory of one CTA (offsets from a 1 KB-aligned base): the K and V
// rings (KS / VS tiles), the query rows and P^T buffers, barriers, scratch
// and the groups' tables.
struct TLayout {
    uint32_t kring, vring, q, p, bars, red, misc, gcum, vg, total;
    int KS, VS;
    __host__ __device__ TLayout(int KS_, int VS_, int K) : KS(KS_), VS(VS_) {
        uint32_t off = 0;
        kring = off;   off += KVTILE * (uint32_t)KS;
        vring = off;   off += KVTILE * (uint32_t)VS;
        q = off;       off += 2u * QBUF;
        p = off;       off += 2u * PBUF;      // by unit parity
        bars = off;    off += 8u * (uint32_t)(2 * KS + 2 * VS + B_N);
        off = (off + 15u) & ~15u;
        red = off;     off += 4u * (2 * NSOFT * NR + NSOFT * NR);
        misc = off;    off += 4u * 40;
        gcum = off;    off += 4u * (uint32_t)(K + 1);
        vg = off;      off += 4u * 3u * (uint32_t)K;
        total = off;
    }
    __host__ __device__ uint32_t kfull(int s) const { return bars + 8u * s; }
    __host__ __device__ uint32_t kempty(int s) const { return bars + 8u * (KS + s); }
    __host__ __device__ uint32_t vfull(int s) const { return bars + 8u * (2 * KS + s); }
    __host__ __device__ uint32_t vempty(int s) const { return bars + 8u * (2 * KS + VS + s); }
    __host__ __device__ uint32_t bar(int i) const { return bars + 8u * (2 * KS + 2 * VS + i); }
};

// Instruction descriptor of kind::f16 (fp32 accumulator, A and B of one
// 16-bit type), either operand K- or MN-major.
__host__ __device__ constexpr uint32_t idesc(uint32_t fmt, uint32_t a_mn, uint32_t b_mn, uint32_t M,
                                             uint32_t N) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

// Barrier among the softmax warps (id 1, 128 threads) that also tells every
// thread whether any of them passed `fail`.
__device__ __forceinline__ bool soft_sync_any(bool fail) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"((uint32_t)fail), "n"(NSOFT * 32)
        : "memory");
    return r != 0;
}

// One butterfly step of warp_rows: lanes with bit BIT set keep rows
// HALF .. 2 HALF - 1 of their 2 HALF and send the lower half, the others the
// reverse; each combines what it kept with its partner's.
template <bool MAX, int HALF, int BIT>
__device__ __forceinline__ void rows_step(float (&v)[NR], int lane) {
    const bool up = (lane & BIT) != 0;
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
        const float keep = up ? v[i + HALF] : v[i];
        const float send = up ? v[i] : v[i + HALF];
        const float got = __shfl_xor_sync(FULL, send, BIT);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
}
// Per row r of the 16: reduce v[r] over the warp's lanes (max or sum).  On
// return, lane l holds row row_of(l)'s result in v[0].
template <bool MAX>
__device__ __forceinline__ void warp_rows(float (&v)[NR], int lane) {
    rows_step<MAX, 8, 16>(v, lane);
    rows_step<MAX, 4, 8>(v, lane);
    rows_step<MAX, 2, 4>(v, lane);
    rows_step<MAX, 1, 2>(v, lane);
    const float got = __shfl_xor_sync(FULL, v[0], 1);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
}
__device__ __forceinline__ int row_of(int lane) {
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

// Bounded wait by one lane, outcome shared by the warp.  The lane sleeps in
// the barrier between polls (the hardware wakes it when the phase
// completes), so a waiting role takes no issue slots from the softmax warps
// on its sub-partition.  On expiry, or when another role has
// already given up, it raises the abort flag and returns false.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, unsigned long long limit, int lane) {
    int ok = 1;
    if (lane == 0) {
        ok = limit == 0 ? dec::mbar_test(bar, parity) : dec::mbar_try(bar, parity);
        if (!ok && !*abort_flag && limit > 0) ok = dec::mbar_wait_sleep(bar, parity, limit);
        if (!ok) {
            *abort_flag = 1;
            atomicOr(err, KV_DEVERR_TIMEOUT);
        }
    }
    return __shfl_sync(FULL, ok, 0) != 0;
}

// T: the pool's (and the queries') 16-bit type; BS: block size (16 or 32).
// p.stages is the depth of each ring.  The per-sequence pass's work unit is
// one block here, so the prefix is counted in blocks.
template <typename T, int G, int BS>
__global__ void __launch_bounds__(NTHREADS, 1) paged_decode_prefix_tc(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const PParams p) {
    constexpr uint32_t fmt = pf::H16<T>::kFmt;
    constexpr int TB = TOK / BS;                  // blocks per full tile
    constexpr int MS = NR / G;                    // members per sub-group
    constexpr int NT = NTHREADS;
    constexpr int ub = 1;                         // blocks per unit of the per-sequence pass
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = dec::smem_align_1k(smem_raw);
    const uint32_t sbase = dec::smem_u32(smem);
    const int K = p.num_groups, H = p.num_kv_heads, B = p.batch;
    const int KS = p.stages, VS = p.stages;
    const TLayout lay(KS, VS, K);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.misc) + 1;
    int* warp_tot = reinterpret_cast<int*>(smem + lay.misc) + 8;
    int* gcum = reinterpret_cast<int*>(smem + lay.gcum);
    int* vg = reinterpret_cast<int*>(smem + lay.vg);
    const int* gfirst = vg;
    const int* gsize = vg + K;
    const int* gunits = vg + 2 * K;               // shared blocks (units of `ub` blocks)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cap = p.max_blocks * BS;

    if (tid == 0) {
        for (int s = 0; s < KS; ++s) {
            dec::mbar_init(sbase + lay.kfull(s), 1);
            dec::mbar_init(sbase + lay.kempty(s), 1);
        }
        for (int s = 0; s < VS; ++s) {
            dec::mbar_init(sbase + lay.vfull(s), 1);
            dec::mbar_init(sbase + lay.vempty(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            dec::mbar_init(sbase + lay.bar(B_QFULL + x), 1);
            dec::mbar_init(sbase + lay.bar(B_QEMPTY + x), 1);
            dec::mbar_init(sbase + lay.bar(B_SFULL + x), 1);
            dec::mbar_init(sbase + lay.bar(B_SFREE + x), NSOFT);
            dec::mbar_init(sbase + lay.bar(B_PFULL + x), NSOFT);
            dec::mbar_init(sbase + lay.bar(B_PVDONE + x), 1);
            dec::mbar_init(sbase + lay.bar(B_DRAIN + x), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // The second pass is let in only after this wait: the pool is then
    // complete, so that pass may stream its blocks before this one ends.
    dec::pdl_wait();
    dec::pdl_launch_dependents();

    // -- used groups and their units (sub-groups x KV heads x tiles) ----------
    const int NG = dec::load_groups(p.g_first, p.g_size, p.g_blocks, K, p.seq_lens, B, BS, cap, ub,
                                    vg, warp_tot, p.err);
    auto tiles_of = [&](int k) { return (gunits[k] * ub + TB - 1) / TB; };
    {
        const int per = (NG + NT - 1) / NT;
        const int k0 = min(NG, tid * per), k1 = min(NG, k0 + per);
        int local = 0;
        for (int k = k0; k < k1; ++k) local += ((gsize[k] + MS - 1) / MS) * H * tiles_of(k);
        int total = 0;
        int run = dec::block_excl_sum(local, warp_tot, &total);
        for (int k = k0; k < k1; ++k) {
            gcum[k] = run;
            run += ((gsize[k] + MS - 1) / MS) * H * tiles_of(k);
        }
        if (tid == 0) gcum[NG] = total;
    }
    __syncthreads();

    const int U = gcum[NG];
    const int chunk = dec::unit_chunk(U, p.num_ctas);
    const int start = blockIdx.x * chunk;
    const int end = min(U, start + chunk);
    if (start >= end) return;                     // whole CTA, before TMEM is allocated

    if (warp == WARP_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         sbase + lay.misc + 4u),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pf::tc_fence_before();
    __syncthreads();
    pf::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // unit u: group k, sub-group, KV head g, tile j of the segment
    struct Unit {
        int k, sub, g, j, seg, tiles, nb;
    };
    auto unit = [&](int u) {
        Unit x;
        x.k = dec::find_le(gcum, NG, u);
        x.tiles = tiles_of(x.k);
        const int r = u - gcum[x.k];
        const int sg = r / x.tiles;
        x.sub = sg / H;
        x.g = sg % H;
        x.j = r % x.tiles;
        x.seg = gcum[x.k] + sg * x.tiles;
        x.nb = min(TB, gunits[x.k] * ub - x.j * TB);
        return x;
    };
    // the unit after x (every role walks its range in order, so the search
    // and divisions of unit() run once per role)
    auto advance = [&](Unit& x) {
        if (++x.j < x.tiles) {
            x.nb = min(TB, gunits[x.k] * ub - x.j * TB);
            return;
        }
        x.j = 0;
        x.seg += x.tiles;
        if (++x.g == H) {
            x.g = 0;
            if (++x.sub == (gsize[x.k] + MS - 1) / MS) {
                x.sub = 0;
                ++x.k;
                x.tiles = tiles_of(x.k);
            }
        }
        x.nb = min(TB, gunits[x.k] * ub);
    };
    auto first_of = [&](int u, const Unit& x) { return u == start || u == x.seg; };
    auto last_of = [&](int u, const Unit& x) { return u == end - 1 || u == x.seg + x.tiles - 1; };

    if (warp == WARP_PK || warp == WARP_PV_LOAD) {
        // -------------------------------------------------------- producers --
        // One warp for K tiles (and the pieces' query rows), one for V tiles,
        // so a K tile is fetched as soon as the S^T before it has freed its
        // stage, however long the V tiles stay in use.
        const bool is_k = warp == WARP_PK;
        const int nst = is_k ? KS : VS;
        const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
        int issued = 0, pi = -1;
        bool ok = true;
        auto full_of = [&](int s) { return is_k ? lay.kfull(s) : lay.vfull(s); };
        auto empty_of = [&](int s) { return is_k ? lay.kempty(s) : lay.vempty(s); };
        // Block ids, a batch of 32 / TB units at a time: lane l holds block
        // l % TB of unit b0 + l / TB; the next batch's table loads are in
        // flight while the current batch's units are issued.
        constexpr int UPB = 32 / TB;              // units per batch
        auto fetch = [&](int b0) {
            const int v = b0 + lane / TB, blk = lane % TB;
            if (v >= end) return -1;
            const Unit y = unit(v);
            return blk < y.nb
                       ? __ldg(p.block_tables + (size_t)gfirst[y.k] * p.max_blocks + y.j * TB + blk)
                       : -1;
        };
        int ids_cur = fetch(start), ids_nxt = fetch(start + UPB);
        Unit x = unit(start);
        for (int u = start; ok && u < end; ++u) {
            const int i = u - start;
            if (i > 0) advance(x);
            if (i > 0 && i % UPB == 0) {
                ids_cur = ids_nxt;
                ids_nxt = fetch(u + UPB);
            }
            const int id = __shfl_sync(FULL, ids_cur, ((i % UPB) * TB + lane) & 31);
            // A piece's first unit (K side): its 16 query rows are loaded into
            // registers first, the tile's copies issued, and only then does the
            // warp wait for Q buffer pi % 2 and store the rows, so the query
            // loads and the tile's copies are in flight together.
            const bool qpiece = is_k && first_of(u, x);
            const int c = lane >> 1, h = lane & 1, m = c / G, hh = c % G;   // (row c, 64-dim half h)
            uint4 raw[8];
            int qb = 0;
            if (qpiece) {
                ++pi;
                qb = pi & 1;
                const int m0 = gfirst[x.k] + x.sub * MS;
                const int msz = min(MS, gsize[x.k] - x.sub * MS);
                const T* src = static_cast<const T*>(p.q) +
                               ((size_t)(m0 + m) * p.num_q_heads + x.g * G + hh) * D + h * 64;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    raw[ch] = m < msz ? __ldg(reinterpret_cast<const uint4*>(src) + ch)
                                      : make_uint4(0u, 0u, 0u, 0u);
            }
            // the tile's blocks: lane 2 b + c makes copy c of block b
            const int s = i % nst;
            if (i >= nst)
                ok = warp_wait(sbase + empty_of(s), ((i / nst) - 1) & 1, abort_flag, p.err, p.wait_ns,
                               lane);
            if (!ok) break;
            bool load = false;
            if (lane < x.nb) {
                load = id >= 0 && id < p.num_blocks;
                if (!load && is_k) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
            }
            const unsigned mask = __ballot_sync(FULL, load);
            const uint32_t fb = sbase + full_of(s);
            constexpr uint32_t per_block = 2u * BS * 128u;   // both 64-dim halves
            if (lane == 0) dec::mbar_arrive_tx(fb, (uint32_t)__popc(mask) * per_block);
            __syncwarp();
            const int bb = lane >> 1, cc = lane & 1;
            const int bid = __shfl_sync(FULL, id, bb);
            if (bb < TB && ((mask >> bb) & 1u)) {
                // cc = the 64-dim half
                const uint32_t d = sbase + (is_k ? lay.kring : lay.vring) + (uint32_t)s * KVTILE +
                                   (uint32_t)cc * KVHALF + (uint32_t)bb * BS * 128u;
                dec::tma_load_3d(d, map, cc * 64, x.g, bid * BS, fb);
            }
            issued = i + 1;
            if (qpiece) {
                if (pi >= 2)
                    ok = warp_wait(sbase + lay.bar(B_QEMPTY + qb), ((pi >> 1) - 1) & 1, abort_flag,
                                   p.err, p.wait_ns, lane);
                if (!ok) break;
                unsigned char* qdst = smem + lay.q + (uint32_t)qb * QBUF + (uint32_t)h * QHALF + c * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4*>(qdst + ((ch ^ (c & 7)) << 4)) = raw[ch];
                dec::fence_proxy_async();
                __syncwarp();
                if (lane == 0) dec::mbar_arrive(sbase + lay.bar(B_QFULL + qb));
            }
        }
        // Drain (full limit): no copy may still be landing at exit.
        if (lane == 0) {
            bool dok = true;
            for (int i = max(0, issued - nst); i < issued; ++i)
                dok &= dec::mbar_wait(sbase + full_of(i % nst), (i / nst) & 1, kWaitLimitNs);
            if (!dok) atomicOr(p.err, KV_DEVERR_TIMEOUT);
        }
    } else if (warp == WARP_MMA || warp == WARP_PV) {
        // -------------------------------------------------------------- MMA --
        // Two issuing warps, so a product waits only for its own inputs: S^T
        // of unit i needs its K tile and the free S^T buffer i % 2; O^T of
        // unit i needs P^T buffer i % 2 and the V tile.  One elected lane
        // issues each instruction.
        constexpr uint32_t id_s = idesc(fmt, 0, 0, TOK, NR);    // S^T = K Q^T
        constexpr uint32_t id_pv = idesc(fmt, 1, 0, D, 2 * NR); // O^T += V^T P^T (V^T MN-major)
        const uint32_t tm = __shfl_sync(FULL, tmem, 0);
        const int n = end - start;
        auto wait = [&](uint32_t b, uint32_t par) {
            return warp_wait(sbase + b, par, abort_flag, p.err, p.wait_ns, lane);
        };
        const int xw = warp == WARP_MMA ? 0 : 1;
        Unit x = unit(start);
        if (xw == 0) {
            const uint64_t dq = pf::sdesc_sw128(sbase + lay.q, 16u, 1024u);
            const uint64_t dk = pf::sdesc_sw128(sbase + lay.kring, 16u, 1024u);
            int pi = -1;
            for (int i = 0; i < n; ++i) {
                const int u = start + i, s = i % KS;
                if (i > 0) advance(x);
                if (!wait(lay.kfull(s), (i / KS) & 1)) break;
                if (first_of(u, x)) {
                    ++pi;
                    if (!wait(lay.bar(B_QFULL + (pi & 1)), (pi >> 1) & 1)) break;
                }
                if (i >= 2 && !wait(lay.bar(B_SFREE + (i & 1)), ((i >> 1) - 1) & 1)) break;
                pf::tc_fence_after();
                if (pf::elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ko = ((uint32_t)s * KVTILE + (uint32_t)(kk >> 2) * KVHALF +
                                             (uint32_t)(kk & 3) * 32u) >> 4;
                        const uint32_t qo = ((uint32_t)(pi & 1) * QBUF + (uint32_t)(kk >> 2) * QHALF +
                                             (uint32_t)(kk & 3) * 32u) >> 4;
                        pf::mma_ss(tm + COL_S + 16u * (uint32_t)(i & 1), dk + ko, dq + qo, id_s,
                                   kk > 0 ? 1u : 0u);
                    }
                    pf::mma_commit(sbase + lay.bar(B_SFULL + (i & 1)));
                    pf::mma_commit(sbase + lay.kempty(s));
                    if (last_of(u, x)) pf::mma_commit(sbase + lay.bar(B_QEMPTY + (pi & 1)));
                }
                __syncwarp();
            }
        } else {
            const uint64_t dv = pf::sdesc_sw128(sbase + lay.vring, KVHALF, 1024u);
            const uint64_t dp = pf::sdesc_sw128(sbase + lay.p, 16u, 1024u);
            for (int i = 0; i < n; ++i) {
                const int u = start + i, s = i % VS;
                if (i > 0) advance(x);
                if (!wait(lay.bar(B_PFULL + (i & 1)), (i >> 1) & 1)) break;
                if (!wait(lay.vfull(s), (i / VS) & 1)) break;
                pf::tc_fence_after();
                if (pf::elect_one()) {
                    const int nk = x.nb * BS / 16;   // the tile's tokens, 16 per K step
                    const uint32_t pb = (uint32_t)(i & 1) * PBUF;
                    for (int kk = 0; kk < nk; ++kk) {
                        // 16 tokens = two 8-row swizzle atoms (2 KB) of V; the two
                        // 64-dim halves are KVHALF apart (leading byte offset)
                        const uint64_t vd =
                            dv + (uint64_t)(((uint32_t)s * KVTILE + (uint32_t)kk * 2048u) >> 4);
                        const uint32_t po = (pb + (uint32_t)(kk >> 2) * PHALF + (uint32_t)(kk & 3) * 32u) >> 4;
                        const uint32_t acc = (first_of(u, x) && kk == 0) ? 0u : 1u;
                        pf::mma_ss(tm + COL_O, vd, dp + po, id_pv, acc);
                    }
                    pf::mma_commit(sbase + lay.vempty(s));
                    pf::mma_commit(sbase + lay.bar(B_PVDONE + (i & 1)));
                }
                __syncwarp();
            }
        }
        // Drain (full limit, after an abort too): every MMA this warp issued
        // has completed before TMEM is freed.
        if (pf::elect_one()) pf::mma_commit(sbase + lay.bar(B_DRAIN + xw));
        __syncwarp();
        if (!__all_sync(FULL, dec::mbar_wait(sbase + lay.bar(B_DRAIN + xw), 0, kWaitLimitNs)))
            atomicOr(p.err, KV_DEVERR_TIMEOUT);
    } else if (warp < NSOFT) {
        // ----------------------------------------------- softmax, epilogue --
        const int t = tid;                        // token of a tile / dim of O^T
        const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
        float* red = reinterpret_cast<float*>(smem + lay.red);   // [2][NR][NSOFT] maxima, [NR][NSOFT] sums
        float m[NR], l[NR];
        bool ok = true;
        int pi = -1;
        Unit x = unit(start);
        for (int u = start; u < end; ++u) {
            const int i = u - start;
            if (i > 0) advance(x);
            const int ntok = x.nb * BS;
            const bool first = first_of(u, x), last = last_of(u, x);
            if (first) {
                ++pi;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    m[r] = -CUDART_INF_F;
                    l[r] = 0.f;
                }
            }
            // -- the tile's scores (this thread: token t, all 16 rows) -------
            float sv[NR];
            ok = ok && warp_wait(sbase + lay.bar(B_SFULL + (i & 1)), (i >> 1) & 1, abort_flag, p.err,
                                 p.wait_ns, lane);
            if (ok) {
                uint32_t raw[NR];
                pf::tc_fence_after();
                tmem_ld16(trow + COL_S + 16u * (uint32_t)(i & 1), raw);
                pf::tmem_wait_ld();
                pf::tc_fence_before();
                __syncwarp();
                if (lane == 0) dec::mbar_arrive(sbase + lay.bar(B_SFREE + (i & 1)));
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    sv[r] = t < ntok ? __uint_as_float(raw[r]) * p.qscale : -CUDART_INF_F;
                float mx[NR];
#pragma unroll
                for (int r = 0; r < NR; ++r) mx[r] = sv[r];
                warp_rows<true>(mx, lane);
                if ((lane & 1) == 0) red[((i & 1) * NR + row_of(lane)) * NSOFT + warp] = mx[0];
            }
            if (soft_sync_any(!ok)) {
                ok = false;
                break;
            }
            // -- lazy running maximum, P = hi + lo -----------------------------
            bool grow = false;
            float alpha[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float4 w4 = *reinterpret_cast<const float4*>(red + ((i & 1) * NR + r) * NSOFT);
                const float tmax = fmaxf(fmaxf(w4.x, w4.y), fmaxf(w4.z, w4.w));
                alpha[r] = 1.f;
                if (tmax > m[r] + kRescaleLog2) {
                    alpha[r] = dec::fast_exp2(m[r] - tmax);      // 0 while m is -inf
                    m[r] = tmax;
                    grow = true;
                }
            }
            uint32_t ph[NR / 2], pl[NR / 2];
#pragma unroll
            for (int r = 0; r < NR; r += 2) {
                float pp[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float mu = m[r + e] == -CUDART_INF_F ? 0.f : m[r + e];
                    pp[e] = dec::fast_exp2(sv[r + e] - mu);
                    l[r + e] = l[r + e] * alpha[r + e] + pp[e];
                }
                pf::H16<T>::split(pp[0], pp[1], ph[r / 2], pl[r / 2]);
            }
            // -- P^T buffer i % 2 free (O^T of unit i - 2 done); a rescale also
            // needs O^T current (unit i - 1 done) ---------------------------
            if (i >= 2)
                ok = ok && warp_wait(sbase + lay.bar(B_PVDONE + (i & 1)), ((i >> 1) - 1) & 1,
                                     abort_flag, p.err, p.wait_ns, lane);
            if (grow && !first)
                ok = ok && warp_wait(sbase + lay.bar(B_PVDONE + ((i - 1) & 1)), ((i - 1) >> 1) & 1,
                                     abort_flag, p.err, p.wait_ns, lane);
            if (ok) {
                pf::tc_fence_after();
                if (grow && !first) {
                    uint32_t ov[2 * NR];
                    pf::tmem_ld32(trow + COL_O, ov);
                    pf::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 2 * NR; ++c)
                        ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha[c % NR]);
                    pf::tmem_st32(trow + COL_O, ov);
                    pf::tmem_wait_st();
                }
                // P^T rows r (hi) and 16 + r (lo), token t: 64-token half t / 64,
                // 128-byte row, swizzled 16-byte chunk
                const uint32_t base = (uint32_t)(i & 1) * PBUF + (uint32_t)(t >> 6) * PHALF +
                                      (uint32_t)(t & 7) * 2u;
                const int ck = (t & 63) >> 3;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const uint32_t off = base + (uint32_t)r * 128u + (uint32_t)((ck ^ (r & 7)) << 4);
                    const uint32_t hv = (r & 1) ? (ph[r / 2] >> 16) : (ph[r / 2] & 0xffffu);
                    const uint32_t lv = (r & 1) ? (pl[r / 2] >> 16) : (pl[r / 2] & 0xffffu);
                    *reinterpret_cast<unsigned short*>(smem + lay.p + off) = (unsigned short)hv;
                    *reinterpret_cast<unsigned short*>(smem + lay.p + off + NR * 128u) =
                        (unsigned short)lv;
                }
                dec::fence_proxy_async();
                pf::tc_fence_before();
                __syncwarp();
                if (lane == 0) dec::mbar_arrive(sbase + lay.bar(B_PFULL + (i & 1)));
            }
            if (!last) continue;
            // -- piece end: O^T / l -> prefix states or the CTA's partial slot --
            ok = ok && warp_wait(sbase + lay.bar(B_PVDONE + (i & 1)), (i >> 1) & 1, abort_flag, p.err,
                                 p.wait_ns, lane);
            float ls[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) ls[r] = l[r];
            warp_rows<false>(ls, lane);
            if ((lane & 1) == 0) red[(2 * NR + row_of(lane)) * NSOFT + warp] = ls[0];
            if (soft_sync_any(!ok)) {
                ok = false;
                break;
            }
            uint32_t ov[2 * NR];
            pf::tc_fence_after();
            pf::tmem_ld32(trow + COL_O, ov);
            pf::tmem_wait_ld();
            pf::tc_fence_before();
            const int m0 = gfirst[x.k] + x.sub * MS;
            const int msz = min(MS, gsize[x.k] - x.sub * MS);
            const int rows = msz * G;
            const bool complete = x.seg >= start && x.seg + x.tiles <= end;
            // slot 0 holds the CTA's first piece, slot 1 its last
            const size_t ps = (size_t)blockIdx.x * 2 + (max(x.seg, start) == start ? 0 : 1);
            float* slot_o = p.part_o + ps * NR * D;
            float* slot_lse = p.part_lse + ps * NR;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float4 w4 = *reinterpret_cast<const float4*>(red + (2 * NR + r) * NSOFT);
                const float L = (w4.x + w4.y) + (w4.z + w4.w);
                if (r >= rows) continue;
                const float inv = L > 0.f ? 1.f / L : 0.f;
                const size_t prow = (size_t)(m0 + r / G) * p.num_q_heads + x.g * G + r % G;
                float* dst = complete ? p.pst_o + prow * D : slot_o + r * D;
                dst[t] = (__uint_as_float(ov[r]) + __uint_as_float(ov[NR + r])) * inv;
                if (t == r) {
                    const float lse = L > 0.f ? m[r] + dec::fast_log2(L) : -CUDART_INF_F;
                    if (complete) p.pst_lse[prow] = lse; else slot_lse[r] = lse;
                }
            }
            if (!complete) {
                // the CTA whose piece completes the segment's count merges; all
                // softmax warps take a share of the element passes
                __threadfence();
                dec::named_sync(2);
                const int c0 = x.seg / chunk, c1 = (x.seg + x.tiles - 1) / chunk;
                int lastp = 0;
                if (warp == 0 && lane == 0)
                    lastp = dec::count_piece(p.counters + 2 * ((size_t)m0 * H + x.g), p.tag,
                                             c1 - c0 + 1);
                if (soft_sync_any(lastp != 0)) {
                    __threadfence();
                    dec::merge_prefix_partials<D, G, 4>(p, x.seg, chunk, c0, c1, rows, m0, x.g, lane,
                                                        warp, NSOFT);
                }
            }
        }
    }

    // -- teardown: free TMEM once every role is done with it ------------------
    pf::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        pf::tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// -- host side ----------------------------------------------------------------
template <typename T, int G, int BS>
cudaError_t prefix_tc_attrs(size_t smem, int* occ) {
    auto k = paged_decode_prefix_tc<T, G, BS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, NTHREADS, smem);
}

// Launched with programmatic stream serialisation (the kernel waits on its
// predecessor with griddepcontrol before it reads anything).
template <typename T, int G, int BS>
cudaError_t prefix_tc_launch(const CUtensorMap& mk, const CUtensorMap& mv, const PParams& p,
                             size_t smem, int grid, cudaStream_t stream) {
    auto k = paged_decode_prefix_tc<T, G, BS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, mk, mv, p);
}

// Instances by (type, group, block size).
template <class F>
cudaError_t by_tc_shape(const kv_pool& pool, int group, F&& f) {
    const int bs = pool.block_size;
#define PKV_T(TT, GG, BB) \
    if (group == GG && bs == BB) return f.template operator()<TT, GG, BB>();
    if (pool.dtype == KV_BF16) {
        PKV_T(__nv_bfloat16, 1, 16) PKV_T(__nv_bfloat16, 2, 16) PKV_T(__nv_bfloat16, 4, 16)
        PKV_T(__nv_bfloat16, 8, 16) PKV_T(__nv_bfloat16, 1, 32) PKV_T(__nv_bfloat16, 2, 32)
        PKV_T(__nv_bfloat16, 4, 32) PKV_T(__nv_bfloat16, 8, 32)
    } else {
        PKV_T(__half, 1, 16) PKV_T(__half, 2, 16) PKV_T(__half, 4, 16) PKV_T(__half, 8, 16)
        PKV_T(__half, 1, 32) PKV_T(__half, 2, 32) PKV_T(__half, 4, 32) PKV_T(__half, 8, 32)
    }
#undef PKV_T
    return cudaErrorNotSupported;
}

}  // namespace ptc
}  // namespace pagedkv
