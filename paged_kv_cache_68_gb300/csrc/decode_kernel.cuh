// PagedAttention decode for sm_103a: a persistent, token-balanced split kernel
// fed by TMA, and a log-sum-exp combine kernel.
//
// What is computed ("Lecture 3", semidirectx.com CS349D notes, sec. 3.2; S06
// "Implementation", llminference.xinbetween.com): for each sequence b and
// query head h, softmax(scale * q K^T) V over the sequence's L tokens, K and V
// read through the block table inside the kernel.  Block-wise partial
// softmaxes are merged with a running maximum and sum ("Lecture 24",
// semidirectx.com CMU 11-868 notes, sec. 3.2 -- the FlashAttention /
// Flash-Decoding trick); partial results of one sequence computed on
// different CTAs are merged by log-sum-exp in the combine kernel.
//
// Work decomposition.  A unit is one (sequence b, KV head g, logical block j).
// Units are ordered b-major, then g, then j, and the U units are cut into
// equal contiguous ranges, one per CTA of a persistent grid (#SMs x resident
// CTAs), so every CTA streams the same number of KV blocks whatever the
// length mix.  Every CTA derives the cut itself from seq_lens (a prefix sum in
// shared memory): no host synchronisation, no atomics, no extra launch.  The
// run of units of one (b, g) inside a CTA is a "piece".  A piece that is a
// whole (b, g) is finished in the CTA and written to `out`; a piece cut by a
// range boundary is written as a partial (normalised o, log2-sum-exp) to one
// of two workspace slots of its CTA -- slot 0 for the CTA's first piece, slot
// 1 for its last -- and the combine kernel merges those.
//
// One CTA = 1 producer warp + NCW consumer warps.  The producer walks the
// CTA's units, looks each block id up in the block table, and issues two TMA
// tile loads per unit (the K and V rows of that block for KV head g: a
// [block_size, head_dim] box of the pool viewed as [N*bs, Hkv, D]) into a ring
// of S shared-memory stages guarded by full/empty mbarriers.  Consumer warp w
// takes units w, w+NCW, ... of each piece (one warp per KV block), so the K/V
// of a block is loaded once for the whole GQA group of G query heads.
//   QK: TPT lanes per token, each holding D/TPT dims of all G (pre-scaled)
//       query rows in registers; the G partial dot products are reduced across
//       the TPT lanes with a transposing shuffle reduction.
//   softmax: per block, per head, fp32, base 2 (q carries scale*log2 e).
//   PV: each lane owns 4 dims of the G output rows; p is broadcast from
//       shared memory.  Rows past the sequence end are never touched.
// At the end of a piece the NCW warps' (m, l, o) are merged through shared
// memory (double-buffered, one named barrier per piece).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "pagedkv_internal.cuh"

namespace pagedkv {
namespace dec {

constexpr int NCW = 4;                       // consumer warps per CTA
constexpr int NTHREADS = (NCW + 1) * 32;     // + one producer warp
constexpr unsigned FULL = 0xffffffffu;
constexpr int kMinChunk = 8;                 // fewest units a CTA is given

struct Params {
    const void* q;
    void* out;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    int* err;
    int* ws_prefix;        // [batch + 1]: blocks-per-sequence prefix (CTA 0 writes)
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
};

// ---------------------------------------------------------------- layout ---
struct Layout {
    uint32_t full, empty, valid, misc, prefix, lens, sbuf, abuf, merge_o, merge_ml, ring;
    uint32_t stage_bytes, total;
    __host__ __device__ Layout(int S, int B, int bs, int G, int D, int elt) {
        uint32_t off = 0;
        full = off;   off += 8u * S;
        empty = off;  off += 8u * S;
        valid = off;  off += 4u * S;
        misc = off;   off += 4u * 40;            // abort flag + warp totals
        prefix = off; off += 4u * (B + 1);
        lens = off;   off += 4u * B;
        off = (off + 15u) & ~15u;
        sbuf = off;   off += 4u * NCW * bs * G;
        abuf = off;   off += 4u * NCW * G;
        off = (off + 15u) & ~15u;
        merge_o = off;  off += 2u * 4u * NCW * G * D;
        merge_ml = off; off += 2u * 2u * 4u * NCW * G;
        off = (off + 1023u) & ~1023u;
        ring = off;
        stage_bytes = 2u * bs * D * elt;         // K tile then V tile, 128-byte multiples
        off += stage_bytes * S;
        total = off;
    }
};

// ------------------------------------------------------------- PTX helpers --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with `parity` to complete; give up after
// kWaitLimitNs and return false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
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
__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
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

// ------------------------------------------------------------ split kernel --
template <typename T, int D, int G>
__global__ void __launch_bounds__(NTHREADS) paged_decode_split(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const Params p) {
    using C = Cfg<T, D, G>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int B = p.batch, bs = p.bs, S = p.stages, H = p.num_kv_heads;
    const Layout lay(S, B, bs, G, D, C::ELT);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + lay.empty);
    volatile int* valid = reinterpret_cast<volatile int*>(smem + lay.valid);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc);
    int* warp_tot = reinterpret_cast<int*>(smem + lay.misc) + 8;
    int* prefix = reinterpret_cast<int*>(smem + lay.prefix);
    int* lens = reinterpret_cast<int*>(smem + lay.lens);
    unsigned char* ring = smem + lay.ring;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // -- 1. clamped lengths and the blocks-per-sequence prefix --------------
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {
        const int cap = p.max_blocks * bs;
        const int per = (B + NTHREADS - 1) / NTHREADS;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        int local = 0;
        bool over = false;
        for (int b = b0; b < b1; ++b) {
            int L = p.seq_lens[b];
            L = L < 0 ? 0 : L;
            if (L > cap) { over = true; L = cap; }
            lens[b] = L;
            local += (L + bs - 1) / bs;
        }
        if (over && blockIdx.x == 0) atomicOr(p.err, KV_DEVERR_SEQ_RANGE);
        int x = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        int woff = 0;
        for (int w = 0; w < warp; ++w) woff += warp_tot[w];
        int run = woff + x - local;
        for (int b = b0; b < b1; ++b) {
            prefix[b] = run;
            run += (lens[b] + bs - 1) / bs;
        }
        if (tid == NTHREADS - 1) prefix[B] = woff + x;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int i = tid; i <= B; i += NTHREADS) p.ws_prefix[i] = prefix[i];

    const int U = prefix[B] * H;
    const int chunk = unit_chunk(U, p.num_ctas);
    const int start = blockIdx.x * chunk;
    const int end = min(U, start + chunk);
    if (start >= end) return;

    if (warp == NCW) {
        // ---------------------------------------------------- producer warp --
        // Lanes look up the block ids of the next 32 units in parallel; lane 0
        // then issues the TMA loads one unit at a time.
        auto fetch = [&](int uu, int& id, int& gg) {
            id = -1;
            gg = 0;
            if (uu < end) {
                const int b = find_seq(prefix, B, uu, H);
                const int nb = prefix[b + 1] - prefix[b];
                const int r = uu - prefix[b] * H;
                gg = r / nb;
                id = __ldg(p.block_tables + (size_t)b * p.max_blocks + (r - gg * nb));
            }
        };
        int id_cur, g_cur, id_nxt, g_nxt;
        fetch(start + lane, id_cur, g_cur);
        int k = 0;
        for (int base = start; base < end; base += 32) {
            fetch(base + 32 + lane, id_nxt, g_nxt);
            const int n = min(32, end - base);
            for (int i = 0; i < n; ++i, ++k) {
                const int id = __shfl_sync(FULL, id_cur, i);
                const int gg = __shfl_sync(FULL, g_cur, i);
                if (lane == 0) {
                    const int s = k % S, ph = k / S;
                    bool ok = *abort_flag == 0;
                    if (ok && ph > 0 && !mbar_wait(smem_u32(&empty[s]), (ph - 1) & 1)) {
                        *abort_flag = 1;
                        atomicOr(p.err, KV_DEVERR_TIMEOUT);
                        ok = false;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    if (ok && id >= 0 && id < p.num_blocks) {
                        valid[s] = 1;
                        mbar_arrive_tx(fb, lay.stage_bytes);
                        const uint32_t dst = smem_u32(ring + (size_t)s * lay.stage_bytes);
                        tma_load_3d(dst, &tmap_k, 0, gg, id * bs, fb);
                        tma_load_3d(dst + lay.stage_bytes / 2, &tmap_v, 0, gg, id * bs, fb);
                    } else {
                        valid[s] = 0;
                        if (ok) atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                        mbar_arrive(fb);
                    }
                }
            }
            __syncwarp();
            id_cur = id_nxt;
            g_cur = g_nxt;
        }
        // Drain: no copy may still be landing in shared memory at exit.
        if (lane == 0)
            for (int kk = max(0, k - S); kk < k; ++kk)
                if (!mbar_wait(smem_u32(&full[kk % S]), (kk / S) & 1))
                    atomicOr(p.err, KV_DEVERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int w = warp;
    const int tg = lane / C::TPT, jl = lane % C::TPT;
    const int hsel = (jl >> C::HSHIFT) & (G - 1);
    const bool leader = (jl & ((1 << C::HSHIFT) - 1)) == 0;
    const int hh = lane % G;                       // head this lane tracks in softmax
    const int tv = lane / C::LPV, dl = lane % C::LPV;
    float* sb = reinterpret_cast<float*>(smem + lay.sbuf) + w * bs * G;   // [bs][G]
    float* ab = reinterpret_cast<float*>(smem + lay.abuf) + w * G;
    const T* qbase = static_cast<const T*>(p.q);
    T* obase = static_cast<T*>(p.out);

    int sel = 0;
    for (int u = start; u < end;) {
        const int b = find_seq(prefix, B, u, H);
        const int nb = prefix[b + 1] - prefix[b];
        const int r = u - prefix[b] * H;
        const int g = r / nb;
        const int j0 = r - g * nb;
        const int seg_start = prefix[b] * H + g * nb;
        const int piece_end = min(end, seg_start + nb);
        const int Lb = lens[b];

        // query rows of the group, scaled by scale * log2(e), in registers
        float qf[G][C::QE];
        {
            const T* qp = qbase + ((size_t)b * p.num_q_heads + (size_t)g * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int i = 0; i < C::NCH; ++i) {
                    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
                        qp + (size_t)h * D + (jl + C::TPT * i) * C::VE));
                    float f[C::VE];
                    Elt<T>::chunk(raw, f);
#pragma unroll
                    for (int e = 0; e < C::VE; ++e) qf[h][i * C::VE + e] = f[e] * p.qscale;
                }
        }
        float m_run = -CUDART_INF_F, l_run = 0.f;
        float o[G][4];
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[h][e] = 0.f;

        for (int uu = u + w; uu < piece_end; uu += NCW) {
            const int k = uu - start, s = k % S;
            bool ok = *abort_flag == 0;
            if (ok && !mbar_wait(smem_u32(&full[s]), (k / S) & 1)) {
                *abort_flag = 1;
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(FULL, ok);
            if (ok && valid[s]) {
                const int j = j0 + (uu - u);
                const int n_valid = min(bs, Lb - j * bs);
                const unsigned char* Ks = ring + (size_t)s * lay.stage_bytes;
                const unsigned char* Vs = Ks + lay.stage_bytes / 2;
                // -- scores --------------------------------------------------
                for (int t0 = 0; t0 < bs; t0 += C::TPS) {
                    const int t = t0 + tg;
                    float acc[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h] = 0.f;
                    if (t < n_valid) {
#pragma unroll
                        for (int i = 0; i < C::NCH; ++i) {
                            const uint4 raw = *reinterpret_cast<const uint4*>(
                                Ks + ((size_t)t * C::CHUNKS + jl + C::TPT * i) * 16);
                            float kf[C::VE];
                            Elt<T>::chunk(raw, kf);
#pragma unroll
                            for (int h = 0; h < G; ++h)
#pragma unroll
                                for (int e = 0; e < C::VE; ++e)
                                    acc[h] = fmaf(qf[h][i * C::VE + e], kf[e], acc[h]);
                        }
                    }
                    TReduce<G, C::TPT / 2>::run(acc, lane);
                    if (leader && t < bs) sb[t * G + hsel] = (t < n_valid) ? acc[0] : -CUDART_INF_F;
                }
                __syncwarp();
                // -- online softmax, per head -----------------------------------
                float mloc = -CUDART_INF_F;
                for (int t = lane / G; t < bs; t += 32 / G) mloc = fmaxf(mloc, sb[t * G + hh]);
#pragma unroll
                for (int off = 16; off >= G; off >>= 1)
                    mloc = fmaxf(mloc, __shfl_xor_sync(FULL, mloc, off));
                const float m_new = fmaxf(m_run, mloc);
                float alpha = 1.f, lsum = 0.f;
                if (m_new != -CUDART_INF_F) {
                    alpha = fast_exp2(m_run - m_new);
                    for (int t = lane / G; t < bs; t += 32 / G) {
                        const float pe = fast_exp2(sb[t * G + hh] - m_new);
                        sb[t * G + hh] = pe;
                        lsum += pe;
                    }
                } else {
                    for (int t = lane / G; t < bs; t += 32 / G) sb[t * G + hh] = 0.f;
                }
#pragma unroll
                for (int off = 16; off >= G; off >>= 1) lsum += __shfl_xor_sync(FULL, lsum, off);
                l_run = l_run * alpha + lsum;
                m_run = m_new;
                if (lane < G) ab[lane] = alpha;
                __syncwarp();
                // -- weighted sum of V -------------------------------------------
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float a = ab[h];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[h][e] *= a;
                }
                for (int t = tv; t < n_valid; t += C::TPSV) {
                    float vf[4];
                    Elt<T>::four(Vs + ((size_t)t * D + dl * 4) * C::ELT, vf);
                    float pr[G];
#pragma unroll
                    for (int h = 0; h < G; ++h) pr[h] = sb[t * G + h];
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[h][e] = fmaf(pr[h], vf[e], o[h][e]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        // -- merge the NCW warps' partial softmaxes of this piece -------------
        float* mo = reinterpret_cast<float*>(smem + lay.merge_o) + sel * NCW * G * D;
        float* mm = reinterpret_cast<float*>(smem + lay.merge_ml) + sel * 2 * NCW * G;
#pragma unroll
        for (int off = C::LPV; off < 32; off <<= 1)
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[h][e] += __shfl_xor_sync(FULL, o[h][e], off);
        if (lane < C::LPV) {
#pragma unroll
            for (int h = 0; h < G; ++h)
                *reinterpret_cast<float4*>(mo + (w * G + h) * D + dl * 4) =
                    make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
        }
        if (lane < G) {
            mm[w * G + lane] = m_run;
            mm[NCW * G + w * G + lane] = l_run;
        }
        consumer_barrier();
        const bool complete = seg_start >= start && seg_start + nb <= end;
        const int slot = (u == start) ? 0 : 1;
        for (int idx = tid; idx < G * D; idx += NCW * 32) {
            const int h = idx / D, d = idx % D;
            float M = -CUDART_INF_F;
#pragma unroll
            for (int w2 = 0; w2 < NCW; ++w2) M = fmaxf(M, mm[w2 * G + h]);
            float den = 0.f, num = 0.f;
            if (M != -CUDART_INF_F) {
#pragma unroll
                for (int w2 = 0; w2 < NCW; ++w2) {
                    const float sc = fast_exp2(mm[w2 * G + h] - M);
                    den += sc * mm[NCW * G + w2 * G + h];
                    num += sc * mo[(w2 * G + h) * D + d];
                }
            }
            const float val = den > 0.f ? num / den : 0.f;
            if (complete) {
                obase[((size_t)b * p.num_q_heads + (size_t)g * G + h) * D + d] = Elt<T>::store(val);
            } else {
                const size_t ps = (size_t)blockIdx.x * 2 + slot;
                p.part_o[(ps * G + h) * D + d] = val;
                if (d == 0) p.part_lse[ps * G + h] = den > 0.f ? M + fast_log2(den) : -CUDART_INF_F;
            }
        }
        sel ^= 1;
        u = piece_end;
    }
}

// ---------------------------------------------------------- combine kernel --
// One CTA per (sequence, KV head): merge the partials of a (b, g) that was cut
// across CTAs (weights 2^(lse_p - max)), write zeros for empty sequences, and
// leave whole pieces (already written by the split kernel) alone.
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) paged_decode_combine(const Params p) {
    const int H = p.num_kv_heads;
    const int b = blockIdx.x / H, g = blockIdx.x % H;
    const int* prefix = p.ws_prefix;
    const int nb = prefix[b + 1] - prefix[b];
    T* o = static_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)g * G) * D;
    if (nb == 0) {
        for (int idx = threadIdx.x; idx < G * D; idx += 128) o[idx] = Elt<T>::store(0.f);
        return;
    }
    const int U = prefix[p.batch] * H;
    const int chunk = unit_chunk(U, p.num_ctas);
    const int S0 = prefix[b] * H + g * nb;
    const int c0 = S0 / chunk, c1 = (S0 + nb - 1) / chunk;
    if (c0 == c1) return;
    const int slot0 = (S0 == c0 * chunk) ? 0 : 1;
    for (int idx = threadIdx.x; idx < G * D; idx += 128) {
        const int h = idx / D, d = idx % D;
        float M = -CUDART_INF_F;
        for (int c = c0; c <= c1; ++c) {
            const size_t ps = (size_t)c * 2 + (c == c0 ? slot0 : 0);
            M = fmaxf(M, p.part_lse[ps * G + h]);
        }
        float den = 0.f, num = 0.f;
        if (M != -CUDART_INF_F) {
            for (int c = c0; c <= c1; ++c) {
                const size_t ps = (size_t)c * 2 + (c == c0 ? slot0 : 0);
                const float wgt = fast_exp2(p.part_lse[ps * G + h] - M);
                den += wgt;
                num += wgt * p.part_o[(ps * G + h) * D + d];
            }
        }
        o[idx] = Elt<T>::store(den > 0.f ? num / den : 0.f);
    }
}

// ------------------------------------------------------------- host side --
template <typename T, int D, int G>
cudaError_t launch_typed(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                         cudaStream_t stream) {
    auto split = paged_decode_split<T, D, G>;
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
    p.ws_prefix = reinterpret_cast<int*>(ws + plan.ws_prefix_off);
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
    split<<<plan.num_ctas, NTHREADS, plan.smem_bytes, stream>>>(pool.tmap_k, pool.tmap_v, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    paged_decode_combine<T, D, G><<<call.batch * pool.num_kv_heads, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T, int D, int G>
cudaError_t attrs_typed(size_t smem, int* ctas_per_sm) {
    auto split = paged_decode_split<T, D, G>;
    cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, split, NTHREADS, smem);
}

template <typename T>
cudaError_t dispatch(const kv_pool& pool, const DecodeCall& call, const DecodePlan& plan,
                     cudaStream_t stream) {
#define PKV_CASE(DD, GG) \
    if (pool.head_dim == DD && plan.group == GG) return launch_typed<T, DD, GG>(pool, call, plan, stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t attrs(int head_dim, int group, size_t smem, int* ctas_per_sm) {
#define PKV_CASE(DD, GG) \
    if (head_dim == DD && group == GG) return attrs_typed<T, DD, GG>(smem, ctas_per_sm);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
    return cudaErrorNotSupported;
}

}  // namespace dec
}  // namespace pagedkv
