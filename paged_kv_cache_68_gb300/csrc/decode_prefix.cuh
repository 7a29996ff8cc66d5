// Cascade (shared-prefix) decode, first pass: attention of many sequences'
// queries over the KV blocks their tables share.
//
// Parallel samples or beams forked from one prompt point their block tables
// at the same physical prefix blocks ("Lecture 3", semidirectx.com CS349D
// notes, sec. 4.1; "Lecture 24", semidirectx.com CMU 11-868 notes, sec. 4.1).
// Plain decode reads such a block once per sequence.  This pass reads it once
// for a whole group: a unit is (group k, sub-group s, KV head g, prefix block
// j), and the block's K/V tile is multiplied against the query rows of every
// member of the sub-group at once -- up to 16 rows (members x G heads) on the
// two N tiles of mma.sync m16n8k16.  For each member sequence b and head h the
// pass leaves a normalised partial output and its log2-sum-exp ("prefix
// state"); the second pass (the plain split kernel over each sequence's
// remaining blocks) folds it into the final log-sum-exp merge, the same trick
// the pages credit to Flash-Decoding ("Lecture 24", sec. 3.2) and that the S06
// page names for vLLM's cascade path (llminference.xinbetween.com, "In
// production").  The result equals plain decode up to fp32 rounding.
//
// The frame is the split kernel's: a persistent grid cut into equal unit
// ranges, one TMA producer warp feeding a ring of 128-byte-swizzled tiles,
// four consumer warps (unit k to stage k % S and warp k % 4), a per-piece warp
// merge, and tagged piece counters so the CTA that finishes the last piece
// of a (group, sub-group, head) segment merges the pieces cut across CTAs.
#pragma once

#include "decode_kernel.cuh"

namespace pagedkv {
namespace dec {

constexpr int kRows = 16;   // query rows per segment: (members of a sub-group) x G

struct PParams {
    const void* q;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    const int32_t* g_first;        // [num_groups] first member (sequence index)
    const int32_t* g_size;         // [num_groups] members
    const int32_t* g_blocks;       // [num_groups] leading blocks shared by all members
    int* err;
    float* pst_o;                  // out [batch][num_q_heads][D], members of used groups
    float* pst_lse;                // out [batch][num_q_heads]
    unsigned long long* counters;  // [batch][num_kv_heads][2], by a sub-group's first
                                   // member: {tag, pieces done}
    unsigned long long tag;        // this call's random counter tag
    float* part_o;                 // [num_ctas][2][kRows][D]
    float* part_lse;               // [num_ctas][2][kRows]
    int num_groups;
    int max_blocks;
    int batch;
    int num_q_heads;
    int num_kv_heads;
    int num_blocks;
    int bs;
    int stages;
    int num_ctas;
    float qscale;
    unsigned long long wait_ns;    // limit of one pipeline wait (the pool's setting)
};

struct PLayout {
    uint32_t full, empty, valid, misc, gcum, vg, merge_o, merge_ml, ring;
    uint32_t stage_bytes, total;
    __host__ __device__ PLayout(int S, int K, int bs, int D, int elt) {
        uint32_t off = 0;
        full = off;   off += 8u * S;
        empty = off;  off += 8u * S;
        valid = off;  off += 4u * S;
        misc = off;   off += 4u * 40;
        gcum = off;   off += 4u * (K + 1);
        vg = off;     off += 4u * 3u * K;            // used groups: first, size, blocks
        off = (off + 15u) & ~15u;
        merge_o = off;  off += 4u * (NCW - 1) * kRows * D;
        merge_ml = off; off += 2u * 4u * (NCW - 1) * kRows;
        off = (off + 1023u) & ~1023u;
        ring = off;
        stage_bytes = 2u * bs * D * elt;
        off += stage_bytes * S;
        total = off;
    }
};

// Largest i in [0, n) with a[i] <= u (a[0] = 0 <= u, a non-decreasing).
__device__ __forceinline__ int find_le(const int* a, int n, int u) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= u) lo = mid; else hi = mid;
    }
    return lo;
}

// Tensor-core policy over up to 16 rows.  Lane roles as in TcPolicy: gid =
// lane / 4, tig = lane % 4; on N tile nt the lane holds columns (rows of the
// output) nt*8 + 2 tig + {0, 1}; column c is member c / G, head c % G.
template <typename T, int D, int G, int BSC>
struct TcRows {
    static_assert(sizeof(T) == 2 && BSC % 16 == 0 && (G == 1 || G == 2 || G == 4 || G == 8),
                  "tensor-core shapes");
    static constexpr int NT = kRows / 8;
    static constexpr int KS = D / 16;
    static constexpr int MT = D / 16;
    static constexpr int TT = BSC / 16;

    uint32_t qb[KS][NT][2];
    float oacc[MT][NT][4];
    float m_run[NT][2], l_run[NT][2];
    int lc[NT][2];                      // context length of the column's member (0: padding)

    __device__ static __forceinline__ uint32_t swz(uint32_t tile, int r, int c) {
        return tile + (uint32_t)((c >> 3) * BSC * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    }

    // members m0 .. m0 + msz - 1, KV head g
    __device__ __forceinline__ void begin(const T* q, int m0, int msz, int g, int hq,
                                          const int32_t* seq_lens, int cap, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = nt * 8 + gid, m = row / G, h = row % G;
            const T* qr = q + ((size_t)(m0 + m) * hq + g * G + h) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    qb[ks][nt][j] =
                        m < msz ? __ldg(reinterpret_cast<const uint32_t*>(qr + ks * 16 + j * 8 + tig * 2))
                                : 0u;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = nt * 8 + 2 * tig + j, mc = c / G;
                lc[nt][j] = mc < msz ? min(max(seq_lens[m0 + mc], 0), cap) : 0;
                m_run[nt][j] = -CUDART_INF_F;
                l_run[nt][j] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
        }
    }

    __device__ __forceinline__ void block(const unsigned char* Ks, const unsigned char* Vs,
                                          int jblk, float qscale, int lane) {
        const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, r8 = lane & 7;
        const uint32_t kbase = smem_u32(Ks), vbase = smem_u32(Vs);
        int nv[NT][2], nvmax = 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                nv[nt][j] = min(BSC, lc[nt][j] - jblk * BSC);
                nvmax = max(nvmax, nv[nt][j]);
            }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) nvmax = max(nvmax, __shfl_xor_sync(FULL, nvmax, off));
        if (nvmax < BSC) {
            // rows no member reaches: P is 0 there, but 0 * NaN would poison the MMA
            unsigned char* V = const_cast<unsigned char*>(Vs);
            const int from = max(nvmax, 0);
            const int nbytes = (BSC - from) * 128;
            for (int i = lane * 16; i < nbytes; i += 32 * 16)
#pragma unroll
                for (int hf = 0; hf < D / 64; ++hf)
                    *reinterpret_cast<uint4*>(V + hf * BSC * 128 + from * 128 + i) =
                        make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async();
            __syncwarp();
        }
        // -- S^T = K_blk Q^T over both N tiles --------------------------------
        float s[TT][NT][4];
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            // even and odd k-steps accumulate apart: two independent MMA chains
            float acc[2][NT][4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    acc[h2][nt][0] = acc[h2][nt][1] = acc[h2][nt][2] = acc[h2][nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(a, swz(kbase, tt * 16 + (mi & 1) * 8 + r8, ks * 2 + (mi >> 1)));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    Mma<T>::run(acc[ks & 1][nt], a, qb[ks][nt][0], qb[ks][nt][1]);
            }
            const int t0 = tt * 16 + gid, t1 = t0 + 8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                s[tt][nt][0] = t0 < nv[nt][0] ? (acc[0][nt][0] + acc[1][nt][0]) * qscale : -CUDART_INF_F;
                s[tt][nt][1] = t0 < nv[nt][1] ? (acc[0][nt][1] + acc[1][nt][1]) * qscale : -CUDART_INF_F;
                s[tt][nt][2] = t1 < nv[nt][0] ? (acc[0][nt][2] + acc[1][nt][2]) * qscale : -CUDART_INF_F;
                s[tt][nt][3] = t1 < nv[nt][1] ? (acc[0][nt][3] + acc[1][nt][3]) * qscale : -CUDART_INF_F;
            }
        }
        // -- online softmax per column ----------------------------------------
        float alpha[NT][2], mnew[NT][2], lsum[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float mx = -CUDART_INF_F;
#pragma unroll
                for (int tt = 0; tt < TT; ++tt) mx = fmaxf(mx, fmaxf(s[tt][nt][j], s[tt][nt][j + 2]));
                mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
                mnew[nt][j] = fmaxf(m_run[nt][j], mx);
                alpha[nt][j] = mnew[nt][j] == -CUDART_INF_F ? 1.f : fast_exp2(m_run[nt][j] - mnew[nt][j]);
                lsum[nt][j] = 0.f;
            }
#pragma unroll
        for (int tt = 0; tt < TT; ++tt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = e & 1;
                    const float pe = mnew[nt][j] == -CUDART_INF_F ? 0.f : fast_exp2(s[tt][nt][e] - mnew[nt][j]);
                    s[tt][nt][e] = pe;
                    lsum[nt][j] += pe;
                }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                lsum[nt][j] += __shfl_xor_sync(FULL, lsum[nt][j], 4);
                lsum[nt][j] += __shfl_xor_sync(FULL, lsum[nt][j], 8);
                lsum[nt][j] += __shfl_xor_sync(FULL, lsum[nt][j], 16);
                l_run[nt][j] = l_run[nt][j] * alpha[nt][j] + lsum[nt][j];
                m_run[nt][j] = mnew[nt][j];
            }
        // rescale the accumulators only when some running maximum moved
        bool same = true;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) same = same && alpha[nt][0] == 1.f && alpha[nt][1] == 1.f;
        if (!__all_sync(FULL, same))
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float2 a2 = make_float2(alpha[nt][0], alpha[nt][1]);
                const float2 lo = __fmul2_rn(make_float2(oacc[mt][nt][0], oacc[mt][nt][1]), a2);
                const float2 hi = __fmul2_rn(make_float2(oacc[mt][nt][2], oacc[mt][nt][3]), a2);
                oacc[mt][nt][0] = lo.x; oacc[mt][nt][1] = lo.y;
                oacc[mt][nt][2] = hi.x; oacc[mt][nt][3] = hi.y;
            }
        // -- O^T += V_blk^T P^T, P as hi + lo halves ---------------------------
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float* sv = s[tt][nt];
                const uint32_t h01 = Mma<T>::pack(sv[0], sv[1]), h23 = Mma<T>::pack(sv[2], sv[3]);
                const float2 f01 = Mma<T>::unpack(h01), f23 = Mma<T>::unpack(h23);
                const uint32_t l01 = Mma<T>::pack(sv[0] - f01.x, sv[1] - f01.y);
                const uint32_t l23 = Mma<T>::pack(sv[2] - f23.x, sv[3] - f23.y);
                bh[nt][0] = movm_t(h01); bh[nt][1] = movm_t(h23);
                bl[nt][0] = movm_t(l01); bl[nt][1] = movm_t(l23);
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                ldsm_x4_t(a, swz(vbase, tt * 16 + (mi >> 1) * 8 + r8, mt * 2 + (mi & 1)));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    Mma<T>::run(oacc[mt][nt], a, bh[nt][0], bh[nt][1]);
                    Mma<T>::run(oacc[mt][nt], a, bl[nt][0], bl[nt][1]);
                }
            }
        }
    }

    // merge area: o [NCW-1][kRows][D], m [NCW-1][kRows], l [NCW-1][kRows]
    __device__ __forceinline__ void put(float* mo, float* mm, int w, int rows, int lane) const {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = nt * 8 + 2 * tig + j;
                if (c >= rows) continue;
                float* row = mo + ((w - 1) * kRows + c) * D;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    row[mt * 16 + gid] = oacc[mt][nt][j];
                    row[mt * 16 + gid + 8] = oacc[mt][nt][j + 2];
                }
                if (gid == 0) {
                    mm[(w - 1) * kRows + c] = m_run[nt][j];
                    mm[(NCW - 1) * kRows + (w - 1) * kRows + c] = l_run[nt][j];
                }
            }
    }

    // Warp 0: merge the warps' states; a complete segment goes straight to the
    // prefix states of its members, a cut piece to the CTA's partial slot.
    __device__ __forceinline__ void merge_store(const float* mo, const float* mm, int rows,
                                                bool complete, float* pst_o, float* pst_lse,
                                                int m0, int g, int hq, float* slot_o,
                                                float* slot_lse, int lane) const {
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c = nt * 8 + 2 * tig + j;
                if (c >= rows) continue;
                float M = m_run[nt][j];
#pragma unroll
                for (int w2 = 1; w2 < NCW; ++w2) M = fmaxf(M, mm[(w2 - 1) * kRows + c]);
                float cw[NCW];
                cw[0] = M == -CUDART_INF_F ? 0.f : fast_exp2(m_run[nt][j] - M);
                float den = cw[0] * l_run[nt][j];
#pragma unroll
                for (int w2 = 1; w2 < NCW; ++w2) {
                    cw[w2] = M == -CUDART_INF_F ? 0.f : fast_exp2(mm[(w2 - 1) * kRows + c] - M);
                    den += cw[w2] * mm[(NCW - 1) * kRows + (w2 - 1) * kRows + c];
                }
                const float inv = den > 0.f ? 1.f / den : 0.f;
                const size_t prow = (size_t)(m0 + c / G) * hq + g * G + c % G;
                float* dst = complete ? pst_o + prow * D : slot_o + c * D;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int d = mt * 16 + gid + 8 * hf;
                        float num = cw[0] * oacc[mt][nt][j + 2 * hf];
#pragma unroll
                        for (int w2 = 1; w2 < NCW; ++w2) num += cw[w2] * mo[((w2 - 1) * kRows + c) * D + d];
                        dst[d] = num * inv;
                    }
                if (gid == 0) {
                    const float lse = den > 0.f ? M + fast_log2(den) : -CUDART_INF_F;
                    if (complete) pst_lse[prow] = lse; else slot_lse[c] = lse;
                }
            }
    }
};

// One warp: merge the partials of a cut segment into the prefix states.
template <int D, int G>
__device__ __forceinline__ void merge_prefix_partials(const PParams& p, int seg_start, int chunk,
                                                      int c0, int c1, int rows, int m0, int g,
                                                      int lane) {
    merge_cut<kRows, D>(p.part_o, p.part_lse, c0, c1, seg_start == c0 * chunk ? 0 : 1, nullptr,
                        nullptr, lane, [&](int r, int d0, const float* v, float lse) {
                            if (r >= rows) return;
                            const size_t prow = (size_t)(m0 + r / G) * p.num_q_heads + g * G + r % G;
#pragma unroll
                            for (int k = 0; k < merge_epl<kRows, D>(); ++k)
                                p.pst_o[prow * D + d0 + k] = v[k];
                            if (d0 == 0) p.pst_lse[prow] = lse;
                        });
}

template <typename T, int D, int G, int BSC>
__global__ void __launch_bounds__(NTHREADS, 2) paged_decode_prefix(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const PParams p) {
    using Pol = TcRows<T, D, G, BSC>;
    constexpr int ELT = sizeof(T);
    constexpr int MS = kRows / G;                   // members per sub-group
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_align_1k(smem_raw);
    const int K = p.num_groups, S = p.stages, H = p.num_kv_heads, B = p.batch;
    const PLayout lay(S, K, BSC, D, ELT);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + lay.empty);
    volatile int* valid = reinterpret_cast<volatile int*>(smem + lay.valid);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc);
    int* warp_tot = reinterpret_cast<int*>(smem + lay.misc) + 8;
    int* gcum = reinterpret_cast<int*>(smem + lay.gcum);
    int* vg = reinterpret_cast<int*>(smem + lay.vg);
    const int* gfirst = vg;
    const int* gsize = vg + K;
    const int* gblk = vg + 2 * K;
    unsigned char* ring = smem + lay.ring;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cap = p.max_blocks * BSC;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_launch_dependents();
    pdl_wait();

    // -- used groups, their units (sub-groups x KV heads x shared blocks) ------
    const int NG = load_groups(p.g_first, p.g_size, p.g_blocks, K, p.seq_lens, B, BSC, cap, vg,
                               warp_tot, p.err);
    {
        const int per = (NG + NTHREADS - 1) / NTHREADS;
        const int k0 = min(NG, tid * per), k1 = min(NG, k0 + per);
        int local = 0;
        for (int k = k0; k < k1; ++k) local += ((gsize[k] + MS - 1) / MS) * H * gblk[k];
        int total = 0;
        int run = block_excl_sum(local, warp_tot, &total);
        for (int k = k0; k < k1; ++k) {
            gcum[k] = run;
            run += ((gsize[k] + MS - 1) / MS) * H * gblk[k];
        }
        if (tid == 0) gcum[NG] = total;
    }
    __syncthreads();

    const int U = gcum[NG];
    const int chunk = unit_chunk(U, p.num_ctas);
    const int start = blockIdx.x * chunk;
    const int end = min(U, start + chunk);
    if (start >= end) return;

    if (warp == NCW) {
        // ---------------------------------------------------- producer warp --
        auto fetch = [&](int uu, int& id, int& gg) {
            id = -1;
            gg = 0;
            if (uu < end) {
                const int k = find_le(gcum, NG, uu);
                const int P = gblk[k];
                const int r = uu - gcum[k];
                gg = (r / P) % H;
                id = __ldg(p.block_tables + (size_t)gfirst[k] * p.max_blocks + r % P);
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
                int stop = 0;
                if (lane == 0) {
                    const int s = k % S, ph = k / S;
                    bool ok = *abort_flag == 0;
                    if (ok && ph > 0 &&
                        !mbar_wait_sleep(smem_u32(&empty[s]), (ph - 1) & 1, p.wait_ns)) {
                        *abort_flag = 1;
                        atomicOr(p.err, KV_DEVERR_TIMEOUT);
                        ok = false;
                    }
                    const uint32_t fb = smem_u32(&full[s]);
                    // after an abort no barrier is touched again (a full
                    // stage's last phase may still be waiting for bytes)
                    stop = !ok;
                    if (stop) {
                    } else if (id >= 0 && id < p.num_blocks) {
                        valid[s] = 1;
                        mbar_arrive_tx(fb, lay.stage_bytes);
                        const uint32_t dst = smem_u32(ring + (size_t)s * lay.stage_bytes);
                        // one 4-D copy per block: both 128-byte halves, [half][rows]
                        tma_load_4d(dst, &tmap_k, 0, id * BSC, 0, gg, fb);
                        tma_load_4d(dst + lay.stage_bytes / 2, &tmap_v, 0, id * BSC, 0, gg, fb);
                    } else {
                        valid[s] = 0;
                        atomicOr(p.err, KV_DEVERR_BLOCK_RANGE);
                        mbar_arrive(fb);
                    }
                }
                if (__shfl_sync(FULL, stop, 0)) break;
            }
            __syncwarp();
            if (k < base + n - start) break;      // stopped early (abort)
            id_cur = id_nxt;
            g_cur = g_nxt;
        }
        // Drain (full limit whatever the pool's setting): the issues that
        // reached a barrier are the first k, each stage with at most its last
        // phase outstanding (a stage is refilled only after it was released).
        if (lane == 0)
            for (int kk = max(0, k - S); kk < k; ++kk)
                if (!mbar_wait_sleep(smem_u32(&full[kk % S]), (kk / S) & 1, kWaitLimitNs))
                    atomicOr(p.err, KV_DEVERR_TIMEOUT);
        return;
    }

    // ---------------------------------------------------- consumer warps ----
    const int w = warp;
    float* mo = reinterpret_cast<float*>(smem + lay.merge_o);
    float* mm = reinterpret_cast<float*>(smem + lay.merge_ml);
    const T* qbase = static_cast<const T*>(p.q);
    Pol pol;
    bool first_piece = true;
    for (int u = start; u < end;) {
        const int k = find_le(gcum, NG, u);
        const int P = gblk[k];
        const int r = u - gcum[k];
        const int sg = r / P;                      // sub-group * H + kv head
        const int sub = sg / H, g = sg % H;
        const int j0 = r % P;
        const int seg_start = gcum[k] + sg * P;
        const int piece_end = min(end, seg_start + P);
        const int m0 = gfirst[k] + sub * MS;
        const int msz = min(MS, gsize[k] - sub * MS);
        const int rows = msz * G;

        pol.begin(qbase, m0, msz, g, p.num_q_heads, p.seq_lens, cap, lane);
        const int first = u + ((w - (u - start) % NCW) + NCW) % NCW;
        for (int uu = first; uu < piece_end; uu += NCW) {
            const int kk = uu - start, s = kk % S;
            bool ok = *abort_flag == 0;
            if (ok && !mbar_wait_sleep(smem_u32(&full[s]), (kk / S) & 1, p.wait_ns)) {
                *abort_flag = 1;
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ok = false;
            }
            ok = __all_sync(FULL, ok);
            if (ok && valid[s]) {
                const unsigned char* Ks = ring + (size_t)s * lay.stage_bytes;
                pol.block(Ks, Ks + lay.stage_bytes / 2, j0 + (uu - u), p.qscale, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }
        if (w != 0) {
            if (!first_piece) named_sync(2);
            pol.put(mo, mm, w, rows, lane);
            named_arrive(1);
        } else {
            named_sync(1);
            const bool complete = seg_start >= start && seg_start + P <= end;
            const size_t ps = (size_t)blockIdx.x * 2 + ((u == start) ? 0 : 1);
            pol.merge_store(mo, mm, rows, complete, p.pst_o, p.pst_lse, m0, g, p.num_q_heads,
                            p.part_o + ps * kRows * D, p.part_lse + ps * kRows, lane);
            if (!complete) {
                __threadfence();
                __syncwarp();
                const int c0 = seg_start / chunk, c1 = (seg_start + P - 1) / chunk;
                int last = 0;
                if (lane == 0)
                    last = count_piece(p.counters + 2 * ((size_t)m0 * H + g), p.tag, c1 - c0 + 1);
                if (__shfl_sync(FULL, last, 0)) {
                    __threadfence();
                    merge_prefix_partials<D, G>(p, seg_start, chunk, c0, c1, rows, m0, g, lane);
                }
            }
            named_arrive(2);
        }
        first_piece = false;
        u = piece_end;
    }
    if (w != 0 && !first_piece) named_sync(2);
}

}  // namespace dec
}  // namespace pagedkv
