// Cascade (shared-prefix) decode, first pass, for 8-bit pools: attention of
// many sequences' queries over the KV blocks their tables share.
//
// Parallel samples or beams forked from one prompt point their block tables
// at the same physical prefix blocks ("Lecture 3", semidirectx.com CS349D
// notes, sec. 4.1; "Lecture 24", semidirectx.com CMU 11-868 notes, sec. 4.1).
// Plain decode reads such a block once per sequence.  This pass reads it once
// for a whole group: a unit is (group k, sub-group s, KV head g, 32 shared
// tokens j), and the unit's K/V code tile is multiplied against the query rows
// of every member of the sub-group at once -- up to 16 rows (members x G
// heads) on the two N tiles of mma.sync m16n8k16, the codes turned into f16 in
// registers.  For each member sequence b and head h the pass leaves a
// normalised partial output and its log2-sum-exp ("prefix state"); the second
// pass (the plain split kernel over each sequence's remaining blocks) folds it
// into the final log-sum-exp merge, the same trick the pages credit to
// Flash-Decoding ("Lecture 24", sec. 3.2) and that the S06 page names for
// vLLM's cascade path (llminference.xinbetween.com, "In production").  The
// result equals plain decode up to fp32 rounding.  (16-bit pools take the
// tcgen05 pass of decode_prefix_tc.cuh; the two share the parameters, the
// group tables, the partial slots and their merge, defined here.)
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
    const float* k_scales;         // INT8 pools: [num_blocks][num_kv_heads][bs]
    const float* v_scales;
    float vscale;                  // FP8 pools: the pool's V scale (its K scale is in qscale)
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

// Shared memory of one CTA: S stages of a unit's K then V tile (`rows` token
// rows each), and for INT8 pools S pairs of the unit's K and V scale rows.
struct PLayout {
    uint32_t full, empty, valid, misc, gcum, vg, merge_o, merge_ml, sring, ring;
    uint32_t stage_bytes, tx_bytes, total;
    __host__ __device__ PLayout(int S, int K, int rows, int D, int elt, bool scales) {
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
        sring = off;    off += scales ? 2u * 4u * rows * S : 0u;
        off = (off + 1023u) & ~1023u;
        ring = off;
        stage_bytes = 2u * rows * D * elt;
        tx_bytes = stage_bytes + (scales ? 2u * 4u * rows : 0u);
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

// The state of up to 16 query rows on mma.sync tiles, and its merge.  Lane
// roles as in TcPolicy: gid = lane / 4, tig = lane % 4; on N tile nt the lane
// holds columns (rows of the output) nt*8 + 2 tig + {0, 1}; column c is member
// c / G, head c % G.  PERM: the accumulators' dims are permuted (as the 8-bit
// policy below leaves them).  The policy supplies begin() and block().
template <typename T, int D, int G, int BSC, bool PERM = false>
struct TcRows {
    static_assert(sizeof(T) == 2 && BSC % 16 == 0 && (G == 1 || G == 2 || G == 4 || G == 8),
                  "tensor-core shapes");
    static constexpr int NT = kRows / 8;
    static constexpr int KS = D / 16;
    static constexpr int MT = D / 16;
    static constexpr int TT = BSC / 16;
    static constexpr int kTileRows = BSC;          // token rows of a unit's tile

    // The output dim of accumulator oacc[mt][.][j + 2 hf] in the lane of row gid.
    __device__ static __forceinline__ int dim(int mt, int gid, int hf) {
        return PERM ? 16 * gid + 2 * mt + hf : mt * 16 + gid + 8 * hf;
    }

    uint32_t qb[KS][NT][2];
    float oacc[MT][NT][4];
    float m_run[NT][2], l_run[NT][2];
    int lc[NT][2];                      // context length of the column's member (0: padding)

    // Before the warp merge (the 8-bit policy's accumulators are scaled).
    __device__ __forceinline__ void finish() {}

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
                    row[dim(mt, gid, 0)] = oacc[mt][nt][j];
                    row[dim(mt, gid, 1)] = oacc[mt][nt][j + 2];
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
                        const int d = dim(mt, gid, hf);
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

// 8-bit pools (FP8 E4M3 with one K and one V scale per pool, INT8 with a
// scale per token and head): a unit is a 32-row tile of 128-byte code rows
// (two blocks of 16 or one of 32), 128-byte swizzled.  As in the split
// kernel's 8-bit policy the codes turn into f16 exactly in registers and the
// MMAs run on f16; each query row is held as f16 times a power of two 2^e of
// its own (its largest |q| lands in [2^14, 2^15), so bf16 and f16 queries
// convert exactly), and a score is acc * scale * log2(e) * 2^-e (times the
// FP8 K scale, folded into qscale, or the token's INT8 K scale).  P is
// multiplied by vscale_t / R before its hi + lo split, R the largest V scale
// met so far (FP8: the pool's V scale, constant), and the accumulators hold
// O / R until finish().  The dims are permuted: the contraction over the
// head dim pairs Q and K in one permuted order (a dot product does not care),
// and the accumulator element (mt, gid, hf) is dim 16 gid + 2 mt + hf.
template <typename T, int G, int FMT>
struct Tc8Rows : TcRows<T, 128, G, 32, true> {
    using Base = TcRows<T, 128, G, 32, true>;
    static constexpr int NT = Base::NT, KS = Base::KS, MT = Base::MT, TT = Base::TT;
    static constexpr int kTileRows = 32;
    static constexpr bool kScales = FMT == kFmtInt8;

    float qinv[NT][2];    // 2^-e of the lane's score columns' query rows
    float R;              // the accumulators hold O / R
    float Rinv;           // INT8: 1 / R (0 while R is 0)

    // 16-byte chunk c of row r of a 128-byte-swizzled tile (1 KB-aligned base)
    __device__ static __forceinline__ uint4 chunk(const unsigned char* tile, int r, int c) {
        return *reinterpret_cast<const uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4));
    }

    // members m0 .. m0 + msz - 1, KV head g; vq: the FP8 pool's V scale
    __device__ __forceinline__ void begin(const T* q, int m0, int msz, int g, int hq,
                                          const int32_t* seq_lens, int cap, float vq, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        float rinv[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = nt * 8 + gid, m = row / G, h = row % G;
            const T* qr = q + ((size_t)(m0 + m) * hq + g * G + h) * 128;
            // lane (gid, tig) holds dims 32 tig + 4 ks + {0..3} of its row
            float2 qf[KS][2];
            float amax = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint2 raw = make_uint2(0u, 0u);
                if (m < msz) raw = __ldg(reinterpret_cast<const uint2*>(qr + 32 * tig + 4 * ks));
                qf[ks][0] = Mma<T>::unpack(raw.x);
                qf[ks][1] = Mma<T>::unpack(raw.y);
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    amax = fmaxf(amax, fmaxf(fabsf(qf[ks][j].x), fabsf(qf[ks][j].y)));
            }
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
            // 2^e with amax * 2^e in [2^14, 2^15): the exponent field of amax
            int e = 0;
            if (amax > 0.f && amax <= 3.0e38f) {
                const int ex = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 126;   // amax < 2^ex
                e = min(max(15 - ex, -120), 120);
            }
            const float up = __uint_as_float((uint32_t)(e + 127) << 23);
            rinv[nt] = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const __half2 hv = __floats2half2_rn(qf[ks][j].x * up, qf[ks][j].y * up);
                    this->qb[ks][nt][j] = *reinterpret_cast<const uint32_t*>(&hv);
                }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // score column c = nt*8 + 2 tig + j is query row c: lanes 4 (2 tig + j) ..
                qinv[nt][j] = __shfl_sync(FULL, rinv[nt], (2 * tig + j) * 4);
                const int c = nt * 8 + 2 * tig + j, mc = c / G;
                this->lc[nt][j] = mc < msz ? min(max(seq_lens[m0 + mc], 0), cap) : 0;
                this->m_run[nt][j] = -CUDART_INF_F;
                this->l_run[nt][j] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
                this->oacc[mt][nt][0] = this->oacc[mt][nt][1] = this->oacc[mt][nt][2] =
                    this->oacc[mt][nt][3] = 0.f;
        }
        R = FMT == kFmtInt8 ? 0.f : vq;
        Rinv = 0.f;
    }

    // Unit ju of the segment: K and V code tiles, sc = K scales [32] then V
    // scales [32] (INT8).
    __device__ __forceinline__ void block(const unsigned char* Ks, const unsigned char* Vs,
                                          const float* sc, int ju, float qscale, int lane) {
        const int gid = lane >> 2, tig = lane & 3;
        int nv[NT][2], nvmax = 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                nv[nt][j] = min(32, this->lc[nt][j] - ju * 32);
                nvmax = max(nvmax, nv[nt][j]);
            }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) nvmax = max(nvmax, __shfl_xor_sync(FULL, nvmax, off));
        // -- S^T = K_tile Q^T over both N tiles -------------------------------
        float s[TT][NT][4];
        float sv[TT][2];          // INT8: V scales of the lane's token rows (0 past nvmax)
        float smax = 0.f;
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            float acc[2][NT][4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    acc[h2][nt][0] = acc[h2][nt][1] = acc[h2][nt][2] = acc[h2][nt][3] = 0.f;
            const unsigned char* Kt = Ks + tt * 16 * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4 ra = chunk(Kt, gid, 2 * tig + h), rb = chunk(Kt, gid + 8, 2 * tig + h);
                const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    uint32_t a[4];
                    cvt4<FMT>(wa[qq], a[0], a[2]);
                    cvt4<FMT>(wb[qq], a[1], a[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        Mma<__half>::run(acc[qq & 1][nt], a, this->qb[4 * h + qq][nt][0],
                                         this->qb[4 * h + qq][nt][1]);
                }
            }
            const int t0 = tt * 16 + gid, t1 = t0 + 8;
            float f0 = qscale, f1 = qscale;
            sv[tt][0] = sv[tt][1] = 0.f;
            if constexpr (FMT == kFmtInt8) {
                f0 *= t0 < nvmax ? sc[t0] : 0.f;
                f1 *= t1 < nvmax ? sc[t1] : 0.f;
                sv[tt][0] = t0 < nvmax ? sc[32 + t0] : 0.f;
                sv[tt][1] = t1 < nvmax ? sc[32 + t1] : 0.f;
                smax = fmaxf(smax, fmaxf(sv[tt][0], sv[tt][1]));
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float q0 = qinv[nt][0], q1 = qinv[nt][1];
                s[tt][nt][0] = t0 < nv[nt][0] ? (acc[0][nt][0] + acc[1][nt][0]) * (f0 * q0) : -CUDART_INF_F;
                s[tt][nt][1] = t0 < nv[nt][1] ? (acc[0][nt][1] + acc[1][nt][1]) * (f0 * q1) : -CUDART_INF_F;
                s[tt][nt][2] = t1 < nv[nt][0] ? (acc[0][nt][2] + acc[1][nt][2]) * (f1 * q0) : -CUDART_INF_F;
                s[tt][nt][3] = t1 < nv[nt][1] ? (acc[0][nt][3] + acc[1][nt][3]) * (f1 * q1) : -CUDART_INF_F;
            }
        }
        // -- online softmax per column; INT8: R follows the largest V scale ---
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
                mnew[nt][j] = fmaxf(this->m_run[nt][j], mx);
                alpha[nt][j] = mnew[nt][j] == -CUDART_INF_F ? 1.f : fast_exp2(this->m_run[nt][j] - mnew[nt][j]);
                lsum[nt][j] = 0.f;
            }
        float rf = 1.f;
        if constexpr (FMT == kFmtInt8) {
            float mx = smax;
#pragma unroll
            for (int off = 16; off >= 4; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
            if (mx > R) {                     // (uniform: every lane sees every token row's max)
                Rinv = __frcp_rn(mx);
                rf = R * Rinv;
                R = mx;
            }
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
                this->l_run[nt][j] = this->l_run[nt][j] * alpha[nt][j] + lsum[nt][j];
                this->m_run[nt][j] = mnew[nt][j];
            }
        // rescale the accumulators only when a running maximum or R moved
        bool same = rf == 1.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) same = same && alpha[nt][0] == 1.f && alpha[nt][1] == 1.f;
        if (!__all_sync(FULL, same))
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 a2 = make_float2(alpha[nt][0] * rf, alpha[nt][1] * rf);
                    const float2 lo = __fmul2_rn(make_float2(this->oacc[mt][nt][0], this->oacc[mt][nt][1]), a2);
                    const float2 hi = __fmul2_rn(make_float2(this->oacc[mt][nt][2], this->oacc[mt][nt][3]), a2);
                    this->oacc[mt][nt][0] = lo.x; this->oacc[mt][nt][1] = lo.y;
                    this->oacc[mt][nt][2] = hi.x; this->oacc[mt][nt][3] = hi.y;
                }
        // -- O^T += V_tile^T P'^T, P' = P * vscale_t / R as hi + lo halves -----
#pragma unroll
        for (int tt = 0; tt < TT; ++tt) {
            if constexpr (FMT == kFmtInt8) {
                const float w0 = sv[tt][0] * Rinv, w1 = sv[tt][1] * Rinv;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    s[tt][nt][0] *= w0; s[tt][nt][1] *= w0;
                    s[tt][nt][2] *= w1; s[tt][nt][3] *= w1;
                }
            }
            uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float* x = s[tt][nt];
                const uint32_t h01 = Mma<__half>::pack(x[0], x[1]), h23 = Mma<__half>::pack(x[2], x[3]);
                const float2 f01 = Mma<__half>::unpack(h01), f23 = Mma<__half>::unpack(h23);
                const uint32_t l01 = Mma<__half>::pack(x[0] - f01.x, x[1] - f01.y);
                const uint32_t l23 = Mma<__half>::pack(x[2] - f23.x, x[3] - f23.y);
                bh[nt][0] = movm_t(h01); bh[nt][1] = movm_t(h23);
                bl[nt][0] = movm_t(l01); bl[nt][1] = movm_t(l23);
            }
            // V rows 2 tig, 2 tig + 1, + 8, + 9 of the 16-row tile, chunk gid
            // (dims 16 gid ..); rows no member reaches read as zero codes (P' is
            // 0 there, but an E4M3 NaN code would still poison the MMA)
            const int tv = tt * 16;
            const unsigned char* Vt = Vs + tv * 128;
            uint32_t vw[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 2 * tig + (i & 1) + 8 * (i >> 1);
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (tv + r < nvmax) v = chunk(Vt, r, gid);
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
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    Mma<__half>::run(this->oacc[mt][nt], a, bh[nt][0], bh[nt][1]);
                    Mma<__half>::run(this->oacc[mt][nt], a, bl[nt][0], bl[nt][1]);
                }
            }
        }
    }

    // The accumulators become O itself.
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) this->oacc[mt][nt][i] *= R;
    }
};

// Merge the partials of a cut segment into the prefix states (pass0, pstep:
// the element passes this warp takes when several warps share the merge;
// BATCH: slots whose loads are in flight together).
template <int D, int G, int BATCH = kMergeBatch>
__device__ __forceinline__ void merge_prefix_partials(const PParams& p, int seg_start, int chunk,
                                                      int c0, int c1, int rows, int m0, int g,
                                                      int lane, int pass0 = 0, int pstep = 1) {
    merge_slots<kRows, D, BATCH>(p.part_o, p.part_lse, c0, c1, seg_start == c0 * chunk ? 0 : 1,
                                 nullptr, nullptr, lane, pass0, pstep,
                                 [&](int r, int d0, const float* v, float lse) {
                                     if (r >= rows) return;
                                     const size_t prow =
                                         (size_t)(m0 + r / G) * p.num_q_heads + g * G + r % G;
#pragma unroll
                                     for (int k = 0; k < merge_epl<kRows, D>(); ++k)
                                         p.pst_o[prow * D + d0 + k] = v[k];
                                     if (d0 == 0) p.pst_lse[prow] = lse;
                                 });
}

// Pol: Tc8Rows (3-D swizzled maps of 128-byte code rows, UB blocks of BS
// rows per unit).
template <typename T, int D, int G, int BS, class Pol>
__global__ void __launch_bounds__(NTHREADS, 2) paged_decode_prefix(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const PParams p) {
    constexpr int ROWS = Pol::kTileRows;            // token rows per unit
    constexpr int UB = ROWS / BS;                   // pool blocks per unit
    static_assert(UB * BS == ROWS, "unit shape");
    constexpr int ELT = 1;                          // one code per element
    constexpr bool SCALES = Pol::kScales;
    constexpr int MS = kRows / G;                   // members per sub-group
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_align_1k(smem_raw);
    const int K = p.num_groups, S = p.stages, H = p.num_kv_heads, B = p.batch;
    const PLayout lay(S, K, ROWS, D, ELT, SCALES);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + lay.empty);
    volatile int* valid = reinterpret_cast<volatile int*>(smem + lay.valid);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + lay.misc);
    int* warp_tot = reinterpret_cast<int*>(smem + lay.misc) + 8;
    // the CTA's last piece, when it completes a cut segment's count: {merge,
    // seg_start, c0, c1, rows, m0, g}, posted by warp 0 for every attending warp
    volatile int* fm = reinterpret_cast<volatile int*>(smem + lay.misc) + 1;
    int* gcum = reinterpret_cast<int*>(smem + lay.gcum);
    int* vg = reinterpret_cast<int*>(smem + lay.vg);
    const int* gfirst = vg;
    const int* gsize = vg + K;
    const int* gblk = vg + 2 * K;
    unsigned char* ring = smem + lay.ring;
    float* sring = reinterpret_cast<float*>(smem + lay.sring);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cap = p.max_blocks * BS;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // The second pass is let in only after this wait: the pool is then
    // complete, so that pass may stream its blocks before this one ends.
    pdl_wait();
    pdl_launch_dependents();

    // -- used groups, their units (sub-groups x KV heads x shared units) -------
    const int NG = load_groups(p.g_first, p.g_size, p.g_blocks, K, p.seq_lens, B, BS, cap, UB, vg,
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
        // unit uu: its blocks (the second -1 when UB = 1) and KV head
        auto fetch = [&](int uu, int& id, int& id2, int& gg) {
            id = -1;
            id2 = -1;
            gg = 0;
            if (uu < end) {
                const int k = find_le(gcum, NG, uu);
                const int P = gblk[k];
                const int r = uu - gcum[k];
                gg = (r / P) % H;
                const int32_t* row = p.block_tables + (size_t)gfirst[k] * p.max_blocks + (r % P) * UB;
                id = __ldg(row);
                if (UB == 2) id2 = __ldg(row + 1);
            }
        };
        auto in_pool = [&](int x) { return x >= 0 && x < p.num_blocks; };
        int id_cur, id2_cur, g_cur, id_nxt, id2_nxt, g_nxt;
        fetch(start + lane, id_cur, id2_cur, g_cur);
        int k = 0;
        for (int base = start; base < end; base += 32) {
            fetch(base + 32 + lane, id_nxt, id2_nxt, g_nxt);
            const int n = min(32, end - base);
            for (int i = 0; i < n; ++i, ++k) {
                const int id = __shfl_sync(FULL, id_cur, i);
                const int id2 = __shfl_sync(FULL, id2_cur, i);
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
                    } else if (in_pool(id) && (UB == 1 || in_pool(id2))) {
                        valid[s] = 1;
                        mbar_arrive_tx(fb, lay.tx_bytes);
                        const uint32_t dst = smem_u32(ring + (size_t)s * lay.stage_bytes);
                        const uint32_t vdst = dst + lay.stage_bytes / 2;
                        // one 3-D copy per block: BS code rows of 128 bytes
#pragma unroll
                        for (int x = 0; x < UB; ++x) {
                            const int bid = x == 0 ? id : id2;
                            tma_load_3d(dst + x * BS * 128, &tmap_k, 0, gg, bid * BS, fb);
                            tma_load_3d(vdst + x * BS * 128, &tmap_v, 0, gg, bid * BS, fb);
                            if constexpr (SCALES) {
                                // the unit's K scales [ROWS], then its V scales [ROWS]
                                const size_t srow = ((size_t)bid * H + gg) * BS;
                                const uint32_t sdst = smem_u32(sring + s * 2 * ROWS + x * BS);
                                bulk_load(sdst, p.k_scales + srow, BS * 4u, fb);
                                bulk_load(sdst + ROWS * 4u, p.v_scales + srow, BS * 4u, fb);
                            }
                        }
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
            id2_cur = id2_nxt;
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

        pol.begin(qbase, m0, msz, g, p.num_q_heads, p.seq_lens, cap, p.vscale, lane);
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
                pol.block(Ks, Ks + lay.stage_bytes / 2, sring + s * 2 * ROWS, j0 + (uu - u),
                          p.qscale, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }
        pol.finish();
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
            const bool final_piece = piece_end == end;
            int merge = 0;
            if (!complete) {
                __threadfence();
                __syncwarp();
                const int c0 = seg_start / chunk, c1 = (seg_start + P - 1) / chunk;
                int last = 0;
                if (lane == 0)
                    last = count_piece(p.counters + 2 * ((size_t)m0 * H + g), p.tag, c1 - c0 + 1);
                merge = __shfl_sync(FULL, last, 0);
                if (merge) __threadfence();
                if (final_piece) {
                    // the other warps are done: they share this merge below
                    if (lane == 0) {
                        fm[1] = seg_start; fm[2] = c0; fm[3] = c1; fm[4] = rows; fm[5] = m0;
                        fm[6] = g;
                    }
                } else if (merge) {
                    merge_prefix_partials<D, G>(p, seg_start, chunk, c0, c1, rows, m0, g, lane);
                }
            }
            if (final_piece && lane == 0) fm[0] = merge;
            __syncwarp();
            named_arrive(2);
        }
        first_piece = false;
        u = piece_end;
    }
    if (first_piece) return;
    if (w != 0) named_sync(2);
    if (fm[0]) {                                   // every warp: a share of the last piece's merge
        __threadfence();
        merge_prefix_partials<D, G>(p, fm[1], chunk, fm[2], fm[3], fm[4], fm[5], fm[6], lane, w, NCW);
    }
}

// -- host side: occupancy and launch of one instance ------------------------
template <typename T, int G, int BS, class Pol>
cudaError_t prefix_attrs(size_t smem, int* occ) {
    auto k = paged_decode_prefix<T, 128, G, BS, Pol>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, k, NTHREADS, smem);
}

// Launched with programmatic stream serialisation (the kernel waits on its
// predecessor with griddepcontrol before it reads anything).
template <typename T, int G, int BS, class Pol>
cudaError_t prefix_launch(const CUtensorMap& mk, const CUtensorMap& mv, const PParams& p,
                          size_t smem, int grid, cudaStream_t stream) {
    auto k = paged_decode_prefix<T, 128, G, BS, Pol>;
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

// The instances for 8-bit pools, one translation unit per query type: by the
// pool's code format, block size (16 or 32) and the group.
template <typename T, class F>
cudaError_t by_q8_shape(const kv_pool& pool, int group, F&& f) {
    const bool i8 = pool.cache_dtype == KV_INT8;
    const int bs = pool.block_size;
#define PKV_Q(FF, GG, BB)                                          \
    if ((FF == kFmtInt8) == i8 && group == GG && bs == BB)         \
        return f.template operator()<T, GG, BB, Tc8Rows<T, GG, FF>>();
    PKV_Q(kFmtE4M3, 1, 16) PKV_Q(kFmtE4M3, 2, 16) PKV_Q(kFmtE4M3, 4, 16) PKV_Q(kFmtE4M3, 8, 16)
    PKV_Q(kFmtE4M3, 1, 32) PKV_Q(kFmtE4M3, 2, 32) PKV_Q(kFmtE4M3, 4, 32) PKV_Q(kFmtE4M3, 8, 32)
    PKV_Q(kFmtInt8, 1, 16) PKV_Q(kFmtInt8, 2, 16) PKV_Q(kFmtInt8, 4, 16) PKV_Q(kFmtInt8, 8, 16)
    PKV_Q(kFmtInt8, 1, 32) PKV_Q(kFmtInt8, 2, 32) PKV_Q(kFmtInt8, 4, 32) PKV_Q(kFmtInt8, 8, 32)
#undef PKV_Q
    return cudaErrorNotSupported;
}

}  // namespace dec

// 8-bit prefix kernels by query type (decode_cascade_q8_*.cu).
cudaError_t prefix_q8_attrs_bf16(const kv_pool& pool, int group, size_t smem, int* occ);
cudaError_t prefix_q8_attrs_f16(const kv_pool& pool, int group, size_t smem, int* occ);
cudaError_t prefix_q8_launch_bf16(const kv_pool& pool, int group, const dec::PParams& p,
                                  size_t smem, int grid, cudaStream_t stream);
cudaError_t prefix_q8_launch_f16(const kv_pool& pool, int group, const dec::PParams& p,
                                 size_t smem, int grid, cudaStream_t stream);

}  // namespace pagedkv
