/*
 * pagedkv_oracle.c -- plain, slow, obviously correct CPU oracle for the paged
 * KV cache hot path: slot-mapped append, block copy, and PagedAttention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; it is written from the definitions on the source pages:
 *
 *  [CS349D-L3]  "Lecture 3: memory and prefix reuse in serving engines --
 *               vLLM PagedAttention and SGLang RadixAttention"
 *               (semidirectx.com, Stanford CS349D lecture 3 notes)
 *  [11868-L24]  "Lecture 24: PagedAttention and vLLM"
 *               (semidirectx.com, CMU 11-868 lecture 24 notes)
 *  [RL-Part3]   "Part 3: single node -- engines that optimise memory"
 *               (random-liu.github.io, LLM inference from principle to production)
 *  [S06]        "S06 memory and KV cache: PagedAttention"
 *               (llminference.xinbetween.com)
 *
 * Arithmetic: every floating-point step is done in fp64 with libm's exp.
 * No blocking, no split, no online softmax: the attention is the textbook
 * softmax(q K^T * scale) V over the gathered context.
 *
 * Layout (the pool layout [S06] "Implementation" gives for k_cache):
 *   pool  [num_blocks, block_size, num_kv_heads, head_dim]   (K and V separate)
 *   q/out [batch, num_q_heads, head_dim]
 *   block_tables int32 [batch, max_blocks_per_seq], seq_lens int32 [batch]
 *   slot_mapping int64 [num_tokens]
 *   pairs int32 [num_pairs, 2] = (src, dst)
 *
 * Element types: 0 = IEEE binary32, 1 = IEEE binary16, 2 = bfloat16 (the top
 * 16 bits of a binary32).  Decoding is written from the formats' definitions.
 * 8-bit pools (FP8 E4M3 with a per-pool scale, INT8 with per-token scales)
 * are described at their section below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };

static size_t elem_size(int dtype) { return dtype == OR_F32 ? 4u : 2u; }

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-14 / 1024 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return sign ? -v : v;
}

/* bfloat16: the 16 high-order bits of a binary32. */
static double decode_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double load_elem(const void* base, size_t idx, int dtype) {
    if (dtype == OR_F32) {
        float x;
        memcpy(&x, (const char*)base + 4 * idx, 4);
        return (double)x;
    }
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * idx, 2);
    return dtype == OR_F16 ? decode_f16(h) : decode_bf16(h);
}

/* Exposed so the tests can pin the element decoders against library ones. */
double oracle_decode_elem(const void* base, size_t idx, int dtype) {
    return load_elem(base, idx, dtype);
}

/*
 * Slot-mapped append ([RL-Part3] ch. 13 sec. 1, "slot_mapping": the GPU does
 * kv_cache[slot_mapping[i]] = new_kv; [CS349D-L3] sec. 3.1 slot arithmetic).
 * A slot addresses one token row of the pool: block slot / bs, row slot % bs,
 * which in the [num_blocks, bs, Hkv, D] layout is row `slot` of the pool viewed
 * as [num_blocks * bs, Hkv * D].  Each row is copied byte for byte.
 * Negative slots are padding and are skipped; slots >= num_blocks * bs are
 * skipped and counted.  Returns the number of out-of-range slots.
 */
long oracle_append(void* k_pool, void* v_pool, long num_blocks, long block_size,
                   long num_kv_heads, long head_dim, int dtype,
                   const void* k_new, const void* v_new,
                   const int64_t* slot_mapping, long num_tokens) {
    size_t row = (size_t)num_kv_heads * head_dim * elem_size(dtype);
    long nrows = num_blocks * block_size;
    long bad = 0;
    for (long i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= nrows) { ++bad; continue; }
        long blk = (long)(slot / block_size), off = (long)(slot % block_size);
        size_t dst = ((size_t)blk * block_size + off) * row;
        memcpy((char*)k_pool + dst, (const char*)k_new + (size_t)i * row, row);
        memcpy((char*)v_pool + dst, (const char*)v_new + (size_t)i * row, row);
    }
    return bad;
}

/*
 * Copy-on-write block copy ([CS349D-L3] sec. 4.1: allocate, copy the content,
 * remap, then write; sec. 3.2: the many small copies go in one launch).
 * For each pair in order: K[dst] <- K[src], V[dst] <- V[src], whole blocks.
 * Pairs with an id outside [0, num_blocks) are skipped and counted.
 */
long oracle_copy_blocks(void* k_pool, void* v_pool, long num_blocks,
                        long block_size, long num_kv_heads, long head_dim,
                        int dtype, const int32_t* pairs, long num_pairs) {
    size_t blk = (size_t)block_size * num_kv_heads * head_dim * elem_size(dtype);
    long bad = 0;
    for (long p = 0; p < num_pairs; ++p) {
        long src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        memmove((char*)k_pool + dst * blk, (const char*)k_pool + src * blk, blk);
        memmove((char*)v_pool + dst * blk, (const char*)v_pool + src * blk, blk);
    }
    return bad;
}

/* ------------------------------------------------------- 8-bit KV cache --
 *
 * [RL-Part3] ch. 10 (KV cache quantisation): a new token's K and V are scaled
 * and rounded to 8 bits before they are stored, and turned back into wider
 * numbers when the attention reads them (sec. 1); INT8 is a scale plus a
 * rounding to integers, with a fine-grained (per-token) scale (sec. 3); FP8 is
 * a shorter float (sec. 3).  Readings where the chapter is silent:
 *   OR_E4M3: E4M3 (bias 7, 3 mantissa bits, S.1111.111 = NaN, max 448), one
 *     scale per pool: code = E4M3(x / scale) with the division in fp32,
 *     nearest-even rounding, saturation to +-448 (infinities too), NaN -> 0x7F;
 *     value = decode(code) * scale.
 *   OR_INT8: one scale per (token, KV head): amax = max |x| over the row,
 *     inv = 127 / amax and scale = amax / 127 in fp32, code = rint(x * inv)
 *     (fp32 product, ties to even) clipped to [-127, 127]; all-zero row:
 *     scale 0, codes 0; a row holding NaN or an infinity: scale NaN, codes 0.
 *     value = code * scale.
 *   Codes use the pool layout [num_blocks, block_size, Hkv, D], one byte each;
 *   INT8 scales are fp32 [num_blocks, Hkv, block_size].
 */
enum { OR_E4M3 = 3, OR_INT8 = 4 };

static double e4m3_decode(uint8_t c) {
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);                 /* m/8 * 2^-6 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

static uint8_t e4m3_encode(float t) {
    if (isnan(t)) return 0x7F;
    uint8_t sign = signbit(t) ? 0x80 : 0;
    double a = fabs((double)t);
    if (a > 448.0) a = 448.0;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                          /* a in [2^(e-1), 2^e) */
    int E = e - 1;
    if (E < -6) E = -6;                    /* below 2^-6 the grid is 2^-9 */
    double step = ldexp(1.0, E - 3);
    double v = nearbyint(a / step) * step; /* exact quotient; ties to even */
    if (v == 0.0) return sign;
    frexp(v, &e);
    E = e - 1;
    if (E < -6) return (uint8_t)(sign | (int)(v / ldexp(1.0, -9)));
    return (uint8_t)(sign | ((E + 7) << 3) | ((int)(v / ldexp(1.0, E - 3)) - 8));
}

static void int8_quantize_row(const float* x, long n, int8_t* codes, float* scale) {
    float amax = 0.0f;
    int finite = 1;
    for (long i = 0; i < n; ++i) {
        if (!isfinite(x[i])) finite = 0;
        else if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    }
    for (long i = 0; i < n; ++i) codes[i] = 0;
    if (!finite) { *scale = NAN; return; }
    if (amax == 0.0f) { *scale = 0.0f; return; }
    float inv = 127.0f / amax;
    for (long i = 0; i < n; ++i) {
        float t = x[i] * inv;
        float r = nearbyintf(t);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        codes[i] = (int8_t)r;
    }
    *scale = amax / 127.0f;
}

static double dequant(const void* codes, size_t idx, int fmt, float row_scale,
                      double pool_scale) {
    uint8_t c = ((const uint8_t*)codes)[idx];
    if (fmt == OR_E4M3) return e4m3_decode(c) * pool_scale;
    return (double)(int8_t)c * (double)row_scale;
}

/* Exposed for the tests. */
double oracle_e4m3_decode(int code) { return e4m3_decode((uint8_t)code); }
int oracle_e4m3_encode(float t) { return e4m3_encode(t); }
void oracle_int8_quantize_row(const float* x, long n, int8_t* codes, float* scale) {
    int8_quantize_row(x, n, codes, scale);
}

/*
 * Quantising append: kv_append's slot rule, with each (token, KV head) row of
 * the new K and V (elements of `dtype`, read as fp32) quantised to `fmt`.
 * Returns the number of out-of-range slots.
 */
long oracle_append_q8(uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales,
                      long num_blocks, long block_size, long num_kv_heads, long head_dim,
                      int fmt, int dtype, const void* k_new, const void* v_new,
                      const int64_t* slot_mapping, long num_tokens,
                      float fp8_k_scale, float fp8_v_scale) {
    long nrows = num_blocks * block_size, D = head_dim, Hkv = num_kv_heads;
    long bad = 0;
    float* x = (float*)malloc(sizeof(float) * (size_t)D);
    int8_t* c8 = (int8_t*)malloc((size_t)D);
    if (!x || !c8) { free(x); free(c8); return -1; }
    for (long i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= nrows) { ++bad; continue; }
        long blk = (long)(slot / block_size), off = (long)(slot % block_size);
        for (int kv = 0; kv < 2; ++kv) {
            const void* src = kv ? v_new : k_new;
            uint8_t* codes = kv ? v_codes : k_codes;
            float* scales = kv ? v_scales : k_scales;
            float s8 = kv ? fp8_v_scale : fp8_k_scale;
            for (long g = 0; g < Hkv; ++g) {
                size_t in = ((size_t)i * Hkv + g) * D;
                size_t dst = (((size_t)blk * block_size + off) * Hkv + g) * D;
                for (long d = 0; d < D; ++d) x[d] = (float)load_elem(src, in + d, dtype);
                if (fmt == OR_E4M3) {
                    for (long d = 0; d < D; ++d) codes[dst + d] = e4m3_encode(x[d] / s8);
                } else {
                    float sc;
                    int8_quantize_row(x, D, c8, &sc);
                    memcpy(codes + dst, c8, (size_t)D);
                    scales[((size_t)blk * Hkv + g) * block_size + off] = sc;
                }
            }
        }
    }
    free(x);
    free(c8);
    return bad;
}

/* copy_blocks for an 8-bit pool: codes, and INT8 scales when given. */
long oracle_copy_blocks_q8(uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales,
                           long num_blocks, long block_size, long num_kv_heads, long head_dim,
                           const int32_t* pairs, long num_pairs) {
    size_t blk = (size_t)block_size * num_kv_heads * head_dim;
    size_t sblk = (size_t)num_kv_heads * block_size;
    long bad = 0;
    for (long p = 0; p < num_pairs; ++p) {
        long src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { ++bad; continue; }
        memmove(k_codes + dst * blk, k_codes + src * blk, blk);
        memmove(v_codes + dst * blk, v_codes + src * blk, blk);
        if (k_scales) memmove(k_scales + dst * sblk, k_scales + src * sblk, sblk * 4);
        if (v_scales) memmove(v_scales + dst * sblk, v_scales + src * sblk, sblk * 4);
    }
    return bad;
}


typedef struct {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    int dtype;          /* element type of q and out, and of the pool if fmt < 0 */
    int fmt;            /* -1: pool holds `dtype` elements; OR_E4M3 / OR_INT8: 8-bit codes */
    const float* k_scales, *v_scales;   /* OR_INT8: [num_blocks, Hkv, block_size] */
    double fp8_k_scale, fp8_v_scale;    /* OR_E4M3: one scale per pool */
    long num_blocks, block_size, num_kv_heads, head_dim;
    const int32_t* block_tables;
    long max_blocks_per_seq;
    const int32_t* seq_lens;
    long batch, num_q_heads;
    double scale;
    double* out;        /* [batch, num_q_heads, head_dim], fp64 */
    long b_begin, b_end;
    long bad;           /* out-of-range block ids met */
} decode_job;

/*
 * Attention for one sequence ([S06] "Implementation": walk the block table,
 * take the first n rows of each physical block, score q . k / sqrt(d), one
 * softmax over every position of every block, weighted sum of V;
 * [CS349D-L3] sec. 3.2: the softmax denominator sums over all positions of all
 * blocks, and only the written rows of the last block take part;
 * [RL-Part3] ch. 9 sec. 1: query heads are grouped, each group shares one KV
 * head, here in contiguous groups: kv head g = h / (Hq / Hkv)).
 *
 * Steps, all in fp64:
 *   1. gather K and V of kv head g for positions 0..L-1 through the table
 *      into contiguous arrays (the "gather" the pages describe);
 *   2. s_t = scale * sum_d q[d] k_t[d];
 *   3. w = softmax(s) with the maximum subtracted;
 *   4. out = sum_t w_t v_t.
 * L = 0 gives zeros.
 */
static void decode_one_seq(decode_job* J, long b, double* kbuf, double* vbuf,
                           double* s, double* qbuf) {
    long bs = J->block_size, Hkv = J->num_kv_heads, D = J->head_dim;
    long Hq = J->num_q_heads, group = Hq / Hkv;
    long L = J->seq_lens[b];
    if (L > J->max_blocks_per_seq * bs) {  /* table too short: use what exists */
        J->bad++;
        L = J->max_blocks_per_seq * bs;
    }
    const int32_t* table = J->block_tables + b * J->max_blocks_per_seq;
    for (long h = 0; h < Hq; ++h) {
        double* o = J->out + ((size_t)b * Hq + h) * D;
        for (long d = 0; d < D; ++d) o[d] = 0.0;
        if (L <= 0) continue;
        long g = h / group;
        /* 1. gather */
        long n = 0;
        for (long t = 0; t < L; ++t) {
            long phys = table[t / bs];
            if (phys < 0 || phys >= J->num_blocks) {  /* invalid entry: skip */
                J->bad++;
                continue;
            }
            size_t row = (((size_t)phys * bs + t % bs) * Hkv + g) * D;
            if (J->fmt < 0) {
                for (long d = 0; d < D; ++d) {
                    kbuf[n * D + d] = load_elem(J->k_pool, row + d, J->dtype);
                    vbuf[n * D + d] = load_elem(J->v_pool, row + d, J->dtype);
                }
            } else {
                size_t srow = ((size_t)phys * Hkv + g) * bs + t % bs;
                for (long d = 0; d < D; ++d) {
                    kbuf[n * D + d] = dequant(J->k_pool, row + d, J->fmt,
                                              J->k_scales ? J->k_scales[srow] : 0.0f,
                                              J->fp8_k_scale);
                    vbuf[n * D + d] = dequant(J->v_pool, row + d, J->fmt,
                                              J->v_scales ? J->v_scales[srow] : 0.0f,
                                              J->fp8_v_scale);
                }
            }
            ++n;
        }
        if (n == 0) continue;
        /* 2. scores */
        size_t qoff = ((size_t)b * Hq + h) * D;
        for (long d = 0; d < D; ++d) qbuf[d] = load_elem(J->q, qoff + d, J->dtype);
        for (long t = 0; t < n; ++t) {
            double acc = 0.0;
            for (long d = 0; d < D; ++d) acc += qbuf[d] * kbuf[t * D + d];
            s[t] = J->scale * acc;
        }
        /* 3. softmax with max subtraction */
        double m = -INFINITY;
        for (long t = 0; t < n; ++t) if (s[t] > m) m = s[t];
        double denom = 0.0;
        for (long t = 0; t < n; ++t) { s[t] = exp(s[t] - m); denom += s[t]; }
        /* 4. weighted sum of V */
        for (long t = 0; t < n; ++t) {
            double w = s[t] / denom;
            for (long d = 0; d < D; ++d) o[d] += w * vbuf[t * D + d];
        }
    }
}

static void* decode_worker(void* arg) {
    decode_job* J = (decode_job*)arg;
    long maxL = J->max_blocks_per_seq * J->block_size;
    double* kbuf = (double*)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1) * J->head_dim);
    double* vbuf = (double*)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1) * J->head_dim);
    double* s = (double*)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    double* qbuf = (double*)malloc(sizeof(double) * (size_t)J->head_dim);
    if (!kbuf || !vbuf || !s || !qbuf) {
        J->bad = -1;
    } else {
        for (long b = J->b_begin; b < J->b_end; ++b) decode_one_seq(J, b, kbuf, vbuf, s, qbuf);
    }
    free(kbuf);
    free(vbuf);
    free(s);
    free(qbuf);
    return NULL;
}

/*
 * PagedAttention decode for a batch.  Sequences are independent; with
 * num_threads > 1 contiguous ranges of sequences go to separate threads (the
 * arithmetic of each sequence is unchanged).  Returns 0 when every table entry
 * that was read is a valid block id and every seq_len fits its table, a
 * positive count of such problems otherwise (the offending positions are
 * skipped), or -1 on bad arguments / no memory.
 */
static long run_decode(const void* q, const void* k_pool, const void* v_pool, int dtype,
                       int fmt, const float* k_scales, const float* v_scales,
                       double fp8_k_scale, double fp8_v_scale,
                       long num_blocks, long block_size, long num_kv_heads, long head_dim,
                       const int32_t* block_tables, long max_blocks_per_seq,
                       const int32_t* seq_lens, long batch, long num_q_heads,
                       double scale, double* out, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 ||
        head_dim <= 0 || batch < 0)
        return -1;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > batch) num_threads = batch > 0 ? (int)batch : 1;
    decode_job* jobs = (decode_job*)calloc((size_t)num_threads, sizeof(decode_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    for (int i = 0; i < num_threads; ++i) {
        decode_job* J = &jobs[i];
        J->q = q; J->k_pool = k_pool; J->v_pool = v_pool; J->dtype = dtype;
        J->fmt = fmt; J->k_scales = k_scales; J->v_scales = v_scales;
        J->fp8_k_scale = fp8_k_scale; J->fp8_v_scale = fp8_v_scale;
        J->num_blocks = num_blocks; J->block_size = block_size;
        J->num_kv_heads = num_kv_heads; J->head_dim = head_dim;
        J->block_tables = block_tables; J->max_blocks_per_seq = max_blocks_per_seq;
        J->seq_lens = seq_lens; J->batch = batch; J->num_q_heads = num_q_heads;
        J->scale = scale; J->out = out;
        J->b_begin = batch * i / num_threads;
        J->b_end = batch * (i + 1) / num_threads;
    }
    long bad = 0;
    if (num_threads == 1) {
        decode_worker(&jobs[0]);
    } else {
        for (int i = 0; i < num_threads; ++i)
            pthread_create(&tids[i], NULL, decode_worker, &jobs[i]);
        for (int i = 0; i < num_threads; ++i) pthread_join(tids[i], NULL);
    }
    for (int i = 0; i < num_threads; ++i) {
        if (jobs[i].bad < 0) { bad = -1; break; }
        bad += jobs[i].bad;
    }
    free(jobs);
    free(tids);
    return bad;
}

long oracle_decode(const void* q, const void* k_pool, const void* v_pool, int dtype,
                   long num_blocks, long block_size, long num_kv_heads, long head_dim,
                   const int32_t* block_tables, long max_blocks_per_seq,
                   const int32_t* seq_lens, long batch, long num_q_heads,
                   double scale, double* out, int num_threads) {
    return run_decode(q, k_pool, v_pool, dtype, -1, NULL, NULL, 1.0, 1.0, num_blocks,
                      block_size, num_kv_heads, head_dim, block_tables, max_blocks_per_seq,
                      seq_lens, batch, num_q_heads, scale, out, num_threads);
}

/*
 * The same decode over an 8-bit pool: every K/V element read is the
 * dequantised value of its code (fmt OR_E4M3 or OR_INT8, see above); q and
 * out are `dtype` elements.
 */
long oracle_decode_q8(const void* q, int dtype, const uint8_t* k_codes, const uint8_t* v_codes,
                      const float* k_scales, const float* v_scales, int fmt,
                      double fp8_k_scale, double fp8_v_scale,
                      long num_blocks, long block_size, long num_kv_heads, long head_dim,
                      const int32_t* block_tables, long max_blocks_per_seq,
                      const int32_t* seq_lens, long batch, long num_q_heads,
                      double scale, double* out, int num_threads) {
    if (fmt != OR_E4M3 && fmt != OR_INT8) return -1;
    if (fmt == OR_INT8 && (!k_scales || !v_scales)) return -1;
    return run_decode(q, k_codes, v_codes, dtype, fmt, k_scales, v_scales, fp8_k_scale,
                      fp8_v_scale, num_blocks, block_size, num_kv_heads, head_dim,
                      block_tables, max_blocks_per_seq, seq_lens, batch, num_q_heads, scale,
                      out, num_threads);
}

/*
 * Swap to host ("Lecture 3", CS349D notes, sec. 5.2; "Part 3: single node",
 * ch. 14 sec. 3): a preempted request's blocks go to CPU memory and come back
 * when it resumes.  For each (gpu_block, host_block) pair in order, every
 * array of the pool (n_arrays of them: K, V, and INT8 scales when present,
 * block_bytes[a] bytes per block) is copied whole: host <- gpu (direction 0,
 * out) or gpu <- host (direction 1, in).  Pairs outside either pool are
 * skipped and counted.
 */
long oracle_swap_blocks(void* const* gpu, void* const* host, const long* block_bytes, int n_arrays,
                        long num_gpu_blocks, long num_host_blocks, const int32_t* pairs,
                        long num_pairs, int direction) {
    long bad = 0;
    for (long p = 0; p < num_pairs; ++p) {
        long g = pairs[2 * p], h = pairs[2 * p + 1];
        if (g < 0 || g >= num_gpu_blocks || h < 0 || h >= num_host_blocks) { ++bad; continue; }
        for (int a = 0; a < n_arrays; ++a) {
            char* gp = (char*)gpu[a] + (size_t)g * block_bytes[a];
            char* hp = (char*)host[a] + (size_t)h * block_bytes[a];
            if (direction == 0) memmove(hp, gp, (size_t)block_bytes[a]);
            else memmove(gp, hp, (size_t)block_bytes[a]);
        }
    }
    return bad;
}

/*
 * Paged (chunked) prefill ("Part 3: single node", ch. 13 sec. 1-2): request
 * b's C_b = cu_seqlens[b+1] - cu_seqlens[b] queries (rows cu_seqlens[b] ..
 * of q and out) are its last C_b positions of L_b = seq_lens[b]; query i
 * attends to positions 0 .. L_b - C_b + i through the block table.  Same
 * fp64 gather-then-softmax as oracle_decode; requests are independent and may
 * go to separate threads.  Returns the count of invalid table entries / too
 * long lengths met (skipped), or -1 on bad arguments / no memory.
 */
typedef struct {
    const void* q; const void* k_pool; const void* v_pool; int dtype;
    long num_blocks, block_size, num_kv_heads, head_dim;
    const int32_t* cu; const int32_t* block_tables; long max_blocks_per_seq;
    const int32_t* seq_lens; long num_q_heads; double scale; double* out;
    long b_begin, b_end; long bad;
} prefill_job;

static void* prefill_worker(void* arg) {
    prefill_job* J = (prefill_job*)arg;
    long bs = J->block_size, Hkv = J->num_kv_heads, D = J->head_dim, Hq = J->num_q_heads;
    long group = Hq / Hkv, maxL = J->max_blocks_per_seq * bs;
    double* kbuf = (double*)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1) * D);
    double* vbuf = (double*)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1) * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    long* pos = (long*)malloc(sizeof(long) * (size_t)(maxL > 0 ? maxL : 1));
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    if (!kbuf || !vbuf || !s || !pos || !qv) { J->bad = -1; goto done; }
    for (long b = J->b_begin; b < J->b_end; ++b) {
        long C = J->cu[b + 1] - J->cu[b], L = J->seq_lens[b];
        if (C <= 0 || L <= 0) continue;
        if (L > maxL) { J->bad++; L = maxL; }
        const int32_t* table = J->block_tables + b * J->max_blocks_per_seq;
        for (long g = 0; g < Hkv; ++g) {
            /* gather positions 0..L-1 of kv head g (skipping invalid blocks) */
            long n = 0;
            for (long t = 0; t < L; ++t) {
                long phys = table[t / bs];
                if (phys < 0 || phys >= J->num_blocks) { J->bad++; continue; }
                size_t row = (((size_t)phys * bs + t % bs) * Hkv + g) * D;
                for (long d = 0; d < D; ++d) {
                    kbuf[n * D + d] = load_elem(J->k_pool, row + d, J->dtype);
                    vbuf[n * D + d] = load_elem(J->v_pool, row + d, J->dtype);
                }
                pos[n++] = t;
            }
            for (long i = 0; i < C; ++i) {
                long p = J->seq_lens[b] - C + i;       /* query position */
                long row_q = J->cu[b] + i;
                for (long hh = 0; hh < group; ++hh) {
                    long h = g * group + hh;
                    double* o = J->out + ((size_t)row_q * Hq + h) * D;
                    for (long d = 0; d < D; ++d) o[d] = 0.0;
                    if (p < 0) continue;
                    for (long d = 0; d < D; ++d)
                        qv[d] = load_elem(J->q, ((size_t)row_q * Hq + h) * D + d, J->dtype);
                    long m = 0;
                    double mx = -INFINITY;
                    for (long t = 0; t < n && pos[t] <= p; ++t, ++m) {
                        double acc = 0.0;
                        for (long d = 0; d < D; ++d) acc += qv[d] * kbuf[t * D + d];
                        s[t] = J->scale * acc;
                        if (s[t] > mx) mx = s[t];
                    }
                    if (m == 0) continue;
                    double den = 0.0;
                    for (long t = 0; t < m; ++t) { s[t] = exp(s[t] - mx); den += s[t]; }
                    for (long t = 0; t < m; ++t) {
                        double w = s[t] / den;
                        for (long d = 0; d < D; ++d) o[d] += w * vbuf[t * D + d];
                    }
                }
            }
        }
    }
done:
    free(kbuf); free(vbuf); free(s); free(pos); free(qv);
    return NULL;
}

long oracle_prefill(const void* q, const void* k_pool, const void* v_pool, int dtype,
                    long num_blocks, long block_size, long num_kv_heads, long head_dim,
                    const int32_t* cu_seqlens, const int32_t* block_tables, long max_blocks_per_seq,
                    const int32_t* seq_lens, long batch, long num_q_heads, double scale,
                    double* out, int num_threads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 ||
        head_dim <= 0 || batch < 0)
        return -1;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > batch) num_threads = batch > 0 ? (int)batch : 1;
    prefill_job* jobs = (prefill_job*)calloc((size_t)num_threads, sizeof(prefill_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -1; }
    for (int i = 0; i < num_threads; ++i) {
        prefill_job* J = &jobs[i];
        J->q = q; J->k_pool = k_pool; J->v_pool = v_pool; J->dtype = dtype;
        J->num_blocks = num_blocks; J->block_size = block_size; J->num_kv_heads = num_kv_heads;
        J->head_dim = head_dim; J->cu = cu_seqlens; J->block_tables = block_tables;
        J->max_blocks_per_seq = max_blocks_per_seq; J->seq_lens = seq_lens;
        J->num_q_heads = num_q_heads; J->scale = scale; J->out = out;
        J->b_begin = batch * i / num_threads; J->b_end = batch * (i + 1) / num_threads;
    }
    if (num_threads == 1) prefill_worker(&jobs[0]);
    else {
        for (int i = 0; i < num_threads; ++i) pthread_create(&tids[i], NULL, prefill_worker, &jobs[i]);
        for (int i = 0; i < num_threads; ++i) pthread_join(tids[i], NULL);
    }
    long bad = 0;
    for (int i = 0; i < num_threads; ++i) {
        if (jobs[i].bad < 0) { bad = -1; break; }
        bad += jobs[i].bad;
    }
    free(jobs); free(tids);
    return bad;
}
