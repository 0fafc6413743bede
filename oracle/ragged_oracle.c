/*
 * ragged_oracle.c -- plain, slow CPU oracle for one attention layer's forward
 * over a ragged batch with a block-indexed KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it follows (page titles and sections of the source pages):
 *  - "DeepSpeed Inference v2" (pyshine.com/deepspeed-2), section "Ragged
 *    batches: packing a whole server into four tensors": the tokens of all
 *    sequences are concatenated into one stream, with per-sequence metadata in
 *    parallel buffers and a token-to-sequence map; kernels address the KV pools
 *    through the integer block ids each sequence owns.
 *  - same page, section "The front desk": each sequence descriptor keeps its
 *    integer block ids; pools are flat block-indexed tensors.
 *  - "DeepSpeed-Inference and DeepSpeed-MII" tutorial (jwzheng96, ch. 10),
 *    section 10.10: the ragged batch carries offset / cu_seqlens metadata.
 *  - The computed result is the exact causal softmax attention of every new
 *    token over all earlier positions of its own sequence (the cached history
 *    plus the earlier new tokens of the same chunk, and itself), with rotary
 *    position embedding applied to the new queries and keys before the keys
 *    are stored.  The pages name the kernels ("blocked flash attention") but
 *    print none of their math, so the oracle is the plain definition.
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes of the repository):
 *  - rotary embedding: frequencies f_k = theta^(-2k/d), k < d/2; "half" pairing
 *    (x_k, x_{k+d/2}) by default, "interleaved" pairing (x_{2k}, x_{2k+1}) on
 *    request; position p = seen + j for the j-th new token.
 *  - keys/values stored in the pool are the rotated keys and the raw values,
 *    rounded to the storage type; the rotation for stored keys (and for the
 *    optional rotated-query output) is evaluated in fp32 in a fixed, plain
 *    operation order (below), then rounded to the storage type with
 *    round-to-nearest-even.  The query used for attention is rotated in fp64
 *    and is not rounded.
 *  - pool layout [num_blocks][2 (K,V)][Hkv][block_size][d]; position p of
 *    sequence i lives in block block_table_i[p / bs] at offset p % bs.
 *  - query head h reads KV head floor(h / (Hq/Hkv)); softmax scale 1/sqrt(d)
 *    unless the caller gives one.
 *
 * Every floating-point value here is fp64 except the fp32 rotary evaluation
 * that defines the stored keys.  Build with -ffp-contract=off so that no
 * multiply-add is fused.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_FP16 0
#define OR_BF16 1
#define OR_ROPE_HALF 0
#define OR_ROPE_INTERLEAVED 1

/* ------------------------------------------------------------------------- */
/* Storage types: IEEE binary16 and bfloat16 (the upper half of a binary32).  */
/* ------------------------------------------------------------------------- */

static double fp16_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double storage_to_double(uint16_t bits, int dtype) {
    return dtype == OR_BF16 ? bf16_bits_to_double(bits) : fp16_bits_to_double(bits);
}

/* binary32 -> bfloat16, round to nearest, ties to even. */
static uint16_t float_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) {
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u); /* quiet NaN */
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* binary32 -> binary16, round to nearest, ties to even.  Works on the exact
 * value in fp64: scale so that the kept bits are the integer part, then round
 * with rint (the default rounding mode is to-nearest-even). */
static uint16_t float_to_fp16_bits(float f) {
    double x = (double)f;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* rounds past 65504 */
    if (a < ldexp(1.0, -14)) {                            /* subnormal range */
        double m = rint(ldexp(a, 24));                    /* units of 2^-24 */
        return (uint16_t)(sign | (uint16_t)m);            /* m == 1024 is 2^-14 */
    }
    int E;
    (void)frexp(a, &E);                     /* a = f * 2^E, f in [0.5, 1) */
    double m = rint(ldexp(a, 11 - E));      /* in [1024, 2048] */
    int ex = E - 1;
    if (m >= 2048.0) {
        m = 1024.0;
        ex += 1;
    }
    int biased = ex + 15;
    if (biased >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)((int)m - 1024));
}

static uint16_t float_to_storage(float f, int dtype) {
    return dtype == OR_BF16 ? float_to_bf16_bits(f) : float_to_fp16_bits(f);
}

/* ------------------------------------------------------------------------- */
/* Rotary position embedding.                                                 */
/* ------------------------------------------------------------------------- */

static void pair_index(int k, int d, int style, int* i0, int* i1) {
    if (style == OR_ROPE_INTERLEAVED) {
        *i0 = 2 * k;
        *i1 = 2 * k + 1;
    } else {
        *i0 = k;
        *i1 = k + d / 2;
    }
}

/* fp32 rotary evaluation that defines the stored keys:
 *   f_k  = fp32(pow(theta, -2k/d))            (pow in fp64, then rounded)
 *   a    = fp32(fp32(p) * f_k)
 *   c, s = fp32(cos(a)), fp32(sin(a))          (cos/sin in fp64 of the fp32 a)
 *   y0   = fp32(fp32(x0*c) - fp32(x1*s))
 *   y1   = fp32(fp32(x1*c) + fp32(x0*s))
 */
static void rope_fp32(const float* x, float* y, int64_t p, int d, int style, float theta) {
    for (int k = 0; k < d / 2; ++k) {
        int i0, i1;
        pair_index(k, d, style, &i0, &i1);
        float fk = (float)pow((double)theta, -2.0 * (double)k / (double)d);
        float pf = (float)p;
        float a = pf * fk;
        float c = (float)cos((double)a);
        float s = (float)sin((double)a);
        float x0 = x[i0], x1 = x[i1];
        float t0 = x0 * c;
        float t1 = x1 * s;
        float t2 = x1 * c;
        float t3 = x0 * s;
        y[i0] = t0 - t1;
        y[i1] = t2 + t3;
    }
}

/* fp64 rotary evaluation used for the attention query. */
static void rope_fp64(const double* x, double* y, int64_t p, int d, int style, double theta) {
    for (int k = 0; k < d / 2; ++k) {
        int i0, i1;
        pair_index(k, d, style, &i0, &i1);
        double fk = pow(theta, -2.0 * (double)k / (double)d);
        double a = (double)p * fk;
        double c = cos(a), s = sin(a);
        double x0 = x[i0], x1 = x[i1];
        y[i0] = x0 * c - x1 * s;
        y[i1] = x1 * c + x0 * s;
    }
}

/* ------------------------------------------------------------------------- */
/* Exported helpers (used by the pins in the tests).                          */
/* ------------------------------------------------------------------------- */

void oracle_storage_to_f64(const uint16_t* bits, int64_t n, int32_t dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = storage_to_double(bits[i], dtype);
}

void oracle_f32_to_storage(const float* in, int64_t n, int32_t dtype, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_storage(in[i], dtype);
}

void oracle_rope_vec_f32(const float* x, float* y, int64_t p, int32_t d, int32_t style, float theta) {
    rope_fp32(x, y, p, d, style, theta);
}

void oracle_rope_vec_f64(const double* x, double* y, int64_t p, int32_t d, int32_t style, double theta) {
    rope_fp64(x, y, p, d, style, theta);
}

/* ------------------------------------------------------------------------- */
/* Ragged metadata.                                                           */
/* ------------------------------------------------------------------------- */

/* From S descriptors (seen_i, new_i, the ids a sequence owns) build:
 *   cu_seqlens[S+1]  exclusive prefix sum of new_i
 *   seq_seen[S], seq_new[S]
 *   blk_off[S+1]     exclusive prefix sum of nb_i = ceil((seen_i+new_i)/bs)
 *   block_table      the first nb_i ids of each sequence, in batch order
 *   tok_seq[N]       sequence of each packed token
 *   tok_pos[N]       position seen_i + j of the j-th new token of sequence i
 * Returns the number of block-table entries, or -1 when a sequence owns fewer
 * than nb_i ids, has new_i < 1 or seen_i < 0. */
int64_t oracle_meta_build(int32_t S, const int32_t* seen, const int32_t* new_tokens,
                          const int64_t* ids_off, const int32_t* ids_flat, int32_t bs,
                          int32_t* cu_seqlens, int32_t* seq_seen, int32_t* seq_new,
                          int32_t* blk_off, int32_t* block_table, int32_t* tok_seq,
                          int32_t* tok_pos) {
    cu_seqlens[0] = 0;
    blk_off[0] = 0;
    for (int32_t i = 0; i < S; ++i) {
        if (new_tokens[i] < 1 || seen[i] < 0) return -1;
        int64_t L = (int64_t)seen[i] + new_tokens[i];
        int64_t nb = (L + bs - 1) / bs;
        if (ids_off[i + 1] - ids_off[i] < nb) return -1;
        seq_seen[i] = seen[i];
        seq_new[i] = new_tokens[i];
        cu_seqlens[i + 1] = cu_seqlens[i] + new_tokens[i];
        blk_off[i + 1] = blk_off[i] + (int32_t)nb;
        for (int64_t b = 0; b < nb; ++b) block_table[blk_off[i] + b] = ids_flat[ids_off[i] + b];
        for (int32_t j = 0; j < new_tokens[i]; ++j) {
            tok_seq[cu_seqlens[i] + j] = i;
            tok_pos[cu_seqlens[i] + j] = seen[i] + j;
        }
    }
    return S ? blk_off[S] : 0;
}

/* ------------------------------------------------------------------------- */
/* Rotary embedding + KV append.                                              */
/* ------------------------------------------------------------------------- */

static int64_t pool_index(int64_t blk, int kv, int h, int off, int e, int Hkv, int bs, int d) {
    return ((((blk * 2 + kv) * Hkv + h) * (int64_t)bs + off) * d) + e;
}

/* For every packed token t (sequence i, position p): rotate its K heads and
 * store them with its V heads in slot (block_table_i[p/bs], p % bs) of the
 * pool; optionally write its rotated Q heads (fp32 rotation, storage-rounded)
 * to q_out[N][Hq*d].  slot_block/slot_off receive each token's slot.
 * Returns 0, or -1 on an out-of-range block id. */
int oracle_rope_append(int32_t N, const int32_t* tok_seq, const int32_t* tok_pos,
                       const int32_t* blk_off, const int32_t* block_table, int32_t num_blocks,
                       int32_t Hq, int32_t Hkv, int32_t d, int32_t bs, int32_t dtype,
                       int32_t style, float theta, const uint16_t* qkv, uint16_t* pool,
                       uint16_t* q_out, int32_t* slot_block, int32_t* slot_off) {
    int64_t W = (int64_t)(Hq + 2 * Hkv) * d;
    float* x = (float*)malloc(sizeof(float) * (size_t)d);
    float* y = (float*)malloc(sizeof(float) * (size_t)d);
    int rc = 0;
    for (int32_t t = 0; t < N && rc == 0; ++t) {
        int32_t i = tok_seq[t];
        int64_t p = tok_pos[t];
        int32_t blk = block_table[blk_off[i] + p / bs];
        int32_t off = (int32_t)(p % bs);
        if (blk < 0 || blk >= num_blocks) {
            rc = -1;
            break;
        }
        slot_block[t] = blk;
        slot_off[t] = off;
        const uint16_t* row = qkv + (int64_t)t * W;
        for (int32_t h = 0; h < Hkv; ++h) {
            const uint16_t* k = row + (int64_t)(Hq + h) * d;
            const uint16_t* v = row + (int64_t)(Hq + Hkv + h) * d;
            for (int e = 0; e < d; ++e) x[e] = (float)storage_to_double(k[e], dtype);
            rope_fp32(x, y, p, d, style, theta);
            for (int e = 0; e < d; ++e) {
                pool[pool_index(blk, 0, h, off, e, Hkv, bs, d)] = float_to_storage(y[e], dtype);
                pool[pool_index(blk, 1, h, off, e, Hkv, bs, d)] = v[e];
            }
        }
        if (q_out) {
            for (int32_t h = 0; h < Hq; ++h) {
                const uint16_t* q = row + (int64_t)h * d;
                for (int e = 0; e < d; ++e) x[e] = (float)storage_to_double(q[e], dtype);
                rope_fp32(x, y, p, d, style, theta);
                for (int e = 0; e < d; ++e)
                    q_out[(int64_t)t * Hq * d + (int64_t)h * d + e] = float_to_storage(y[e], dtype);
            }
        }
    }
    free(x);
    free(y);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Causal attention over the block-indexed cache.                             */
/* ------------------------------------------------------------------------- */

typedef struct {
    int32_t n_rows;
    const int32_t* rows;
    const int32_t* tok_seq;
    const int32_t* tok_pos;
    const int32_t* blk_off;
    const int32_t* block_table;
    int32_t Hq, Hkv, d, bs, dtype, style;
    double theta, scale;
    const uint16_t* qkv;
    const uint16_t* pool;
    double* out;
    int32_t n_threads, tid;
} attn_job;

/* One (row, head): O = sum_u softmax_u(scale * <q_rot, K[u]>) V[u], u = 0..p. */
static void attend_one(const attn_job* J, int32_t r, int32_t h, double* q, double* qr, double* z) {
    int32_t t = J->rows[r];
    int32_t i = J->tok_seq[t];
    int64_t p = J->tok_pos[t];
    int32_t g = J->Hq / J->Hkv;
    int32_t c = h / g;
    int32_t d = J->d;
    int64_t W = (int64_t)(J->Hq + 2 * J->Hkv) * d;
    const uint16_t* qbits = J->qkv + (int64_t)t * W + (int64_t)h * d;
    for (int e = 0; e < d; ++e) q[e] = storage_to_double(qbits[e], J->dtype);
    rope_fp64(q, qr, p, d, J->style, J->theta);
    double zmax = -INFINITY;
    for (int64_t u = 0; u <= p; ++u) {
        int64_t blk = J->block_table[J->blk_off[i] + u / J->bs];
        int off = (int)(u % J->bs);
        const uint16_t* k = J->pool + pool_index(blk, 0, c, off, 0, J->Hkv, J->bs, d);
        double acc = 0.0;
        for (int e = 0; e < d; ++e) acc += qr[e] * storage_to_double(k[e], J->dtype);
        z[u] = J->scale * acc;
        if (z[u] > zmax) zmax = z[u];
    }
    double* o = J->out + ((int64_t)r * J->Hq + h) * d;
    for (int e = 0; e < d; ++e) o[e] = 0.0;
    double l = 0.0;
    for (int64_t u = 0; u <= p; ++u) {
        int64_t blk = J->block_table[J->blk_off[i] + u / J->bs];
        int off = (int)(u % J->bs);
        const uint16_t* v = J->pool + pool_index(blk, 1, c, off, 0, J->Hkv, J->bs, d);
        double w = exp(z[u] - zmax);
        l += w;
        for (int e = 0; e < d; ++e) o[e] += w * storage_to_double(v[e], J->dtype);
    }
    for (int e = 0; e < d; ++e) o[e] /= l;
}

static void* attend_worker(void* arg) {
    const attn_job* J = (const attn_job*)arg;
    int64_t maxp = 0;
    for (int32_t r = 0; r < J->n_rows; ++r)
        if (J->tok_pos[J->rows[r]] > maxp) maxp = J->tok_pos[J->rows[r]];
    double* q = (double*)malloc(sizeof(double) * (size_t)J->d);
    double* qr = (double*)malloc(sizeof(double) * (size_t)J->d);
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxp + 1));
    int64_t total = (int64_t)J->n_rows * J->Hq;
    for (int64_t w = J->tid; w < total; w += J->n_threads)
        attend_one(J, (int32_t)(w / J->Hq), (int32_t)(w % J->Hq), q, qr, z);
    free(q);
    free(qr);
    free(z);
    return NULL;
}

/* Attention output of the listed packed tokens, all query heads, in fp64:
 * out[n_rows][Hq][d].  The pool must already hold this batch's appended K/V.
 * scale <= 0 selects 1/sqrt(d).  Work is split over n_threads POSIX threads
 * (row-head items dealt round-robin); the result does not depend on it. */
int oracle_attention_rows(int32_t n_rows, const int32_t* rows, const int32_t* tok_seq,
                          const int32_t* tok_pos, const int32_t* blk_off,
                          const int32_t* block_table, int32_t Hq, int32_t Hkv, int32_t d,
                          int32_t bs, int32_t dtype, int32_t style, float theta, float scale,
                          const uint16_t* qkv, const uint16_t* pool, double* out,
                          int32_t n_threads) {
    if (Hkv <= 0 || Hq % Hkv != 0) return -1;
    if (n_threads < 1) n_threads = 1;
    attn_job* jobs = (attn_job*)malloc(sizeof(attn_job) * (size_t)n_threads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int32_t k = 0; k < n_threads; ++k) {
        attn_job J = {n_rows, rows, tok_seq, tok_pos, blk_off, block_table, Hq, Hkv, d, bs,
                      dtype, style, (double)theta,
                      scale > 0.0f ? (double)scale : 1.0 / sqrt((double)d),
                      qkv, pool, out, n_threads, k};
        jobs[k] = J;
    }
    for (int32_t k = 1; k < n_threads; ++k) pthread_create(&th[k], NULL, attend_worker, &jobs[k]);
    attend_worker(&jobs[0]);
    for (int32_t k = 1; k < n_threads; ++k) pthread_join(th[k], NULL);
    free(jobs);
    free(th);
    return 0;
}
