/*
 * pagedkv_oracle.c -- the CPU oracle for paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) may include, link or call this file.  It is read by the
 * tests, by __graft_entry__.smoke() and by the CPU-baseline leg of bench.py.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of each step, in fp64, with no
 * tiling, splitting or fusion:
 *
 *   - kv bytes per token:  2 x layers x KV heads x head dim x bytes per value
 *       ("KV cache, PagedAttention and FlashAttention", Problem 3, "The
 *        concepts"; "Memory Management in LLM Serving Systems", "KV cache
 *        sizing").
 *   - paged address arithmetic: block = p // B, offset = p % B, physical
 *       location = block_table[seq][block], offset
 *       ("KV cache, PagedAttention and FlashAttention", Problem 4, "The idea").
 *   - append: one new key row and value row per token written into its slot
 *       ("The KV Cache from First Principles", "Deriving the cache").
 *   - decode attention for one new query per sequence:
 *       out_h = sum_p softmax_p(scale * q_h . k_p) v_p over every cached
 *       position p of the sequence, with query head h reading KV head
 *       h // (n_q / n_kv)
 *       ("The KV Cache from First Principles", "Implementation" and
 *        "Grouped-query attention: the compromise"; the max-subtracted
 *        softmax of "Memory Management in LLM Serving Systems",
 *        "FlashAttention").
 *   - prefill (chunked) attention over the cache: a sequence's chunk of T new
 *       tokens, already appended at positions C-T .. C-1, each attending to
 *       every cached position up to and including its own (causal), with
 *       the same per-head definition as decode ("Memory Management in LLM
 *       Serving Systems", "FlashAttention" and its causal prefill; "The KV
 *       Cache from First Principles", "Deriving the cache": the prefill
 *       populates the cache and computes attention for the prompt).
 *   - FP8 E4M3 codec: decode from the bit-field definition, encode by brute
 *       force over all finite codes (nearest, ties to the even code,
 *       saturating to +-448).  The pages say only "FP8"; E4M3 with a
 *       per-KV-head fp32 scale is the stated reading.
 *   - 4-bit KV: the pages ask for "per-channel keys" and cite KIVI and
 *       KVQuant ("KV cache, PagedAttention and FlashAttention", Problem 3,
 *       "Trade-offs").  Reading: asymmetric 4-bit codes c in [0, 15] with
 *       x ~ c * s + z; keys use one (s, z) per (KV head, channel), fixed on
 *       the pool; values use one (s, z) per (token, KV head), from that
 *       row's min and max (s = (max - min) / 15, or 1 when max == min;
 *       z = min, a negative zero taken as +0).  c = clamp(rint((x - z) / s), 0, 15) in fp32 with
 *       round-half-to-even.  Codes are packed two per byte, the even
 *       channel in the low nibble.
 *
 * Pool contents mirrored here as two logical arrays, keys and values, each
 * [num_blocks][n_kv][block_size][d_head], so element (blk, g, off, d) sits at
 * ((blk*n_kv + g)*block_size + off)*d_head + d (the library stores a (block,
 * KV head)'s key and value rows side by side; tests read them through its
 * reported strides as these arrays).  Elements are bf16 (2 bytes, stored as
 * raw 16-bit patterns) or E4M3 (1 byte).
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC pagedkv_oracle.c -lm -lpthread.
 * No -ffast-math: fp32 division and fp64 arithmetic must be IEEE.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_BF16 0
#define ORC_E4M3 1
#define ORC_INT4 2

/* ------------------------------------------------------------------------ */
/* Sizing: "KV cache, PagedAttention and FlashAttention", Problem 3,          */
/* per-token cost = 2 x L x n_kv x d_head x bytes_per_value.                  */
/* ------------------------------------------------------------------------ */
double orc_kv_bytes_per_token(int layers, int n_kv, int d_head, double bytes_per_value)
{
    return 2.0 * (double)layers * (double)n_kv * (double)d_head * bytes_per_value;
}

/* ------------------------------------------------------------------------ */
/* Address arithmetic: "KV cache, PagedAttention and FlashAttention",        */
/* Problem 4, "The idea": block = p // B, offset = p % B, and the physical    */
/* block comes from block_table[seq][block].  Returns the slot index          */
/* phys * B + offset, or -1 when the table entry is outside [0, num_blocks). */
/* ------------------------------------------------------------------------ */
int64_t orc_slot_of(const int32_t *table_row, int64_t pos, int block_size, int64_t num_blocks)
{
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    int64_t phys = table_row[logical_block];
    if (phys < 0 || phys >= num_blocks) return -1;
    return phys * block_size + offset;
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

float orc_bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent
 * field 0 holds subnormals m/8 * 2^-6; the all-ones pattern S.1111.111 is
 * NaN; there is no infinity, so the largest finite magnitude is
 * 1.75 * 2^8 = 448. */
double orc_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Decoded values of all 256 codes, filled once from orc_e4m3_decode. */
static double orc_e4m3_values[256];
static pthread_once_t orc_e4m3_once = PTHREAD_ONCE_INIT;
static void orc_e4m3_fill(void)
{
    for (int c = 0; c < 256; ++c) orc_e4m3_values[c] = orc_e4m3_decode((uint8_t)c);
}

/* Brute-force encoder: among all finite codes of the same sign as y, take
 * the one nearest to y; on an exact tie take the code whose mantissa LSB is
 * 0 (neighbouring codes of one sign differ by one in the code, so "even code"
 * is "even mantissa").  Anything above 448 in magnitude, infinity
 * included, lands on +-448 because only finite codes are candidates.  The
 * sign of zero is kept.  NaN maps to the NaN code 0x7F. */
uint8_t orc_e4m3_encode(float y)
{
    pthread_once(&orc_e4m3_once, orc_e4m3_fill);
    if (isnan(y)) return 0x7F;
    int want_sign = signbit(y) ? 1 : 0;
    /* Saturation: a magnitude at or beyond the largest finite value (448),
     * infinity included, is +-448.  Stated directly rather than left to the
     * nearest-code search, whose fp64 distances stop telling codes apart once
     * |y| passes about 2^53 times their spacing. */
    if (fabs((double)y) >= 448.0) return (uint8_t)((want_sign << 7) | 0x7E);
    uint8_t best = (uint8_t)(want_sign << 7);
    double best_dist = INFINITY;
    for (int c = 0; c < 256; ++c) {
        if (((c >> 7) & 1) != want_sign) continue;
        double v = orc_e4m3_values[c];
        if (isnan(v)) continue;
        double dist = fabs(v - (double)y);
        if (dist < best_dist || (dist == best_dist && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_dist = dist;
        }
    }
    return best;
}

/* Quantise one bf16 value with a per-head fp32 scale: fp32 division x/scale
 * rounded to nearest even (IEEE single), then the brute-force encoder. */
uint8_t orc_quantise_e4m3(uint16_t bf16_bits, float scale)
{
    volatile float x = orc_bf16_to_float(bf16_bits);
    volatile float y = x / scale;
    return orc_e4m3_encode(y);
}

/* ------------------------------------------------------------------------ */
/* Append: "The KV Cache from First Principles", "Deriving the cache": the   */
/* new k_t and v_t are appended once and never recomputed.  Each token t     */
/* carries a slot (phys * B + offset); slot < 0 marks padding and is skipped.*/
/* k_new and v_new are [T][n_kv][d_head] bf16 bit patterns.  Returns the     */
/* number of tokens skipped because their slot was past the pool's end.      */
/* ------------------------------------------------------------------------ */
int64_t orc_append(void *k_pool, void *v_pool, int dtype, int64_t num_blocks, int block_size,
                   int n_kv, int d_head, const uint16_t *k_new, const uint16_t *v_new,
                   const int64_t *slot_mapping, int64_t n_tokens, const float *k_scale,
                   const float *v_scale)
{
    /* For large E4M3 appends the quantiser is memoised: for one head and one
     * scale it is a function of the 16-bit bf16 pattern alone, so a table of
     * its 65536 results is the same function evaluated ahead of time. */
    uint8_t *lut = NULL;
    if (dtype == ORC_E4M3 && n_tokens * (int64_t)d_head > 4 * 65536) {
        lut = (uint8_t *)malloc((size_t)2 * n_kv * 65536);
        if (lut) {
            for (int g = 0; g < n_kv; ++g)
                for (int x = 0; x < 65536; ++x) {
                    lut[(size_t)(2 * g) * 65536 + x] = orc_quantise_e4m3((uint16_t)x, k_scale[g]);
                    lut[(size_t)(2 * g + 1) * 65536 + x] = orc_quantise_e4m3((uint16_t)x, v_scale[g]);
                }
        }
    }
    int64_t out_of_range = 0;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) {
            ++out_of_range;
            continue;
        }
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int g = 0; g < n_kv; ++g) {
            int64_t dst = ((blk * n_kv + g) * block_size + off) * (int64_t)d_head;
            int64_t src = (t * n_kv + g) * (int64_t)d_head;
            for (int d = 0; d < d_head; ++d) {
                if (dtype == ORC_BF16) {
                    ((uint16_t *)k_pool)[dst + d] = k_new[src + d];
                    ((uint16_t *)v_pool)[dst + d] = v_new[src + d];
                } else if (lut) {
                    ((uint8_t *)k_pool)[dst + d] = lut[(size_t)(2 * g) * 65536 + k_new[src + d]];
                    ((uint8_t *)v_pool)[dst + d] = lut[(size_t)(2 * g + 1) * 65536 + v_new[src + d]];
                } else {
                    ((uint8_t *)k_pool)[dst + d] = orc_quantise_e4m3(k_new[src + d], k_scale[g]);
                    ((uint8_t *)v_pool)[dst + d] = orc_quantise_e4m3(v_new[src + d], v_scale[g]);
                }
            }
        }
    }
    free(lut);
    return out_of_range;
}

/* ------------------------------------------------------------------------ */
/* Decode attention                                                           */
/* ------------------------------------------------------------------------ */

/* ------------------------------------------------------------------------ */
/* 4-bit codes (the reading stated in the header).                            */
/* ------------------------------------------------------------------------ */

/* c = clamp(rint((x - z) / s), 0, 15), every step in fp32. */
uint8_t orc_int4_code(float x, float s, float z)
{
    volatile float t = x - z;
    volatile float u = t / s;
    float r = rintf(u); /* round half to even in the default rounding mode */
    if (!(r >= 0.0f)) r = 0.0f; /* also NaN */
    if (r > 15.0f) r = 15.0f;
    return (uint8_t)r;
}

/* A value row's (s, z): z = min, s = (max - min) / 15 in fp32, 1 if max == min. */
void orc_int4_row_params(const uint16_t *row_bits, int d, float *s_out, float *z_out)
{
    float mn = orc_bf16_to_float(row_bits[0]), mx = mn;
    for (int c = 1; c < d; ++c) {
        float x = orc_bf16_to_float(row_bits[c]);
        if (x < mn) mn = x;
        if (x > mx) mx = x;
    }
    volatile float range = mx - mn;
    volatile float s = range / 15.0f;
    if (s == 0.0f) s = 1.0f;
    volatile float z = mn + 0.0f; /* a negative-zero minimum is stored as +0 */
    *s_out = s;
    *z_out = z;
}

static void orc_put_nibble(uint8_t *row, int c, uint8_t code)
{
    uint8_t *b = row + c / 2;
    if (c & 1) *b = (uint8_t)((*b & 0x0F) | (code << 4));
    else *b = (uint8_t)((*b & 0xF0) | code);
}

static uint8_t orc_get_nibble(const uint8_t *row, int c)
{
    uint8_t b = row[c / 2];
    return (c & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0x0F);
}

/* Append into a 4-bit pool mirror: K and V codes [num_blocks][n_kv][B][d/2]
 * bytes, value params [num_blocks][n_kv][B][2] fp32 (s, z); key params
 * k_scale, k_zero [n_kv][d].  Returns the number of slots past the pool. */
int64_t orc_append_int4(uint8_t *k_codes, uint8_t *v_codes, float *v_params, int64_t num_blocks, int block_size,
                        int n_kv, int d_head, const uint16_t *k_new, const uint16_t *v_new,
                        const int64_t *slot_mapping, int64_t n_tokens, const float *k_scale, const float *k_zero)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * block_size) {
            ++bad;
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int g = 0; g < n_kv; ++g) {
            int64_t r = (blk * n_kv + g) * block_size + off;
            const uint16_t *kx = k_new + (t * n_kv + g) * (int64_t)d_head;
            const uint16_t *vx = v_new + (t * n_kv + g) * (int64_t)d_head;
            uint8_t *krow = k_codes + r * (d_head / 2), *vrow = v_codes + r * (d_head / 2);
            for (int c = 0; c < d_head; ++c)
                orc_put_nibble(krow, c, orc_int4_code(orc_bf16_to_float(kx[c]), k_scale[g * d_head + c],
                                                      k_zero[g * d_head + c]));
            float s, z;
            orc_int4_row_params(vx, d_head, &s, &z);
            for (int c = 0; c < d_head; ++c) orc_put_nibble(vrow, c, orc_int4_code(orc_bf16_to_float(vx[c]), s, z));
            v_params[2 * r] = s;
            v_params[2 * r + 1] = z;
        }
    }
    return bad;
}

typedef struct {
    const void *k_pool, *v_pool;
    int dtype;
    int64_t num_blocks;
    int block_size, n_kv, d_head;
    const uint16_t *q;
    int batch, n_q;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    double scale;
    const float *k_scale, *v_scale;
    const float *k_zero, *v_params; /* 4-bit pools: key zero points; value (s, z) per row */
    const int32_t *qo_indptr;       /* prefill: query rows of sequence b are qo_indptr[b] .. qo_indptr[b+1] */
    double *out;
    /* work distribution */
    int64_t next_task;
    pthread_mutex_t lock;
    int status;
} orc_decode_job;

/* Stored element -> real value.  bf16 widens exactly; E4M3 decodes exactly and
 * the per-head scale multiplies in fp64. */
static double orc_load(const void *pool, int dtype, int64_t idx, double head_scale)
{
    if (dtype == ORC_BF16) return orc_bf16_to_double(((const uint16_t *)pool)[idx]);
    return orc_e4m3_decode(((const uint8_t *)pool)[idx]) * head_scale;
}

/* One (sequence b, KV head g): gather K and V of every cached position
 * through the block table into contiguous fp64 arrays, then for each query
 * head of the group compute softmax(scale * q K^T) V with the row max
 * subtracted.  Returns 0, or -1 if a table entry needed by the sequence is
 * outside the pool (those sequences are left unwritten). */
static int orc_decode_one(orc_decode_job *job, int b, int g)
{
    const int D = job->d_head, BS = job->block_size;
    const int group = job->n_q / job->n_kv;
    int64_t C = job->context_lens[b];
    if (job->qo_indptr && job->qo_indptr[b + 1] - job->qo_indptr[b] > C) return -1; /* chunk longer than the cache */
    if (C <= 0) {
        int64_t r0 = b, r1 = (int64_t)b + 1;
        if (job->qo_indptr) {
            r0 = job->qo_indptr[b];
            r1 = job->qo_indptr[b + 1];
        }
        for (int64_t r = r0; r < r1; ++r)
            for (int hh = 0; hh < group; ++hh)
                for (int d = 0; d < D; ++d) job->out[(r * job->n_q + g * group + hh) * D + d] = 0.0;
        return 0;
    }
    if (C > (int64_t)job->max_blocks_per_seq * BS) return -1;

    double ks = job->dtype == ORC_E4M3 ? (double)job->k_scale[g] : 1.0;
    double vs = job->dtype == ORC_E4M3 ? (double)job->v_scale[g] : 1.0;
    double *Kc = (double *)malloc(sizeof(double) * (size_t)C * D);
    double *Vc = (double *)malloc(sizeof(double) * (size_t)C * D);
    double *s = (double *)malloc(sizeof(double) * (size_t)C);
    if (!Kc || !Vc || !s) {
        free(Kc); free(Vc); free(s);
        return -2;
    }
    const int32_t *row = job->block_tables + (int64_t)b * job->max_blocks_per_seq;
    for (int64_t p = 0; p < C; ++p) {
        int64_t slot = orc_slot_of(row, p, BS, job->num_blocks);
        if (slot < 0) {
            free(Kc); free(Vc); free(s);
            return -1;
        }
        int64_t blk = slot / BS, off = slot % BS;
        int64_t base = ((blk * job->n_kv + g) * BS + off) * (int64_t)D;
        if (job->dtype == ORC_INT4) { /* x = c * s + z, in fp64 */
            int64_t r = (blk * job->n_kv + g) * BS + off;
            const uint8_t *krow = (const uint8_t *)job->k_pool + r * (D / 2);
            const uint8_t *vrow = (const uint8_t *)job->v_pool + r * (D / 2);
            double vsc = job->v_params[2 * r], vz = job->v_params[2 * r + 1];
            for (int d = 0; d < D; ++d) {
                Kc[p * D + d] = orc_get_nibble(krow, d) * (double)job->k_scale[g * D + d] + job->k_zero[g * D + d];
                Vc[p * D + d] = orc_get_nibble(vrow, d) * vsc + vz;
            }
            continue;
        }
        for (int d = 0; d < D; ++d) {
            Kc[p * D + d] = orc_load(job->k_pool, job->dtype, base + d, ks);
            Vc[p * D + d] = orc_load(job->v_pool, job->dtype, base + d, vs);
        }
    }
    /* decode: one query row (position C-1) per sequence; prefill: rows
     * r0 .. r1-1 hold the chunk's tokens at positions C-T .. C-1 */
    int64_t r0 = b, r1 = (int64_t)b + 1;
    if (job->qo_indptr) {
        r0 = job->qo_indptr[b];
        r1 = job->qo_indptr[b + 1];
    }
    for (int64_t r = r0; r < r1; ++r) {
        int64_t n_keys = C - (r1 - r) + 1; /* causal: keys 0 .. own position */
        for (int hh = 0; hh < group; ++hh) {
            int h = g * group + hh; /* query head h reads KV head h // group */
            const uint16_t *qh = job->q + (r * job->n_q + h) * D;
            double m = -INFINITY;
            for (int64_t p = 0; p < n_keys; ++p) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += orc_bf16_to_double(qh[d]) * Kc[p * D + d];
                s[p] = job->scale * dot;
                if (s[p] > m) m = s[p];
            }
            double denom = 0.0;
            double *o = job->out + (r * job->n_q + h) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t p = 0; p < n_keys; ++p) {
                double w = exp(s[p] - m);
                denom += w;
                for (int d = 0; d < D; ++d) o[d] += w * Vc[p * D + d];
            }
            for (int d = 0; d < D; ++d) o[d] /= denom;
        }
    }
    free(Kc); free(Vc); free(s);
    return 0;
}

static void *orc_decode_worker(void *arg)
{
    orc_decode_job *job = (orc_decode_job *)arg;
    int64_t n_tasks = (int64_t)job->batch * job->n_kv;
    for (;;) {
        pthread_mutex_lock(&job->lock);
        int64_t task = job->next_task++;
        pthread_mutex_unlock(&job->lock);
        if (task >= n_tasks) break;
        int rc = orc_decode_one(job, (int)(task / job->n_kv), (int)(task % job->n_kv));
        if (rc != 0) {
            pthread_mutex_lock(&job->lock);
            if (job->status == 0) job->status = rc;
            pthread_mutex_unlock(&job->lock);
        }
    }
    return NULL;
}

/* q is [batch][n_q][d_head] bf16 bit patterns; block_tables [batch][W] int32;
 * context_lens [batch] int32 (the length after this step's append, so the
 * new token attends to itself); scale is the fp32 value the caller passes
 * (widened exactly); out is [batch][n_q][d_head] fp64.  Returns 0, -1 if a
 * sequence needed a table entry outside the pool or a length above W * B,
 * -2 on allocation failure, -3 on bad arguments. */
int orc_decode(const void *k_pool, const void *v_pool, int dtype, int64_t num_blocks,
               int block_size, int n_kv, int d_head, const uint16_t *q, int batch, int n_q,
               const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
               float scale, const float *k_scale, const float *v_scale, double *out,
               int n_threads)
{
    if (n_kv <= 0 || n_q <= 0 || n_q % n_kv != 0 || batch < 0 || d_head <= 0 || block_size <= 0)
        return -3;
    orc_decode_job job;
    memset(&job, 0, sizeof job);
    job.k_pool = k_pool; job.v_pool = v_pool; job.dtype = dtype;
    job.num_blocks = num_blocks; job.block_size = block_size; job.n_kv = n_kv; job.d_head = d_head;
    job.q = q; job.batch = batch; job.n_q = n_q;
    job.block_tables = block_tables; job.max_blocks_per_seq = max_blocks_per_seq;
    job.context_lens = context_lens; job.scale = (double)scale;
    job.k_scale = k_scale; job.v_scale = v_scale; job.out = out;
    pthread_mutex_init(&job.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t tids[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&tids[started], NULL, orc_decode_worker, &job) == 0) ++started;
    orc_decode_worker(&job);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}

/* orc_decode for a 4-bit pool: codes k_codes / v_codes, value params
 * v_params, key params k_scale / k_zero [n_kv][d_head] (see
 * orc_append_int4).  Same arguments and results otherwise. */
int orc_decode_int4(const uint8_t *k_codes, const uint8_t *v_codes, const float *v_params, int64_t num_blocks,
                    int block_size, int n_kv, int d_head, const uint16_t *q, int batch, int n_q,
                    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens, float scale,
                    const float *k_scale, const float *k_zero, double *out, int n_threads)
{
    if (n_kv <= 0 || n_q <= 0 || n_q % n_kv != 0 || batch < 0 || d_head <= 0 || d_head % 2 || block_size <= 0)
        return -3;
    orc_decode_job job;
    memset(&job, 0, sizeof job);
    job.k_pool = k_codes; job.v_pool = v_codes; job.dtype = ORC_INT4;
    job.num_blocks = num_blocks; job.block_size = block_size; job.n_kv = n_kv; job.d_head = d_head;
    job.q = q; job.batch = batch; job.n_q = n_q;
    job.block_tables = block_tables; job.max_blocks_per_seq = max_blocks_per_seq;
    job.context_lens = context_lens; job.scale = (double)scale;
    job.k_scale = k_scale; job.k_zero = k_zero; job.v_params = v_params; job.out = out;
    pthread_mutex_init(&job.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t tids[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&tids[started], NULL, orc_decode_worker, &job) == 0) ++started;
    orc_decode_worker(&job);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}

/* Prefill: query rows [qo_indptr[b], qo_indptr[b+1]) of q ([rows][n_q][d]
 * bf16) are sequence b's newest tokens, at positions C-T .. C-1 of its cache
 * (C = context_lens[b], T the row count), each attending causally.  out is
 * [rows][n_q][d] fp64.  bf16 and E4M3 pools.  Returns as orc_decode (-1 also
 * when a chunk is longer than its cache). */
int orc_prefill(const void *k_pool, const void *v_pool, int dtype, int64_t num_blocks, int block_size, int n_kv,
                int d_head, const uint16_t *q, const int32_t *qo_indptr, int batch, int n_q,
                const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens, float scale,
                const float *k_scale, const float *v_scale, double *out, int n_threads)
{
    if (n_kv <= 0 || n_q <= 0 || n_q % n_kv != 0 || batch < 0 || d_head <= 0 || block_size <= 0 || !qo_indptr ||
        dtype == ORC_INT4)
        return -3;
    orc_decode_job job;
    memset(&job, 0, sizeof job);
    job.k_pool = k_pool; job.v_pool = v_pool; job.dtype = dtype;
    job.num_blocks = num_blocks; job.block_size = block_size; job.n_kv = n_kv; job.d_head = d_head;
    job.q = q; job.batch = batch; job.n_q = n_q; job.qo_indptr = qo_indptr;
    job.block_tables = block_tables; job.max_blocks_per_seq = max_blocks_per_seq;
    job.context_lens = context_lens; job.scale = (double)scale;
    job.k_scale = k_scale; job.v_scale = v_scale; job.out = out;
    pthread_mutex_init(&job.lock, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t tids[256];
    int started = 0;
    for (int i = 1; i < n_threads; ++i)
        if (pthread_create(&tids[started], NULL, orc_decode_worker, &job) == 0) ++started;
    orc_decode_worker(&job);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    pthread_mutex_destroy(&job.lock);
    return job.status;
}

/* Number of threads the decode oracle can use on this host. */
int orc_hardware_threads(void)
{
#ifdef _SC_NPROCESSORS_ONLN
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
#else
    return 1;
#endif
}
