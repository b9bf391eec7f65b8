/*
 * oracle.c -- plain, slow CPU oracle for the DeepSeek-V4.1 sparse latent attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file exists to check the CUDA library against the pages that
 * define the method.  Only the tests, the smoke check and the CPU-baseline leg of the benchmark
 * may load it.  It shares no code, header, table or constant with the CUDA path, and the CUDA
 * path never calls it.
 *
 * Sources (page title, section):
 *   [attend]   "DeepSeek V4.1", blocks/.../attention/attend: get_window_topk_idxs,
 *              sparse_attn_kernel, sparse_attn wrapper.
 *   [latent]   "DeepSeek V4.1", blocks/.../attention/query-latent: Attention.__init__
 *              (window_kv_cache ring buffer), Attention.forward (window + compressed concat).
 *   [attn]     "Module attn" (deepseek_v41_ref API page): the Precision paragraph, the ring-cache
 *              paragraph, FP8_BLOCK, act_quant_inplace, pow2_ceil, sparse_attn, window_topk_idxs,
 *              apply_rotary, freqs_cis.
 *   [latent] also gives precompute_freqs_cis and apply_rotary_emb (RoPE) and the remark that the
 *              compressed cache holds quantised values (the fp8 row store below keeps them as
 *              e4m3 codes plus scale exponents).
 *
 * Everything here is written as plain loops in the order the pages state the steps.  The
 * precision is the pages' own: the fp8 round trip decides its scale in f32 ([attn] pow2_ceil
 * works on the IEEE fields of an f32), and sparse_attn runs in f32 with a bf16 result ([attn]
 * Precision).  A float64 variant of sparse_attn is kept for the pinning tests.
 *
 * Every function is pinned by tests that do not re-type it: the ring-cache worked example of
 * [attn], brute-force dense masked softmax, closed forms, invariances, and PyTorch's own
 * float8_e4m3fn conversion (see tests/test_oracle_pins.py).
 *
 * Build (plain C11, no intrinsics, no fast-math, no contraction so x86 and Arm agree):
 *   gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared -o liboracle.so oracle.c -lm -lpthread
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* bf16 <-> f32, written from the format: bf16 is the top 16 bits of an IEEE binary32.         */
/* ------------------------------------------------------------------------------------------ */

static float bf16_bits_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an f32 to the nearest bf16, ties to even.  NaN stays NaN (quiet). */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;          /* truncated result                     */
    uint32_t dropped = u & 0xffffu;   /* the 16 bits that do not fit          */
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;                   /* carries into the exponent if needed  */
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------------------------------ */
/* window_topk_idxs  ([attend] get_window_topk_idxs; [attn] window_topk_idxs)                  */
/* ------------------------------------------------------------------------------------------ */

/*
 * Ring-slot index rows for the sliding window.
 * start_pos == 0 (prefill, s queries): cols = min(s, window); row q lists the causal window of
 *   query q starting at max(0, q - window + 1); an entry past q holds nothing and is -1.
 * start_pos > 0 (decode, one query): cols = window; the whole ring oldest first, i.e. slots
 *   oldest..window-1 then 0..oldest-1 with oldest = start_pos % window + 1; a slot whose value
 *   exceeds start_pos is still empty and is -1.
 * Writes out[q * cols + j].  Returns cols, or -1 for a chunked prefill (start_pos > 0, s > 1),
 * which the pages do not define.
 */
int oracle_window_topk_idxs(int32_t *out, int s, int64_t start_pos, int window) {
    if (s <= 0 || window <= 0 || start_pos < 0) return -1;
    if (start_pos == 0) {
        int cols = s < window ? s : window;
        for (int q = 0; q < s; ++q) {
            int first = q - window + 1;
            if (first < 0) first = 0;
            for (int j = 0; j < cols; ++j) {
                int v = first + j;
                out[(int64_t)q * cols + j] = v > q ? -1 : v;
            }
        }
        return cols;
    }
    if (s != 1) return -1;
    int oldest = (int)(start_pos % window) + 1;
    int k = 0;
    for (int v = oldest; v < window; ++v) out[k++] = (int64_t)v > start_pos ? -1 : v;
    for (int v = 0; v < oldest; ++v) out[k++] = (int64_t)v > start_pos ? -1 : v;
    return window;
}

/* ------------------------------------------------------------------------------------------ */
/* fp8 round trip  ([attn] FP8_BLOCK, pow2_ceil, act_quant_inplace, Precision)                 */
/* ------------------------------------------------------------------------------------------ */

#define ORACLE_FP8_BLOCK 32
#define ORACLE_E4M3_MAX 448.0f

/* 2 ** ceil(log2(v)) for a positive normal f32, read off the IEEE fields: a value whose
 * mantissa field is zero is already a power of two; otherwise the next power up is the one
 * with the exponent field plus one and a zero mantissa. */
float oracle_pow2_ceil(float v) {
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    uint32_t exponent = (u >> 23) & 0xffu;
    uint32_t mantissa = u & 0x7fffffu;
    if (mantissa == 0u) return v;
    uint32_t r = (exponent + 1u) << 23;
    float out;
    memcpy(&out, &r, sizeof out);
    return out;
}

/* The 127 non-negative finite values of e4m3fn (1 sign, 4 exponent, 3 mantissa bits, bias 7;
 * exponent field 0 is subnormal with step 2^-9; code 0x7f is NaN and is not a value).  The codes
 * are in ascending order of value. */
static double e4m3_table[127];
static pthread_once_t e4m3_once = PTHREAD_ONCE_INIT;

static void e4m3_build_table(void) {
    for (int code = 0; code < 127; ++code) {
        int e = code >> 3, m = code & 7;
        e4m3_table[code] = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    }
}

/* Code (0..126, the table position) of the e4m3fn magnitude nearest to a >= 0, ties to the even
 * code (even mantissa).  a must lie in [0, 448]. */
static int e4m3_nearest_code(double a) {
    pthread_once(&e4m3_once, e4m3_build_table);
    int k = 0;                               /* largest code with value <= a */
    while (k + 1 < 127 && e4m3_table[k + 1] <= a) ++k;
    int pick = k;
    if (k + 1 < 127 && a > e4m3_table[k]) {
        double below = a - e4m3_table[k], above = e4m3_table[k + 1] - a;
        if (above < below) pick = k + 1;
        else if (above == below) pick = (k % 2 == 0) ? k : k + 1;
    }
    return pick;
}

/* Nearest e4m3fn value to y, ties to the even code (even mantissa).  y must lie in [-448, 448]. */
float oracle_e4m3_round(float y) {
    double r = e4m3_table[e4m3_nearest_code(fabs((double)y))];
    return (float)(signbit(y) ? -r : r);     /* sign-magnitude: -0 stays -0 */
}

/* One block of FP8_BLOCK bf16 values, in place: amax floored at 1e-4, scale = pow2_ceil of
 * amax / 448 (f32 division), each value divided by the scale, clamped to +-448, rounded to
 * e4m3 (RNE), multiplied back and rounded to bf16 (exact: e4m3 times a power of two). */
static void quant_block(uint16_t *x) {
    float amax = 0.0f;
    for (int i = 0; i < ORACLE_FP8_BLOCK; ++i) {
        float a = fabsf(bf16_bits_to_f32(x[i]));
        if (a > amax) amax = a;
    }
    if (amax < 1e-4f) amax = 1e-4f;
    float scale = oracle_pow2_ceil(amax / ORACLE_E4M3_MAX);
    for (int i = 0; i < ORACLE_FP8_BLOCK; ++i) {
        float y = bf16_bits_to_f32(x[i]) / scale;
        if (y > ORACLE_E4M3_MAX) y = ORACLE_E4M3_MAX;
        if (y < -ORACLE_E4M3_MAX) y = -ORACLE_E4M3_MAX;
        float qv = oracle_e4m3_round(y);
        x[i] = f32_to_bf16_bits(qv * scale);
    }
}

/* act_quant_inplace over n bf16 values (n a multiple of FP8_BLOCK).  Returns 0, or -1. */
int oracle_act_quant_inplace(uint16_t *x, int64_t n) {
    if (n < 0 || n % ORACLE_FP8_BLOCK != 0) return -1;
    for (int64_t i = 0; i < n; i += ORACLE_FP8_BLOCK) quant_block(x + i);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* fp8 row store: the quantised values kept as e4m3fn codes plus one power-of-two scale        */
/* exponent per block ([attn] act_quant_inplace, Precision; [query-latent] the compressed      */
/* cache holds quantised values).  Decoding a row gives exactly the bf16 round trip above.     */
/* ------------------------------------------------------------------------------------------ */

/* One block: the same scale and rounding as quant_block, kept as codes (bit 7 the sign, bits
 * 0-6 the position in the ascending table of magnitudes, i.e. the e4m3fn bit pattern) and the
 * scale's exponent k (scale = 2^k). */
static void quant_block_codes(const uint16_t *x, uint8_t *codes, int8_t *k_out) {
    float amax = 0.0f;
    for (int i = 0; i < ORACLE_FP8_BLOCK; ++i) {
        float a = fabsf(bf16_bits_to_f32(x[i]));
        if (a > amax) amax = a;
    }
    if (amax < 1e-4f) amax = 1e-4f;
    float scale = oracle_pow2_ceil(amax / ORACLE_E4M3_MAX);
    int k;
    frexpf(scale, &k);                       /* scale = 0.5 * 2^k, so scale = 2^(k - 1) */
    *k_out = (int8_t)(k - 1);
    for (int i = 0; i < ORACLE_FP8_BLOCK; ++i) {
        float y = bf16_bits_to_f32(x[i]) / scale;
        if (y > ORACLE_E4M3_MAX) y = ORACLE_E4M3_MAX;
        if (y < -ORACLE_E4M3_MAX) y = -ORACLE_E4M3_MAX;
        int code = e4m3_nearest_code(fabs((double)y));
        codes[i] = (uint8_t)((signbit(y) ? 0x80 : 0) | code);
    }
}

/* rows x d bf16 values (row-major, d a multiple of FP8_BLOCK) into codes[rows][d] and
 * exps[rows][d / FP8_BLOCK].  Returns 0, or -1. */
int oracle_kv_quantize_fp8(const uint16_t *x, int64_t rows, int d, uint8_t *codes, int8_t *exps) {
    if (rows < 0 || d <= 0 || d % ORACLE_FP8_BLOCK != 0) return -1;
    const int nb = d / ORACLE_FP8_BLOCK;
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < nb; ++c)
            quant_block_codes(x + r * d + (int64_t)c * ORACLE_FP8_BLOCK, codes + r * d + (int64_t)c * ORACLE_FP8_BLOCK,
                              exps + r * nb + c);
    return 0;
}

/* codes[rows][d] and exps[rows][d / FP8_BLOCK] back to bf16: value = (+-table[code]) * 2^k,
 * exact in bf16.  The NaN codes 0x7f / 0xff (never written by the quantiser) decode to NaN. */
int oracle_kv_dequantize_fp8(const uint8_t *codes, const int8_t *exps, int64_t rows, int d, uint16_t *out) {
    if (rows < 0 || d <= 0 || d % ORACLE_FP8_BLOCK != 0) return -1;
    pthread_once(&e4m3_once, e4m3_build_table);
    const int nb = d / ORACLE_FP8_BLOCK;
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < d; ++c) {
            uint8_t code = codes[r * d + c];
            int k = exps[r * nb + c / ORACLE_FP8_BLOCK];
            if ((code & 0x7f) == 0x7f) {
                out[r * d + c] = 0x7fc0u;
                continue;
            }
            double v = ldexp(e4m3_table[code & 0x7f], k);
            out[r * d + c] = f32_to_bf16_bits((float)((code & 0x80) ? -v : v));
        }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Ring write  ([latent] window_kv_cache; [attn] ring-cache paragraph, WindowCache, attention) */
/* ------------------------------------------------------------------------------------------ */

/*
 * New KV rows kv[bi][t][0:d] (row stride d, batch stride kv_bstride) are rounded through fp8 in
 * place; the token at absolute position start_pos + t is then stored in ring slot
 * (start_pos + t) % window when it is among the last `window` rows of the chunk
 * (t >= s - window).  ring[bi][slot][0:d] has batch stride ring_bstride.
 */
int oracle_kv_quant_ring_write(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride,
                               int b, int s, int d, int64_t start_pos, int window) {
    if (b < 0 || s < 0 || d <= 0 || d % ORACLE_FP8_BLOCK != 0 || window <= 0 || start_pos < 0) return -1;
    for (int bi = 0; bi < b; ++bi) {
        for (int t = 0; t < s; ++t) {
            uint16_t *row = kv + (int64_t)bi * kv_bstride + (int64_t)t * d;
            oracle_act_quant_inplace(row, d);
            if (t >= s - window) {
                int64_t slot = (start_pos + t) % window;
                memcpy(ring + (int64_t)bi * ring_bstride + slot * d, row, (size_t)d * sizeof(uint16_t));
            }
        }
    }
    return 0;
}

/*
 * The ring write with an fp8 row store as the ring: kv rows rounded in place as above, and the
 * ring slot of each of the last `window` rows receives that row's codes and exponents, computed
 * from the row as given (one quantisation pass, so its decode equals the rounded row).  ring
 * slots are rows of codes[bi][slot][d] and exps[bi][slot][d / FP8_BLOCK], batch stride
 * ring_bstride rows.
 */
int oracle_kv_quant_ring_write_fp8(uint16_t *kv, int64_t kv_bstride, uint8_t *codes, int8_t *exps,
                                   int64_t ring_bstride, int b, int s, int d, int64_t start_pos, int window) {
    if (b < 0 || s < 0 || d <= 0 || d % ORACLE_FP8_BLOCK != 0 || window <= 0 || start_pos < 0) return -1;
    const int nb = d / ORACLE_FP8_BLOCK;
    for (int bi = 0; bi < b; ++bi) {
        for (int t = 0; t < s; ++t) {
            uint16_t *row = kv + (int64_t)bi * kv_bstride + (int64_t)t * d;
            if (t >= s - window) {
                int64_t slot = (int64_t)bi * ring_bstride + (start_pos + t) % window;
                oracle_kv_quantize_fp8(row, 1, d, codes + slot * d, exps + slot * nb);
            }
            oracle_act_quant_inplace(row, d);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* RoPE  ([attn] freqs_cis, apply_rotary, Precision; [latent] precompute_freqs_cis,            */
/* apply_rotary_emb and Attention.forward: rotate the last rope_dim of q and of the kv row,    */
/* then the inverse rotation on the output)                                                      */
/* ------------------------------------------------------------------------------------------ */

/*
 * The ratio-0 table (no YaRN): for position p and pair j < dim/2,
 *   freq_j = 1 / base^(2j / dim)        (f32: the exponent 2j/dim, the power and the reciprocal)
 *   angle  = p * freq_j                 (f32 product)
 *   table[p][j] = (cos angle, sin angle) in f32.
 * out has npos * dim/2 * 2 floats.
 */
int oracle_rope_table(float *out, int64_t npos, int dim, double base) {
    if (npos < 0 || dim <= 0 || dim % 2 != 0 || !(base > 0.0)) return -1;
    for (int j = 0; j < dim / 2; ++j) {
        float e = (float)(2 * j) / (float)dim;
        float pw = (float)pow(base, (double)e);
        float freq = 1.0f / pw;
        for (int64_t p = 0; p < npos; ++p) {
            float ang = (float)p * freq;
            out[(p * (dim / 2) + j) * 2] = (float)cos((double)ang);
            out[(p * (dim / 2) + j) * 2 + 1] = (float)sin((double)ang);
        }
    }
    return 0;
}

/*
 * Rotate the last rd values of each row_len-wide row of x (bf16, in place): pair j of the rotated
 * part, (a, b) = (x[2j], x[2j+1]), is the complex number a + ib, multiplied by cos + i sin of row
 * r's position (sin negated when inverse) in f32, each product and sum rounded separately:
 *   a' = a c - b s,  b' = a s + b c,  written back as bf16 (nearest even).
 * Row r sits at position start_pos + (r / rows_per_pos) % positions_per_seq (e.g. rows of
 * q or o [b][m][h][d]: rows_per_pos = h, positions_per_seq = m).
 */
int oracle_apply_rotary(uint16_t *x, int64_t rows, int row_len, int rd, int64_t rows_per_pos,
                        int64_t positions_per_seq, int64_t start_pos, const float *table, int64_t table_rows,
                        int inverse) {
    if (rows < 0 || rd <= 0 || rd % 2 != 0 || rd > row_len || rows_per_pos < 1 || positions_per_seq < 1)
        return -1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t pos = start_pos + (r / rows_per_pos) % positions_per_seq;
        if (pos < 0 || pos >= table_rows) return -1;
        uint16_t *v = x + r * row_len + (row_len - rd);
        for (int j = 0; j < rd / 2; ++j) {
            float a = bf16_bits_to_f32(v[2 * j]), bb = bf16_bits_to_f32(v[2 * j + 1]);
            float c = table[(pos * (rd / 2) + j) * 2], sn = table[(pos * (rd / 2) + j) * 2 + 1];
            if (inverse) sn = -sn;
            float ac = a * c, bs = bb * sn, as = a * sn, bc = bb * c;
            v[2 * j] = f32_to_bf16_bits(ac - bs);
            v[2 * j + 1] = f32_to_bf16_bits(as + bc);
        }
    }
    return 0;
}

/*
 * The ring write of a ratio-0 layer's new kv rows with their RoPE first ([attn] module text: RoPE
 * on the last rope_dim, then the fp8 round trip in place, then the ring): row t of the chunk is
 * at position start_pos + t.
 */
int oracle_kv_rope_quant_ring_write(uint16_t *kv, int64_t kv_bstride, uint16_t *ring, int64_t ring_bstride, int b,
                                    int s, int d, int64_t start_pos, int window, int rd, const float *table,
                                    int64_t table_rows) {
    if (b < 0 || s < 0 || d <= 0 || d % ORACLE_FP8_BLOCK != 0) return -1;
    for (int bi = 0; bi < b; ++bi)
        if (oracle_apply_rotary(kv + (int64_t)bi * kv_bstride, s, d, rd, 1, s, start_pos, table, table_rows, 0) != 0)
            return -1;
    return oracle_kv_quant_ring_write(kv, kv_bstride, ring, ring_bstride, b, s, d, start_pos, window);
}

/* ------------------------------------------------------------------------------------------ */
/* Indexer scoring and top-k  ([latent] Indexer.forward: the index score of every compressed   */
/* position, the causal compress_lens mask, top-k re-sorted by position, -1 and the offset)    */
/* ------------------------------------------------------------------------------------------ */

/*
 * For sequence bi and query i (position start_pos + i) over compressed positions t < T:
 *   score[t] = sum_h relu(dot(q[bi][i][h], k[bi][t])) * w[bi][i][h]      (f32, h and d in order)
 * q and k are taken as given: their RoPE and fp4 rounding happen before (the pages only name the
 * fp4 step), and w already holds the weights projection times softmax_scale * H^-0.5.
 * compress_lens = (start_pos + i + 1) / ratio (integer division): positions t >= compress_lens
 * are not visible yet (score -inf in the prefill; in a decode step T equals it).
 * kk = min(topk, (start_pos + s) / ratio) entries are kept: the kk largest scores, equal scores
 * by the smaller position first (the pages leave the order of ties open; this is one valid
 * choice), re-sorted by position; an entry t >= compress_lens becomes -1, the others t + offset.
 * idx_out[bi][i][0..kk), scores_out[bi][i][0..T) (optional).  Returns kk, or -1.
 */
static int cmp_desc_score(const void *pa, const void *pb, void *ctx) {
    const float *sc = (const float *)ctx;
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    if (sc[a] > sc[b]) return -1;
    if (sc[a] < sc[b]) return 1;
    return a < b ? -1 : (a > b ? 1 : 0);
}

static int cmp_i64(const void *pa, const void *pb) {
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    return a < b ? -1 : (a > b ? 1 : 0);
}

/* insertion sort with a context (qsort_r is not portable C11); the oracle's sizes are small */
static void sort_ctx(int64_t *v, int64_t n, int (*cmp)(const void *, const void *, void *), void *ctx) {
    for (int64_t i = 1; i < n; ++i) {
        int64_t x = v[i], j = i - 1;
        while (j >= 0 && cmp(&v[j], &x, ctx) > 0) {
            v[j + 1] = v[j];
            --j;
        }
        v[j + 1] = x;
    }
}

/* kk entries of one row of T scores: the kk largest (ties: smaller position first), by position */
static void select_row(const float *sc, int64_t *ord, int64_t T, int64_t lens, int64_t kk, int64_t offset,
                       int32_t *out) {
    for (int64_t t = 0; t < T; ++t) ord[t] = t;
    sort_ctx(ord, T, cmp_desc_score, (void *)sc);
    qsort(ord, (size_t)kk, sizeof(int64_t), cmp_i64);
    for (int64_t j = 0; j < kk; ++j) out[j] = ord[j] < lens ? (int32_t)(ord[j] + offset) : -1;
}

int oracle_indexer_topk(const uint16_t *q, const uint16_t *k, const float *w, int b, int s, int H, int D, int64_t T,
                        int64_t start_pos, int ratio, int topk, int64_t offset, float *scores_out, int32_t *idx_out) {
    if (b < 0 || s < 1 || H < 1 || D < 1 || T < 0 || start_pos < 0 || ratio < 1 || topk < 0) return -1;
    int64_t kk = (start_pos + s) / ratio;
    if (kk > topk) kk = topk;
    if (kk > T) return -1;
    float *sc = (float *)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
    int64_t *ord = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    if (!sc || !ord) {
        free(sc);
        free(ord);
        return -1;
    }
    for (int bi = 0; bi < b; ++bi) {
        for (int i = 0; i < s; ++i) {
            const int64_t lens = (start_pos + i + 1) / ratio;
            for (int64_t t = 0; t < T; ++t) {
                float acc = 0.0f;
                for (int h = 0; h < H; ++h) {
                    const uint16_t *qv = q + (((int64_t)bi * s + i) * H + h) * D;
                    const uint16_t *kv = k + ((int64_t)bi * T + t) * D;
                    float dot = 0.0f;
                    for (int d = 0; d < D; ++d) dot += bf16_bits_to_f32(qv[d]) * bf16_bits_to_f32(kv[d]);
                    float r = dot > 0.0f ? dot : 0.0f;
                    acc += r * w[((int64_t)bi * s + i) * H + h];
                }
                sc[t] = t < lens ? acc : -INFINITY;
                if (scores_out) scores_out[((int64_t)bi * s + i) * T + t] = sc[t];
            }
            select_row(sc, ord, T, lens, kk, offset, idx_out + ((int64_t)bi * s + i) * kk);
        }
    }
    free(sc);
    free(ord);
    return (int)kk;
}

/*
 * The selection alone, from given scores: row (bi, i) is scores[(bi * s + i) * ld + t] for
 * t < Tv = (start_pos + s) / ratio; positions t >= compress_lens count as -inf whatever the row
 * holds there.  The kept entries follow the rule above.  Returns kk, or -1.
 */
int oracle_indexer_select(const float *scores, int64_t ld, int b, int s, int64_t start_pos, int ratio, int topk,
                          int64_t offset, int32_t *idx_out) {
    if (b < 0 || s < 1 || start_pos < 0 || ratio < 1 || topk < 0) return -1;
    const int64_t Tv = (start_pos + s) / ratio;
    if (ld < Tv) return -1;
    const int64_t kk = topk < Tv ? topk : Tv;
    float *sc = (float *)malloc(sizeof(float) * (size_t)(Tv > 0 ? Tv : 1));
    int64_t *ord = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Tv > 0 ? Tv : 1));
    if (!sc || !ord) {
        free(sc);
        free(ord);
        return -1;
    }
    for (int bi = 0; bi < b; ++bi)
        for (int i = 0; i < s; ++i) {
            const int64_t lens = (start_pos + i + 1) / ratio;
            const float *row = scores + ((int64_t)bi * s + i) * ld;
            for (int64_t t = 0; t < Tv; ++t) sc[t] = t < lens ? row[t] : -INFINITY;
            select_row(sc, ord, Tv, lens, kk, offset, idx_out + ((int64_t)bi * s + i) * kk);
        }
    free(sc);
    free(ord);
    return (int)kk;
}

/* ------------------------------------------------------------------------------------------ */
/* sparse_attn  ([attn] sparse_attn and Precision; [attend] sparse_attn_kernel, wrapper)       */
/* ------------------------------------------------------------------------------------------ */

/*
 * For query token (bi, t) and head hh:
 *   s_j = scale * sum_c q[bi][t][hh][c] * kv[bi][idx_j][c]     for every entry idx_j >= 0
 *   M   = max(sink[hh], max_j s_j)                              (subtracted for range only)
 *   den = exp(sink[hh] - M) + sum_j exp(s_j - M)                the sink is in the denominator only
 *   o   = sum_j exp(s_j - M) / den * kv[bi][idx_j][:]           V is the same gathered row
 * Entries < 0 are skipped; a row with no entry >= 0 gives o = 0.  All arithmetic in f32 in the
 * order written, result rounded to bf16 (f32 variant) or kept as double (f64 variant).
 *
 * Layouts: q, o [b][m][h][d]; kv [b][n][d]; sink [h]; idx [b][m][topk]; all contiguous.
 * tokens: optional list of flattened token numbers bi*m + t to compute (NULL = all b*m); the
 * output then holds one [h][d] block per listed token, in list order.
 */
typedef struct {
    const uint16_t *q, *kv;
    int64_t n;
    const float *sink;
    const int32_t *idx;
    int topk;
    float scale;
    int b, m, h, d;
    const int64_t *tokens;
    int64_t ntok;
    uint16_t *o_bf16;     /* f32 variant */
    double *o_f64;        /* f64 variant */
    int thread_id, nthreads;
    int status;
} attn_job;

static void attn_token_f32(const attn_job *J, int64_t tok, int64_t out_slot, float *qf, float *sc, float *acc) {
    const int d = J->d, topk = J->topk;
    const int64_t bi = tok / J->m;
    const int32_t *irow = J->idx + tok * topk;
    const uint16_t *kvb = J->kv + bi * J->n * d;
    for (int hh = 0; hh < J->h; ++hh) {
        const uint16_t *qrow = J->q + (tok * J->h + hh) * (int64_t)d;
        for (int c = 0; c < d; ++c) qf[c] = bf16_bits_to_f32(qrow[c]);
        /* scores, and their maximum together with the sink */
        float M = J->sink[hh];
        for (int j = 0; j < topk; ++j) {
            if (irow[j] < 0) continue;
            const uint16_t *r = kvb + (int64_t)irow[j] * d;
            float dot = 0.0f;
            for (int c = 0; c < d; ++c) dot += qf[c] * bf16_bits_to_f32(r[c]);
            sc[j] = J->scale * dot;
            if (sc[j] > M) M = sc[j];
        }
        /* denominator: every gathered row plus the sink */
        float den = expf(J->sink[hh] - M);
        for (int j = 0; j < topk; ++j)
            if (irow[j] >= 0) den += expf(sc[j] - M);
        /* probabilities, then the weighted sum of the same gathered rows */
        for (int c = 0; c < d; ++c) acc[c] = 0.0f;
        for (int j = 0; j < topk; ++j) {
            if (irow[j] < 0) continue;
            float p = expf(sc[j] - M) / den;
            const uint16_t *r = kvb + (int64_t)irow[j] * d;
            for (int c = 0; c < d; ++c) acc[c] += p * bf16_bits_to_f32(r[c]);
        }
        uint16_t *orow = J->o_bf16 + (out_slot * J->h + hh) * (int64_t)d;
        for (int c = 0; c < d; ++c) orow[c] = f32_to_bf16_bits(acc[c]);
    }
}

static void attn_token_f64(const attn_job *J, int64_t tok, int64_t out_slot, double *qf, double *sc, double *acc) {
    const int d = J->d, topk = J->topk;
    const int64_t bi = tok / J->m;
    const int32_t *irow = J->idx + tok * topk;
    const uint16_t *kvb = J->kv + bi * J->n * d;
    for (int hh = 0; hh < J->h; ++hh) {
        const uint16_t *qrow = J->q + (tok * J->h + hh) * (int64_t)d;
        for (int c = 0; c < d; ++c) qf[c] = (double)bf16_bits_to_f32(qrow[c]);
        double M = (double)J->sink[hh];
        for (int j = 0; j < topk; ++j) {
            if (irow[j] < 0) continue;
            const uint16_t *r = kvb + (int64_t)irow[j] * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += qf[c] * (double)bf16_bits_to_f32(r[c]);
            sc[j] = (double)J->scale * dot;
            if (sc[j] > M) M = sc[j];
        }
        double den = exp((double)J->sink[hh] - M);
        for (int j = 0; j < topk; ++j)
            if (irow[j] >= 0) den += exp(sc[j] - M);
        for (int c = 0; c < d; ++c) acc[c] = 0.0;
        for (int j = 0; j < topk; ++j) {
            if (irow[j] < 0) continue;
            double p = exp(sc[j] - M) / den;
            const uint16_t *r = kvb + (int64_t)irow[j] * d;
            for (int c = 0; c < d; ++c) acc[c] += p * (double)bf16_bits_to_f32(r[c]);
        }
        double *orow = J->o_f64 + (out_slot * J->h + hh) * (int64_t)d;
        for (int c = 0; c < d; ++c) orow[c] = acc[c];
    }
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    int use64 = J->o_f64 != NULL;
    size_t es = use64 ? sizeof(double) : sizeof(float);
    void *qf = malloc((size_t)J->d * es);
    void *acc = malloc((size_t)J->d * es);
    void *sc = malloc((size_t)(J->topk > 0 ? J->topk : 1) * es);
    if (!qf || !sc || !acc) {
        J->status = -1;
    } else {
        for (int64_t k = J->thread_id; k < J->ntok; k += J->nthreads) {
            int64_t tok = J->tokens ? J->tokens[k] : k;
            if (use64) attn_token_f64(J, tok, k, (double *)qf, (double *)sc, (double *)acc);
            else attn_token_f32(J, tok, k, (float *)qf, (float *)sc, (float *)acc);
        }
    }
    free(qf);
    free(sc);
    free(acc);
    return NULL;
}

static int attn_run(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx,
                    int topk, float scale, int b, int m, int h, int d, const int64_t *tokens, int64_t ntok,
                    uint16_t *o_bf16, double *o_f64, int nthreads) {
    if (b < 0 || m < 0 || h <= 0 || d <= 0 || topk < 0 || n < 0) return -1;
    if (!tokens) ntok = (int64_t)b * m;
    for (int64_t k = 0; k < ntok; ++k) {       /* caller contract: every index < n */
        int64_t tok = tokens ? tokens[k] : k;
        if (tok < 0 || tok >= (int64_t)b * m) return -1;
        for (int j = 0; j < topk; ++j)
            if (idx[tok * topk + j] >= n) return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    attn_job jobs[256];
    pthread_t th[256];
    for (int i = 0; i < nthreads; ++i) {
        attn_job J = {q, kv, n, sink, idx, topk, scale, b, m, h, d, tokens, ntok, o_bf16, o_f64, i, nthreads, 0};
        jobs[i] = J;
    }
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, attn_worker, &jobs[i]) != 0) break;
        started = i;
    }
    if (started < nthreads - 1) {              /* could not start every thread: run serially */
        for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
        attn_job J = {q, kv, n, sink, idx, topk, scale, b, m, h, d, tokens, ntok, o_bf16, o_f64, 0, 1, 0};
        attn_worker(&J);
        return J.status;
    }
    attn_worker(&jobs[0]);
    int status = jobs[0].status;
    for (int i = 1; i < nthreads; ++i) {
        pthread_join(th[i], NULL);
        if (jobs[i].status) status = jobs[i].status;
    }
    return status;
}

int oracle_sparse_attn(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx,
                       int topk, float scale, uint16_t *o, int b, int m, int h, int d,
                       const int64_t *tokens, int64_t ntok, int nthreads) {
    return attn_run(q, kv, n, sink, idx, topk, scale, b, m, h, d, tokens, ntok, o, NULL, nthreads);
}

int oracle_sparse_attn_f64(const uint16_t *q, const uint16_t *kv, int64_t n, const float *sink, const int32_t *idx,
                           int topk, float scale, double *o, int b, int m, int h, int d,
                           const int64_t *tokens, int64_t ntok, int nthreads) {
    return attn_run(q, kv, n, sink, idx, topk, scale, b, m, h, d, tokens, ntok, NULL, o, nthreads);
}
