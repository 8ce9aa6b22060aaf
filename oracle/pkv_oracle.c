/*
 * pkv_oracle.c -- float64 CPU oracle for paged grouped-query decode attention
 * and for the per-step KV append into the page pool.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the CUDA
 * library in paged_kv_decode_16_gb300/.  Only the test suite, the smoke check
 * and the benchmark's CPU-baseline / reference leg load it.  It shares no code,
 * header, table or helper with the CUDA path and includes none of its files.
 *
 * What is computed, and where the pages define it
 * ------------------------------------------------
 *  Decode attention (one query token per sequence):
 *    CacheIR, "Compiler Example": in the decode graph the roped query and the
 *      cached keys/values feed paged_attention_decode.
 *    CacheIR, "Boundaries": multi-batch page-table decode attention with a GQA
 *      mapping; batched decode over shared page tables ("Current Capabilities",
 *      Runtime row).
 *    TorchInferno, "Runtime Scaffolds": runtime.paged is the page-table-shaped
 *      KV allocation and materialization; runtime.paged_attention is the paged
 *      causal attention reference.  "Custom Kernels": paged_decode_attention and
 *      batched_paged_decode_attention (one query token per request).
 *  The pages never print the formula.  The plain reading, used here, is scaled
 *  dot-product attention of the single query over every cached token of the
 *  sequence (the causal mask admits all of them), with no soft-cap, bias or
 *  window:
 *      s_t   = scale * sum_d q[d] * k_t[d]          t = 0 .. L-1
 *      out   = sum_t exp(s_t - M) v_t / sum_t exp(s_t - M),   M = max_t s_t
 *  Subtracting M changes no value (the factor exp(-M) cancels); it only keeps
 *  exp() finite.  L = 0 gives out = 0.
 *
 *  Token t of sequence b lives in physical page table[b][t / P], slot t % P.
 *  Pool layout [num_pages][n_kv_heads][P][D] (one contiguous block per page and
 *  KV head).  GQA: query head hq reads KV head hq / (n_q_heads / n_kv_heads),
 *  i.e. consecutive query heads share one KV head.
 *
 *  KV append (TorchInferno, "OpenAI-Compatible Serving" knob list: a KV-append
 *  kernel; CacheIR, "Compiler Example": the new token's K/V are written before
 *  paged_attention_decode runs): for every sequence with position p >= 0 the
 *  new row of every KV head is copied bit for bit into page table[b][p / P],
 *  slot p % P.  A negative position marks a padded batch slot that must not
 *  write anything (TorchInferno, "Quickstart": decode graphs were switched off
 *  because bucket padding let a dummy batch slot alias a live KV row).
 *
 *  Gather: materialise a sequence's cached K or V as a dense [Hkv][L][D] block
 *  by reading through the page table (TorchInferno, "Runtime Scaffolds",
 *  runtime.paged materialization).  Bit copy.
 *
 *  Rotary position embedding before the append (CacheIR, "Compiler Example":
 *  rope(q, k) produces the q and k that attention consumes; "Complete Tech
 *  Stack": Llama/Mistral/Qwen-style blocks with RoPE; TorchInferno,
 *  "OpenAI-Compatible Serving" knob list: a fused decode rotary + KV append
 *  kernel).  The pages print no formula.  The plain reading, used here, is the
 *  rotary embedding of those model families with the rotate-half pairing:
 *  element i of the first half of a head pairs with element i + D/2, and the
 *  pair is turned by the angle pos * theta^(-2i/D), i = 0 .. D/2-1:
 *      y_i       = x_i cos(a_i) - x_{i+D/2} sin(a_i)
 *      y_{i+D/2} = x_{i+D/2} cos(a_i) + x_i sin(a_i)
 *  with theta given by the caller and pos the token's position.  The rotated
 *  row is rounded to the storage format (round to nearest, ties to even).
 *
 * Precision: every product, sum and exp is in IEEE double.  fp16 / bf16 inputs
 * are decoded from their sign / exponent / fraction fields (IEEE 754 binary16,
 * and bfloat16 = the upper half of binary32), which is exact in double.
 *
 * Return codes: 0 ok, 1 invalid argument, 2 page id outside the pool,
 *               3 context length beyond the page-table row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_INVALID 1
#define ORC_BAD_PAGE 2
#define ORC_BAD_LEN 3

enum { ORC_F16 = 0, ORC_BF16 = 1 };

/* Decode a 16-bit float from its fields.  ebits exponent bits, mbits fraction
 * bits, bias 2^(ebits-1) - 1.  binary16: (5, 10); bfloat16: (8, 7). */
static double decode_fields(uint16_t bits, int ebits, int mbits) {
    const int sign = (bits >> 15) & 1;
    const int emax = (1 << ebits) - 1;
    const int bias = (1 << (ebits - 1)) - 1;
    const int e = (bits >> mbits) & emax;
    const int m = bits & ((1 << mbits) - 1);
    double mag;
    if (e == emax) {
        mag = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        /* subnormal: 0.m * 2^(1 - bias) */
        mag = ldexp((double)m, 1 - bias - mbits);
    } else {
        /* normal: 1.m * 2^(e - bias) */
        mag = ldexp((double)((1 << mbits) + m), e - bias - mbits);
    }
    return sign ? -mag : mag;
}

double pkv_oracle_decode_bits(uint16_t bits, int dtype) {
    return dtype == ORC_BF16 ? decode_fields(bits, 8, 7) : decode_fields(bits, 5, 10);
}

/* Encode x as a 16-bit float with ebits exponent and mbits fraction bits,
 * rounding to nearest with ties to even (IEEE 754 roundTiesToEven): find the
 * binade of |x|, express |x| in units of that binade's spacing (exact: a power
 * of two scale), round that to an integer, and carry into the exponent when
 * the rounding reaches the next binade.  Below the normal range the spacing is
 * that of the subnormals; beyond the largest finite value the result is inf.
 * NaN gives the quiet NaN with the sign kept. */
static uint16_t encode_fields(double x, int ebits, int mbits) {
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << (ebits + mbits)) : 0;
    const int bias = (1 << (ebits - 1)) - 1;
    const uint16_t exp_all = (uint16_t)(((1u << ebits) - 1) << mbits);
    if (isnan(x)) return (uint16_t)(sign | exp_all | (1u << (mbits - 1)));
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | exp_all);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;               /* a in [2^e, 2^(e+1)) */
    const int emin = 1 - bias;
    if (e < emin) {               /* subnormal: spacing 2^(emin - mbits) */
        const double r = nearbyint(ldexp(a, mbits - emin));
        /* r = 2^mbits lands on the smallest normal: the same bit pattern */
        return (uint16_t)(sign | (uint16_t)r);
    }
    double r = nearbyint(ldexp(a, mbits - e));   /* in [2^mbits, 2^(mbits+1)] */
    if (r == ldexp(1.0, mbits + 1)) {
        r = ldexp(1.0, mbits);
        e += 1;
    }
    if (e > bias) return (uint16_t)(sign | exp_all);  /* beyond the largest finite value */
    return (uint16_t)(sign | ((uint16_t)(e + bias) << mbits) | (uint16_t)(r - ldexp(1.0, mbits)));
}

static uint16_t encode_dtype(double x, int dtype) {
    return dtype == ORC_F16 ? encode_fields(x, 5, 10) : encode_fields(x, 8, 7);
}

/* Encode n doubles (used by the tests to pin the encoder). */
int pkv_oracle_encode_array(const double* x, int64_t n, int dtype, uint16_t* out) {
    if (!x || !out || n < 0 || (dtype != ORC_F16 && dtype != ORC_BF16)) return ORC_INVALID;
    for (int64_t i = 0; i < n; ++i) out[i] = encode_dtype(x[i], dtype);
    return ORC_OK;
}

/*
 * Rotary embedding of rows x [batch][heads][head_dim] at positions[b] (every
 * head of sequence b turns by the same angles), theta > 0, head_dim even.
 * out: the rotated rows rounded to dtype; out_f64 (nullable): the same rows
 * before rounding.
 */
int pkv_oracle_rope(const uint16_t* x, const int32_t* positions, int batch, int heads,
                    int head_dim, double theta, int dtype, uint16_t* out, double* out_f64) {
    if (!x || !positions || !out || batch < 0 || heads <= 0 || head_dim <= 0 ||
        head_dim % 2 || !(theta > 0.0) || (dtype != ORC_F16 && dtype != ORC_BF16))
        return ORC_INVALID;
    const int half = head_dim / 2;
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < heads; ++h) {
            const int64_t row = ((int64_t)b * heads + h) * head_dim;
            for (int i = 0; i < half; ++i) {
                const double ang = (double)positions[b] * pow(theta, -2.0 * i / head_dim);
                const double c = cos(ang), sn = sin(ang);
                const double x0 = pkv_oracle_decode_bits(x[row + i], dtype);
                const double x1 = pkv_oracle_decode_bits(x[row + half + i], dtype);
                const double y0 = x0 * c - x1 * sn;
                const double y1 = x1 * c + x0 * sn;
                if (out_f64) {
                    out_f64[row + i] = y0;
                    out_f64[row + half + i] = y1;
                }
                out[row + i] = encode_dtype(y0, dtype);
                out[row + half + i] = encode_dtype(y1, dtype);
            }
        }
    }
    return ORC_OK;
}

/*
 * Per-head RMS normalisation of q or k before the rotary embedding (the
 * Q/K-normalised decoders of Experimental LibTorch prefix cache, "Current
 * execution limits": normalised keys written straight into the attention
 * arenas).  Row x of head_dim elements becomes
 *     n_d = x_d * w_d / sqrt(mean_d(x_d^2) + eps),
 * which is then turned exactly as pkv_oracle_rope turns its rows, at
 * positions[b]; one rounding to the storage format at the end.  w (16-bit
 * patterns, head_dim of them) is shared by every head.
 */
int pkv_oracle_norm_rope(const uint16_t* x, const int32_t* positions, int batch, int heads,
                         int head_dim, const uint16_t* w, double eps, double theta, int dtype,
                         uint16_t* out, double* out_f64) {
    if (!x || !positions || !w || !out || batch < 0 || heads <= 0 || head_dim <= 0 ||
        head_dim % 2 || !(theta > 0.0) || !(eps >= 0.0) ||
        (dtype != ORC_F16 && dtype != ORC_BF16))
        return ORC_INVALID;
    const int half = head_dim / 2;
    double* n = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!n) return ORC_INVALID;
    for (int b = 0; b < batch; ++b) {
        for (int h = 0; h < heads; ++h) {
            const int64_t row = ((int64_t)b * heads + h) * head_dim;
            double ss = 0.0;
            for (int d = 0; d < head_dim; ++d) {
                const double v = pkv_oracle_decode_bits(x[row + d], dtype);
                ss += v * v;
            }
            const double inv_rms = 1.0 / sqrt(ss / head_dim + eps);
            for (int d = 0; d < head_dim; ++d)
                n[d] = pkv_oracle_decode_bits(x[row + d], dtype) * inv_rms *
                       pkv_oracle_decode_bits(w[d], dtype);
            for (int i = 0; i < half; ++i) {
                const double ang = (double)positions[b] * pow(theta, -2.0 * i / head_dim);
                const double c = cos(ang), sn = sin(ang);
                const double y0 = n[i] * c - n[half + i] * sn;
                const double y1 = n[half + i] * c + n[i] * sn;
                if (out_f64) {
                    out_f64[row + i] = y0;
                    out_f64[row + half + i] = y1;
                }
                out[row + i] = encode_dtype(y0, dtype);
                out[row + half + i] = encode_dtype(y1, dtype);
            }
        }
    }
    free(n);
    return ORC_OK;
}

/* Decode n elements (used by the tests to pin the decoder). */
int pkv_oracle_decode_array(const uint16_t* bits, int64_t n, int dtype, double* out) {
    if (!bits || !out || n < 0 || (dtype != ORC_F16 && dtype != ORC_BF16)) return ORC_INVALID;
    for (int64_t i = 0; i < n; ++i) out[i] = pkv_oracle_decode_bits(bits[i], dtype);
    return ORC_OK;
}

typedef struct {
    const uint16_t* q;
    const uint16_t* k_pool;
    const uint16_t* v_pool;
    int dtype;
    const int32_t* table;
    int table_stride;
    const int32_t* lens;
    int batch, n_q_heads, n_kv_heads, head_dim, page_size, num_pages;
    double scale;
} decode_args;

static int check_decode_args(const decode_args* a) {
    if (!a->q || !a->k_pool || !a->v_pool || !a->table || !a->lens) return ORC_INVALID;
    if (a->dtype != ORC_F16 && a->dtype != ORC_BF16) return ORC_INVALID;
    if (a->batch < 0 || a->n_q_heads <= 0 || a->n_kv_heads <= 0 || a->head_dim <= 0 ||
        a->page_size <= 0 || a->num_pages < 0 || a->table_stride < 0)
        return ORC_INVALID;
    if (a->n_q_heads % a->n_kv_heads != 0) return ORC_INVALID;
    return ORC_OK;
}

/* One output row: sequence b, query head hq.  out_row has head_dim doubles. */
/* One output row: query row qsel (NULL: row (b, hq) of a->q) of sequence b
 * over the first n_att of its tokens (n_att < 0: all of them). */
static int decode_row_at(const decode_args* a, int b, int hq, const uint16_t* qsel, int n_att,
                         double* out_row) {
    const int D = a->head_dim, P = a->page_size;
    const int group = a->n_q_heads / a->n_kv_heads;
    const int hkv = hq / group; /* consecutive query heads share a KV head */
    const int Lseq = a->lens[b];
    for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    if (Lseq < 0) return ORC_BAD_LEN;
    if ((int64_t)Lseq > (int64_t)a->table_stride * P) return ORC_BAD_LEN;
    const int L = n_att < 0 ? Lseq : (n_att < Lseq ? n_att : Lseq);  /* tokens attended */
    if (L <= 0) return ORC_OK;

    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    if (!qd || !s) { free(qd); free(s); return ORC_INVALID; }
    const uint16_t* qrow = qsel ? qsel : a->q + ((int64_t)b * a->n_q_heads + hq) * D;
    for (int d = 0; d < D; ++d) qd[d] = pkv_oracle_decode_bits(qrow[d], a->dtype);

    int rc = ORC_OK;
    /* scores s_t = scale * q . k_t */
    for (int t = 0; t < L && rc == ORC_OK; ++t) {
        const int32_t page = a->table[(int64_t)b * a->table_stride + t / P];
        if (page < 0 || page >= a->num_pages) { rc = ORC_BAD_PAGE; break; }
        const uint16_t* krow =
            a->k_pool + (((int64_t)page * a->n_kv_heads + hkv) * P + (t % P)) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qd[d] * pkv_oracle_decode_bits(krow[d], a->dtype);
        s[t] = a->scale * dot;
    }
    if (rc == ORC_OK) {
        double M = s[0];
        for (int t = 1; t < L; ++t) if (s[t] > M) M = s[t];
        double den = 0.0;
        for (int t = 0; t < L; ++t) {
            const int32_t page = a->table[(int64_t)b * a->table_stride + t / P];
            const uint16_t* vrow =
                a->v_pool + (((int64_t)page * a->n_kv_heads + hkv) * P + (t % P)) * D;
            const double w = exp(s[t] - M);
            den += w;
            for (int d = 0; d < D; ++d) out_row[d] += w * pkv_oracle_decode_bits(vrow[d], a->dtype);
        }
        for (int d = 0; d < D; ++d) out_row[d] /= den;
    } else {
        for (int d = 0; d < D; ++d) out_row[d] = 0.0;
    }
    free(qd);
    free(s);
    return rc;
}

static int decode_row(const decode_args* a, int b, int hq, double* out_row) {
    return decode_row_at(a, b, hq, NULL, -1, out_row);
}

/*
 * Several query tokens per sequence (speculative or suffix decoding).  The
 * n_queries new tokens of sequence b are its last ones, so query j stands at
 * position L - n_queries + j and, causally, attends to tokens
 * t = 0 .. L - n_queries + j (its own and every earlier one).
 * q and out [batch][n_queries][n_q_heads][head_dim].  A query with no token
 * to attend to (L < n_queries - j) gives zeros.
 */
int pkv_oracle_paged_decode_multi(const uint16_t* q, const uint16_t* k_pool,
                                  const uint16_t* v_pool, int dtype, const int32_t* table,
                                  int table_stride, const int32_t* lens, int batch, int n_queries,
                                  int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                                  int num_pages, double scale, double* out) {
    decode_args a = {q, k_pool, v_pool, dtype, table, table_stride, lens, batch, n_q_heads,
                     n_kv_heads, head_dim, page_size, num_pages, scale};
    int rc = check_decode_args(&a);
    if (rc != ORC_OK || !out || n_queries <= 0) return rc != ORC_OK ? rc : ORC_INVALID;
    const int64_t rows = (int64_t)batch * n_queries * n_q_heads;
    int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r) {
        const int hq = (int)(r % n_q_heads);
        const int j = (int)((r / n_q_heads) % n_queries);
        const int b = (int)(r / ((int64_t)n_q_heads * n_queries));
        const uint16_t* qsel = q + r * head_dim;  /* row (b, j, hq) */
        const int n_att = lens[b] - n_queries + j + 1;
        /* before the first token (n_att <= 0) the query sees nothing: zeros */
        const int e = decode_row_at(&a, b, hq, qsel, n_att > 0 ? n_att : 0, out + r * head_dim);
        if (e != ORC_OK) {
#pragma omp critical
            err = e;
        }
    }
    return err;
}

/*
 * Full decode: out[b][hq][d] for every sequence and query head, as double.
 * q [batch][n_q_heads][head_dim]; k_pool, v_pool [num_pages][n_kv_heads]
 * [page_size][head_dim]; table [batch][table_stride]; lens [batch].
 */
int pkv_oracle_paged_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                            int dtype, const int32_t* table, int table_stride,
                            const int32_t* lens, int batch, int n_q_heads, int n_kv_heads,
                            int head_dim, int page_size, int num_pages, double scale,
                            double* out) {
    decode_args a = {q, k_pool, v_pool, dtype, table, table_stride, lens,
                     batch, n_q_heads, n_kv_heads, head_dim, page_size, num_pages, scale};
    int rc = check_decode_args(&a);
    if (rc != ORC_OK || !out) return rc != ORC_OK ? rc : ORC_INVALID;
    const int64_t rows = (int64_t)batch * n_q_heads;
    int worst = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1) reduction(max : worst)
    for (int64_t r = 0; r < rows; ++r) {
        const int b = (int)(r / n_q_heads), hq = (int)(r % n_q_heads);
        const int rr = decode_row(&a, b, hq, out + r * head_dim);
        if (rr > worst) worst = rr;
    }
    return worst;
}

/*
 * Selected rows only: rows[2*i] = b, rows[2*i+1] = hq; out [n_rows][head_dim].
 * Lets a test check sampled outputs of a workload too large to recompute whole.
 */
int pkv_oracle_paged_decode_rows(const uint16_t* q, const uint16_t* k_pool,
                                 const uint16_t* v_pool, int dtype, const int32_t* table,
                                 int table_stride, const int32_t* lens, int batch,
                                 int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                                 int num_pages, double scale, const int32_t* rows, int n_rows,
                                 double* out) {
    decode_args a = {q, k_pool, v_pool, dtype, table, table_stride, lens,
                     batch, n_q_heads, n_kv_heads, head_dim, page_size, num_pages, scale};
    int rc = check_decode_args(&a);
    if (rc != ORC_OK) return rc;
    if (!rows || !out || n_rows < 0) return ORC_INVALID;
    for (int i = 0; i < n_rows; ++i) {
        if (rows[2 * i] < 0 || rows[2 * i] >= batch || rows[2 * i + 1] < 0 ||
            rows[2 * i + 1] >= n_q_heads)
            return ORC_INVALID;
    }
    int worst = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1) reduction(max : worst)
    for (int i = 0; i < n_rows; ++i) {
        const int rr = decode_row(&a, rows[2 * i], rows[2 * i + 1], out + (int64_t)i * head_dim);
        if (rr > worst) worst = rr;
    }
    return worst;
}

/*
 * KV append: k_new, v_new [batch][n_kv_heads][head_dim] are copied bit for bit
 * into slot positions[b] % P of page table[b][positions[b] / P].  Negative
 * positions skip the sequence.  Pools are modified in place.
 */
int pkv_oracle_kv_append(uint16_t* k_pool, uint16_t* v_pool, const uint16_t* k_new,
                         const uint16_t* v_new, const int32_t* table, int table_stride,
                         const int32_t* positions, int batch, int n_kv_heads, int head_dim,
                         int page_size, int num_pages) {
    if (!k_pool || !v_pool || !k_new || !v_new || !table || !positions) return ORC_INVALID;
    if (batch < 0 || n_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages < 0 ||
        table_stride < 0)
        return ORC_INVALID;
    /* validate everything first so that a bad entry leaves the pools untouched */
    for (int b = 0; b < batch; ++b) {
        const int32_t p = positions[b];
        if (p < 0) continue;
        if (p / page_size >= table_stride) return ORC_BAD_LEN;
        const int32_t page = table[(int64_t)b * table_stride + p / page_size];
        if (page < 0 || page >= num_pages) return ORC_BAD_PAGE;
    }
    for (int b = 0; b < batch; ++b) {
        const int32_t p = positions[b];
        if (p < 0) continue;
        const int32_t page = table[(int64_t)b * table_stride + p / page_size];
        for (int h = 0; h < n_kv_heads; ++h) {
            const int64_t dst = (((int64_t)page * n_kv_heads + h) * page_size + p % page_size) * head_dim;
            const int64_t src = ((int64_t)b * n_kv_heads + h) * head_dim;
            memcpy(k_pool + dst, k_new + src, sizeof(uint16_t) * (size_t)head_dim);
            memcpy(v_pool + dst, v_new + src, sizeof(uint16_t) * (size_t)head_dim);
        }
    }
    return ORC_OK;
}

/*
 * Gather (materialisation): dense[b][h][t][d] = pool[table[b][t/P]][h][t%P][d]
 * for t < lens[b]; entries with t >= lens[b] are left as they are.
 * dense is [batch][n_kv_heads][max_len][head_dim].
 */
int pkv_oracle_gather(const uint16_t* pool, const int32_t* table, int table_stride,
                      const int32_t* lens, int batch, int n_kv_heads, int head_dim,
                      int page_size, int num_pages, int max_len, uint16_t* dense) {
    if (!pool || !table || !lens || !dense) return ORC_INVALID;
    if (batch < 0 || n_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || max_len < 0)
        return ORC_INVALID;
    for (int b = 0; b < batch; ++b) {
        const int L = lens[b];
        if (L < 0 || L > max_len || (int64_t)L > (int64_t)table_stride * page_size) return ORC_BAD_LEN;
        for (int t = 0; t < L; ++t) {
            const int32_t page = table[(int64_t)b * table_stride + t / page_size];
            if (page < 0 || page >= num_pages) return ORC_BAD_PAGE;
            for (int h = 0; h < n_kv_heads; ++h) {
                const int64_t src = (((int64_t)page * n_kv_heads + h) * page_size + t % page_size) * head_dim;
                const int64_t dst = (((int64_t)b * n_kv_heads + h) * max_len + t) * head_dim;
                memcpy(dense + dst, pool + src, sizeof(uint16_t) * (size_t)head_dim);
            }
        }
    }
    return ORC_OK;
}

int pkv_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int pkv_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
