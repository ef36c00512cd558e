/*
 * uly_oracle.c -- plain, slow CPU oracle for the Ulysses attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only on the bytes of seeded synthetic inputs.
 *
 * What it computes (all citations are to the source pages by title):
 *
 *  - orc_to_heads / orc_to_seq: the Ulysses sequence<->head exchange written
 *    as an explicit per-element index map.  The all-to-all is a pure
 *    permutation of bytes ("Add head-group pipelined Ulysses exchange",
 *    sglang PR #43521, section "First-sight check": the exchange's bytes do
 *    not depend on the transport), so the oracle moves bytes and never
 *    interprets them.  The map follows
 *      * flashdreams core/attention/cp.py, ContextParallelAttention.
 *        _impl_ulysses (rank r receives heads [r*H/P,(r+1)*H/P) of every
 *        shard, gathered sender-rank-major along the sequence), and
 *      * sglang multimodal_gen attention/layer.py, USPAttention.
 *        _forward_with_replicated_prefix / _suffix / _kv_prefix (replicated
 *        rows stay out of the all-to-all, each rank head-slices its own copy,
 *        prefix rows go before the gathered rows, suffix rows after them in
 *        "tail order", and the replicated output is gathered over heads so
 *        every shard gets all heads of those rows).
 *
 *  - orc_attention: non-causal scaled-dot-product attention in fp64 by its
 *    plain definition (sglang layer.py, LocalAttention.forward: softmax of
 *    scale*q.k over the keys the mask admits, weights times V; GQA maps
 *    q head h to kv head h / (Hq/Hkv), the repeat_interleave of the same
 *    function).  Masked keys are excluded exactly instead of through the
 *    finite -finfo.max bias; a query with no admitted key returns 0.
 *    fp8 e4m3 inputs are decoded from the OCP FP8 definition (bias 7, three
 *    mantissa bits, subnormals, S.1111.111 = NaN) and multiplied by their
 *    per-head scale before the dot product (LightX2V PR #1235: the fp8
 *    payload travels with a separate scale tensor).
 *
 * Every function is pinned by the tests against facts that do not come from
 * this file: closed forms, a hand-worked 2x2 case, invariants (round trip,
 * P=1 identity, iota images, key-permutation invariance, masked-key
 * invariance), torch's own float8 decode and torch's fp64 SDPA.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_REP_NONE = 0, ORC_REP_PREFIX = 1, ORC_REP_SUFFIX = 2, ORC_REP_KV_PREFIX = 3 };
enum { ORC_BF16 = 0, ORC_E4M3 = 1, ORC_F64 = 2 };

/* Shape of one Ulysses exchange: B batches, P virtual ranks, S_l image rows
 * per shard, R replicated rows, rep mode, Hq/Hkv heads, head dim D; lens,
 * when not NULL, gives each shard's own number of image rows (uneven
 * shards: sglang layer.py passes seq_lens to _usp_input_all_to_all_varlen)
 * and S_l is then unused. */
typedef struct {
    int32_t B, P, S_l, R, mode, Hq, Hkv, D;
    const int32_t *lens;
} orc_shape;

/* ---------------------------------------------------------------- sizes -- */

/* Image rows of shard p, and the image rows of the shards before it. */
static int64_t img_len(const orc_shape *s, int p) { return s->lens ? s->lens[p] : s->S_l; }
static int64_t img_off(const orc_shape *s, int p)
{
    int64_t o = 0;
    for (int q = 0; q < p; ++q) o += img_len(s, q);
    return o;
}

/* Rows shard p holds for q (is_kv=0) or k/v (is_kv=1). */
int64_t orc_shard_rows_p(const orc_shape *s, int p, int is_kv)
{
    const int64_t L = img_len(s, p);
    switch (s->mode) {
    case ORC_REP_NONE: return L;
    case ORC_REP_PREFIX:
    case ORC_REP_SUFFIX: return (int64_t)s->R + L;
    case ORC_REP_KV_PREFIX: return is_kv ? (int64_t)s->R + L : L;
    }
    return -1;
}

/* Rows every shard holds (even shards). */
int64_t orc_shard_rows(const orc_shape *s, int is_kv) { return orc_shard_rows_p(s, 0, is_kv); }

/* Rows of the head-sharded (gathered) sequence each rank attends over. */
int64_t orc_heads_rows(const orc_shape *s, int is_kv)
{
    int64_t img = img_off(s, s->P);
    switch (s->mode) {
    case ORC_REP_NONE: return img;
    case ORC_REP_PREFIX:
    case ORC_REP_SUFFIX: return img + s->R;
    case ORC_REP_KV_PREFIX: return is_kv ? img + s->R : img;
    }
    return -1;
}

/* 0 when the shape is one the pages accept (heads divisible by the number of
 * ranks, q heads a multiple of kv heads, replicated rows only with a mode). */
int orc_check(const orc_shape *s)
{
    if (s->B < 1 || s->P < 1 || s->S_l < 0 || s->R < 0 || s->D < 1) return 1;
    if (s->lens)
        for (int p = 0; p < s->P; ++p)
            if (s->lens[p] < 0) return 1;
    if (s->Hq < 1 || s->Hkv < 1) return 1;
    if (s->Hq % s->P || s->Hkv % s->P) return 1;
    if (s->Hq % s->Hkv) return 1;
    if (s->mode < ORC_REP_NONE || s->mode > ORC_REP_KV_PREFIX) return 1;
    if (s->mode == ORC_REP_NONE && s->R != 0) return 1;
    if (s->mode != ORC_REP_NONE && s->R < 1) return 1;
    return 0;
}

/* ------------------------------------------------------------ index map -- */

/* Shard holding image row i of the global sequence (shards in rank order). */
static int img_shard(const orc_shape *s, int64_t i)
{
    int p = 0;
    while (p + 1 < s->P && i >= img_off(s, p + 1)) ++p;
    return p;
}

/* Source of row n of rank r's gathered sequence: which shard holds it and at
 * which of its rows.  Image row i of the global sequence lives in the shard
 * whose image rows cover it (rows are gathered in rank order); a replicated
 * row is taken from rank r's own shard. */
void orc_src_row(const orc_shape *s, int is_kv, int r, int64_t n, int32_t *shard, int64_t *row)
{
    int64_t img = img_off(s, s->P);
    int has_prefix = (s->mode == ORC_REP_PREFIX) || (s->mode == ORC_REP_KV_PREFIX && is_kv);
    int has_suffix = (s->mode == ORC_REP_SUFFIX);
    if (has_prefix) {
        if (n < s->R) { *shard = r; *row = n; return; }
        int64_t i = n - s->R;
        int p = img_shard(s, i);
        *shard = p;
        *row = s->R + (i - img_off(s, p));
        return;
    }
    if (has_suffix && n >= img) {
        *shard = r;
        *row = img_len(s, r) + (n - img);
        return;
    }
    int p = img_shard(s, n);
    *shard = p;
    *row = n - img_off(s, p);
}

/* Inverse direction for outputs: the gathered row that shard p's output row
 * `row` comes back from.  Replicated rows map to the same gathered row for
 * every shard (the head all-gather gives each shard every head of them). */
int64_t orc_out_row(const orc_shape *s, int p, int64_t row)
{
    int64_t img = img_off(s, s->P);
    if (s->mode == ORC_REP_PREFIX) {
        if (row < s->R) return row;
        return s->R + img_off(s, p) + (row - s->R);
    }
    if (s->mode == ORC_REP_SUFFIX) {
        if (row >= img_len(s, p)) return img + (row - img_len(s, p));
        return img_off(s, p) + row;
    }
    return img_off(s, p) + row;
}

/* Seq-sharded -> head-sharded.  src[p] is shard p's [B, rows_shard, H, D]
 * tensor, dst[r] is rank r's [B, rows_heads, H/P, D] tensor; elements are
 * `esize` opaque bytes.  Literal loops over (r, b, n, j, d). */
int orc_to_heads(const orc_shape *s, int is_kv, int esize, const void *const *src, void *const *dst)
{
    if (orc_check(s)) return 1;
    const int H = is_kv ? s->Hkv : s->Hq;
    const int Hl = H / s->P;
    const int64_t N = orc_heads_rows(s, is_kv);
    for (int r = 0; r < s->P; ++r)
        for (int b = 0; b < s->B; ++b)
            for (int64_t n = 0; n < N; ++n) {
                int32_t p;
                int64_t row;
                orc_src_row(s, is_kv, r, n, &p, &row);
                const int64_t Rs = orc_shard_rows_p(s, p, is_kv);
                for (int j = 0; j < Hl; ++j)
                    for (int d = 0; d < s->D; ++d) {
                        int64_t di = (((int64_t)b * N + n) * Hl + j) * s->D + d;
                        int64_t si = (((int64_t)b * Rs + row) * H + (int64_t)r * Hl + j) * s->D + d;
                        memcpy((char *)dst[r] + di * esize, (const char *)src[p] + si * esize, (size_t)esize);
                    }
            }
    return 0;
}

/* Head-sharded -> seq-sharded for the attention output (q-shaped).  src[r]
 * is rank r's [B, rows_heads(q), Hq/P, D]; dst[p] is shard p's
 * [B, rows_shard(q), Hq, D].  Head h of every output row comes from rank
 * h / (Hq/P), local head h % (Hq/P). */
int orc_to_seq(const orc_shape *s, int esize, const void *const *src, void *const *dst)
{
    if (orc_check(s)) return 1;
    const int H = s->Hq;
    const int Hl = H / s->P;
    const int64_t N = orc_heads_rows(s, 0);
    for (int p = 0; p < s->P; ++p) {
        const int64_t Rs = orc_shard_rows_p(s, p, 0);
        for (int b = 0; b < s->B; ++b)
            for (int64_t row = 0; row < Rs; ++row) {
                int64_t n = orc_out_row(s, p, row);
                for (int h = 0; h < H; ++h) {
                    int r = h / Hl, j = h % Hl;
                    for (int d = 0; d < s->D; ++d) {
                        int64_t di = (((int64_t)b * Rs + row) * H + h) * s->D + d;
                        int64_t si = (((int64_t)b * N + n) * Hl + j) * s->D + d;
                        memcpy((char *)dst[p] + di * esize, (const char *)src[r] + si * esize, (size_t)esize);
                    }
                }
            }
    }
    return 0;
}

/* ------------------------------------------------------------- decoding -- */

/* bf16: the upper 16 bits of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent 0 is subnormal (2^-6 * m/8); S.1111.111 is NaN and
 * there is no infinity. */
double orc_e4m3_to_f64(uint8_t x)
{
    int sgn = (x >> 7) & 1, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

static double load_elem(const void *base, int64_t i, int dtype)
{
    switch (dtype) {
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t *)base)[i]);
    case ORC_E4M3: return orc_e4m3_to_f64(((const uint8_t *)base)[i]);
    default: return ((const double *)base)[i];
    }
}

/* ------------------------------------------------------------ attention -- */

/*
 * Attention over one gathered problem:
 *   q [B, Nq, Hq, D], k/v [B, Nk, Hkv, D] of `dtype`;
 *   key_mask [B, Nk] (nonzero = key admitted) or NULL (all admitted);
 *   q_scale[Hq], k_scale[Hkv], v_scale[Hkv] multiply the decoded values (NULL
 *   means 1);
 *   zero_masked_rows: 1 = query row n is written as 0 if the key at the same
 *   token (n + q_key_offset) is masked -- the zero-fill convention of
 *   sglang's varlen fast path (USPAttention.forward docstring: masked query
 *   rows read as zeros); 2 = masked query rows attend only to the masked
 *   keys and admitted rows only to the admitted keys (the masked rows as a
 *   varlen segment of their own, LightX2V PR #1235); 0 = every row attends
 *   to the admitted keys;
 *   sel: NULL for every (b, n, h) -> out [B, Nq, Hq, D]; otherwise n_sel
 *   triples (b, n, h) -> out [n_sel, D].
 * Per query:  s_m = scale * sum_d q_d k_md  over admitted m;
 *             o = sum_m exp(s_m - max s) v_m / sum_m exp(s_m - max s).
 * Returns the number of threads used.
 */
int orc_attention_lse(int B, int Nq, int Nk, int Hq, int Hkv, int D, int dtype,
                      const void *q, const void *k, const void *v,
                      const uint8_t *key_mask, double scale,
                      const float *q_scale, const float *k_scale, const float *v_scale,
                      int zero_masked_rows, int q_key_offset,
                      int64_t n_sel, const int32_t *sel, double *out, double *lse);

int orc_attention(int B, int Nq, int Nk, int Hq, int Hkv, int D, int dtype,
                  const void *q, const void *k, const void *v,
                  const uint8_t *key_mask, double scale,
                  const float *q_scale, const float *k_scale, const float *v_scale,
                  int zero_masked_rows, int q_key_offset,
                  int64_t n_sel, const int32_t *sel, double *out)
{
    return orc_attention_lse(B, Nq, Nk, Hq, Hkv, D, dtype, q, k, v, key_mask, scale, q_scale, k_scale, v_scale,
                             zero_masked_rows, q_key_offset, n_sel, sel, out, NULL);
}

/* As orc_attention, and when lse is not NULL also the log-sum-exp of each
 * query's admitted scores, lse = ln sum_m exp(s_m) = max s + ln sum_m
 * exp(s_m - max s) (the compute_log_sumexp output of the SDPA calls in
 * flashdreams cp.py), -inf for a query with no admitted key or one written
 * as zero; one value per output row ([B, Nq, Hq] or [n_sel]). */
int orc_attention_lse(int B, int Nq, int Nk, int Hq, int Hkv, int D, int dtype,
                      const void *q, const void *k, const void *v,
                      const uint8_t *key_mask, double scale,
                      const float *q_scale, const float *k_scale, const float *v_scale,
                      int zero_masked_rows, int q_key_offset,
                      int64_t n_sel, const int32_t *sel, double *out, double *lse)
{
    const int G = Hq / Hkv;
    const int64_t total = sel ? n_sel : (int64_t)B * Nq * Hq;
    int used = 1;
#ifdef _OPENMP
    used = omp_get_max_threads();
#endif
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < total; ++t) {
            int b, n, h;
            double *o;
            if (sel) {
                b = sel[3 * t];
                n = sel[3 * t + 1];
                h = sel[3 * t + 2];
                o = out + t * D;
            } else {
                h = (int)(t % Hq);
                n = (int)((t / Hq) % Nq);
                b = (int)(t / ((int64_t)Hq * Nq));
                o = out + t * D;
            }
            const int hk = h / G;
            const double sq = q_scale ? q_scale[h] : 1.0;
            const double sk = k_scale ? k_scale[hk] : 1.0;
            const double sv = v_scale ? v_scale[hk] : 1.0;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            if (lse) lse[t] = -INFINITY;
            /* the query's own token: admitted or masked (for the zero-fill and
             * separate-segment conventions) */
            int row_valid = 1;
            if (key_mask) {
                int64_t kp = (int64_t)n + q_key_offset;
                if (kp >= 0 && kp < Nk) row_valid = key_mask[(int64_t)b * Nk + kp] != 0;
            }
            if (zero_masked_rows == 1 && !row_valid) continue;
            /* zero_masked_rows == 2: masked query rows form a sequence of their
             * own (LightX2V PR #1235 cu_seqlens builders: the masked text rows
             * are a separate varlen segment): a query attends to the keys whose
             * admission equals its own token's */
            const int self_seg = zero_masked_rows == 2 && key_mask;
            const int64_t qi = (((int64_t)b * Nq + n) * Hq + h) * D;
            for (int d = 0; d < D; ++d)
                qd[d] = sq * load_elem(q, qi + d, dtype);
            /* scores of admitted keys and their maximum */
            double mx = -INFINITY;
            int any = 0;
            for (int m = 0; m < Nk; ++m) {
                if (key_mask && (self_seg ? ((key_mask[(int64_t)b * Nk + m] != 0) != row_valid)
                                          : !key_mask[(int64_t)b * Nk + m])) continue;
                const int64_t ki = (((int64_t)b * Nk + m) * Hkv + hk) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d)
                    acc += qd[d] * (sk * load_elem(k, ki + d, dtype));
                sc[m] = scale * acc;
                if (sc[m] > mx) mx = sc[m];
                any = 1;
            }
            if (!any) continue; /* no admitted key: output 0 */
            double l = 0.0;
            for (int m = 0; m < Nk; ++m) {
                if (key_mask && (self_seg ? ((key_mask[(int64_t)b * Nk + m] != 0) != row_valid)
                                          : !key_mask[(int64_t)b * Nk + m])) continue;
                const double pm = exp(sc[m] - mx);
                l += pm;
                const int64_t vi = (((int64_t)b * Nk + m) * Hkv + hk) * D;
                for (int d = 0; d < D; ++d)
                    o[d] += pm * (sv * load_elem(v, vi + d, dtype));
            }
            for (int d = 0; d < D; ++d)
                o[d] /= l;
            if (lse) lse[t] = mx + log(l);
        }
        free(sc);
        free(qd);
    }
    return used;
}

/* Merge two attention results over disjoint key sets of the same queries
 * (ring attention, flashdreams cp.py ContextParallelAttention._impl_ring):
 *   out = prev_out - sigmoid(lse - prev_lse) * (prev_out - out)
 *   lse = prev_lse - logsigmoid(prev_lse - lse)
 * per row of D values.  A part with lse = -inf (no admitted key) leaves the
 * other unchanged; the formula's 0*inf and inf-inf are resolved that way
 * (its limit). o_* are [rows, D], lse_* are [rows]; results may overwrite
 * the "prev" inputs. */
void orc_lse_merge(int64_t rows, int D, const double *prev_out, const double *prev_lse,
                   const double *o, const double *l, double *out, double *lse_out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double pl = prev_lse[r], cl = l[r];
        if (cl == -INFINITY) {
            for (int d = 0; d < D; ++d) out[r * D + d] = prev_out[r * D + d];
            lse_out[r] = pl;
            continue;
        }
        if (pl == -INFINITY) {
            for (int d = 0; d < D; ++d) out[r * D + d] = o[r * D + d];
            lse_out[r] = cl;
            continue;
        }
        const double sig = 1.0 / (1.0 + exp(-(cl - pl)));                  /* sigmoid(lse - prev_lse) */
        const double x = pl - cl;
        const double logsig = x >= 0 ? -log1p(exp(-x)) : x - log1p(exp(x)); /* logsigmoid(prev_lse - lse) */
        for (int d = 0; d < D; ++d)
            out[r * D + d] = prev_out[r * D + d] - sig * (prev_out[r * D + d] - o[r * D + d]);
        lse_out[r] = pl - logsig;
    }
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
