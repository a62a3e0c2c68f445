/*
 * oracle.c -- plain fp64 CPU oracle for paged-KV decode attention and for the
 * MLA paged causal prefill variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every stored value is exact: fp16/bf16 inputs are widened to double bit by
 * bit (no rounding), all arithmetic is double, and nothing is blocked, fused or
 * reordered beyond the definitions below, so that a reader can check each
 * function against the pages it cites.
 *
 * Sources (page title, then the function or docstring section):
 *   [V2]  "paged_attention_v2_triton.py -- CCCL-derived Triton PagedAttention V2":
 *         _partition_attn_kernel (docstring "Algorithm"), _reduce_partitions_kernel,
 *         the key/value cache layout comments of its argument list.
 *         Its launcher, paged_attention_v2_triton, also takes kv_cache_dtype,
 *         k_scale and v_scale (and ignores them); the fp8 KV cache here reads
 *         them the plainest way: cache bytes are OCP FP8 E4M3 values and
 *         K = k_scale * fp8, V = v_scale * fp8.  The same launcher takes
 *         alibi_slopes (ignored too); read as ALiBi's additive bias: the score
 *         of key position t for query head h gains slopes[h] * (t - pos), pos
 *         the query's own position -- zero there, decreasing linearly with
 *         distance.
 *   [FD]  "koas-w.github.io flash-decode post": Decode_Paged_GQAAttention_Kernel,
 *         _flash_decode_partial_kernel, _flash_decode_combine_kernel.
 *   [MTD] Several query tokens per sequence (speculative / multi-token decode):
 *         the bottom-right causal rule of [MLA] section "3. Pass 1" applied to
 *         the [FD] cache layouts.  A sequence of context length n carries q_len
 *         query tokens, the last q_len of its n positions: query i (0-based)
 *         sits at pos = n - q_len + i and attends keys t <= pos.  Where
 *         n - q_len + i < 0 the window is empty and the row is zero (the [FD]
 *         empty-context reading, extended per query).  q_len = 1 is plain decode.
 *   [MLA] "kernelindex.com flashinfer gemini-2.5-pro triton xvhq2i"
 *         (mla_paged_prefill_causal_h16_ckv512_kpe64_ps1): sections
 *         "2. Determine Sequence Boundaries", "3. Pass 1", "4. Pass 2".
 *
 * Status codes returned (same numbers as the library's, written out here):
 *   0 ok, 1 invalid argument, 5 bad block table / bad page index.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

enum { OR_OK = 0, OR_INVALID = 1, OR_BAD_TABLE = 5 };
enum { OR_F16 = 0, OR_BF16 = 1, OR_FP8 = 2 };
enum { OR_NHD = 0, OR_VLLM = 1 };

/* ---- exact widening of 16-bit floats ------------------------------------ */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 (8 exponent bits, bias 127). */
static double bf16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* subnormal: f * 2^-126 / 2^7 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 128), e - 134);     /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

static double widen(uint16_t h, int dtype)
{
    return dtype == OR_BF16 ? bf16_bits_to_double(h) : f16_bits_to_double(h);
}

/* Exported so the tests can check the widening against a library routine. */
double oracle_widen(uint16_t h, int dtype) { return widen(h, dtype); }

/* OCP FP8 E4M3 (the "e4m3fn" encoding): 1 sign, 4 exponent (bias 7) and 3
 * fraction bits; exponent 0 is subnormal, S.1111.111 is NaN, there is no
 * infinity (largest finite 1.75 * 2^8 = 448). */
static double e4m3_bits_to_double(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 0xf && f == 0x7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);                  /* subnormal: f/8 * 2^-6 */
    else
        v = ldexp((double)(f + 8), e - 10);        /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

double oracle_widen8(uint8_t b) { return e4m3_bits_to_double(b); }

/* ---- paged K/V addressing ------------------------------------------------ */

/*
 * Element d of token slot o in physical page p, KV head g.
 *   NHD  : k_cache / v_cache [num_blocks][n_kv_heads][block_size][head_dim]
 *          ([FD] Decode_Paged_GQAAttention_Kernel argument comments).
 *   VLLM : key_cache   [num_blocks][kv_heads][head_size/x][block_size][x]
 *          value_cache [num_blocks][kv_heads][head_size][block_size]
 *          ([V2] _partition_attn_kernel argument comments and its K/V gathers).
 */
static size_t k_index(int layout, int Hkv, int BS, int D, int x,
                      long long p, int g, int o, int d)
{
    if (layout == OR_NHD)
        return (((size_t)p * Hkv + g) * BS + o) * D + d;
    return ((((size_t)p * Hkv + g) * (D / x) + d / x) * BS + o) * x + d % x;
}

static size_t v_index(int layout, int Hkv, int BS, int D,
                      long long p, int g, int o, int d)
{
    if (layout == OR_NHD)
        return (((size_t)p * Hkv + g) * BS + o) * D + d;
    return (((size_t)p * Hkv + g) * D + d) * BS + o;
}

typedef struct {
    int B, Hq, Hkv, D, BS, MBPS, NB, dtype, layout, x;
    int kv_dtype;              /* dtype of the caches: OR_F16, OR_BF16 or OR_FP8 */
    int q_len;                 /* query tokens per sequence ([MTD]); 1 = plain decode */
    const uint16_t* q;         /* [B][q_len][Hq][D] */
    const void *k, *v;         /* 16-bit or 8-bit elements per kv_dtype */
    const int32_t *table, *ctx;
    double scale, k_scale, v_scale;   /* k_scale, v_scale multiply fp8 cache values (1 otherwise) */
    const double* alibi;       /* per query head ALiBi slope, or NULL */
} decode_args;

/* Value of cache element i: exact widening, times the fp8 scale. */
static double cache_value(const decode_args* a, const void* base, size_t i, double fp8_scale)
{
    if (a->kv_dtype == OR_FP8) return fp8_scale * e4m3_bits_to_double(((const uint8_t*)base)[i]);
    return widen(((const uint16_t*)base)[i], a->kv_dtype);
}

/* Checks the arguments shared by every decode entry point. */
static int check_decode(const decode_args* a)
{
    if (a->B < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->D <= 0 || a->BS <= 0 ||
        a->MBPS < 0 || a->NB < 0 || a->q_len <= 0)
        return OR_INVALID;
    if (a->Hq % a->Hkv != 0) return OR_INVALID;
    if (a->dtype != OR_F16 && a->dtype != OR_BF16) return OR_INVALID;
    if (a->kv_dtype != a->dtype && !(a->kv_dtype == OR_FP8 && a->layout == OR_NHD)) return OR_INVALID;
    if (a->layout == OR_VLLM && (a->x <= 0 || a->D % a->x != 0)) return OR_INVALID;
    if (a->layout != OR_NHD && a->layout != OR_VLLM) return OR_INVALID;
    return OR_OK;
}

/* Context length of sequence b, or -1 if it is out of range. */
static int seq_len(const decode_args* a, int b)
{
    int n = a->ctx[b];
    if (n < 0 || (long long)n > (long long)a->MBPS * a->BS) return -1;
    return n;
}

/* Physical page of token t of sequence b, or -1 if the table entry is bad.
 * Token t lives in logical block t / block_size at slot t % block_size
 * ([V2] "Paged K gather"; [FD] block_table comment: -1 = unallocated). */
static long long page_of(const decode_args* a, int b, int t)
{
    long long p = a->table[(size_t)b * a->MBPS + t / a->BS];
    if (p < 0 || p >= a->NB) return -1;
    return p;
}

/* Score of token t for query token i, head h:  scale * sum_d q[b][i][h][d] * K_t[d]. */
static double score(const decode_args* a, int b, int i, int h, int g, long long p, int o)
{
    double s = 0.0;
    for (int d = 0; d < a->D; ++d) {
        double qd = widen(a->q[(((size_t)b * a->q_len + i) * a->Hq + h) * a->D + d], a->dtype);
        double kd = cache_value(a, a->k, k_index(a->layout, a->Hkv, a->BS, a->D, a->x, p, g, o, d), a->k_scale);
        s += qd * kd;
    }
    return a->scale * s;
}

static double value(const decode_args* a, int g, long long p, int o, int d)
{
    return cache_value(a, a->v, v_index(a->layout, a->Hkv, a->BS, a->D, p, g, o, d), a->v_scale);
}

/*
 * Softmax attention of query token i, head h over tokens [t0, t1) of sequence b
 * (the caller keeps t1 inside the query's causal window), returned unnormalised: m = max_t s_t, l = sum_t exp(s_t - m),
 * acc[d] = sum_t exp(s_t - m) * V_t[d].  An empty range gives (-inf, 0, 0),
 * the sentinel of [FD] _flash_decode_partial_kernel ("empty splits").
 * Returns -1 on a bad table entry.
 */
static int attend_range(const decode_args* a, int b, int i, int h, int t0, int t1,
                        double* m_out, double* l_out, double* acc, double* sbuf)
{
    int G = a->Hq / a->Hkv;
    int g = h / G;           /* consecutive grouping: kv head = q head / group size */
    for (int d = 0; d < a->D; ++d) acc[d] = 0.0;
    if (t1 <= t0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return 0;
    }
    double m = -INFINITY;
    int pos = seq_len(a, b) - a->q_len + i;   /* the query's own position */
    for (int t = t0; t < t1; ++t) {
        long long p = page_of(a, b, t);
        if (p < 0) return -1;
        sbuf[t - t0] = score(a, b, i, h, g, p, t % a->BS);
        if (a->alibi) sbuf[t - t0] += a->alibi[h] * (double)(t - pos);
        if (sbuf[t - t0] > m) m = sbuf[t - t0];
    }
    double l = 0.0;
    for (int t = t0; t < t1; ++t) {
        long long p = page_of(a, b, t);
        double w = exp(sbuf[t - t0] - m);
        l += w;
        for (int d = 0; d < a->D; ++d) acc[d] += w * value(a, g, p, t % a->BS, d);
    }
    *m_out = m;
    *l_out = l;
    return 0;
}

/* End of query token i's causal window in a sequence of n tokens ([MTD]):
 * it attends keys t < n - q_len + i + 1 (t <= its position); <= 0 is empty. */
static int window_end(int n, int q_len, int i) { return n - q_len + i + 1; }

/*
 * Paged GQA decode attention, the plain definition:
 *   out[b][i][h][:] = sum_t softmax_t(scale * q[b][i][h] . K_t) * V_t,
 *   t in [0, window_end(ctx[b], q_len, i)),
 * K_t, V_t gathered for KV head h / (Hq/Hkv) through block_table.
 * An empty window (ctx[b] == 0 in plain decode) gives a zero row (the reading
 * taken for the empty context; [FD] _flash_decode_combine_kernel writes zeros
 * there).  Only sequences b in [b_lo, b_hi) are computed and written.
 * sbuf: caller scratch of at least max ctx doubles; acc: D doubles.
 */
int oracle_decode(int B, int Hq, int Hkv, int D, int BS, int MBPS, int NB,
                  int dtype, int layout, int x, int kv_dtype, int q_len,
                  const uint16_t* q, const void* k, const void* v,
                  const int32_t* table, const int32_t* ctx, double scale, double k_scale, double v_scale,
                  const double* alibi, int b_lo, int b_hi, double* out, double* sbuf, double* acc)
{
    decode_args a = {B, Hq, Hkv, D, BS, MBPS, NB, dtype, layout, x, kv_dtype, q_len, q, k, v, table, ctx,
                     scale, k_scale, v_scale, alibi};
    int st = check_decode(&a);
    if (st) return st;
    if (b_lo < 0 || b_hi > B || b_lo > b_hi) return OR_INVALID;
    for (int b = b_lo; b < b_hi; ++b) {
        int n = seq_len(&a, b);
        if (n < 0) return OR_INVALID;
        for (int i = 0; i < q_len; ++i) {
            int end = window_end(n, q_len, i);
            for (int h = 0; h < Hq; ++h) {
                double m, l;
                double* o = out + (((size_t)b * q_len + i) * Hq + h) * D;
                if (end <= 0) {
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    continue;
                }
                if (attend_range(&a, b, i, h, 0, end, &m, &l, acc, sbuf)) return OR_BAD_TABLE;
                for (int d = 0; d < D; ++d) o[d] = acc[d] / l;
            }
        }
    }
    return OR_OK;
}

/*
 * Split mode ([V2] phase 1 with fixed partitions; [FD] partial kernel):
 * split s covers tokens [s*P, min((s+1)*P, ctx[b])), cut further at the end of
 * each query's causal window.  For each (b, i, h, s) it stores the
 * unnormalised partial (m, l, acc) of attend_range, with the (-inf, 0, 0)
 * sentinel where that range is empty.  Layouts: m, l [B][q_len][Hq][NS],
 * acc [B][q_len][Hq][NS][D].
 */
int oracle_decode_partials(int B, int Hq, int Hkv, int D, int BS, int MBPS, int NB,
                           int dtype, int layout, int x, int kv_dtype, int q_len,
                           const uint16_t* q, const void* k, const void* v,
                           const int32_t* table, const int32_t* ctx, double scale, double k_scale,
                           double v_scale, const double* alibi, int P, int NS, int b_lo, int b_hi,
                           double* pm, double* pl, double* pacc, double* sbuf)
{
    decode_args a = {B, Hq, Hkv, D, BS, MBPS, NB, dtype, layout, x, kv_dtype, q_len, q, k, v, table, ctx,
                     scale, k_scale, v_scale, alibi};
    int st = check_decode(&a);
    if (st) return st;
    if (P <= 0 || NS <= 0 || b_lo < 0 || b_hi > B || b_lo > b_hi) return OR_INVALID;
    for (int b = b_lo; b < b_hi; ++b) {
        int n = seq_len(&a, b);
        if (n < 0) return OR_INVALID;
        if ((long long)NS * P < n) return OR_INVALID;   /* splits must cover the context */
        for (int i = 0; i < q_len; ++i) {
            int end = window_end(n, q_len, i);
            for (int h = 0; h < Hq; ++h) {
                for (int s = 0; s < NS; ++s) {
                    long long t0 = (long long)s * P, t1 = t0 + P;
                    if (t1 > end) t1 = end;
                    if (t0 > t1) t0 = t1;
                    size_t r = (((size_t)b * q_len + i) * Hq + h) * NS + s;
                    if (attend_range(&a, b, i, h, (int)t0, (int)t1, &pm[r], &pl[r], &pacc[r * D], sbuf))
                        return OR_BAD_TABLE;
                }
            }
        }
    }
    return OR_OK;
}

/*
 * Cross-split combine ([FD] _flash_decode_combine_kernel; [V2]
 * _reduce_partitions_kernel docstring):  M = max_s m_s, f_s = exp(m_s - M),
 * out = sum_s f_s acc_s / sum_s f_s l_s.  Sentinel splits (m = -inf) get
 * f_s = 0.  Rows are (b, i, h), i < q_len; an empty causal window
 * (ctx[b] == 0 in plain decode) gives zeros.
 */
int oracle_combine(int B, int q_len, int Hq, int D, int NS, const int32_t* ctx,
                   const double* pm, const double* pl, const double* pacc,
                   int b_lo, int b_hi, double* out)
{
    if (B < 0 || q_len <= 0 || Hq <= 0 || D <= 0 || NS <= 0 || b_lo < 0 || b_hi > B || b_lo > b_hi)
        return OR_INVALID;
    for (int b = b_lo; b < b_hi; ++b) {
        for (long long r = (long long)b * q_len * Hq; r < (long long)(b + 1) * q_len * Hq; ++r) {
            int i = (int)((r / Hq) % q_len);
            double* o = out + (size_t)r * D;
            const double* m = pm + (size_t)r * NS;
            const double* l = pl + (size_t)r * NS;
            const double* acc = pacc + (size_t)r * NS * D;
            if (window_end(ctx[b], q_len, i) <= 0) {
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                continue;
            }
            double M = -INFINITY;
            for (int s = 0; s < NS; ++s) if (m[s] > M) M = m[s];
            double L = 0.0;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int s = 0; s < NS; ++s) {
                double f = (m[s] == -INFINITY) ? 0.0 : exp(m[s] - M);
                L += f * l[s];
                for (int d = 0; d < D; ++d) o[d] += f * acc[(size_t)s * D + d];
            }
            for (int d = 0; d < D; ++d) o[d] /= L;
        }
    }
    return OR_OK;
}

/*
 * MLA paged causal prefill, page_size 1 ([MLA] sections 2-4):
 * for query token t of sequence b (qo_indptr[b] <= t < qo_indptr[b+1]) and
 * head h,
 *   kv_len = kv_indptr[b+1] - kv_indptr[b],  q_len = qo_indptr[b+1] - qo_indptr[b],
 *   prefix = kv_len - q_len,  pos = prefix + (t - qo_indptr[b])   (bottom-right causal),
 *   for j in [0, kv_len) with j <= pos:  page = kv_indices[kv_indptr[b] + j],
 *     logit_j = sm_scale * (q_nope[t][h] . ckv[page] + q_pe[t][h] . kpe[page]),
 *   out[t][h] = sum_j softmax(logit)_j * ckv[page_j]       (V is ckv),
 *   lse[t][h] = log2 sum_j exp(logit_j)                     (base-2 LSE).
 * kv_len == 0 gives out = 0 and lse = -inf ([MLA] section 2).
 * Tensors (bf16 bits): q_nope [total_q][H][Dc], q_pe [total_q][H][Dr],
 * ckv [num_pages][1][Dc], kpe [num_pages][1][Dr].  Only tokens in [t_lo, t_hi)
 * are computed.  sbuf: at least max kv_len doubles.
 */
int oracle_mla(int total_q, int H, int Dc, int Dr, int batch, int num_pages,
               const uint16_t* q_nope, const uint16_t* q_pe,
               const uint16_t* ckv, const uint16_t* kpe,
               const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
               double sm_scale, int t_lo, int t_hi, double* out, double* lse, double* sbuf)
{
    if (total_q < 0 || H <= 0 || Dc <= 0 || Dr < 0 || batch < 0 || num_pages < 0)
        return OR_INVALID;
    if (t_lo < 0 || t_hi > total_q || t_lo > t_hi) return OR_INVALID;
    if (qo_indptr[0] != 0 || kv_indptr[0] != 0 || qo_indptr[batch] != total_q) return OR_INVALID;
    for (int t = t_lo; t < t_hi; ++t) {
        int b = 0;
        while (b < batch && !(qo_indptr[b] <= t && t < qo_indptr[b + 1])) ++b;
        if (b == batch) return OR_INVALID;
        int q_len = qo_indptr[b + 1] - qo_indptr[b];
        int kv_len = kv_indptr[b + 1] - kv_indptr[b];
        if (kv_len < 0) return OR_INVALID;
        int pos = (kv_len - q_len) + (t - qo_indptr[b]);
        for (int h = 0; h < H; ++h) {
            double* o = out + ((size_t)t * H + h) * Dc;
            for (int d = 0; d < Dc; ++d) o[d] = 0.0;
            if (kv_len == 0) {
                lse[(size_t)t * H + h] = -INFINITY;
                continue;
            }
            if (kv_len < q_len) return OR_INVALID;   /* negative prefix */
            const uint16_t* qn = q_nope + ((size_t)t * H + h) * Dc;
            const uint16_t* qp = q_pe + ((size_t)t * H + h) * Dr;
            int nkeys = pos + 1 < kv_len ? pos + 1 : kv_len;
            double m = -INFINITY;
            for (int j = 0; j < nkeys; ++j) {
                long long pg = kv_indices[kv_indptr[b] + j];
                if (pg < 0 || pg >= num_pages) return OR_BAD_TABLE;
                double s = 0.0;
                for (int d = 0; d < Dc; ++d)
                    s += bf16_bits_to_double(qn[d]) * bf16_bits_to_double(ckv[(size_t)pg * Dc + d]);
                for (int d = 0; d < Dr; ++d)
                    s += bf16_bits_to_double(qp[d]) * bf16_bits_to_double(kpe[(size_t)pg * Dr + d]);
                sbuf[j] = sm_scale * s;
                if (sbuf[j] > m) m = sbuf[j];
            }
            double z = 0.0;
            for (int j = 0; j < nkeys; ++j) {
                long long pg = kv_indices[kv_indptr[b] + j];
                double w = exp(sbuf[j] - m);
                z += w;
                for (int d = 0; d < Dc; ++d) o[d] += w * bf16_bits_to_double(ckv[(size_t)pg * Dc + d]);
            }
            for (int d = 0; d < Dc; ++d) o[d] /= z;
            lse[(size_t)t * H + h] = (m + log(z)) / log(2.0);
        }
    }
    return OR_OK;
}
