/*
 * fia_oracle.c -- the ORACLE for the fused inference attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, fp64 CPU statement of
 * what the operators compute.  It exists so that the CUDA path can be checked
 * against something written directly from the operator descriptions.  Only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark may load it;
 * the product library never links, loads or calls it, and it shares no code,
 * header, table or constant with the CUDA sources.
 *
 * Sources (operator documentation pages):
 *   [IFA]  aclnnIncreFlashAttentionV3 -- "Function" (formula
 *          Attention = Softmax(Q K^T / sqrt(d)) V, scaleValue), parameter table
 *          (antiquantScale/antiquantOffset shapes, blocktable, actualSeqLengths,
 *          numKeyValueHeads) and "Constraints" (page attention scenario).
 *   [RAU]  aclnnRingAttentionUpdate -- "功能说明 / 计算公式" (merge of two
 *          FlashAttention results by their softmax max and sum).
 *   [FAS]  aclnnFlashAttentionScoreV4 -- "计算公式" (learnable sink:
 *          m = max(sink, max S), Attention = sum e^{S-m} V / (sum e^{S-m} + e^{sink-m}))
 *          and the TND / actualSeqQLen rules in "约束说明".
 *   [FIA]  FusedInferAttentionScore 全解析 -- prefill (Q_S > 1) and decode
 *          (Q_S = 1) in one operator, sparseMode 3 = rightDownCausal, and the
 *          empty-tensor rules ("约束说明 / 空入参").
 *
 * Readings where the pages are silent or garbled (each one is listed with its
 * justification in the design notes):
 *   R1  GQA grouping: query head h reads kv head h / (Nq / Nkv) (contiguous groups).
 *   R2  int8 dequant: k = fl32(fl32((float)x - offset) * scale), two separate
 *       round-to-nearest fp32 operations (no fused multiply-add), then widened.
 *   R3  The sink is added in the domain of the scaled logits, unscaled.
 *   R4  softmax_max / softmax_sum are the natural-exp max and sum of the scaled
 *       logits, sink included; one value per (row, head).
 *   R5  RingAttentionUpdate: each partial's output is normalised by its own sum,
 *       so the merge weights it by sum_i * e^{max_i - max}  (the printed formula
 *       drops these sum factors; only the weighted form is exact).
 *   R6  A row with no visible key and no sink: out = 0, max = -inf, sum = 0.
 *       With a sink: out = 0, max = sink, sum = 1.
 *   R7  Causal mask (rightDownCausal): key j is visible to query i of a sequence
 *       iff j <= i + (Lkv - Lq).
 *   R13 attenMask (decode): a byte per (batch, key); nonzero = the key is masked
 *       out (the causal forms the pages describe keep the diagonal at 0), and a
 *       masked key is left out of the softmax entirely.
 *   R16 Decode with several query positions (speculative drafts, Q_S > 1 over the
 *       paged cache): the s queries of a batch are its last s positions, each seeing
 *       the keys up to its own position (rightDownCausal with Lq = s).
 *   R14 Post-quant output: y = out * quantScale2 + quantOffset2 in the
 *       attention's own precision, rounded to nearest with ties to even and
 *       saturated to int8; per-channel parameters index the output's N * D
 *       channels (N = query heads, the heads of attentionOut).
 *   R15 Band (sparseMode 4, preTokens / nextTokens): aligned on the same
 *       diagonal as rightDownCausal: key j is visible to query i iff
 *       i + (Lkv - Lq) - preTokens <= j <= i + (Lkv - Lq) + nextTokens.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC.
 * -ffp-contract=off is required: R2 forbids contracting the dequant into an FMA.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes used by this file's interface (its own numbering). */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_I8 = 3, OR_F64 = 4 };

/* ---- scalar decoding of the stored formats, from the IEEE-754 definitions ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^-24 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 1024), expo - 25);  /* (1 + frac/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of a binary32. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int dtype, int64_t idx)
{
    switch (dtype) {
    case OR_F32: return (double)((const float *)base)[idx];
    case OR_F16: return half_bits_to_double(((const uint16_t *)base)[idx]);
    case OR_BF16: return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    case OR_F64: return ((const double *)base)[idx];
    default: return NAN;
    }
}

/* R2: per-channel antiquant of one int8 code, in fp32 with two roundings. */
float oracle_dequant_i8(int8_t x, float offset, float scale)
{
    float xf = (float)x;
    float centred = xf - offset;
    float r = centred * scale;
    return r;
}

/* R2 over arrays: out[i] = dequant of x[i] with its own offset and scale. */
void oracle_dequant_i8_array(const int8_t *x, const float *offset, const float *scale, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_dequant_i8(x[i], offset[i], scale[i]);
}

/* [IFA] Constraints / page attention, as raw bytes: copies the stored rows of
 * tokens 0..L-1 of (batch b, kv head hk) out of a (blocknum, KV_N, blocksize, D)
 * pool into dst (L x D elements of elem_bytes each), token t from block
 * block_table[b][t / block_size], in-block row t - (t / block_size) * block_size. */
int oracle_gather_rows(const void *cache, int elem_bytes, const int32_t *block_table, int64_t bt_stride,
                       int b, int hk, int64_t L, int Nkv, int D, int block_size, void *dst)
{
    const int64_t row_bytes = (int64_t)D * elem_bytes;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t logical = t / block_size;
        const int64_t in_block = t - logical * block_size;
        const int64_t blk = block_table[(int64_t)b * bt_stride + logical];
        if (blk < 0)
            return -1;
        const int64_t row = (blk * Nkv + hk) * block_size + in_block;
        memcpy((char *)dst + t * row_bytes, (const char *)cache + row * row_bytes, (size_t)row_bytes);
    }
    return 0;
}

/* ---- the attention of one query row over a dense list of visible keys ----
 *
 * [IFA] Function: out = Softmax(scale * q K^T) V, written out as its definition.
 * [FAS] sink: m = max(sink, max_t s_t); l = sum_t e^{s_t - m} + e^{sink - m};
 *       out = sum_t e^{s_t - m} v_t / l.
 * q: D values; K, V: n x D row-major; sink may be NULL. */
static void attend_row(const double *q, const double *K, const double *V, int64_t n, int D,
                       double scale, const double *sink, double *s /* scratch, n */,
                       double *out, double *smax, double *ssum)
{
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * K[t * D + d];
        s[t] = scale * dot;
        if (s[t] > m)
            m = s[t];
    }
    if (sink && *sink > m)
        m = *sink;
    if (m == -INFINITY) {            /* R6: nothing visible and no sink */
        for (int d = 0; d < D; ++d)
            out[d] = 0.0;
        *smax = -INFINITY;
        *ssum = 0.0;
        return;
    }
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t)
        l += exp(s[t] - m);
    if (sink)
        l += exp(*sink - m);
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t t = 0; t < n; ++t)
            acc += exp(s[t] - m) * V[t * D + d];
        out[d] = acc / l;
    }
    *smax = m;
    *ssum = l;
}

/* ---- decode (query S = 1) ------------------------------------------------
 *
 * [IFA] Constraints / page attention: token t of batch b lives in physical block
 * block_table[b][t / block_size], row t % block_size; the KV cache layout is
 * (blocknum, KV_N, blocksize, D).  When block_table is NULL the cache is read as
 * the contiguous layout (B, KV_N, kv_rows, D) instead (BNSD without paging).
 *
 * q: (B, Nq, D) in q_dtype (F16/BF16/F32/F64).  k_cache / v_cache in kv_dtype;
 * for OR_I8 the codes are dequantised with aq_scale / aq_offset of shape
 * (2, Nkv, D), index 0 for K and 1 for V ([IFA] parameter table, per-channel);
 * aq_offset may be NULL (zero).  sink: fp32 (Nq) or NULL.
 * mask: [IFA] attenMask of shape (B, 1, 1, S), one byte per (b, t) at
 * mask[b * mask_stride + t], or NULL; a nonzero byte removes key t of batch b
 * from the attention (1 = masked out, 0 = attended), so a batch whose keys are
 * all masked is handled like one of length 0.
 * q_len (R16): s >= 1 query positions per batch, q laid out (B, s, Nq, D); position i
 * sits at qp = L - s + i of a batch of length L; rows run over B * s * Nq.  A mask needs
 * s = 1.
 * pre_tokens / next_tokens: the band of R15, key t visible iff
 * qp - pre_tokens <= t <= qp + next_tokens; (large, 0) is rightDownCausal with Lq = s
 * (for s = 1: every key), the default.
 * rows: the (b * Nq + h) rows to compute, or NULL for all B * Nq rows; results
 * are written compactly: out[i * D + d], smax[i], ssum[i] for the i-th row.
 * Returns 0, or -1 on an argument it cannot handle. */
int oracle_decode(const void *q, int q_dtype,
                  const void *k_cache, const void *v_cache, int kv_dtype,
                  const int32_t *block_table, int64_t bt_stride,
                  const int64_t *seq_lens,
                  int B, int Nq, int Nkv, int D, int block_size, int64_t kv_rows,
                  double scale, const float *aq_scale, const float *aq_offset,
                  const float *sink, const uint8_t *mask, int64_t mask_stride,
                  int64_t pre_tokens, int64_t next_tokens, int q_len,
                  const int64_t *rows, int64_t n_rows, int nthreads,
                  double *out, double *smax, double *ssum)
{
    if (Nkv == 0)
        Nkv = Nq;                         /* [IFA] numKeyValueHeads = 0 means equal */
    if (Nq <= 0 || Nkv <= 0 || Nq % Nkv != 0 || D <= 0)
        return -1;
    if (kv_dtype == OR_I8 && !aq_scale)
        return -1;
    if (q_len < 1)
        q_len = 1;
    if (mask && q_len != 1)
        return -1;
    const int G = Nq / Nkv;
    const int64_t total = rows ? n_rows : (int64_t)B * q_len * Nq;
    int64_t max_len = 0;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] > max_len)
            max_len = seq_lens[b];
    int bad = 0;

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel reduction(| : bad)
#endif
    {
        double *Kd = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1) * D);
        double *Vd = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1) * D);
        double *qd = (double *)malloc(sizeof(double) * D);
        double *sc = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!Kd || !Vd || !qd || !sc)
            bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < total; ++i) {
            if (bad)
                continue;
            const int64_t r = rows ? rows[i] : i;
            const int64_t bi = r / Nq;                          /* b * q_len + position */
            const int b = (int)(bi / q_len), h = (int)(r % Nq);
            const int64_t pos = bi % q_len;
            const int hk = h / G;                               /* R1 */
            const int64_t L = seq_lens[b];
            const int64_t qp = L - q_len + pos;                 /* the query's position, R16 */
            for (int d = 0; d < D; ++d)
                qd[d] = load_elem(q, q_dtype, r * D + d);
            /* gather the visible keys/values of (b, hk) into dense rows; n of them
             * survive the mask */
            int64_t n = 0;
            for (int64_t t = 0; t < L; ++t) {
                if (mask && mask[(int64_t)b * mask_stride + t] != 0)
                    continue;
                if (t < qp - pre_tokens || t > qp + next_tokens)            /* R15, R16 */
                    continue;
                int64_t src;                                    /* element offset of row t */
                if (block_table) {
                    const int64_t blk = block_table[(int64_t)b * bt_stride + t / block_size];
                    src = ((blk * Nkv + hk) * (int64_t)block_size + t % block_size) * D;
                } else {
                    src = (((int64_t)b * Nkv + hk) * kv_rows + t) * D;
                }
                for (int d = 0; d < D; ++d) {
                    if (kv_dtype == OR_I8) {
                        const float ko = aq_offset ? aq_offset[(0 * Nkv + hk) * D + d] : 0.0f;
                        const float vo = aq_offset ? aq_offset[(1 * Nkv + hk) * D + d] : 0.0f;
                        Kd[n * D + d] = (double)oracle_dequant_i8(((const int8_t *)k_cache)[src + d],
                                                                  ko, aq_scale[(0 * Nkv + hk) * D + d]);
                        Vd[n * D + d] = (double)oracle_dequant_i8(((const int8_t *)v_cache)[src + d],
                                                                  vo, aq_scale[(1 * Nkv + hk) * D + d]);
                    } else {
                        Kd[n * D + d] = load_elem(k_cache, kv_dtype, src + d);
                        Vd[n * D + d] = load_elem(v_cache, kv_dtype, src + d);
                    }
                }
                ++n;
            }
            double sk;
            attend_row(qd, Kd, Vd, n, D, scale, sink ? (sk = sink[h], &sk) : NULL, sc,
                       out + i * D, smax + i, ssum + i);
        }
        free(Kd);
        free(Vd);
        free(qd);
        free(sc);
    }
    return bad ? -1 : 0;
}

/* ---- prefill, TND layout ---------------------------------------------------
 *
 * [FIA] prefill (Q_S > 1) runs the same attention over whole prompts; [FAS] TND:
 * the tokens of all sequences are concatenated; cu_q / cu_kv hold B + 1
 * cumulative lengths starting at 0 (the RingAttentionUpdate page's form of
 * actual_seq_qlen).  q/out: (T, Nq, D); k, v: (Tkv, Nkv, D).
 * sparse_mode ([FIA] sparseMode): 0 no mask, 3 rightDownCausal (R7), 4 band (R15):
 * with d = Lkv - Lq, key j is visible to query i iff
 *     i + d - pre_tokens <= j <= i + d + next_tokens.
 * rows: (t * Nq + h) rows or NULL for all. */
int oracle_prefill(const void *q, const void *k, const void *v, int dtype,
                   const int64_t *cu_q, const int64_t *cu_kv,
                   int B, int Nq, int Nkv, int D, double scale, int sparse_mode,
                   int64_t pre_tokens, int64_t next_tokens, const float *sink,
                   const int64_t *rows, int64_t n_rows, int nthreads,
                   double *out, double *smax, double *ssum)
{
    if (Nkv == 0)
        Nkv = Nq;
    if (Nq <= 0 || Nkv <= 0 || Nq % Nkv != 0 || D <= 0 || B <= 0)
        return -1;
    if (sparse_mode != 0 && sparse_mode != 3 && sparse_mode != 4)
        return -1;
    const int G = Nq / Nkv;
    const int64_t T = cu_q[B];
    const int64_t total = rows ? n_rows : T * Nq;
    int64_t max_kv = 0;
    for (int b = 0; b < B; ++b)
        if (cu_kv[b + 1] - cu_kv[b] > max_kv)
            max_kv = cu_kv[b + 1] - cu_kv[b];
    int bad = 0;

#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel reduction(| : bad)
#endif
    {
        const size_t cap = (size_t)(max_kv > 0 ? max_kv : 1);
        double *Kd = (double *)malloc(sizeof(double) * cap * D);
        double *Vd = (double *)malloc(sizeof(double) * cap * D);
        double *qd = (double *)malloc(sizeof(double) * D);
        double *sc = (double *)malloc(sizeof(double) * cap);
        if (!Kd || !Vd || !qd || !sc)
            bad = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
        for (int64_t i = 0; i < total; ++i) {
            if (bad)
                continue;
            const int64_t r = rows ? rows[i] : i;
            const int64_t t = r / Nq;
            const int h = (int)(r % Nq), hk = h / G;
            int b = 0;
            while (b < B && !(cu_q[b] <= t && t < cu_q[b + 1]))
                ++b;
            if (b == B) {
                bad = 1;
                continue;
            }
            const int64_t qi = t - cu_q[b];
            const int64_t Lq = cu_q[b + 1] - cu_q[b], Lkv = cu_kv[b + 1] - cu_kv[b];
            int64_t first = 0, n = Lkv;                     /* keys first .. first + n - 1 */
            if (sparse_mode == 3) {                         /* R7 */
                const int64_t last = qi + (Lkv - Lq);       /* last visible key index */
                n = last + 1 < 0 ? 0 : (last + 1 < Lkv ? last + 1 : Lkv);
            } else if (sparse_mode == 4) {                  /* R15 */
                int64_t lo = qi + (Lkv - Lq) - pre_tokens, hi = qi + (Lkv - Lq) + next_tokens;
                if (lo < 0)
                    lo = 0;
                if (hi > Lkv - 1)
                    hi = Lkv - 1;
                first = lo;
                n = hi >= lo ? hi - lo + 1 : 0;
            }
            for (int d = 0; d < D; ++d)
                qd[d] = load_elem(q, dtype, r * D + d);
            for (int64_t j = 0; j < n; ++j)
                for (int d = 0; d < D; ++d) {
                    const int64_t src = ((cu_kv[b] + first + j) * Nkv + hk) * D + d;
                    Kd[j * D + d] = load_elem(k, dtype, src);
                    Vd[j * D + d] = load_elem(v, dtype, src);
                }
            double sk;
            attend_row(qd, Kd, Vd, n, D, scale, sink ? (sk = sink[h], &sk) : NULL, sc,
                       out + i * D, smax + i, ssum + i);
        }
        free(Kd);
        free(Vd);
        free(qd);
        free(sc);
    }
    return bad ? -1 : 0;
}

/* ---- RingAttentionUpdate ---------------------------------------------------
 *
 * [RAU] merge of two attention results (prev, cur), each with its per-row
 * softmax max and sum, read per R5:
 *   m   = max(m_p, m_c)
 *   w_p = l_p e^{m_p - m},  w_c = l_c e^{m_c - m}     (a side with m = -inf weighs 0)
 *   l   = w_p + w_c
 *   out = (o_p w_p + o_c w_c) / l
 * rows x N (max/sum) and rows x N x D (out), all fp64 here. */
int oracle_rau(const double *prev_out, const double *prev_max, const double *prev_sum,
               const double *cur_out, const double *cur_max, const double *cur_sum,
               int64_t rows, int N, int D,
               double *out, double *max_out, double *sum_out)
{
    for (int64_t r = 0; r < rows * N; ++r) {
        const double mp = prev_max[r], mc = cur_max[r];
        const double m = mp > mc ? mp : mc;
        if (m == -INFINITY) {
            for (int d = 0; d < D; ++d)
                out[r * D + d] = 0.0;
            max_out[r] = -INFINITY;
            sum_out[r] = 0.0;
            continue;
        }
        const double wp = (mp == -INFINITY) ? 0.0 : prev_sum[r] * exp(mp - m);
        const double wc = (mc == -INFINITY) ? 0.0 : cur_sum[r] * exp(mc - m);
        const double l = wp + wc;
        for (int d = 0; d < D; ++d)
            out[r * D + d] = l > 0.0 ? (prev_out[r * D + d] * wp + cur_out[r * D + d] * wc) / l : 0.0;
        max_out[r] = m;
        sum_out[r] = l;
    }
    return 0;
}

/* ---- int8 post-quant output ----------------------------------------------
 *
 * [IFA] quantScale2 / quantOffset2 (output quantisation, symmetric without an
 * offset, asymmetric with one): y = out * scale2[c] + offset2[c] for channel
 * c = h * D + d of the (N, D) output row, rounded to the nearest integer with
 * ties to even and saturated to [-128, 127].  per_channel = 0 reads scale2[0]
 * (and offset2[0]) for every channel.  x: rows x C in fp64 (C = N * D);
 * offset2 may be NULL.  y (the unrounded value, may be NULL) and code get
 * rows x C entries. */
void oracle_post_quant(const double *x, int64_t rows, int64_t C, const float *scale2,
                       const float *offset2, int per_channel, double *y, int8_t *code)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < C; ++c) {
            const int64_t i = r * C + c;
            const int64_t pc = per_channel ? c : 0;
            const double v = x[i] * (double)scale2[pc] + (offset2 ? (double)offset2[pc] : 0.0);
            double q = nearbyint(v);                    /* default rounding: ties to even */
            if (q > 127.0)
                q = 127.0;
            if (q < -128.0)
                q = -128.0;
            if (y)
                y[i] = v;
            code[i] = (int8_t)q;
        }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
