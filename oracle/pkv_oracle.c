/*
 * pkv_oracle.c -- CPU oracle for paged-KV attention with asymmetric K/V head
 * dimensions (K 192 / V 128, GQA, and the MLA-shaped 576 / 512 variant).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the GPU library computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant with the CUDA library: every definition below is
 * written out here from the sources cited next to it.
 *
 * Sources (web pages; cited by title and section):
 *   [PR64064]  vLLM PR #64064 "ROCm AITER unified attention for MiMo-V2.6",
 *              section "Details" (the reshape_and_cache_flash fix: V has its
 *              own head size and head stride; one packed (head_size +
 *              head_size_v) row per KV head, K first) and section "Tests"
 *              (bf16 / fp8 caches, per-tensor and per-head scales, both
 *              layouts, slack past the cache).
 *   [PR50371]  vLLM PR #50371 "Enable 12-head MLA persistent decode",
 *              sections "Purpose" and "Test Plan" (12 -> 16 zero-padded query
 *              heads, D 576 -> 512 output, FP32 SDPA reference) and the
 *              discussion of split-KV with runtime split selection.
 *   [MiMo-2xRTX] Hugging Face model card
 *              "diffbot/MiMo-V2.6-Flash-MOPD-FP8KV-W4A8-2x-RTX-PRO-6000",
 *              sections "What the kernels do" (split-KV for the verify step,
 *              FP8 E4M3 K/V) and "Update 2026-10-01" (rows with no visible
 *              keys give 0, not NaN, in the split-KV reducer; the attention
 *              sink taken as one extra logit in the softmax denominator,
 *              vLLM #58235).
 *
 * Precision: the FP8 encode divides in IEEE binary32 (that division decides
 * the code byte, and the GPU takes the same decision in the same precision);
 * everything in attention and the split merge is accumulated in binary64.
 *
 * Every function here is pinned by the CPU tests to something other than
 * itself (closed forms, brute force, a library conversion, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---------------------------------------------------------------- types --- */

/* Cache description.  Field meanings follow the packed-row layout of
 * [PR64064] "Details": every KV head of every token slot owns one row of
 * row_elems elements; K sits at [k_off, k_off + head_size) and V at
 * [v_off, v_off + head_size_v) of that row. */
typedef struct {
    int dtype;        /* 0 = bf16, 1 = fp8 e4m3 */
    int layout;       /* 0 = NHD [blk][bs][H][R], 1 = HND [blk][H][bs][R] */
    int num_blocks;
    int block_size;
    int num_kv_heads;
    int row_elems;
    int k_off, head_size;
    int v_off, head_size_v;
    int scale_mode;   /* 0 = none, 1 = per tensor, 2 = per KV head */
} oracle_cache_desc;

/* ----------------------------------------------------------- bf16 / e4m3 --- */

/* bfloat16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448;
 * subnormals are m * 2^-9.  Decoding straight from that definition. */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);        /* normal */
    return s ? -v : v;
}

/* Encode a binary32 value as E4M3 with round-to-nearest-even and saturation
 * to the largest finite magnitude (448).  NaN encodes as 0x7F. */
uint8_t oracle_e4m3_encode(float x)
{
    double a;
    uint8_t sign;
    int e;
    double frac, q;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;                      /* saturate, inf included */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: value = m * 2^-9, m = RNE(a / 2^-9) in [0, 8];
         * m == 8 is the smallest normal (code 0x08), which the code layout
         * produces by itself. */
        q = rint(ldexp(a, 9));
        return sign | (uint8_t)q;
    }
    frexp(a, &e);                                 /* a = f * 2^e, f in [0.5,1) */
    e -= 1;                                       /* a = 1.x * 2^e */
    frac = ldexp(a, -e) - 1.0;                    /* exact: [0, 1) */
    q = rint(frac * 8.0);                         /* RNE on the 3-bit mantissa */
    if (q == 8.0) {
        q = 0.0;
        e += 1;
    }
    /* a < 448 and RNE cannot produce a value above 448 here, so e + 7 <= 15
     * and the code is at most 0x7E. */
    return sign | (uint8_t)(((e + 7) << 3) | (int)q);
}

/* ------------------------------------------------------------ addressing --- */

static int64_t row_offset_elems(const oracle_cache_desc *d, int64_t block,
                                int64_t off, int64_t head)
{
    if (d->layout == 0)
        return ((block * d->block_size + off) * d->num_kv_heads + head) *
               (int64_t)d->row_elems;
    return ((block * d->num_kv_heads + head) * d->block_size + off) *
           (int64_t)d->row_elems;
}

static float scale_of(const float *scale, int mode, int head)
{
    if (mode == 1)
        return scale[0];
    if (mode == 2)
        return scale[head];
    return 1.0f;
}

/* ------------------------------------------------------------ cache write --- */

/* [PR64064] "Details": for each token t with slot s = slot_mapping[t] >= 0,
 * block b = s / block_size and offset o = s % block_size; for every KV head h
 * the K vector (head_size elements, read with K's own token and head strides)
 * goes to row[k_off ...] and the V vector (head_size_v elements, read with
 * V's own strides) goes to row[v_off ...].  A negative slot is skipped.
 * value == NULL writes K only (MLA, where V is a prefix of K).
 * fp8 caches store e4m3(x / scale) with the division in binary32.
 * Returns 0, or -1 for an argument it cannot honour. */
int oracle_kv_cache_write(const uint16_t *key, int64_t k_tok_stride,
                          int64_t k_head_stride, const uint16_t *value,
                          int64_t v_tok_stride, int64_t v_head_stride,
                          const int64_t *slot_mapping, int num_tokens,
                          void *cache, const oracle_cache_desc *d,
                          const float *k_scale, const float *v_scale)
{
    int t, h, i;
    int64_t nslots = (int64_t)d->num_blocks * d->block_size;
    for (t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        int64_t blk, off;
        if (s < 0)
            continue;
        if (s >= nslots)
            return -1;
        blk = s / d->block_size;
        off = s % d->block_size;
        for (h = 0; h < d->num_kv_heads; ++h) {
            int64_t row = row_offset_elems(d, blk, off, h);
            const uint16_t *ks = key + t * k_tok_stride + h * k_head_stride;
            const uint16_t *vs =
                value ? value + t * v_tok_stride + h * v_head_stride : NULL;
            if (d->dtype == 0) {
                uint16_t *c = (uint16_t *)cache + row;
                for (i = 0; i < d->head_size; ++i)
                    c[d->k_off + i] = ks[i];
                if (vs)
                    for (i = 0; i < d->head_size_v; ++i)
                        c[d->v_off + i] = vs[i];
            } else {
                uint8_t *c = (uint8_t *)cache + row;
                float ksc = scale_of(k_scale, d->scale_mode, h);
                float vsc = scale_of(v_scale, d->scale_mode, h);
                for (i = 0; i < d->head_size; ++i) {
                    float x = (float)oracle_bf16_to_double(ks[i]);
                    float y = x / ksc;                   /* binary32 divide */
                    c[d->k_off + i] = oracle_e4m3_encode(y);
                }
                if (vs)
                    for (i = 0; i < d->head_size_v; ++i) {
                        float x = (float)oracle_bf16_to_double(vs[i]);
                        float y = x / vsc;
                        c[d->v_off + i] = oracle_e4m3_encode(y);
                    }
            }
        }
    }
    return 0;
}

/* Dequantised read of one cache element: bf16 widens exactly; an fp8 code is
 * decoded and multiplied by its scale ([MiMo-2xRTX] "What the kernels do":
 * the E4M3 K/V path converts in the kernel). */
static double cache_read(const void *cache, const oracle_cache_desc *d,
                         int64_t elem, double scale)
{
    if (d->dtype == 0)
        return oracle_bf16_to_double(((const uint16_t *)cache)[elem]);
    return oracle_e4m3_decode(((const uint8_t *)cache)[elem]) * scale;
}

/* -------------------------------------------------------------- attention --- */

/* Paged attention for one query row (token t, query head h).
 *
 * The sequence b that owns t has q_len = qsl[b+1] - qsl[b] query tokens and
 * L = seq_lens[b] keys in total (the new tokens included).  Query i of the
 * sequence sits at position L - q_len + i and sees keys 0 .. L - q_len + i
 * (causal, bottom-right aligned), so n_vis = clamp(L - q_len + i + 1, 0, L).
 * Key j lives at page block_table[b][j / bs], offset j % bs.  Query head h
 * reads KV head h / G, G = Hq / Hkv.
 *
 * When num_splits > 0 only the keys of segment `split` are used: with
 * P = ceil(L / bs) pages and pps = ceil(P / num_splits) pages per segment,
 * segment s covers pages [s*pps, min((s+1)*pps, P)); the keys it contributes
 * are those of its pages that are also visible to the row.
 *
 * out[0 .. dv) = sum_j softmax_j * V_j and *lse = m + log(sum exp(s_j - m)),
 * computed in two passes (max, then sums).  No visible key: out = 0 and
 * lse = -inf ([MiMo-2xRTX] "Update 2026-10-01": such rows are 0, never NaN).
 *
 * Attention sink ([MiMo-2xRTX] "Update 2026-10-01", vLLM #58235: the sink is
 * an extra softmax-denominator logit): `sink` is one more logit with no value
 * vector, out = sum_j exp(s_j) V_j / (exp(sink) + sum_j exp(s_j)) and
 * lse = log(exp(sink) + sum_j exp(s_j)).  sink = -inf is no sink.  With a
 * finite sink a row without visible keys is 0 with lse = sink.
 */
static void attend_row(const uint16_t *q_row, const void *cache,
                       const oracle_cache_desc *d, const int32_t *bt_row,
                       int64_t key_lo, int64_t key_hi, int g, double scale,
                       double ks, double vs, double sink, double *out,
                       double *lse)
{
    int64_t j;
    int i;
    double m = sink, l;
    int dk = d->head_size, dv = d->head_size_v;

    for (i = 0; i < dv; ++i)
        out[i] = 0.0;
    if (key_hi <= key_lo) {
        *lse = sink;
        return;
    }
    /* pass 1: the row maximum of the scaled scores (and the sink) */
    for (j = key_lo; j < key_hi; ++j) {
        int64_t row = row_offset_elems(d, bt_row[j / d->block_size],
                                       j % d->block_size, g);
        double s = 0.0;
        for (i = 0; i < dk; ++i)
            s += oracle_bf16_to_double(q_row[i]) *
                 cache_read(cache, d, row + d->k_off + i, ks);
        s *= scale;
        if (s > m)
            m = s;
    }
    /* pass 2: exponentials, their sum (the sink's term first) and the
     * weighted sum of V */
    l = exp(sink - m);
    for (j = key_lo; j < key_hi; ++j) {
        int64_t row = row_offset_elems(d, bt_row[j / d->block_size],
                                       j % d->block_size, g);
        double s = 0.0, p;
        for (i = 0; i < dk; ++i)
            s += oracle_bf16_to_double(q_row[i]) *
                 cache_read(cache, d, row + d->k_off + i, ks);
        s *= scale;
        p = exp(s - m);
        l += p;
        for (i = 0; i < dv; ++i)
            out[i] += p * cache_read(cache, d, row + d->v_off + i, vs);
    }
    for (i = 0; i < dv; ++i)
        out[i] /= l;
    *lse = m + log(l);
}

/* Page range [*plo, *phi) of segment `split` of sequence b, the pages of
 * the sequence being P = ceil(L / block_size).
 *
 * Equal segments (split_ranges == 0; the split-KV of [MiMo-2xRTX] "What the
 * kernels do" with page-aligned segments): pps = ceil(P / num_splits) pages
 * per segment, segment s = [s * pps, min((s + 1) * pps, P)).
 *
 * Balanced ranges (split_ranges = W > 0; split selection from the sequence
 * lengths on the device, [PR50371] discussion): the pages of all sequences
 * are laid end to end in sequence order, sequence b starting at global page
 * G_b = sum of P over the sequences before it, Ptot pages in all.  That line
 * is cut into ranges of R pages, R = max(ceil(Ptot / W), Rmin, 1), where
 * Rmin keeps every sequence within num_splits segments: Rmin = Ptot when
 * num_splits is 1, else floor(max(Pmax - 2, 0) / (num_splits - 1)) + 1
 * (Pmax the largest P; a sequence of P >= 2 pages meets at most
 * floor((P - 2) / R) + 2 ranges).  Segment s of sequence b is the part of
 * the sequence inside range floor(G_b / R) + s, in the sequence's own page
 * numbers; it is empty when that range holds none of its pages. */
static void segment_pages(const int32_t *seq_lens, int num_seqs, int b,
                          int block_size, int num_splits, int split_ranges,
                          int split, int64_t *plo, int64_t *phi)
{
    int64_t P = ((int64_t)seq_lens[b] + block_size - 1) / block_size;
    if (split_ranges <= 0) {
        int64_t pps = (P + num_splits - 1) / num_splits;
        int64_t lo = (int64_t)split * pps, hi = lo + pps;
        *plo = lo < P ? lo : P;
        *phi = hi < P ? hi : P;
    } else {
        int64_t Ptot = 0, Pmax = 0, G = 0, R, Rmin, r, lo, hi;
        int i;
        for (i = 0; i < num_seqs; ++i) {
            int64_t Pi = ((int64_t)seq_lens[i] + block_size - 1) / block_size;
            if (i < b)
                G += Pi;
            Ptot += Pi;
            if (Pi > Pmax)
                Pmax = Pi;
        }
        R = (Ptot + split_ranges - 1) / split_ranges;
        if (num_splits == 1)
            Rmin = Ptot;
        else
            Rmin = (Pmax > 2 ? Pmax - 2 : 0) / (num_splits - 1) + 1;
        if (R < Rmin)
            R = Rmin;
        if (R < 1)
            R = 1;
        r = G / R + split;            /* the range of segment `split` */
        lo = r * R > G ? r * R : G;   /* its global pages, clipped to b */
        hi = (r + 1) * R < G + P ? (r + 1) * R : G + P;
        if (hi < lo)
            hi = lo;
        *plo = lo - G;
        *phi = hi - G;
    }
}

/* Attention over the paged cache for a list of query tokens.
 *
 * tokens[0 .. n_tokens) selects the query tokens (global token indices);
 * tokens == NULL means all num_tokens of them.  q is [num_tokens][Hq][dk]
 * bf16 (raw bits), out_o is [n][Hq][dv] and out_lse is [n][Hq], binary64.
 * split < 0 computes the whole row; otherwise the partial of segment
 * `split` of `num_splits`, cut as segment_pages describes (equal segments
 * when split_ranges is 0, balanced ranges otherwise).  Returns 0, or -1
 * when a token index is outside every sequence.  sinks (NULL: none) holds
 * one sink logit per query head; it enters whole rows only (split < 0): a
 * segment's partial is sink-free and the merge adds the sink once. */
int oracle_paged_attn(const uint16_t *q, int num_q_heads, int num_tokens,
                      const void *cache, const oracle_cache_desc *d,
                      const int32_t *block_table, int max_blocks_per_seq,
                      const int32_t *seq_lens, const int32_t *query_start_loc,
                      int num_seqs, float softmax_scale, const float *k_scale,
                      const float *v_scale, const int32_t *tokens, int n_tokens,
                      int num_splits, int split, int split_ranges, double *out_o,
                      double *out_lse, const float *sinks)
{
    int n = tokens ? n_tokens : num_tokens;
    int G = num_q_heads / d->num_kv_heads;
    int k, h, b;
    for (k = 0; k < n; ++k) {
        int t = tokens ? tokens[k] : k;
        int64_t L, qlen, i, n_vis, lo, hi;
        const int32_t *bt_row;
        for (b = 0; b < num_seqs; ++b)
            if (t >= query_start_loc[b] && t < query_start_loc[b + 1])
                break;
        if (b == num_seqs)
            return -1;
        L = seq_lens[b];
        qlen = query_start_loc[b + 1] - query_start_loc[b];
        i = t - query_start_loc[b];
        n_vis = L - qlen + i + 1;
        if (n_vis < 0)
            n_vis = 0;
        if (n_vis > L)
            n_vis = L;
        lo = 0;
        hi = n_vis;
        if (split >= 0) {
            int64_t plo, phi;
            segment_pages(seq_lens, num_seqs, b, d->block_size, num_splits,
                          split_ranges, split, &plo, &phi);
            lo = plo * d->block_size;
            if (phi * d->block_size < hi)
                hi = phi * d->block_size;
        }
        bt_row = block_table + (int64_t)b * max_blocks_per_seq;
        for (h = 0; h < num_q_heads; ++h) {
            int g = h / G;
            attend_row(q + ((int64_t)t * num_q_heads + h) * d->head_size, cache,
                       d, bt_row, lo, hi, g, (double)softmax_scale,
                       (double)scale_of(k_scale, d->scale_mode, g),
                       (double)scale_of(v_scale, d->scale_mode, g),
                       (sinks && split < 0) ? (double)sinks[h] : -INFINITY,
                       out_o + ((int64_t)k * num_q_heads + h) * d->head_size_v,
                       out_lse + (int64_t)k * num_q_heads + h);
        }
    }
    return 0;
}

/* ------------------------------------------------------- split-KV merge --- */

/* Merge of split-KV partials ([MiMo-2xRTX] "What the kernels do" and
 * "Update 2026-10-01"; [PR50371] discussion of the two-stage split decode).
 * For each row r: M = max_s lse[s][r].  If M is -inf no segment saw a key and
 * the row is 0 with lse -inf.  Otherwise w_s = exp(lse_s - M) (0 for empty
 * segments), out = sum_s w_s * o_s / sum_s w_s and lse = M + log(sum_s w_s).
 * partial_o is [S][rows][dv] and partial_lse [S][rows] (binary32, the
 * library's partial format); o_s of an empty segment is never read.
 * sinks (NULL: none): the sink logit of row r is sinks[r % num_q_heads] (rows
 * are (token, query head) pairs); it joins the merge as one more segment
 * with lse = sink and o = 0, so M also covers it and W gains exp(sink - M):
 * a row whose segments are all empty is then 0 with lse = sink. */
void oracle_splitkv_reduce(const float *partial_o, const float *partial_lse,
                           int num_splits, int64_t rows, int dv, double *out,
                           double *lse_out, const float *sinks, int num_q_heads)
{
    int64_t r;
    int s, i;
    for (r = 0; r < rows; ++r) {
        double sink = sinks ? (double)sinks[r % num_q_heads] : -INFINITY;
        double M = sink, W;
        double *o = out + r * dv;
        for (i = 0; i < dv; ++i)
            o[i] = 0.0;
        for (s = 0; s < num_splits; ++s) {
            double x = partial_lse[(int64_t)s * rows + r];
            if (x > M)
                M = x;
        }
        if (M == -INFINITY) {
            lse_out[r] = -INFINITY;
            continue;
        }
        W = exp(sink - M);
        for (s = 0; s < num_splits; ++s) {
            double x = partial_lse[(int64_t)s * rows + r];
            double w;
            if (x == -INFINITY)
                continue;
            w = exp(x - M);
            W += w;
            for (i = 0; i < dv; ++i)
                o[i] += w * partial_o[((int64_t)s * rows + r) * dv + i];
        }
        for (i = 0; i < dv; ++i)
            o[i] /= W;
        lse_out[r] = M + log(W);
    }
}
