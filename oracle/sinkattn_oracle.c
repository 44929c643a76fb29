/*
 * fp64 CPU oracle for paged grouped-query attention with per-head attention sinks.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header or table with
 * the CUDA library: it walks the block tables itself, converts bf16 to double itself
 * and evaluates the attention in double precision straight from its definition.
 *
 * What is computed (sources are the extracted pages "GPT-OSS on Day 0"
 * (perplexity.ai, section "Sink Attention"), "Hosting Qwen on Blackwell"
 * (perplexity.ai, KV-cache layout paragraph of "Prefill") and TensorSharp
 * "docs/models/gptoss.md" (section 3 "Forward graph" and section 4.1 "Attention")):
 *
 *   For query head h with KV head g = h / (Hq / Hkv), query vector q and the set J
 *   of keys the query may see:
 *       s_j  = scale * <q, k_j>
 *       m    = max(sink_h, max_j s_j)
 *       den  = exp(sink_h - m) + sum_j exp(s_j - m)
 *       out  = sum_j exp(s_j - m) * v_j / den
 *       lse  = m + ln(den)
 *   i.e. softmax attention over J plus one virtual token whose logit is sink_h and
 *   whose value is the zero vector (gptoss.md 4.1: a virtual token with zero K and V;
 *   section 3: the sink term enters the max and the exp-sum, not the numerator).
 *   A NULL sinks pointer means every sink is -inf (plain GQA attention).
 *
 *   J is: decode - every cached token [0, L_b); causal prefill - tokens 0..t of the
 *   same sequence; chunked prefill - all P_i prefix tokens plus new tokens 0..t,
 *   the new token t sitting at absolute position P_i + t; non-causal prefill (an
 *   encoder without a KV cache) - every token of the same sequence.
 *
 *   Sliding window W > 0 (gptoss.md section 4: even layers attend a local window of
 *   128 positions, odd layers the full causal range; the window is passed per call to
 *   the paged kernel): J keeps only the keys at absolute positions pos - W < j <= pos,
 *   pos being the query's own position (decode: L_b - 1).  W <= 0: no window.
 *
 *   KV pages are HND: [num_pages, Hkv, page_size, head_dim], the tokens of one
 *   (page, head) contiguous (Hosting Qwen on Blackwell, KV-cache layout paragraph).
 *   Token j of sequence b lives in page block_table[b][j / page_size], slot
 *   j % page_size.
 *
 * Conventions where the pages are silent:
 *   - the sink is a raw logit in the same (already scaled) domain as s_j;
 *   - exp and log are natural; lse includes the sink term;
 *   - no visible key and no sink (m = -inf): out = 0, lse = -inf.
 *
 * Also here, for checking the split-KV method the GPU uses (GPT-OSS on Day 0,
 * "Sink Attention": online softmax with the running max seeded by the sink; the
 * sink counted in one block only when the sequence is split):
 *   oracle_partial  - unnormalised state (m, l, acc) of one key range, no sink;
 *   oracle_merge    - log-sum-exp combination of partial states plus the sink;
 *   oracle_online   - block-by-block online softmax seeded with m = sink, d = 1.
 *
 * bf16 arguments are passed as raw uint16 bit patterns; outputs are double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sink_of(const float *sinks, int h) {
    return sinks ? (double)sinks[h] : -INFINITY;
}

/* The definition above, for one query over n keys given by row pointers.
 * s is caller scratch of n doubles. */
static void attend(const uint16_t *q, int D, double scale, double sink, int64_t n,
                   const uint16_t *const *krow, const uint16_t *const *vrow, double *s,
                   double *out, double *lse) {
    double m = sink;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(krow[j][d]);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    if (m == -INFINITY) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double den = exp(sink - m);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double w = exp(s[j] - m);
        den += w;
        for (int d = 0; d < D; ++d) out[d] += w * bf16_to_double(vrow[j][d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    *lse = m + log(den);
}

/* Address of token `slot` of KV head g in physical page `page` (HND layout). */
static const uint16_t *page_row(const uint16_t *pages, int64_t page, int Hkv, int P, int D, int g,
                                int slot) {
    return pages + (((page * Hkv + g) * (int64_t)P + slot) * D);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Decode: one query token per sequence.
 *   q [B, Hq, D]; k_pages, v_pages [num_pages, Hkv, P, D]; block_table [B, max_pages];
 *   seq_lens [B]; sinks [Hq] or NULL; out [B, Hq, D]; lse [B, Hq].
 *   select [B * Hq] or NULL: compute only entries with select != 0 (others untouched).
 * Returns 0, or -1 if a length or page index is out of range (nothing is read then).
 */
int oracle_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                  const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                  double scale, int B, int Hq, int Hkv, int D, int P, int64_t num_pages,
                  int max_pages, int window, const uint8_t *select, double *out, double *lse) {
    if (Hq % Hkv) return -1;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 0 || (int64_t)L > (int64_t)max_pages * P) return -1;
        for (int j = 0; j < (L + P - 1) / P; ++j) {
            int32_t pg = block_table[(int64_t)b * max_pages + j];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
        if (select && !select[bh]) continue;
        const int b = (int)(bh / Hq), h = (int)(bh % Hq), g = h / G;
        const int64_t L = seq_lens[b];
        /* keys [lo, L): the query sits at position L - 1 */
        const int64_t lo = (window > 0 && L > window) ? L - window : 0;
        const int64_t nk = L - lo;
        const uint16_t **krow = malloc(sizeof(*krow) * (size_t)(nk + 1));
        const uint16_t **vrow = malloc(sizeof(*vrow) * (size_t)(nk + 1));
        double *s = malloc(sizeof(double) * (size_t)(nk + 1));
        if (!krow || !vrow || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
            for (int64_t j = lo; j < L; ++j) {
                int64_t pg = block_table[(int64_t)b * max_pages + j / P];
                krow[j - lo] = page_row(k_pages, pg, Hkv, P, D, g, (int)(j % P));
                vrow[j - lo] = page_row(v_pages, pg, Hkv, P, D, g, (int)(j % P));
            }
            attend(q + bh * D, D, scale, sink_of(sinks, h), nk, krow, vrow, s, out + bh * D,
                   lse + bh);
        }
        free(krow);
        free(vrow);
        free(s);
    }
    return bad ? -2 : 0;
}

/*
 * Prefill over packed ragged sequences, optionally after a paged prefix.
 *   q [T, Hq, D]; k, v [T, Hkv, D] (new tokens); cu_seqlens [n + 1];
 *   prefix: k_pages / v_pages [num_pages, Hkv, P, D], prefix_block_table [n, max_pages],
 *   prefix_lens [n]; all NULL for a plain causal prefill.
 *   out [T, Hq, D]; lse [T, Hq]; select [T * Hq] or NULL.
 */
int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *cu_seqlens, int n, const uint16_t *k_pages,
                   const uint16_t *v_pages, const int32_t *prefix_block_table,
                   const int32_t *prefix_lens, int64_t num_pages, int max_pages,
                   const float *sinks, double scale, int Hq, int Hkv, int D, int P, int window,
                   const uint8_t *select, double *out, double *lse) {
    if (Hq % Hkv) return -1;
    const int G = Hq / Hkv;
    const int64_t T = cu_seqlens[n];
    int32_t *seq_of = malloc(sizeof(int32_t) * (size_t)(T + 1));
    if (!seq_of) return -2;
    for (int i = 0; i < n; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i]) { free(seq_of); return -1; }
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) seq_of[t] = i;
        int Pi = prefix_lens ? prefix_lens[i] : 0;
        if (Pi < 0 || (Pi > 0 && (int64_t)Pi > (int64_t)max_pages * P)) { free(seq_of); return -1; }
        for (int j = 0; j < (Pi + P - 1) / P; ++j) {
            int32_t pg = prefix_block_table[(int64_t)i * max_pages + j];
            if (pg < 0 || pg >= num_pages) { free(seq_of); return -1; }
        }
    }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t th = 0; th < T * Hq; ++th) {
        if (select && !select[th]) continue;
        const int64_t t = th / Hq;
        const int h = (int)(th % Hq), g = h / G, i = seq_of[t];
        const int64_t Pi = prefix_lens ? prefix_lens[i] : 0;
        const int64_t tl = t - cu_seqlens[i]; /* position among the new tokens */
        const int64_t pos = Pi + tl;           /* absolute position of the query */
        /* keys at absolute positions [lo, pos]: prefix 0..Pi-1, then new tokens */
        const int64_t lo = (window > 0 && pos + 1 > window) ? pos + 1 - window : 0;
        const int64_t nk = pos + 1 - lo;
        const uint16_t **krow = malloc(sizeof(*krow) * (size_t)nk);
        const uint16_t **vrow = malloc(sizeof(*vrow) * (size_t)nk);
        double *s = malloc(sizeof(double) * (size_t)nk);
        if (!krow || !vrow || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
            for (int64_t j = lo; j <= pos; ++j) {
                if (j < Pi) {
                    int64_t pg = prefix_block_table[(int64_t)i * max_pages + j / P];
                    krow[j - lo] = page_row(k_pages, pg, Hkv, P, D, g, (int)(j % P));
                    vrow[j - lo] = page_row(v_pages, pg, Hkv, P, D, g, (int)(j % P));
                } else {
                    int64_t row = cu_seqlens[i] + (j - Pi);
                    krow[j - lo] = k + (row * Hkv + g) * D;
                    vrow[j - lo] = v + (row * Hkv + g) * D;
                }
            }
            attend(q + th * D, D, scale, sink_of(sinks, h), nk, krow, vrow, s, out + th * D,
                   lse + th);
        }
        free(krow);
        free(vrow);
        free(s);
    }
    free(seq_of);
    return bad ? -2 : 0;
}

/*
 * Non-causal prefill over packed ragged sequences, without a KV cache: the attention of
 * an embedding (encoder) model served through ragged kernels with no KV cache ("Fast
 * embeddings on GPUs", the section on attention kernels).  The pages give no mask for
 * it; the reading here is the plain bidirectional one: query t of sequence i sees
 * every token of sequence i, before and after it, and nothing outside it.
 *   q [T, Hq, D]; k, v [T, Hkv, D]; cu_seqlens [n + 1]; out [T, Hq, D]; lse [T, Hq].
 */
int oracle_prefill_noncausal(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const int32_t *cu_seqlens, int n, const float *sinks, double scale,
                             int Hq, int Hkv, int D, const uint8_t *select, double *out,
                             double *lse) {
    if (Hq % Hkv) return -1;
    for (int i = 0; i < n; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i]) return -1;
    const int G = Hq / Hkv;
    int bad = 0;
    for (int i = 0; i < n; ++i) {
        const int64_t first = cu_seqlens[i], len = cu_seqlens[i + 1] - cu_seqlens[i];
        if (len == 0) continue;
        /* the same key set for every query of the sequence */
        const uint16_t **krow = malloc(sizeof(*krow) * (size_t)len * Hkv);
        const uint16_t **vrow = malloc(sizeof(*vrow) * (size_t)len * Hkv);
        if (!krow || !vrow) {
            free(krow);
            free(vrow);
            return -2;
        }
        for (int g = 0; g < Hkv; ++g)
            for (int64_t j = 0; j < len; ++j) {
                krow[g * len + j] = k + ((first + j) * Hkv + g) * D;
                vrow[g * len + j] = v + ((first + j) * Hkv + g) * D;
            }
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t e = 0; e < len * Hq; ++e) {
            const int64_t th = first * Hq + e; /* (token, head) pair */
            if (select && !select[th]) continue;
            const int h = (int)(e % Hq);
            double *s = malloc(sizeof(double) * (size_t)len);
            if (!s) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            attend(q + th * D, D, scale, sink_of(sinks, h), len, krow + (h / G) * len,
                   vrow + (h / G) * len, s, out + th * D, lse + th);
            free(s);
        }
        free(krow);
        free(vrow);
    }
    return bad ? -2 : 0;
}

/*
 * Append new K/V rows into HND pages (each layer stores its K and V in the cache before
 * its attention, gptoss.md section 3).  Token t of sequence i goes to position
 * pos = start_pos[i] + (t - cu_seqlens[i]): page block_table[i][pos / P], slot pos % P.
 * Copies bit patterns; pages are modified in place.  Returns -1 (nothing written)
 * if any destination is out of range.
 */
int oracle_append_kv(const uint16_t *k, const uint16_t *v, const int32_t *cu_seqlens, int n,
                     const int32_t *block_table, const int32_t *start_pos, int max_pages,
                     int64_t num_pages, int Hkv, int D, int P, uint16_t *k_pages,
                     uint16_t *v_pages) {
    for (int i = 0; i < n; ++i) {
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
            int64_t pos = start_pos[i] + (t - cu_seqlens[i]);
            if (pos < 0 || pos / P >= max_pages) return -1;
            int32_t pg = block_table[(int64_t)i * max_pages + pos / P];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    for (int i = 0; i < n; ++i) {
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
            int64_t pos = start_pos[i] + (t - cu_seqlens[i]);
            int64_t pg = block_table[(int64_t)i * max_pages + pos / P];
            for (int g = 0; g < Hkv; ++g) {
                uint16_t *kd = (uint16_t *)page_row(k_pages, pg, Hkv, P, D, g, (int)(pos % P));
                uint16_t *vd = (uint16_t *)page_row(v_pages, pg, Hkv, P, D, g, (int)(pos % P));
                memcpy(kd, k + (t * Hkv + g) * D, sizeof(uint16_t) * (size_t)D);
                memcpy(vd, v + (t * Hkv + g) * D, sizeof(uint16_t) * (size_t)D);
            }
        }
    }
    return 0;
}

/*
 * Split-KV pieces, on contiguous keys k, v [n, D] and one query q [D].
 *
 * oracle_partial: state of keys [j0, j1) without the sink:
 *   m = max s_j (-inf if the range is empty), l = sum exp(s_j - m),
 *   acc = sum exp(s_j - m) v_j.
 */
void oracle_partial(const uint16_t *q, const uint16_t *k, const uint16_t *v, int D, double scale,
                    int64_t j0, int64_t j1, double *m_out, double *l_out, double *acc) {
    double m = -INFINITY;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(k[j * D + d]);
        if (scale * dot > m) m = scale * dot;
    }
    double l = 0.0;
    if (m > -INFINITY) {
        for (int64_t j = j0; j < j1; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(k[j * D + d]);
            double w = exp(scale * dot - m);
            l += w;
            for (int d = 0; d < D; ++d) acc[d] += w * bf16_to_double(v[j * D + d]);
        }
    }
    *m_out = m;
    *l_out = l;
}

/* oracle_merge: combine S partial states (m[s], l[s], acc[s][D]) and the sink:
 *   M = max(sink, max_s m_s); den = exp(sink - M) + sum_s l_s exp(m_s - M);
 *   out = sum_s acc_s exp(m_s - M) / den; lse = M + ln(den). */
void oracle_merge(int S, const double *m, const double *l, const double *acc, int D, double sink,
                  double *out, double *lse) {
    double M = sink;
    for (int s = 0; s < S; ++s)
        if (m[s] > M) M = m[s];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double den = exp(sink - M);
    for (int s = 0; s < S; ++s) {
        if (m[s] == -INFINITY) continue;
        double w = exp(m[s] - M);
        den += l[s] * w;
        for (int d = 0; d < D; ++d) out[d] += acc[s * D + d] * w;
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
    *lse = M + log(den);
}

/* oracle_online: the streaming form, keys visited in blocks of `block` keys.
 * The running max starts at the sink and the running denominator at 1
 * (= exp(sink - m) with m = sink); each block raises the max, rescales the
 * denominator and the accumulator by exp(m_old - m_new) and adds its own terms.
 * When split_at > 0 the keys are cut at that index into two independent
 * streams, only the first of which is seeded with the sink; the two states are
 * then combined with oracle_merge's rule (sink already counted, so -inf there). */
static void online_range(const uint16_t *q, const uint16_t *k, const uint16_t *v, int D,
                         double scale, int64_t j0, int64_t j1, int block, double m0, double d0,
                         double *m_out, double *d_out, double *acc) {
    double m = m0, den = d0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int64_t b0 = j0; b0 < j1; b0 += block) {
        int64_t b1 = b0 + block < j1 ? b0 + block : j1;
        double mb = m;
        for (int64_t j = b0; j < b1; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(k[j * D + d]);
            if (scale * dot > mb) mb = scale * dot;
        }
        if (mb == -INFINITY) continue;
        double r = (m == -INFINITY) ? 0.0 : exp(m - mb);
        den *= r;
        for (int d = 0; d < D; ++d) acc[d] *= r;
        for (int64_t j = b0; j < b1; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(k[j * D + d]);
            double w = exp(scale * dot - mb);
            den += w;
            for (int d = 0; d < D; ++d) acc[d] += w * bf16_to_double(v[j * D + d]);
        }
        m = mb;
    }
    *m_out = m;
    *d_out = den;
}

void oracle_online(const uint16_t *q, const uint16_t *k, const uint16_t *v, int D, double scale,
                   double sink, int64_t n, int block, int64_t split_at, double *out, double *lse) {
    double *acc = malloc(sizeof(double) * 2 * (size_t)D);
    double m[2], den[2];
    if (!acc) return;
    int64_t cut = (split_at > 0 && split_at < n) ? split_at : n;
    /* first stream: seeded with the sink (d0 = 1 means exp(sink - m0) with m0 = sink;
     * when the sink is -inf that term is 0 and the first block's rescale zeroes it). */
    online_range(q, k, v, D, scale, 0, cut, block, sink, sink == -INFINITY ? 0.0 : 1.0, &m[0],
                 &den[0], acc);
    int S = 1;
    if (cut < n) {
        online_range(q, k, v, D, scale, cut, n, block, -INFINITY, 0.0, &m[1], &den[1], acc + D);
        S = 2;
    }
    oracle_merge(S, m, den, acc, D, -INFINITY, out, lse);
    free(acc);
}

/* ------------------------------------------------------------------------------
 * FP8 KV cache.  The pages name an FP8 serving precision ("GPT-OSS on Day 0",
 * section "GPT-OSS on Hopper") and an 8-bit KV-cache type (TensorSharp gptoss.md
 * section 10, "Memory and KV cache strategy") but give no scale convention.  The
 * reading taken here: each K/V element is one OCP FP8 E4M3 code (1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN;
 * largest finite 448), and its value is scale[g] * e4m3(code) with one fp32 scale
 * per KV head g, separately for K and for V.
 *
 * Quantisation (the fp8 append): x is the bf16 value as float; y = x / scale[g] in
 * IEEE single precision (round to nearest); the code is y rounded to the nearest
 * E4M3 value, ties to the even mantissa, with finite overflow and infinities
 * saturated to +-448 and NaN kept NaN (0x7F with the sign bit of y).
 */

/* The value of an E4M3 code, from the format's definition. */
double oracle_e4m3_value(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
    else
        mag = ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* Nearest E4M3 code of a float (ties to even, saturating, NaN preserved). */
uint8_t oracle_e4m3_code(float y) {
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    if (isnan(y)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* saturation: 448 is code 0x7E */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; rint rounds half to even */
        double q = rint(ldexp(a, 9)); /* 0..8; 8 is the smallest normal, code 0x08 */
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e2;
    frexp(a, &e2);    /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;   /* a in [2^e, 2^(e+1)), e in [-6, 8] */
    double q = rint(ldexp(a, 3 - e)); /* 8..16: significand with 3 fraction bits */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    int field = e + 7; /* 1..15 */
    if (field > 15 || (field == 15 && q - 8.0 > 6.0)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)(field << 3) | (uint8_t)(q - 8.0));
}

/* attend() over E4M3 rows: the key and value elements are scale * e4m3(code). */
static void attend_e4m3(const uint16_t *q, int D, double scale, double sink, int64_t n,
                        const uint8_t *const *krow, const uint8_t *const *vrow, double kscale,
                        double vscale, double *s, double *out, double *lse) {
    double top = sink; /* m of the definition */
    for (int64_t j = 0; j < n; ++j) {
        double qk = 0.0;
        for (int d = 0; d < D; ++d)
            qk += bf16_to_double(q[d]) * (kscale * oracle_e4m3_value(krow[j][d]));
        s[j] = scale * qk;
        if (s[j] > top) top = s[j];
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (top == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = exp(sink - top); /* the denominator, starting with the sink's term */
    for (int64_t j = 0; j < n; ++j) {
        double e = exp(s[j] - top);
        z += e;
        for (int d = 0; d < D; ++d) out[d] += e * (vscale * oracle_e4m3_value(vrow[j][d]));
    }
    for (int d = 0; d < D; ++d) out[d] /= z;
    *lse = top + log(z);
}

/*
 * Decode over an FP8 E4M3 cache: oracle_decode with byte pages
 * k_pages, v_pages uint8 [num_pages, Hkv, P, D] and fp32 scales k_scale, v_scale [Hkv]
 * (NULL: 1).  Same visible keys, sinks, window and return codes.
 */
int oracle_decode_fp8(const uint16_t *q, const uint8_t *k_pages, const uint8_t *v_pages,
                      const float *k_scale, const float *v_scale, const int32_t *block_table,
                      const int32_t *seq_lens, const float *sinks, double scale, int B, int Hq,
                      int Hkv, int D, int P, int64_t num_pages, int max_pages, int window,
                      const uint8_t *select, double *out, double *lse) {
    if (Hq % Hkv) return -1;
    const int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        if (L < 0 || (int64_t)L > (int64_t)max_pages * P) return -1;
        for (int j = 0; j < (L + P - 1) / P; ++j) {
            int32_t pg = block_table[(int64_t)b * max_pages + j];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
        if (select && !select[bh]) continue;
        const int b = (int)(bh / Hq), h = (int)(bh - (int64_t)b * Hq), g = h / G;
        const int64_t L = seq_lens[b];
        const int64_t first = (window > 0 && L > window) ? L - window : 0; /* first visible key */
        const int64_t nk = L - first;
        const uint8_t **krow = malloc(sizeof(*krow) * (size_t)(nk + 1));
        const uint8_t **vrow = malloc(sizeof(*vrow) * (size_t)(nk + 1));
        double *s = malloc(sizeof(double) * (size_t)(nk + 1));
        if (!krow || !vrow || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
            for (int64_t j = first; j < L; ++j) {
                int64_t pg = block_table[(int64_t)b * max_pages + j / P];
                int64_t off = ((pg * Hkv + g) * (int64_t)P + j % P) * D;
                krow[j - first] = k_pages + off;
                vrow[j - first] = v_pages + off;
            }
            attend_e4m3(q + bh * D, D, scale, sink_of(sinks, h), nk, krow, vrow,
                        k_scale ? (double)k_scale[g] : 1.0, v_scale ? (double)v_scale[g] : 1.0, s,
                        out + bh * D, lse + bh);
        }
        free(krow);
        free(vrow);
        free(s);
    }
    return bad ? -2 : 0;
}

/*
 * Append into an FP8 E4M3 cache: token placement as oracle_append_kv; each element
 * x (bf16) is stored as oracle_e4m3_code(x / scale[g]), the division in single
 * precision.  k_scale, v_scale [Hkv] (NULL: 1).
 */
int oracle_append_kv_fp8(const uint16_t *k, const uint16_t *v, const float *k_scale,
                         const float *v_scale, const int32_t *cu_seqlens, int n,
                         const int32_t *block_table, const int32_t *start_pos, int max_pages,
                         int64_t num_pages, int Hkv, int D, int P, uint8_t *k_pages,
                         uint8_t *v_pages) {
    for (int i = 0; i < n; ++i) {
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
            int64_t pos = start_pos[i] + (t - cu_seqlens[i]);
            if (pos < 0 || pos / P >= max_pages) return -1;
            int32_t pg = block_table[(int64_t)i * max_pages + pos / P];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    for (int i = 0; i < n; ++i) {
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) {
            int64_t pos = start_pos[i] + (t - cu_seqlens[i]);
            int64_t pg = block_table[(int64_t)i * max_pages + pos / P];
            for (int g = 0; g < Hkv; ++g) {
                const float ks = k_scale ? k_scale[g] : 1.0f, vs = v_scale ? v_scale[g] : 1.0f;
                int64_t off = ((pg * Hkv + g) * (int64_t)P + pos % P) * D;
                for (int d = 0; d < D; ++d) {
                    float kx = (float)bf16_to_double(k[(t * Hkv + g) * D + d]);
                    float vx = (float)bf16_to_double(v[(t * Hkv + g) * D + d]);
                    k_pages[off + d] = oracle_e4m3_code(kx / ks);
                    v_pages[off + d] = oracle_e4m3_code(vx / vs);
                }
            }
        }
    }
    return 0;
}

/* Element-wise oracle_e4m3_code / oracle_e4m3_value over arrays. */
void oracle_e4m3_codes(const float *y, int64_t n, uint8_t *codes) {
    for (int64_t i = 0; i < n; ++i) codes[i] = oracle_e4m3_code(y[i]);
}

void oracle_e4m3_values(const uint8_t *codes, int64_t n, double *values) {
    for (int64_t i = 0; i < n; ++i) values[i] = oracle_e4m3_value(codes[i]);
}

/* ------------------------------------------------------------------------------
 * Rotary position embedding, NeoX layout, with YaRN frequency scaling: the step the
 * pages put on Q and K right before the K/V append and the attention (TensorSharp
 * gptoss.md section 3 "Forward graph": RoPE_NeoX with YaRN scaling, original context
 * 4096, freqScale = 1 / RopeScale, beta_fast = 32, beta_slow = 1; section 4.1
 * "Attention"; "GPT-OSS on Day 0": YaRN position encoding as in DeepSeek-V3).  The pages
 * name the parameters only.  The reading taken - the YaRN "by parts" interpolation as
 * the rotary routine those pages call computes it:
 *   - NeoX layout: element i < D/2 forms a pair with element i + D/2;
 *   - base frequency of pair i: w_i = base^(-2i/D) radians per position;
 *   - the pair index at which a full turn takes L0 / r positions (r turns over the
 *     original context L0): c(r) = D ln(L0 / (2 pi r)) / (2 ln base);
 *     lo = max(0, floor(c(beta_fast))), hi = min(D - 1, ceil(c(beta_slow)));
 *   - blend over the pair index, y_i = clamp((i - lo) / max(0.001, hi - lo), 0, 1):
 *     theta_i = (1 - y_i) w_i + y_i w_i / factor  (fast pairs keep their frequency,
 *     slow pairs are interpolated by the factor, a linear ramp in between);
 *   - magnitude: mscale = 1 + 0.1 ln(factor) multiplies both outputs of every pair;
 *   - at position p, with a = p theta_i:
 *       out[i]       = mscale (x[i] cos a - x[i + D/2] sin a)
 *       out[i + D/2] = mscale (x[i + D/2] cos a + x[i] sin a).
 * The rotated query and key are bf16 activations: rounded to the nearest bf16 value,
 * ties to even, when they are used (oracle_bf16_round).
 */
void oracle_rope_freqs(int D, double base, double factor, int L0, double beta_fast,
                       double beta_slow, double *theta, double *mscale) {
    const double two_pi = 2.0 * acos(-1.0);
    double lo = floor(D * log(L0 / (two_pi * beta_fast)) / (2.0 * log(base)));
    double hi = ceil(D * log(L0 / (two_pi * beta_slow)) / (2.0 * log(base)));
    if (lo < 0.0) lo = 0.0;
    if (hi > D - 1) hi = D - 1;
    const double span = (hi - lo) > 0.001 ? (hi - lo) : 0.001;
    for (int i = 0; i < D / 2; ++i) {
        const double w = pow(base, -2.0 * i / D);
        double y = (i - lo) / span;
        if (y < 0.0) y = 0.0;
        if (y > 1.0) y = 1.0;
        theta[i] = (1.0 - y) * w + y * (w / factor);
    }
    *mscale = 1.0 + 0.1 * log(factor);
}

/* Rotate rows x [n, H, D] (bf16 bits): row r at position pos[r], every head the same
 * way; out [n, H, D] in double (not rounded). */
void oracle_rope(const uint16_t *x, int64_t n, int H, int D, const int64_t *pos, double base,
                 double factor, int L0, double beta_fast, double beta_slow, double *out) {
    double *theta = malloc(sizeof(double) * (size_t)(D / 2));
    double ms;
    if (!theta) return;
    oracle_rope_freqs(D, base, factor, L0, beta_fast, beta_slow, theta, &ms);
    for (int64_t r = 0; r < n; ++r)
        for (int h = 0; h < H; ++h) {
            const uint16_t *xr = x + (r * H + h) * D;
            double *o = out + (r * H + h) * D;
            for (int i = 0; i < D / 2; ++i) {
                const double a = (double)pos[r] * theta[i];
                const double c = cos(a), s = sin(a);
                const double x0 = bf16_to_double(xr[i]), x1 = bf16_to_double(xr[i + D / 2]);
                o[i] = ms * (x0 * c - x1 * s);
                o[i + D / 2] = ms * (x1 * c + x0 * s);
            }
        }
    free(theta);
}

/* The bf16 value nearest to x (ties to the even significand), as its bit pattern:
 * 8 significant bits, exponents down to the subnormal step 2^-133, +-inf past the
 * largest finite value, NaN kept. */
uint16_t oracle_bf16_round(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
    int e;
    frexp(x, &e);            /* |x| = f 2^e, f in [0.5, 1): the leading bit is 2^(e-1) */
    int ulp = e - 8;         /* 8 significant bits */
    if (ulp < -133) ulp = -133;
    double r = ldexp(rint(ldexp(x, -ulp)), ulp); /* rint: nearest, ties to even */
    float f = (float)r;      /* exact: r has at most 8 significant bits */
    if (fabs(r) > 3.3895313892515355e38) f = signbit(x) ? -INFINITY : INFINITY;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void oracle_bf16_round_array(const double *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}

/* ------------------------------------------------------------------------------
 * Chunked prefill over an FP8 E4M3 paged prefix: oracle_prefill with the prefix pages in
 * the FP8 cache convention above (value = scale[g] * e4m3(code), per KV head, separately
 * for K and V) and the new tokens' keys and values in bf16 as given.  Query t of request
 * i at absolute position P_i + t sees the prefix keys 0 .. P_i - 1 and the new keys 0 .. t
 * (with a window W > 0, only those at positions > P_i + t - W).
 */
static void attend_fp8_prefix(const uint16_t *q, int D, double scale, double sink, int64_t np,
                              const uint8_t *const *kp, const uint8_t *const *vp, double ks, double vs,
                              int64_t nn, const uint16_t *const *kn, const uint16_t *const *vn,
                              double *s, double *out, double *lse) {
    double m = sink;
    for (int64_t j = 0; j < np; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * (ks * oracle_e4m3_value(kp[j][d]));
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    for (int64_t j = 0; j < nn; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(kn[j][d]);
        s[np + j] = scale * dot;
        if (s[np + j] > m) m = s[np + j];
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double z = exp(sink - m); /* the denominator, from the sink's term */
    for (int64_t j = 0; j < np; ++j) {
        double wt = exp(s[j] - m);
        z += wt;
        for (int d = 0; d < D; ++d) out[d] += wt * (vs * oracle_e4m3_value(vp[j][d]));
    }
    for (int64_t j = 0; j < nn; ++j) {
        double wt = exp(s[np + j] - m);
        z += wt;
        for (int d = 0; d < D; ++d) out[d] += wt * bf16_to_double(vn[j][d]);
    }
    for (int d = 0; d < D; ++d) out[d] /= z;
    *lse = m + log(z);
}

int oracle_prefill_fp8(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *cu_seqlens, int n, const uint8_t *k_pages,
                       const uint8_t *v_pages, const float *k_scale, const float *v_scale,
                       const int32_t *prefix_block_table, const int32_t *prefix_lens,
                       int64_t num_pages, int max_pages, const float *sinks, double scale, int Hq,
                       int Hkv, int D, int P, int window, const uint8_t *select, double *out,
                       double *lse) {
    if (Hq % Hkv) return -1;
    const int G = Hq / Hkv;
    const int64_t T = cu_seqlens[n];
    int32_t *seq_of = malloc(sizeof(int32_t) * (size_t)(T + 1));
    if (!seq_of) return -2;
    for (int i = 0; i < n; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i]) { free(seq_of); return -1; }
        for (int64_t t = cu_seqlens[i]; t < cu_seqlens[i + 1]; ++t) seq_of[t] = i;
        int Pi = prefix_lens[i];
        if (Pi < 0 || (int64_t)Pi > (int64_t)max_pages * P) { free(seq_of); return -1; }
        for (int j = 0; j < (Pi + P - 1) / P; ++j) {
            int32_t pg = prefix_block_table[(int64_t)i * max_pages + j];
            if (pg < 0 || pg >= num_pages) { free(seq_of); return -1; }
        }
    }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t th = 0; th < T * Hq; ++th) {
        if (select && !select[th]) continue;
        const int64_t t = th / Hq;
        const int h = (int)(th % Hq), i = seq_of[t], g = h / G;
        const int64_t Pi = prefix_lens[i];
        const int64_t tl = t - cu_seqlens[i];
        const int64_t pos = Pi + tl;
        const int64_t lo = (window > 0 && pos >= window) ? pos - window + 1 : 0; /* first visible */
        /* visible prefix keys [lo, Pi) and new keys [max(lo, Pi) - Pi, tl] */
        const int64_t np = lo < Pi ? Pi - lo : 0;
        const int64_t n0 = lo > Pi ? lo - Pi : 0;
        const int64_t nn = tl + 1 - n0;
        const uint8_t **kp = malloc(sizeof(*kp) * (size_t)(np + 1));
        const uint8_t **vp = malloc(sizeof(*vp) * (size_t)(np + 1));
        const uint16_t **kn = malloc(sizeof(*kn) * (size_t)(nn + 1));
        const uint16_t **vn = malloc(sizeof(*vn) * (size_t)(nn + 1));
        double *s = malloc(sizeof(double) * (size_t)(np + nn + 1));
        if (!kp || !vp || !kn || !vn || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
            for (int64_t j = 0; j < np; ++j) {
                const int64_t key = lo + j;
                const int64_t pg = prefix_block_table[(int64_t)i * max_pages + key / P];
                const int64_t off = ((pg * Hkv + g) * (int64_t)P + key % P) * D;
                kp[j] = k_pages + off;
                vp[j] = v_pages + off;
            }
            for (int64_t j = 0; j < nn; ++j) {
                const int64_t row = cu_seqlens[i] + n0 + j;
                kn[j] = k + (row * Hkv + g) * D;
                vn[j] = v + (row * Hkv + g) * D;
            }
            attend_fp8_prefix(q + th * D, D, scale, sink_of(sinks, h), np, kp, vp,
                              k_scale == NULL ? 1.0 : (double)k_scale[g],
                              v_scale == NULL ? 1.0 : (double)v_scale[g],
                              nn, kn, vn, s, out + th * D, lse + th);
        }
        free(kp);
        free(vp);
        free(kn);
        free(vn);
        free(s);
    }
    free(seq_of);
    return bad ? -2 : 0;
}
