/*
 * smla_oracle.c -- CPU oracle for sparse MLA decode attention.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline / reference leg may load, link or call this code. It shares no
 * source, header, table or helper with the CUDA path, and the CUDA path never
 * calls it.
 *
 * What it computes follows two pages:
 *
 *  [DSv4] vllm.models.deepseek_v41.nvidia.specialized_decode.attention.
 *         sparse_mla_cute -- module docstring, "What this module computes":
 *         per token t and head h, over the active columns c (c < lens[t] and
 *         indices[t, c] >= 0), scores s_c = bmm1_scale * q[t,h] . kv[c],
 *         p_c = exp(s_c - m) with m the maximum of the scores and the sink,
 *         out = bmm2_scale * sum_c p_c kv[c] / (sum_c p_c + exp(sink_h - m));
 *         columns below the sliding-window width read the first pool, the rest
 *         the second; a token with no active column gets zeros.
 *
 *  [K3]   vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.dsa.
 *         attn_sparse -- module docstring (the per-chunk datapath and the
 *         "Precision" paragraph) and SparseDcpDecode.merge: FP32 logits, a
 *         base-2 online softmax per chunk of keys, P = exp2(s*scale_log2 - max
 *         + log2 448) rounded to E4M3 (RN, satfinite) against the running max
 *         of the split, FP32 sums of the unquantised P, FP32 accumulation of
 *         E4M3(P) x E4M3(V), the splits merged with weights exp2(max_c - max),
 *         one BF16 rounding of out = sum * k_scale / total, and
 *         LSE = max + log2(total / 448).  Count-0 rows: zeros and LSE -inf.
 *
 * Two modes:
 *   smla_oracle_fp64     the plain definition [DSv4], every step in double.
 *   smla_oracle_emulate  the [K3] datapath replayed step by step on a given
 *                        partition (splits, keys per chunk), with FP32
 *                        roundings where the datapath has them. Flags switch
 *                        the E4M3 rounding of P and the FP32 roundings off, so
 *                        that the online/merge algebra can be checked against
 *                        the plain definition.
 *
 * Readings where the pages are silent:
 *   - logits use bmm1_scale only; the output multiplier is bmm2_scale*k_scale;
 *   - the LSE is base 2 and includes the sink term of the denominator;
 *   - sinks are in score units (already scaled), base 2 = sink * log2(e);
 *   - lens is clamped to [0, width];
 *   - an index outside [0, pool rows) is treated as a hole;
 *   - a 576-byte row feeds QK with all 576 bytes and PV with its first 512.
 *
 * Numbers: E4M3 is OCP "E4M3FN" (bias 7, no infinities, S.1111.111 = NaN,
 * largest finite 448). BF16 is the upper half of binary32, rounded to
 * nearest-even. Built with -ffp-contract=off so that every float operation
 * rounds once, on x86-64 and aarch64 alike.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "smla_oracle.h"

#define LATENT 512

/* ---------------------------------------------------------------- numbers */

/* OCP FP8 E4M3FN byte -> exact real value. */
double smla_oracle_e4m3_to_double(uint8_t byte) {
    int sign = byte >> 7;
    int exponent = (byte >> 3) & 0xF;
    int mantissa = byte & 0x7;
    double magnitude;
    if (exponent == 0xF && mantissa == 0x7) return NAN;
    if (exponent == 0)
        magnitude = ldexp((double)mantissa, -9); /* subnormal: m/8 * 2^-6 */
    else
        magnitude = ldexp(8.0 + mantissa, exponent - 7 - 3); /* (1+m/8) 2^(e-7) */
    return sign ? -magnitude : magnitude;
}

/* float -> E4M3FN, round to nearest even, saturating to +-448; NaN -> 0x7F. */
uint8_t smla_oracle_e4m3_from_float(float value) {
    double x = (double)value;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isnan(x)) return 0x7F;
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal */
        double q = nearbyint(ldexp(a, 9)); /* exact scaling, RN-even */
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;               /* a in [2^e, 2^(e+1)) */
    double q = nearbyint(ldexp(a, 3 - e)); /* in [8, 16] */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    int biased = e + 7;
    if (biased > 15 || (biased == 15 && q - 8.0 > 6.0)) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (biased << 3) | (int)(q - 8.0));
}

/* float -> BF16 bits, round to nearest even (NaN kept quiet). */
uint16_t smla_oracle_bf16_from_float(float value) {
    uint32_t bits;
    memcpy(&bits, &value, 4);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu)) return 0x7FC0;
    uint32_t rounding = 0x7FFFu + ((bits >> 16) & 1u);
    return (uint16_t)((bits + rounding) >> 16);
}

float smla_oracle_bf16_to_float(uint16_t bits) {
    uint32_t wide = (uint32_t)bits << 16;
    float value;
    memcpy(&value, &wide, 4);
    return value;
}

/* ------------------------------------------------------------ the columns */

static int clamp_count(const smla_oracle_problem* p, int t) {
    int n = p->lens[t];
    if (n < 0) n = 0;
    if (n > p->width) n = p->width;
    return n;
}

/* Row of column c of token t, or NULL for an inactive column ([DSv4]: active
 * iff c < lens[t] and indices[t,c] >= 0; the first pool_split columns read
 * pool 0, the others pool 1). The caller has already applied c < count. */
static const uint8_t* column_row(const smla_oracle_problem* p, int t, int c) {
    int32_t index = p->indices[(int64_t)t * p->idx_stride_token + c];
    int pool = (p->num_pools == 2 && c >= p->pool_split) ? 1 : 0;
    if (index < 0 || (int64_t)index >= p->pool_rows[pool]) return NULL;
    return p->pool[pool] + (int64_t)index * p->head_dim;
}

static const uint8_t* query_row(const smla_oracle_problem* p, int t, int h) {
    return p->q + (int64_t)t * p->q_stride_token + (int64_t)h * p->q_stride_head;
}

/* q . kv over all head_dim bytes, exact: every E4M3 x E4M3 product and their
 * sum over <= 576 terms are exact in double (products span 2^-18 .. 2^17.6). */
static double exact_dot(const uint8_t* q, const uint8_t* kv, int dim) {
    double sum = 0.0;
    for (int d = 0; d < dim; ++d)
        sum += smla_oracle_e4m3_to_double(q[d]) * smla_oracle_e4m3_to_double(kv[d]);
    return sum;
}

/* ------------------------------------------------------- fp64 definition */

int smla_oracle_fp64(const smla_oracle_problem* p, int t, int h, double* out, double* lse2) {
    const double log2e = 1.4426950408889634074;
    int count = clamp_count(p, t);
    const uint8_t* q = query_row(p, t, h);

    /* pass 1: scores of the active columns and their maximum (with the sink) */
    double* score = (double*)malloc(sizeof(double) * (count > 0 ? count : 1));
    int active = 0;
    double m = -INFINITY;
    for (int c = 0; c < count; ++c) {
        const uint8_t* row = column_row(p, t, c);
        if (!row) {
            score[c] = -INFINITY;
            continue;
        }
        score[c] = p->bmm1_scale * exact_dot(q, row, p->head_dim);
        if (score[c] > m) m = score[c];
        ++active;
    }
    for (int j = 0; j < LATENT; ++j) out[j] = 0.0;
    if (active == 0) { /* no active column: zeros, LSE -inf (sink ignored) */
        *lse2 = -INFINITY;
        free(score);
        return 0;
    }
    double sink = p->sinks ? (double)p->sinks[h] : 0.0;
    if (p->sinks && sink > m) m = sink;

    /* pass 2: weights, denominator and the weighted sum of the V rows */
    double den = p->sinks ? exp(sink - m) : 0.0;
    for (int c = 0; c < count; ++c) {
        if (score[c] == -INFINITY) continue;
        const uint8_t* row = column_row(p, t, c);
        double w = exp(score[c] - m);
        den += w;
        for (int j = 0; j < LATENT; ++j) out[j] += w * smla_oracle_e4m3_to_double(row[j]);
    }
    double scale = p->bmm2_scale * p->k_scale / den;
    for (int j = 0; j < LATENT; ++j) out[j] *= scale;
    *lse2 = (m + log(den)) * log2e;
    free(score);
    return 0;
}

/* ------------------------------------------------------ emulating datapath */

/* One rounding to binary32, or none when the caller asked for exact math. */
static double r32(double x, int exact) { return exact ? x : (double)(float)x; }

/* The E4M3 code of P is a rounding decision that the datapath takes on an
 * FP32 value whose last bits the pages leave open: the logits come from FP8
 * products summed in FP32 in an order they do not fix, and exp2 is a fast
 * approximation (Kimi K3.1 attn_sparse page, "Precision"). A P within a
 * relative 2^-16 of a rounding midpoint may therefore take either neighbouring
 * code. The emulation keeps the round-to-nearest code and reports, per output
 * element, the most that taking the other code at every such P can move it. */
#define TIE_WINDOW (1.0 / 65536.0)

static double code_value(double x) {
    return smla_oracle_e4m3_to_double(smla_oracle_e4m3_from_float((float)x));
}

int smla_oracle_emulate(const smla_oracle_problem* p, int t, int h, int splits, int chunk,
                        int flags, double* out_value, uint16_t* out_bf16, double* lse2_out,
                        double* tie_out) {
    const int exact = (flags & SMLA_ORACLE_EXACT) != 0;
    const int keep_p = (flags & SMLA_ORACLE_NO_P_ROUNDING) != 0;
    /* P moved to either edge of the tie window before its rounding (the two
     * codes a tie-ambiguous P may take; the sums keep the unmoved P) */
    const double nudge = (flags & SMLA_ORACLE_P_UP) ? 1.0 + TIE_WINDOW
                       : (flags & SMLA_ORACLE_P_DOWN) ? 1.0 - TIE_WINDOW : 1.0;
    const double log2_448 = log2(448.0);
    if (splits < 1 || chunk < 1) return -1;

    const double log2e = 1.4426950408889634074;
    const double scale_log2 = r32(p->bmm1_scale * log2e, exact);
    const double out_scale = r32(p->bmm2_scale * p->k_scale, exact);
    const double anchor = r32(log2_448, exact);

    int count = clamp_count(p, t);
    const uint8_t* q = query_row(p, t, h);

    /* The partition the GPU replays: columns [0, count) in chunks of `chunk`,
     * consecutive chunks dealt to the splits, ceil(chunks / splits) each. */
    int chunks = (count + chunk - 1) / chunk;
    int per_split = (chunks + splits - 1) / splits;

    double* m_split = (double*)malloc(sizeof(double) * splits);
    double* l_split = (double*)malloc(sizeof(double) * splits);
    double* acc = (double*)calloc((size_t)splits * LATENT, sizeof(double));
    double* tie_acc = (double*)calloc((size_t)splits * LATENT, sizeof(double));
    double* s2 = (double*)malloc(sizeof(double) * chunk);
    double* prob = (double*)malloc(sizeof(double) * chunk);
    double* spread = (double*)malloc(sizeof(double) * chunk);

    for (int s = 0; s < splits; ++s) {
        double m_run = -INFINITY, l_run = 0.0;
        double* a = acc + (size_t)s * LATENT;
        double* ta = tie_acc + (size_t)s * LATENT;
        int c_first = s * per_split;
        int c_last = c_first + per_split < chunks ? c_first + per_split : chunks;
        for (int ck = c_first; ck < c_last; ++ck) {
            int base = ck * chunk;
            int n = count - base < chunk ? count - base : chunk;
            /* FP32 logits in log2 units; masked columns score -inf */
            double chunk_max = -INFINITY;
            for (int i = 0; i < n; ++i) {
                const uint8_t* row = column_row(p, t, base + i);
                if (!row) {
                    s2[i] = -INFINITY;
                    continue;
                }
                double logit = r32(exact_dot(q, row, p->head_dim), exact);
                s2[i] = r32(logit * scale_log2, exact);
                if (s2[i] > chunk_max) chunk_max = s2[i];
            }
            /* running max and the rescale factor of what was accumulated */
            double m_new = chunk_max > m_run ? chunk_max : m_run;
            double alpha = 1.0;
            if (m_run != -INFINITY) alpha = r32(exp2(m_run - m_new), exact);
            /* P against the running max, scaled so the maximum maps to 448 */
            double bias = r32(m_new - anchor, exact);
            double chunk_sum = 0.0;
            for (int i = 0; i < n; ++i) {
                double x = 0.0;
                if (s2[i] != -INFINITY) x = r32(exp2(r32(s2[i] - bias, exact)), exact);
                chunk_sum = r32(chunk_sum + x, exact); /* sums of the unquantised P */
                prob[i] = keep_p ? x : code_value(x * nudge);
                /* the two codes P may take within the tie window */
                spread[i] = keep_p ? 0.0 : code_value(x * (1.0 + TIE_WINDOW)) - code_value(x * (1.0 - TIE_WINDOW));
            }
            l_run = r32(r32(l_run * alpha, exact) + chunk_sum, exact);
            m_run = m_new;
            /* PV: E4M3(P) x E4M3(V) products are exact; one FP32 rounding */
            for (int j = 0; j < LATENT; ++j) {
                double pv = 0.0;
                for (int i = 0; i < n; ++i) {
                    if (prob[i] == 0.0) continue;
                    const uint8_t* row = column_row(p, t, base + i);
                    pv += prob[i] * smla_oracle_e4m3_to_double(row[j]);
                }
                a[j] = r32(r32(a[j] * alpha, exact) + pv, exact);
                double tie = 0.0;
                for (int i = 0; i < n; ++i) {
                    if (spread[i] == 0.0) continue;
                    tie += spread[i] * fabs(smla_oracle_e4m3_to_double(column_row(p, t, base + i)[j]));
                }
                ta[j] = ta[j] * alpha + tie;
            }
        }
        m_split[s] = m_run;
        l_split[s] = l_run;
    }

    /* merge of the splits (and the sink) */
    double top = -INFINITY;
    for (int s = 0; s < splits; ++s)
        if (m_split[s] > top) top = m_split[s];
    int empty = (top == -INFINITY);
    if (!empty && p->sinks) {
        double sink2 = r32((double)p->sinks[h] * log2e, exact);
        if (sink2 > top) top = sink2;
    }
    double total = 0.0;
    double* merged = (double*)calloc(LATENT, sizeof(double));
    double* tie_merged = (double*)calloc(LATENT, sizeof(double));
    if (!empty) {
        for (int s = 0; s < splits; ++s) {
            if (m_split[s] == -INFINITY) continue;
            double w = r32(exp2(m_split[s] - top), exact);
            total = r32(total + r32(w * l_split[s], exact), exact);
            for (int j = 0; j < LATENT; ++j) {
                merged[j] = r32(merged[j] + r32(w * acc[(size_t)s * LATENT + j], exact), exact);
                tie_merged[j] += w * tie_acc[(size_t)s * LATENT + j];
            }
        }
        if (p->sinks) {
            double sink2 = r32((double)p->sinks[h] * log2e, exact);
            double w = r32(448.0 * r32(exp2(sink2 - top), exact), exact);
            total = r32(total + w, exact);
        }
    }
    if (empty || !(total > 0.0)) {
        for (int j = 0; j < LATENT; ++j) {
            if (out_value) out_value[j] = 0.0;
            if (out_bf16) out_bf16[j] = 0;
            if (tie_out) tie_out[j] = 0.0;
        }
        if (lse2_out) *lse2_out = -INFINITY;
    } else {
        /* out = merged * (bmm2_scale * k_scale) / total, one BF16 rounding */
        double inverse = r32(out_scale / total, exact);
        for (int j = 0; j < LATENT; ++j) {
            double value = exact ? merged[j] * out_scale / total : r32(merged[j] * inverse, 0);
            if (out_value) out_value[j] = value;
            if (out_bf16) out_bf16[j] = smla_oracle_bf16_from_float((float)value);
            if (tie_out) tie_out[j] = tie_merged[j] * fabs(out_scale) / total;
        }
        if (lse2_out) *lse2_out = top - log2_448 + log2(total);
    }
    free(tie_merged);
    free(merged);
    free(spread);
    free(prob);
    free(s2);
    free(tie_acc);
    free(acc);
    free(l_split);
    free(m_split);
    return 0;
}

/* ----------------------------------------------- LSE merge of partial sets */
/*
 * [DCP]  vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.dcp --
 *        DcpValue (class docstring and merge): the owner weights each source
 *        s of a (token, head) by exp2(lse_s - max) / sum over the sources, in
 *        FP32; a source whose LSE is NaN, -inf or +inf (or a token of count
 *        0) is empty and weighs nothing; the weighted sum of the sources' BF16
 *        rows is taken in FP32 and rounded to BF16 once. A token with no
 *        source left gets zeros.
 * Readings: an LSE that is not finite marks an empty source; the merged LSE,
 * which the page does not output, is max + log2(sum of weights) (base 2),
 * -inf for an empty result.
 */

/* The merge in double: `sources` rows of 512 values with base-2 LSEs. */
int smla_oracle_merge_f64(int sources, const double* rows, const double* lses, double* out, double* lse2) {
    double top = -INFINITY;
    for (int s = 0; s < sources; ++s)
        if (isfinite(lses[s]) && lses[s] > top) top = lses[s];
    double total = 0.0;
    for (int s = 0; s < sources; ++s)
        if (isfinite(lses[s])) total += exp2(lses[s] - top);
    for (int j = 0; j < LATENT; ++j) out[j] = 0.0;
    if (!(total > 0.0)) {
        *lse2 = -INFINITY;
        return 0;
    }
    for (int s = 0; s < sources; ++s) {
        if (!isfinite(lses[s])) continue;
        double weight = exp2(lses[s] - top) / total;
        for (int j = 0; j < LATENT; ++j) out[j] += weight * rows[(size_t)s * LATENT + j];
    }
    *lse2 = top + log2(total);
    return 0;
}

/* The merge of (t, h) from BF16 rows: out_value (double, before rounding),
 * out_bf16 (bits) and the merged LSE; any may be NULL. */
int smla_oracle_merge(const smla_oracle_merge_problem* m, int t, int h, double* out_value,
                      uint16_t* out_bf16, double* lse2_out) {
    double* rows = (double*)malloc(sizeof(double) * (size_t)m->sources * LATENT);
    double* lses = (double*)malloc(sizeof(double) * (size_t)(m->sources > 0 ? m->sources : 1));
    double out[LATENT];
    double lse2 = -INFINITY;
    if (!rows || !lses) {
        free(rows);
        free(lses);
        return -1;
    }
    int live = !(m->lens && m->lens[t] <= 0);
    for (int s = 0; s < m->sources; ++s) {
        const uint16_t* part = m->parts + s * m->part_stride_source + (int64_t)t * m->part_stride_token +
                               (int64_t)h * m->part_stride_head;
        for (int j = 0; j < LATENT; ++j) rows[(size_t)s * LATENT + j] = smla_oracle_bf16_to_float(part[j]);
        lses[s] = live ? (double)m->lses[s * m->lse_stride_source + (int64_t)t * m->lse_stride_token + h]
                       : -INFINITY;
    }
    smla_oracle_merge_f64(m->sources, rows, lses, out, &lse2);
    for (int j = 0; j < LATENT; ++j) {
        if (out_value) out_value[j] = out[j];
        if (out_bf16) out_bf16[j] = smla_oracle_bf16_from_float((float)out[j]);
    }
    if (lse2_out) *lse2_out = lse2;
    free(rows);
    free(lses);
    return 0;
}

int smla_oracle_merge_pairs(const smla_oracle_merge_problem* m, const int32_t* tokens,
                            const int32_t* heads, int n, double* out_value, uint16_t* out_bf16,
                            double* lse2, int threads) {
    int bad = 0;
#ifdef _OPENMP
    const int team = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(team) schedule(dynamic, 4) reduction(| : bad)
#endif
    for (int i = 0; i < n; ++i)
        bad |= smla_oracle_merge(m, tokens[i], heads[i], out_value ? out_value + (size_t)i * LATENT : NULL,
                                 out_bf16 ? out_bf16 + (size_t)i * LATENT : NULL, lse2 ? lse2 + i : NULL) != 0;
    (void)threads;
    return bad ? -1 : 0;
}

/* ------------------------------------------ MXFP4 quantisation of the query */
/*
 * [MXFP4] vllm.models.kimi_k3.nvidia.ops.dsa_indexer_mxfp4 -- mxfp4_q_quant,
 *         _mxfp4_q_quant_kernel and _mxfp4_quant: each head's 128 query
 *         values (taken as FP32) form 4 blocks of 32; a block's UE8M0 scale is
 *         2^e with e = ceil(log2(max(amax, 6 * 2^-126) / 6)) clamped to
 *         [-127, 127] and stored as e + 127; the values divided by 2^e are
 *         rounded to FP4 E2M1 and packed two per byte, the even element in
 *         the low nibble; a head's four scale bytes form one int32 (block b
 *         in byte b); the head weights are multiplied by weight_scale in FP32;
 *         heads [H, P) of the padded outputs are zero.
 * Readings: the ceiling of log2 is taken exactly on the FP32 quotient (a power
 * of two gives its own exponent, anything above it the next one); E2M1 is the
 * OCP MX element format (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), rounded to
 * nearest with ties to the even code, saturating at 6, keeping the sign of
 * zero.
 */

/* FP32 -> E2M1 code (sign in bit 3), round to nearest even, saturating. */
uint8_t smla_oracle_e2m1_from_float(float value) {
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint8_t sign = signbit(value) ? 8u : 0u;
    float a = fabsf(value);
    if (a >= 6.0f) return (uint8_t)(sign | 7u);
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        float d_best = fabsf(a - grid[best]), d = fabsf(a - grid[c]);
        if (d < d_best || (d == d_best && (c & 1) == 0)) best = c;
    }
    return (uint8_t)(sign | (uint8_t)best);
}

double smla_oracle_e2m1_to_double(uint8_t code) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = grid[code & 7u];
    return (code & 8u) ? -v : v;
}

/* e = ceil(log2(q)) for a positive finite float q, exactly. */
static int ceil_log2_exact(float q) {
    int e;
    double m = frexp((double)q, &e); /* q = m * 2^e, m in [0.5, 1) */
    return m == 0.5 ? e - 1 : e;
}

/* One token: q [heads][128] FP32 values, weights [heads]; outputs for the
 * padded heads: packed [padded][64] bytes, scale [padded] int32, w_out [padded]. */
int smla_oracle_mxfp4_q_quant(int heads, int padded, const float* q, const float* weights, float weight_scale,
                              uint8_t* packed, int32_t* scale, float* w_out) {
    const int D = 128, B = 32;
    for (int h = 0; h < padded; ++h) {
        if (h >= heads) {
            memset(packed + (size_t)h * (D / 2), 0, D / 2);
            scale[h] = 0;
            w_out[h] = 0.0f;
            continue;
        }
        const float* x = q + (size_t)h * D;
        uint32_t bytes = 0;
        for (int b = 0; b < D / B; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < B; ++i) amax = fmaxf(amax, fabsf(x[b * B + i]));
            float floor_amax = 6.0f * ldexpf(1.0f, -126);
            float quotient = fmaxf(amax, floor_amax) / 6.0f;
            int e = ceil_log2_exact(quotient);
            if (e < -127) e = -127;
            if (e > 127) e = 127;
            bytes |= (uint32_t)(uint8_t)(e + 127) << (8 * b);
            for (int i = 0; i < B; i += 2) {
                float lo = (float)ldexp((double)x[b * B + i], -e);     /* exact: a power-of-two scaling */
                float hi = (float)ldexp((double)x[b * B + i + 1], -e);
                packed[(size_t)h * (D / 2) + (b * B + i) / 2] =
                    (uint8_t)(smla_oracle_e2m1_from_float(lo) | (smla_oracle_e2m1_from_float(hi) << 4));
            }
        }
        memcpy(&scale[h], &bytes, 4);
        w_out[h] = weights[h] * weight_scale;
    }
    return 0;
}

/* ------------------------------- value projection and gate after the merge */
/*
 * [DCP]  DcpValue (class docstring and merge, the lines after the merged
 *        rows): out[t, h*128 + v] = BF16(BF16(sum_j latent[t, h, j] *
 *        W[h, j, v]) * sigmoid(gate[t, h*128 + v])), the sum over the 512
 *        latents (BF16 operands, FP32 accumulation on the page), sigmoid(x) =
 *        1 / (1 + e^-x); rows of a token whose count is <= 0 are zero.
 * Readings: the count is per token (the page's per-request totals with one
 * token per request); the sum is taken exactly (double) before its BF16
 * rounding.
 */
int smla_oracle_value_gate(int tokens, int heads, const uint16_t* latent, const uint16_t* w_uv,
                           const uint16_t* gate, const int32_t* lens, double* out_value, uint16_t* out_bf16) {
    const int J = LATENT, V = 128;
    for (int t = 0; t < tokens; ++t)
        for (int h = 0; h < heads; ++h)
            for (int v = 0; v < V; ++v) {
                size_t o = ((size_t)t * heads + h) * V + v;
                double value = 0.0;
                if (!(lens && lens[t] <= 0)) {
                    double acc = 0.0;
                    for (int j = 0; j < J; ++j)
                        acc += (double)smla_oracle_bf16_to_float(latent[((size_t)t * heads + h) * J + j]) *
                               (double)smla_oracle_bf16_to_float(w_uv[((size_t)h * J + j) * V + v]);
                    double rounded = smla_oracle_bf16_to_float(smla_oracle_bf16_from_float((float)acc));
                    double g = smla_oracle_bf16_to_float(gate[o]);
                    value = rounded * (1.0 / (1.0 + exp(-g)));
                }
                if (out_value) out_value[o] = value;
                if (out_bf16) out_bf16[o] = smla_oracle_bf16_from_float((float)value);
            }
    return 0;
}

/* ------------------------------------------------------------ batch drivers */

/* FP64 definition over every (token, head); OpenMP over the pairs. */
int smla_oracle_fp64_all(const smla_oracle_problem* p, double* out, double* lse2, int threads) {
    int pairs = p->tokens * p->heads;
#ifdef _OPENMP
    const int team = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(team) schedule(dynamic, 1)
#endif
    for (int i = 0; i < pairs; ++i)
        smla_oracle_fp64(p, i / p->heads, i % p->heads, out + (size_t)i * LATENT, lse2 + i);
    (void)threads;
    return 0;
}

/* FP64 definition over a list of (token, head) pairs. */
int smla_oracle_fp64_pairs(const smla_oracle_problem* p, const int32_t* tokens,
                           const int32_t* heads, int n, double* out, double* lse2, int threads) {
#ifdef _OPENMP
    const int team = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(team) schedule(dynamic, 1)
#endif
    for (int i = 0; i < n; ++i)
        smla_oracle_fp64(p, tokens[i], heads[i], out + (size_t)i * LATENT, lse2 + i);
    (void)threads;
    return 0;
}

/* Emulating datapath over a list of (token, head) pairs. */
int smla_oracle_emulate_pairs(const smla_oracle_problem* p, const int32_t* tokens,
                              const int32_t* heads, int n, int splits, int chunk, int flags,
                              double* out_value, uint16_t* out_bf16, double* lse2, double* tie,
                              int threads) {
    int bad = 0;
#ifdef _OPENMP
    const int team = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(team) schedule(dynamic, 1) reduction(| : bad)
#endif
    for (int i = 0; i < n; ++i)
        bad |= smla_oracle_emulate(p, tokens[i], heads[i], splits, chunk, flags,
                                   out_value ? out_value + (size_t)i * LATENT : NULL,
                                   out_bf16 ? out_bf16 + (size_t)i * LATENT : NULL,
                                   lse2 ? lse2 + i : NULL,
                                   tie ? tie + (size_t)i * LATENT : NULL) != 0;
    (void)threads;
    return bad ? -1 : 0;
}

int smla_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
