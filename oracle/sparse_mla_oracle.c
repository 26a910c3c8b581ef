/*
 * Oracle for the token-sparse MLA attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg load it.  It shares no code, header, table or constant with the CUDA
 * library; both sides only read the same seeded inputs.
 *
 * What it computes (the plain definition, in fp64, two passes, no blocking):
 * for every query token t and head h, with the per-token list idx[t, 0:topk]
 * of int32 slots into a latent KV cache whose rows have 576 dims (512 latent +
 * 64 rope, one KV head):
 *
 *   valid(j)  <=>  0 <= idx[t,j] < num_slots          (-1 marks an invalid entry)
 *   s_j       =   scale * sum_{d<576} q[t,h,d] * kv[idx[t,j], d]
 *   m         =   max_{valid j} s_j
 *   l         =   sum_{valid j} exp(s_j - m)
 *   O[t,h,d]  =   sum_{valid j} exp(s_j - m) * kv[idx[t,j], d] / l,  d < 512
 *   LSE[t,h]  =   m + ln(l)          (natural log of the sum of exp of SCALED logits)
 *   no valid j:   O = 0, LSE = -inf
 *
 * Each list entry is its own softmax term, so a slot listed k times weighs k.
 *
 * Sources (page title, section):
 *  - vLLM PR #60220 "FlashMLA sparse: stage fp8 mixed-batch q/out in the
 *    workspace", Claims: q is T x heads x 576 bf16 and the output is
 *    T x heads x 512 bf16; Details: the kernel also returns lse (T x 64 x 4 B).
 *  - PR #55738 report, 功能与动机 (motivation): prefill tokens go through a
 *    "per-token top-k MQA kernel" -- one KV head shared by all query heads,
 *    each token attending to its own top-k rows.
 *  - PR #55738 report, `_is_masked_mha_available` geometry table:
 *    kv_lora_rank 512 and qk_rope_head_dim 64, hence 576-dim keys whose first
 *    512 dims are the values.
 *  - vLLM PR #54951 "Shard long-context indexer prefill rows", Summary and
 *    Additional checks: the index lists are fixed-width int32 and only the SET
 *    of selected rows matters (top-k order is not deterministic).
 *  - vLLM PR #60220, Overview: the sparse kernel also reads a quantised
 *    latent cache (fp8_ds_mla).  The pages do not give its byte layout; this
 *    oracle reads [512 x e4m3 | 4 x fp32 scale per 128 dims | 64 x bf16 rope]
 *    (656 bytes) and computes latent[d] = e4m3(byte[d]) * scale[d / 128]
 *    exactly in fp64.
 *
 * bf16 -> fp64 and e4m3 -> fp64 are exact; the e4m3 values come from the
 * format's definition (OCP 8-bit floating point, E4M3: bias 7, 3 mantissa bits,
 * exponent field 0 = subnormal, S.1111.111 = NaN, no infinities, max 448).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DQK 576
#define ORACLE_DV 512
#define ORACLE_FP8_ROW 656

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_FP8 = 1 };

static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 value of one byte, from the format definition. */
double oracle_e4m3_value(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);      /* subnormal: m/8 * 2^(1-bias) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: (1 + m/8) * 2^(e-bias) */
    return sign ? -v : v;
}

void oracle_e4m3_table(double *out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e4m3_value((uint8_t)c);
}

double oracle_bf16_value(uint16_t bits) { return bf16_bits_to_double(bits); }

/* Decode one cache row to 576 fp64 values. */
void oracle_decode_row(const void *kv, int kv_format, int64_t slot, double *row) {
    if (kv_format == ORACLE_KV_BF16) {
        const uint16_t *r = (const uint16_t *)kv + slot * (int64_t)ORACLE_DQK;
        for (int d = 0; d < ORACLE_DQK; ++d) row[d] = bf16_bits_to_double(r[d]);
    } else {
        const uint8_t *r = (const uint8_t *)kv + slot * (int64_t)ORACLE_FP8_ROW;
        float tile_scale[4];
        memcpy(tile_scale, r + 512, sizeof tile_scale);
        for (int d = 0; d < 512; ++d)
            row[d] = oracle_e4m3_value(r[d]) * (double)tile_scale[d / 128];
        for (int d = 0; d < 64; ++d) {
            uint16_t b;
            memcpy(&b, r + 528 + 2 * d, sizeof b);
            row[512 + d] = bf16_bits_to_double(b);
        }
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * q        [T, h, 576] bf16 bit patterns
 * kv       [num_slots, 576] bf16, or [num_slots] rows of 656 bytes (fp8)
 * idx      [T, topk] int32
 * tokens   optional list of n_tokens token ids to evaluate (NULL: all T, n_tokens = T)
 * out      [n_tokens, h, 512] fp64;  lse [n_tokens, h] fp64
 * returns 0 on success, 1 on a bad argument, 2 if memory ran out
 */
int oracle_sparse_mla_fwd(const uint16_t *q, const void *kv, int kv_format,
                          const int32_t *idx, int64_t T, int h, int topk,
                          int64_t num_slots, double scale, const int64_t *tokens,
                          int64_t n_tokens, double *out, double *lse, int nthreads) {
    if (T < 0 || h <= 0 || topk <= 0 || num_slots <= 0 || n_tokens < 0) return 1;
    if (kv_format != ORACLE_KV_BF16 && kv_format != ORACLE_KV_FP8) return 1;
    if (n_tokens > 0 && (!q || !kv || !idx || !out || !lse)) return 1;
    if (!tokens && n_tokens != T) return 1;
    if (tokens)
        for (int64_t i = 0; i < n_tokens; ++i)
            if (tokens[i] < 0 || tokens[i] >= T) return 1;

    int failed = 0;
    int64_t pairs = n_tokens * (int64_t)h;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)topk);
        double *row = (double *)malloc(sizeof(double) * ORACLE_DQK);
        double qv[ORACLE_DQK], acc[ORACLE_DV];
        if (!s || !row) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t p = 0; p < pairs; ++p) {
            if (!s || !row) continue;
            int64_t i = p / h;
            int hh = (int)(p % h);
            int64_t t = tokens ? tokens[i] : i;
            const uint16_t *qr = q + (t * h + hh) * (int64_t)ORACLE_DQK;
            const int32_t *list = idx + t * (int64_t)topk;
            double *o = out + (i * h + hh) * (int64_t)ORACLE_DV;

            for (int d = 0; d < ORACLE_DQK; ++d) qv[d] = bf16_bits_to_double(qr[d]);

            /* pass 1: scaled logits of the valid entries and their maximum */
            double m = -INFINITY;
            int n_valid = 0;
            for (int j = 0; j < topk; ++j) {
                int64_t slot = list[j];
                if (slot < 0 || slot >= num_slots) continue;
                oracle_decode_row(kv, kv_format, slot, row);
                double dot = 0.0;
                for (int d = 0; d < ORACLE_DQK; ++d) dot += qv[d] * row[d];
                s[j] = scale * dot;
                if (s[j] > m) m = s[j];
                ++n_valid;
            }
            if (n_valid == 0) {
                for (int d = 0; d < ORACLE_DV; ++d) o[d] = 0.0;
                lse[i * h + hh] = -INFINITY;
                continue;
            }

            /* pass 2: softmax weights and the weighted sum of the value rows */
            double l = 0.0;
            for (int d = 0; d < ORACLE_DV; ++d) acc[d] = 0.0;
            for (int j = 0; j < topk; ++j) {
                int64_t slot = list[j];
                if (slot < 0 || slot >= num_slots) continue;
                double w = exp(s[j] - m);
                l += w;
                oracle_decode_row(kv, kv_format, slot, row);
                for (int d = 0; d < ORACLE_DV; ++d) acc[d] += w * row[d];
            }
            for (int d = 0; d < ORACLE_DV; ++d) o[d] = acc[d] / l;
            lse[i * h + hh] = m + log(l);
        }
        free(s);
        free(row);
    }
    return failed ? 2 : 0;
}

/*
 * Merge of the partial results of one list split into parts: the "DCP merge"
 * that consumes out and lse (vLLM PR #60220, Details: the output "is consumed
 * by the v_up projection or the DCP merge"; vLLM PR #64510, Details: heads
 * gathered by DCP).  The pages do not write the merge.  Read as the exact
 * combination of softmax results over disjoint parts of one list, each part p
 * given as its normalised O_p and natural-log LSE_p (what the forward returns):
 *
 *   M        = max_p LSE_p
 *   LSE      = M + ln sum_p exp(LSE_p - M)
 *   O[d]     = sum_p exp(LSE_p - LSE) * O_p[d]
 *   a part with LSE_p = -inf is empty and weighs 0; no non-empty part: O = 0,
 *   LSE = -inf.
 *
 * o_parts   [n][rows][512], fp64 (o_bf16 = 0) or bf16 bit patterns (o_bf16 = 1)
 * lse_parts [n][rows] fp64
 * out       [rows][512] fp64;  lse [rows] fp64
 * Returns 0, or 1 for n < 1 or rows < 0.
 */
int oracle_merge(const void *o_parts, int o_bf16, const double *lse_parts, int n, int64_t rows,
                 double *out, double *lse) {
    if (n < 1 || rows < 0) return 1;
    const double *of = (const double *)o_parts;
    const uint16_t *ob = (const uint16_t *)o_parts;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int p = 0; p < n; ++p)
            if (lse_parts[p * rows + r] > m) m = lse_parts[p * rows + r];
        double *o = out + r * ORACLE_DV;
        if (m == -INFINITY) {
            for (int d = 0; d < ORACLE_DV; ++d) o[d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int p = 0; p < n; ++p) {
            double l = lse_parts[p * rows + r];
            if (l != -INFINITY) sum += exp(l - m);
        }
        double total = m + log(sum);
        for (int d = 0; d < ORACLE_DV; ++d) o[d] = 0.0;
        for (int p = 0; p < n; ++p) {
            double l = lse_parts[p * rows + r];
            if (l == -INFINITY) continue;
            double w = exp(l - total);
            int64_t base = (p * rows + r) * ORACLE_DV;
            for (int d = 0; d < ORACLE_DV; ++d)
                o[d] += w * (o_bf16 ? bf16_bits_to_double(ob[base + d]) : of[base + d]);
        }
        lse[r] = total;
    }
    return 0;
}

/*
 * The v_up projection of the attention output (vLLM PR #60220, Details: the output "is
 * consumed by the v_up projection or the DCP merge").  Shapes from the PR #55738 report,
 * `_is_masked_mha_available` geometry table: kv_lora_rank 512 with v_head_dim 128
 * (DeepSeek-V3.2) or 256 (GLM-5).  Per head h the 512-dim latent output goes through that
 * head's value up-projection (512 -> v):
 *
 *   y[t, h, n] = sum_{k < 512} O[t, h, k] * W[h, n, k]        (n < v)
 *
 * O [T, h, 512] bf16, W [h, v, 512] bf16 (row n of head h: the 512 weights of output n; the
 * pages give no layout, this one keeps each output's weights contiguous), y [T, h, v] fp64.
 * Returns 0, or 1 for a bad size.
 */
int oracle_v_up(const uint16_t *o, const uint16_t *w, int64_t T, int h, int v, double *y) {
    if (T < 0 || h < 1 || v < 1) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int hh = 0; hh < h; ++hh) {
            const uint16_t *orow = o + (t * h + hh) * ORACLE_DV;
            for (int n = 0; n < v; ++n) {
                const uint16_t *wrow = w + ((int64_t)hh * v + n) * ORACLE_DV;
                double acc = 0.0;
                for (int k = 0; k < ORACLE_DV; ++k)
                    acc += bf16_bits_to_double(orow[k]) * bf16_bits_to_double(wrow[k]);
                y[(t * h + hh) * v + n] = acc;
            }
        }
    }
    return 0;
}

/*
 * Top-k selection of a token's index list from per-position scores: the step before the
 * sparse attention (vLLM PR #54951, Summary: the indexer's "MQA logits and top-k" produce the
 * fixed-width int32 lists; Additional checks: the top-k order is not deterministic, only the
 * set matters).  The pages do not give the indexer's scoring; this takes the scores as input.
 * Row t keeps the `topk` positions with the largest scores among its causal history
 * [0, len[t]) -- ties broken towards the lower position -- lists them in ascending position
 * order, maps position p to slot block_table[p / 64] * 64 + p % 64 (block_table may be NULL:
 * slot = p), and pads with -1 when len[t] < topk.
 * scores [T, S] fp32, len [T] int32 (0 <= len <= S), out [T, topk] int32.
 * Returns 0, or 1 for bad sizes.
 */
typedef struct {
    float score;
    int32_t pos;
} oracle_scored;

static int oracle_by_score_desc(const void *a, const void *b) {
    const oracle_scored *x = (const oracle_scored *)a, *y = (const oracle_scored *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int oracle_by_pos(const void *a, const void *b) {
    const int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

int oracle_topk(const float *scores, int64_t T, int64_t S, const int32_t *len, int topk,
                const int32_t *block_table, int32_t *out) {
    if (T < 0 || S < 0 || topk < 1) return 1;
    for (int64_t t = 0; t < T; ++t)
        if (len[t] < 0 || len[t] > S) return 1;
    int failed = 0;
#pragma omp parallel
    {
        oracle_scored *row = (oracle_scored *)malloc(sizeof(oracle_scored) * (size_t)(S > 0 ? S : 1));
        int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)topk);
        if (!row || !sel) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < T; ++t) {
            if (!row || !sel) continue;
            const int64_t n = len[t];
            for (int64_t p = 0; p < n; ++p) {
                row[p].score = scores[t * S + p];
                row[p].pos = (int32_t)p;
            }
            qsort(row, (size_t)n, sizeof(oracle_scored), oracle_by_score_desc);
            const int k = n < topk ? (int)n : topk;
            for (int i = 0; i < k; ++i) sel[i] = row[i].pos;
            qsort(sel, (size_t)k, sizeof(int32_t), oracle_by_pos);
            for (int i = 0; i < topk; ++i) {
                int32_t v = -1;
                if (i < k) v = block_table ? block_table[sel[i] / 64] * 64 + sel[i] % 64 : sel[i];
                out[t * topk + i] = v;
            }
        }
        free(row);
        free(sel);
    }
    return failed ? 2 : 0;
}

/*
 * The masked dense route for short prefill (PR #55738 report, 实现拆解 items 2 and 5 and the
 * key-files list: the top-k lists are scattered into a dense mask and a masked MHA runs over
 * the request's decompressed per-head K and V, instead of the per-token sparse kernel).  The
 * pages name the steps (a scatter kernel, a `mask_mod` attention) but give neither the mask's
 * layout nor the arithmetic.  Read as:
 *
 *   scatter:  mask[t, s] = 1  <=>  some j has idx[t, j] == s, 0 <= s < S
 *             (-1 and every other value outside [0, S) set nothing; a position listed twice
 *             sets its bit once).  Stored as bits: bit (s % 32) of word s / 32 of row t,
 *             W = ceil(S / 32) uint32 words a row, the bits past S zero.
 *   masked MHA, per token t and head h, over the positions s with mask[t, s] = 1:
 *             s_ts    = scale * sum_{d < dqk} q[t, h, d] * k[s, h, d]
 *             O[t, h] = sum_s softmax(s_t.)_s * v[s, h, 0:dv]
 *             LSE     = natural log of sum_s exp(s_ts);  no position: O = 0, LSE = -inf.
 *
 * The mask alone decides which positions attend: lists drawn over a token's causal history
 * are causal by construction.  Since the mask holds a set, this equals the sparse forward
 * over the same lists exactly when no list repeats a position.
 */
int oracle_scatter_mask(const int32_t *idx, int64_t T, int topk, int64_t S, uint32_t *mask) {
    if (T < 0 || topk < 1 || S < 1) return 1;
    const int64_t W = (S + 31) / 32;
    for (int64_t i = 0; i < T * W; ++i) mask[i] = 0u;
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < topk; ++j) {
            const int64_t s = idx[t * topk + j];
            if (s < 0 || s >= S) continue;
            mask[t * W + s / 32] |= 1u << (s % 32);
        }
    return 0;
}

/*
 * q [T, h, dqk], k [S, h, dqk], v [S, h, dv] fp64 values (the caller decodes bf16 exactly);
 * mask [T, ceil(S / 32)] bits as oracle_scatter_mask writes them;
 * out [T, h, dv] fp64;  lse [T, h] fp64.
 * Returns 0, 1 for a bad size, 2 if memory ran out.
 */
int oracle_masked_mha(const double *q, const double *k, const double *v, const uint32_t *mask,
                      int64_t T, int64_t S, int h, int dqk, int dv, double scale, double *out,
                      double *lse) {
    if (T < 0 || S < 1 || h < 1 || dqk < 1 || dv < 1) return 1;
    const int64_t W = (S + 31) / 32;
    int failed = 0;
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)S);
        double *acc = (double *)malloc(sizeof(double) * (size_t)dv);
        if (!sc || !acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < T * (int64_t)h; ++p) {
            if (!sc || !acc) continue;
            const int64_t t = p / h;
            const int hh = (int)(p % h);
            const double *qr = q + p * dqk;
            const uint32_t *mrow = mask + t * W;
            double *o = out + p * dv;

            /* pass 1: scaled logits of the masked-in positions and their maximum */
            double m = -INFINITY;
            int64_t n_in = 0;
            for (int64_t s = 0; s < S; ++s) {
                if (!((mrow[s / 32] >> (s % 32)) & 1u)) continue;
                const double *kr = k + (s * h + hh) * (int64_t)dqk;
                double dot = 0.0;
                for (int d = 0; d < dqk; ++d) dot += qr[d] * kr[d];
                sc[s] = scale * dot;
                if (sc[s] > m) m = sc[s];
                ++n_in;
            }
            if (n_in == 0) {
                for (int d = 0; d < dv; ++d) o[d] = 0.0;
                lse[p] = -INFINITY;
                continue;
            }

            /* pass 2: softmax weights and the weighted sum of the value rows */
            double l = 0.0;
            for (int d = 0; d < dv; ++d) acc[d] = 0.0;
            for (int64_t s = 0; s < S; ++s) {
                if (!((mrow[s / 32] >> (s % 32)) & 1u)) continue;
                const double *vr = v + (s * h + hh) * (int64_t)dv;
                const double w = exp(sc[s] - m);
                l += w;
                for (int d = 0; d < dv; ++d) acc[d] += w * vr[d];
            }
            for (int d = 0; d < dv; ++d) o[d] = acc[d] / l;
            lse[p] = m + log(l);
        }
        free(sc);
        free(acc);
    }
    return failed ? 2 : 0;
}
