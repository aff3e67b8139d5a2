/*
 * oracle.c -- plain CPU reference for the MoE dispatch/combine path.
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Single-threaded plain loops,
 * double accumulation, one rounding per output value.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- values */

static double f32_at(const void* base, int64_t i) {
    return (double)((const float*)base)[i];
}

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double bf16_at(const void* base, int64_t i) {
    return bf16_bits_to_double(((const uint16_t*)base)[i]);
}

static double load_elem(const void* base, int dtype, int64_t i) {
    return dtype == ORACLE_F32 ? f32_at(base, i) : bf16_at(base, i);
}

/* bf16 keeps 8 significant bits (1 implicit + 7 stored) and float's exponent
 * range.  Round |v| to a multiple of its quantum 2^(lead-7), where lead is
 * the exponent of the leading bit (clamped at -126 for subnormals); rint()
 * rounds to nearest with ties to even.  The rounded value has at most 9
 * significant bits, so it converts to float exactly (or to inf on overflow)
 * and the bf16 pattern is the float's upper half. */
static uint16_t double_to_bf16_bits(double v) {
    if (isnan(v)) return 0x7FC0u;
    if (isinf(v)) return v > 0 ? 0x7F80u : 0xFF80u;
    if (v == 0.0) return signbit(v) ? 0x8000u : 0x0000u;
    int ex;
    (void)frexp(v, &ex);
    int lead = ex - 1;
    if (lead < -126) lead = -126;
    double q = ldexp(1.0, lead - 7);
    double r = rint(v / q) * q;
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static void store_elem(void* base, int dtype, int64_t i, double v) {
    if (dtype == ORACLE_F32)
        ((float*)base)[i] = (float)v;
    else
        ((uint16_t*)base)[i] = double_to_bf16_bits(v);
}

static int dtype_ok(int dtype) { return dtype == ORACLE_F32 || dtype == ORACLE_BF16; }

int oracle_bf16_from_double(const double* v, int64_t n, uint16_t* out) {
    if (n < 0 || (n > 0 && (!v || !out))) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_bits(v[i]);
    return 0;
}

/* ---------------------------------------------------------------- top-k */

typedef struct {
    float value;
    int32_t id;
} scored_expert;

/* Larger logit first; equal logits: lower expert id first. */
static int by_score_then_id(const void* pa, const void* pb) {
    const scored_expert* a = (const scored_expert*)pa;
    const scored_expert* b = (const scored_expert*)pb;
    if (a->value > b->value) return -1;
    if (a->value < b->value) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

int oracle_topk_softmax(const float* logits, int64_t T, int E, int k,
                        int32_t* topk_idx, float* topk_w, double* topk_w_f64) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    if (T > 0 && (!logits || !topk_idx || !topk_w)) return -1;
    scored_expert* row = (scored_expert*)malloc(sizeof(scored_expert) * (size_t)E);
    double* ex = (double*)malloc(sizeof(double) * (size_t)k);
    if (!row || !ex) { free(row); free(ex); return -2; }
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            row[e].value = logits[t * E + e];
            row[e].id = e;
        }
        qsort(row, (size_t)E, sizeof(scored_expert), by_score_then_id);
        /* softmax over the k chosen scores; row[0] holds the largest */
        double s0 = (double)row[0].value;
        double total = 0.0;
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)row[j].value - s0);
            total += ex[j];
        }
        for (int j = 0; j < k; ++j) {
            double w = ex[j] / total;
            topk_idx[t * k + j] = row[j].id;
            topk_w[t * k + j] = (float)w;
            if (topk_w_f64) topk_w_f64[t * k + j] = w;
        }
    }
    free(row);
    free(ex);
    return 0;
}

int oracle_topk_softmax_grouped(const float* logits, int64_t T, int E, int k, int n_groups,
                                int topk_groups, int32_t* topk_idx, float* topk_w,
                                double* topk_w_f64) {
    if (T < 0 || E < 1 || k < 1 || n_groups < 1 || E % n_groups != 0) return -1;
    if (topk_groups < 1 || topk_groups > n_groups) return -1;
    const int gsize = E / n_groups;
    if (k > topk_groups * gsize) return -1;
    if (T > 0 && (!logits || !topk_idx || !topk_w)) return -1;
    scored_expert* groups = (scored_expert*)malloc(sizeof(scored_expert) * (size_t)n_groups);
    scored_expert* row = (scored_expert*)malloc(sizeof(scored_expert) * (size_t)E);
    uint8_t* keep = (uint8_t*)malloc((size_t)n_groups);
    double* ex = (double*)malloc(sizeof(double) * (size_t)k);
    if (!groups || !row || !keep || !ex) { free(groups); free(row); free(keep); free(ex); return -2; }
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        /* score every group by its largest logit, then keep the best groups */
        for (int g = 0; g < n_groups; ++g) {
            float best = l[g * gsize];
            for (int i = 1; i < gsize; ++i)
                if (l[g * gsize + i] > best) best = l[g * gsize + i];
            groups[g].value = best;
            groups[g].id = g;
        }
        qsort(groups, (size_t)n_groups, sizeof(scored_expert), by_score_then_id);
        memset(keep, 0, (size_t)n_groups);
        for (int i = 0; i < topk_groups; ++i) keep[groups[i].id] = 1;
        /* top-k among the experts of the kept groups */
        int n = 0;
        for (int e = 0; e < E; ++e) {
            if (!keep[e / gsize]) continue;
            row[n].value = l[e];
            row[n].id = e;
            ++n;
        }
        qsort(row, (size_t)n, sizeof(scored_expert), by_score_then_id);
        double s0 = (double)row[0].value;
        double total = 0.0;
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)row[j].value - s0);
            total += ex[j];
        }
        for (int j = 0; j < k; ++j) {
            double w = ex[j] / total;
            topk_idx[t * k + j] = row[j].id;
            topk_w[t * k + j] = (float)w;
            if (topk_w_f64) topk_w_f64[t * k + j] = w;
        }
    }
    free(groups);
    free(row);
    free(keep);
    free(ex);
    return 0;
}

/* ------------------------------------------------------ routing indices */

int oracle_route_indices(const int32_t* topk_idx, const float* topk_w,
                         int64_t T, int E, int k, uint8_t* routing_map,
                         int32_t* counts, int32_t* offsets, int32_t* group_list,
                         int32_t* sorted_indices, int32_t* slot_pos,
                         float* permuted_probs) {
    if (T < 0 || E < 1 || k < 1) return -1;
    if (!counts || !offsets || !group_list) return -1;
    if (T > 0 && (!topk_idx || !sorted_indices || !slot_pos)) return -1;
    if (permuted_probs && !topk_w && T > 0) return -1;

    /* routing_map[t][e]: token t picked expert e */
    uint8_t* map = (uint8_t*)calloc((size_t)(T * E > 0 ? T * E : 1), 1);
    /* probs[t][e]: the weight token t gives expert e (0 where not picked) */
    float* probs = permuted_probs ? (float*)calloc((size_t)(T * E > 0 ? T * E : 1), sizeof(float)) : NULL;
    if (!map || (permuted_probs && !probs)) { free(map); free(probs); return -2; }
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t e = topk_idx[t * k + j];
            if (e == -1) continue;
            if (e < -1 || e >= E || map[t * E + e]) { free(map); free(probs); return -1; }
            map[t * E + e] = 1;
            if (probs) probs[t * E + e] = topk_w[t * k + j];
        }
    }
    if (routing_map) memcpy(routing_map, map, (size_t)(T * E));

    /* tokens per expert = column sums of the routing map */
    for (int e = 0; e < E; ++e) {
        int64_t c = 0;
        for (int64_t t = 0; t < T; ++t) c += map[t * E + e];
        counts[e] = (int32_t)c;
    }
    /* group_list: inclusive running total; offsets: the exclusive one */
    int64_t run = 0;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        run += counts[e];
        group_list[e] = (int32_t)run;
        offsets[e + 1] = (int32_t)run;
    }

    /* Scan the transposed map row by row (expert by expert, tokens in
     * ascending order) and keep the token ids where it is set: the order a
     * masked_select over routing_map.T yields.  Probabilities follow the
     * same scan. */
    int64_t p = 0;
    for (int e = 0; e < E; ++e) {
        for (int64_t t = 0; t < T; ++t) {
            if (!map[t * E + e]) continue;
            sorted_indices[p] = (int32_t)t;
            if (permuted_probs) permuted_probs[p] = probs[t * E + e];
            ++p;
        }
    }
    for (int64_t q = p; q < T * k; ++q) {
        sorted_indices[q] = -1;
        if (permuted_probs) permuted_probs[q] = 0.0f;
    }

    /* slot_pos: invert sorted_indices.  Row p of expert e's segment holds
     * token sorted_indices[p]; find the slot j in which that token chose e. */
    for (int64_t i = 0; i < T * k; ++i) slot_pos[i] = -1;
    for (int e = 0; e < E; ++e) {
        for (int64_t q = offsets[e]; q < offsets[e + 1]; ++q) {
            int64_t t = sorted_indices[q];
            for (int j = 0; j < k; ++j)
                if (topk_idx[t * k + j] == e) slot_pos[t * k + j] = (int32_t)q;
        }
    }
    free(map);
    free(probs);
    return 0;
}

/* ----------------------------------------------- capacity / padded layout */

int64_t oracle_expert_capacity(int64_t tokens, int top_k, int num_experts,
                               double capacity_factor) {
    if (tokens < 0 || top_k < 1 || num_experts < 1 || !(capacity_factor > 0.0)) return -1;
    return (int64_t)ceil((double)tokens * (double)top_k / (double)num_experts * capacity_factor);
}

int oracle_route_layout(const int32_t* topk_idx, const float* topk_w, int64_t T, int E, int k,
                        int capacity, int pad, int alignment, int64_t max_rows,
                        int32_t* counts, int32_t* offsets, int32_t* group_list,
                        int32_t* sorted_indices, int32_t* slot_pos, float* permuted_probs) {
    if (T < 0 || E < 1 || k < 1 || capacity < 0 || alignment < 1 || max_rows < 0) return -1;
    if (pad && capacity < 1) return -1;
    if (!counts || !offsets || !group_list) return -1;
    if (T > 0 && (!topk_idx || !slot_pos)) return -1;
    if (max_rows > 0 && !sorted_indices) return -1;
    if (permuted_probs && !topk_w && T > 0) return -1;
    /* rank of each (token, slot) inside its expert, tokens in order */
    int64_t* seen = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    if (!seen) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t e = topk_idx[t * k + j];
            slot_pos[t * k + j] = -1;
            if (e == -1) continue;
            int dup = 0;
            for (int q = 0; q < j; ++q) dup |= topk_idx[t * k + q] == e;
            if (e < -1 || e >= E || dup) { free(seen); return -1; }
            int64_t r = seen[e]++;
            /* keep the rank for now; turned into a row below */
            slot_pos[t * k + j] = (capacity > 0 && r >= capacity) ? -1 : (int32_t)r;
        }
    }
    /* segments and their prefixes */
    int64_t run = 0;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int64_t kept = capacity > 0 && seen[e] > capacity ? capacity : seen[e];
        counts[e] = (int32_t)kept;
        int64_t seg = pad ? capacity : (kept + alignment - 1) / alignment * alignment;
        run += seg;
        offsets[e + 1] = (int32_t)run;
        group_list[e] = (int32_t)run;
    }
    free(seen);
    if (run > max_rows) return -1;
    for (int64_t p = 0; p < max_rows; ++p) {
        sorted_indices[p] = -1;
        if (permuted_probs) permuted_probs[p] = 0.0f;
    }
    /* rank r of expert e goes to row offsets[e] + r */
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int32_t r = slot_pos[t * k + j];
            if (r < 0) continue;
            int32_t e = topk_idx[t * k + j];
            int64_t p = offsets[e] + r;
            slot_pos[t * k + j] = (int32_t)p;
            sorted_indices[p] = (int32_t)t;
            if (permuted_probs) permuted_probs[p] = topk_w[t * k + j];
        }
    }
    return 0;
}

/* -------------------------------------------------------------- FP8 e4m3 */

/* e4m3fn: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; normal values
 * (1 + m/8) * 2^(e-7) for e = 1..15 (e = 15, m = 7 is NaN), subnormals
 * m/8 * 2^-6.  Round |f| to a multiple of its quantum (2^(lead-3), or 2^-9
 * below 2^-6) with ties to even, saturate at 448, then encode. */
static uint8_t e4m3_bits(float f) {
    if (isnan(f)) return 0x7F;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    int ex;
    (void)frexp(a, &ex);
    int lead = ex - 1;
    if (lead < -6) lead = -6;
    double q = ldexp(1.0, lead - 3);
    double r = rint(a / q) * q;
    if (r > 448.0) r = 448.0;
    if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    (void)frexp(r, &ex);
    int e = ex - 1;                                   /* r in [2^e, 2^(e+1)) */
    int m = (int)(r / ldexp(1.0, e - 3)) - 8;         /* 0..7 */
    return (uint8_t)(sign | ((e + 7) << 3) | m);
}

static double e4m3_value(uint8_t b) {
    int e = (b >> 3) & 0xF, m = b & 7;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return (b & 0x80) ? -v : v;
}

int oracle_e4m3_from_float(const float* v, int64_t n, uint8_t* out) {
    if (n < 0 || (n > 0 && (!v || !out))) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_bits(v[i]);
    return 0;
}

int oracle_quantize_fp8(const uint16_t* x, int64_t T, int64_t H, int block, uint8_t* q,
                        float* scales) {
    if (T < 0 || H < 0 || block < 1 || H % block != 0) return -1;
    if (T > 0 && H > 0 && (!x || !q || !scales)) return -1;
    int64_t nb = H / block;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int64_t i = 0; i < block; ++i) {
                float v = fabsf((float)bf16_bits_to_double(x[t * H + b * block + i]));
                if (v > amax) amax = v;
            }
            float s = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[t * nb + b] = s;
            for (int64_t i = 0; i < block; ++i) {
                float v = (float)bf16_bits_to_double(x[t * H + b * block + i]);
                q[t * H + b * block + i] = e4m3_bits(v / s);
            }
        }
    }
    return 0;
}

int oracle_dequantize_fp8(const uint8_t* q, const float* scales, int64_t N, int64_t H,
                          int block, uint16_t* out) {
    if (N < 0 || H < 0 || block < 1 || H % block != 0) return -1;
    if (N > 0 && H > 0 && (!q || !scales || !out)) return -1;
    int64_t nb = H / block;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t h = 0; h < H; ++h)
            out[r * H + h] = double_to_bf16_bits(e4m3_value(q[r * H + h]) *
                                                 (double)scales[r * nb + h / block]);
    return 0;
}

/* --------------------------------------------------------------- permute */

int oracle_permute(const void* x, int elem_size, int64_t T, int64_t H,
                   const int32_t* sorted_indices, int64_t n_rows, void* out) {
    if (T < 0 || H < 0 || n_rows < 0 || (elem_size != 1 && elem_size != 2 && elem_size != 4))
        return -1;
    if (n_rows > 0 && (!x || !sorted_indices || !out)) return -1;
    size_t row = (size_t)(H * elem_size);
    for (int64_t p = 0; p < n_rows; ++p) {
        int64_t t = sorted_indices[p];
        if (t < 0 || t >= T) return -1;
        memcpy((char*)out + (size_t)p * row, (const char*)x + (size_t)t * row, row);
    }
    return 0;
}

/* ----------------------------------------------------------- sort_chunks */

int oracle_chunk_idxs(int R, int L, int inverse, int32_t* idxs) {
    if (R < 1 || L < 1 || !idxs) return -1;
    /* A matrix [A x B] numbered row-major, read column by column: entry
     * (a, b) has number a*B + b and is read at position b*A + a. */
    if (!inverse) {
        for (int r = 0; r < R; ++r)
            for (int l = 0; l < L; ++l) idxs[l * R + r] = r * L + l;
    } else {
        for (int l = 0; l < L; ++l)
            for (int r = 0; r < R; ++r) idxs[r * L + l] = l * R + r;
    }
    return 0;
}

int oracle_sort_chunks(const void* in, int64_t row_bytes, int64_t N,
                       const int32_t* split_sizes, const int32_t* sorted_idxs,
                       int C, void* out) {
    if (row_bytes < 0 || N < 0 || C < 0) return -1;
    if (C > 0 && (!split_sizes || !sorted_idxs)) return -1;
    int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)(C + 1));
    uint8_t* seen = (uint8_t*)calloc((size_t)(C + 1), 1);
    if (!start || !seen) { free(start); free(seen); return -2; }
    /* chunks = in.split(split_sizes): chunk c starts where chunk c-1 ended */
    start[0] = 0;
    for (int c = 0; c < C; ++c) {
        if (split_sizes[c] < 0) { free(start); free(seen); return -1; }
        start[c + 1] = start[c] + split_sizes[c];
    }
    if (start[C] != N) { free(start); free(seen); return -1; }
    /* out = cat([chunks[i] for i in sorted_idxs]) */
    int64_t dst = 0;
    for (int i = 0; i < C; ++i) {
        int c = sorted_idxs[i];
        if (c < 0 || c >= C || seen[c]) { free(start); free(seen); return -1; }
        seen[c] = 1;
        int64_t rows = split_sizes[c];
        if (rows > 0)
            memcpy((char*)out + dst * row_bytes, (const char*)in + start[c] * row_bytes,
                   (size_t)(rows * row_bytes));
        dst += rows;
    }
    free(start);
    free(seen);
    return 0;
}

/* --------------------------------------------------------------- combine */

int oracle_combine(const void* y, int dtype, int64_t T, int64_t H, int k,
                   const int32_t* slot_pos, const float* topk_w, void* out,
                   double* out_f64) {
    if (!dtype_ok(dtype) || T < 0 || H < 0 || k < 1) return -1;
    if (T > 0 && H > 0 && (!y || !slot_pos || !out)) return -1;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!acc) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
        for (int j = 0; j < k; ++j) {           /* slot order */
            int64_t p = slot_pos[t * k + j];
            if (p < 0) continue;
            double w = topk_w ? (double)topk_w[t * k + j] : 1.0;
            for (int64_t h = 0; h < H; ++h) acc[h] += w * load_elem(y, dtype, p * H + h);
        }
        for (int64_t h = 0; h < H; ++h) {
            store_elem(out, dtype, t * H + h, acc[h]);
            if (out_f64) out_f64[t * H + h] = acc[h];
        }
    }
    free(acc);
    return 0;
}

int oracle_unpermute(const void* y, int dtype, int64_t T, int64_t H,
                     const int32_t* sorted_indices, const float* probs,
                     int64_t n_valid, void* out, double* out_f64) {
    if (!dtype_ok(dtype) || T < 0 || H < 0 || n_valid < 0) return -1;
    double* acc = (double*)calloc((size_t)(T * H > 0 ? T * H : 1), sizeof(double));
    if (!acc) return -2;
    for (int64_t p = 0; p < n_valid; ++p) {
        int64_t t = sorted_indices[p];
        if (t < 0 || t >= T) { free(acc); return -1; }
        double w = probs ? (double)probs[p] : 1.0;
        for (int64_t h = 0; h < H; ++h) acc[t * H + h] += w * load_elem(y, dtype, p * H + h);
    }
    for (int64_t i = 0; i < T * H; ++i) {
        store_elem(out, dtype, i, acc[i]);
        if (out_f64) out_f64[i] = acc[i];
    }
    free(acc);
    return 0;
}

int oracle_combine_backward(const void* grad_out, const void* y, int dtype,
                            int64_t T, int64_t H, int k,
                            const int32_t* slot_pos, const float* topk_w,
                            void* grad_y, float* grad_probs,
                            double* grad_probs_f64) {
    if (!dtype_ok(dtype) || T < 0 || H < 0 || k < 1) return -1;
    if (T > 0 && (!grad_out || !y || !slot_pos || !grad_y || !grad_probs)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int64_t p = slot_pos[t * k + j];
            if (p < 0) {
                grad_probs[t * k + j] = 0.0f;
                if (grad_probs_f64) grad_probs_f64[t * k + j] = 0.0;
                continue;
            }
            double w = topk_w ? (double)topk_w[t * k + j] : 1.0;
            double dot = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                double g = load_elem(grad_out, dtype, t * H + h);
                store_elem(grad_y, dtype, p * H + h, w * g);
                dot += g * load_elem(y, dtype, p * H + h);
            }
            grad_probs[t * k + j] = (float)dot;
            if (grad_probs_f64) grad_probs_f64[t * k + j] = dot;
        }
    }
    return 0;
}

/* ---------------------------------------------------------- router backward */

int oracle_route_backward(const int32_t* topk_idx, const float* topk_w,
                          const float* grad_probs, int64_t T, int E, int k,
                          float* grad_logits) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    if (T > 0 && (!topk_idx || !topk_w || !grad_probs || !grad_logits)) return -1;
    for (int64_t t = 0; t < T; ++t) {
        const int32_t* id = topk_idx + t * k;
        for (int j = 0; j < k; ++j) {
            if (id[j] < -1 || id[j] >= E) return -1;
            for (int i = 0; i < j; ++i)
                if (id[j] >= 0 && id[i] == id[j]) return -1;
        }
        double dot = 0.0;
        for (int j = 0; j < k; ++j)
            if (id[j] >= 0)
                dot += (double)topk_w[t * k + j] * (double)grad_probs[t * k + j];
        for (int e = 0; e < E; ++e) grad_logits[t * E + e] = 0.0f;
        for (int i = 0; i < k; ++i) {
            if (id[i] < 0) continue;
            double d = (double)grad_probs[t * k + i] - dot;
            grad_logits[t * E + id[i]] = (float)((double)topk_w[t * k + i] * d);
        }
    }
    return 0;
}

/* ---------------------------------------------------------- stand-in expert */

int oracle_expert_scale(const void* x_perm, int dtype, int64_t H, int E,
                        const int32_t* offsets, const float* scale, void* y) {
    if (!dtype_ok(dtype) || H < 0 || E < 1 || !offsets || !scale) return -1;
    for (int e = 0; e < E; ++e) {
        double s = (double)scale[e];
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p)
            for (int64_t h = 0; h < H; ++h)
                store_elem(y, dtype, p * H + h, load_elem(x_perm, dtype, p * H + h) * s);
    }
    return 0;
}

/* -------------------------------------------------------- grouped SwiGLU */

static double silu(double z) { return z / (1.0 + exp(-z)); }

static int expert_of_row(const int32_t* offsets, int E, int64_t p) {
    for (int e = 0; e < E; ++e)
        if (p >= offsets[e] && p < offsets[e + 1]) return e;
    return -1;
}

int oracle_grouped_swiglu(const uint16_t* x, const uint16_t* w_up,
                          const uint16_t* w_down, const int32_t* offsets,
                          int E, int64_t H, int64_t I,
                          const int64_t* rows, int64_t n_rows,
                          uint16_t* y, double* y_f64,
                          uint16_t* gate_up_out, uint16_t* hidden_out) {
    if (E < 1 || H < 1 || I < 1 || !x || !w_up || !w_down || !offsets || !y) return -1;
    int64_t total = offsets[E];
    int64_t count = rows ? n_rows : total;
    double* gate_up = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* hidden = (double*)malloc(sizeof(double) * (size_t)I);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    if (!gate_up || !hidden || !acc) { free(gate_up); free(hidden); free(acc); return -2; }
    for (int64_t r = 0; r < count; ++r) {
        int64_t p = rows ? rows[r] : r;
        int e = expert_of_row(offsets, E, p);
        if (e < 0) { free(gate_up); free(hidden); free(acc); return -1; }
        const uint16_t* up_e = w_up + (size_t)e * (size_t)(H * 2 * I);
        const uint16_t* down_e = w_down + (size_t)e * (size_t)(I * H);
        /* GMM1: gate_up = x[p] @ w_up[e] */
        for (int64_t c = 0; c < 2 * I; ++c) gate_up[c] = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            double xv = bf16_bits_to_double(x[p * H + h]);
            const uint16_t* wrow = up_e + h * 2 * I;
            for (int64_t c = 0; c < 2 * I; ++c) gate_up[c] += xv * bf16_bits_to_double(wrow[c]);
        }
        /* SwiGLU: first I columns are the gate, last I the up projection */
        for (int64_t i = 0; i < I; ++i)
            hidden[i] = bf16_bits_to_double(double_to_bf16_bits(silu(gate_up[i]) * gate_up[I + i]));
        if (gate_up_out)
            for (int64_t c = 0; c < 2 * I; ++c)
                gate_up_out[p * 2 * I + c] = double_to_bf16_bits(gate_up[c]);
        if (hidden_out)
            for (int64_t i = 0; i < I; ++i) hidden_out[p * I + i] = double_to_bf16_bits(hidden[i]);
        /* GMM2: y[p] = hidden @ w_down[e] */
        for (int64_t h = 0; h < H; ++h) acc[h] = 0.0;
        for (int64_t i = 0; i < I; ++i) {
            const uint16_t* wrow = down_e + i * H;
            for (int64_t h = 0; h < H; ++h) acc[h] += hidden[i] * bf16_bits_to_double(wrow[h]);
        }
        for (int64_t h = 0; h < H; ++h) {
            y[p * H + h] = double_to_bf16_bits(acc[h]);
            if (y_f64) y_f64[p * H + h] = acc[h];
        }
    }
    free(gate_up);
    free(hidden);
    free(acc);
    return 0;
}

/* ------------------------------------------------- grouped SwiGLU backward */

int oracle_swiglu_dgrad(const uint16_t* dy, const uint16_t* w_up, const uint16_t* w_down,
                        const int32_t* offsets, const uint16_t* gate_up, int E, int64_t H,
                        int64_t I, const int64_t* rows, int64_t n_rows, uint16_t* dgate_up,
                        double* dgate_up_f64, uint16_t* dx, double* dx_f64) {
    if (E < 1 || H < 1 || I < 1 || !dy || !w_up || !w_down || !offsets || !gate_up ||
        !dgate_up || !dx)
        return -1;
    int64_t count = rows ? n_rows : offsets[E];
    double* dh = (double*)malloc(sizeof(double) * (size_t)I);
    double* dgu = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    if (!dh || !dgu) { free(dh); free(dgu); return -2; }
    for (int64_t r = 0; r < count; ++r) {
        int64_t p = rows ? rows[r] : r;
        int e = expert_of_row(offsets, E, p);
        if (e < 0) { free(dh); free(dgu); return -1; }
        const uint16_t* up_e = w_up + (size_t)e * (size_t)(H * 2 * I);
        const uint16_t* down_e = w_down + (size_t)e * (size_t)(I * H);
        /* GMM2 backward: dh = dy[p] @ w_down[e]^T */
        for (int64_t i = 0; i < I; ++i) {
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += bf16_bits_to_double(dy[p * H + h]) * bf16_bits_to_double(down_e[i * H + h]);
            dh[i] = acc;
        }
        /* SwiGLU backward at the stored gate / up values */
        for (int64_t i = 0; i < I; ++i) {
            double g = bf16_bits_to_double(gate_up[p * 2 * I + i]);
            double u = bf16_bits_to_double(gate_up[p * 2 * I + I + i]);
            double sg = 1.0 / (1.0 + exp(-g));
            dgu[i] = dh[i] * u * sg * (1.0 + g * (1.0 - sg));
            dgu[I + i] = dh[i] * g * sg;
        }
        for (int64_t c = 0; c < 2 * I; ++c) {
            dgate_up[p * 2 * I + c] = double_to_bf16_bits(dgu[c]);
            if (dgate_up_f64) dgate_up_f64[p * 2 * I + c] = dgu[c];
        }
        /* GMM1 backward from the stored (bf16) dgate_up: dx = dgate_up @ w_up[e]^T */
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t c = 0; c < 2 * I; ++c)
                acc += bf16_bits_to_double(dgate_up[p * 2 * I + c]) *
                       bf16_bits_to_double(up_e[h * 2 * I + c]);
            dx[p * H + h] = double_to_bf16_bits(acc);
            if (dx_f64) dx_f64[p * H + h] = acc;
        }
    }
    free(dh);
    free(dgu);
    return 0;
}

int oracle_swiglu_wgrad_at(const uint16_t* x, const uint16_t* hidden, const uint16_t* dy,
                           const uint16_t* dgate_up, const int32_t* offsets, int E, int64_t H,
                           int64_t I, int which, const int64_t* coords, int64_t n,
                           double* out) {
    if (E < 1 || H < 1 || I < 1 || !offsets || !coords || (n > 0 && !out)) return -1;
    if (which != 0 && which != 1) return -1;
    if (which == 0 && (!x || !dgate_up)) return -1;
    if (which == 1 && (!hidden || !dy)) return -1;
    for (int64_t q = 0; q < n; ++q) {
        int64_t e = coords[3 * q], a = coords[3 * q + 1], b = coords[3 * q + 2];
        if (e < 0 || e >= E || a < 0 || b < 0) return -1;
        double acc = 0.0;
        if (which == 0) {            /* dW_up[e][h=a][c=b] = sum_p x[p,h] dgate_up[p,c] */
            if (a >= H || b >= 2 * I) return -1;
            for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p)
                acc += bf16_bits_to_double(x[p * H + a]) *
                       bf16_bits_to_double(dgate_up[p * 2 * I + b]);
        } else {                     /* dW_down[e][i=a][h=b] = sum_p hidden[p,i] dy[p,h] */
            if (a >= I || b >= H) return -1;
            for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p)
                acc += bf16_bits_to_double(hidden[p * I + a]) * bf16_bits_to_double(dy[p * H + b]);
        }
        out[q] = acc;
    }
    return 0;
}
