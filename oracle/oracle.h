/*
 * oracle.h -- plain, slow CPU reference for the MoE dispatch/combine path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include,
 * link or call this code; only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no source with the CUDA
 * path: its own types, its own bf16 conversion, its own loops.
 *
 * Every floating-point result is accumulated in IEEE double and rounded once
 * (round-to-nearest-even) to the output type.  All loops run in the order the
 * definitions below state; there is no blocking, fusion or reordering.
 *
 * Sources (web pages, cited by title and section):
 *  [MOE-OPS]  "从零理解 MoE 算子：路由、专家并行与 Token 重排"
 *             (www.171host.com/746420.html) -- a from-scratch MoE operator
 *             tutorial: §3 Router, §7 GroupedMatMul, §8 expert FFN,
 *             §11-13 rank-major / expert-major, §16 top-k merge.
 *  [COMBINE]  "03 · Combine 与 forward / backward 对称性"
 *             (llm-infra-atlas.github.io/parallel/05_ep/03_combine_and_backward/)
 *             -- §1 combine formula, §2.1 sort_chunks inverse, §2.3
 *             unpermute = scatter_add, §4 backward symmetry table.
 *  [DISPATCH] "token dispatcher + fuse_a2a" (obnotes-4iw.pages.dev, Megatron
 *             transformer-moe notes) -- §1.1 Alltoall: the permute()
 *             walk-through (transposed routing map, masked_select, index_select)
 *             and its worked example.
 *
 * Conventions: tensors are row-major and contiguous.  bf16 values are passed
 * as their 16-bit patterns (uint16_t).  An expert id of -1 in topk_idx marks an
 * empty slot: it routes nothing and its slot position is -1.
 * Return value: 0 on success, a negative number on invalid arguments.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Round each double to bf16 (nearest, ties to even; subnormals and overflow
 * to infinity handled).  Exported so tests can pin it to a library routine. */
int oracle_bf16_from_double(const double* v, int64_t n, uint16_t* out);

/* [MOE-OPS] §3: topk_scores, topk_indices = topk(router_logits, k);
 * topk_weights = softmax(topk_scores).
 * Slot order: descending logit; equal logits go to the lower expert id.
 * Softmax over the k chosen scores, stabilised by the largest one, in double;
 * topk_w is that value rounded to float, topk_w_f64 (nullable) the double. */
int oracle_topk_softmax(const float* logits, int64_t T, int E, int k,
                        int32_t* topk_idx, float* topk_w, double* topk_w_f64);

/* Group-limited top-k, [MOE-OPS] §21: the E experts form n_groups
 * consecutive groups of E/n_groups; a group's score is its largest logit;
 * the topk_groups groups with the largest scores are kept (equal scores: the
 * lower group id); then top-k as in oracle_topk_softmax over the experts of
 * the kept groups only, and the softmax over those k scores.
 * Requires E % n_groups == 0, 1 <= topk_groups <= n_groups and
 * k <= topk_groups * (E / n_groups). */
int oracle_topk_softmax_grouped(const float* logits, int64_t T, int E, int k, int n_groups,
                                int topk_groups, int32_t* topk_idx, float* topk_w,
                                double* topk_w_f64);

/* From topk_idx [T,k] build, following [DISPATCH] §1.1 and [MOE-OPS] §7:
 *  routing_map [T,E]   1 where expert e is among token t's choices (nullable)
 *  counts [E]          tokens per expert (column sums of the routing map)
 *  offsets [E+1]       exclusive prefix of counts, offsets[0] = 0
 *  group_list [E]      inclusive prefix of counts
 *  sorted_indices [T*k] token ids, expert-major, ascending token inside an
 *                      expert (the order of a row-major scan of the
 *                      transposed routing map); entries past offsets[E] = -1
 *  slot_pos [T,k]      position of (t, topk_idx[t,j]) in sorted_indices, -1
 *                      for an empty slot
 *  permuted_probs [T*k] topk_w rearranged into sorted_indices order; entries
 *                      past offsets[E] = 0 (nullable; needs topk_w)
 * Fails on an expert id outside [-1, E) or a token naming an expert twice. */
int oracle_route_indices(const int32_t* topk_idx, const float* topk_w,
                         int64_t T, int E, int k, uint8_t* routing_map,
                         int32_t* counts, int32_t* offsets, int32_t* group_list,
                         int32_t* sorted_indices, int32_t* slot_pos,
                         float* permuted_probs);

/* [MOE-OPS] §18: expert_capacity = ceil(tokens * top_k / num_experts *
 * capacity_factor), evaluated in double. */
int64_t oracle_expert_capacity(int64_t tokens, int top_k, int num_experts,
                               double capacity_factor);

/* Capacity-bounded, padded or aligned layout of the permuted rows
 * ([MOE-OPS] §18 capacity, [DISPATCH] §1.1 drop_and_pad, DeepEP
 * expert_alignment in [COMBINE] §6):
 *  - the tokens of expert e, in token order, get ranks 0, 1, ...; with
 *    capacity > 0 only ranks < capacity are kept, the others dropped (their
 *    slot_pos is -1; they contribute nothing downstream)
 *  - counts[e] = kept tokens of expert e
 *  - segment of e: capacity rows if pad, else counts[e] rounded up to a
 *    multiple of alignment (>= 1)
 *  - offsets / group_list: exclusive / inclusive prefix of the segments
 *  - sorted_indices[offsets[e] + r] = token of rank r; padding rows and rows
 *    from offsets[E] to max_rows are -1 (permuted_probs 0 there)
 * Fails if offsets[E] would exceed max_rows. */
int oracle_route_layout(const int32_t* topk_idx, const float* topk_w, int64_t T, int E, int k,
                        int capacity, int pad, int alignment, int64_t max_rows,
                        int32_t* counts, int32_t* offsets, int32_t* group_list,
                        int32_t* sorted_indices, int32_t* slot_pos, float* permuted_probs);

/* FP8 dispatch ([COMBINE] §3: the dispatch moves FP8 rows with scales, the
 * combine stays BF16; [DISPATCH] names x_scales / num_scales): per token and
 * per block of `block` consecutive elements, scale = amax / 448 (448 = the
 * largest finite e4m3 value; an all-zero block gets scale 1), and each
 * element becomes e4m3(x / scale): the float quotient rounded to nearest
 * even e4m3, saturated to +-448.  x: bf16 [T,H]; q: e4m3 bytes [T,H];
 * scales: float [T, H/block]. */
int oracle_quantize_fp8(const uint16_t* x, int64_t T, int64_t H, int block, uint8_t* q,
                        float* scales);

/* out = bf16(q * scale): the exact product rounded once. */
int oracle_dequantize_fp8(const uint8_t* q, const float* scales, int64_t N, int64_t H,
                          int block, uint16_t* out);

/* e4m3 (fn: no infinities, 0x7F/0xFF NaN) of a float: nearest, ties to even,
 * saturated to +-448.  Exported for the pins. */
int oracle_e4m3_from_float(const float* v, int64_t n, uint8_t* out);

/* [DISPATCH] §1.1 permuted_input = tokens.index_select(0, sorted_indices):
 * out[p] = x[sorted_indices[p]] for p < n_rows; elem_size 4, 2 or 1 bytes. */
int oracle_permute(const void* x, int elem_size, int64_t T, int64_t H,
                   const int32_t* sorted_indices, int64_t n_rows, void* out);

/* Chunk orders for a [R source ranks x L local experts] split matrix,
 * [COMBINE] §2.1 and [MOE-OPS] §11-13:
 *  inverse = 0: rank-major -> expert-major, idxs[l*R + r] = r*L + l
 *  inverse = 1: expert-major -> rank-major, idxs[r*L + l] = l*R + r          */
int oracle_chunk_idxs(int R, int L, int inverse, int32_t* idxs);

/* sort_chunks_by_idxs: cut `in` [N rows] into C consecutive chunks of
 * split_sizes[c] rows, then write chunk sorted_idxs[0], sorted_idxs[1], ...
 * back to back into `out`.  Requires sum(split_sizes) == N and sorted_idxs a
 * permutation of 0..C-1. */
int oracle_sort_chunks(const void* in, int64_t row_bytes, int64_t N,
                       const int32_t* split_sizes, const int32_t* sorted_idxs,
                       int C, void* out);

/* [COMBINE] §1, [MOE-OPS] §16:
 * out[t] = sum_{j=0..k-1} topk_w[t,j] * y[slot_pos[t,j]], accumulated in
 * double in slot order j = 0..k-1, rounded once to `dtype`.
 * topk_w = NULL gives the unweighted sum.  out_f64 (nullable) keeps the
 * double sums. */
int oracle_combine(const void* y, int dtype, int64_t T, int64_t H, int k,
                   const int32_t* slot_pos, const float* topk_w, void* out,
                   double* out_f64);

/* [COMBINE] §2.3 unpermute as a scatter-add: out = zeros([T,H]);
 * out[sorted_indices[p]] += probs[p] * y[p] for p < n_valid (probs NULL = 1),
 * in double, in ascending p, rounded once.  A second statement of the same
 * combine, used to cross-check oracle_combine. */
int oracle_unpermute(const void* y, int dtype, int64_t T, int64_t H,
                     const int32_t* sorted_indices, const float* probs,
                     int64_t n_valid, void* out, double* out_f64);

/* Router backward: only the chosen experts' probabilities carry gradient
 * ([COMBINE] §6, backward pseudocode), and w is the softmax over the k chosen
 * logits ([MOE-OPS] §3).  With g = dL/dw (grad_probs of the combine backward)
 * the softmax Jacobian dw_j/ds_i = w_j (delta_ij - w_i) gives
 *   grad_logits[t, topk_idx[t,i]] = w_i * (g_i - sum_j w_j g_j)
 * and 0 for every expert not chosen.  Double arithmetic: the sum over the
 * valid slots in slot order, then the difference, the product, one rounding
 * to float.  Slots with id -1 are skipped.  Fails on an id >= E or < -1, or
 * an id repeated within a token. */
int oracle_route_backward(const int32_t* topk_idx, const float* topk_w,
                          const float* grad_probs, int64_t T, int E, int k,
                          float* grad_logits);

/* [COMBINE] §4 (the backward of the linear combine is its transpose):
 *  grad_y[slot_pos[t,j]] = topk_w[t,j] * grad_out[t]      (rounded once)
 *  grad_probs[t,j]       = sum_h grad_out[t,h] * y[slot_pos[t,j],h]
 *                          (double, ascending h, rounded to float)
 * topk_w = NULL means every weight is 1.  Empty slots give grad_probs 0 and
 * write no row.  grad_probs_f64 (nullable) keeps the double dots. */
int oracle_combine_backward(const void* grad_out, const void* y, int dtype,
                            int64_t T, int64_t H, int k,
                            const int32_t* slot_pos, const float* topk_w,
                            void* grad_y, float* grad_probs,
                            double* grad_probs_f64);

/* Stand-in expert: y[p] = x_perm[p] * scale[e] for offsets[e] <= p <
 * offsets[e+1], product in double, rounded once. */
int oracle_expert_scale(const void* x_perm, int dtype, int64_t H, int E,
                        const int32_t* offsets, const float* scale, void* y);

/* [MOE-OPS] §7-8 GMM1 -> SwiGLU -> GMM2 per expert over group_list segments:
 *  gate_up = X_e @ w_up[e]            [n, 2I]  (double)
 *  gate, up = gate_up[:, :I], gate_up[:, I:]
 *  hidden = silu(gate) * up           rounded to bf16 (the stored activation)
 *  y_e = hidden @ w_down[e]           [n, H]   (double, rounded to bf16)
 * x [N,H], w_up [E,H,2I], w_down [E,I,H], y [N,H], all bf16 patterns.
 * rows (nullable): compute only these n_rows row ids; otherwise every row in
 * [0, offsets[E]).  y_f64 (nullable) has the same layout as y.
 * gate_up_out [N,2I] and hidden_out [N,I] (nullable): the bf16 gate_up and
 * hidden a training forward keeps for the backward. */
int oracle_grouped_swiglu(const uint16_t* x, const uint16_t* w_up,
                          const uint16_t* w_down, const int32_t* offsets,
                          int E, int64_t H, int64_t I,
                          const int64_t* rows, int64_t n_rows,
                          uint16_t* y, double* y_f64,
                          uint16_t* gate_up_out, uint16_t* hidden_out);

/* Backward of the grouped SwiGLU, [MOE-OPS] §22 (GMM2 backward -> SwiGLU
 * backward -> GMM1 backward, giving dX, dW1, dW2) and [COMBINE] §4.2 (dgrad
 * m-grouped, wgrad k-grouped), per expert segment, from the stored bf16
 * gate_up [N,2I] and upstream gradient dy [N,H]:
 *  dh       = dy @ w_down[e]^T                               (double)
 *  s        = sigmoid(gate)
 *  d_gate   = dh * up * s * (1 + gate * (1 - s))   (derivative of gate*s)
 *  d_up     = dh * gate * s                        (= dh * silu(gate))
 *  dgate_up = [d_gate | d_up]                      rounded to bf16 (stored)
 *  dx       = dgate_up @ w_up[e]^T   from the stored bf16 dgate_up, rounded
 * rows (nullable) as in oracle_grouped_swiglu.  The *_f64 outputs
 * (nullable) keep the unrounded doubles. */
int oracle_swiglu_dgrad(const uint16_t* dy, const uint16_t* w_up, const uint16_t* w_down,
                        const int32_t* offsets, const uint16_t* gate_up, int E, int64_t H,
                        int64_t I, const int64_t* rows, int64_t n_rows, uint16_t* dgate_up,
                        double* dgate_up_f64, uint16_t* dx, double* dx_f64);

/* Weight gradients (the k-grouped GEMMs: a sum over each expert's rows), in
 * double, at n coordinates (e, a, b) given as coords[3q..3q+2]:
 *  which 0: dW_up[e][h=a][c=b]   = sum_{p in e} x[p,h] * dgate_up[p,c]
 *  which 1: dW_down[e][i=a][h=b] = sum_{p in e} hidden[p,i] * dy[p,h]
 * An expert with no rows has zero gradient. */
int oracle_swiglu_wgrad_at(const uint16_t* x, const uint16_t* hidden, const uint16_t* dy,
                           const uint16_t* dgate_up, const int32_t* offsets, int E, int64_t H,
                           int64_t I, int which, const int64_t* coords, int64_t n,
                           double* out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ORACLE_H */
