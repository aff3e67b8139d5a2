/*
 * moe.h -- C ABI of libmoe, the GB300 (sm_103a) MoE token dispatch/combine
 * library.  One GPU, one stream per call, hand-written CUDA kernels only.
 *
 * Sources (web pages, cited by title and section):
 *  [MOE-OPS]  "从零理解 MoE 算子：路由、专家并行与 Token 重排"
 *             (www.171host.com/746420.html): §3 Router and top-k, §6 grouping
 *             tokens by expert, §7 GroupedMatMul and group_list, §8 expert
 *             FFN (GMM1 -> SwiGLU -> GMM2), §11-13 rank-major / expert-major
 *             permute and unpermute, §16 merging the top-k outputs, §26 edge
 *             cases.
 *  [COMBINE]  "03 · Combine 与 forward / backward 对称性"
 *             (llm-infra-atlas.github.io/parallel/05_ep/03_combine_and_backward/):
 *             §1 the combine formula, §2.1 unpermute-2 with transposed splits,
 *             §2.3 unpermute as a (weighted) scatter-add, §4 the backward
 *             symmetry table.
 *  [DISPATCH] "token dispatcher + fuse_a2a" (obnotes-4iw.pages.dev, Megatron
 *             transformer-moe notes): §1.1 the permute() walk-through.
 *
 * Conventions for every entry point
 *  - Tensors are caller-owned DEVICE pointers (unless a parameter says
 *    "host"), row-major and contiguous.  The library never allocates device
 *    memory; scratch space is a caller-provided workspace whose size the
 *    matching *_workspace_size call returns.  Workspaces must be 256-byte
 *    aligned and may be reused across calls on the same stream.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  Host-side validation happens before
 *    any launch and returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE with nothing launched.  A failed launch returns
 *    MOE_ERR_CUDA.  Problems only the device can see (an expert id out of
 *    range, splits that do not add up) are recorded in the workspace's
 *    status word and read back with moe_workspace_status(); device code never
 *    traps.
 *  - Sizes: T tokens, H hidden elements per row, E experts, k = top_k.
 *    1 <= k <= min(E, 32), 1 <= E <= 1024, T*k < 2^31, H*element < 2^31.
 *    T = 0 and H = 0 are valid and do nothing (routing outputs still zeroed).
 *  - Activations are MOE_F32 or MOE_BF16; logits, weights and probabilities
 *    are float32; indices int32.  Rows whose byte length is a multiple of 16
 *    and whose base pointers are 16-byte aligned take the vectorised path;
 *    anything else takes an element-wise path with identical results.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad pointer, size or dtype: nothing launched */
    MOE_ERR_UNSUPPORTED = 2,   /* outside the supported ranges above           */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned   */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed         */
    MOE_ERR_TIMEOUT = 5,       /* a bounded device wait gave up                */
    MOE_ERR_DEVICE_CHECK = 6   /* the device found invalid data (see above)    */
} moe_status_t;

/* Element types.  MOE_FP8_E4M3 (one byte: 1 sign, 4 exponent, 3 mantissa
 * bits, no infinities) is accepted by the row-movement calls only
 * (moe_permute, moe_sort_chunks, moe_fill_pad_rows). */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8_E4M3 = 2 } moe_dtype_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status_t status);

/* ABI version of this header (bumped on any signature change): 2. */
int moe_abi_version(void);

/* ------------------------------------------------------------------ route
 * [MOE-OPS] §3: topk_scores, topk_indices = topk(router_logits, k);
 * topk_weights = softmax(topk_scores).  [DISPATCH] §1.1 and [MOE-OPS] §7:
 * routing map, tokens per expert, group_list, and the expert-major
 * sorted_indices that a masked_select over the transposed routing map yields.
 *
 * Inputs
 *   logits [T,E] float32 (finite values).
 * Outputs (all device, caller-owned, written completely)
 *   topk_idx [T,k] int32   chosen experts, descending logit; equal logits go
 *                          to the lower expert id
 *   topk_w [T,k] float32   softmax over the k chosen logits (fp32, stabilised
 *                          by the largest); rows sum to 1
 *   counts [E] int32       tokens routed to each expert
 *   offsets [E+1] int32    exclusive prefix of counts (offsets[0] = 0): expert
 *                          e owns permuted rows [offsets[e], offsets[e+1])
 *   group_list [E] int32   inclusive prefix of counts ([3,2,4] -> [3,5,9])
 *   sorted_indices [T*k]   source token of each permuted row: expert-major,
 *                          ascending token inside an expert; entries past
 *                          offsets[E] are -1
 *   slot_pos [T,k] int32   permuted row of (t, slot j); -1 for an empty slot.
 *                          sorted_indices[slot_pos[t,j]] == t.
 *   permuted_probs [T*k]   topk_w[t,j] stored at row slot_pos[t,j]; 0 past
 *                          offsets[E]
 *   routing_map [T,E] u8   1 where token t picked expert e (NULL: not written)
 * Every integer output is bit-exact and independent of launch order.
 * Workspace: moe_route_workspace_size(T, E, k) bytes.  Nothing in it needs to
 * be cleared, and between calls it may hold anything (other data, random
 * bytes): every call writes the scratch it reads, except the fused route's
 * grid-barrier count and marker.  A call checks those against what the
 * previous call on this workspace left; if either differs, it passes the
 * barrier by per-block flags, which are correct for any contents (about
 * 1 us slower), and leaves the count and marker ready for the next call.
 * Calls that share a workspace must not overlap on the GPU.  Device status:
 * up to 256 experts the logits reach shared memory through bounded
 * bulk-copy waits; one that gives up records MOE_ERR_TIMEOUT in the
 * library's device status word (moe_device_status). */
moe_status_t moe_route_workspace_size(int64_t T, int E, int k, size_t* bytes);

moe_status_t moe_route(const float* logits, int64_t T, int E, int k,
                       int32_t* topk_idx, float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* group_list,
                       int32_t* sorted_indices, int32_t* slot_pos,
                       float* permuted_probs, uint8_t* routing_map,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Group-limited routing, [MOE-OPS] §21: the E experts form n_groups
 * consecutive groups of E/n_groups (n_groups <= 32, E % n_groups == 0); a
 * group's score is its largest logit; the topk_groups best groups are kept
 * (equal scores: the lower group id) and the k experts are chosen among the
 * kept groups' experts only (k <= topk_groups * E/n_groups), with the same
 * tie rule, softmax and outputs as moe_route.  n_groups = topk_groups gives
 * exactly moe_route.  Workspace: moe_route_workspace_size(T, E, k). */
moe_status_t moe_route_grouped(const float* logits, int64_t T, int E, int k,
                               int n_groups, int topk_groups,
                               int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* group_list,
                               int32_t* sorted_indices, int32_t* slot_pos,
                               float* permuted_probs, uint8_t* routing_map,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The index half of moe_route for a caller that already has the top-k
 * choices.  topk_idx [T,k] may contain -1 for an empty slot; topk_w (nullable)
 * only feeds permuted_probs (NULL: permuted_probs is not written and may be
 * NULL).  An id outside [-1, E) or an expert named twice by one token marks
 * the workspace status MOE_ERR_DEVICE_CHECK and that slot is treated as
 * empty. */
moe_status_t moe_route_indices(const int32_t* topk_idx, const float* topk_w,
                               int64_t T, int E, int k,
                               int32_t* counts, int32_t* offsets, int32_t* group_list,
                               int32_t* sorted_indices, int32_t* slot_pos,
                               float* permuted_probs, uint8_t* routing_map,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The same routing as moe_route for callers that cannot allocate device
 * memory: a plugin or runtime that works inside a fixed, pre-reserved memory
 * budget and has no allocator of its own, or code that must not call
 * cudaMalloc because cudaMalloc can synchronise the device.  (The pages have
 * no counterpart: this is a property of the library, not of the method.)
 * The caller still passes every input and output; the scratch space that
 * moe_route takes as a workspace comes instead from a fixed array of
 * MOE_ROUTE_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library keeps until the process exits.
 *  - Problems needing more than that (moe_route_workspace_size(T, E, k) >
 *    MOE_ROUTE_NOALLOC_SCRATCH_BYTES; e.g. T = 16384, E = 256 needs 772 KB,
 *    and at E = 256 the limit is about 87,000 tokens) return
 *    MOE_ERR_UNSUPPORTED before anything runs.
 *  - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *    call.  Its first call on each device looks up the array's device address
 *    (once per device, with that device current); make that first call before
 *    any stream capture.  The address is kept for the life of the process:
 *    after cudaDeviceReset (or anything else that destroys and re-creates the
 *    device's primary context) it is stale, so do not use this entry point
 *    on a device that has been reset.  (moe_device_status caches the address
 *    of the device status word the same way.)
 *  - Every call shares the one array.  Each call writes all the scratch it
 *    reads, so nothing has to be cleared between calls, but calls that
 *    overlap on the GPU (other streams, other host threads) race: serialise
 *    them.
 *  - There is no workspace to pass to moe_workspace_status; a bulk-copy
 *    wait that gives up is recorded in the device status word as for
 *    moe_route (moe_device_status). */
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (1u << 20)

moe_status_t moe_route_noalloc(const float* logits, int64_t T, int E, int k,
                               int32_t* topk_idx, float* topk_w,
                               int32_t* counts, int32_t* offsets, int32_t* group_list,
                               int32_t* sorted_indices, int32_t* slot_pos,
                               float* permuted_probs, uint8_t* routing_map, void* stream);

/* ------------------------------------------ capacity, drop and pad, alignment
 * [MOE-OPS] §18 capacity, the drop_and_pad branch of [DISPATCH] §1.1 and the
 * expert_alignment of the DeepEP dispatch in [COMBINE] §6.
 *
 * moe_expert_capacity (host): ceil(tokens * top_k / num_experts *
 * capacity_factor) in double ([MOE-OPS] §18: 1024*2/8*1.25 -> 320).
 *
 * moe_route_layout: the index outputs of moe_route_indices for a bounded or
 * padded layout of the permuted rows.
 *  - the tokens of expert e, in token order, get ranks 0, 1, ...; with
 *    capacity > 0 an expert keeps ranks < capacity and drops the rest (the
 *    dropped slots' slot_pos is -1: they move no row and add nothing in the
 *    combine; the kept weights are not renormalised)
 *  - counts[e] = kept tokens
 *  - expert e's segment is `capacity` rows if pad (capacity > 0), else
 *    counts[e] rounded up to a multiple of alignment (>= 1)
 *  - offsets [E+1] / group_list [E]: exclusive / inclusive prefix of the
 *    segments
 *  - sorted_indices and permuted_probs have max_rows entries; padding rows
 *    and rows from offsets[E] on hold -1 / 0
 * max_rows: the caller's capacity for rows, at least
 * moe_route_layout_rows(...) (E*capacity when padding, else
 * T*k + E*(alignment-1)); if the layout would still need more, rows past
 * max_rows are not written and the workspace status is
 * MOE_ERR_DEVICE_CHECK.  topk_idx may hold -1 (empty slots); invalid ids are
 * handled as in moe_route_indices.  Workspace: moe_route_workspace_size.
 *
 * moe_fill_pad_rows: zero the padding rows [offsets[e] + counts[e],
 * offsets[e+1]) (clipped to max_rows) of a permuted buffer [max_rows, H], so
 * a grouped GEMM over the padded segments reads zeros there. */
moe_status_t moe_expert_capacity(int64_t tokens, int top_k, int num_experts,
                                 double capacity_factor, int64_t* capacity);

moe_status_t moe_route_layout_rows(int64_t T, int E, int k, int capacity, int pad,
                                   int alignment, int64_t* max_rows);

moe_status_t moe_route_layout(const int32_t* topk_idx, const float* topk_w, int64_t T,
                              int E, int k, int capacity, int pad, int alignment,
                              int64_t max_rows, int32_t* counts, int32_t* offsets,
                              int32_t* group_list, int32_t* sorted_indices,
                              int32_t* slot_pos, float* permuted_probs,
                              void* workspace, size_t workspace_bytes, void* stream);

moe_status_t moe_fill_pad_rows(void* rows, moe_dtype_t dtype, int64_t max_rows, int64_t H,
                               const int32_t* offsets, const int32_t* counts, int E,
                               void* stream);

/* ---------------------------------------------------------------- permute
 * [DISPATCH] §1.1 permuted_input = tokens.index_select(0, sorted_indices),
 * computed token by token: every row x[t] is read once and written to rows
 * slot_pos[t, 0..k-1] of `out` (the dedup form: one read, k writes).
 *   x [T,H] (dtype), slot_pos [T,k] (from moe_route*), out [n_rows,H] (dtype);
 *   n_rows = T*k for the plain layout, max_rows for moe_route_layout.
 * Rows of `out` that no slot names are left untouched.  Entries of slot_pos
 * outside [0, n_rows) are skipped.  Rows that are 16-byte multiples move with
 * bulk copies (one load and one store instruction per row piece); a wait on
 * such a copy that gives up is reported by moe_device_status. */
moe_status_t moe_permute(const void* x, moe_dtype_t dtype, int64_t T, int64_t H, int k,
                         int64_t n_rows, const int32_t* slot_pos, void* out, void* stream);

/* ------------------------------------------------------------ sort_chunks
 * [COMBINE] §2.1 and [MOE-OPS] §11-13: cut `in` [N,H] into C consecutive
 * chunks of split_sizes[c] rows and write chunk sorted_idxs[0],
 * sorted_idxs[1], ... back to back into `out` [N,H].
 *   split_sizes [C] int32 (device), sorted_idxs [C] int32 (device).
 * If the sizes do not add up to N, or sorted_idxs is not a permutation of
 * 0..C-1, nothing is written and the workspace status becomes
 * MOE_ERR_DEVICE_CHECK.  1 <= C <= 65536.  Up to 1024 chunks of rows that
 * are 16-byte multiples take one launch that copies with bulk copies; a
 * bounded wait there that gives up is reported by moe_device_status.
 * Workspace: moe_sort_chunks_workspace_size(C) bytes. */
moe_status_t moe_sort_chunks_workspace_size(int C, size_t* bytes);

moe_status_t moe_sort_chunks(const void* in, moe_dtype_t dtype, int64_t N, int64_t H,
                             const int32_t* split_sizes, const int32_t* sorted_idxs, int C,
                             void* out, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Host helper: chunk orders for an [R source ranks x L local experts] split
 * matrix M (row-major, M.ravel() are the rank-major splits).
 *   inverse = 0: rank-major -> expert-major, idxs[l*R + r] = r*L + l
 *   inverse = 1: expert-major -> rank-major (use the splits M.T.ravel()),
 *                idxs[r*L + l] = l*R + r.
 * The two orders are mutually inverse ([COMBINE] §2.1).  idxs is HOST memory
 * of R*L ints. */
moe_status_t moe_chunk_idxs(int R, int L, int inverse, int32_t* idxs);

/* ---------------------------------------------------------------- combine
 * [COMBINE] §1 and [MOE-OPS] §16:
 *   out[t] = sum_{j=0..k-1} topk_w[t,j] * expert_out[slot_pos[t,j]]
 * A deterministic gather-reduce that replaces the scatter-add of [COMBINE]
 * §2.3.  Accumulation is float32 in slot order with a certified rounding
 * test; elements the test cannot certify are recomputed in double in the same
 * order.  The result is the double slot-order sum rounded once to `dtype`.
 * topk_w = NULL gives the plain sum (the unweighted combine, and the backward
 * of moe_permute).  Empty or dropped slots (-1) contribute nothing; a token
 * with no valid slot gets a zero row.
 *   expert_out [n_rows,H] (n_rows = T*k, or max_rows of a padded layout),
 *   slot_pos [T,k], topk_w [T,k] or NULL, out [T,H]. */
moe_status_t moe_combine(const void* expert_out, moe_dtype_t dtype, int64_t T, int64_t H,
                         int k, int64_t n_rows, const int32_t* slot_pos, const float* topk_w,
                         void* out, void* stream);

/* [COMBINE] §4: the combine is linear in expert_out and in the weights, so
 *   grad_expert_out[slot_pos[t,j]] = topk_w[t,j] * grad_out[t]
 *                                    (exact product rounded once to dtype)
 *   grad_probs[t,j] = sum_h grad_out[t,h] * expert_out[slot_pos[t,j],h]
 *                     (float32 with error-free compensated summation)
 * topk_w = NULL means weights of 1.  Empty slots write no row and give
 * grad_probs 0.
 *   grad_out [T,H], expert_out and grad_expert_out [n_rows,H] (dtype);
 *   grad_probs [T,k] float32. */
moe_status_t moe_combine_backward(const void* grad_out, const void* expert_out,
                                  moe_dtype_t dtype, int64_t T, int64_t H, int k, int64_t n_rows,
                                  const int32_t* slot_pos, const float* topk_w,
                                  void* grad_expert_out, float* grad_probs, void* stream);

/* ---------------------------------------------------------- stand-in expert
 * A per-expert elementwise scale on expert-contiguous rows, used as a
 * stand-in for the expert FFN when exercising dispatch and combine:
 *   out[p] = in[p] * scale[e] for offsets[e] <= p < offsets[e+1]
 * (exact product rounded once to dtype).  Rows at or past offsets[E] are
 * untouched.  in, out [n_rows,H]; offsets [E+1] and scale [E] on the device;
 * n_rows bounds the rows the kernel may touch (normally T*k). */
moe_status_t moe_expert_scale(const void* in, moe_dtype_t dtype, int64_t n_rows, int64_t H,
                              int E, const int32_t* offsets, const float* scale, void* out,
                              void* stream);

/* --------------------------------------------------------- grouped SwiGLU
 * [MOE-OPS] §8 (and §7 for the segments): each expert e applies its SwiGLU
 * FFN to its rows [offsets[e], offsets[e+1]) of the permuted activations:
 *   gate_up = x_e @ w_up[e]            [n_e, 2I]  (fp32 accumulation)
 *   hidden  = silu(gate) * up          gate = first I columns, up = last I;
 *                                      stored as bf16
 *   y_e     = hidden @ w_down[e]       [n_e, H]   (fp32 accumulation, bf16 out)
 * on the tcgen05 tensor cores.  Weights are prepacked once (a model-load
 * step, not part of the per-batch path) by moe_grouped_swiglu_pack:
 *   w_up [E,H,2I] bf16  -> w_up_packed [E,2I,H]  (K-major; rows in blocks of
 *                          256 = [128 gate rows | the matching 128 up rows])
 *   w_down [E,I,H] bf16 -> w_down_packed [E,H,I] (K-major)
 * Shapes: H a multiple of 256, I a multiple of 128, E <= 1024, all bf16
 * 16-byte aligned.  offsets [E+1] int32 stays on the device (no host sync):
 * rows past offsets[E] of y are untouched.  x, y [N,H].  Workspace
 * (moe_grouped_swiglu_workspace_size) holds the bf16 hidden [N,I] and the
 * status word (MOE_ERR_TIMEOUT if a bounded tensor-core pipeline wait gave
 * up; read with moe_workspace_status). */
moe_status_t moe_grouped_swiglu_pack(const void* w_up, const void* w_down, int E, int64_t H,
                                     int64_t I, void* w_up_packed, void* w_down_packed,
                                     void* stream);

moe_status_t moe_grouped_swiglu_workspace_size(int64_t N, int E, int64_t H, int64_t I,
                                               size_t* bytes);

moe_status_t moe_grouped_swiglu(const void* x, const void* w_up_packed,
                                const void* w_down_packed, const int32_t* offsets,
                                int64_t N, int E, int64_t H, int64_t I, void* y,
                                void* workspace, size_t workspace_bytes, void* stream);

/* moe_grouped_swiglu_fp8: moe_grouped_swiglu with the activations in FP8
 * dispatch form ([COMBINE] §3: e4m3 rows with per-block scales, as
 * moe_permute_quantize_fp8 leaves them): x_q [N,H] e4m3 codes and scales
 * [N, H/128] float (block = 128).  GMM1 reads the codes and converts each
 * stage in shared memory to bf16(code * scale), the exact product rounded
 * once -- the values moe_dequantize_fp8 would write -- so y and hidden are
 * bit for bit those of moe_grouped_swiglu on moe_dequantize_fp8(x_q,
 * scales), with no dequantized copy in memory.  H a multiple of 512 (the
 * scale rows are read by TMA, 16 bytes at a time; else MOE_ERR_UNSUPPORTED),
 * x_q and scales 16-byte aligned (else MOE_ERR_INVALID_ARG); weights,
 * offsets, y, the other shapes and workspace as moe_grouped_swiglu. */
moe_status_t moe_grouped_swiglu_fp8(const void* x_q, const float* scales,
                                    const void* w_up_packed, const void* w_down_packed,
                                    const int32_t* offsets, int64_t N, int E, int64_t H,
                                    int64_t I, void* y, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* ------------------------------------------- grouped SwiGLU, training path
 * [MOE-OPS] §22 (GMM2 backward -> SwiGLU backward -> GMM1 backward, giving
 * dX, dW1 and dW2, with d_gate and d_up from hidden = silu(gate) * up) and
 * [COMBINE] §4.2 / §5 (the expert backward is an m-grouped dgrad on the
 * critical path plus a k-grouped wgrad that may be deferred).  Shapes and
 * alignment as moe_grouped_swiglu (H a multiple of 256, I of 128, all bf16
 * buffers 16-byte aligned); all buffers are caller-owned device memory.
 * `workspace` here is only the status header: MOE_STATUS_WORKSPACE_BYTES,
 * 256-byte aligned; read with moe_workspace_status (MOE_ERR_TIMEOUT if a
 * bounded tensor-core pipeline wait gave up).
 *
 * moe_grouped_swiglu_save: the forward of moe_grouped_swiglu that keeps what
 * the backward needs: hidden [N,I] (bf16, the GMM2 input) and gate_up [N,2I]
 * (bf16 GMM1 output, gate columns first) in caller buffers.
 *
 * moe_grouped_swiglu_dgrad (m-grouped, per expert segment of offsets):
 *   dh       = dy @ w_down[e]^T                 (fp32 accumulation)
 *   s        = sigmoid(gate), gate / up from the stored gate_up
 *   dgate_up = [dh*up*s*(1 + gate*(1-s)) | dh*gate*s]     -> bf16 [N,2I]
 *   dx       = dgate_up @ w_up[e]^T             -> bf16 [N,H]
 * w_up [E,H,2I] and w_down [E,I,H] in their ORIGINAL layouts (not packed):
 * for these two products they are already K-major.
 *
 * moe_grouped_swiglu_wgrad (k-grouped: sums over each expert's rows):
 *   dw_up[e]   = x_e^T @ dgate_up_e       fp32 [E,H,2I]
 *   dw_down[e] = hidden_e^T @ dy_e        fp32 [E,I,H]
 * Either output may be NULL (not computed).  Experts with no rows get zeros.
 * For all three calls, offsets outside [0, N] or decreasing are clamped into
 * [0, N] (no row outside the buffers is read or written) and reported as
 * MOE_ERR_DEVICE_CHECK in the workspace status.
 * Segments need no alignment; segments that are multiples of 64 rows (an
 * aligned layout, moe_route_layout) skip the in-kernel zeroing of a
 * segment's last partial stage.  With padded or aligned layouts the pad rows
 * of x, dy and dgate_up must be zero (moe_fill_pad_rows; dgrad keeps
 * dgate_up's pad rows zero when gate_up's are, since d_gate and d_up vanish
 * where gate and up do). */
#define MOE_STATUS_WORKSPACE_BYTES 256

moe_status_t moe_grouped_swiglu_save(const void* x, const void* w_up_packed,
                                     const void* w_down_packed, const int32_t* offsets,
                                     int64_t N, int E, int64_t H, int64_t I, void* y,
                                     void* hidden, void* gate_up, void* workspace,
                                     size_t workspace_bytes, void* stream);

moe_status_t moe_grouped_swiglu_dgrad(const void* dy, const void* w_up, const void* w_down,
                                      const int32_t* offsets, const void* gate_up, int64_t N,
                                      int E, int64_t H, int64_t I, void* dgate_up, void* dx,
                                      void* workspace, size_t workspace_bytes, void* stream);

moe_status_t moe_grouped_swiglu_wgrad(const void* x, const void* hidden, const void* dy,
                                      const void* dgate_up, const int32_t* offsets, int64_t N,
                                      int E, int64_t H, int64_t I, float* dw_up, float* dw_down,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ router backward
 * Gradient of the router logits from the gradient of the routing weights.
 * Only the chosen experts' probabilities carry gradient ([COMBINE] §6,
 * backward pseudocode) and w is the softmax over the k chosen logits
 * ([MOE-OPS] §3), so with g = grad_probs (moe_combine_backward's output):
 *   grad_logits[t, topk_idx[t,i]] = w_i * (g_i - sum_j w_j g_j)
 * and 0 for the other experts of the row.  Computed in double (the sum in
 * slot order), rounded once to float.
 * topk_idx int32 [T,k] (-1 = empty slot, skipped), topk_w and grad_probs
 * float [T,k], grad_logits float [T,E] (every element written); all device
 * memory owned by the caller.  1 <= k <= min(E, 32), E <= 1024.  Ids outside
 * [0,E) other than -1, or repeated within a token, are skipped and recorded
 * as MOE_ERR_DEVICE_CHECK in the device status word (moe_device_status). */
moe_status_t moe_route_backward(const int32_t* topk_idx, const float* topk_w,
                                const float* grad_probs, int64_t T, int E, int k,
                                float* grad_logits, void* stream);

/* ------------------------------------------------------------ FP8 dispatch
 * [COMBINE] §3 (the dispatch moves FP8 rows with scales, the combine stays
 * BF16) and the x_scales / num_scales of [DISPATCH]'s DeepEP dispatch.
 * moe_quantize_fp8: per token and per block of `block` consecutive elements
 * (block = 32, 64, 128 or 256; H a multiple of it), scale = amax / 448 (the
 * largest finite e4m3 value; an all-zero block gets scale 1) and
 * x_q = e4m3(x / scale), the float quotient rounded to nearest even e4m3 and
 * saturated to +-448.  x bf16 [T,H]; x_q e4m3 bytes [T,H]; scales float
 * [T, H/block].  Move x_q with moe_permute(dtype MOE_FP8_E4M3) and the
 * scales with moe_permute(dtype MOE_F32, H/block columns) using the same
 * slot_pos.
 * moe_dequantize_fp8: out = bf16(x_q * scale), the exact product rounded
 * once; x_q [N,H], scales [N, H/block], out bf16 [N,H].
 * All buffers are device memory owned by the caller; bf16 pointers 16-byte,
 * e4m3 pointers 8-byte and scales 4-byte aligned, else MOE_ERR_INVALID_ARG.
 * A block size other than 32/64/128/256 is MOE_ERR_UNSUPPORTED. */
moe_status_t moe_quantize_fp8(const void* x, int64_t T, int64_t H, int block, void* x_q,
                              float* scales, void* stream);

moe_status_t moe_dequantize_fp8(const void* x_q, const float* scales, int64_t N, int64_t H,
                                int block, void* out, void* stream);

/* moe_permute_fp8: moe_permute of the e4m3 rows x_q [T,H] and of their scale
 * rows scales [T, H/block] with the same slot_pos, in one launch: each token's
 * scale row travels in the same copy stage as its data row.  out_q
 * [n_rows,H], out_scales [n_rows, H/block]; rows no slot names are left as
 * they were; errors as moe_permute.  Buffers whose rows are not 16-byte
 * multiples or not 16-byte aligned take two moe_permute launches instead. */
moe_status_t moe_permute_fp8(const void* x_q, const float* scales, int64_t T, int64_t H,
                             int block, int k, int64_t n_rows, const int32_t* slot_pos,
                             void* out_q, float* out_scales, void* stream);

/* moe_permute_quantize_fp8: moe_quantize_fp8 then moe_permute_fp8 in one
 * launch, with no token-order e4m3 copy in between: each token's bf16 row
 * x [T,H] is read once, quantized (the same scales and codes as
 * moe_quantize_fp8, bit for bit) and written to every slot row slot_pos
 * [T,k] names: out_q [n_rows,H] e4m3, out_scales [n_rows, H/block] float.
 * Slots outside [0, n_rows) (dropped, -1) are skipped; rows no slot names are
 * left as they were.  Requires x and out_q 16-byte aligned, out_scales 4-byte
 * aligned (else MOE_ERR_INVALID_ARG) and H <= 8192 (else
 * MOE_ERR_UNSUPPORTED: use the two calls); block and H as moe_quantize_fp8;
 * 1 <= k <= 32.  A bounded copy wait that gives up is reported by
 * moe_device_status. */
moe_status_t moe_permute_quantize_fp8(const void* x, int64_t T, int64_t H, int block, int k,
                                      int64_t n_rows, const int32_t* slot_pos, void* out_q,
                                      float* out_scales, void* stream);

/* ------------------------------------------------- workspace status word
 * Waits for `stream`, then reads the status a previous call left in
 * `workspace`: MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_TIMEOUT.  Each call
 * that takes a workspace resets its status word. */
moe_status_t moe_workspace_status(const void* workspace, void* stream);

/* Waits for `stream`, then reads and clears the library's device status word
 * of the current device, which kernels that take no workspace set: the
 * bulk-copy permutes when one of their bounded pipeline waits gives up
 * (MOE_ERR_TIMEOUT), moe_route_backward on an invalid or repeated expert id
 * (MOE_ERR_DEVICE_CHECK); MOE_OK if neither happened since the last read.
 * One word per device, shared by all streams. */
moe_status_t moe_device_status(void* stream);

/* Health check of the failure path that the pipelined kernels (the grouped
 * GEMMs and the bulk-copy permutes) rely on; no counterpart on the pages.
 * One block waits on an mbarrier that nothing completes, through the same
 * bounded poll loop those kernels use but limited to `polls` polls
 * (1 <= polls <= 2^20; each poll of mbarrier.try_wait suspends the thread for
 * at most a short hardware-defined time), gives up, records MOE_ERR_TIMEOUT
 * in the workspace status word (detail = polls) and returns normally, so the
 * context stays usable.  Read the outcome with moe_workspace_status().
 *   workspace: device memory, 256-byte aligned, >= 256 bytes (only its
 *   status header is written).
 * Returns MOE_ERR_WORKSPACE or MOE_ERR_INVALID_ARG before any launch on bad
 * arguments, MOE_ERR_CUDA if the launch fails. */
moe_status_t moe_selftest_timeout(void* workspace, size_t workspace_bytes, uint32_t polls,
                                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
