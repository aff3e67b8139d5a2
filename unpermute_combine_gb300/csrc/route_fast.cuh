// route_fast.cuh -- the top-k route for up to 256 experts (route_fast.cu),
// called by moe_route / moe_route_grouped in route.cu.
#pragma once

#include "common.cuh"

namespace moe {

// Largest expert count the route_fast kernels take.
constexpr int kFastMaxExperts = 256;

// Can route_fast take this problem?  (E <= 256; for group-limited routing,
// each lane's experts must lie in one group and a group must span a
// power-of-two number of lanes.)
bool fast_route_supported(int E, int n_groups);

// Histogram scratch route_fast needs after the 256-byte workspace header.
size_t fast_hist_bytes(int64_t T, int E);

// Top-k + softmax, counts, offsets, group_list, sorted_indices, slot_pos and
// permuted_probs from fp32 logits [T, E] (n_groups = 0: plain top-k).
// `scratch` points at fast_hist_bytes(T, E) bytes of workspace past `header`.
moe_status_t fast_route(const float* logits, int64_t T, int E, int k, int n_groups,
                        int topk_groups, int32_t* topk_idx, float* topk_w, int32_t* counts,
                        int32_t* offsets, int32_t* group_list, int32_t* sorted_indices,
                        int32_t* slot_pos, float* permuted_probs, uint8_t* routing_map,
                        WsHeader* header, int32_t* scratch, cudaStream_t stream);

}  // namespace moe
