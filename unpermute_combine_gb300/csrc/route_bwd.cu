// route_bwd.cu -- moe_route_backward: gradient of the router logits.
//
// Only the chosen experts' probabilities carry gradient ("03 · Combine 与
// forward / backward 对称性" §6, backward pseudocode), and the probabilities
// are a softmax over the k chosen logits ("从零理解 MoE 算子" §3).  With
// g = dL/dw (the grad_probs of the combine backward), the softmax Jacobian
// dw_j/ds_i = w_j (delta_ij - w_i) gives, per token,
//   grad_logits[t, topk_idx[t,i]] = w_i * (g_i - sum_j w_j g_j)
// and zero for the other E - k experts.
//
// Arithmetic: double, the sum over the valid slots in slot order, then the
// difference and the product, one rounding to float -- the products of two
// floats are exact in double, so the result does not depend on contraction.
//
// Layout of the work: a warp owns 32 consecutive tokens, one per lane, so
// each fp64 instruction serves 32 tokens (FP64 issue is scarce on this part).
// The warp first zero-fills the 32 rows it owns -- one contiguous run of
// 32*E floats, written with coalesced vector stores -- then, after a
// __syncwarp (which orders the warp's memory accesses), each lane writes its
// token's k values.  Ids outside [0, E), other than the empty id -1, and ids
// repeated within a token are skipped and recorded as MOE_ERR_DEVICE_CHECK in
// the library's device status word.
#include "common.cuh"
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int kBwdThreads = 64;
constexpr int kBwdWarps = kBwdThreads / 32;

__global__ void __launch_bounds__(kBwdThreads)
route_backward_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                      const float* __restrict__ grad_probs, int64_t T, int E, int k,
                      float* __restrict__ grad_logits, bool vec, uint32_t* __restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = int64_t(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5);
    const int64_t t0 = warp * 32;
    if (t0 >= T) return;
    const int64_t t = t0 + lane;
    const bool active = t < T;
    const int64_t base = t * k;

    // pass 1: validity and the slot-order sum of w_j g_j
    double dot = 0.0;
    bool bad = false;
    if (active) {
        for (int j = 0; j < k; ++j) {
            const int32_t id = topk_idx[base + j];
            if (id < 0 || id >= E) {
                bad |= id != -1;
                continue;
            }
            for (int i = 0; i < j; ++i) bad |= topk_idx[base + i] == id;
            dot = __dadd_rn(dot, __dmul_rn(double(topk_w[base + j]), double(grad_probs[base + j])));
        }
    }

    // zero-fill rows [t0, t0 + 32) (or up to T)
    const int64_t rows = min64(int64_t(32), T - t0);
    float* row0 = grad_logits + t0 * E;
    if (vec) {
        float4* v = reinterpret_cast<float4*>(row0);
        const int64_t n = rows * E / 4;
        for (int64_t i = lane; i < n; i += 32) v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        const int64_t n = rows * E;
        for (int64_t i = lane; i < n; i += 32) row0[i] = 0.0f;
    }
    __syncwarp();

    // pass 2: each lane's k values (a repeated id keeps its first slot)
    if (active) {
        for (int j = 0; j < k; ++j) {
            const int32_t id = topk_idx[base + j];
            if (id < 0 || id >= E) continue;
            bool seen = false;
            for (int i = 0; i < j; ++i) seen |= topk_idx[base + i] == id;
            if (seen) continue;
            const double d = __dsub_rn(double(grad_probs[base + j]), dot);
            grad_logits[t * E + id] = __double2float_rn(__dmul_rn(double(topk_w[base + j]), d));
        }
    }
    if (bad && status) atomicExch(status, uint32_t(MOE_ERR_DEVICE_CHECK));
}

// k <= KMAX: the token's k (id, w, g) are loaded into registers before the
// zero-fill, so their latency overlaps the fill's stores; same arithmetic.
template <int KMAX>
__global__ void __launch_bounds__(kBwdThreads)
route_backward_regs_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                           const float* __restrict__ grad_probs, int64_t T, int E, int k,
                           float* __restrict__ grad_logits, bool vec,
                           uint32_t* __restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = int64_t(blockIdx.x) * kBwdWarps + (threadIdx.x >> 5);
    const int64_t t0 = warp * 32;
    if (t0 >= T) return;
    const int64_t t = t0 + lane;
    const bool active = t < T;
    const int64_t base = t * k;
    int32_t id[KMAX];
    float w[KMAX], g[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const bool on = active && j < k;
        id[j] = on ? __ldg(topk_idx + base + j) : -1;
        w[j] = on ? __ldg(topk_w + base + j) : 0.0f;
        g[j] = on ? __ldg(grad_probs + base + j) : 0.0f;
    }

    const int64_t rows = min64(int64_t(32), T - t0);
    float* row0 = grad_logits + t0 * E;
    if (vec) {
        float4* v = reinterpret_cast<float4*>(row0);
        const int64_t n = rows * E / 4;
        for (int64_t i = lane; i < n; i += 32) v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        const int64_t n = rows * E;
        for (int64_t i = lane; i < n; i += 32) row0[i] = 0.0f;
    }

    bool bad = false;
    bool keep[KMAX];
    double dot = 0.0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        const bool valid = id[j] >= 0 && id[j] < E;
        bad |= !valid && id[j] != -1;
        bool seen = false;
#pragma unroll
        for (int i = 0; i < j; ++i) seen |= valid && id[i] == id[j];
        bad |= seen;
        keep[j] = valid && !seen;
        if (valid) dot = __dadd_rn(dot, __dmul_rn(double(w[j]), double(g[j])));
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
        if (keep[j])
            grad_logits[t * E + id[j]] =
                __double2float_rn(__dmul_rn(double(w[j]), __dsub_rn(double(g[j]), dot)));
    if (bad && status) atomicExch(status, uint32_t(MOE_ERR_DEVICE_CHECK));
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_backward(const int32_t* topk_idx, const float* topk_w,
                                           const float* grad_probs, int64_t T, int E, int k,
                                           float* grad_logits, void* stream) {
    MOE_TRACE(__func__);
    if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > kMaxTopK || T * int64_t(E) >= (int64_t(1) << 40))
        return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!topk_idx || !topk_w || !grad_probs || !grad_logits) return MOE_ERR_INVALID_ARG;
    const bool vec = E % 4 == 0 && aligned16(grad_logits);
    const int64_t warps = (T + 31) / 32;
    const int64_t blocks = (warps + kBwdWarps - 1) / kBwdWarps;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (k <= 8)
        route_backward_regs_kernel<8><<<unsigned(blocks), kBwdThreads, 0, s>>>(
            topk_idx, topk_w, grad_probs, T, E, k, grad_logits, vec, device_status_word());
    else
        route_backward_kernel<<<unsigned(blocks), kBwdThreads, 0, s>>>(
            topk_idx, topk_w, grad_probs, T, E, k, grad_logits, vec, device_status_word());
    return launch_status();
}
