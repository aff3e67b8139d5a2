// fp8.cu -- moe_quantize_fp8 / moe_dequantize_fp8.
//
// FP8 dispatch ("03 · Combine 与 forward / backward 对称性" §3: the dispatch
// moves FP8 rows with scales and the combine stays BF16; "token dispatcher +
// fuse_a2a" names x_scales / num_scales): per token and per block of `block`
// elements, scale = amax / 448 (the largest finite e4m3 value; an all-zero
// block gets scale 1) and q = e4m3(x / scale), rounded to nearest even and
// saturated.  The quantized rows and the [T, H/block] scale rows then move
// through moe_permute / moe_sort_chunks like any other rows (FP8 halves the
// permute's write bytes).  Dequantization is the exact product q * scale
// rounded once to bf16.
//
// The [rows, H] tensor is a flat run of 16-byte vectors of 8 bf16 (8 e4m3
// bytes on the quantized side), and every block is G = block/8 consecutive
// vectors, so a block never straddles rows and lane groups of G lanes own
// whole blocks.  A lane keeps several vectors in flight; the block amax is a
// max over the group (xor shuffles) of the magnitude bits, which order like
// the magnitudes for non-negative floats.  The quotient is IEEE division, the
// encoding cvt.rn.satfinite.e4m3x2.f32 (and cvt.rn.f16x2.e4m3x2 back).
#include <cuda_fp16.h>

#include "common.cuh"
#include "pipeline.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kUnrollQ = 4;    // 16-byte bf16 vectors in flight per lane (quantize)
constexpr int kUnrollD = 8;    // 8-byte e4m3 vectors in flight per lane (dequantize)

// two floats -> two e4m3 bytes (low byte = a, high byte = b)
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// four floats -> four e4m3 bytes of f / s
__device__ __forceinline__ uint32_t q4(const float* f, float s) {
    return e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
           (e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
}

template <int G>   // lanes per block: block = 8 * G elements
__global__ void __launch_bounds__(kThreads)
quantize_fp8_kernel(const uint4* __restrict__ x, int64_t nvec, uint2* __restrict__ q,
                    float* __restrict__ scales) {
    static_assert(G == 4 || G == 8 || G == 16 || G == 32, "block of 32..256 elements");
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (kThreads / 32);
    for (int64_t base = (int64_t(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5)) * 32 * kUnrollQ;
         base < nvec; base += warps * 32 * kUnrollQ) {
        uint4 xv[kUnrollQ];
#pragma unroll
        for (int u = 0; u < kUnrollQ; ++u) {
            const int64_t v = base + u * 32 + lane;
            xv[u] = v < nvec ? ld_nc_v4(x + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnrollQ; ++u) {
            const int64_t v = base + u * 32 + lane;
            const uint32_t w[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
            float f[8];
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                m = max(m, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
            }
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1)
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            const float amax = __uint_as_float(m);
            const float s = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
            if (v < nvec) {
                q[v] = make_uint2(q4(f, s), q4(f + 4, s));
                if ((lane & (G - 1)) == 0) scales[v / G] = s;
            }
        }
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads)
dequantize_fp8_kernel(const uint2* __restrict__ q, const float* __restrict__ scales,
                      int64_t nvec, uint4* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (kThreads / 32);
    for (int64_t base = (int64_t(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5)) * 32 * kUnrollD;
         base < nvec; base += warps * 32 * kUnrollD) {
        uint2 qv[kUnrollD];
        float sv[kUnrollD];
#pragma unroll
        for (int u = 0; u < kUnrollD; ++u) {
            const int64_t v = base + u * 32 + lane;
            qv[u] = v < nvec ? __ldcs(q + v) : make_uint2(0, 0);
            sv[u] = v < nvec ? __ldg(scales + v / G) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < kUnrollD; ++u) {
            const int64_t v = base + u * 32 + lane;
            const uint32_t bytes[2] = {qv[u].x, qv[u].y};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float a, b;
                e4m3x2_to_f32(bytes[i >> 1] >> (16 * (i & 1)), a, b);
                o[i] = mul_bf16_rn(a, sv[u]) | (mul_bf16_rn(b, sv[u]) << 16);
            }
            if (v < nvec) out[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// ------------------------------------------- fused quantize + permute
// One CTA of 8 warps per token at a time.  Thread 0 bulk-loads the token's
// bf16 row into a ring stage; all threads quantize it into the stage's e4m3
// area with the arithmetic of quantize_fp8_kernel (16-byte vectors, lane
// groups of G owning a block, IEEE quotient, cvt.rn.satfinite); the scale of
// each block goes straight to the token's slot rows of out_scales, and lanes
// 0..k-1 of warp 0 each bulk-store the e4m3 row to their slot row.  The
// input area is refilled as soon as every thread has read it; the output
// area is written again only after the stores from it have read it.  So the
// row is read from HBM once and written k times in e4m3, with no
// token-order e4m3 copy in between.  (Measured at T=16384, H=7168, k=8:
// 8 warps and 3 stages 193 us; 4 warps 235 us, 16 warps 208 us; 2 stages
// 210-212 us, 4 stages 316 us.)
constexpr int kPQThreads = 256;
constexpr int kPQStages = 3;
constexpr int kPQRowMax = 16384;              // bf16 bytes of a row in one stage (H <= 8192)

template <int G>
__global__ void __launch_bounds__(kPQThreads)
permute_quantize_fp8_kernel(const uint8_t* __restrict__ x, int64_t T, int H, int k,
                            int64_t n_rows, const int32_t* __restrict__ slot_pos,
                            uint8_t* __restrict__ out_q, float* __restrict__ out_scales,
                            uint32_t* __restrict__ status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[kPQStages];
    __shared__ int32_t s_slot[2][kMaxTopK];
    __shared__ int s_failed;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t in_bytes = uint32_t(H) * 2u, stage_bytes = uint32_t(H) * 3u;
    const int nvec = H / 8;                    // 16-byte bf16 vectors of a row
    const int nb = H / (8 * G);                // scale blocks of a row
    const int64_t first = blockIdx.x;
    const int64_t my = first < T ? (T - first + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t smem0 = smem_addr(smem);
    if (tid == 0) {
        for (int st = 0; st < kPQStages; ++st) mbar_init(smem_addr(&full_bar[st]), 1);
        mbar_fence_init();
        s_failed = 0;
    }
    __syncthreads();
    auto issue_load = [&](int64_t q) {
        const int64_t t = first + q * int64_t(gridDim.x);
        const int st = int(q % kPQStages);
        const uint32_t fb = smem_addr(&full_bar[st]);
        mbar_expect_tx(fb, in_bytes);
        bulk_load(smem0 + uint32_t(st) * stage_bytes, x + t * int64_t(in_bytes), in_bytes, fb);
    };
    if (tid == 0)
        for (int64_t q = 0; q < my && q < kPQStages; ++q) issue_load(q);

    int64_t q_fail = 0;
    for (int64_t q = 0; q < my; ++q) {
        const int64_t t = first + q * int64_t(gridDim.x);
        const int st = int(q % kPQStages);
        const uint32_t ph = uint32_t(q / kPQStages) & 1u;
        int32_t* slots = s_slot[q & 1];
        int32_t p = -1;
        if (warp == 0 && lane < k) {
            // this lane's store of token q - kPQStages (same stage) has read it
            bulk_wait_read<kPQStages - 1>();
            p = slot_pos[t * k + lane];
            if (p < 0 || p >= n_rows) p = -1;
            slots[lane] = p;
        }
        if (!mbar_wait(smem_addr(&full_bar[st]), ph)) s_failed = 1;
        __syncthreads();
        if (s_failed) {
            q_fail = q;
            break;
        }

        const uint8_t* in = smem + uint32_t(st) * stage_bytes;
        uint8_t* outq = smem + uint32_t(st) * stage_bytes + in_bytes;
        // warp-uniform trip count; a G-group is wholly inside or outside the row
        for (int v0 = warp * 32; v0 < nvec; v0 += kPQThreads) {
            const int v = v0 + lane;
            const bool live = v < nvec;
            const uint4 xv = live ? *reinterpret_cast<const uint4*>(in + v * 16)
                                  : make_uint4(0, 0, 0, 0);
            const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
            float f[8];
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                m = max(m, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
            }
#pragma unroll
            for (int off = G / 2; off > 0; off >>= 1)
                m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            const float amax = __uint_as_float(m);
            const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
            if (live) {
                *reinterpret_cast<uint2*>(outq + v * 8) = make_uint2(q4(f, sc), q4(f + 4, sc));
                if ((lane & (G - 1)) == 0) {
                    const int blk = v / G;
                    for (int j = 0; j < k; ++j) {
                        const int32_t pj = slots[j];
                        if (pj >= 0) out_scales[int64_t(pj) * nb + blk] = sc;
                    }
                }
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (warp == 0 && lane < k) {
            if (p >= 0) bulk_store(out_q + int64_t(p) * H, smem_addr(outq), uint32_t(H));
            bulk_commit();
        }
        if (tid == 0 && q + kPQStages < my) issue_load(q + kPQStages);
    }
    if (warp == 0 && lane < k) bulk_wait_all();
    if (tid == 0 && s_failed) {
        // loads issued but never consumed (items q_fail .. q_fail + stages - 1)
        // may still be landing in this CTA's shared memory: wait for each
        // (bounded) before the CTA exits and the memory is reused
        for (int64_t i = q_fail; i < my && i < q_fail + kPQStages; ++i)
            mbar_wait(smem_addr(&full_bar[i % kPQStages]), uint32_t(i / kPQStages) & 1u);
        if (status) atomicExch(status, uint32_t(MOE_ERR_TIMEOUT));
    }
}

int grid_pq(const void* kernel, size_t smem, int64_t T) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kPQThreads, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    return int(T < cap ? (T > 0 ? T : 1) : cap);
}

int grid_for(const void* kernel, int64_t nvec, int unroll) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (per_sm < 1) per_sm = 1;
    const int64_t per_block = int64_t(kThreads) * unroll;
    const int64_t want = (nvec + per_block - 1) / per_block;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    return int(want < cap ? (want > 0 ? want : 1) : cap);
}

moe_status_t check_block(int64_t rows, int64_t H, int block) {
    if (rows < 0 || H < 0) return MOE_ERR_INVALID_ARG;
    if (block != 32 && block != 64 && block != 128 && block != 256) return MOE_ERR_UNSUPPORTED;
    if (H % block != 0) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_quantize_fp8(const void* x, int64_t T, int64_t H, int block,
                                         void* x_q, float* scales, void* stream) {
    MOE_TRACE(__func__);
    const moe_status_t st = check_block(T, H, block);
    if (st != MOE_OK) return st;
    if (T == 0 || H == 0) return MOE_OK;
    if (!x || !x_q || !scales) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(x_q) & 7) ||
        (reinterpret_cast<uintptr_t>(scales) & 3))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t nvec = T * H / 8;
    const uint4* xv = static_cast<const uint4*>(x);
    uint2* qv = static_cast<uint2*>(x_q);
#define MOE_QUANT(G_)                                                                          \
    quantize_fp8_kernel<G_><<<grid_for((const void*)quantize_fp8_kernel<G_>, nvec, kUnrollQ), kThreads, 0, \
                              s>>>(xv, nvec, qv, scales)
    switch (block) {
        case 32: MOE_QUANT(4); break;
        case 64: MOE_QUANT(8); break;
        case 128: MOE_QUANT(16); break;
        default: MOE_QUANT(32); break;
    }
#undef MOE_QUANT
    return launch_status();
}

extern "C" moe_status_t moe_dequantize_fp8(const void* x_q, const float* scales, int64_t N,
                                           int64_t H, int block, void* out, void* stream) {
    MOE_TRACE(__func__);
    const moe_status_t st = check_block(N, H, block);
    if (st != MOE_OK) return st;
    if (N == 0 || H == 0) return MOE_OK;
    if (!x_q || !scales || !out) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x_q) & 7) || (reinterpret_cast<uintptr_t>(scales) & 3) ||
        !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t nvec = N * H / 8;
    const uint2* qv = static_cast<const uint2*>(x_q);
    uint4* ov = static_cast<uint4*>(out);
#define MOE_DEQUANT(G_)                                                                  \
    dequantize_fp8_kernel<G_><<<grid_for((const void*)dequantize_fp8_kernel<G_>, nvec, kUnrollD), \
                                kThreads, 0, s>>>(qv, scales, nvec, ov)
    switch (block) {
        case 32: MOE_DEQUANT(4); break;
        case 64: MOE_DEQUANT(8); break;
        case 128: MOE_DEQUANT(16); break;
        default: MOE_DEQUANT(32); break;
    }
#undef MOE_DEQUANT
    return launch_status();
}

extern "C" moe_status_t moe_permute_quantize_fp8(const void* x, int64_t T, int64_t H, int block,
                                                 int k, int64_t n_rows,
                                                 const int32_t* slot_pos, void* out_q,
                                                 float* out_scales, void* stream) {
    MOE_TRACE(__func__);
    const moe_status_t st = check_block(T, H, block);
    if (st != MOE_OK) return st;
    if (k < 1 || k > kMaxTopK || n_rows < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0 || H == 0) return MOE_OK;
    if (H * 2 > kPQRowMax) return MOE_ERR_UNSUPPORTED;
    if (!x || !slot_pos || !out_q || !out_scales) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out_q) || (reinterpret_cast<uintptr_t>(out_scales) & 3))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t smem = size_t(kPQStages) * size_t(H) * 3;
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    uint8_t* qb = static_cast<uint8_t*>(out_q);
#define MOE_PQ(G_)                                                                              \
    do {                                                                                        \
        const void* kern = (const void*)permute_quantize_fp8_kernel<G_>;                        \
        if (!opt_in_smem(kern, int(smem))) return MOE_ERR_CUDA;                                 \
        permute_quantize_fp8_kernel<G_><<<grid_pq(kern, smem, T), kPQThreads, smem, s>>>(        \
            xb, T, int(H), k, n_rows, slot_pos, qb, out_scales, device_status_word());         \
    } while (0)
    switch (block) {
        case 32: MOE_PQ(4); break;
        case 64: MOE_PQ(8); break;
        case 128: MOE_PQ(16); break;
        default: MOE_PQ(32); break;
    }
#undef MOE_PQ
    return launch_status();
}
