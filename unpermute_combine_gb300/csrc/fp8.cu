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

// two e4m3 bytes (low byte first) -> two floats (exact)
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t v, float& a, float& b) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(v)));
    a = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
    b = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
}

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
