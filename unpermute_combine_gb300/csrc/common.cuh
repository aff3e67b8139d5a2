// common.cuh -- helpers shared by the libmoe CUDA sources (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ host side

constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 1024;
constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// NVTX range around one C-ABI call (named after the entry point), so a
// profiler's timeline shows which library call launched which kernels.
// Without a tool attached a push/pop is a check of a null function pointer.
struct NvtxScope {
    explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope&) = delete;
    NvtxScope& operator=(const NvtxScope&) = delete;
};
#define MOE_TRACE(name) ::moe::NvtxScope moe_trace_scope_(name)

inline size_t elem_size(moe_dtype_t d) { return d == MOE_F32 ? 4 : d == MOE_BF16 ? 2 : 1; }

// dtypes the arithmetic ops take
inline bool dtype_ok(int d) { return d == MOE_F32 || d == MOE_BF16; }

// dtypes the row-movement ops take (rows are moved as bytes)
inline bool dtype_ok_move(int d) { return d == MOE_F32 || d == MOE_BF16 || d == MOE_FP8_E4M3; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Number of SMs of the current device (cached per device id).
int sm_count();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device (once per device, kernel and size; safe from several host threads).
bool opt_in_smem(const void* kernel, int bytes);

// Launch-error check after a kernel launch.
inline moe_status_t launch_status() {
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Workspace header: the first 256 bytes of every workspace.
struct WsHeader {
    uint32_t status;      // moe_status_t of the last call that used the workspace
    uint32_t detail;      // call-specific detail (first offending index, ...)
    uint32_t reserved[62];
};
static_assert(sizeof(WsHeader) == kWsAlign, "header is one alignment unit");

// --------------------------------------------------------------- device side

// bf16 <-> f32 on packed pairs (bit manipulation; exact).
__device__ __forceinline__ float bf16lo_to_f32(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Round two floats to bf16 (nearest even) and pack: low half = a, high = b.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float a) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(a));
}

// double -> bf16, one rounding to nearest even, via round-to-odd: truncate to
// float (24 significant bits) and set the last bit if anything was dropped;
// rounding that float to bf16 (8 bits) is then the correct rounding of the
// double (Boldo & Melquiond, "Emulation of FMA and correctly rounded sums:
// proved algorithms using rounding to odd", 2008).
__device__ __forceinline__ uint16_t f64_to_bf16_rn(double v) {
    float t;
    asm("cvt.rz.f32.f64 %0, %1;" : "=f"(t) : "d"(v));
    uint32_t u = __float_as_uint(t);
    if ((double)t != v && (u & 0x7F800000u) != 0x7F800000u) u |= 1u;
    if (v != v) return 0x7FC0u;
    return f32_to_bf16_rn(__uint_as_float(u));
}

__device__ __forceinline__ float f64_to_f32_rn(double v) { return __double2float_rn(v); }

// Two e4m3 codes (low byte first) -> their exact float values
// (cvt.rn.f16x2.e4m3x2 is exact: every e4m3 value is an f16 value).
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t v, float& a, float& b) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(v)));
    a = __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
    b = __half2float(__ushort_as_half(uint16_t(h2 >> 16)));
}

// bf16 of the exact product a*b.  p = fl(a*b) is within half a float ulp of
// it, so p rounds like the exact product unless p sits exactly on a bf16
// midpoint; then the sign of the product's error e = fma(a,b,-p) breaks the
// tie (Dekker/Knuth error-free product).  The bf16 bits come back in the low
// half of a 32-bit word (callers pack pairs of them).
__device__ __forceinline__ uint32_t mul_bf16_rn(float a, float b) {
    const float p = __fmul_rn(a, b);
    const uint32_t u = __float_as_uint(p);
    if ((u & 0xFFFFu) == 0x8000u) {
        const float e = __fmaf_rn(a, b, -p);
        if (e != 0.0f) {
            const bool same = ((__float_as_uint(e) ^ u) & 0x80000000u) == 0;
            return (same ? u + 0x8000u : u - 0x8000u) >> 16;
        }
    }
    return f32_to_bf16_rn(p);
}

// Programmatic dependent launch: the kernel may start while its predecessor
// in the stream is finishing; it must call wait_for_predecessor() before it
// touches anything the predecessor writes (or reads what it may overwrite).
__device__ __forceinline__ void wait_for_predecessor() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Streaming 16-byte global accesses.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

}  // namespace moe
