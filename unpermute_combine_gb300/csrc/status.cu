// status.cu -- status strings, ABI version, workspace status read-back, the
// per-device SM count used to size persistent grids, and the one-time
// dynamic shared-memory opt-in of the kernels that need more than 48 KB.
#include <mutex>
#include <map>

#include "pipeline.cuh"

// Status word of kernels that take no workspace (set to MOE_ERR_TIMEOUT by a
// bounded wait that gave up; read and cleared by moe_device_status).
static __device__ uint32_t g_device_status;

namespace moe {

uint32_t* device_status_word() {
    static std::mutex m;
    static uint32_t* cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(m);
    if (!cached[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<uint32_t*>(p);
    }
    return cached[dev];
}

bool opt_in_smem(const void* kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    static std::mutex m;
    // the largest limit set so far per (device, kernel): the attribute is
    // only ever raised, so a call with a smaller row size can never lower it
    // under a size an earlier call still launches with
    static std::map<std::pair<int, const void*>, int> limit;
    std::lock_guard<std::mutex> lock(m);
    const auto key = std::make_pair(dev, kernel);
    const auto it = limit.find(key);
    if (it != limit.end() && it->second >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    limit[key] = bytes;
    return true;
}

int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

namespace {

// One block waits on an mbarrier that nothing completes, through the same
// bounded poll loop as the pipelined kernels, gives up after `polls` polls
// and records the timeout in the workspace header.  Nothing is in flight on
// the barrier, so the block simply returns.
__global__ void timeout_selftest_kernel(WsHeader* header, uint32_t polls) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_addr(&bar), 1);
    mbar_fence_init();
    const bool done = mbar_wait_bounded(smem_addr(&bar), 0, polls);
    header->status = done ? MOE_OK : MOE_ERR_TIMEOUT;
    header->detail = done ? 0u : polls;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_selftest_timeout(void* workspace, size_t workspace_bytes,
                                             uint32_t polls, void* stream) {
    MOE_TRACE(__func__);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (moe::kWsAlign - 1)) ||
        workspace_bytes < moe::kWsAlign)
        return MOE_ERR_WORKSPACE;
    if (polls < 1 || polls > moe::kSpinLimit) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    moe::timeout_selftest_kernel<<<1, 32, 0, s>>>(static_cast<moe::WsHeader*>(workspace), polls);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" const char* moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    }
    return "MOE_ERR_UNKNOWN";
}

extern "C" int moe_abi_version(void) { return 2; }

extern "C" moe_status_t moe_workspace_status(const void* workspace, void* stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (moe::kWsAlign - 1)))
        return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    switch (word) {
        case MOE_OK:
        case MOE_ERR_DEVICE_CHECK:
        case MOE_ERR_TIMEOUT: return static_cast<moe_status_t>(word);
    }
    return MOE_ERR_DEVICE_CHECK;
}

extern "C" moe_status_t moe_device_status(void* stream) {
    uint32_t* word = moe::device_status_word();
    if (!word) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(word, 0, sizeof v, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (v == 0) return MOE_OK;
    return v == uint32_t(MOE_ERR_DEVICE_CHECK) ? MOE_ERR_DEVICE_CHECK : MOE_ERR_TIMEOUT;
}
