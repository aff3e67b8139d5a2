// status.cu -- status strings, ABI version, workspace status read-back, and
// the per-device SM count used to size persistent grids.
#include "common.cuh"

namespace moe {

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

}  // namespace moe

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

extern "C" int moe_abi_version(void) { return 1; }

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
