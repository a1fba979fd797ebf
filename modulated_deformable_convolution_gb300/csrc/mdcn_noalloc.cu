// Allocation-free forward: mdcn_forward with its workspace taken from a
// fixed device array that lives in this library, for callers that cannot
// allocate device memory on their execution path. Examples: a deployment that
// reserves all device memory at start-up and forbids allocation while
// serving; a plugin or runtime whose execute step must not call cudaMalloc;
// plain C code that has no device allocator of its own to hand out scratch.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "mdcn.h"

namespace {

// Largest workspace this entry point can serve (mdcn_workspace_size of the
// call must not exceed it).
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};  // set once per device, on success only

// Device address of the array on the current device. The device is checked
// first (compute capability 10.3, the only architecture the library is built
// for), so a call on another GPU gets MDCN_ERR_ARCH, as mdcn_forward returns.
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up with cudaGetSymbolAddress, once per device with that
// device current, and cached; a failed look-up is not cached and is retried
// by the next call.
mdcn_status scratch_on_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MDCN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MDCN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MDCN_ERR_CUDA;
        if (major != 10 || minor != 3) return MDCN_ERR_ARCH;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MDCN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MDCN_OK;
}

}  // namespace

extern "C" mdcn_status mdcn_forward_noalloc(mdcn_handle handle, const void* x, const void* offset, const void* mask,
                                            const void* weight, const void* bias_or_null, void* out,
                                            const mdcn_dims* dims, mdcn_dtype dtype, void* stream) {
    size_t need = 0;
    mdcn_status s = mdcn_workspace_size(handle, dims, dtype, &need);
    if (s != MDCN_OK) return s;
    if (need > kNoAllocScratchBytes) return MDCN_ERR_WORKSPACE;
    void* scratch = nullptr;
    s = scratch_on_current_device(&scratch);
    if (s != MDCN_OK) return s;
    // Same kernels, same validation and same results as mdcn_forward; the
    // first of them clears the status word, and every other byte the forward
    // reads from scratch is written earlier in the same call.
    return mdcn_forward(handle, x, offset, mask, weight, bias_or_null, out, scratch, kNoAllocScratchBytes, dims, dtype,
                        stream);
}

// The status word of the fixed array on the current device: what the last
// mdcn_forward_noalloc on this device left there, read and cleared like
// mdcn_query_status does for a caller's workspace.
extern "C" mdcn_status mdcn_noalloc_query_status(void* stream, uint32_t* device_bits) {
    void* scratch = nullptr;
    const mdcn_status s = scratch_on_current_device(&scratch);
    if (s != MDCN_OK) return s;
    return mdcn_query_status(scratch, stream, device_bits);
}
