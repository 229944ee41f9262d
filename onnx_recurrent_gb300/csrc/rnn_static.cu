// Fixed device scratch for rnn_run_static_scratch(), the entry point for
// callers that cannot allocate device memory during a run.
//
// The scratch is one file-scope __device__ array: every GPU on which the
// library is loaded holds kStaticScratchBytes of it until the process exits.
// In host code `g_static_scratch` names a host-side stand-in, not device
// memory, so its device address is looked up here with cudaGetSymbolAddress,
// once per device with that device current, and cached; that address is what
// the kernels receive.  The first call on a device performs this look-up, so
// it should come before any stream capture.  The cache lives as long as the
// process: after cudaDeviceReset the module is loaded again in a new context
// and the cached address would be stale, so the entry point is not for use on
// a device that has been reset.
#include <mutex>

#include "rnn_internal.h"

namespace rnngb {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;   // 32 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

cudaError_t static_scratch(void** ptr, size_t* bytes)
{
    static std::mutex mu;
    static void* cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        cache[dev] = p;
    }
    *ptr = cache[dev];
    *bytes = kStaticScratchBytes;
    return cudaSuccess;
}

}  // namespace rnngb
