// attend_noalloc.cu -- kvc_decode_attend_noalloc: decode attention whose split
// scratch lives in a fixed array owned by the library instead of a caller
// workspace.
//
// Who needs it: callers that must not allocate device memory on their decode
// path.  Examples are a serving engine that hands all free device memory to
// its KV-cache pool at start-up and so has nothing left to cudaMalloc from,
// and a plugin host that offers no allocator and forbids cudaMalloc /
// cudaFree in its enqueue callback because those calls synchronise the
// device.  Such a caller still passes its own inputs and outputs; only the
// scratch (the per-split partial results that the combine step merges) comes
// from here.
//
// The scratch is one file-scope device array of KVC_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Its
// host-side name is only a stand-in for the symbol, so the host looks up the
// real device address with cudaGetSymbolAddress once per device (with that
// device current) on the first call that needs scratch, and passes that
// address to the kernels; later calls read the cached address without taking
// the lock.  A cudaDeviceReset unloads the module the address belongs to, so
// the entry point must not be used after one.  Every call on a device shares
// the array: two calls whose kernels overlap on the GPU (different streams
// without ordering) race on it.  Each call overwrites every scratch word it
// reads, so nothing has to be cleared.
#include "kvc_internal.h"

#include <atomic>
#include <mutex>

namespace kvc {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVC_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::atomic<void *> g_scratch_addr[MAX_DEVICES];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (nullptr on failure).
void *scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return nullptr;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p)
        return p;
    std::lock_guard<std::mutex> lk(g_scratch_mu);   // first call on this device: set-up
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess)
            return nullptr;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    return p;
}

} // namespace
} // namespace kvc

extern "C" kvc_status kvc_decode_attend_noalloc(const kvc_attend_args *args, cudaStream_t stream)
{
    if (!args)
        return KVC_ERR_INVALID_ARG;
    kvc_attend_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    const size_t need = kvc_workspace_size(&a);
    if (need > (size_t)KVC_NOALLOC_SCRATCH_BYTES)
        return KVC_ERR_WORKSPACE;   // these shapes need more scratch than the fixed array holds
    if (need > 0) {
        void *p = kvc::scratch_address();
        if (!p)
            return KVC_ERR_CUDA;
        a.workspace = p;
        a.workspace_bytes = (size_t)KVC_NOALLOC_SCRATCH_BYTES;
    }
    return kvc_decode_attend(&a, stream);
}
