// noalloc.cu -- ssd_fwd_noalloc: the forward scan with its scratch memory in a
// library-owned static device array instead of a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// scan: code that runs while a CUDA graph is being captured (cudaMalloc is not
// a capturable operation), serving runtimes that reserve the whole device
// memory up front in their own pools and hand out no extra buffers, and
// real-time or embedded loops that must not touch the allocator at all.  This
// entry point lets them run the scan with only their inputs and outputs.
//
// The array lives in this translation unit's module, so it occupies device
// memory only on devices where this entry point is used (the module is loaded
// on first use) and stays allocated until the process exits.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;   // SSD_NOALLOC_SCRATCH_BYTES

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_addr[64] = {nullptr};   // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch array on the current device (looked up once per
// device, with that device current).  nullptr on failure.
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_addr[dev] = ptr;
    }
    return g_addr[dev];
}

}  // namespace

extern "C" ssd_status ssd_fwd_noalloc(const ssd_problem *prob, const ssd_fwd_args *args, void *stream) {
    size_t need = 0;
    ssd_status s = ssd_fwd_workspace_size(prob, args, &need);
    if (s != SSD_OK) return s;
    if (need > kNoAllocScratchBytes) return SSD_ERR_WORKSPACE_TOO_SMALL;
    void *ws = scratch_address();
    if (ws == nullptr) return SSD_ERR_CUDA;
    return ssd_fwd(prob, args, ws, kNoAllocScratchBytes, stream);
}
