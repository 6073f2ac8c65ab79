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
// on first use) and stays allocated until the process exits.  In host code its
// name is only a host-side stand-in: the device address is looked up with
// cudaGetSymbolAddress, with the device current, once per device and context (a
// context that was torn down and rebuilt, e.g. after cudaDeviceReset, gets a new
// lookup), and that address is what the kernels receive.
#include <cuda.h>
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;   // SSD_NOALLOC_SCRATCH_BYTES
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);

struct Slot {
    void *addr = nullptr;
    unsigned long long ctx_id = 0;
};
std::mutex g_mu;
Slot g_slot[kMaxDevices];   // per device ordinal: the scratch address and the context it belongs to

// Unique id of the current context (0 if there is none yet or the query is unavailable).
unsigned long long current_ctx_id() {
    static PfnCtxGetCurrent get_cur = nullptr;
    static PfnCtxGetId get_id = nullptr;
    static bool looked = false;
    if (!looked) {
        void *p1 = nullptr, *p2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 4000, cudaEnableDefault, &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PfnCtxGetCurrent>(p1);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PfnCtxGetId>(p2);
        looked = true;
    }
    if (get_cur == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_noalloc_scratch on the current device; nullptr on failure (an
// ordinal beyond kMaxDevices included: the cache has one slot per ordinal).
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    Slot &sl = g_slot[dev];
    const unsigned long long id = current_ctx_id();
    if (sl.addr == nullptr || id == 0 || id != sl.ctx_id) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        sl.addr = ptr;
        sl.ctx_id = current_ctx_id();   // the lookup made the device's context current
    }
    return sl.addr;
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

extern "C" ssd_status ssd_noalloc_query_status(void *stream) {
    void *ws = scratch_address();
    if (ws == nullptr) return SSD_ERR_CUDA;
    return ssd_query_status(ws, stream);
}
