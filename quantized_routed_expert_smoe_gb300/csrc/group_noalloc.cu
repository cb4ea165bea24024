// group_noalloc.cu -- smoe_group_noalloc: the grouping step with its scratch space inside the library, for callers
// that cannot allocate device memory themselves.
//
// smoe_group needs a scratch buffer of smoe_group_work_bytes(n, E) bytes (per-chunk expert counts).  Some callers
// cannot provide one: a runtime whose device memory is planned once up front (a fixed arena with no room set aside
// for library scratch), or a serving loop that must not call cudaMalloc between requests because the call can
// synchronise the device and stall the streams already in flight.  For them this entry point keeps the scratch in a
// file-scope __device__ array that every GPU loading the library holds until the process exits.
//
// The array holds the largest scratch any valid call needs: 48 chunks x 1024 experts of int32 counts (192 KiB).  The
// counts pass overwrites every entry a call later reads, so nothing has to be cleared between calls; the contents
// left by the previous call are simply replaced.  All calls on one device share the one array: two calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on it and give wrong tables.
// The first call on a device looks up the array's device address (cudaGetSymbolAddress with that device current);
// that first call should come before any stream capture.  The address is kept per device together with the identity
// of the device's CUDA context; a call that finds a different context (the old one was destroyed, e.g. by
// cudaDeviceReset, and the library's module loaded again) looks the address up again instead of using a stale one.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "smoe.h"
#include "smoe_internal.h"

namespace {

constexpr size_t kNoallocScratchInts = 48 * SMOE_MAX_EXPERTS;  // 196,608 bytes
static __device__ __align__(256) int32_t g_group_scratch[kNoallocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
struct ScratchAddr {
    int32_t* ptr;
    unsigned long long ctx_id;  // the context the address belongs to (0: not known)
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

bool aligned16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

// The unique id of the calling thread's current CUDA context (driver entry points looked up through the runtime,
// so that the library needs no link to the driver library); false when there is none yet or the lookup fails.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// The device address of this device's copy of the array, looked up with that device current on the first call and
// again whenever the device's context has changed since.  In host code the array's name stands for a host-side
// shadow, never for device memory, so the kernels get this address.
smoe_status scratch_address(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SMOE_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchAddr& c = g_scratch_addr[dev];
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    if (c.ptr == nullptr || !known || c.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_group_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            c.ptr = nullptr;
            return SMOE_ERR_LAUNCH;
        }
        c.ptr = static_cast<int32_t*>(p);
        // the lookup has made the context current if it was not yet; a context that still cannot be identified
        // leaves ctx_id 0, and every call then looks the address up again
        unsigned long long id2 = 0;
        c.ctx_id = current_context_id(&id2) ? id2 : 0ull;
    }
    *out = c.ptr;
    return SMOE_OK;
}

}  // namespace

extern "C" smoe_status smoe_group_noalloc(const int32_t* ids, int64_t T, int K, int E, int32_t* counts,
                                          int32_t* offsets, int32_t* src, int32_t* slot, int32_t* tiles,
                                          size_t tiles_bytes, void* stream) {
    if (T < 0 || E < 1 || E > SMOE_MAX_EXPERTS || K < 1 || K > SMOE_MAX_TOPK) return SMOE_ERR_ARG;
    if (T > (int64_t)(INT32_MAX / 2) / K) return SMOE_ERR_ARG;  // checked before T * K can overflow
    const int64_t n = T * K;
    if (!aligned16(counts) || !aligned16(offsets) || !aligned16(tiles)) return SMOE_ERR_ARG;
    if (n > 0 && (!aligned16(ids) || !aligned16(src) || !aligned16(slot))) return SMOE_ERR_ARG;
    if (tiles_bytes < smoe_tiles_bytes(n, E)) return SMOE_ERR_ARG;
    // the built-in scratch covers every valid (n, E); a size beyond it is refused rather than overrun
    if (smoe_group_work_bytes(n, E) > kNoallocScratchInts * sizeof(int32_t)) return SMOE_ERR_UNSUPPORTED;
    if (smoe_device_check() != SMOE_OK) return SMOE_ERR_UNSUPPORTED;
    int32_t* scratch = nullptr;
    const smoe_status st = scratch_address(&scratch);
    if (st != SMOE_OK) return st;
    const cudaError_t err =
        smoe::launch_group(ids, n, K, E, counts, offsets, src, slot, tiles, scratch, (cudaStream_t)stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SMOE_ERR_LAUNCH;
    }
    return SMOE_OK;
}
