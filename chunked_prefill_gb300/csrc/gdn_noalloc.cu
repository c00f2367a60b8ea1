// gdn_chunk_fwd_noalloc: the forward with its scratch memory in a fixed-size device array
// that belongs to this library, for callers that cannot allocate device memory.
//
// Why some callers cannot allocate: a runtime that hands all device memory to its own pool
// at start-up (so a driver allocation would fail or break its accounting), a real-time or
// latency-critical loop where cudaMalloc/cudaFree may synchronise the device, or a plug-in
// interface that passes only the input and output buffers.  Those callers use this entry
// point; everyone else uses gdn_chunk_fwd with a workspace they allocate.
//
// The scratch is a file-scope __device__ array: every GPU that loads this library holds
// GDN_NOALLOC_SCRATCH_BYTES of it until the process exits.  In host code the array's name
// is only a host-side stand-in, so its device address is taken with cudaGetSymbolAddress,
// with the device current, on the first call made on that device -- and again whenever the
// device's context has changed since (after cudaDeviceReset the module, and the array, may
// be loaded at another address).  The context is told apart by its driver ID (cuCtxGetId),
// which is unique for the life of the process; without that driver entry point the lookup
// is simply repeated on every call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/gdn.h"

namespace {

constexpr size_t kScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct ScratchCache {
    unsigned long long ctx_id = 0;  // 0: nothing cached
    void* addr = nullptr;
};

std::mutex g_setup_mutex;
ScratchCache g_cache[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// ID of the calling thread's current context, or 0 when there is none yet (the runtime
// creates the primary context lazily) or the driver entry points are unavailable.
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        looked_up = true;
    }
    if (!get_cur || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

namespace gdn {
void set_last_error(const char* msg);  // defined with gdn_last_error
}

namespace {

// Device address of the scratch array for the current device and context (looked up again
// when the context changed); GDN_OK or GDN_ERR_CUDA with the message set.
gdn_status scratch_address(const char* who, void** out) {
    char msg[256];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "%s: no usable current device (%s)", who,
                 e != cudaSuccess ? cudaGetErrorString(e) : "device ordinal out of range");
        gdn::set_last_error(msg);
        return GDN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchCache& c = g_cache[dev];
    const unsigned long long id = current_ctx_id();
    if (id == 0 || c.ctx_id != id || !c.addr) {
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess || !addr) {
            snprintf(msg, sizeof(msg),
                     "%s: cudaGetSymbolAddress of the scratch array failed on device %d (%s)", who,
                     dev, e != cudaSuccess ? cudaGetErrorString(e) : "null address");
            gdn::set_last_error(msg);
            c = ScratchCache{};
            return GDN_ERR_CUDA;
        }
        c.addr = addr;
        c.ctx_id = current_ctx_id();  // the lookup has created the context if there was none
    }
    *out = c.addr;
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(const gdn_problem* p, const void* q, const void* k,
                                            const void* v, const float* g, const float* beta,
                                            const float* h0, void* o, float* ht, void* stream) {
    char msg[256];
    size_t need = 0;
    gdn_status st = gdn_chunk_fwd_workspace_size(p, &need);
    if (st != GDN_OK) return st;  // message already set by the size query
    if (need > kScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "gdn_chunk_fwd_noalloc: this problem needs %zu bytes of scratch, more than the "
                 "fixed %zu-byte array; call gdn_chunk_fwd with a caller-allocated workspace, "
                 "or use fewer context-parallel segments (cp_mode / cp_segment_chunks)",
                 need, kScratchBytes);
        gdn::set_last_error(msg);
        return GDN_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    st = scratch_address("gdn_chunk_fwd_noalloc", &scratch);
    if (st != GDN_OK) return st;
    return gdn_chunk_fwd(p, q, k, v, g, beta, h0, o, ht, scratch, kScratchBytes, stream);
}

// The failure report of the calls above: their error word is the first 4 bytes of the
// library's array, which only this file can address.
extern "C" gdn_status gdn_noalloc_device_status(void* stream) {
    void* scratch = nullptr;
    const gdn_status st = scratch_address("gdn_noalloc_device_status", &scratch);
    if (st != GDN_OK) return st;
    return gdn_device_status(scratch, stream);
}

extern "C" gdn_status gdn_noalloc_debug_wait_timeout(int32_t limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) {
        gdn::set_last_error("gdn_noalloc_debug_wait_timeout: limit_us must be in [1, 1000000]");
        return GDN_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    const gdn_status st = scratch_address("gdn_noalloc_debug_wait_timeout", &scratch);
    if (st != GDN_OK) return st;
    return gdn_debug_wait_timeout(scratch, limit_us, stream);
}
