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
// once per device, with that device current, on the first call made on that device.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/gdn.h"

namespace {

constexpr size_t kScratchBytes = GDN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

namespace gdn {
void set_last_error(const char* msg);  // defined with gdn_last_error
}

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
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "gdn_chunk_fwd_noalloc: no usable current device (%s)",
                 e != cudaSuccess ? cudaGetErrorString(e) : "device ordinal out of range");
        gdn::set_last_error(msg);
        return GDN_ERR_CUDA;
    }
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_addr[dev]) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
            if (e != cudaSuccess || !addr) {
                snprintf(msg, sizeof(msg),
                         "gdn_chunk_fwd_noalloc: cudaGetSymbolAddress of the scratch array "
                         "failed on device %d (%s)",
                         dev, e != cudaSuccess ? cudaGetErrorString(e) : "null address");
                gdn::set_last_error(msg);
                return GDN_ERR_CUDA;
            }
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    return gdn_chunk_fwd(p, q, k, v, g, beta, h0, o, ht, scratch, kScratchBytes, stream);
}
