// Internal launch interface between the C ABI layer and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "gdn_plan.h"

namespace gdn {

// Chunk size of the kernels for a dtype (bf16: 64; fp32 test mode: 32).
int fwd_chunk_size(int dtype);

// Plan kernel + (phase A + fix-up when P.cp != CP_NONE) + phase C.  hist=true replaces
// the output stage by a store of every chunk's entering state into P.hist.
cudaError_t launch_fwd(const Problem& P, int dtype, bool hist, cudaStream_t st);

// The plan kernel (work decomposition from the device cu_seqlens) and the serial fix-up of
// the exact context-parallel mode, shared by the CUDA-core and tensor-core paths.
void launch_plan(const Problem& P, int C, cudaStream_t st);
// Multiprocessors of the current device.
int sm_count();
// Groups of 8 state columns per fix-up CTA for a launch over this many (sequence, head) chains.
int fixup_groups(int chains);
void launch_fixup(const Problem& P, cudaStream_t st);
// The backward's reverse fix-up (bf16 path: reads the untransposed transitions P.mbuf_t).
void launch_bwd_fixup_tc(const BwdProblem& B, cudaStream_t st);

// TMA descriptors of k, q, v for the tensor-core path.
struct TcMaps {
    CUtensorMap k, q, v;
};
// [T_total, H, 128] bf16 viewed as (d, head, token), box 64 x 1 x 64 (one 64-column block of
// a 64-token tile), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int H, int64_t T_total);
// [rows, 128] bf16 (rows of 256 bytes), box 64 x 128 (one 64-column block of a 128-row
// tile), 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows);
// Chunk-parallel preparation of the tensor-core path into P.prep: per (chunk, v-head) one
// record of P.prep_stride bytes holding W' = -T diag(beta e) K (bf16 64 x 128, two
// 128-byte-swizzled 64-column blocks), TU = T diag(beta) and P (bf16 64 x 64, swizzled), and
// for the backward also T itself (bf16 64 x 64, swizzled).
constexpr int PREP_W = 0, PREP_TU = 16384, PREP_P = 24576, PREP_T = 32768;
constexpr int PREP_FWD_BYTES = 32768, PREP_BWD_BYTES = 40960;
void launch_prep(const Problem& P, const TcMaps& maps, cudaStream_t st);


// Tensor-core (tcgen05) forward for bf16: same phases as launch_fwd.
cudaError_t launch_fwd_tc(const Problem& P, bool hist, int64_t T_total, cudaStream_t st);
// Tensor-core reverse dh scan of the backward (bf16; needs the forward's chunk records):
// which = 0 first context-parallel phase, 1 the rerun storing dh per chunk.
cudaError_t launch_bwd_scan_tc(const BwdProblem& B, int which, int64_t T_total, cudaStream_t st);

// Tensor-core local gradients of the backward (bf16): one persistent CTA per SM over the
// (chunk, v-head) items; needs the chunk records (with T), the states per chunk in B.f.hist and
// the gradients per chunk in B.dhist.
cudaError_t launch_bwd_local_tc(const BwdProblem& B, int64_t T_total, cudaStream_t st);

// Backward: reverse dh scan (with the same context-parallel segments as the forward) and
// the chunk-parallel local gradients; expects the forward recompute (states per chunk in
// B.f.hist, transitions in B.f.mbuf) to have run on the same stream.
cudaError_t launch_bwd(const BwdProblem& B, int dtype, cudaStream_t st);

// Fused prologue (q/k L2 norm, gate and beta activations) and its reverse mode.
struct PrologueArgs {
    int dtype;            // 0 bf16, 1 fp32 (q, k and their gradients)
    int64_t rows;         // T_total * Hqk rows of 128 for q and for k
    int64_t gates;        // T_total * Hv gate elements
    int Hv;
    const void* q_raw;
    const void* k_raw;
    const float* a;       // [T, Hv] gate pre-activation
    const float* b;       // [T, Hv] beta pre-activation
    const float* A_log;   // [Hv]
    const float* dt_bias; // [Hv]
    void* q;              // forward outputs
    void* k;
    float* g;
    float* beta;
    const void* dq;       // backward inputs
    const void* dk;
    const float* dg;
    const float* dbeta;
    void* dq_raw;         // backward outputs
    void* dk_raw;
    float* da;
    float* db;
    float* dA_log;
    float* ddt_bias;
    float* part;          // backward workspace (prologue_bwd_workspace bytes)
};
size_t prologue_bwd_workspace(int Hv);
cudaError_t launch_prologue_fwd(const PrologueArgs& A, cudaStream_t st);
cudaError_t launch_prologue_bwd(const PrologueArgs& A, cudaStream_t st);

// Test hook of the device failure report: a bounded wait that gives up after limit_us.
cudaError_t launch_debug_wait(int* err, int limit_us, cudaStream_t st);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device): the attribute
// persists, and setting it again on every call costs host time the small problems feel.
cudaError_t smem_attr_once(const void* kern, int bytes);
template <typename... KArgs>
cudaError_t smem_attr(void (*kern)(KArgs...), int bytes) {
    return smem_attr_once(reinterpret_cast<const void*>(kern), bytes);
}

// Per-kernel event timing hooks (no-ops unless gdn_timing_enable(1)).
void timing_begin(const char* name, cudaStream_t st);
void timing_end(cudaStream_t st);

// Launch with programmatic stream serialisation: the kernel may begin launching while the
// previous kernel in the stream drains; it must call pdl_wait() (tc05.cuh) before touching
// anything that kernel (or an earlier one) wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace gdn
