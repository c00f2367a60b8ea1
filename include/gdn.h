/*
 * gdn.h -- C ABI of the chunked gated delta rule (GDN) prefill library for NVIDIA GB300
 * (sm_103a).
 *
 * The operation (FlashQLA pages: agentlenshq "GDN chunked prefill optimisation" and the
 * aisparkup "usage" section, which gives the high-level call
 * chunk_gated_delta_rule(q, k, v, g, beta, scale, initial_state, output_final_state,
 * cu_seqlens) -> (o, final_state) and the low-level forward/backward entry points):
 *
 *   per sequence, per v-head j (q/k head j / G, G = Hv / Hqk), state S_t in R^{V x K}:
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale * S_t q_t
 *   S_0 = initial state (zero when absent); the final state is S after the last token.
 *
 * States cross this ABI transposed, as h = S^T stored [K][V] (row-major, V fastest).
 *
 * Tensor layouts (row-major, contiguous; "T_total" = B*T, or T when varlen):
 *   q, k      [T_total, Hqk, K]   dtype (bf16 or fp32)
 *   v, o, dO  [T_total, Hv,  V]   dtype
 *   g, beta   [T_total, Hv]       fp32   (g: natural-log decay, beta: write strength)
 *   h0, ht, dht, dh0  [N_seq, Hv, K, V]  fp32
 *   dq, dk    like q;  dv like v;  dg, dbeta like g (fp32)
 *
 * Conventions, for every entry point:
 *   - Pointers are DEVICE pointers unless the field says host.  Every device pointer must
 *     be 16-byte aligned.  The caller owns all memory; the library never allocates, frees
 *     or synchronises.  Work is enqueued on `stream` (a cudaStream_t; NULL = legacy stream)
 *     and runs asynchronously.
 *   - Arguments are validated before anything is launched; on a non-OK status nothing has
 *     been written and gdn_last_error() (thread-local) says why.
 *   - Results are deterministic: repeated calls give bitwise-identical outputs.
 *   - K = V = 128 only (GDN_ERR_UNSUPPORTED otherwise).
 *   - Stream order holds as for any launch.  Inside a call, kernels overlap their
 *     predecessors' ends by programmatic dependent launch, each waiting for its predecessor
 *     (griddepcontrol.wait) before it reads anything that one wrote; the library's kernels
 *     signal their dependents early, so a caller's kernel launched right after a call WITH
 *     programmatic stream serialisation must itself wait (cudaGridDependencySynchronize)
 *     before it reads the call's outputs.  Ordinary launches, copies and events need nothing.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment or cu_seqlens */
    GDN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. K != 128) */
    GDN_ERR_WORKSPACE = 3,     /* workspace missing or smaller than the *_workspace_size */
    GDN_ERR_CUDA = 4,          /* a CUDA launch or attribute call failed */
    GDN_ERR_TIMEOUT = 5,       /* a device-side wait gave up (gdn_device_status) */
    GDN_ERR_BOUNDS = 6         /* checked build: a store index fell outside its tensor (gdn_device_status) */
} gdn_status;

typedef enum { GDN_BF16 = 0, GDN_FP32 = 1 } gdn_dtype;

/* Intra-GPU context parallelism over chunk ranges (FlashQLA pages, "AutoCP" section: when
 * batch * heads leaves SMs idle, each sequence's chunks are split into segments). */
typedef enum {
    GDN_CP_AUTO = 0,    /* exact; the planner picks the segment length L: by default the L
                           that minimises a cost model of the launches on this GPU (waves of
                           one CTA per SM, chunk steps, fix-up steps); with cp_lambda > 0 the
                           pages' rule L = cp_lambda * sqrt(chunks) instead */
    GDN_CP_OFF = 1,     /* one segment per sequence: a plain serial chunk scan */
    GDN_CP_EXACT = 2,   /* segments of cp_segment_chunks chunks; transition fix-up, exact */
    GDN_CP_WARMUP = 3,  /* opt-in approximation: each segment starts warmup_chunks chunks
                           early from a zero state instead of the exact fix-up (FlashQLA
                           pages, "warm-up" paragraph: 6-8 chunks); NOT exact */
    GDN_CP_EXACT_FULL = 4 /* as GDN_CP_EXACT, with every segment's transition computed and
                           composed and every segment rerun from its entering state */
} gdn_cp_mode;

/* How the exact modes (AUTO, EXACT) skip work without changing the result.  Every chunk's
 * state transition X -> prod_t exp(g_t) (I - beta_t k_t k_t^T) X has 2-norm at most
 * B = exp(sum_t g_t) prod_t max(1, |1 - beta_t |k_t|^2|), computed per (chunk, v-head) from
 * the inputs (bf16 path).  Where the product of these bounds over a prefix of a segment falls
 * below 2^-126, the smallest normal fp32 number, whatever enters the segment changes the states
 * past that prefix by less than 2^-126 times its norm: the segment's transition is then not
 * computed (the fix-up takes the segment's state from zero as its result) and only the
 * prefix's outputs are recomputed from the true entering state.  Elsewhere the transition is
 * computed, composed and the whole segment rerun, as in GDN_CP_EXACT_FULL.  The fp32 test mode
 * always works as GDN_CP_EXACT_FULL. */

typedef struct gdn_problem {
    int32_t B;                        /* batch; must be 1 when cu_seqlens is given */
    int32_t T;                        /* tokens per sequence (total tokens when varlen) */
    int32_t Hqk;                      /* q/k heads */
    int32_t Hv;                       /* v heads; multiple of Hqk */
    int32_t K;                        /* key dim (128) */
    int32_t V;                        /* value dim (128) */
    int32_t dtype;                    /* gdn_dtype of q, k, v, o, dO, dq, dk, dv */
    float scale;                      /* output scale, finite and > 0 (GDN_ERR_INVALID_ARG
                                         otherwise); usually K^-0.5 */
    const int32_t* cu_seqlens;        /* device [num_seqs+1] or NULL (then B sequences of T) */
    const int32_t* cu_seqlens_host;   /* HOST copy with the same contents; required iff
                                         cu_seqlens != NULL (sizes the launch grids) */
    int32_t num_seqs;                 /* N_seq when varlen */
    int32_t cp_mode;                  /* gdn_cp_mode */
    int32_t cp_segment_chunks;        /* EXACT, EXACT_FULL, WARMUP: chunks per segment
                                         (0 = auto) */
    int32_t warmup_chunks;            /* WARMUP: warm-up chunks (0 = 8) */
    float cp_lambda;                  /* AUTO: lambda in L = lambda sqrt(N) (0 = cost model) */
} gdn_problem;

/* Bytes of device workspace gdn_chunk_fwd needs for *p (written to *bytes). */
gdn_status gdn_chunk_fwd_workspace_size(const gdn_problem* p, size_t* bytes);

/*
 * Forward (FlashQLA pages: the low-level forward of the aisparkup "usage" section; the
 * chunk-local prep, the chunk-serial state scan and the output stage of the agentlenshq
 * "GDN chunked prefill" section).
 *   h0  : initial states or NULL (zero).       o  : output, written for every token.
 *   ht  : final states or NULL (not returned).
 *   workspace: device scratch of at least gdn_chunk_fwd_workspace_size bytes (contents
 *   are overwritten; it may be reused across calls on the same stream).
 */
gdn_status gdn_chunk_fwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, void* o,
                         float* ht, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace gdn_chunk_bwd needs for *p (written to *bytes). */
gdn_status gdn_chunk_bwd_workspace_size(const gdn_problem* p, size_t* bytes);

/*
 * Backward (FlashQLA pages, agentlenshq "backward pass" paragraph: the dv, dh-scan,
 * dq/dk/dw/dg and WY-backward steps).  Gradients of
 *   L = <o, dO> + <ht, dht>
 * with respect to q, k, v, g, beta and h0, for the forward defined above with the same
 * inputs.  The forward intermediates are recomputed from q, k, v, g, beta, h0.
 *   dht : NULL = zero.   dh0 : NULL = not returned.
 *   dq, dk are summed over the G v-heads that share each q/k head.
 *   Context parallelism in the backward is always exact (GDN_CP_WARMUP is treated as
 *   GDN_CP_EXACT here).
 */
gdn_status gdn_chunk_bwd(const gdn_problem* p, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, const void* dO,
                         const float* dht, void* dq, void* dk, void* dv, float* dg,
                         float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                         void* stream);

/* ------------------------------------------------------------------------------------
 * Low-level forward / backward pair with saved intermediates (FlashQLA pages, aisparkup
 * "usage" section: the low-level forward returns g, A, o, h and the final state, and the
 * backward is called separately).  The pages name the tuple but do not define its members;
 * this library reads them as
 *   g_cum : [T_total, Hv] fp32, gamma, the cumulative sum of g within each chunk (it restarts
 *           at every chunk start and at every sequence start);
 *   A     : [T_total, Hv, C] dtype, for every token its row of its chunk's
 *           T = (I + diag(beta) (K K^T * Dm))^-1 (unit lower triangular; Dm_ij =
 *           exp(gamma_i - gamma_j) for i > j, else 0); column i of a token's row refers to
 *           the chunk's i-th token, columns past the token's own position are 0;
 *   h     : [total_chunks, Hv, K, V] dtype, the state h = S^T entering every chunk, chunks
 *           numbered over all sequences in order (sequence s holds ceil(len_s / C) of them,
 *           its first one being h0, or 0).
 * C is the kernels' chunk size (64 for bf16, 32 in the fp32 test mode); gdn_chunk_layout
 * reports it and total_chunks.
 *
 * gdn_chunk_fwd_saved computes what gdn_chunk_fwd computes and also writes g_cum and A (when
 * non-NULL) and h (required).  It runs the backward's decomposition of the problem
 * (context parallelism is exact; GDN_CP_WARMUP is treated as GDN_CP_EXACT) and leaves in
 * the workspace the chunk records and segment transitions that the backward needs: the
 * workspace must hold gdn_chunk_bwd_workspace_size bytes.
 *
 * gdn_chunk_bwd_saved computes what gdn_chunk_bwd computes for the same inputs, without
 * recomputing the forward: it reads h and the workspace exactly as gdn_chunk_fwd_saved left
 * them for the same problem (the caller keeps both unchanged between the two calls, and
 * orders the calls, e.g. on one stream).  h0 is not needed (h holds it).  g_cum and A are
 * outputs only; the backward does not read them.
 * ------------------------------------------------------------------------------------ */
gdn_status gdn_chunk_layout(const gdn_problem* p, int32_t* chunk_size, int64_t* total_chunks);

gdn_status gdn_chunk_fwd_saved(const gdn_problem* p, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const float* h0, void* o,
                               float* ht, float* g_cum, void* A, void* h, void* workspace,
                               size_t workspace_bytes, void* stream);

gdn_status gdn_chunk_bwd_saved(const gdn_problem* p, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const void* h, const void* dO,
                               const float* dht, void* dq, void* dk, void* dv, float* dg,
                               float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                               void* stream);

/* ------------------------------------------------------------------------------------
 * Fused prologue: the activations that turn a layer's raw projections into the inputs of
 * gdn_chunk_fwd, in one pass (read once, write once), and their reverse mode.  The FlashQLA
 * pages take q, k, g, beta as given (g a log-decay, beta a write strength, q and k the unit
 * keys of the delta rule) and do not say how they are formed; this library reads them as
 *   q = q_raw / sqrt(sum(q_raw^2) + 1e-6)  and  k likewise   (per token and q/k head, over K)
 *   g = -exp(A_log[j]) * softplus(a + dt_bias[j])           (per token and v-head j)
 *   beta = 1 / (1 + exp(-b))
 * with softplus(x) = log(1 + exp(x)) (x itself above 20).
 *
 * Shapes from *p (B, T or varlen total T, Hqk, Hv, K = 128, dtype; cu_seqlens unused):
 *   q_raw, k_raw, q, k, dq, dk, dq_raw, dk_raw   [T_total, Hqk, K]  dtype
 *   a, b, g, beta, dg, dbeta, da, db             [T_total, Hv]      fp32
 *   A_log, dt_bias, dA_log, ddt_bias             [Hv]               fp32
 * gdn_prologue_fwd may run in place (q == q_raw, k == k_raw, g == a, beta == b).
 * gdn_prologue_bwd takes dq, dk, dg, dbeta (the gradients gdn_chunk_bwd returns) and the
 * forward's raw inputs, and writes the gradients of L with respect to q_raw, k_raw, a, b,
 * A_log and dt_bias; dA_log and ddt_bias are sums over all tokens taken in a fixed order.
 * Its workspace (gdn_prologue_bwd_workspace_size bytes) holds per-head partial sums.
 * ------------------------------------------------------------------------------------ */
gdn_status gdn_prologue_fwd(const gdn_problem* p, const void* q_raw, const void* k_raw,
                            const float* a, const float* b, const float* A_log,
                            const float* dt_bias, void* q, void* k, float* g, float* beta,
                            void* stream);

gdn_status gdn_prologue_bwd_workspace_size(const gdn_problem* p, size_t* bytes);

gdn_status gdn_prologue_bwd(const gdn_problem* p, const void* q_raw, const void* k_raw,
                            const float* a, const float* b, const float* A_log,
                            const float* dt_bias, const void* dq, const void* dk,
                            const float* dg, const float* dbeta, void* dq_raw, void* dk_raw,
                            float* da, float* db, float* dA_log, float* ddt_bias,
                            void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------
 * Per-kernel timing (instrumentation for benchmarks; not needed for computation).
 * While enabled, every kernel the library launches is bracketed by two CUDA events
 * recorded on the launching stream.  gdn_timing_collect waits for the recorded events
 * (it synchronises on them), sums the elapsed time per kernel name, writes up to
 * max_entries records, sets *n_entries to the number of distinct kernels, releases the
 * events and clears the record.  Not thread-safe: time one thread's calls at a time.
 * ------------------------------------------------------------------------------------ */
typedef struct gdn_kernel_time {
    char name[48];     /* kernel name, e.g. "fwd_phase_c" */
    int32_t launches;  /* launches recorded since the last collect */
    float total_ms;    /* summed event-to-event time of those launches */
} gdn_kernel_time;

gdn_status gdn_timing_enable(int32_t enable);
gdn_status gdn_timing_collect(gdn_kernel_time* out, int32_t max_entries, int32_t* n_entries);

/* ------------------------------------------------------------------------------------
 * Allocation-free forward.  The FlashQLA pages have no counterpart to this entry point: it
 * exists for callers that cannot allocate device memory themselves -- a runtime that has
 * handed all device memory to its own pool, a latency-critical loop where cudaMalloc or
 * cudaFree may synchronise the device, or a plug-in interface that passes only inputs and
 * outputs.  It computes exactly what gdn_chunk_fwd computes, with the same arguments minus
 * the workspace.
 *
 * Its scratch is one fixed device array of GDN_NOALLOC_SCRATCH_BYTES inside the library;
 * every GPU that loads the library holds that memory until the process exits.  Problems
 * whose gdn_chunk_fwd_workspace_size exceeds it are rejected with GDN_ERR_WORKSPACE and a
 * message (nothing is launched); fewer context-parallel segments (cp_mode /
 * cp_segment_chunks) shrink the need.  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.  The lookup is
 * repeated when the device's context has changed since (e.g. after cudaDeviceReset, which
 * may load the array at another address), so such a call, too, belongs outside a capture.
 * All calls share the one array and it keeps the last call's contents (every byte a call
 * reads is written earlier by the same call), so calls whose GPU work overlaps -- on
 * different streams, or from different threads -- race on it and must be serialised by the
 * caller.
 *
 * gdn_noalloc_device_status is gdn_device_status for these calls: it waits for `stream` and
 * reads the error word that the calls keep at the start of the array (their device-side
 * failure report, see below).  gdn_noalloc_debug_wait_timeout is gdn_debug_wait_timeout on
 * that word (a test hook).
 * ------------------------------------------------------------------------------------ */
#define GDN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

gdn_status gdn_chunk_fwd_noalloc(const gdn_problem* p, const void* q, const void* k,
                                 const void* v, const float* g, const float* beta,
                                 const float* h0, void* o, float* ht, void* stream);

gdn_status gdn_noalloc_device_status(void* stream);

gdn_status gdn_noalloc_debug_wait_timeout(int32_t limit_us, void* stream);

/* ------------------------------------------------------------------------------------
 * Device-side failure report.  Every wait of the tensor-core kernels on an mbarrier (a TMA
 * copy landing, a tensor-core product completing, a warp role handing over) is bounded: after
 * 2 s of wall time it gives up, sets a bit in the call's error word -- the first 4 bytes of
 * its workspace, cleared by the first kernel of every gdn_chunk_fwd, gdn_chunk_bwd,
 * gdn_chunk_fwd_saved and gdn_chunk_bwd_saved call -- and the kernel winds down (issued copies
 * and products drained, tensor memory released) instead of hanging; the outputs of that call
 * are then not valid.
 *
 * gdn_device_status waits for `stream` (this call does synchronise), reads the error word of
 * `workspace` (the workspace of the call(s) just enqueued on that stream) and returns GDN_OK,
 * or GDN_ERR_TIMEOUT with the word's bits in gdn_last_error().  workspace: device pointer, at
 * least 4 bytes, 16-byte aligned.
 *
 * Checked builds of this library (compiled with -DGDN_CHECK; libgdn_check.so, for tests)
 * also test the element index of every output store of the bf16 path (o, dq, dk, dv, dg,
 * dbeta, gamma and the rows of T) against the tensor's extent; a store outside it is skipped
 * and sets bit 31 of the error word, and gdn_device_status then returns GDN_ERR_BOUNDS.
 * Release builds do not test and never set that bit.
 * ------------------------------------------------------------------------------------ */
gdn_status gdn_device_status(const void* workspace, void* stream);

/* Test hook of the planner (host only, no GPU work): the segmentation that gdn_chunk_fwd (and
 * gdn_chunk_bwd) would use for `p` on a GPU with `sms` multiprocessors -- chunks per
 * context-parallel segment and the number of segments over all sequences (one per sequence
 * when the planner does not split them).  GDN_ERR_INVALID_ARG for an invalid problem, NULL
 * outputs or sms <= 0. */
gdn_status gdn_debug_plan(const gdn_problem* p, int32_t sms, int32_t* chunks_per_segment,
                          int32_t* segments);

/* Test hook of the failure report: one block waits on an mbarrier that no thread ever
 * completes, gives up after limit_us microseconds (1 .. 1000000) and sets its bit in the error
 * word of `workspace` (only those 4 bytes are touched).  Asynchronous on `stream`. */
gdn_status gdn_debug_wait_timeout(void* workspace, int32_t limit_us, void* stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char* gdn_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H */
