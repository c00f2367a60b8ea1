// Forward chunk scan on the 5th-generation tensor cores (bf16 operands, fp32 accumulation).
//
// Same chunk algebra and the same context-parallel phases as the CUDA-core kernels in
// gdn_fwd.cu (FlashQLA pages, agentlenshq "GDN chunked prefill optimisation": chunk-local
// W/U preparation, the serial state S and the output O kept on-chip; "AutoCP" segments);
// what changes is where the data live and who moves them:
//
//   * the state is kept TRANSPOSED in tensor memory, Xt[v][dk] = h[dk][v] (fp32 master,
//     128 columns) plus a bf16 copy (64 columns) that is the A operand of the V' and Q h
//     products straight from TMEM;
//   * K, Q, V chunk tiles arrive by TMA (128-byte swizzle) and the chunk-local W', TU, P
//     tiles of the preparation kernel by bulk copies, into a 2-stage ring;
//   * per chunk of 64 tokens (i, j tokens; dk key dim; v value dim):
//       D3  = V^T TU^T + Xt W'^T = V'^T  (v x i)       -> bf16 V'^T and diag(kd) V'^T in TMEM
//       D4a = Xt Q^T     = (Q h)^T       (v x i)
//       D4b = V'^T P^T   = (P V')^T      (v x i)       -> O = scale (e * D4a + D4b)
//       Xt  = e^{gamma_C} Xt + (diag(kd) V')^T K       (v x dk)
//
// Warp roles (16 warps): 0 TMA producer; 1 state-chain MMA issuer (V' with D4a, state
// update); 2 gates (cumsum of g and its exponentials); 3 output MMA issuer (U, D4b), or U alone
// without an output side; 4-11 state warps, one warpgroup per half of the key columns (state
// hand-off, V' conversion); 12-15 output warps.  The two issuers run independently: the state
// chain never queues behind the output products.  Every wait on an mbarrier is bounded; on a
// timeout the kernel records an error word and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc05.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int TCT = 512;  // threads (16 warps)
constexpr int CH = 64;    // chunk

// tensor-memory columns: Xt (fp32 state, transposed), its bf16 copy, two chunk buffers DD
// (by chunk parity) and D4b.  A DD buffer holds [V'^T | (Q h)^T] (64 + 64 columns): U^T is
// written first (the (Q h)^T half is zero: the output warps clear it after reading it), then
// one MMA over [W'; Q] adds Xt W'^T and Xt Q^T (as two products of N = 64, V' first, the
// whole scan ran slower: more tensor-pipe instructions per chunk).  D4b = (P V')^T; the
// output warps combine O = scale (e (Q h) + P V').
constexpr uint32_t T_XF = 0, T_XB = 128, T_D4B = 448;
__device__ __forceinline__ uint32_t t_dd(int k) { return (k & 1) ? 320u : 192u; }
// converted V' in a DD buffer: tokens [0,32) at columns [0,16) (V'^T) and [16,32)
// (diag(kd) V'^T), tokens [32,64) at [32,48) and [48,64); K step s covers 16 tokens
__device__ __forceinline__ uint32_t p_col(int s) { return uint32_t((s >> 1) * 32 + (s & 1) * 8); }
__device__ __forceinline__ uint32_t kd_col(int s) { return uint32_t((s >> 1) * 32 + 16 + (s & 1) * 8); }

// shared-memory layout (offsets from a 1024-aligned base), two stages of
//   K     [64 tok][128 dk]          2 x 8 KB column blocks (MN-major B of the state update)
//   WQ    [W' 64 rows; Q 64 rows]   2 column blocks of 16 KB (K-major B of the V'/Qh MMA)
//   V     [64 tok][128 v]           MN-major A of the U MMA
//   TU    [64 i][64 j]              K-major B of the U MMA
// and a ring of NP P tiles ([64 i][64 j], K-major B of the P V' MMA) that the output issuer
// fills and drains on its own, so the output side never holds back the stage ring.
constexpr uint32_t S_K = 0, S_K_STRIDE = 16384;
constexpr uint32_t S_WQ = 32768, S_WQ_STRIDE = 32768;
constexpr uint32_t S_V = 98304, S_V_STRIDE = 16384;
constexpr uint32_t S_TU = 131072, S_TU_STRIDE = 8192;
constexpr uint32_t S_P = 147456, S_P_STRIDE = 8192;
constexpr int NP = 4;
constexpr uint32_t S_GATE = 180224;     // NGATE gate buffers
constexpr int NGATE = 4;
constexpr uint32_t GATE_BYTES = 1088;
constexpr int LDO = 136;                              // output staging row stride (bf16)
constexpr uint32_t S_O = S_GATE + NGATE * GATE_BYTES; // 64 x 136 bf16 output staging
constexpr uint32_t S_BAR = S_O + 64 * LDO * 2;        // mbarriers
constexpr uint32_t S_END = S_BAR + 512;              // B_COUNT barriers, TMEM slot, error word
constexpr uint32_t SMEM_BYTES = S_END + 1024;         // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct alignas(16) Gate {
    float gam[CH];
    float e[CH];     // exp(gamma)
    float kd[CH];    // exp(gamma_C - gamma)
    float eC;
    int c;           // valid rows
    int store;       // store this chunk's outputs (and entering state, when asked)
    int pad;
};

// First pass of the decay-bounded exact mode (see k_tc_phase_c): which chunks' results this
// CTA stores and where its decisions go.
struct ScanRule {
    int n_own;       // chunks of the own segment (the scan may run on into the next one)
    int e_own;       // leading chunks of the own segment that the previous CTA stores (0: none)
    int lj;          // segment index within the sequence (reverse scan: 0 for every segment but
                     // the last, whose scan starts from the true gradient)
    int* dec;        // -1: the own segment's transition is not negligible, else 0 (or null)
    int ext_ok;      // reverse scan: the own segment's transition is negligible (the forward's
                     // decision), so the scan past it starts from a true state
    int* rerun;      // 1: some output of the own segment is left to the correction pass
    float* x_mid;    // the state at the end of the own segment, when the scan runs on (or null)
};
static_assert(sizeof(Gate) <= GATE_BYTES && sizeof(Gate) % 16 == 0, "gate buffer");

enum Bar { B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_GATE0, B_GATE1, B_GATE2, B_GATE3, B_GFREE0,
           B_GFREE1, B_GFREE2, B_GFREE3, B_MMA3, B_MMA5, B_MMA4_0, B_MMA4_1, B_DRAIN, B_EX, B_EV0,
           B_EV1, B_EPI0, B_EPI1, B_M5C0, B_M5C1, B_U0, B_U1, B_FULLP0, B_EMPTYP0 = B_FULLP0 + NP,
           B_COUNT = B_EMPTYP0 + NP };

static_assert(B_COUNT * 8 + 8 <= 512, "barrier area");

enum TcKind { TK_STATE = 0, TK_TRANS = 1, TK_OUT = 2, TK_HIST = 3 };

#ifdef GDN_TRACE
#ifndef GDN_TRACE_X
#define GDN_TRACE_X 0
#define GDN_TRACE_Y 0
#endif
// debug builds only: SM-clock timestamps of the pipeline events of one CTA
__device__ unsigned long long g_trace[64][32];
__device__ unsigned long long g_cta_trace[2][512][4];  // [phase A, C][cta]: globaltimer at entry, scan start, scan end, exit
#define CTRACE(ph, e)                                                                          \
    do {                                                                                       \
        if (threadIdx.x == 0 && blockIdx.x * gridDim.y + blockIdx.y < 512) {                   \
            unsigned long long t_;                                                             \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                             \
            g_cta_trace[ph][blockIdx.x * gridDim.y + blockIdx.y][e] = t_;                      \
        }                                                                                      \
    } while (0)
#define TRACE(k, ev)                                                                           \
    do {                                                                                       \
        if (blockIdx.x == GDN_TRACE_X && blockIdx.y == GDN_TRACE_Y && blockIdx.z == 0 && (k) >= 0 && (k) < 64) \
            g_trace[(k)][(ev)] = clock64();                                                    \
    } while (0)
#else
#define TRACE(k, ev) \
    do {             \
    } while (0)
#define CTRACE(ph, e) \
    do {              \
    } while (0)
#endif

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) {  // K-major SW128 operand
    return make_desc(addr, 0, 1024);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t addr, uint32_t lbo) {  // MN-major SW128
    return make_desc(addr, lbo, 1024);
}


__device__ __forceinline__ bool wait_bar(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    if (mbar_wait_spin(&bars[b], parity)) return true;
    atomicOr(errflag, 1 << (b % 27));
    return false;
}
// a wait of a role that is not on the state chain: it backs off between tries
__device__ __forceinline__ bool wait_bar_lazy(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    if (mbar_wait_sleep(&bars[b], parity, 64)) return true;
    atomicOr(errflag, 1 << (b % 27));
    return false;
}
// warp-uniform wait: lane 0 waits, the result is broadcast, then the warp synchronises
template <bool LAZY = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0)
        ok = LAZY ? wait_bar_lazy(bars, b, parity, errflag) : wait_bar(bars, b, parity, errflag);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}

// Entering state (fp32, [dk][v] in global memory; null = zero, or the identity for the
// transition kind) into key columns [64 half, 64 half + 64) of the transposed TMEM state.
template <int KIND>
__device__ __forceinline__ void init_state_half(uint32_t tm, uint32_t lb, int half, int v,
                                                const float* x0, uint32_t xf = T_XF) {
    float xv[16];
    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int dk = c0 + i;
            xv[i] = x0 ? x0[dk * VD + v] : ((KIND == TK_TRANS && dk == v) ? 1.f : 0.f);
        }
        tmem_st16(tm + lb + xf + c0, xv);
    }
    tmem_st_wait();
}

// The same hand-off in two parts, so that the chain's next products can start after the
// first: (1) read the fp32 state of one half and write its bf16 copy (all the next products
// read); (2) after the hand-off has been signalled, store the state for the backward when
// asked and decay the fp32 state by exp(gamma_C) in place -- the state update accumulates onto
// it only after the V' conversion, whose store wait and arrival follow.  Part 1 leaves the 64
// values in x for part 2.
__device__ __forceinline__ void state_bf16_half(uint32_t tm, uint32_t lb, uint32_t xb, int half,
                                                uint32_t xf, float (&x)[64]) {
    const int c0 = 64 * half;
    tmem_ld32(tm + lb + xf + c0, x);
    tmem_ld32(tm + lb + xf + c0 + 32, x + 32);
    tmem_ld_wait();
    float pk[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) pk[i] = __uint_as_float(pack_bf16(x[2 * i], x[2 * i + 1]));
    tmem_st16(tm + lb + xb + c0 / 2, pk);
    tmem_st16(tm + lb + xb + c0 / 2 + 16, pk + 16);
    tmem_st_wait();
}
template <int KIND>
__device__ __forceinline__ void state_decay_half(const Problem& P, uint32_t tm, uint32_t lb, int half,
                                                 int v, float eC, int64_t chunk, int j, uint32_t xf,
                                                 float (&x)[64], bool store = true) {
    const int c0 = 64 * half;
    if ((KIND == TK_HIST || (KIND == TK_OUT && P.hist)) && store) {
        __nv_bfloat16* hp = reinterpret_cast<__nv_bfloat16*>(P.hist) + (chunk * P.Hv + j) * (KD * VD);
#pragma unroll
        for (int i = 0; i < 64; ++i) hp[(c0 + i) * VD + v] = __float2bfloat16_rn(x[i]);
    }
#pragma unroll
    for (int i = 0; i < 64; ++i) x[i] *= eC;
    tmem_st32(tm + lb + xf + c0, x);
    tmem_st32(tm + lb + xf + c0 + 32, x + 32);
}

// The two parts for a warp that hands off all 128 columns (too many to keep in registers
// between the parts: the second reads the fp32 state again), 32 columns at a time.
__device__ __forceinline__ void state_bf16_all(uint32_t tm, uint32_t lb, uint32_t xb, uint32_t xf) {
#pragma unroll 1
    for (int c0 = 0; c0 < KD; c0 += 32) {
        float x[32], pk[16];
        tmem_ld32(tm + lb + xf + c0, x);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = __uint_as_float(pack_bf16(x[2 * i], x[2 * i + 1]));
        tmem_st16(tm + lb + xb + c0 / 2, pk);
    }
    tmem_st_wait();
}
__device__ __forceinline__ void state_decay_all(uint32_t tm, uint32_t lb, uint32_t xf, float eC) {
#pragma unroll 1
    for (int c0 = 0; c0 < KD; c0 += 32) {
        float x[32];
        tmem_ld32(tm + lb + xf + c0, x);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] *= eC;
        tmem_st32(tm + lb + xf + c0, x);
    }
}

// x_out_t (TK_TRANS only, or null): the transition also untransposed.  rule (or null: store
// everything): the gate warp sums the own chunks' transition log-bounds (P.logb); with P_c the
// sum over chunks [0, c), chunk c's entering state depends on the scan's entering state by less
// than 2^-126 of its norm when P_c < LOG_NEGLIGIBLE.  An own chunk's results are stored when
// the previous CTA does not store them (c >= e_own) and P_c is below it (a chunk at or past
// e_own that fails is left to the correction: rerun); the chunks past the own segment are
// stored when the scan reached them from a true state (the first segment, or P_n below it).
// The scan's barriers, its tensor memory and (with an output side) the zeroed (Q h)^T halves;
// nothing here reads memory that an earlier kernel writes, so a kernel may run it before it
// waits for its predecessor (then tc_scan is called with ready, or tc_scan_release frees the
// tensor memory on a path that does not scan).
template <int KIND>
__device__ void tc_scan_setup(unsigned char* sm) {
    constexpr bool OUT = KIND == TK_OUT;
    constexpr bool NEEDU = KIND != TK_TRANS;
    const int tid = threadIdx.x, w = tid >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + B_COUNT * 8);
    int* errflag = reinterpret_cast<int*>(sm + S_BAR + B_COUNT * 8 + 4);
    if (tid == 0) {
        mbar_init(&bars[B_FULL0], 1);
        mbar_init(&bars[B_FULL1], 1);
        mbar_init(&bars[B_EMPTY0], 1);  // released by the state-chain issuer
        mbar_init(&bars[B_EMPTY1], 1);
        for (int b = 0; b < NP; ++b) {
            mbar_init(&bars[B_FULLP0 + b], 1);
            mbar_init(&bars[B_EMPTYP0 + b], 1);
        }
        for (int b = 0; b < NGATE; ++b) {
            mbar_init(&bars[B_GATE0 + b], 1);
            mbar_init(&bars[B_GFREE0 + b], OUT ? 12 : 8);  // 8 state warps (+ 4 output warps)
        }
        mbar_init(&bars[B_MMA3], 1);
        mbar_init(&bars[B_MMA5], 1);
        mbar_init(&bars[B_MMA4_0], 1);
        mbar_init(&bars[B_MMA4_1], 1);
        mbar_init(&bars[B_DRAIN], NEEDU ? 2 : 1);  // the state-chain issuer and warp 3
        mbar_init(&bars[B_EX], 8);
        mbar_init(&bars[B_EV0], 8);
        mbar_init(&bars[B_EV1], 8);
        mbar_init(&bars[B_EPI0], 4);
        mbar_init(&bars[B_EPI1], 4);
        mbar_init(&bars[B_M5C0], 1);  // per chunk parity: the state update has completed
        mbar_init(&bars[B_M5C1], 1);
        mbar_init(&bars[B_U0], 1);
        mbar_init(&bars[B_U1], 1);
        *errflag = 0;
        mbar_fence_init();
    }
    if (w == 0) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;
    if (OUT) {  // the (Q h)^T halves of both DD buffers start at zero
        if (w >= 12) {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
            const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                tmem_st32(tm + lb + t_dd(b) + 64, z);
                tmem_st32(tm + lb + t_dd(b) + 96, z);
            }
            tmem_st_wait();
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
}
__device__ void tc_scan_release(unsigned char* sm) {
    fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        fence_after_sync();
        tmem_dealloc(*reinterpret_cast<uint32_t*>(sm + S_BAR + B_COUNT * 8), 512);
    }
}

template <int KIND>
__device__ void tc_scan(const Problem& P, const TcMaps& maps, unsigned char* sm, int j,
                        int64_t t0, int64_t t1, int cb, int ce, const float* x0, float* x_out,
                        int64_t hist_base, float* x_out_t = nullptr, const ScanRule* rule = nullptr,
                        bool ready = false) {
    constexpr bool OUT = KIND == TK_OUT;
    constexpr bool NEEDU = KIND != TK_TRANS;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + B_COUNT * 8);
    int* errflag = reinterpret_cast<int*>(sm + S_BAR + B_COUNT * 8 + 4);
    Gate* gates = reinterpret_cast<Gate*>(sm + S_GATE);
    const int G = P.Hv / P.Hqk, qh = j / G;
    const int n = ce - cb;

    if (!ready) tc_scan_setup<KIND>(sm);
    CTRACE(OUT || KIND == TK_HIST ? 1 : 0, 2);
    const uint32_t tm = *tmem_slot;
    if (w == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t bytes = 16384u + 16384u + (OUT ? 16384u : 0u) + (NEEDU ? 16384u + 8192u : 0u);
            int issued = 0;
            for (int k = 0; k < n; ++k) {
                const int st = k & 1;
                if (k >= 2 && !wait_bar_lazy(bars, B_EMPTY0 + st, ((k - 2) >> 1) & 1, errflag)) break;
                TRACE(k, 3);
                const int tc = int(t0 + int64_t(cb + k) * CH);
                uint64_t* full = &bars[B_FULL0 + st];
                unsigned char* kt = sm + S_K + st * S_K_STRIDE;
                unsigned char* wq = sm + S_WQ + st * S_WQ_STRIDE;
                const unsigned char* rec = static_cast<const unsigned char*>(P.prep) +
                                           ((hist_base + cb + k) * P.Hv + j) * P.prep_stride;
                mbar_expect_tx(full, bytes);
                tma_load_3d(kt, &maps.k, full, 0, qh, tc);
                tma_load_3d(kt + 8192, &maps.k, full, 64, qh, tc);
                bulk_load(wq, rec + PREP_W, 8192, full);                // W' columns 0-63
                bulk_load(wq + 16384, rec + PREP_W + 8192, 8192, full); // W' columns 64-127
                if (OUT) {
                    tma_load_3d(wq + 8192, &maps.q, full, 0, qh, tc);
                    tma_load_3d(wq + 16384 + 8192, &maps.q, full, 64, qh, tc);
                }
                if (NEEDU) {
                    unsigned char* vt = sm + S_V + st * S_V_STRIDE;
                    tma_load_3d(vt, &maps.v, full, 0, j, tc);
                    tma_load_3d(vt + 8192, &maps.v, full, 64, j, tc);
                    bulk_load(sm + S_TU + st * S_TU_STRIDE, rec + PREP_TU, 8192, full);
                }
                issued = k + 1;
            }
            // drain: every issued load has landed before the CTA may exit
            for (int k = max(0, issued - 2); k < issued; ++k)
                mbar_wait(&bars[B_FULL0 + (k & 1)], (k >> 1) & 1);
        }
        __syncwarp();
    } else if (w == 1) {
        // ------------------------------------------------------------ state-chain MMA issuer
        // per chunk k: [V'|Q h] (V' alone without an output side), then the state update; U
        // of each chunk comes from warp 3.  Lane 0 alone runs the loop: issued from
        // warp-uniform code (elect.sync) the MMAs leave the tensor pipe sooner, but the whole
        // scan runs slower (the state warps that share this warp's SMSP lose issue slots).
        if (lane == 0) {
            constexpr uint32_t IDV = make_idesc(128, OUT ? 128 : 64, 0, 0);
            constexpr uint32_t ID5 = make_idesc(128, 128, 0, 1);
            const uint32_t k0a = smem_addr(sm + S_K), wq0 = smem_addr(sm + S_WQ);
            bool ok = true;
            for (int k = 0; ok && k < n; ++k) {
                const int st = k & 1;
                const uint32_t dd = tm + t_dd(k);
                const uint64_t dWQ = kdesc(wq0 + st * S_WQ_STRIDE), dK = mdesc(k0a + st * S_K_STRIDE, 8192);
                TRACE(k, 0);
                if ((!NEEDU && !wait_bar(bars, B_FULL0 + st, (k >> 1) & 1, errflag)) ||
                    (NEEDU && !wait_bar(bars, B_U0 + st, (k >> 1) & 1, errflag)) ||
                    !wait_bar(bars, B_EX, k & 1, errflag)) {
                    ok = false;
                    break;
                }
                TRACE(k, 1);
                fence_after_sync();
                // [V'^T | (Q h)^T] in one product over [W'; Q]; the (Q h)^T half of this DD
                // buffer last held chunk k-2's, read (and cleared) by its output warps
                if (OUT && k >= 2 && !wait_bar(bars, B_EPI0 + (k & 1), ((k - 2) >> 1) & 1, errflag)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_bf16_ta(dd, tm + T_XB + 8 * s, dWQ + (off >> 4), IDV, (NEEDU || s > 0) ? 1u : 0u);
                }
                commit(&bars[B_MMA3]);
                TRACE(k, 2);
                if (!wait_bar(bars, B_EV0 + (k & 1), (k >> 1) & 1, errflag)) { ok = false; break; }
                TRACE(k, 4);
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16_ta(tm + T_XF, dd + (OUT ? kd_col(s) : p_col(s)), dK + (s * 2048 >> 4), ID5, 1u);
                commit(&bars[B_MMA5]);
                if (NEEDU) commit(&bars[B_M5C0 + (k & 1)]);
                commit(&bars[B_EMPTY0 + st]);  // last reader of this stage on this issuer
                TRACE(k, 5);
                TRACE(k, 7);
            }
            // drain: every MMA issued here has completed before TMEM may be released
            commit(&bars[B_DRAIN]);
            mbar_wait(&bars[B_DRAIN], 0);
        }
        __syncwarp();
    } else if (w == 2) {
        // ------------------------------------------------------------ gates
        float lb_run = 0.f;  // sum of the own chunks' transition log-bounds so far (rule)
        bool bad = rule && rule->lj >= 1 && rule->e_own == 0, ext_ok = true, nm = false;
        for (int k = 0; k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const int64_t tc = t0 + int64_t(cb + k) * CH;
            const int c = int((t1 - tc) < int64_t(CH) ? (t1 - tc) : int64_t(CH));
            float gv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // issue the global loads before waiting for a buffer
                const int r = 2 * lane + u;
                gv[u] = r < c ? P.g[(tc + r) * P.Hv + j] : 0.f;
            }
            int store = 1;
            if (rule) {
                if (k < rule->n_own) {
                    const float lb = P.logb[(hist_base + cb + k) * P.Hv + j];
                    if (rule->lj >= 1) {
                        if (rule->e_own == 0 || k < rule->e_own) {
                            store = 0;
                        } else {
                            store = lb_run < LOG_NEGLIGIBLE ? 1 : 0;  // (NaN: not negligible)
                            if (!store) bad = true;
                        }
                    }
                    lb_run += lb;
                    if (k == rule->n_own - 1) {
                        nm = !(lb_run < LOG_NEGLIGIBLE);
                        ext_ok = rule->lj == 0 || !nm;
                    }
                } else {
                    store = ext_ok ? 1 : 0;
                }
            }
            TRACE(k, 21);
            if (k >= NGATE && !warp_wait<true>(bars, B_GFREE0 + gs, ((k - NGATE) >> 2) & 1, errflag)) break;
            TRACE(k, 22);
            Gate& gb = gates[gs];
            float run0 = gv[0], run1 = gv[0] + gv[1];
            float tot = run1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, tot, off);
                if (lane >= off) tot += y;
            }
            const float excl = tot - run1;
            const float last = __shfl_sync(0xffffffffu, tot, 31);
            const float gm[2] = {run0 + excl, run1 + excl};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                gb.gam[r] = gm[u];
                gb.e[r] = expf(gm[u]);
                gb.kd[r] = expf(last - gm[u]);
            }
            if (lane == 0) {
                gb.eC = expf(last);
                gb.c = c;
                gb.store = store;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_GATE0 + gs]);
            TRACE(k, 23);
        }
        if (rule && lane == 0) {  // (the first segment's dec serves the backward's reverse scan)
            if (rule->dec) *rule->dec = nm ? -1 : 0;
            *rule->rerun = bad ? 1 : 0;
        }
    } else if (w == 3 && OUT) {
        // ------------------------------------------------------------ output MMA issuer
        // D4b = (P V')^T once V' of chunk k is converted and the output warps have read D4b
        // of chunk k-1; U of chunk k+1 before that, right after the last reader of its buffer
        // (the P V' product of chunk k-1, issued here), so the state chain never waits on it.
        if (lane == 0) {
            constexpr uint32_t ID4 = make_idesc(128, 64, 0, 0);
            const uint32_t p0 = smem_addr(sm + S_P);
            auto load_p = [&](int q) {  // P of chunk q into ring slot q % NP
                const int b = q % NP;
                const unsigned char* rec = static_cast<const unsigned char*>(P.prep) +
                                           ((hist_base + cb + q) * P.Hv + j) * P.prep_stride;
                mbar_expect_tx(&bars[B_FULLP0 + b], 8192);
                bulk_load(sm + S_P + b * S_P_STRIDE, rec + PREP_P, 8192, &bars[B_FULLP0 + b]);
            };
            constexpr uint32_t IDU = make_idesc(128, 64, 1, 0);
            const uint32_t v0a = smem_addr(sm + S_V), tu0 = smem_addr(sm + S_TU);
            // U^T = V^T TU^T of chunk q into the V' half of its DD buffer, whose last reader
            // (the P V' product of chunk q-2) was issued here before
            auto issue_u = [&](int q) {
                const int st = q & 1;
                const uint64_t dV = mdesc(v0a + st * S_V_STRIDE, 8192), dTU = kdesc(tu0 + st * S_TU_STRIDE);
                TRACE(q, 8);
                if (!wait_bar(bars, B_FULL0 + st, (q >> 1) & 1, errflag)) return false;
                TRACE(q, 6);
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + t_dd(q), dV + (s * 2048 >> 4), dTU + (s * 32 >> 4), IDU, s > 0);
                commit(&bars[B_U0 + st]);
                return true;
            };
            int issued = 0, used = 0;
            for (; issued < NP - 1 && issued < n; ++issued) load_p(issued);
            bool uok = n > 0 ? issue_u(0) : true;
            for (int k = 0; uok && k < n; ++k) {
                const int b = k % NP;
                if (k + 1 < n && !issue_u(k + 1)) break;
                if (!wait_bar(bars, B_FULLP0 + b, (k / NP) & 1, errflag)) break;
                used = k + 1;
                if (k >= 1 && !wait_bar(bars, B_EPI0 + ((k - 1) & 1), ((k - 1) >> 1) & 1, errflag)) break;
                // after the state update of chunk k (so P V' never queues ahead of it); V' of
                // chunk k is converted by then as well
                if (!wait_bar(bars, B_M5C0 + (k & 1), (k >> 1) & 1, errflag)) break;
                TRACE(k, 10);
                fence_after_sync();
                const uint32_t dd = tm + t_dd(k);
                const uint64_t dP = kdesc(p0 + b * S_P_STRIDE);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16_ta(tm + T_D4B, dd + p_col(s), dP + (s * 32 >> 4), ID4, s > 0);
                commit(&bars[B_MMA4_0 + (k & 1)]);
                commit(&bars[B_EMPTYP0 + b]);
                TRACE(k, 11);
                const int q = k + NP - 1;  // refill the slot chunk k-1 used
                if (q < n) {
                    if (q >= NP && !wait_bar(bars, B_EMPTYP0 + q % NP, ((q - NP) / NP) & 1, errflag)) break;
                    load_p(q);
                    issued = q + 1;
                }
            }
            for (int q = used; q < issued; ++q) mbar_wait(&bars[B_FULLP0 + q % NP], (q / NP) & 1);
            commit(&bars[B_DRAIN]);
        }
        __syncwarp();
    } else if (w == 3 && NEEDU) {
        // ------------------------------------------------------------ U issuer (no output side)
        // U of chunk k+1 once the state update of chunk k-1, the last reader of its buffer, has
        // completed (and its tiles have landed), so the state chain never waits on it
        if (lane == 0) {
            constexpr uint32_t IDU = make_idesc(128, 64, 1, 0);
            const uint32_t v0a = smem_addr(sm + S_V), tu0 = smem_addr(sm + S_TU);
            for (int q = 0; q < n; ++q) {
                const int st = q & 1;
                if (q >= 2 && !wait_bar(bars, B_M5C0 + st, ((q - 2) >> 1) & 1, errflag)) break;
                if (!wait_bar(bars, B_FULL0 + st, (q >> 1) & 1, errflag)) break;
                fence_after_sync();
                const uint64_t dV = mdesc(v0a + st * S_V_STRIDE, 8192), dTU = kdesc(tu0 + st * S_TU_STRIDE);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + t_dd(q), dV + (s * 2048 >> 4), dTU + (s * 32 >> 4), IDU, s > 0);
                commit(&bars[B_U0 + st]);
            }
            commit(&bars[B_DRAIN]);
        }
        __syncwarp();
    } else if (w >= 4 && w < 12) {
        // ------------------------------------------------------------ state warps
        // two warpgroups, one per half of the key columns of the state (hf); each converts
        // the V' columns of its half of the chunk's tokens
        const int hf = w >= 8 ? 1 : 0;
        const int v = tid - (hf ? 256 : 128);        // TMEM lane = value column
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        init_state_half<KIND>(tm, lb, hf, v, x0);
        bool ok = true;
        for (int k = 0; ok && k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!warp_wait(bars, B_GATE0 + gs, (k >> 2) & 1, errflag)) { ok = false; break; }
            if (v == 0 && !hf) TRACE(k, 16);
            if (k >= 1) {
                if (!warp_wait(bars, B_MMA5, (k - 1) & 1, errflag)) { ok = false; break; }
                fence_after_sync();
            }
            if (v == 0 && !hf) TRACE(k, 17);
            {
                float xs[64];
                state_bf16_half(tm, lb, T_XB, hf, T_XF, xs);
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_EX]);
                if (rule && rule->x_mid && k == rule->n_own) {
                    // the state at the end of the own segment (read again from TMEM in a rolled
                    // loop: once per scan, so the loop body's code stays small)
#pragma unroll 1
                    for (int c0 = 64 * hf; c0 < 64 * hf + 64; c0 += 16) {
                        float xv[16];
                        tmem_ld16(tm + lb + T_XF + c0, xv);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) rule->x_mid[(c0 + i) * VD + v] = xv[i];
                    }
                }
                state_decay_half<KIND>(P, tm, lb, hf, v, gb.eC, hist_base + cb + k, j, T_XF, xs,
                                       gb.store != 0);
            }
            if (v == 0 && !hf) TRACE(k, 18);
            // V' of tokens [32 hf, 32 hf + 32): fp32 -> bf16 V'^T and bf16 diag(kd) V'^T, both
            // inside the 32 columns just read (no other warp touches them)
            if (!warp_wait(bars, B_MMA3, k & 1, errflag)) { ok = false; break; }
            if (v == 0 && !hf) TRACE(k, 19);
            fence_after_sync();
            const uint32_t d3 = tm + lb + t_dd(k) + 32 * hf;
            float vp[32];
            tmem_ld32(d3, vp);
            tmem_ld_wait();
            float p1[16], h1[16], kd[32];
            {
                const uint32_t ka = smem_addr(&gb.kd[32 * hf]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 f = lds128f(ka + 16 * i);
                    kd[4 * i] = f.x;
                    kd[4 * i + 1] = f.y;
                    kd[4 * i + 2] = f.z;
                    kd[4 * i + 3] = f.w;
                }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = vp[2 * i], b = vp[2 * i + 1];
                p1[i] = __uint_as_float(pack_bf16(a, b));
                h1[i] = __uint_as_float(pack_bf16(a * kd[2 * i], b * kd[2 * i + 1]));
            }
            if (OUT) {
                tmem_st16(d3, p1);
                tmem_st16(d3 + 16, h1);
            } else {  // only diag(kd) V' is read again (by the state update)
                tmem_st16(d3, h1);
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_EV0 + (k & 1)]);
                mbar_arrive(&bars[B_GFREE0 + gs]);  // done with this chunk's gates
            }
            if (v == 0 && !hf) TRACE(k, 20);
        }
        if (ok && warp_wait(bars, B_MMA5, (n - 1) & 1, errflag)) {
            fence_after_sync();
            if (x_out) {
                for (int c0 = 64 * hf; c0 < 64 * hf + 64; c0 += 16) {
                    float xv[16];
                    tmem_ld16(tm + lb + T_XF + c0, xv);
                    tmem_ld_wait();
                    if (KIND == TK_TRANS) {  // segment transitions are stored transposed (M^T)
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(x_out + v * VD + c0 + i) =
                                make_float4(xv[i], xv[i + 1], xv[i + 2], xv[i + 3]);
                        if (x_out_t) {  // and untransposed, for the backward's reverse fix-up
#pragma unroll
                            for (int i = 0; i < 16; ++i) x_out_t[(c0 + i) * VD + v] = xv[i];
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) x_out[(c0 + i) * VD + v] = xv[i];
                    }
                }
            }
        }
    } else if (w >= 12 && OUT) {
        // ------------------------------------------------------------ output warps
        // per chunk: read (Q h)^T (clearing it) and D4b, then O = scale (e (Q h) + P V')
        const int v = tid - 384;                     // TMEM lane = value column
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        const uint32_t so = smem_addr(sm + S_O);
        for (int k = 0; k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!named_and(2, 128, warp_wait<true>(bars, B_GATE0 + gs, (k >> 2) & 1, errflag) &&
                                   warp_wait<true>(bars, B_MMA4_0 + (k & 1), (k >> 1) & 1, errflag)))
                break;
            if (v == 0) TRACE(k, 14);
            fence_after_sync();
            const float sc = P.scale;
            const uint32_t dqa = tm + lb + t_dd(k) + 64;
            const uint32_t ge = smem_addr(&gb.e[0]);
            // a rolled loop over four 16-column groups: this role's code stays small (the 16
            // warps' roles share each SMSP's instruction cache)
            float z16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z16[i] = 0.f;
#pragma unroll 1
            for (int g4 = 0; g4 < 4; ++g4) {
                float qa[16], pb[16];
                tmem_ld16(dqa + 16 * g4, qa);
                tmem_ld16(tm + lb + T_D4B + 16 * g4, pb);
                tmem_ld_wait();
                tmem_st16(dqa + 16 * g4, z16);  // clear for the chunk that reuses this buffer
                float ev[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 e4 = lds128f(ge + 4 * (16 * g4 + 4 * i));
                    ev[4 * i] = e4.x;
                    ev[4 * i + 1] = e4.y;
                    ev[4 * i + 2] = e4.z;
                    ev[4 * i + 3] = e4.w;
                }
                const uint32_t sb = so + ((16 * g4) * LDO + v) * 2;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    sts16(sb + u * LDO * 2,
                          __bfloat16_as_ushort(__float2bfloat16_rn(sc * fmaf(ev[u], qa[u], pb[u]))));
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EPI0 + (k & 1)]);
            if (v == 0) TRACE(k, 28);
            named_sync(2, 128);
            // rows of O leave as 16-byte vectors (only the rows of this sequence)
            const int64_t tc = t0 + int64_t(cb + k) * CH;
            const int c = gb.c;
            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(P.o) + (tc * P.Hv + j) * VD;
            const int64_t rs = int64_t(P.Hv) * VD;
            const int64_t o_n = (P.cu ? int64_t(P.T) : int64_t(P.N) * P.T) * rs;
            for (int idx = v; idx < (gb.store ? c * 16 : 0); idx += 128) {
                const int r = idx >> 4, cv = idx & 15;
                if (in_range((tc * P.Hv + j) * VD + r * rs + cv * 8 + 7, o_n, P.err))
                    *reinterpret_cast<uint4*>(ob + r * rs + cv * 8) = lds128(so + (r * LDO + cv * 8) * 2);
            }
            named_sync(2, 128);
            if (lane == 0) mbar_arrive(&bars[B_GFREE0 + gs]);  // done with this chunk's gates
            if (v == 0) TRACE(k, 15);
        }
    }

    fence_before_sync();
    __syncthreads();
    if (*errflag && tid == 0 && P.err) atomicOr(P.err, *errflag);
    if (w == 0) {
        fence_after_sync();
        tmem_dealloc(tm, 512);
    }
}

// Exact context parallelism, first phase, for a segment past the first: the segment's state
// from zero (S) and its transition (M, from the identity) share the chunk tiles and run as two
// independent chains in one CTA, so that the tensor-core work of one chain overlaps the
// CUDA-core hand-offs of the other.  Tensor memory: S chain at columns [0, 256), M chain at
// [256, 512) (fp32 state, bf16 copy, one V' buffer each).
//
// Warp roles: 0 TMA producer; 1 MMA issuer of S (U, V', state update); 2 gates; 3 MMA issuer
// of M (V', state update); 4-11 state warps of S (one warpgroup per half of the key columns);
// 12-15 state warps of M (both halves).
constexpr uint32_t PM = 256;  // tensor-memory column offset of the M chain
__device__ void tc_scan_pair(const Problem& P, const TcMaps& maps, unsigned char* sm, int j,
                             int64_t t0, int64_t t1, int cb, int ce, float* s_out, float* m_out,
                             float* m_out_t, int64_t hist_base) {
    enum PB { Q_FULL0 = 0, Q_FULL1, Q_EMPTY0, Q_EMPTY1, Q_GATE0, Q_GFREE0 = Q_GATE0 + NGATE,
              Q_MMA3S = Q_GFREE0 + NGATE, Q_MMA5S, Q_MMA3M, Q_MMA5M, Q_EXS, Q_EVS, Q_EXM, Q_EVM,
              Q_DRAIN, Q_COUNT };
    static_assert(Q_COUNT * 8 + 8 <= 512, "barrier area");
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + Q_COUNT * 8);
    int* errflag = reinterpret_cast<int*>(sm + S_BAR + Q_COUNT * 8 + 4);
    Gate* gates = reinterpret_cast<Gate*>(sm + S_GATE);
    const int G = P.Hv / P.Hqk, qh = j / G;
    const int n = ce - cb;
    constexpr uint32_t S_DD = 192, M_XF = PM + T_XF, M_XB = PM + T_XB, M_DD = PM + 192;

    if (tid == 0) {
        mbar_init(&bars[Q_FULL0], 1);
        mbar_init(&bars[Q_FULL1], 1);
        mbar_init(&bars[Q_EMPTY0], 2);  // released by both issuers
        mbar_init(&bars[Q_EMPTY1], 2);
        for (int b = 0; b < NGATE; ++b) {
            mbar_init(&bars[Q_GATE0 + b], 1);
            mbar_init(&bars[Q_GFREE0 + b], 12);
        }
        mbar_init(&bars[Q_MMA3S], 1);
        mbar_init(&bars[Q_MMA5S], 1);
        mbar_init(&bars[Q_MMA3M], 1);
        mbar_init(&bars[Q_MMA5M], 1);
        mbar_init(&bars[Q_EXS], 8);
        mbar_init(&bars[Q_EVS], 8);
        mbar_init(&bars[Q_EXM], 4);
        mbar_init(&bars[Q_EVM], 4);
        mbar_init(&bars[Q_DRAIN], 2);
        *errflag = 0;
        mbar_fence_init();
    }
    if (w == 0) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    CTRACE(0, 2);
    const uint32_t tm = *tmem_slot;
    const uint32_t k0a = smem_addr(sm + S_K), wq0 = smem_addr(sm + S_WQ);

    if (w == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t bytes = 16384u + 16384u + 16384u + 8192u;
            int issued = 0;
            for (int k = 0; k < n; ++k) {
                const int st = k & 1;
                if (k >= 2 && !wait_bar_lazy(bars, Q_EMPTY0 + st, ((k - 2) >> 1) & 1, errflag)) break;
                const int tc = int(t0 + int64_t(cb + k) * CH);
                uint64_t* full = &bars[Q_FULL0 + st];
                unsigned char* kt = sm + S_K + st * S_K_STRIDE;
                unsigned char* wq = sm + S_WQ + st * S_WQ_STRIDE;
                unsigned char* vt = sm + S_V + st * S_V_STRIDE;
                const unsigned char* rec = static_cast<const unsigned char*>(P.prep) +
                                           ((hist_base + cb + k) * P.Hv + j) * P.prep_stride;
                mbar_expect_tx(full, bytes);
                tma_load_3d(kt, &maps.k, full, 0, qh, tc);
                tma_load_3d(kt + 8192, &maps.k, full, 64, qh, tc);
                bulk_load(wq, rec + PREP_W, 8192, full);
                bulk_load(wq + 16384, rec + PREP_W + 8192, 8192, full);
                tma_load_3d(vt, &maps.v, full, 0, j, tc);
                tma_load_3d(vt + 8192, &maps.v, full, 64, j, tc);
                bulk_load(sm + S_TU + st * S_TU_STRIDE, rec + PREP_TU, 8192, full);
                issued = k + 1;
            }
            for (int k = max(0, issued - 2); k < issued; ++k)
                mbar_wait(&bars[Q_FULL0 + (k & 1)], (k >> 1) & 1);
        }
        __syncwarp();
    } else if (w == 1 || w == 3) {
        // ------------------------------------------------------------ MMA issuers (S: w1, M: w3)
        if (lane == 0) {
            const bool isS = w == 1;
            constexpr uint32_t IDU = make_idesc(128, 64, 1, 0);
            constexpr uint32_t IDV = make_idesc(128, 64, 0, 0);
            constexpr uint32_t ID5 = make_idesc(128, 128, 0, 1);
            const uint32_t v0a = smem_addr(sm + S_V), tu0 = smem_addr(sm + S_TU);
            const uint64_t dK[2] = {mdesc(k0a, 8192), mdesc(k0a + S_K_STRIDE, 8192)};
            const uint64_t dWQ[2] = {kdesc(wq0), kdesc(wq0 + S_WQ_STRIDE)};
            const uint64_t dV[2] = {mdesc(v0a, 8192), mdesc(v0a + S_V_STRIDE, 8192)};
            const uint64_t dTU[2] = {kdesc(tu0), kdesc(tu0 + S_TU_STRIDE)};
            const uint32_t xf = tm + (isS ? T_XF : M_XF), xb = tm + (isS ? T_XB : M_XB);
            const uint32_t dd = tm + (isS ? S_DD : M_DD);
            const int bEX = isS ? Q_EXS : Q_EXM, bEV = isS ? Q_EVS : Q_EVM;
            const int b3 = isS ? Q_MMA3S : Q_MMA3M, b5 = isS ? Q_MMA5S : Q_MMA5M;
            auto issue_u = [&](int k) {
                const int st = k & 1;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(dd, (st ? dV[1] : dV[0]) + (s * 2048 >> 4), (st ? dTU[1] : dTU[0]) + (s * 32 >> 4),
                             IDU, s > 0);
            };
            bool ok = true;
            if (isS) {
                ok = wait_bar(bars, Q_FULL0, 0, errflag);
                if (ok) {
                    fence_after_sync();
                    issue_u(0);
                }
            }
            for (int k = 0; ok && k < n; ++k) {
                const int st = k & 1;
                if ((!isS && !wait_bar(bars, Q_FULL0 + st, (k >> 1) & 1, errflag)) ||
                    !wait_bar(bars, bEX, k & 1, errflag)) {
                    ok = false;
                    break;
                }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_bf16_ta(dd, xb + 8 * s, (st ? dWQ[1] : dWQ[0]) + (off >> 4), IDV, (isS || s > 0) ? 1u : 0u);
                }
                commit(&bars[b3]);
                if (!wait_bar(bars, bEV, k & 1, errflag)) { ok = false; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16_ta(xf, dd + p_col(s), (st ? dK[1] : dK[0]) + (s * 2048 >> 4), ID5, 1u);
                commit(&bars[b5]);
                commit(&bars[Q_EMPTY0 + st]);
                if (isS && k + 1 < n) {
                    if (!wait_bar(bars, Q_FULL0 + ((k + 1) & 1), ((k + 1) >> 1) & 1, errflag)) {
                        ok = false;
                        break;
                    }
                    fence_after_sync();
                    issue_u(k + 1);
                }
            }
            commit(&bars[Q_DRAIN]);
            if (isS) mbar_wait(&bars[Q_DRAIN], 0);
        }
        __syncwarp();
    } else if (w == 2) {
        // ------------------------------------------------------------ gates
        for (int k = 0; k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const int64_t tc = t0 + int64_t(cb + k) * CH;
            const int c = int((t1 - tc) < int64_t(CH) ? (t1 - tc) : int64_t(CH));
            float gv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                gv[u] = r < c ? P.g[(tc + r) * P.Hv + j] : 0.f;
            }
            if (k >= NGATE && !warp_wait<true>(bars, Q_GFREE0 + gs, ((k - NGATE) >> 2) & 1, errflag)) break;
            Gate& gb = gates[gs];
            float run0 = gv[0], run1 = gv[0] + gv[1];
            float tot = run1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, tot, off);
                if (lane >= off) tot += y;
            }
            const float excl = tot - run1;
            const float last = __shfl_sync(0xffffffffu, tot, 31);
            const float gm[2] = {run0 + excl, run1 + excl};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                gb.gam[r] = gm[u];
                gb.e[r] = expf(gm[u]);
                gb.kd[r] = expf(last - gm[u]);
            }
            if (lane == 0) {
                gb.eC = expf(last);
                gb.c = c;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Q_GATE0 + gs]);
        }
    } else {
        // ------------------------------------------------------------ state warps
        // S: warps 4-11, one warpgroup per key half and per half of the chunk's tokens;
        // M: warps 12-15, everything
        const bool isS = w < 12;
        const int hf = (w >= 8 && w < 12) ? 1 : 0;
        const int v = tid & 127;                     // TMEM lane = value column
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        const uint32_t xf = isS ? T_XF : M_XF, xb = isS ? T_XB : M_XB, ddc = isS ? S_DD : M_DD;
        const int bEX = isS ? Q_EXS : Q_EXM, bEV = isS ? Q_EVS : Q_EVM;
        const int b3 = isS ? Q_MMA3S : Q_MMA3M, b5 = isS ? Q_MMA5S : Q_MMA5M;
        if (isS) {
            init_state_half<TK_STATE>(tm, lb, hf, v, nullptr, xf);
        } else {
            init_state_half<TK_TRANS>(tm, lb, 0, v, nullptr, xf);
            init_state_half<TK_TRANS>(tm, lb, 1, v, nullptr, xf);
        }
        bool ok = true;
        for (int k = 0; ok && k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!warp_wait(bars, Q_GATE0 + gs, (k >> 2) & 1, errflag)) { ok = false; break; }
            if (k >= 1) {
                if (!warp_wait(bars, b5, (k - 1) & 1, errflag)) { ok = false; break; }
                fence_after_sync();
            }
            if (isS) {
                float xs[64];
                state_bf16_half(tm, lb, xb, hf, xf, xs);
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[bEX]);
                state_decay_half<TK_STATE>(P, tm, lb, hf, v, gb.eC, 0, j, xf, xs);
            } else {
                state_bf16_all(tm, lb, xb, xf);
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[bEX]);
                state_decay_all(tm, lb, xf, gb.eC);
            }
            if (!warp_wait(bars, b3, k & 1, errflag)) { ok = false; break; }
            fence_after_sync();
            // diag(kd) V' in bf16 over the fp32 V' of the same tokens (S: one half of them)
            for (int th = isS ? hf : 0; th < (isS ? hf + 1 : 2); ++th) {
                const uint32_t d3 = tm + lb + ddc + 32 * th;
                float vp[32], h1[16];
                tmem_ld32(d3, vp);
                const uint32_t ka = smem_addr(&gb.kd[32 * th]);
                float kd[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 f = lds128f(ka + 16 * i);
                    kd[4 * i] = f.x;
                    kd[4 * i + 1] = f.y;
                    kd[4 * i + 2] = f.z;
                    kd[4 * i + 3] = f.w;
                }
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    h1[i] = __uint_as_float(pack_bf16(vp[2 * i] * kd[2 * i], vp[2 * i + 1] * kd[2 * i + 1]));
                tmem_st16(d3, h1);
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[bEV]);
                mbar_arrive(&bars[Q_GFREE0 + gs]);
            }
        }
        if (ok && warp_wait(bars, b5, (n - 1) & 1, errflag)) {
            fence_after_sync();
            float* out = isS ? s_out : m_out;
            const int c_lo = isS ? 64 * hf : 0, c_hi = isS ? 64 * hf + 64 : 128;
            for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
                float xv[16];
                tmem_ld16(tm + lb + xf + c0, xv);
                tmem_ld_wait();
                if (!isS) {  // transitions are stored transposed (M^T), and for the backward also as M
#pragma unroll
                    for (int i = 0; i < 16; i += 4)
                        *reinterpret_cast<float4*>(out + v * VD + c0 + i) =
                            make_float4(xv[i], xv[i + 1], xv[i + 2], xv[i + 3]);
                    if (m_out_t) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) m_out_t[(c0 + i) * VD + v] = xv[i];
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) out[(c0 + i) * VD + v] = xv[i];
                }
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (*errflag && tid == 0 && P.err) atomicOr(P.err, *errflag);
    if (w == 0) {
        fence_after_sync();
        tmem_dealloc(tm, 512);
    }
}

__device__ __forceinline__ unsigned char* aligned_smem() {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void seq_range(const Problem& P, int s, int64_t& t0, int64_t& t1) {
    if (P.cu) {
        t0 = P.cu[s];
        t1 = P.cu[s + 1];
    } else {
        t0 = int64_t(s) * P.T;
        t1 = t0 + P.T;
    }
}

constexpr int64_t KVN = int64_t(KD) * VD;

// copy (or zero / identity) a state without touching the tensor cores (empty ranges)
__device__ void copy_state(const float* x0, float* x_out, bool ident) {
    if (!x_out) return;
    for (int i = threadIdx.x; i < KD * VD; i += blockDim.x)
        x_out[i] = x0 ? x0[i] : ((ident && (i / VD) == (i % VD)) ? 1.f : 0.f);
}

__global__ void __launch_bounds__(TCT, 1) k_tc_phase_a(Problem P, const __grid_constant__ TcMaps maps) {
    CTRACE(0, 0);
    pdl_launch_dependents();
    pdl_wait();
    CTRACE(0, 1);
    unsigned char* sm = aligned_smem();
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) return;
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + CH - 1) / CH);
    const float* h0 = P.h0 ? P.h0 + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    if (P.cp == CP_EXACT && !P.full_cp) {
        // decay-bounded exact mode: only the transitions that are not negligible, of the
        // segments between the first and the last (the first output pass has stored every
        // segment's state from zero, S, where the fix-up reads it)
        if (lj < 1 || lj >= nseg - 1) return;
        if (P.dec[int64_t(gseg) * P.Hv + j] >= 0) return;
        const int cb = lj * P.L, ce = min(cb + P.L, nt);
        float* mout = P.mbuf + (int64_t(gseg) * P.Hv + j) * KVN;
        float* mout_t = P.mbuf_t ? P.mbuf_t + (int64_t(gseg) * P.Hv + j) * KVN : nullptr;
        tc_scan<TK_TRANS>(P, maps, sm, j, t0, t1, cb, ce, nullptr, mout, plan_chunk_off(P.plan, s), mout_t);
        return;
    }
    if (P.cp == CP_EXACT) {
        if (lj >= nseg - 1) return;
        const int cb = lj * P.L, ce = min(cb + P.L, nt);
        float* out = P.hin + (int64_t(gseg + 1) * P.Hv + j) * KVN;
        if (lj == 0) {  // the first segment starts from h0 and needs no transition
            if (ce <= cb) { copy_state(h0, out, false); return; }
            tc_scan<TK_STATE>(P, maps, sm, j, t0, t1, cb, ce, h0, out, plan_chunk_off(P.plan, s));
        } else {
            float* mout = P.mbuf + (int64_t(gseg) * P.Hv + j) * KVN;
            float* mout_t = P.mbuf_t ? P.mbuf_t + (int64_t(gseg) * P.Hv + j) * KVN : nullptr;
            if (ce <= cb) {
                copy_state(nullptr, out, false);
                copy_state(nullptr, mout, true);
                if (mout_t) copy_state(nullptr, mout_t, true);
                return;
            }
            tc_scan_pair(P, maps, sm, j, t0, t1, cb, ce, out, mout, mout_t, plan_chunk_off(P.plan, s));
            CTRACE(0, 3);
        }
    } else {
        if (lj == 0) return;
        const int cb = lj * P.L, w0 = cb - P.warmup;
        const float* x0 = w0 <= 0 ? h0 : nullptr;
        float* out = P.hin + (int64_t(gseg) * P.Hv + j) * KVN;
        tc_scan<TK_STATE>(P, maps, sm, j, t0, t1, max(w0, 0), cb, x0, out, plan_chunk_off(P.plan, s));
    }
}

// g-only extension length of a segment starting at chunk cs with n chunks: the smallest e in
// [1, min(n, EXT_MAX)] whose first e chunks' gate sum is below LOG_NEGLIGIBLE, else 0.  Since
// beta |k|^2 terms only raise a chunk's log-bound above its gate sum, chunks before e are
// certainly not decoupled from the segment's entering state.  Every warp computes it with the
// same code and summation order, so the CTA of segment lj (looking ahead) and that of lj + 1
// (looking at itself) agree bit for bit.  In two steps (the gate loads, ext_load, then the sum,
// ext_sum), so that a caller that needs two lengths issues all their loads at once.
constexpr int EXT_MAX = 4;
__device__ __forceinline__ void ext_load(const Problem& P, int64_t t0, int64_t t1, int cs, int n, int j,
                                         float (&gv)[EXT_MAX][2]) {
    const int lane = threadIdx.x & 31;
    const int m = min(n, EXT_MAX);
#pragma unroll
    for (int e = 0; e < EXT_MAX; ++e)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t t = t0 + int64_t(cs + e) * CH + 2 * lane + u;
            gv[e][u] = (e < m && t < t1) ? P.g[t * P.Hv + j] : 0.f;
        }
}
__device__ __forceinline__ int ext_sum(const float (&gv)[EXT_MAX][2], int n) {
    const int m = min(n, EXT_MAX);
    float run = 0.f;
#pragma unroll
    for (int e = 0; e < EXT_MAX; ++e) {
        if (e >= m) break;
        float v = gv[e][0] + gv[e][1];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        run += v;
        if (run < LOG_NEGLIGIBLE) return e + 1;
    }
    return 0;
}

// Output stage (KIND = TK_OUT) or the backward's recompute of the state entering every chunk
// (TK_HIST), one CTA per (segment, v-head).  mode 0: every segment from its entering state
// (h0, or the fix-up's), the last one's final state to ht.  Decay-bounded exact mode: mode 1,
// the first pass, runs every segment from h0 (the first) or from zero (the others) and stores
// only the results that provably do not depend on that start (ScanRule); the leading chunks of
// segment lj + 1 that the bound does not reach are scanned by the CTA of segment lj right after
// its own, from its own final state -- the true entering state of lj + 1 when lj's transition
// is negligible (or lj is the first).  Each segment's state from zero, S, goes to the entering
// slot of the next (the last one's to ht), with the decisions (P.dec, P.rerun).  mode 2, the
// correction, reruns from its true entering state every segment with an unwritten result: one
// flagged by its own CTA, one that follows a segment whose transition is not negligible, and
// a last segment whose own transition is not negligible (its final state).
// (mode is a template parameter: each kernel holds one copy of the scan, whose code is larger
// than an SM's instruction cache)
template <int KIND, int MODE>
__global__ void __launch_bounds__(TCT, 1) k_tc_phase_c(Problem P, const __grid_constant__ TcMaps maps) {
    constexpr int mode = MODE;
    if (mode != 2) CTRACE(1, 0);
    pdl_launch_dependents();
    unsigned char* sm = aligned_smem();
    // the passes that scan in every CTA set up while the previous kernel finishes
    const bool pre = mode != 2;
    if (pre) tc_scan_setup<KIND>(sm);
    pdl_wait();
    if (mode != 2) CTRACE(1, 1);
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) {
        if (pre) tc_scan_release(sm);
        return;
    }
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + CH - 1) / CH);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const int64_t sjh = int64_t(gseg) * P.Hv + j;
    const bool last = lj == nseg - 1;
    const float* h0 = P.h0 ? P.h0 + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    float* ht = P.ht ? P.ht + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    if (mode == 1) {
        const float* x0 = lj == 0 ? h0 : nullptr;
        float* x_seg = last ? ht : P.hin + (sjh + P.Hv) * KVN;
        if (ce <= cb) {  // only an empty sequence
            copy_state(x0, x_seg, false);
            tc_scan_release(sm);
            return;
        }
        // both extension lengths from one round of gate loads
        const int n_own = lj >= 1 ? ce - cb : 0, n_next = last ? 0 : min(P.L, nt - ce);
        float g_own[EXT_MAX][2], g_next[EXT_MAX][2];
        ext_load(P, t0, t1, cb, n_own, j, g_own);
        ext_load(P, t0, t1, ce, n_next, j, g_next);
        ScanRule rule;
        rule.n_own = ce - cb;
        rule.e_own = lj >= 1 ? ext_sum(g_own, n_own) : 0;
        const int e_next = last ? 0 : ext_sum(g_next, n_next);
        rule.lj = lj;
        rule.dec = P.dec + sjh;
        rule.rerun = P.rerun + sjh;
        rule.x_mid = e_next > 0 ? x_seg : nullptr;
        tc_scan<KIND>(P, maps, sm, j, t0, t1, cb, ce + e_next, x0, e_next > 0 ? nullptr : x_seg,
                      plan_chunk_off(P.plan, s), nullptr, &rule, true);
        CTRACE(1, 3);
        return;
    }
    if (mode == 2) {
        if (lj == 0 || ce <= cb) return;
        if (!(P.rerun[sjh] != 0 || (lj >= 2 && P.dec[sjh - P.Hv] < 0) || (last && P.dec[sjh] < 0))) return;
        tc_scan<KIND>(P, maps, sm, j, t0, t1, cb, ce, P.hin + sjh * KVN, last ? ht : nullptr,
                      plan_chunk_off(P.plan, s));
        return;
    }
    const float* x0 = (lj == 0) ? h0 : P.hin + sjh * KVN;
    float* x_out = last ? ht : nullptr;
    if (ce <= cb) {
        copy_state(x0, x_out, false);
        tc_scan_release(sm);
        return;
    }
    tc_scan<KIND>(P, maps, sm, j, t0, t1, cb, ce, x0, x_out, plan_chunk_off(P.plan, s), nullptr, nullptr, true);
    CTRACE(1, 3);
}

// =====================================================================================
// Backward: the reverse dh scan on the tensor cores (bf16).  Per chunk, in reverse order,
// with dOs = scale dO, W' = -W and P from the forward's chunk records:
//     dV'^T   = dOs^T P + (dh^T K^T) diag(kd)                 (D_a off the chain, D_b on it)
//     dh_in^T = e_C dh^T + dOs^T diag(e) Q + dV'^T W'
// The state is kept transposed in TMEM (Xt[v][dk] = dh[dk][v], fp32 + bf16 copy), exactly like
// the forward scan.  Warp roles: 0 TMA producer; 1 MMA issuer; 2 gates; 4-11 state warps (one
// warpgroup per half of the key columns / of the chunk's tokens); 12-15 scale dO rows by
// scale e_i into the operand of the dOs^T diag(e) Q product (rows past the sequence end -> 0).
// =====================================================================================
constexpr uint32_t R_K = 0, R_Q = 32768, R_DO = 65536, R_DOE = 98304, R_W = 131072, R_P = 163840;
static_assert(R_P + 2 * 8192 <= S_GATE, "backward scan stages fit below the gate buffers");
constexpr uint32_t T_DB = 192, T_DA = 256;

// rule (or null: store everything): the first pass of the decay-bounded exact mode, in
// reverse.  The own segment is the first rule->n_own chunks of the scan (from its right end);
// the gate warp sums their transition log-bounds in scan order, and the gradient leaving a
// chunk is stored when the next segment's CTA does not store it (k >= e_own) and the sum over
// the chunks scanned before it is below LOG_NEGLIGIBLE (else the segment is left to the
// correction: rerun); the chunks past the own segment are stored when rule->ext_ok.
enum RB { R_FULL0 = 0, R_FULL1, R_EMPTY0, R_EMPTY1, R_GATE0, R_GFREE0 = R_GATE0 + NGATE,
          R_MMA3 = R_GFREE0 + NGATE, R_MMA5, R_EX, R_EV, R_DOE0, R_DOE1, R_DRAIN, R_DEC, R_COUNT };
static_assert(R_COUNT * 8 + 8 <= 512, "barrier area");
// The reverse scan's barriers and tensor memory (reads nothing an earlier kernel writes: may
// run before the wait for it; tc_bwd_release frees the tensor memory on a path that does not
// scan).
__device__ void tc_bwd_setup(unsigned char* sm) {
    const int tid = threadIdx.x, w = tid >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + R_COUNT * 8);
    int* errflag = reinterpret_cast<int*>(sm + S_BAR + R_COUNT * 8 + 4);
    if (tid == 0) {
        mbar_init(&bars[R_FULL0], 1);
        mbar_init(&bars[R_FULL1], 1);
        mbar_init(&bars[R_EMPTY0], 1);
        mbar_init(&bars[R_EMPTY1], 1);
        for (int b = 0; b < NGATE; ++b) {
            mbar_init(&bars[R_GATE0 + b], 1);
            mbar_init(&bars[R_GFREE0 + b], 12);  // 8 state warps + 4 dO-scaling warps
        }
        mbar_init(&bars[R_MMA3], 1);
        mbar_init(&bars[R_MMA5], 1);
        mbar_init(&bars[R_EX], 8);
        mbar_init(&bars[R_EV], 8);
        mbar_init(&bars[R_DOE0], 4);
        mbar_init(&bars[R_DOE1], 4);
        mbar_init(&bars[R_DRAIN], 1);
        mbar_init(&bars[R_DEC], 8);
        *errflag = 0;
        mbar_fence_init();
    }
    if (w == 0) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
}
__device__ void tc_bwd_release(unsigned char* sm) {
    fence_before_sync();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        fence_after_sync();
        tmem_dealloc(*reinterpret_cast<uint32_t*>(sm + S_BAR + R_COUNT * 8), 512);
    }
}

template <bool HIST>
__device__ void tc_bwd_scan(const BwdProblem& B, const TcMaps& maps, const CUtensorMap* mdo,
                            unsigned char* sm, int j, int64_t t0, int64_t t1, int cb, int ce,
                            const float* x0, float* x_out, int64_t gbase,
                            const ScanRule* rule = nullptr, bool ready = false) {
    const Problem& P = B.f;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + R_COUNT * 8);
    int* errflag = reinterpret_cast<int*>(sm + S_BAR + R_COUNT * 8 + 4);
    Gate* gates = reinterpret_cast<Gate*>(sm + S_GATE);
    const int G = P.Hv / P.Hqk, qh = j / G;
    const int n = ce - cb;
    const float sc = P.scale;
    auto chunk_of = [&](int k) { return ce - 1 - k; };  // reverse order

    if (!ready) tc_bwd_setup(sm);
    const uint32_t tm = *tmem_slot;

    if (w == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t bytes = 16384u * 4u + 8192u;
            int issued = 0;
            for (int k = 0; k < n; ++k) {
                const int st = k & 1;
                if (k >= 2 && !wait_bar_lazy(bars, R_EMPTY0 + st, ((k - 2) >> 1) & 1, errflag)) break;
                const int ch = chunk_of(k);
                const int tc = int(t0 + int64_t(ch) * CH);
                uint64_t* full = &bars[R_FULL0 + st];
                const unsigned char* rec = static_cast<const unsigned char*>(P.prep) +
                                           ((gbase + ch) * P.Hv + j) * P.prep_stride;
                unsigned char* kt = sm + R_K + st * 16384;
                unsigned char* qt = sm + R_Q + st * 16384;
                unsigned char* dt = sm + R_DO + st * 16384;
                unsigned char* wt = sm + R_W + st * 16384;
                mbar_expect_tx(full, bytes);
                tma_load_3d(kt, &maps.k, full, 0, qh, tc);
                tma_load_3d(kt + 8192, &maps.k, full, 64, qh, tc);
                tma_load_3d(qt, &maps.q, full, 0, qh, tc);
                tma_load_3d(qt + 8192, &maps.q, full, 64, qh, tc);
                tma_load_3d(dt, mdo, full, 0, j, tc);
                tma_load_3d(dt + 8192, mdo, full, 64, j, tc);
                bulk_load(wt, rec + PREP_W, 8192, full);
                bulk_load(wt + 8192, rec + PREP_W + 8192, 8192, full);
                bulk_load(sm + R_P + st * 8192, rec + PREP_P, 8192, full);
                issued = k + 1;
            }
            for (int k = max(0, issued - 2); k < issued; ++k)
                mbar_wait(&bars[R_FULL0 + (k & 1)], (k >> 1) & 1);
        }
        __syncwarp();
    } else if (w == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDA = make_idesc(128, 64, 1, 1);   // dO^T P
            constexpr uint32_t IDB = make_idesc(128, 64, 0, 0);   // Xt_bf16 K^T
            constexpr uint32_t IDX = make_idesc(128, 128, 1, 1);  // dOe^T Q
            constexpr uint32_t IDW = make_idesc(128, 128, 0, 1);  // dV'^T W'
            const uint32_t k0 = smem_addr(sm + R_K), q0 = smem_addr(sm + R_Q), d0 = smem_addr(sm + R_DO),
                           e0 = smem_addr(sm + R_DOE), w0 = smem_addr(sm + R_W), p0 = smem_addr(sm + R_P);
            const uint64_t dK[2] = {kdesc(k0), kdesc(k0 + 16384)};
            const uint64_t dQ[2] = {mdesc(q0, 8192), mdesc(q0 + 16384, 8192)};
            const uint64_t dD[2] = {mdesc(d0, 8192), mdesc(d0 + 16384, 8192)};
            const uint64_t dE[2] = {mdesc(e0, 8192), mdesc(e0 + 16384, 8192)};
            const uint64_t dW[2] = {mdesc(w0, 8192), mdesc(w0 + 16384, 8192)};
            const uint64_t dP[2] = {mdesc(p0, 8192), mdesc(p0 + 8192, 8192)};
            auto issue_da = [&](int k) {
                const int st = k & 1;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + T_DA, (st ? dD[1] : dD[0]) + (s * 2048 >> 4), (st ? dP[1] : dP[0]) + (s * 2048 >> 4),
                             IDA, s > 0);
            };
            bool ok = wait_bar(bars, R_FULL0, 0, errflag);
            if (ok) {
                fence_after_sync();
                issue_da(0);
            }
            for (int k = 0; ok && k < n; ++k) {
                const int st = k & 1;
                if (!wait_bar(bars, R_EX, k & 1, errflag)) { ok = false; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * 8192 + (s & 3) * 32;
                    mma_bf16_ta(tm + T_DB, tm + T_XB + 8 * s, (st ? dK[1] : dK[0]) + (off >> 4), IDB, s > 0);
                }
                commit(&bars[R_MMA3]);
                if (!wait_bar(bars, R_DOE0 + st, (k >> 1) & 1, errflag)) { ok = false; break; }
                // the state warps have decayed the fp32 state (after the hand-off arrival)
                if (!wait_bar(bars, R_DEC, k & 1, errflag)) { ok = false; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + T_XF, (st ? dE[1] : dE[0]) + (s * 2048 >> 4), (st ? dQ[1] : dQ[0]) + (s * 2048 >> 4),
                             IDX, 1u);
                if (!wait_bar(bars, R_EV, k & 1, errflag)) { ok = false; break; }
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16_ta(tm + T_XF, tm + T_DB + p_col(s), (st ? dW[1] : dW[0]) + (s * 2048 >> 4), IDW, 1u);
                commit(&bars[R_MMA5]);
                commit(&bars[R_EMPTY0 + st]);
                if (k + 1 < n) {
                    if (!wait_bar(bars, R_FULL0 + ((k + 1) & 1), ((k + 1) >> 1) & 1, errflag)) { ok = false; break; }
                    fence_after_sync();
                    issue_da(k + 1);
                }
            }
            commit(&bars[R_DRAIN]);
            mbar_wait(&bars[R_DRAIN], 0);
        }
        __syncwarp();
    } else if (w == 2) {
        // ------------------------------------------------------------ gates
        float lb_run = 0.f;
        bool bad = rule && rule->lj >= 1 && rule->e_own == 0;
        for (int k = 0; k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const int64_t tc = t0 + int64_t(chunk_of(k)) * CH;
            const int c = int((t1 - tc) < int64_t(CH) ? (t1 - tc) : int64_t(CH));
            float gv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                gv[u] = r < c ? P.g[(tc + r) * P.Hv + j] : 0.f;
            }
            int store = 1;
            if (rule) {
                if (k < rule->n_own) {
                    const float lb = P.logb[(gbase + chunk_of(k)) * P.Hv + j];
                    if (rule->lj >= 1) {
                        if (rule->e_own == 0 || k < rule->e_own) {
                            store = 0;
                        } else {
                            store = lb_run < LOG_NEGLIGIBLE ? 1 : 0;  // (NaN: not negligible)
                            if (!store) bad = true;
                        }
                    }
                    lb_run += lb;
                } else {
                    store = rule->ext_ok;
                }
            }
            if (k >= NGATE && !warp_wait<true>(bars, R_GFREE0 + gs, ((k - NGATE) >> 2) & 1, errflag)) break;
            Gate& gb = gates[gs];
            float run0 = gv[0], run1 = gv[0] + gv[1];
            float tot = run1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, tot, off);
                if (lane >= off) tot += y;
            }
            const float excl = tot - run1;
            const float last = __shfl_sync(0xffffffffu, tot, 31);
            const float gm[2] = {run0 + excl, run1 + excl};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                gb.gam[r] = gm[u];
                gb.e[r] = expf(gm[u]);
                gb.kd[r] = expf(last - gm[u]);
            }
            if (lane == 0) {
                gb.eC = expf(last);
                gb.c = c;
                gb.store = store;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[R_GATE0 + gs]);
        }
        if (rule && lane == 0) *rule->rerun = bad ? 1 : 0;
    } else if (w >= 12) {
        // ------------------------------------------------------------ dOe = scale e_i dO_i (i < c)
        const int v = tid - 384;
        for (int k = 0; k < n; ++k) {
            const int st = k & 1, gs = k & (NGATE - 1);
            if (!warp_wait<true>(bars, R_GATE0 + gs, (k >> 2) & 1, errflag) ||
                !warp_wait<true>(bars, R_FULL0 + st, (k >> 1) & 1, errflag))
                break;
            const Gate& gb = gates[gs];
            const uint32_t src = smem_addr(sm + R_DO + st * 16384), dst = smem_addr(sm + R_DOE + st * 16384);
            const uint32_t ge = smem_addr(&gb.e[0]);
            const int c = gb.c;
            uint4 u[8];
            float f[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {  // piece p: 16 bytes of row (p >> 3) & 63, block p >> 9
                const int p = v + 128 * m, r = (p >> 3) & 63;
                u[m] = lds128(src + 16 * p);
                f[m] = r < c ? sc * lds32f(ge + 4 * r) : 0.f;
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                uint32_t* w4 = reinterpret_cast<uint32_t*>(&u[m]);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w4[q]);
                    w4[q] = pack_bf16(f[m] * __low2float(h), f[m] * __high2float(h));
                }
                sts128(dst + 16 * (v + 128 * m), u[m]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[R_DOE0 + st]);
                mbar_arrive(&bars[R_GFREE0 + gs]);
            }
        }
    } else if (w >= 4) {
        // ------------------------------------------------------------ state warps
        const int hf = w >= 8 ? 1 : 0;
        const int v = tid - (hf ? 256 : 128);
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        init_state_half<TK_STATE>(tm, lb, hf, v, x0);
        bool ok = true;
        for (int k = 0; ok && k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!warp_wait(bars, R_GATE0 + gs, (k >> 2) & 1, errflag)) { ok = false; break; }
            if (k >= 1) {
                if (!warp_wait(bars, R_MMA5, (k - 1) & 1, errflag)) { ok = false; break; }
                fence_after_sync();
            }
            // hand-off: bf16 copy (what the chain's next product reads), signalled at once; then
            // (the store of dh of the state leaving the chunk and) the decay by e_C, signalled
            // separately for the products that accumulate onto the state
            {
                float xs[64];
                state_bf16_half(tm, lb, T_XB, hf, T_XF, xs);
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[R_EX]);
                const int c0 = 64 * hf;
                if (rule && rule->x_mid && k == rule->n_own) {  // the own segment's left end
#pragma unroll
                    for (int i = 0; i < 64; ++i) rule->x_mid[(c0 + i) * VD + v] = xs[i];
                }
                if (HIST && gb.store) {
                    __nv_bfloat16* hp = reinterpret_cast<__nv_bfloat16*>(B.dhist) +
                                        ((gbase + chunk_of(k)) * P.Hv + j) * (KD * VD);
#pragma unroll
                    for (int i = 0; i < 64; ++i) hp[(c0 + i) * VD + v] = __float2bfloat16_rn(xs[i]);
                }
#pragma unroll
                for (int i = 0; i < 64; ++i) xs[i] *= gb.eC;
                tmem_st32(tm + lb + T_XF + c0, xs);
                tmem_st32(tm + lb + T_XF + c0 + 32, xs + 32);
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[R_DEC]);
            }
            // dV'^T of tokens [32 hf, 32 hf + 32) = scale D_a + kd D_b, packed bf16 in place
            if (!warp_wait(bars, R_MMA3, k & 1, errflag)) { ok = false; break; }
            fence_after_sync();
            float da[32], db[32], kd[32];
            tmem_ld32(tm + lb + T_DA + 32 * hf, da);
            tmem_ld32(tm + lb + T_DB + 32 * hf, db);
            {
                const uint32_t ka = smem_addr(&gb.kd[32 * hf]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 f4 = lds128f(ka + 16 * i);
                    kd[4 * i] = f4.x;
                    kd[4 * i + 1] = f4.y;
                    kd[4 * i + 2] = f4.z;
                    kd[4 * i + 3] = f4.w;
                }
            }
            tmem_ld_wait();
            float pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = __uint_as_float(pack_bf16(fmaf(sc, da[2 * i], kd[2 * i] * db[2 * i]),
                                                  fmaf(sc, da[2 * i + 1], kd[2 * i + 1] * db[2 * i + 1])));
            tmem_st16(tm + lb + T_DB + 32 * hf, pk);
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[R_EV]);
                mbar_arrive(&bars[R_GFREE0 + gs]);
            }
        }
        if (ok && warp_wait(bars, R_MMA5, (n - 1) & 1, errflag)) {
            fence_after_sync();
            if (x_out) {
                for (int c0 = 64 * hf; c0 < 64 * hf + 64; c0 += 16) {
                    float xv[16];
                    tmem_ld16(tm + lb + T_XF + c0, xv);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) x_out[(c0 + i) * VD + v] = xv[i];
                }
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (*errflag && tid == 0 && P.err) atomicOr(P.err, *errflag);
    if (w == 0) {
        fence_after_sync();
        tmem_dealloc(tm, 512);
    }
}

struct BwdMaps {
    TcMaps f;
    CUtensorMap dO;
};

// first phase of the reverse scan: the gradient entering segment lj >= 1 from its right end,
// started from zero (or from dht for the last segment)
__global__ void __launch_bounds__(TCT, 1) k_tc_bwd_a(BwdProblem B, const __grid_constant__ BwdMaps maps) {
    unsigned char* sm = aligned_smem();
    const Problem& P = B.f;
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N || lj == 0) return;
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + CH - 1) / CH);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const float* x0 = (lj == nseg - 1 && B.dht) ? B.dht + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    float* out = B.dhb + (int64_t(gseg) * P.Hv + j) * KVN;
    if (ce <= cb) { copy_state(x0, out, false); return; }
    tc_bwd_scan<false>(B, maps.f, &maps.dO, sm, j, t0, t1, cb, ce, x0, out, plan_chunk_off(P.plan, s));
}

// g-only extension length of the reverse scan into the segment ending at chunk ce (n chunks):
// the smallest e in [1, min(n, EXT_MAX)] whose last e chunks' gate sum is below
// LOG_NEGLIGIBLE, else 0 (the mirror image of the forward's extension length, with the same
// guarantees; the loads here, the sum in ext_sum).
__device__ __forceinline__ void ext_load_rev(const Problem& P, int64_t t0, int64_t t1, int ce, int n, int j,
                                             float (&gv)[EXT_MAX][2]) {
    const int lane = threadIdx.x & 31;
    const int m = min(n, EXT_MAX);
#pragma unroll
    for (int e = 0; e < EXT_MAX; ++e)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int64_t t = t0 + int64_t(ce - 1 - e) * CH + 2 * lane + u;
            gv[e][u] = (e < m && t < t1) ? P.g[t * P.Hv + j] : 0.f;
        }
}

// The reverse dh scan storing dh for every chunk; the first segment's result is dh0.  mode 0:
// every segment from its true right-end gradient (dht, or the fix-up's).  Decay-bounded exact
// mode (the mirror image of k_tc_phase_c's): mode 1, the first pass, runs every segment from
// its right end from zero (the last from dht), stores the gradients that provably do not
// depend on that start and scans on into the trailing chunks of the previous segment that the
// bound does not reach -- from a true gradient when its own transition is negligible (the
// forward's P.dec) or it is the last; each segment's left-end gradient goes to its slot of
// B.dhb (the first one's to dh0).  mode 2 reruns from its true right-end gradient every
// segment with an unwritten result: flagged by its own CTA, preceding a segment (not the last)
// whose transition is not negligible, or the first segment when its own transition is not
// negligible (dh0).
__global__ void __launch_bounds__(TCT, 1) k_tc_bwd_c(BwdProblem B, const __grid_constant__ BwdMaps maps,
                                                    int mode) {
    pdl_launch_dependents();
    unsigned char* sm = aligned_smem();
    // the passes that scan in every CTA set up while the previous kernel finishes
    const bool pre = mode != 2;
    if (pre) tc_bwd_setup(sm);
    pdl_wait();
    const Problem& P = B.f;
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) {
        if (pre) tc_bwd_release(sm);
        return;
    }
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + CH - 1) / CH);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const int64_t sjh = int64_t(gseg) * P.Hv + j;
    const bool last = lj == nseg - 1;
    const float* dht = B.dht ? B.dht + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    float* dh0 = B.dh0 ? B.dh0 + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    if (mode == 1) {
        const float* x0 = last ? dht : nullptr;
        float* x_seg = lj == 0 ? dh0 : B.dhb + sjh * KVN;
        if (ce <= cb) {  // only an empty sequence
            copy_state(x0, x_seg, false);
            tc_bwd_release(sm);
            return;
        }
        // both extension lengths from one round of gate loads (the previous segment is full)
        const int n_own = last ? 0 : ce - cb, n_prev = lj >= 1 ? P.L : 0;
        float g_own[EXT_MAX][2], g_prev[EXT_MAX][2];
        ext_load_rev(P, t0, t1, ce, n_own, j, g_own);
        ext_load_rev(P, t0, t1, cb, n_prev, j, g_prev);
        ScanRule rule;
        rule.n_own = ce - cb;
        rule.e_own = last ? 0 : ext_sum(g_own, n_own);
        rule.lj = last ? 0 : 1;
        rule.dec = nullptr;
        rule.rerun = B.rrerun + sjh;
        rule.ext_ok = (last || P.dec[sjh] >= 0) ? 1 : 0;
        const int e_prev = lj >= 1 ? ext_sum(g_prev, n_prev) : 0;
        rule.x_mid = e_prev > 0 ? x_seg : nullptr;
        tc_bwd_scan<true>(B, maps.f, &maps.dO, sm, j, t0, t1, cb - e_prev, ce, x0,
                          e_prev > 0 ? nullptr : x_seg, plan_chunk_off(P.plan, s), &rule, true);
        return;
    }
    if (mode == 2) {
        if (last || ce <= cb) return;
        const bool next_inner = lj + 1 <= nseg - 2;  // the next segment is not the last
        if (!(B.rrerun[sjh] != 0 || (next_inner && P.dec[sjh + P.Hv] < 0) || (lj == 0 && P.dec[sjh] < 0)))
            return;
        tc_bwd_scan<true>(B, maps.f, &maps.dO, sm, j, t0, t1, cb, ce, B.dhb + (sjh + P.Hv) * KVN,
                          lj == 0 ? dh0 : nullptr, plan_chunk_off(P.plan, s));
        return;
    }
    const float* x0 = last ? dht : B.dhb + (sjh + P.Hv) * KVN;
    float* x_out = (lj == 0) ? dh0 : nullptr;
    if (ce <= cb) {
        copy_state(x0, x_out, false);
        tc_bwd_release(sm);
        return;
    }
    tc_bwd_scan<true>(B, maps.f, &maps.dO, sm, j, t0, t1, cb, ce, x0, x_out, plan_chunk_off(P.plan, s),
                      nullptr, true);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map(CUtensorMap* m, const void* base, int H, int64_t T_total) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, cuuint64_t(H), cuuint64_t(T_total > 0 ? T_total : 1)};
    const cuuint64_t strides[2] = {cuuint64_t(128 * 2), cuuint64_t(H) * 128 * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, cuuint64_t(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {cuuint64_t(128 * 2)};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


#ifdef GDN_TRACE
extern "C" int gdn_debug_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, g_trace, sizeof(g_trace)));
}
extern "C" int gdn_debug_cta_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, g_cta_trace, sizeof(g_cta_trace)));
}
#endif

cudaError_t launch_fwd_tc(const Problem& P, bool hist, int64_t T_total, cudaStream_t st) {
    TcMaps maps;
    if (!make_map(&maps.k, P.k, P.Hqk, T_total) || !make_map(&maps.q, P.q, P.Hqk, T_total) ||
        !make_map(&maps.v, P.v, P.Hv, T_total))
        return cudaErrorInvalidValue;
    cudaError_t e;
    e = smem_attr(k_tc_phase_a, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    for (auto kern : {k_tc_phase_c<TK_OUT, 0>, k_tc_phase_c<TK_OUT, 1>, k_tc_phase_c<TK_OUT, 2>,
                      k_tc_phase_c<TK_HIST, 0>, k_tc_phase_c<TK_HIST, 1>, k_tc_phase_c<TK_HIST, 2>}) {
        e = smem_attr(kern, SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
#ifdef GDN_CHECK
    launch_plan(P, CH, st);
#else
    // an equal-length batch needs no planner kernel (its decomposition is in closed form): the
    // preparation, the first kernel then, clears the call's error word
    if (P.plan.uni_ns == 0 || P.total_chunks <= 0) launch_plan(P, CH, st);
#endif
    launch_prep(P, maps, st);
    const dim3 grid(P.total_segs, P.Hv);
    auto out_pass = [&](const char* name, int mode) {
        timing_begin(name, st);
        auto kern = hist ? (mode == 1 ? k_tc_phase_c<TK_HIST, 1> : mode == 2 ? k_tc_phase_c<TK_HIST, 2>
                                                                          : k_tc_phase_c<TK_HIST, 0>)
                         : (mode == 1 ? k_tc_phase_c<TK_OUT, 1> : mode == 2 ? k_tc_phase_c<TK_OUT, 2>
                                                                          : k_tc_phase_c<TK_OUT, 0>);
        const cudaError_t r = launch_pdl(kern, grid, dim3(TCT), SMEM_BYTES, st, P, maps);
        timing_end(st);
        return r;
    };
    if (P.cp == CP_EXACT && !P.full_cp) {
        // decay-bounded exact context parallelism: first pass from zero (outputs, segment
        // states, decisions), the transitions and the fix-up only where not negligible, then
        // the correction of the leading chunks of every segment past the first
        e = out_pass(hist ? "fwd_recompute_pass1" : "fwd_pass1", 1);
        if (e != cudaSuccess) return e;
        timing_begin("fwd_transitions", st);
        e = launch_pdl(k_tc_phase_a, grid, dim3(TCT), SMEM_BYTES, st, P, maps);
        timing_end(st);
        if (e != cudaSuccess) return e;
        launch_fixup(P, st);
        e = out_pass(hist ? "fwd_recompute_correction" : "fwd_correction", 2);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (P.cp != CP_NONE) {
        timing_begin("fwd_phase_a", st);
        e = launch_pdl(k_tc_phase_a, grid, dim3(TCT), SMEM_BYTES, st, P, maps);
        if (e != cudaSuccess) return e;
        timing_end(st);
        if (P.cp == CP_EXACT) launch_fixup(P, st);
    }
    e = out_pass(hist ? "fwd_recompute_states" : "fwd_phase_c", 0);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// The reverse-scan launches of the backward (bf16): `which` = 0 first phase, 1 the rerun that
// stores dh per chunk (after the caller's fix-up); decay-bounded exact mode: 2 first pass,
// 3 correction.
cudaError_t launch_bwd_scan_tc(const BwdProblem& B, int which, int64_t T_total, cudaStream_t st) {
    const Problem& P = B.f;
    BwdMaps maps;
    if (!make_map(&maps.f.k, P.k, P.Hqk, T_total) || !make_map(&maps.f.q, P.q, P.Hqk, T_total) ||
        !make_map(&maps.f.v, P.v, P.Hv, T_total) || !make_map(&maps.dO, B.dO, P.Hv, T_total))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (which == 0) {
        e = smem_attr(k_tc_bwd_a, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        k_tc_bwd_a<<<dim3(P.total_segs, P.Hv), TCT, SMEM_BYTES, st>>>(B, maps);
    } else {
        e = smem_attr(k_tc_bwd_c, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = launch_pdl(k_tc_bwd_c, dim3(P.total_segs, P.Hv), dim3(TCT), SMEM_BYTES, st, B, maps, which - 1);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace gdn
