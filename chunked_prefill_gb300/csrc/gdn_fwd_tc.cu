// Forward chunk scan on the 5th-generation tensor cores (bf16 operands, fp32 accumulation).
//
// Same chunk algebra and the same context-parallel phases as the CUDA-core kernels in
// gdn_fwd.cu (FlashQLA pages, agentlenshq "GDN chunked prefill optimisation": chunk-local
// W/U preparation, the serial state S and the output O kept on-chip; "AutoCP" segments);
// what changes is where the data live and who moves them:
//
//   * the state is kept TRANSPOSED in tensor memory, Xt[v][dk] = h[dk][v] (fp32 master,
//     128 columns) plus a bf16 copy (64 columns) that is the A operand of the V' and Q.h
//     products straight from TMEM;
//   * K, Q, V chunk tiles arrive by TMA (128-byte swizzle) into a 2-stage ring;
//   * per chunk of 64 tokens (i, j tokens; dk key dim; v value dim):
//       D1  = [K;Q] K^T                 (128 x 64)    -> A (strictly lower) and P
//       T   = (I + A)^-1 on CUDA cores                -> TW = -T diag(beta e), TU = T diag(beta)
//       D2  = K^T TW^T   = W'^T          (dk x i)      -> smem tile (B operand)
//       D3  = V^T TU^T + Xt W'^T = V'^T  (v x i)       -> bf16 V'^T and diag(kd) V'^T in TMEM
//       D4  = Xt Q^T     = (Q h)^T       (v x i)
//       D5  = V'^T P^T   = (P V')^T      (v x i)       -> O = scale (e * D4 + D5)
//       Xt += (diag(kd) V')^T K          (v x dk)      after Xt was scaled by e^{gamma_C}
//
// Warp roles (12 warps): 0 TMA producer, 1 MMA issuer (one thread), 2 gates (cumsum of g,
// exponentials, partial-chunk row masking), 4-7 state warps (TMEM round trips of the state
// and of V'), 8-11 prep/epilogue warps (A, P, the triangular inverse, TW/TU, W'^T, O).
// Every wait on an mbarrier is bounded; on a timeout the kernel records an error word and
// winds down.
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

// tensor-memory columns
// D3 (U^T, then V'^T) is double-buffered by chunk parity at columns 320 and 448; D4 holds
// O^T = (diag(e) Q h)^T + (P V')^T (the decay e is folded into the Q tile in shared memory).
constexpr uint32_t T_XF = 0, T_XB = 128 /* 2 x 64: bf16 state copy, by chunk parity */,
                   T_D2 = 256, T_D4 = 384;
__device__ __forceinline__ uint32_t t_d3(int k) { return (k & 1) ? 448u : 320u; }

// shared-memory layout (offsets from a 1024-aligned base)
constexpr uint32_t S_KQ = 0;            // 2 x 32 KB: rows 0-63 K, 64-127 Q, 2 column blocks
constexpr uint32_t S_KQ_STRIDE = 32768;
constexpr uint32_t S_V = 65536;         // 2 x 16 KB
constexpr uint32_t S_V_STRIDE = 16384;
constexpr uint32_t S_PR = 98304;        // 2 x 24 KB: TW, TU, P tiles ([64 i][64 j] each)
constexpr uint32_t S_PR_STRIDE = 24576;
constexpr uint32_t S_WT = 147456;       // 16 KB: W'^T [128 dk][64 i]
constexpr uint32_t S_GATE = 163840;     // NGATE gate buffers
constexpr int NGATE = 4;
constexpr uint32_t GATE_BYTES = 1088;
constexpr int LDO = 136;                              // output staging row stride (bf16)
constexpr uint32_t S_O = S_GATE + NGATE * GATE_BYTES; // 64 x 136 bf16 output staging
constexpr uint32_t S_BAR = S_O + 64 * LDO * 2;        // mbarriers
constexpr uint32_t S_END = S_BAR + 256;
constexpr uint32_t SMEM_BYTES = S_END + 1024;         // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct alignas(16) Gate {
    float gam[CH];
    float e[CH];     // exp(gamma)
    float kd[CH];    // exp(gamma_C - gamma)
    float eC;
    int c;           // valid rows
};
static_assert(sizeof(Gate) <= GATE_BYTES && sizeof(Gate) % 16 == 0, "gate buffer");

enum Bar { B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_GATE0, B_GATE1, B_GATE2, B_GATE3, B_GFREE0,
           B_GFREE1, B_GFREE2, B_GFREE3, B_MMA2, B_MMA3, B_MMA5, B_MMA4, B_EW, B_EX, B_EV, B_EPI,
           B_QS0, B_QS1, B_COUNT };

enum TcKind { TK_STATE = 0, TK_TRANS = 1, TK_OUT = 2, TK_HIST = 3 };

#ifdef GDN_TRACE
// debug builds only: SM-clock timestamps of the pipeline events of CTA (0, 0)
__device__ unsigned long long g_trace[64][32];
#define TRACE(k, ev)                                                                           \
    do {                                                                                       \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (k) >= 0 && (k) < 64)     \
            g_trace[(k)][(ev)] = clock64();                                                    \
    } while (0)
#else
#define TRACE(k, ev) \
    do {             \
    } while (0)
#endif

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) {  // K-major SW128 operand
    return make_desc(addr, 0, 1024);
}
__device__ __forceinline__ uint64_t mdesc(uint32_t addr, uint32_t lbo) {  // MN-major SW128
    return make_desc(addr, lbo, 1024);
}

// store 8 consecutive fp32 values as one 16-byte bf16 chunk of row r of an SW128 tile
__device__ __forceinline__ void st_chunk8(unsigned char* tile, int r, int ch, const float* x) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]);
    u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]);
    u.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + r * 128 + ((ch ^ (r & 7)) << 4)) = u;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    if (mbar_wait(&bars[b], parity)) return true;
    atomicOr(errflag, 1 << b);
    return false;
}
// a wait of a role that is not on the state chain: it backs off between tries
__device__ __forceinline__ bool wait_bar_lazy(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    if (mbar_wait_sleep(&bars[b], parity, 64)) return true;
    atomicOr(errflag, 1 << b);
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
                                                const float* x0) {
    float xv[16];
    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int dk = c0 + i;
            xv[i] = x0 ? x0[dk * VD + v] : ((KIND == TK_TRANS && dk == v) ? 1.f : 0.f);
        }
        tmem_st16(tm + lb + T_XF + c0, xv);
    }
    tmem_st_wait();
}

// One half (64 key columns) of the per-chunk state hand-off: read the fp32 state, write its
// bf16 copy (the A operand of the V' and Q h products), store it for the backward when asked,
// and decay the fp32 state by exp(gamma_C) before the chunk's update accumulates onto it.
template <int KIND>
__device__ __forceinline__ void convert_state_half(const Problem& P, uint32_t tm, uint32_t lb,
                                                   uint32_t xb, int half, int v, float eC,
                                                   int64_t chunk, int j) {
#pragma unroll 1
    for (int q = 0; q < 2; ++q) {
        const int c0 = 64 * half + 32 * q;
        float x[32];
        tmem_ld32(tm + lb + T_XF + c0, x);
        tmem_ld_wait();
        if (KIND == TK_HIST) {
            __nv_bfloat16* hp = reinterpret_cast<__nv_bfloat16*>(P.hist) + (chunk * P.Hv + j) * (KD * VD);
#pragma unroll
            for (int i = 0; i < 32; ++i) hp[(c0 + i) * VD + v] = __float2bfloat16_rn(x[i]);
        }
        float pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = __uint_as_float(pack_bf16(x[2 * i], x[2 * i + 1]));
        tmem_st16(tm + lb + xb + c0 / 2, pk);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] *= eC;
        tmem_st16(tm + lb + T_XF + c0, x);
        tmem_st16(tm + lb + T_XF + c0 + 16, x + 16);
    }
    tmem_st_wait();
}

template <int KIND>
__device__ void tc_scan(const Problem& P, const TcMaps& maps, unsigned char* sm, int j,
                        int64_t t0, int64_t t1, int cb, int ce, const float* x0, float* x_out,
                        int64_t hist_base) {
    constexpr bool OUT = KIND == TK_OUT;
    constexpr bool NEEDU = KIND != TK_TRANS;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + S_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S_BAR + B_COUNT * 8);
    int* errflag = reinterpret_cast<int*>(sm + S_BAR + B_COUNT * 8 + 4);
    Gate* gates = reinterpret_cast<Gate*>(sm + S_GATE);
    const int G = P.Hv / P.Hqk, qh = j / G;
    const int n = ce - cb;

    if (tid == 0) {
        mbar_init(&bars[B_FULL0], 1);
        mbar_init(&bars[B_FULL1], 1);
        mbar_init(&bars[B_EMPTY0], 1);
        mbar_init(&bars[B_EMPTY1], 1);
        for (int b = 0; b < NGATE; ++b) {
            mbar_init(&bars[B_GATE0 + b], 1);
            mbar_init(&bars[B_GFREE0 + b], OUT ? 8 : 4);
        }
        mbar_init(&bars[B_MMA2], 1);
        mbar_init(&bars[B_MMA3], 1);
        mbar_init(&bars[B_MMA5], 1);
        mbar_init(&bars[B_MMA4], 1);
        mbar_init(&bars[B_EW], 4);
        mbar_init(&bars[B_EX], 8);
        mbar_init(&bars[B_EV], 4);
        mbar_init(&bars[B_EPI], 4);
        mbar_init(&bars[B_QS0], 1);  // per stage: cannot run two phases ahead of its waiter
        mbar_init(&bars[B_QS1], 1);
        *errflag = 0;
        mbar_fence_init();
    }
    if (w == 0) tmem_alloc(tmem_slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *tmem_slot;

    if (w == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t bytes = 16384u + (OUT ? 16384u : 0u) + (NEEDU ? 16384u : 0u) +
                                   8192u * (1u + (NEEDU ? 1u : 0u) + (OUT ? 1u : 0u));
            int issued = 0;
            for (int k = 0; k < n; ++k) {
                const int st = k & 1;
                if (k >= 2 && !wait_bar_lazy(bars, B_EMPTY0 + st, ((k - 2) >> 1) & 1, errflag)) break;
                const int tc = int(t0 + int64_t(cb + k) * CH);
                uint64_t* full = &bars[B_FULL0 + st];
                unsigned char* kq = sm + S_KQ + st * S_KQ_STRIDE;
                unsigned char* pr = sm + S_PR + st * S_PR_STRIDE;
                const unsigned char* src = static_cast<const unsigned char*>(P.prep) +
                                           ((hist_base + cb + k) * P.Hv + j) * 3 * 8192;
                mbar_expect_tx(full, bytes);
                tma_load_3d(kq, &maps.k, full, 0, qh, tc);
                tma_load_3d(kq + 16384, &maps.k, full, 64, qh, tc);
                bulk_load(pr, src, 8192, full);                       // TW
                if (NEEDU) bulk_load(pr + 8192, src + 8192, 8192, full);   // TU
                if (OUT) {
                    tma_load_3d(kq + 8192, &maps.q, full, 0, qh, tc);
                    tma_load_3d(kq + 16384 + 8192, &maps.q, full, 64, qh, tc);
                    bulk_load(pr + 16384, src + 16384, 8192, full);   // P
                }
                if (NEEDU) {
                    unsigned char* vt = sm + S_V + st * S_V_STRIDE;
                    tma_load_3d(vt, &maps.v, full, 0, j, tc);
                    tma_load_3d(vt + 8192, &maps.v, full, 64, j, tc);
                }
                issued = k + 1;
            }
            // drain: every issued load has landed before the CTA may exit
            for (int k = max(0, issued - 2); k < issued; ++k)
                mbar_wait(&bars[B_FULL0 + (k & 1)], (k >> 1) & 1);
        }
        __syncwarp();
    } else if (w == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID2 = make_idesc(128, 64, 1, 0);
            constexpr uint32_t ID3 = make_idesc(128, 64, 0, 1);
            constexpr uint32_t ID4 = make_idesc(128, 64, 0, 0);
            constexpr uint32_t ID5 = make_idesc(128, 128, 0, 1);
            const uint32_t kq0 = smem_addr(sm + S_KQ), v0 = smem_addr(sm + S_V);
            const uint32_t wt = smem_addr(sm + S_WT), pr0 = smem_addr(sm + S_PR);
            // descriptors are built once; a byte offset `off` within a tile is added to the
            // start-address field as off >> 4 (addresses stay below 2^18, no carry out)
            const uint64_t dKm[2] = {mdesc(kq0, 16384), mdesc(kq0 + S_KQ_STRIDE, 16384)};
            const uint64_t dKk[2] = {kdesc(kq0), kdesc(kq0 + S_KQ_STRIDE)};
            const uint64_t dV[2] = {mdesc(v0, 8192), mdesc(v0 + S_V_STRIDE, 8192)};
            const uint64_t dPr[2] = {kdesc(pr0), kdesc(pr0 + S_PR_STRIDE)};
            const uint64_t dWT = mdesc(wt, 16384);
            bool ok = true;
            int n_mma2 = 0;
            // W'^T = K^T TW^T for chunk k (needs the stage loaded and partial rows masked)
            auto issue_w = [&](int k) -> bool {
                const int st = k & 1;
                if (!wait_bar(bars, B_FULL0 + st, (k >> 1) & 1, errflag)) return false;
                if (!wait_bar(bars, B_GATE0 + (k & (NGATE - 1)), (k >> 2) & 1, errflag)) return false;
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + T_D2, (st ? dKm[1] : dKm[0]) + (s * 2048 >> 4), (st ? dPr[1] : dPr[0]) + (s * 32 >> 4), ID2, s > 0);
                commit(&bars[B_MMA2]);
                ++n_mma2;
                return true;
            };
            // U^T = V^T TU^T for chunk k into D3[k & 1] (needs the stage loaded; issue_w waited)
            auto issue_u = [&](int k) {
                const int st = k & 1;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + t_d3(k), (st ? dV[1] : dV[0]) + (s * 2048 >> 4),
                             (st ? dPr[1] : dPr[0]) + ((8192 + s * 32) >> 4), ID2, s > 0);
            };
            ok = issue_w(0);
            if (ok && NEEDU) issue_u(0);
            // Tensor-pipe order per chunk k: V' (MMA-3), W' of k+1, the state update (MMA-5),
            // U of k+1, then the output products of k -- the state chain never waits behind
            // the output products.
            for (int k = 0; ok && k < n; ++k) {
                const int st = k & 1;
                const uint32_t xb = tm + T_XB + 64 * (k & 1), d3 = tm + t_d3(k);
                TRACE(k, 0);
                if (!wait_bar(bars, B_EX, k & 1, errflag) || !wait_bar(bars, B_EW, k & 1, errflag)) {
                    ok = false;
                    break;
                }
                TRACE(k, 1);
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16_ta(d3, xb + 8 * s, dWT + (s * 2048 >> 4), ID3, (NEEDU || s > 0) ? 1u : 0u);
                commit(&bars[B_MMA3]);
                TRACE(k, 2);
                if (k + 1 < n && !issue_w(k + 1)) { ok = false; break; }
                TRACE(k, 3);
                if (!wait_bar(bars, B_EV, k & 1, errflag)) { ok = false; break; }
                TRACE(k, 4);
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16_ta(tm + T_XF, d3 + 32 + 8 * s, (st ? dKm[1] : dKm[0]) + (s * 2048 >> 4), ID5, 1u);
                commit(&bars[B_MMA5]);
                TRACE(k, 5);
                if (NEEDU && k + 1 < n) issue_u(k + 1);
                if (OUT) {
                    if (k >= 1 && !wait_bar(bars, B_EPI, (k - 1) & 1, errflag)) { ok = false; break; }
                    TRACE(k, 25);
                    if (!wait_bar(bars, B_QS0 + st, (k >> 1) & 1, errflag)) { ok = false; break; }
                    TRACE(k, 26);
                    fence_after_sync();
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t off = 8192 + (s >> 2) * 16384 + (s & 3) * 32;
                        mma_bf16_ta(tm + T_D4, xb + 8 * s, (st ? dKk[1] : dKk[0]) + (off >> 4), ID4, s > 0);
                    }
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16_ta(tm + T_D4, d3 + 8 * s, (st ? dPr[1] : dPr[0]) + ((16384 + s * 32) >> 4), ID4, 1u);
                    commit(&bars[B_MMA4]);
                }
                commit(&bars[B_EMPTY0 + st]);  // every reader of this stage has been issued
                TRACE(k, 7);
            }
            // drain: wait for every issued MMA before TMEM may be released
            commit(&bars[B_MMA2]);
            mbar_wait(&bars[B_MMA2], n_mma2 & 1);
        }
        __syncwarp();
    } else if (w == 2) {
        // ------------------------------------------------------------ gates
        for (int k = 0; k < n; ++k) {
            const int st = k & 1, gs = k & (NGATE - 1);
            const int64_t tc = t0 + int64_t(cb + k) * CH;
            const int c = int((t1 - tc) < int64_t(CH) ? (t1 - tc) : int64_t(CH));
            float gv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // issue the global loads before waiting for a buffer
                const int r = 2 * lane + u;
                gv[u] = r < c ? P.g[(tc + r) * P.Hv + j] : 0.f;
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
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_GATE0 + gs]);
            TRACE(k, 23);
        }
    } else if (w == 3 && OUT) {
        // ------------------------------------------------------------ Q scaling warp
        // Q row i <- exp(gamma_i) Q row i in place, after the stage landed and the gate warp
        // zeroed rows past the sequence end; O = scale (Q~ h + P V') then needs one accumulator.
        for (int k = 0; k < n; ++k) {
            const int st = k & 1, gs = k & (NGATE - 1);
            if (!warp_wait<true>(bars, B_GATE0 + gs, (k >> 2) & 1, errflag)) break;
            if (!warp_wait<true>(bars, B_FULL0 + st, (k >> 1) & 1, errflag)) break;
            TRACE(k, 27);
            const Gate& gb = gates[gs];
            unsigned char* kq = sm + S_KQ + st * S_KQ_STRIDE;
            // lane covers 16-byte piece (lane & 15) of rows 2i + (lane >> 4); eight pieces are
            // loaded before any is rescaled so the shared-memory latency overlaps
#pragma unroll
            for (int b = 0; b < CH / 16; ++b) {
                uint4 u[8];
                float e[8];
                uint4* p[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = (b * 8 + i) * 2 + (lane >> 4), ch = lane & 15;
                    p[i] = reinterpret_cast<uint4*>(kq + (ch >> 3) * 16384 + 8192 + r * 128 + (ch & 7) * 16);
                    u[i] = *p[i];
                    e[i] = gb.e[r];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    uint32_t* w4 = reinterpret_cast<uint32_t*>(&u[i]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w4[q]);
                        w4[q] = pack_bf16(e[i] * __low2float(h), e[i] * __high2float(h));
                    }
                    *p[i] = u[i];
                }
            }
            TRACE(k, 29);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_QS0 + st]);
            TRACE(k, 24);
        }
    } else if (w >= 4 && w < 8) {
        // ------------------------------------------------------------ state warps
        const int v = tid - 128;                     // TMEM lane = value column of h
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        init_state_half<KIND>(tm, lb, 0, v, x0);
        bool ok = true;
        for (int k = 0; ok && k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!warp_wait(bars, B_GATE0 + gs, (k >> 2) & 1, errflag)) { ok = false; break; }
            if (v == 0) TRACE(k, 16);
            if (k >= 1) {
                if (!warp_wait(bars, B_MMA5, (k - 1) & 1, errflag)) { ok = false; break; }
                fence_after_sync();
            }
            if (v == 0) TRACE(k, 17);
            convert_state_half<KIND>(P, tm, lb, T_XB + 64 * (k & 1), 0, v, gb.eC, hist_base + cb + k, j);
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EX]);
            if (v == 0) TRACE(k, 18);
            // V' = D3 -> bf16 V'^T (columns 0-31) and diag(kd) V'^T (columns 32-63)
            if (!warp_wait(bars, B_MMA3, k & 1, errflag)) { ok = false; break; }
            if (v == 0) TRACE(k, 19);
            fence_after_sync();
            float vp[64];
            const uint32_t d3 = t_d3(k);
            tmem_ld32(tm + lb + d3, vp);
            tmem_ld32(tm + lb + d3 + 32, vp + 32);
            tmem_ld_wait();
            float p1[16], p2[16], h1[16], h2[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                p1[i] = __uint_as_float(pack_bf16(vp[2 * i], vp[2 * i + 1]));
                p2[i] = __uint_as_float(pack_bf16(vp[32 + 2 * i], vp[32 + 2 * i + 1]));
                h1[i] = __uint_as_float(pack_bf16(vp[2 * i] * gb.kd[2 * i], vp[2 * i + 1] * gb.kd[2 * i + 1]));
                h2[i] = __uint_as_float(pack_bf16(vp[32 + 2 * i] * gb.kd[32 + 2 * i],
                                                  vp[32 + 2 * i + 1] * gb.kd[32 + 2 * i + 1]));
            }
            tmem_st16(tm + lb + d3, p1);
            tmem_st16(tm + lb + d3 + 16, p2);
            tmem_st16(tm + lb + d3 + 32, h1);
            tmem_st16(tm + lb + d3 + 48, h2);
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_EV]);
                mbar_arrive(&bars[B_GFREE0 + gs]);  // done with this chunk's gates
            }
            if (v == 0) TRACE(k, 20);
        }
        if (ok && warp_wait(bars, B_MMA5, (n - 1) & 1, errflag)) {
            fence_after_sync();
            if (x_out) {
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    float xv[16];
                    tmem_ld16(tm + lb + T_XF + c0, xv);
                    tmem_ld_wait();
                    if (KIND == TK_TRANS) {  // segment transitions are stored transposed (M^T)
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(x_out + v * VD + c0 + i) =
                                make_float4(xv[i], xv[i + 1], xv[i + 2], xv[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) x_out[(c0 + i) * VD + v] = xv[i];
                    }
                }
            }
        }
    } else if (w >= 8 && w < 12) {
        // ------------------------------------------------------------ W'^T + state warps
        const int t = tid - 256;                     // TMEM lane: key row dk / value column v
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        auto convert_w = [&](int k) -> bool {
            if (!warp_wait(bars, B_MMA2, k & 1, errflag)) return false;
            if (t == 0) TRACE(k, 12);
            fence_after_sync();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float d[32];
                tmem_ld32(tm + lb + T_D2 + 32 * half, d);
                tmem_ld_wait();
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) st_chunk8(sm + S_WT, t, 4 * half + ch, d + 8 * ch);
            }
            fence_proxy_async_smem();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EW]);
            if (t == 0) TRACE(k, 13);
            return true;
        };
        init_state_half<KIND>(tm, lb, 1, t, x0);
        bool ok = convert_w(0);
        for (int k = 0; ok && k < n; ++k) {
            const Gate& gb = gates[k & (NGATE - 1)];
            if (!warp_wait(bars, B_GATE0 + (k & (NGATE - 1)), (k >> 2) & 1, errflag)) break;
            if (k >= 1) {
                if (!warp_wait(bars, B_MMA5, (k - 1) & 1, errflag)) break;
                fence_after_sync();
            }
            convert_state_half<KIND>(P, tm, lb, T_XB + 64 * (k & 1), 1, t, gb.eC, hist_base + cb + k, j);
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EX]);
            if (k + 1 < n) ok = convert_w(k + 1);
        }
    } else if (w >= 12 && OUT) {
        // ------------------------------------------------------------ output warps
        const int v = tid - 384;                     // TMEM lane = value column
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        __nv_bfloat16* sO = reinterpret_cast<__nv_bfloat16*>(sm + S_O);
        for (int k = 0; k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!named_and(2, 128, warp_wait<true>(bars, B_MMA4, k & 1, errflag))) break;
            if (v == 0) TRACE(k, 14);
            fence_after_sync();
            const float sc = P.scale;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float d4[32];
                tmem_ld32(tm + lb + T_D4 + 32 * half, d4);
                tmem_ld_wait();
                if (half == 1) {
                    fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_EPI]);
                    if (v == 0) TRACE(k, 28);
                }
#pragma unroll
                for (int qq = 0; qq < 32; ++qq) {
                    const int ii = 32 * half + qq;
                    sO[ii * LDO + v] = __float2bfloat16_rn(sc * d4[qq]);
                }
            }
            named_sync(2, 128);
            // rows of O leave as 16-byte vectors (only the rows of this sequence)
            const int64_t tc = t0 + int64_t(cb + k) * CH;
            const int c = gb.c;
            __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(P.o) + (tc * P.Hv + j) * VD;
            const int64_t rs = int64_t(P.Hv) * VD;
            for (int idx = v; idx < c * 16; idx += 128) {
                const int r = idx >> 4, cv = idx & 15;
                *reinterpret_cast<uint4*>(ob + r * rs + cv * 8) =
                    *reinterpret_cast<const uint4*>(sO + r * LDO + cv * 8);
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
    unsigned char* sm = aligned_smem();
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = P.plan.seg[gseg];
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) return;
    const int nseg = P.plan.seg_off[s + 1] - P.plan.seg_off[s];
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + CH - 1) / CH);
    const float* h0 = P.h0 ? P.h0 + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    if (P.cp == CP_EXACT) {
        if (lj >= nseg - 1) return;
        const int cb = lj * P.L, ce = min(cb + P.L, nt);
        if (blockIdx.z == 0) {
            float* out = P.hin + (int64_t(gseg + 1) * P.Hv + j) * KVN;
            const float* x0 = lj == 0 ? h0 : nullptr;
            if (ce <= cb) { copy_state(x0, out, false); return; }
            tc_scan<TK_STATE>(P, maps, sm, j, t0, t1, cb, ce, x0, out, P.plan.chunk_off[s]);
        } else {
            if (lj == 0) return;
            float* out = P.mbuf + (int64_t(gseg) * P.Hv + j) * KVN;
            if (ce <= cb) { copy_state(nullptr, out, true); return; }
            tc_scan<TK_TRANS>(P, maps, sm, j, t0, t1, cb, ce, nullptr, out, P.plan.chunk_off[s]);
        }
    } else {
        if (lj == 0 || blockIdx.z != 0) return;
        const int cb = lj * P.L, w0 = cb - P.warmup;
        const float* x0 = w0 <= 0 ? h0 : nullptr;
        float* out = P.hin + (int64_t(gseg) * P.Hv + j) * KVN;
        tc_scan<TK_STATE>(P, maps, sm, j, t0, t1, max(w0, 0), cb, x0, out, P.plan.chunk_off[s]);
    }
}

template <int KIND>
__global__ void __launch_bounds__(TCT, 1) k_tc_phase_c(Problem P, const __grid_constant__ TcMaps maps) {
    unsigned char* sm = aligned_smem();
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = P.plan.seg[gseg];
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) return;
    const int nseg = P.plan.seg_off[s + 1] - P.plan.seg_off[s];
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + CH - 1) / CH);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const float* x0 = (lj == 0) ? (P.h0 ? P.h0 + (int64_t(s) * P.Hv + j) * KVN : nullptr)
                                : P.hin + (int64_t(gseg) * P.Hv + j) * KVN;
    float* x_out = (lj == nseg - 1 && P.ht) ? P.ht + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    if (ce <= cb) { copy_state(x0, x_out, false); return; }
    tc_scan<KIND>(P, maps, sm, j, t0, t1, cb, ce, x0, x_out, P.plan.chunk_off[s]);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// [T_total, H, 128] bf16 viewed as (d, head, token); box 64 x 1 x 64, 128-byte swizzle
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

}  // namespace

#ifdef GDN_TRACE
extern "C" int gdn_debug_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, g_trace, sizeof(g_trace)));
}
#endif

cudaError_t launch_fwd_tc(const Problem& P, bool hist, int64_t T_total, cudaStream_t st) {
    TcMaps maps;
    if (!make_map(&maps.k, P.k, P.Hqk, T_total) || !make_map(&maps.q, P.q, P.Hqk, T_total) ||
        !make_map(&maps.v, P.v, P.Hv, T_total))
        return cudaErrorInvalidValue;
    cudaError_t e;
    e = cudaFuncSetAttribute(k_tc_phase_a, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_tc_phase_c<TK_OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_tc_phase_c<TK_HIST>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    launch_plan(P, CH, st);
    launch_prep(P, st);
    if (P.cp != CP_NONE) {
        dim3 ga(P.total_segs, P.Hv, P.cp == CP_EXACT ? 2 : 1);
        timing_begin("fwd_phase_a", st);
        k_tc_phase_a<<<ga, TCT, SMEM_BYTES, st>>>(P, maps);
        timing_end(st);
        if (P.cp == CP_EXACT) launch_fixup(P, st);
    }
    dim3 gc(P.total_segs, P.Hv);
    timing_begin(hist ? "fwd_recompute_states" : "fwd_phase_c", st);
    if (hist)
        k_tc_phase_c<TK_HIST><<<gc, TCT, SMEM_BYTES, st>>>(P, maps);
    else
        k_tc_phase_c<TK_OUT><<<gc, TCT, SMEM_BYTES, st>>>(P, maps);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace gdn
