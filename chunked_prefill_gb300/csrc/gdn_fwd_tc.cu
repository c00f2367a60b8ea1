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
constexpr uint32_t T_XF = 0, T_XB = 128, T_D1 = 192, T_D2 = 256, T_D3 = 320, T_D4 = 384,
                   T_D5 = 448;

// shared-memory layout (offsets from a 1024-aligned base)
constexpr uint32_t S_KQ = 0;            // 2 x 32 KB: rows 0-63 K, 64-127 Q, 2 column blocks
constexpr uint32_t S_KQ_STRIDE = 32768;
constexpr uint32_t S_V = 65536;         // 2 x 16 KB
constexpr uint32_t S_V_STRIDE = 16384;
constexpr uint32_t S_WT = 98304;        // 16 KB: W'^T [128 dk][64 i]
constexpr uint32_t S_TW = 114688;       // 8 KB:  [64 i][64 j]
constexpr uint32_t S_TU = 122880;       // 8 KB
constexpr uint32_t S_P = 131072;        // 2 x 8 KB
constexpr uint32_t S_P_STRIDE = 8192;
constexpr int LDA = 68;                 // fp32 scratch row stride (floats)
constexpr uint32_t S_A = 147456;        // fp32 64 x 68
constexpr uint32_t S_T = S_A + 64 * LDA * 4;
constexpr uint32_t S_TMP = S_T + 64 * LDA * 4;        // 4 warps x 16 x 20 fp32
constexpr uint32_t S_GATE = S_TMP + 5120;             // NGATE gate buffers
constexpr int NGATE = 4;
constexpr uint32_t GATE_BYTES = 1600;
constexpr int LDO = 136;                              // output staging row stride (bf16)
constexpr uint32_t S_O = S_GATE + NGATE * GATE_BYTES; // 64 x 136 bf16 output staging
constexpr uint32_t S_BAR = S_O + 64 * LDO * 2;        // mbarriers
constexpr uint32_t S_END = S_BAR + 256;
constexpr uint32_t SMEM_BYTES = S_END + 1024;         // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct alignas(16) Gate {
    float gam[CH];
    float e[CH];     // exp(gamma)
    float einv[CH];  // exp(-gamma)
    float kd[CH];    // exp(gamma_C - gamma)
    float beta[CH];
    float be[CH];    // beta * exp(gamma)
    float eC;
    int c;           // valid rows
    int pairwise;    // gamma range too wide for the factorised exponentials
};
static_assert(sizeof(Gate) <= GATE_BYTES && sizeof(Gate) % 16 == 0, "gate buffer");

enum Bar { B_FULL0 = 0, B_FULL1, B_GATE0, B_GATE1, B_GATE2, B_GATE3, B_GFREE0, B_GFREE1, B_GFREE2,
           B_GFREE3, B_MMA1, B_MMA2, B_MMA3, B_MMA5, B_ET, B_EW, B_EX, B_EV, B_EPI, B_COUNT };

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
// warp-uniform wait: lane 0 waits, the result is broadcast, then the warp synchronises
__device__ __forceinline__ bool warp_wait(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bars, b, parity, errflag);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
// wait that is uniform over the four prep warps (named barrier 1)
__device__ __forceinline__ bool group_wait(uint64_t* bars, int b, uint32_t parity, int* errflag) {
    const bool ok = warp_wait(bars, b, parity, errflag);
    return named_and(1, 128, ok);
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
        for (int b = 0; b < NGATE; ++b) {
            mbar_init(&bars[B_GATE0 + b], 1);
            mbar_init(&bars[B_GFREE0 + b], OUT ? 12 : 8);
        }
        mbar_init(&bars[B_MMA1], 1);
        mbar_init(&bars[B_MMA2], 1);
        mbar_init(&bars[B_MMA3], 1);
        mbar_init(&bars[B_MMA5], 1);
        mbar_init(&bars[B_ET], 4);
        mbar_init(&bars[B_EW], 4);
        mbar_init(&bars[B_EX], 4);
        mbar_init(&bars[B_EV], 4);
        mbar_init(&bars[B_EPI], 4);
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
            const uint32_t bytes = 16384u + (OUT ? 16384u : 0u) + (NEEDU ? 16384u : 0u);
            int issued = 0;
            for (int k = 0; k < n; ++k) {
                const int st = k & 1;
                if (k >= 2 && !wait_bar(bars, B_MMA5, (k - 2) & 1, errflag)) break;
                const int tc = int(t0 + int64_t(cb + k) * CH);
                uint64_t* full = &bars[B_FULL0 + st];
                unsigned char* kq = sm + S_KQ + st * S_KQ_STRIDE;
                mbar_expect_tx(full, bytes);
                tma_load_3d(kq, &maps.k, full, 0, qh, tc);
                tma_load_3d(kq + 16384, &maps.k, full, 64, qh, tc);
                if (OUT) {
                    tma_load_3d(kq + 8192, &maps.q, full, 0, qh, tc);
                    tma_load_3d(kq + 16384 + 8192, &maps.q, full, 64, qh, tc);
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
            constexpr uint32_t ID1 = make_idesc(128, 64, 0, 0);
            constexpr uint32_t ID2 = make_idesc(128, 64, 1, 0);
            constexpr uint32_t ID3 = make_idesc(128, 64, 0, 1);
            constexpr uint32_t ID4 = make_idesc(128, 64, 0, 0);
            constexpr uint32_t ID5 = make_idesc(128, 128, 0, 1);
            const uint32_t kq0 = smem_addr(sm + S_KQ), v0 = smem_addr(sm + S_V);
            const uint32_t wt = smem_addr(sm + S_WT), tw = smem_addr(sm + S_TW),
                           tu = smem_addr(sm + S_TU), p0 = smem_addr(sm + S_P);
            bool ok = true;
            int n_mma1 = 0;  // commits made on the MMA1 barrier
            auto prep_mma1 = [&](int k) -> bool {
                const int st = k & 1;
                if (!wait_bar(bars, B_FULL0 + st, (k >> 1) & 1, errflag)) return false;
                if (!wait_bar(bars, B_GATE0 + (k & (NGATE - 1)), (k >> 2) & 1, errflag)) return false;
                fence_after_sync();
                const uint32_t kq = kq0 + st * S_KQ_STRIDE;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
                    mma_bf16(tm + T_D1, kdesc(kq + off), kdesc(kq + off), ID1, s > 0);
                }
                commit(&bars[B_MMA1]);
                ++n_mma1;
                return true;
            };
            auto prep_mma2 = [&](int k) -> bool {
                const int st = k & 1;
                if (!wait_bar(bars, B_ET, k & 1, errflag)) return false;
                fence_after_sync();
                const uint32_t kq = kq0 + st * S_KQ_STRIDE;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16(tm + T_D2, mdesc(kq + s * 2048, 16384), kdesc(tw + s * 32), ID2, s > 0);
                commit(&bars[B_MMA2]);
                return true;
            };
            ok = prep_mma1(0) && prep_mma2(0) && wait_bar(bars, B_EW, 0, errflag);
            for (int k = 0; ok && k < n; ++k) {
                const int st = k & 1;
                const uint32_t kq = kq0 + st * S_KQ_STRIDE;
                TRACE(k, 0);
                if (NEEDU) {
                    const uint32_t vt = v0 + st * S_V_STRIDE;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16(tm + T_D3, mdesc(vt + s * 2048, 8192), kdesc(tu + s * 32), ID2, s > 0);
                }
                if (!wait_bar(bars, B_EX, k & 1, errflag)) { ok = false; break; }
                TRACE(k, 1);
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_bf16_ta(tm + T_D3, tm + T_XB + 8 * s, mdesc(wt + s * 2048, 16384), ID3,
                                (NEEDU || s > 0) ? 1u : 0u);
                commit(&bars[B_MMA3]);
                TRACE(k, 2);
                if (OUT) {
                    if (k >= 1 && !wait_bar(bars, B_EPI, (k - 1) & 1, errflag)) { ok = false; break; }
                    fence_after_sync();
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const uint32_t off = 8192 + (s >> 2) * 16384 + (s & 3) * 32;
                        mma_bf16_ta(tm + T_D4, tm + T_XB + 8 * s, kdesc(kq + off), ID4, s > 0);
                    }
                }
                TRACE(k, 30);
                if (k + 1 < n && !prep_mma1(k + 1)) { ok = false; break; }
                TRACE(k, 3);
                if (!wait_bar(bars, B_EV, k & 1, errflag)) { ok = false; break; }
                TRACE(k, 4);
                fence_after_sync();
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_bf16_ta(tm + T_XF, tm + T_D3 + 32 + 8 * s, mdesc(kq + s * 2048, 16384), ID5, 1u);
                if (OUT) {
                    const uint32_t pp = p0 + (k & 1) * S_P_STRIDE;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_bf16_ta(tm + T_D5, tm + T_D3 + 8 * s, kdesc(pp + s * 32), ID4, s > 0);
                }
                commit(&bars[B_MMA5]);
                TRACE(k, 5);
                if (k + 1 < n) {
                    if (!prep_mma2(k + 1)) { ok = false; break; }
                    TRACE(k, 6);
                    if (!wait_bar(bars, B_EW, (k + 1) & 1, errflag)) { ok = false; break; }
                    TRACE(k, 7);
                }
            }
            // drain: wait for every issued MMA before TMEM may be released
            commit(&bars[B_MMA1]);
            mbar_wait(&bars[B_MMA1], n_mma1 & 1);
        }
        __syncwarp();
    } else if (w == 2) {
        // ------------------------------------------------------------ gates
        for (int k = 0; k < n; ++k) {
            const int st = k & 1, gs = k & (NGATE - 1);
            const int64_t tc = t0 + int64_t(cb + k) * CH;
            const int c = int((t1 - tc) < int64_t(CH) ? (t1 - tc) : int64_t(CH));
            float gv[2], bv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {  // issue the global loads before waiting for a buffer
                const int r = 2 * lane + u;
                gv[u] = r < c ? P.g[(tc + r) * P.Hv + j] : 0.f;
                bv[u] = r < c ? P.beta[(tc + r) * P.Hv + j] : 0.f;
            }
            TRACE(k, 21);
            if (k >= NGATE && !warp_wait(bars, B_GFREE0 + gs, ((k - NGATE) >> 2) & 1, errflag)) break;
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
                const float e = expf(gm[u]);
                gb.gam[r] = gm[u];
                gb.e[r] = e;
                gb.einv[r] = expf(-gm[u]);
                gb.kd[r] = expf(last - gm[u]);
                gb.beta[r] = bv[u];
                gb.be[r] = bv[u] * e;
            }
            if (lane == 0) {
                gb.eC = expf(last);
                gb.c = c;
                gb.pairwise = (last < -80.f || !(last == last)) ? 1 : 0;
            }
            if (c < CH) {  // rows past the sequence end: zero them (they may hold other tokens)
                if (!warp_wait(bars, B_FULL0 + st, (k >> 1) & 1, errflag)) break;
                unsigned char* kq = sm + S_KQ + st * S_KQ_STRIDE;
                unsigned char* vt = sm + S_V + st * S_V_STRIDE;
                const int rows = CH - c;
                for (int idx = lane; idx < rows * 16; idx += 32) {
                    const int r = c + idx / 16, ch = idx % 16;
                    const int blk = ch >> 3, cc = ch & 7;
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4*>(kq + blk * 16384 + r * 128 + cc * 16) = z;
                    if (OUT) *reinterpret_cast<uint4*>(kq + blk * 16384 + 8192 + r * 128 + cc * 16) = z;
                    if (NEEDU) *reinterpret_cast<uint4*>(vt + blk * 8192 + r * 128 + cc * 16) = z;
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_GATE0 + gs]);
            TRACE(k, 23);
        }
    } else if (w >= 4 && w < 8) {
        // ------------------------------------------------------------ state warps
        const int v = tid - 128;                     // TMEM lane = value column of h
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        {
            float xv[16];
            for (int c0 = 0; c0 < 128; c0 += 16) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int dk = c0 + i;
                    xv[i] = x0 ? x0[dk * VD + v] : ((KIND == TK_TRANS && dk == v) ? 1.f : 0.f);
                }
                tmem_st16(tm + lb + T_XF + c0, xv);
            }
            tmem_st_wait();
        }
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
            const float eC = gb.eC;
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
                float x[32];
                tmem_ld32(tm + lb + T_XF + c0, x);
                tmem_ld_wait();
                if (KIND == TK_HIST) {
                    __nv_bfloat16* hp = reinterpret_cast<__nv_bfloat16*>(P.hist) +
                                        ((hist_base + cb + k) * P.Hv + j) * (KD * VD);
#pragma unroll
                    for (int i = 0; i < 32; ++i) hp[(c0 + i) * VD + v] = __float2bfloat16_rn(x[i]);
                }
                float pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = __uint_as_float(pack_bf16(x[2 * i], x[2 * i + 1]));
                tmem_st16(tm + lb + T_XB + c0 / 2, pk);
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] *= eC;
                tmem_st16(tm + lb + T_XF + c0, x);
                tmem_st16(tm + lb + T_XF + c0 + 16, x + 16);
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_EX]);
            if (v == 0) TRACE(k, 18);
            // V' = D3 -> bf16 V'^T (columns 0-31) and diag(kd) V'^T (columns 32-63)
            if (!warp_wait(bars, B_MMA3, k & 1, errflag)) { ok = false; break; }
            if (v == 0) TRACE(k, 19);
            fence_after_sync();
            float vp[64];
            tmem_ld32(tm + lb + T_D3, vp);
            tmem_ld32(tm + lb + T_D3 + 32, vp + 32);
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
            tmem_st16(tm + lb + T_D3, p1);
            tmem_st16(tm + lb + T_D3 + 16, p2);
            tmem_st16(tm + lb + T_D3 + 32, h1);
            tmem_st16(tm + lb + T_D3 + 48, h2);
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
        // ------------------------------------------------------------ prep warps
        const int t = tid - 256;                     // TMEM lane
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        float* sA = reinterpret_cast<float*>(sm + S_A);
        float* sT = reinterpret_cast<float*>(sm + S_T);
        float* sTmp = reinterpret_cast<float*>(sm + S_TMP);
        const int i = t & 63;
        for (int k = 0; k < n; ++k) {
            const int st = k & 1;
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (t == 0) TRACE(k, 8);
            if (!group_wait(bars, B_GATE0 + gs, (k >> 2) & 1, errflag)) break;
            if (!group_wait(bars, B_MMA1, k & 1, errflag)) break;
            if (t == 0) TRACE(k, 9);
            fence_after_sync();
            // A (threads 0-63: rows of K K^T) and P (threads 64-127: rows of Q K^T)
            {
                const bool pw = gb.pairwise != 0;
                const float gi = gb.gam[i];
                const float ri = (t < 64) ? gb.be[i] : gb.e[i];   // row factor
                const float bi = gb.beta[i];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float d[32];
                    tmem_ld32(tm + lb + T_D1 + 32 * half, d);
                    tmem_ld_wait();
                    if (t == 0 && half == 0) TRACE(k, 28);
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int jj = 32 * half + q;
                        float f;
                        if (!pw) {
                            f = ri * gb.einv[jj];
                        } else {
                            f = expf(gi - gb.gam[jj]);
                            if (t < 64) f *= bi;
                        }
                        const bool keep = (t < 64) ? (i > jj) : (i >= jj);
                        d[q] = keep ? f * d[q] : 0.f;
                    }
                    if (t < 64) {
#pragma unroll
                        for (int q = 0; q < 32; q += 4)
                            *reinterpret_cast<float4*>(sA + i * LDA + 32 * half + q) =
                                make_float4(d[q], d[q + 1], d[q + 2], d[q + 3]);
                    } else if (OUT) {
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch)
                            st_chunk8(sm + S_P + st * S_P_STRIDE, i, 4 * half + ch, d + 8 * ch);
                    }
                }
                if (OUT && t >= 64) fence_proxy_async_smem();
            }
            named_sync(1, 128);
            if (t == 0) TRACE(k, 10);
            // T = (I + A)^-1.  Diagonal 16 x 16 blocks by substitution: warp q inverts block q
            // (lane = column) ...
            const int q = w - 8;
            if (lane < 16) {
                const int b0 = 16 * q, col = lane;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                    for (int m = 0; m < r; ++m) {
                        if (m & 1) acc1 = fmaf(sA[(b0 + r) * LDA + b0 + m], x[m], acc1);
                        else acc0 = fmaf(sA[(b0 + r) * LDA + b0 + m], x[m], acc0);
                    }
                    x[r] = (r == col) ? 1.f : (r < col ? 0.f : -(acc0 + acc1));
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) sT[(b0 + r) * LDA + b0 + col] = x[r];
            }
            named_sync(1, 128);
            if (t == 0) TRACE(k, 24);
            // ... then the off-diagonal blocks, one block sub-diagonal per step and one block
            // per warp, on TF32 tensor-core tiles:  X = sum_{M=J}^{I-1} A_IM T_MJ,
            // T_IJ = -T_II X.
            {
                const int g = lane >> 2, tq = lane & 3;
                float* xs = sTmp + q * (16 * 20);
#pragma unroll 1
                for (int dd = 1; dd < 4; ++dd) {
                    const int J = q, I = q + dd;
                    if (I < 4) {
                        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        for (int M = J; M < I; ++M) {
#pragma unroll
                            for (int kk = 0; kk < 16; kk += 8) {
                                const float* ar = sA + (16 * I + g) * LDA + 16 * M + kk + tq;
                                const uint32_t a0 = f2tf32(ar[0]), a1 = f2tf32(ar[8 * LDA]),
                                               a2 = f2tf32(ar[4]), a3 = f2tf32(ar[8 * LDA + 4]);
#pragma unroll
                                for (int nt = 0; nt < 2; ++nt) {
                                    const float* br = sT + (16 * M + kk + tq) * LDA + 16 * J + 8 * nt + g;
                                    mma_tf32(acc[nt], a0, a1, a2, a3, f2tf32(br[0]), f2tf32(br[4 * LDA]));
                                }
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            xs[g * 20 + 8 * nt + 2 * tq] = acc[nt][0];
                            xs[g * 20 + 8 * nt + 2 * tq + 1] = acc[nt][1];
                            xs[(g + 8) * 20 + 8 * nt + 2 * tq] = acc[nt][2];
                            xs[(g + 8) * 20 + 8 * nt + 2 * tq + 1] = acc[nt][3];
                        }
                        __syncwarp();
                        float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                        for (int kk = 0; kk < 16; kk += 8) {
                            const float* ar = sT + (16 * I + g) * LDA + 16 * I + kk + tq;
                            const uint32_t a0 = f2tf32(ar[0]), a1 = f2tf32(ar[8 * LDA]),
                                           a2 = f2tf32(ar[4]), a3 = f2tf32(ar[8 * LDA + 4]);
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) {
                                const float* br = xs + (kk + tq) * 20 + 8 * nt + g;
                                mma_tf32(acc2[nt], a0, a1, a2, a3, f2tf32(br[0]), f2tf32(br[4 * 20]));
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            float* tr = sT + (16 * I + g) * LDA + 16 * J + 8 * nt + 2 * tq;
                            tr[0] = -acc2[nt][0];
                            tr[1] = -acc2[nt][1];
                            tr[8 * LDA] = -acc2[nt][2];
                            tr[8 * LDA + 1] = -acc2[nt][3];
                        }
                        __syncwarp();
                    }
                    named_sync(1, 128);
                    if (t == 0) TRACE(k, 24 + dd);
                }
            }
            if (t == 0) TRACE(k, 11);
            // TW = -T diag(beta e) (threads 0-63), TU = T diag(beta) (threads 64-127)
            if (t < 64 || NEEDU) {
                const float* cf = (t < 64) ? gb.be : gb.beta;
                const float sg = (t < 64) ? -1.f : 1.f;
                unsigned char* tile = sm + ((t < 64) ? S_TW : S_TU);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float row[8];
#pragma unroll
                    for (int q = 0; q < 8; q += 4) {
                        const int jj = 8 * ch + q;
                        const float4 tv = *reinterpret_cast<const float4*>(sT + i * LDA + jj);
                        const float4 fv = *reinterpret_cast<const float4*>(cf + jj);
                        row[q + 0] = (jj + 0 <= i) ? sg * tv.x * fv.x : 0.f;
                        row[q + 1] = (jj + 1 <= i) ? sg * tv.y * fv.y : 0.f;
                        row[q + 2] = (jj + 2 <= i) ? sg * tv.z * fv.z : 0.f;
                        row[q + 3] = (jj + 3 <= i) ? sg * tv.w * fv.w : 0.f;
                    }
                    st_chunk8(tile, i, ch, row);
                }
                fence_proxy_async_smem();
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_ET]);
            if (t == 0) TRACE(k, 12);
            // W'^T from D2 -> smem tile rows dk = t
            if (!group_wait(bars, B_MMA2, k & 1, errflag)) break;
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
            if (lane == 0) {
                mbar_arrive(&bars[B_EW]);
                mbar_arrive(&bars[B_GFREE0 + gs]);  // done with this chunk's gates
            }
            if (t == 0) TRACE(k, 13);
        }
    } else if (w >= 12 && OUT) {
        // ------------------------------------------------------------ output warps
        const int v = tid - 384;                     // TMEM lane = value column
        const uint32_t lb = uint32_t(32 * (w & 3)) << 16;
        __nv_bfloat16* sO = reinterpret_cast<__nv_bfloat16*>(sm + S_O);
        for (int k = 0; k < n; ++k) {
            const int gs = k & (NGATE - 1);
            const Gate& gb = gates[gs];
            if (!named_and(2, 128, warp_wait(bars, B_MMA5, k & 1, errflag))) break;
            if (v == 0) TRACE(k, 14);
            fence_after_sync();
            const float sc = P.scale;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float d4[32], d5[32];
                tmem_ld32(tm + lb + T_D4 + 32 * half, d4);
                tmem_ld32(tm + lb + T_D5 + 32 * half, d5);
                tmem_ld_wait();
                if (half == 1) {
                    fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_EPI]);
                }
#pragma unroll
                for (int qq = 0; qq < 32; ++qq) {
                    const int ii = 32 * half + qq;
                    sO[ii * LDO + v] = __float2bfloat16_rn(sc * fmaf(gb.e[ii], d4[qq], d5[qq]));
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
            tc_scan<TK_STATE>(P, maps, sm, j, t0, t1, cb, ce, x0, out, 0);
        } else {
            if (lj == 0) return;
            float* out = P.mbuf + (int64_t(gseg) * P.Hv + j) * KVN;
            if (ce <= cb) { copy_state(nullptr, out, true); return; }
            tc_scan<TK_TRANS>(P, maps, sm, j, t0, t1, cb, ce, nullptr, out, 0);
        }
    } else {
        if (lj == 0 || blockIdx.z != 0) return;
        const int cb = lj * P.L, w0 = cb - P.warmup;
        const float* x0 = w0 <= 0 ? h0 : nullptr;
        float* out = P.hin + (int64_t(gseg) * P.Hv + j) * KVN;
        tc_scan<TK_STATE>(P, maps, sm, j, t0, t1, max(w0, 0), cb, x0, out, 0);
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
