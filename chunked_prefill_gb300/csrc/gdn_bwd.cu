// Backward of the chunked gated delta rule (FlashQLA pages, agentlenshq "backward pass"
// paragraph: the dv, dh-scan, dq/dk/dw/dg and WY-backward steps).
//
// Per chunk, with the forward quantities of that chunk (gamma, e = exp(gamma), kd =
// exp(gamma_C - gamma), A, T = (I + A)^-1, W, U, V' = U - W h, P = (Q K^T) * D), the state h
// entering the chunk and dh the gradient w.r.t. the state leaving it (dOs = scale dO):
//
//   dV'  = P^T dOs + diag(kd) K dh
//   dh_in = e_C dh + Q^T diag(e) dOs - W^T dV'                     (reverse scan)
//   dP   = (dOs V'^T) on i >= j,  dQk = dP * D
//   dQ   = diag(e) dOs h^T + dQk K
//   dK   = dQk^T Q + diag(kd) (V' dh^T) + (dB + dB^T) K + diag(beta e) dYW
//   dW   = -dV' h^T,  dT = dW YW^T + dV' YU^T,  dYW = T^T dW,  dYU = T^T dV'
//   dA   = strictly-lower(-T^T dT T^T),  dB = diag(beta) (dA * Dm)
//   dV   = diag(beta) dYU
//   dbeta_i  = sum_j dA_ij (Bm * Dm)_ij + e_i <dYW_i, K_i> + <dYU_i, V_i>
//   dgamma_i = rowsum - colsum of (dP * P) and of (dA * A) + e_i <dOs_i, (Q h)_i>
//              + beta_i e_i <dYW_i, K_i> - r_i,   r_i = <(V' dh^T)_i, kd_i K_i>
//   dgamma_{C-1} += sum_i r_i + e_C <dh, h>,   dg = reverse in-chunk cumsum of dgamma
//
// Kernels: the reverse dh scan (per segment, context-parallel like the forward: segment
// partials from a zero gradient, a serial fix-up with the transposed segment transitions
// M^T, then the rerun that stores dh for every chunk), the chunk-parallel local-gradient
// kernel (one CTA per (chunk, v-head)) and, when q/k heads are shared, the fixed-order
// reduction of dq, dk over the v-heads of a group (no atomics: deterministic).
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace {

#ifdef GDN_TRACE
__device__ unsigned long long g_loc_trace[16];  // debug builds: SM clock at phase starts of CTA (0, 0)
#define LTRACE(e)                                                                               \
    do {                                                                                        \
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) g_loc_trace[e] = clock64(); \
    } while (0)
#else
#define LTRACE(e) \
    do {          \
    } while (0)
#endif

constexpr int NT = 256;
constexpr int64_t KVN = int64_t(KD) * VD;

__device__ __forceinline__ void seq_range(const Problem& P, int s, int64_t& t0, int64_t& t1) {
    if (P.cu) {
        t0 = P.cu[s];
        t1 = P.cu[s + 1];
    } else {
        t0 = int64_t(s) * P.T;
        t1 = t0 + P.T;
    }
}

template <typename Op, int C>
__device__ __forceinline__ void load_rows(Op* dst, int ld, const Op* src, int64_t gstride,
                                          int valid) {
    constexpr int VEC = 16 / sizeof(Op);
    constexpr int VPR = 128 / VEC;
    for (int idx = threadIdx.x; idx < C * VPR; idx += NT) {
        const int r = idx / VPR, cv = idx % VPR;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < valid) val = *reinterpret_cast<const uint4*>(src + r * gstride + cv * VEC);
        *reinterpret_cast<uint4*>(dst + r * ld + cv * VEC) = val;
    }
}

// in-chunk gates by warp 0: gamma (cumsum), e, kd, beta (rows >= c padded with g = beta = 0)
template <int C>
__device__ __forceinline__ void gates_warp0(float* sGam, float* sE, float* sKd) {
    const int lane = threadIdx.x & 31;
    constexpr int PER = C / 32;
    float vals[PER];
    float run = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        run += sGam[lane * PER + i];
        vals[i] = run;
    }
    float tot = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, tot, off);
        if (lane >= off) tot += y;
    }
    const float excl = tot - run;
    const float last = __shfl_sync(0xffffffffu, tot, 31);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const float gm = vals[i] + excl;
        sGam[lane * PER + i] = gm;
        sE[lane * PER + i] = expf(gm);
        sKd[lane * PER + i] = expf(last - gm);
    }
}

// T = (I + A)^-1 for a C x C strictly lower A in fp32 shared memory (row stride LDF):
// diagonal 16 x 16 blocks by substitution, then the off-diagonal blocks one block
// sub-diagonal at a time (T_IJ = -T_II sum_{M=J}^{I-1} A_IM T_MJ).  All NT threads.
template <int C, int LDF>
__device__ void tri_inverse(const float* sA, float* sT, float* sTmp) {
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    constexpr int NB = C / 16;
    if (w < NB && lane < 16) {
        const int b0 = 16 * w, col = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) acc = fmaf(sA[(b0 + r) * LDF + b0 + m], x[m], acc);
            x[r] = (r == col) ? 1.f : (r < col ? 0.f : -acc);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(b0 + r) * LDF + b0 + col] = x[r];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < NB; ++d) {
        const int nblk = NB - d;
        for (int e = tid; e < nblk * 256; e += NT) {
            const int J = e >> 8, r = (e >> 4) & 15, cc = e & 15, I = J + d;
            float acc = 0.f;
            for (int M = J; M < I; ++M) {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc = fmaf(sA[(16 * I + r) * LDF + 16 * M + m], sT[(16 * M + m) * LDF + 16 * J + cc], acc);
            }
            sTmp[(J * 16 + r) * 17 + cc] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * 256; e += NT) {
            const int J = e >> 8, r = (e >> 4) & 15, cc = e & 15, I = J + d;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                if (m <= r) acc = fmaf(sT[(16 * I + r) * LDF + 16 * I + m], sTmp[(J * 16 + m) * 17 + cc], acc);
            sT[(16 * I + r) * LDF + 16 * J + cc] = -acc;
        }
        __syncthreads();
    }
}

// =====================================================================================
// Reverse dh scan.  State dh (K x V) in registers (warp w: rows 16w..16w+15), an operand
// copy in shared memory.
// =====================================================================================
template <typename Op, int C>
struct ScanSmem {
    static constexpr int LDK = KD + OpTraits<Op>::PAD, LDC = C + OpTraits<Op>::PAD, LDF = C + 1;
    static constexpr size_t TILE = size_t(C) * LDK * sizeof(Op);
    static constexpr size_t CT = size_t(C) * LDC * sizeof(Op);
    static constexpr size_t FT = size_t(C) * LDF * 4;
    static constexpr size_t oK = 0, oQ = oK + TILE, oDO = oQ + TILE, oDOe = oDO + TILE,
                            oW = oDOe + TILE, oDV = oW + TILE, oX = oDV + TILE;
    static constexpr size_t oTW = oX + size_t(KD) * LDK * sizeof(Op), oP = oTW + CT;
    static constexpr size_t oA = oP + CT, oT = oA + FT, oTmp = oT + FT;
    static constexpr size_t oGam = oTmp + 3 * 16 * 17 * 4, oE = oGam + C * 4, oKd = oE + C * 4,
                            oBeta = oKd + C * 4;
    static constexpr size_t bytes = oBeta + C * 4;
    static_assert(bytes <= 232448, "shared memory budget");
};

template <typename Op, int C, bool HIST>
__device__ void bwd_scan(const BwdProblem& B, char* smem, int j, int64_t t0, int64_t t1, int cb,
                         int ce, const float* x0, float* x_out, int64_t hist_base) {
    using S = ScanSmem<Op, C>;
    constexpr int LDK = S::LDK, LDC = S::LDC, LDF = S::LDF;
    const Problem& P = B.f;
    // bf16: the chunk-local W' and P are read from the forward's preparation records
    constexpr bool RECS = sizeof(Op) == 2;
    Op* sK = reinterpret_cast<Op*>(smem + S::oK);
    Op* sQ = reinterpret_cast<Op*>(smem + S::oQ);
    Op* sDO = reinterpret_cast<Op*>(smem + S::oDO);
    Op* sDOe = reinterpret_cast<Op*>(smem + S::oDOe);
    Op* sW = reinterpret_cast<Op*>(smem + S::oW);
    Op* sDV = reinterpret_cast<Op*>(smem + S::oDV);
    Op* sX = reinterpret_cast<Op*>(smem + S::oX);
    Op* sTW = reinterpret_cast<Op*>(smem + S::oTW);
    Op* sP = reinterpret_cast<Op*>(smem + S::oP);
    float* sA = reinterpret_cast<float*>(smem + S::oA);
    float* sT = reinterpret_cast<float*>(smem + S::oT);
    float* sTmp = reinterpret_cast<float*>(smem + S::oTmp);
    float* sGam = reinterpret_cast<float*>(smem + S::oGam);
    float* sE = reinterpret_cast<float*>(smem + S::oE);
    float* sKd = reinterpret_cast<float*>(smem + S::oKd);
    float* sBeta = reinterpret_cast<float*>(smem + S::oBeta);

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int Hqk = P.Hqk, Hv = P.Hv, G = Hv / Hqk, qh = j / G;

    float X[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 16 * w + gq + 8 * h, c = 8 * n + 2 * tq;
            float a = 0.f, b = 0.f;
            if (x0) {
                const float2 v2 = *reinterpret_cast<const float2*>(x0 + r * VD + c);
                a = v2.x;
                b = v2.y;
            }
            X[n][2 * h] = a;
            X[n][2 * h + 1] = b;
        }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int r = 16 * w + gq, c = 8 * n + 2 * tq;
        st2(sX + r * LDK + c, X[n][0], X[n][1]);
        st2(sX + (r + 8) * LDK + c, X[n][2], X[n][3]);
    }

    constexpr int RB = C / 16, WPR = 8 / RB, COLS = 128 / WPR, NTC = COLS / 8;
    const int m0 = 16 * (w % RB), n0 = COLS * (w / RB);
    constexpr int RBk = 2 * C / 16, WPRk = 8 / RBk, COLSk = C / WPRk, NTk = COLSk / 8;
    static_assert(8 % RB == 0 && 8 % RBk == 0 && NTk >= 1, "warp tiling");
    const int mk0 = 16 * (w % RBk), nk0 = COLSk * (w / RBk);

    const int64_t qk_stride = int64_t(Hqk) * KD, v_stride = int64_t(Hv) * VD;
    const Op* qbase = reinterpret_cast<const Op*>(P.q) + qh * KD;
    const Op* kbase = reinterpret_cast<const Op*>(P.k) + qh * KD;
    const Op* dobase = reinterpret_cast<const Op*>(B.dO) + j * VD;
    const float sc = P.scale;

    for (int ch = ce - 1; ch >= cb; --ch) {
        const int64_t tc = t0 + int64_t(ch) * C;
        const int c = int((t1 - tc) < int64_t(C) ? (t1 - tc) : int64_t(C));
        if (HIST) {  // gradient w.r.t. the state leaving this chunk
            Op* hp = reinterpret_cast<Op*>(B.dhist) + ((hist_base + ch) * Hv + j) * KVN;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int r = 16 * w + gq, cc = 8 * n + 2 * tq;
                st2(hp + r * VD + cc, X[n][0], X[n][1]);
                st2(hp + (r + 8) * VD + cc, X[n][2], X[n][3]);
            }
        }
        load_rows<Op, C>(sK, LDK, kbase + tc * qk_stride, qk_stride, c);
        load_rows<Op, C>(sQ, LDK, qbase + tc * qk_stride, qk_stride, c);
        load_rows<Op, C>(sDO, LDK, dobase + tc * v_stride, v_stride, c);
        for (int i = tid; i < C; i += NT) {
            const bool ok = i < c;
            sGam[i] = ok ? P.g[(tc + i) * Hv + j] : 0.f;
            sBeta[i] = ok ? P.beta[(tc + i) * Hv + j] : 0.f;
        }
        __syncthreads();
        if (w == 0) gates_warp0<C>(sGam, sE, sKd);
        if (RECS) {
            // W' = -W and P come from the forward's chunk records (bf16, 128-byte swizzled
            // rows): unswizzle them into the padded operand tiles of this kernel
            const unsigned char* rec = static_cast<const unsigned char*>(P.prep) +
                                       ((hist_base + ch) * Hv + j) * P.prep_stride;
            for (int q = tid; q < 1024 + 512; q += NT) {
                if (q < 1024) {
                    const int blk = q >> 9, r = (q >> 3) & 63, cc = (q & 7) ^ (r & 7);
                    *reinterpret_cast<uint4*>(sW + r * LDK + blk * 64 + cc * 8) =
                        *reinterpret_cast<const uint4*>(rec + PREP_W + q * 16);
                } else {
                    const int q2 = q - 1024, r = q2 >> 3, cc = (q2 & 7) ^ (r & 7);
                    *reinterpret_cast<uint4*>(sP + r * LDC + cc * 8) =
                        *reinterpret_cast<const uint4*>(rec + PREP_P + q2 * 16);
                }
            }
            __syncthreads();  // gates
            for (int idx = tid; idx < C * KD; idx += NT) {
                const int i = idx / KD, v = idx % KD;
                sDOe[i * LDK + v] = from_f<Op>(sc * sE[i] * to_f(sDO[i * LDK + v]));
            }
            __syncthreads();
        } else {
        {
            float acc[NTk][4];
            zero_acc(acc);
            const bool qrows = mk0 >= C;
            warp_mma<NTk, false, true>(acc, qrows ? sQ : sK, LDK, sK, LDK, qrows ? mk0 - C : mk0, nk0, KD);
            float* dst = qrows ? sT : sA;
            const int rb = qrows ? mk0 - C : mk0;
#pragma unroll
            for (int n = 0; n < NTk; ++n) {
                const int cc = nk0 + 8 * n + 2 * tq;
                dst[(rb + gq) * LDF + cc] = acc[n][0];
                dst[(rb + gq) * LDF + cc + 1] = acc[n][1];
                dst[(rb + gq + 8) * LDF + cc] = acc[n][2];
                dst[(rb + gq + 8) * LDF + cc + 1] = acc[n][3];
            }
        }
        __syncthreads();
        for (int idx = tid; idx < C * C; idx += NT) {
            const int i = idx / C, jj = idx % C;
            const float d = expf(sGam[i] - sGam[jj]);
            sA[i * LDF + jj] = (i > jj) ? sBeta[i] * d * sA[i * LDF + jj] : 0.f;
            sP[i * LDC + jj] = from_f<Op>((i >= jj) ? d * sT[i * LDF + jj] : 0.f);
        }
        // dO scaled by scale * e_i (the Q^T diag(e) dOs operand)
        for (int idx = tid; idx < C * KD; idx += NT) {
            const int i = idx / KD, v = idx % KD;
            sDOe[i * LDK + v] = from_f<Op>(sc * sE[i] * to_f(sDO[i * LDK + v]));
        }
        __syncthreads();
        tri_inverse<C, LDF>(sA, sT, sTmp);
        for (int idx = tid; idx < C * C; idx += NT) {
            const int i = idx / C, jj = idx % C;
            const float t = (jj <= i) ? sT[i * LDF + jj] : 0.f;
            sTW[i * LDC + jj] = from_f<Op>(-t * sBeta[jj] * sE[jj]);
        }
        __syncthreads();
        {
            float wacc[NTC][4];
            zero_acc(wacc);
            warp_mma<NTC, false, false>(wacc, sTW, LDC, sK, LDK, m0, n0, C);
#pragma unroll
            for (int n = 0; n < NTC; ++n) {
                const int cc = n0 + 8 * n + 2 * tq;
                st2(sW + (m0 + gq) * LDK + cc, wacc[n][0], wacc[n][1]);
                st2(sW + (m0 + gq + 8) * LDK + cc, wacc[n][2], wacc[n][3]);
            }
        }
        }
        {  // dV' = scale P^T dO + diag(kd) K dh
            float a1[NTC][4], a2[NTC][4];
            zero_acc(a1);
            zero_acc(a2);
            warp_mma<NTC, true, false>(a1, sP, LDC, sDO, LDK, m0, n0, C);
            warp_mma<NTC, false, false>(a2, sK, LDK, sX, LDK, m0, n0, KD);
            const float k0 = sKd[m0 + gq], k1 = sKd[m0 + gq + 8];
#pragma unroll
            for (int n = 0; n < NTC; ++n) {
                const int cc = n0 + 8 * n + 2 * tq;
                st2(sDV + (m0 + gq) * LDK + cc, sc * a1[n][0] + k0 * a2[n][0], sc * a1[n][1] + k0 * a2[n][1]);
                st2(sDV + (m0 + gq + 8) * LDK + cc, sc * a1[n][2] + k1 * a2[n][2], sc * a1[n][3] + k1 * a2[n][3]);
            }
        }
        __syncthreads();
        {  // dh <- e_C dh + Q^T diag(e) dOs - W^T dV'   (sW holds -W)
            const float eC = sE[C - 1];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                X[n][0] *= eC;
                X[n][1] *= eC;
                X[n][2] *= eC;
                X[n][3] *= eC;
            }
            warp_mma<16, true, false>(X, sQ, LDK, sDOe, LDK, 16 * w, 0, C);
            warp_mma<16, true, false>(X, sW, LDK, sDV, LDK, 16 * w, 0, C);
        }
        __syncthreads();
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const int r = 16 * w + gq, cc = 8 * n + 2 * tq;
            st2(sX + r * LDK + cc, X[n][0], X[n][1]);
            st2(sX + (r + 8) * LDK + cc, X[n][2], X[n][3]);
        }
    }
    if (x_out) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const int r = 16 * w + gq, cc = 8 * n + 2 * tq;
            *reinterpret_cast<float2*>(x_out + r * VD + cc) = make_float2(X[n][0], X[n][1]);
            *reinterpret_cast<float2*>(x_out + (r + 8) * VD + cc) = make_float2(X[n][2], X[n][3]);
        }
    }
}

// Phase A of the reverse scan: the gradient entering segment lj >= 1 from its right end,
// started from zero (or from dht for the last segment) -> dhb[g].
template <typename Op, int C>
__global__ void __launch_bounds__(NT, 1) k_bwd_phase_a(BwdProblem B) {
    extern __shared__ __align__(128) char smem[];
    const Problem& P = B.f;
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N || lj == 0) return;
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + C - 1) / C);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const float* x0 = (lj == nseg - 1 && B.dht) ? B.dht + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    bwd_scan<Op, C, false>(B, smem, j, t0, t1, cb, ce, x0, B.dhb + (int64_t(gseg) * P.Hv + j) * KVN,
                           plan_chunk_off(P.plan, s));
}

// Phase C: every segment from its true right-end gradient, storing dh for every chunk; the
// first segment's result is dh0.
template <typename Op, int C>
__global__ void __launch_bounds__(NT, 1) k_bwd_phase_c(BwdProblem B) {
    extern __shared__ __align__(128) char smem[];
    const Problem& P = B.f;
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) return;
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_range(P, s, t0, t1);
    const int nt = int((t1 - t0 + C - 1) / C);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const float* x0 = (lj == nseg - 1) ? (B.dht ? B.dht + (int64_t(s) * P.Hv + j) * KVN : nullptr)
                                       : B.dhb + (int64_t(gseg + 1) * P.Hv + j) * KVN;
    float* x_out = (lj == 0 && B.dh0) ? B.dh0 + (int64_t(s) * P.Hv + j) * KVN : nullptr;
    bwd_scan<Op, C, true>(B, smem, j, t0, t1, cb, ce, x0, x_out, plan_chunk_off(P.plan, s));
}

// Reverse fix-up: dhb[g0+lj] = M_lj^T dhb[g0+lj+1] + dhb[g0+lj] for lj = nseg-2 .. 1.  The
// stored transitions are M^T (mbuf[m][r] = M[r][m]), so M^T x reads mbuf row-major; the
// matrix is staged through shared memory (stride 129: conflict-free row reads).
__global__ void __launch_bounds__(256) k_bwd_fixup(BwdProblem B) {
    extern __shared__ __align__(16) float fsm[];
    float* Ms = fsm;                 // 128 x 129
    float* xs = fsm + KD * 129;      // 128 x 8
    const Problem& P = B.f;
    const int s = blockIdx.x, j = blockIdx.y, cb = blockIdx.z * 8;
    const int g0 = plan_seg_off(P.plan, s), nseg = plan_seg_off(P.plan, s + 1) - g0;
    if (nseg <= 2) return;
    const int row = threadIdx.x & 127, c0 = (threadIdx.x >> 7) * 4;
    {
        const float4 x = *reinterpret_cast<const float4*>(
            B.dhb + (int64_t(g0 + nseg - 1) * P.Hv + j) * KVN + row * VD + cb + c0);
        *reinterpret_cast<float4*>(&xs[row * 8 + c0]) = x;
    }
    for (int lj = nseg - 2; lj >= 1; --lj) {
        const float* Mt = P.mbuf + (int64_t(g0 + lj) * P.Hv + j) * KVN;
        for (int idx = threadIdx.x; idx < KD * KD; idx += 256) Ms[(idx >> 7) * 129 + (idx & 127)] = Mt[idx];
        __syncthreads();
        float4* dst = reinterpret_cast<float4*>(B.dhb + (int64_t(g0 + lj) * P.Hv + j) * KVN + row * VD + cb + c0);
        float4 acc = *dst;
#pragma unroll 8
        for (int m = 0; m < KD; ++m) {
            const float a = Ms[row * 129 + m];
            const float4 xv = *reinterpret_cast<const float4*>(&xs[m * 8 + c0]);
            acc.x = fmaf(a, xv.x, acc.x);
            acc.y = fmaf(a, xv.y, acc.y);
            acc.z = fmaf(a, xv.z, acc.z);
            acc.w = fmaf(a, xv.w, acc.w);
        }
        __syncthreads();
        *reinterpret_cast<float4*>(&xs[row * 8 + c0]) = acc;
        *dst = acc;
    }
}

// =====================================================================================
// Local gradients, one CTA per (chunk, v-head).
// =====================================================================================
template <typename Op, int C>
struct LocSmem {
    static constexpr int LDK = KD + OpTraits<Op>::PAD, LDC = C + OpTraits<Op>::PAD, LDF = C + 1;
    static constexpr size_t TILE = size_t(C) * LDK * sizeof(Op);
    static constexpr size_t CT = size_t(C) * LDC * sizeof(Op);
    static constexpr size_t FT = size_t(C) * LDF * 4;
    // c x 128 tiles
    static constexpr size_t oK = 0, oQ = oK + TILE /* later dW */, oV = oQ + TILE,
                            oW = oV + TILE /* W', later dO */, oVP = oW + TILE, oDV = oVP + TILE;
    // TW, TU staging; fp32 A, T (the states h, dh are read from global memory)
    static constexpr size_t oH = oDV + TILE;
    static constexpr size_t oDH = oH + 2 * CT;
    static constexpr size_t oFDB = oDH + 2 * FT;
    static constexpr size_t oOP = oFDB + FT, oOT = oOP + CT, oO1 = oOT + CT, oO2 = oO1 + CT;
    static constexpr size_t oTmp = oO1;                      // inverse scratch (phase 1 only)
    static constexpr size_t oGam = oO2 + CT, oE = oGam + C * 4, oKd = oE + C * 4,
                            oBeta = oKd + C * 4;
    static constexpr size_t oRow = oBeta + C * 4;            // [4][C] row partials
    static constexpr size_t oCol = oRow + 4 * C * 4;         // [4][C] column partials
    static constexpr size_t oRb = oCol + 4 * C * 4;          // [4][C] dbeta partials
    static constexpr size_t oDg = oRb + 4 * C * 4, oDb = oDg + C * 4, oRed = oDb + C * 4;
    static constexpr size_t bytes = oRed + 64;
    static_assert(CT >= 3 * 16 * 17 * 4, "inverse scratch alias");
    static_assert(bytes <= 232448, "shared memory budget");
};

// sum of v over the four lanes that share a fragment row (t = lane & 3)
__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}
// sum of v over the eight lanes that share a fragment column (g = lane >> 2)
__device__ __forceinline__ float col_sum8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    return v;
}

template <typename Op, int C, int NTL>
__global__ void __launch_bounds__(NTL, 1) k_bwd_local(BwdProblem B, int64_t items) {
    using S = LocSmem<Op, C>;
    constexpr int LDK = S::LDK, LDC = S::LDC, LDF = S::LDF;
    extern __shared__ __align__(128) char smem[];
    const Problem& P = B.f;
    // One CTA per SM walks the (chunk, v-head) items item = chunk Hv + v-head with a stride of
    // the grid (fp32 test mode; bf16 runs the tensor-core kernel of gdn_bwd_tc.cu).
    struct Item {
        int gch, j, s, ch, c, qh;
        int64_t t0, t1, tc;
    };
    auto locate = [&](int64_t item, Item& x) -> bool {
        x.gch = int(item / P.Hv);
        x.j = int(item % P.Hv);
        x.qh = x.j / (P.Hv / P.Hqk);
        if (x.gch >= plan_chunk_off(P.plan, P.N)) return false;
        int lo = 0, hi = P.N - 1;  // chunk -> (sequence, local chunk) by binary search
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (plan_chunk_off(P.plan, mid) <= x.gch) lo = mid;
            else hi = mid - 1;
        }
        x.s = lo;
        x.ch = x.gch - plan_chunk_off(P.plan, x.s);
        seq_range(P, x.s, x.t0, x.t1);
        x.tc = x.t0 + int64_t(x.ch) * C;
        if (x.tc >= x.t1) return false;
        x.c = int((x.t1 - x.tc) < int64_t(C) ? (x.t1 - x.tc) : int64_t(C));
        return true;
    };
#pragma unroll 1
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    Item cur;
    if (!locate(item, cur)) continue;
    const int gch = cur.gch, j = cur.j, s = cur.s, ch = cur.ch;
    const int64_t t0 = cur.t0, t1 = cur.t1, tc = cur.tc;
    (void)s;
    (void)ch;
    (void)t0;
    (void)t1;
    const int c = cur.c;
    Op* tK = reinterpret_cast<Op*>(smem + S::oK);
    Op* tQ = reinterpret_cast<Op*>(smem + S::oQ);
    Op* tDW = tQ;
    Op* tV = reinterpret_cast<Op*>(smem + S::oV);
    Op* tW = reinterpret_cast<Op*>(smem + S::oW);
    Op* tDO = tW;
    Op* tVP = reinterpret_cast<Op*>(smem + S::oVP);
    Op* tDV = reinterpret_cast<Op*>(smem + S::oDV);
    Op* oTW = reinterpret_cast<Op*>(smem + S::oH);
    Op* oTU = reinterpret_cast<Op*>(smem + S::oH + S::CT);
    float* fA = reinterpret_cast<float*>(smem + S::oDH);
    float* fT = reinterpret_cast<float*>(smem + S::oDH + S::FT);
    float* fDB = reinterpret_cast<float*>(smem + S::oFDB);
    Op* oP = reinterpret_cast<Op*>(smem + S::oOP);
    Op* oT = reinterpret_cast<Op*>(smem + S::oOT);
    Op* oX1 = reinterpret_cast<Op*>(smem + S::oO1);
    Op* oX2 = reinterpret_cast<Op*>(smem + S::oO2);
    float* sTmp = reinterpret_cast<float*>(smem + S::oTmp);
    float* sGam = reinterpret_cast<float*>(smem + S::oGam);
    float* sE = reinterpret_cast<float*>(smem + S::oE);
    float* sKd = reinterpret_cast<float*>(smem + S::oKd);
    float* sBeta = reinterpret_cast<float*>(smem + S::oBeta);
    float* rowp = reinterpret_cast<float*>(smem + S::oRow);
    float* rbp = reinterpret_cast<float*>(smem + S::oRb);
    float* colp = reinterpret_cast<float*>(smem + S::oCol);
    float* sDg = reinterpret_cast<float*>(smem + S::oDg);
    float* sDb = reinterpret_cast<float*>(smem + S::oDb);
    float* sRed = reinterpret_cast<float*>(smem + S::oRed);

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int Hqk = P.Hqk, Hv = P.Hv, G = Hv / Hqk, qh = j / G;
    const float sc = P.scale;
    const int64_t qk_stride = int64_t(Hqk) * KD, v_stride = int64_t(Hv) * VD;
    const Op* hsrc = reinterpret_cast<const Op*>(P.hist) + (int64_t(gch) * Hv + j) * KVN;
    const Op* dhsrc = reinterpret_cast<const Op*>(B.dhist) + (int64_t(gch) * Hv + j) * KVN;
    // state operands: the global tensors directly
    const Op* sH = hsrc;
    const Op* sDH = dhsrc;
    constexpr int LDS = VD;

    constexpr int RB = C / 16, WPR = (NTL / 32) / RB, COLS = 128 / WPR, NTC = COLS / 8;
    constexpr int CCOLS = C / WPR, NTS = CCOLS / 8;
    static_assert(NTS >= 1 && WPR <= 4 && RB <= 4, "warp tiling");
    const int m0 = 16 * (w % RB), n0 = COLS * (w / RB), s0 = CCOLS * (w / RB);
    const int cgrp = w / RB, rgrp = w % RB;
    const int r0 = m0 + gq, r1 = m0 + gq + 8;

    LTRACE(0);
    // ---- phase 1: tiles, gates, K K^T, Q K^T, A, P, T
    {
        load_rows<Op, C>(tK, LDK, reinterpret_cast<const Op*>(P.k) + qh * KD + tc * qk_stride, qk_stride, c);
        load_rows<Op, C>(tQ, LDK, reinterpret_cast<const Op*>(P.q) + qh * KD + tc * qk_stride, qk_stride, c);
        load_rows<Op, C>(tV, LDK, reinterpret_cast<const Op*>(P.v) + j * VD + tc * v_stride, v_stride, c);
    }
    for (int i = tid; i < C; i += NTL) {
        const bool ok = i < c;
        sGam[i] = ok ? P.g[(tc + i) * Hv + j] : 0.f;
        sBeta[i] = ok ? P.beta[(tc + i) * Hv + j] : 0.f;
        sDg[i] = 0.f;
        sDb[i] = 0.f;
    }
    __syncthreads();
    if (w == 0) gates_warp0<C>(sGam, sE, sKd);
    float acc[NTC][4];
    {
    {
        float a1[NTS][4], a2[NTS][4];
        zero_acc(a1);
        zero_acc(a2);
        warp_mma<NTS, false, true>(a1, tK, LDK, tK, LDK, m0, s0, KD);
        warp_mma<NTS, false, true>(a2, tQ, LDK, tK, LDK, m0, s0, KD);
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const int cc = s0 + 8 * n + 2 * tq;
            fDB[r0 * LDF + cc] = a1[n][0];
            fDB[r0 * LDF + cc + 1] = a1[n][1];
            fDB[r1 * LDF + cc] = a1[n][2];
            fDB[r1 * LDF + cc + 1] = a1[n][3];
            fT[r0 * LDF + cc] = a2[n][0];
            fT[r0 * LDF + cc + 1] = a2[n][1];
            fT[r1 * LDF + cc] = a2[n][2];
            fT[r1 * LDF + cc + 1] = a2[n][3];
        }
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += NTL) {
        const int i = idx / C, jj = idx % C;
        const float d = expf(sGam[i] - sGam[jj]);
        const float db = (i > jj) ? d * fDB[i * LDF + jj] : 0.f;
        fDB[i * LDF + jj] = db;                       // Dm * Bm
        fA[i * LDF + jj] = sBeta[i] * db;             // A
        oP[i * LDC + jj] = from_f<Op>((i >= jj) ? d * fT[i * LDF + jj] : 0.f);
    }
    __syncthreads();
    tri_inverse<C, LDF>(fA, fT, sTmp);
    for (int idx = tid; idx < C * C; idx += NTL) {
        const int i = idx / C, jj = idx % C;
        const float t = (jj <= i) ? fT[i * LDF + jj] : 0.f;
        oT[i * LDC + jj] = from_f<Op>(t);
        oTW[i * LDC + jj] = from_f<Op>(-t * sBeta[jj] * sE[jj]);
        oTU[i * LDC + jj] = from_f<Op>(t * sBeta[jj]);
    }
    __syncthreads();

    LTRACE(1);
    // ---- phase 2: W' = -T diag(beta e) K, U = T diag(beta) V, V' = U + W' h
    {
        float wacc[NTC][4];
        zero_acc(wacc);
        warp_mma<NTC, false, false>(wacc, oTW, LDC, tK, LDK, m0, n0, C);
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            st2(tW + r0 * LDK + cc, wacc[n][0], wacc[n][1]);
            st2(tW + r1 * LDK + cc, wacc[n][2], wacc[n][3]);
        }
        zero_acc(acc);
        warp_mma<NTC, false, false>(acc, oTU, LDC, tV, LDK, m0, n0, C);
    }
    }
    __syncthreads();  // TW, TU consumed: the h tile may overwrite them
    __syncthreads();
    warp_mma<NTC, false, false>(acc, tW, LDK, sH, LDS, m0, n0, KD);
#pragma unroll
    for (int n = 0; n < NTC; ++n) {
        const int cc = n0 + 8 * n + 2 * tq;
        st2(tVP + r0 * LDK + cc, acc[n][0], acc[n][1]);
        st2(tVP + r1 * LDK + cc, acc[n][2], acc[n][3]);
    }
    __syncthreads();  // W' consumed: dO may overwrite it; T fp32 consumed: dh may overwrite it

    LTRACE(2);
    // ---- phase 3: dO, dh; dV' = scale P^T dO + diag(kd) K dh
    {
        load_rows<Op, C>(tDO, LDK, reinterpret_cast<const Op*>(B.dO) + j * VD + tc * v_stride, v_stride, c);
    }
    __syncthreads();
    {
        float a1[NTC][4], a2[NTC][4];
        zero_acc(a1);
        zero_acc(a2);
        warp_mma<NTC, true, false>(a1, oP, LDC, tDO, LDK, m0, n0, C);
        warp_mma<NTC, false, false>(a2, tK, LDK, sDH, LDS, m0, n0, KD);
        const float k0 = sKd[r0], k1 = sKd[r1];
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            st2(tDV + r0 * LDK + cc, sc * a1[n][0] + k0 * a2[n][0], sc * a1[n][1] + k0 * a2[n][1]);
            st2(tDV + r1 * LDK + cc, sc * a1[n][2] + k1 * a2[n][2], sc * a1[n][3] + k1 * a2[n][3]);
        }
    }
    // dP = scale dO V'^T on i >= j; dgamma += rowsum - colsum of dP * P; dQk = dP * D -> oX1
    {
        float dp[NTS][4];
        zero_acc(dp);
        warp_mma<NTS, false, true>(dp, tDO, LDK, tVP, LDK, m0, s0, VD);
        float rs0 = 0.f, rs1 = 0.f;
        float cs[NTS][2];
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const int cc = s0 + 8 * n + 2 * tq;
            float pp[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rr = (e < 2) ? r0 : r1, cj = cc + (e & 1);
                float v = (rr >= cj) ? sc * dp[n][e] : 0.f;
                dp[n][e] = v;
                pp[e] = v * to_f(oP[rr * LDC + cj]);
            }
            rs0 += pp[0] + pp[1];
            rs1 += pp[2] + pp[3];
            cs[n][0] = pp[0] + pp[2];
            cs[n][1] = pp[1] + pp[3];
        }
        rs0 = quad_sum(rs0);
        rs1 = quad_sum(rs1);
        if (tq == 0) {
            rowp[cgrp * C + r0] = rs0;
            rowp[cgrp * C + r1] = rs1;
        }
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const float c0s = col_sum8(cs[n][0]), c1s = col_sum8(cs[n][1]);
            if (gq == 0) {
                colp[rgrp * C + s0 + 8 * n + 2 * tq] = c0s;
                colp[rgrp * C + s0 + 8 * n + 2 * tq + 1] = c1s;
            }
        }
        // dQk = dP * D
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const int cc = s0 + 8 * n + 2 * tq;
            const float d00 = expf(sGam[r0] - sGam[cc]), d01 = expf(sGam[r0] - sGam[cc + 1]);
            const float d10 = expf(sGam[r1] - sGam[cc]), d11 = expf(sGam[r1] - sGam[cc + 1]);
            st2(oX1 + r0 * LDC + cc, dp[n][0] * (r0 >= cc ? d00 : 0.f), dp[n][1] * (r0 >= cc + 1 ? d01 : 0.f));
            st2(oX1 + r1 * LDC + cc, dp[n][2] * (r1 >= cc ? d10 : 0.f), dp[n][3] * (r1 >= cc + 1 ? d11 : 0.f));
        }
    }
    __syncthreads();
    for (int i = tid; i < C; i += NTL) {  // fold the dP * P row/column sums into dgamma
        float v = 0.f;
        for (int q = 0; q < WPR; ++q) v += rowp[q * C + i];
        for (int q = 0; q < RB; ++q) v -= colp[q * C + i];
        sDg[i] += v;
    }
    __syncthreads();

    LTRACE(3);
    // ---- phase 4: dQ = scale diag(e) dO h^T + dQk K; e_i <dOs_i, (Q h)_i>; <dh, h>
    {
        float a1[NTC][4], a2[NTC][4];
        zero_acc(a1);
        zero_acc(a2);
        warp_mma<NTC, false, true>(a1, tDO, LDK, sH, LDS, m0, n0, VD);
        warp_mma<NTC, false, false>(a2, oX1, LDC, tK, LDK, m0, n0, C);
        const float e0 = sc * sE[r0], e1 = sc * sE[r1];
        float* dqp = B.dqp;
        // <dO_i, (Q h)_i> = <Q_i, (dO h^T)_i>: row sums of Q * (dO h^T), no Q h product needed
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            rs0 += a1[n][0] * to_f(tQ[r0 * LDK + cc]) + a1[n][1] * to_f(tQ[r0 * LDK + cc + 1]);
            rs1 += a1[n][2] * to_f(tQ[r1 * LDK + cc]) + a1[n][3] * to_f(tQ[r1 * LDK + cc + 1]);
        }
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            const float q00 = e0 * a1[n][0] + a2[n][0], q01 = e0 * a1[n][1] + a2[n][1];
            const float q10 = e1 * a1[n][2] + a2[n][2], q11 = e1 * a1[n][3] + a2[n][3];
            if (dqp) {
                if (r0 < c) *reinterpret_cast<float2*>(dqp + ((tc + r0) * Hv + j) * KD + cc) = make_float2(q00, q01);
                if (r1 < c) *reinterpret_cast<float2*>(dqp + ((tc + r1) * Hv + j) * KD + cc) = make_float2(q10, q11);
            } else {
                Op* dq = reinterpret_cast<Op*>(B.dq) + qh * KD;
                if (r0 < c) st2(dq + (tc + r0) * qk_stride + cc, q00, q01);
                if (r1 < c) st2(dq + (tc + r1) * qk_stride + cc, q10, q11);
            }
        }
        rs0 = quad_sum(rs0);
        rs1 = quad_sum(rs1);
        if (tq == 0) {
            rowp[cgrp * C + r0] = rs0;
            rowp[cgrp * C + r1] = rs1;
        }
        // <dh, h>
        float hd = 0.f;
        for (int idx = tid; idx < KD * VD; idx += NTL) {
            const int r = idx / VD, v = idx % VD;
            hd += to_f(sDH[r * LDS + v]) * to_f(sH[r * LDS + v]);
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, off);
        if (lane == 0) sRed[w] = hd;
    }
    __syncthreads();
    for (int i = tid; i < C; i += NTL) {
        float v = 0.f;
        for (int q = 0; q < WPR; ++q) v += rowp[q * C + i];
        sDg[i] += sc * sE[i] * v;
    }
    if (tid == 0) {
        float hd = 0.f;
        for (int q = 0; q < NTL / 32; ++q) hd += sRed[q];
        sRed[8] = hd;
    }
    __syncthreads();

    LTRACE(4);
    // ---- phase 5: dK = dQk^T Q + diag(kd) (V' dh^T) (+ later terms); r_i
    float dk[NTC][4];
    {
        zero_acc(dk);
        warp_mma<NTC, true, false>(dk, oX1, LDC, tQ, LDK, m0, n0, C);
        float a2[NTC][4];
        zero_acc(a2);
        warp_mma<NTC, false, true>(a2, tVP, LDK, sDH, LDS, m0, n0, VD);
        const float k0 = sKd[r0], k1 = sKd[r1];
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            rs0 += a2[n][0] * to_f(tK[r0 * LDK + cc]) + a2[n][1] * to_f(tK[r0 * LDK + cc + 1]);
            rs1 += a2[n][2] * to_f(tK[r1 * LDK + cc]) + a2[n][3] * to_f(tK[r1 * LDK + cc + 1]);
            dk[n][0] += k0 * a2[n][0];
            dk[n][1] += k0 * a2[n][1];
            dk[n][2] += k1 * a2[n][2];
            dk[n][3] += k1 * a2[n][3];
        }
        rs0 = quad_sum(rs0) * k0;
        rs1 = quad_sum(rs1) * k1;
        if (tq == 0) {
            rowp[cgrp * C + r0] = rs0;
            rowp[cgrp * C + r1] = rs1;
        }
    }
    __syncthreads();
    if (tid == 0) {  // r_i enters dgamma_i with a minus sign, and their sum at the chunk end
        float rsum = 0.f;
        for (int i = 0; i < C; ++i) {
            float v = 0.f;
            for (int q = 0; q < WPR; ++q) v += rowp[q * C + i];
            sDg[i] -= v;
            rsum += v;
        }
        sDg[C - 1] += rsum + sE[C - 1] * sRed[8];
    }
    __syncthreads();

    LTRACE(5);
    // ---- phase 6: dW = -dV' h^T -> tile (reuses the Q tile)
    {
        float a1[NTC][4];
        zero_acc(a1);
        warp_mma<NTC, false, true>(a1, tDV, LDK, sH, LDS, m0, n0, VD);
        __syncthreads();  // Q tile no longer read
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            st2(tDW + r0 * LDK + cc, -a1[n][0], -a1[n][1]);
            st2(tDW + r1 * LDK + cc, -a1[n][2], -a1[n][3]);
        }
    }
    __syncthreads();

    LTRACE(6);
    // ---- phase 7: dT = (dW K^T) diag(beta e) + (dV' V^T) diag(beta) -> fA (fp32) -> oX2
    {
        float a1[NTS][4], a2[NTS][4];
        zero_acc(a1);
        zero_acc(a2);
        warp_mma<NTS, false, true>(a1, tDW, LDK, tK, LDK, m0, s0, KD);
        warp_mma<NTS, false, true>(a2, tDV, LDK, tV, LDK, m0, s0, VD);
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const int cc = s0 + 8 * n + 2 * tq;
            const float be0 = sBeta[cc] * sE[cc], be1 = sBeta[cc + 1] * sE[cc + 1];
            const float b0 = sBeta[cc], b1 = sBeta[cc + 1];
            st2(oX2 + r0 * LDC + cc, a1[n][0] * be0 + a2[n][0] * b0, a1[n][1] * be1 + a2[n][1] * b1);
            st2(oX2 + r1 * LDC + cc, a1[n][2] * be0 + a2[n][2] * b0, a1[n][3] * be1 + a2[n][3] * b1);
        }
    }
    __syncthreads();

    LTRACE(7);
    // ---- phase 8: dYW = T^T dW, dYU = T^T dV'; dV = diag(beta) dYU; dK += diag(beta e) dYW
    {
        float yw[NTC][4], yu[NTC][4];
        zero_acc(yw);
        zero_acc(yu);
        warp_mma<NTC, true, false>(yw, oT, LDC, tDW, LDK, m0, n0, C);
        warp_mma<NTC, true, false>(yu, oT, LDC, tDV, LDK, m0, n0, C);
        const float be0 = sBeta[r0] * sE[r0], be1 = sBeta[r1] * sE[r1];
        const float b0 = sBeta[r0], b1 = sBeta[r1];
        float tw0 = 0.f, tw1 = 0.f, tu0 = 0.f, tu1 = 0.f;
        Op* dv = reinterpret_cast<Op*>(B.dv) + j * VD;
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            tw0 += yw[n][0] * to_f(tK[r0 * LDK + cc]) + yw[n][1] * to_f(tK[r0 * LDK + cc + 1]);
            tw1 += yw[n][2] * to_f(tK[r1 * LDK + cc]) + yw[n][3] * to_f(tK[r1 * LDK + cc + 1]);
            tu0 += yu[n][0] * to_f(tV[r0 * LDK + cc]) + yu[n][1] * to_f(tV[r0 * LDK + cc + 1]);
            tu1 += yu[n][2] * to_f(tV[r1 * LDK + cc]) + yu[n][3] * to_f(tV[r1 * LDK + cc + 1]);
            dk[n][0] += be0 * yw[n][0];
            dk[n][1] += be0 * yw[n][1];
            dk[n][2] += be1 * yw[n][2];
            dk[n][3] += be1 * yw[n][3];
            if (r0 < c) st2(dv + (tc + r0) * v_stride + cc, b0 * yu[n][0], b0 * yu[n][1]);
            if (r1 < c) st2(dv + (tc + r1) * v_stride + cc, b1 * yu[n][2], b1 * yu[n][3]);
        }
        tw0 = quad_sum(tw0);
        tw1 = quad_sum(tw1);
        tu0 = quad_sum(tu0);
        tu1 = quad_sum(tu1);
        if (tq == 0) {
            rowp[cgrp * C + r0] = tw0;
            rowp[cgrp * C + r1] = tw1;
            colp[cgrp * C + r0] = tu0;   // (row sums of dYU * V)
            colp[cgrp * C + r1] = tu1;
        }
    }
    __syncthreads();
    for (int i = tid; i < C; i += NTL) {
        float tw = 0.f, tu = 0.f;
        for (int q = 0; q < WPR; ++q) {
            tw += rowp[q * C + i];
            tu += colp[q * C + i];
        }
        sDb[i] += sE[i] * tw + tu;
        sDg[i] += sBeta[i] * sE[i] * tw;
    }
    __syncthreads();

    LTRACE(8);
    // ---- phase 9: Z = dT T^T; dA = strictly-lower(-T^T Z); dB = diag(beta) dA * Dm
    {
        float z[NTS][4];
        zero_acc(z);
        warp_mma<NTS, false, true>(z, oX2, LDC, oT, LDC, m0, s0, C);
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const int cc = s0 + 8 * n + 2 * tq;
            st2(oX1 + r0 * LDC + cc, z[n][0], z[n][1]);
            st2(oX1 + r1 * LDC + cc, z[n][2], z[n][3]);
        }
    }
    __syncthreads();
    {
        float da[NTS][4];
        zero_acc(da);
        warp_mma<NTS, true, false>(da, oT, LDC, oX1, LDC, m0, s0, C);
        float rs0 = 0.f, rs1 = 0.f, ra0 = 0.f, ra1 = 0.f;
        float cs[NTS][2];
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const int cc = s0 + 8 * n + 2 * tq;
            float aa[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int rr = (e < 2) ? r0 : r1, cj = cc + (e & 1);
                const float dav = (rr > cj) ? -da[n][e] : 0.f;
                const float db = fDB[rr * LDF + cj];
                aa[e] = dav * sBeta[rr] * db;                 // dA * A
                // dB = beta_i dA_ij Dm_ij (dav is zero on and above the diagonal), in place of
                // the Dm * Bm entry just read
                fDB[rr * LDF + cj] = (rr > cj) ? sBeta[rr] * dav * expf(sGam[rr] - sGam[cj]) : 0.f;
                if (e < 2) rs0 += dav * db; else rs1 += dav * db;
            }
            ra0 += aa[0] + aa[1];
            ra1 += aa[2] + aa[3];
            cs[n][0] = aa[0] + aa[2];
            cs[n][1] = aa[1] + aa[3];
        }
        rs0 = quad_sum(rs0);
        rs1 = quad_sum(rs1);
        ra0 = quad_sum(ra0);
        ra1 = quad_sum(ra1);
        if (tq == 0) {
            rowp[cgrp * C + r0] = ra0;
            rowp[cgrp * C + r1] = ra1;
            rbp[cgrp * C + r0] = rs0;    // dbeta partial (dA * Dm * Bm row sums)
            rbp[cgrp * C + r1] = rs1;
        }
#pragma unroll
        for (int n = 0; n < NTS; ++n) {
            const float c0s = col_sum8(cs[n][0]), c1s = col_sum8(cs[n][1]);
            if (gq == 0) {
                colp[rgrp * C + s0 + 8 * n + 2 * tq] = c0s;
                colp[rgrp * C + s0 + 8 * n + 2 * tq + 1] = c1s;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < C; i += NTL) {
        float ra = 0.f, ca = 0.f, rb = 0.f;
        for (int q = 0; q < WPR; ++q) {
            ra += rowp[q * C + i];
            rb += rbp[q * C + i];
        }
        for (int q = 0; q < RB; ++q) ca += colp[q * C + i];
        sDg[i] += ra - ca;
        sDb[i] += rb;
    }
    // (dB + dB^T) as an MMA operand
    for (int idx = tid; idx < C * C; idx += NTL) {
        const int i = idx / C, jj = idx % C;
        oX2[i * LDC + jj] = from_f<Op>(fDB[i * LDF + jj] + fDB[jj * LDF + i]);
    }
    __syncthreads();

    LTRACE(9);
    // ---- phase 10: dK += (dB + dB^T) K; store dK
    warp_mma<NTC, false, false>(dk, oX2, LDC, tK, LDK, m0, n0, C);
    {
        float* dkp = B.dkp;
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            if (dkp) {
                if (r0 < c) *reinterpret_cast<float2*>(dkp + ((tc + r0) * Hv + j) * KD + cc) = make_float2(dk[n][0], dk[n][1]);
                if (r1 < c) *reinterpret_cast<float2*>(dkp + ((tc + r1) * Hv + j) * KD + cc) = make_float2(dk[n][2], dk[n][3]);
            } else {
                Op* dkk = reinterpret_cast<Op*>(B.dk) + qh * KD;
                if (r0 < c) st2(dkk + (tc + r0) * qk_stride + cc, dk[n][0], dk[n][1]);
                if (r1 < c) st2(dkk + (tc + r1) * qk_stride + cc, dk[n][2], dk[n][3]);
            }
        }
    }
    LTRACE(10);
    // ---- dg = reverse in-chunk cumsum of dgamma; dbeta
    if (w == 0) {
        constexpr int PER = C / 32;
        float vals[PER];
        float run = 0.f;
#pragma unroll
        for (int i = PER - 1; i >= 0; --i) {   // suffix sums inside the lane's rows
            run += sDg[lane * PER + i];
            vals[i] = run;
        }
        float tot = run;                        // suffix scan over lanes (from the top)
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_down_sync(0xffffffffu, tot, off);
            if (lane + off < 32) tot += y;
        }
        const float excl = tot - run;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int r = lane * PER + i;
            if (r < c) {
                B.dg[(tc + r) * Hv + j] = vals[i] + excl;
                B.dbeta[(tc + r) * Hv + j] = sDb[r];
            }
        }
    }
    __syncthreads();  // the next item re-initialises the gate and partial-sum arrays
    }
}

// dq, dk = sum over the G v-heads of each q/k head, in head order (deterministic).
template <typename Op>
__global__ void k_bwd_reduce(BwdProblem B, int64_t T_total) {
    const Problem& P = B.f;
    const int G = P.Hv / P.Hqk;
    const int64_t n = T_total * P.Hqk * (KD / 2);
    for (int64_t idx = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; idx < n;
         idx += int64_t(gridDim.x) * blockDim.x) {
        const int64_t t = idx / (P.Hqk * (KD / 2));
        const int rem = int(idx % (P.Hqk * (KD / 2)));
        const int qh = rem / (KD / 2), d2 = (rem % (KD / 2)) * 2;
        float q0 = 0.f, q1 = 0.f, k0 = 0.f, k1 = 0.f;
        for (int jj = qh * G; jj < (qh + 1) * G; ++jj) {
            const float2 a = *reinterpret_cast<const float2*>(B.dqp + (t * P.Hv + jj) * KD + d2);
            const float2 b = *reinterpret_cast<const float2*>(B.dkp + (t * P.Hv + jj) * KD + d2);
            q0 += a.x;
            q1 += a.y;
            k0 += b.x;
            k1 += b.y;
        }
        st2(reinterpret_cast<Op*>(B.dq) + (t * P.Hqk + qh) * KD + d2, q0, q1);
        st2(reinterpret_cast<Op*>(B.dk) + (t * P.Hqk + qh) * KD + d2, k0, k1);
    }
}

template <typename Op, int C>
cudaError_t launch_bwd_t(const BwdProblem& B, cudaStream_t st) {
    // bf16: the tensor-core reverse scan and local-gradient kernels; fp32 test mode: the
    // CUDA-core kernels of this file
    const Problem& P = B.f;
    using SS = ScanSmem<Op, C>;
    using LS = LocSmem<Op, C>;
    constexpr bool TC = sizeof(Op) == 2;
    cudaError_t e;
    const int fix_smem = (KD * 129 + KD * 8) * 4;
    e = smem_attr(k_bwd_fixup, fix_smem);
    if (e != cudaSuccess) return e;
    if constexpr (!TC) {
        e = cudaFuncSetAttribute(k_bwd_phase_a<Op, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SS::bytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_bwd_phase_c<Op, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SS::bytes));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(k_bwd_local<Op, C, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(LS::bytes));
        if (e != cudaSuccess) return e;
    }
    const int64_t T_total = P.cu ? P.T : int64_t(P.N) * P.T;
    if (TC && P.dec && B.rrerun) {
        // decay-bounded exact mode (the forward's decisions in P.dec): first pass from the
        // segments' right ends, the reverse fix-up only where a transition is not negligible,
        // the correction of the segments left with unwritten gradients
        timing_begin("bwd_dh_pass1", st);
        e = launch_bwd_scan_tc(B, 2, T_total, st);
        if (e != cudaSuccess) return e;
        timing_end(st);
        timing_begin("bwd_fixup", st);
        launch_bwd_fixup_tc(B, st);
        timing_end(st);
        timing_begin("bwd_dh_correction", st);
        e = launch_bwd_scan_tc(B, 3, T_total, st);
        if (e != cudaSuccess) return e;
        timing_end(st);
    } else if (P.cp != CP_NONE) {
        timing_begin("bwd_phase_a", st);
        if constexpr (TC) {
            e = launch_bwd_scan_tc(B, 0, T_total, st);
            if (e != cudaSuccess) return e;
        } else {
            k_bwd_phase_a<Op, C><<<dim3(P.total_segs, P.Hv), NT, SS::bytes, st>>>(B);
        }
        timing_end(st);
        timing_begin("bwd_fixup", st);
        if (TC && P.mbuf_t)
            launch_bwd_fixup_tc(B, st);
        else
            k_bwd_fixup<<<dim3(P.N, P.Hv, VD / 8), 256, fix_smem, st>>>(B);
        timing_end(st);
    }
    if (!(TC && P.dec && B.rrerun)) {
        timing_begin("bwd_dh_scan", st);
        if constexpr (TC) {
            e = launch_bwd_scan_tc(B, 1, T_total, st);
            if (e != cudaSuccess) return e;
        } else {
            k_bwd_phase_c<Op, C><<<dim3(P.total_segs, P.Hv), NT, SS::bytes, st>>>(B);
        }
        timing_end(st);
    }
    if (P.total_chunks > 0) {
        timing_begin("bwd_local", st);
        if constexpr (TC) {
            e = launch_bwd_local_tc(B, T_total, st);
            if (e != cudaSuccess) return e;
        } else {
            const int64_t items = int64_t(P.total_chunks) * P.Hv;
            const int grid = int(std::min<int64_t>(items, sm_count()));  // one CTA per SM, persistent
            k_bwd_local<Op, C, NT><<<grid, NT, LS::bytes, st>>>(B, items);
        }
        timing_end(st);
    }
    if (B.dqp) {
        const int64_t n = T_total * P.Hqk * (KD / 2);
        const int blocks = int(std::min<int64_t>((n + 255) / 256, 4096));
        if (blocks > 0) {
            timing_begin("bwd_reduce", st);
            k_bwd_reduce<Op><<<blocks, 256, 0, st>>>(B, T_total);
            timing_end(st);
        }
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const BwdProblem& B, int dtype, cudaStream_t st) {
    if (dtype == 0) return launch_bwd_t<__nv_bfloat16, 64>(B, st);
    return launch_bwd_t<float, 32>(B, st);
}

}  // namespace gdn

#ifdef GDN_TRACE
extern "C" int gdn_debug_loc_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, gdn::g_loc_trace, sizeof(gdn::g_loc_trace)));
}
#endif
