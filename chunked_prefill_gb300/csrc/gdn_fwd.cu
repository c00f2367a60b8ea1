// Forward kernels of the chunked gated delta rule.
//
// One CTA scans the chunks of one (sequence, v-head, segment) in order.  Per chunk of C
// tokens (FlashQLA pages, agentlenshq "GDN chunked prefill optimisation": the chunk-local
// W/U preparation, the serial state S and the output O, kept on-chip here instead of
// round-tripping HBM), with gamma the in-chunk cumsum of g and X the state (K x 128):
//
//   A   = diag(beta) (K K^T * exp(gamma_i - gamma_j))   strictly lower
//   T   = (I + A)^-1                                    blocked forward substitution, fp32
//   -W  = -T diag(beta e^gamma) K          U = T diag(beta) V
//   V'  = U - W X                          (corrected values)
//   O   = scale (diag(e^gamma) Q X + (Q K^T * D) V')
//   X  <- e^{gamma_C} X + K^T diag(e^{gamma_C - gamma}) V'
//
// The state X lives in registers as fp32 mma accumulators (warp w owns rows 16w..16w+15);
// a bf16 (or fp32 in the test mode) copy sits in shared memory as the MMA operand.
//
// Context parallelism (FlashQLA pages, "AutoCP" and the warm-up paragraph): the chunk map
// is affine in X, so a segment maps its entering state by X_out = M X_in + S.  Phase A
// computes S (from a zero state, or from h0 for the first segment) and M (from X = I,
// without the U term) per segment; the fix-up composes them serially per (sequence,
// head); phase C reruns every segment from its true entering state and writes O.  The
// opt-in warm-up mode replaces phase A + fix-up by a scan of the warmup chunks before each
// segment from a zero state.
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc05.cuh"

namespace gdn {

enum Kind { K_STATE = 0, K_TRANS = 1, K_OUT = 2, K_HIST = 3 };

constexpr int NTHREADS = 256;

template <typename Op, int C>
struct FwdSmem {
    static constexpr int LDK = KD + OpTraits<Op>::PAD;  // 128-wide operand rows
    static constexpr int LDC = C + OpTraits<Op>::PAD;   // C-wide operand rows
    static constexpr int LDF = C + 1;                   // fp32 C x C scratch
    static constexpr size_t TILE = size_t(C) * LDK * sizeof(Op);
    static constexpr size_t CT = size_t(C) * LDC * sizeof(Op);
    static constexpr size_t FT = size_t(C) * LDF * 4;
    static constexpr size_t oK = 0, oQ = oK + TILE, oV = oQ + TILE, oW = oV + TILE,
                            oVp = oW + TILE, oVh = oVp + TILE, oX = oVh + TILE;
    static constexpr size_t oTW = oX + size_t(KD) * LDK * sizeof(Op);
    static constexpr size_t oTU = oTW + CT, oP = oTU + CT, oA = oP + CT, oT = oA + FT;
    static constexpr size_t oTmp = oT + FT;
    static constexpr size_t oGam = oTmp + 3 * 16 * 17 * 4;
    static constexpr size_t oE = oGam + C * 4, oKd = oE + C * 4, oBeta = oKd + C * 4;
    static constexpr size_t bytes = oBeta + C * 4;
    static_assert(bytes <= 232448, "shared memory budget");
    static_assert(TILE % 16 == 0 && CT % 16 == 0 && FT % 16 == 0, "16-byte alignment");
};

// Copy `valid` rows of 128 elements (row stride `gstride` elements) into shared rows of
// stride `ld`, zero-filling rows valid..C-1.  16-byte vectors.
template <typename Op, int C>
__device__ __forceinline__ void load_tile(Op* dst, int ld, const Op* src, int64_t gstride,
                                          int valid) {
    constexpr int VEC = 16 / sizeof(Op);
    constexpr int VPR = 128 / VEC;
    for (int idx = threadIdx.x; idx < C * VPR; idx += NTHREADS) {
        const int r = idx / VPR, cv = idx % VPR;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < valid) val = *reinterpret_cast<const uint4*>(src + r * gstride + cv * VEC);
        *reinterpret_cast<uint4*>(dst + r * ld + cv * VEC) = val;
    }
}

__device__ __forceinline__ void seq_bounds(const Problem& P, int s, int64_t& t0, int64_t& t1) {
    if (P.cu) {
        t0 = P.cu[s];
        t1 = P.cu[s + 1];
    } else {
        t0 = int64_t(s) * P.T;
        t1 = t0 + P.T;
    }
}

// Scan chunks [cb, ce) of sequence s (tokens [t0, t1)), v-head j, starting from state x0
// (fp32 [128][128] in global memory; null = zero, or the identity for K_TRANS).  Writes
// the final state to x_out if non-null.
template <typename Op, int C, int KIND>
__device__ void scan_chunks(const Problem& P, char* smem, int s, int j, int64_t t0, int64_t t1,
                            int cb, int ce, const float* x0, float* x_out, int64_t hist_base) {
    using S = FwdSmem<Op, C>;
    constexpr int LDK = S::LDK, LDC = S::LDC, LDF = S::LDF;
    Op* sK = reinterpret_cast<Op*>(smem + S::oK);
    Op* sQ = reinterpret_cast<Op*>(smem + S::oQ);
    Op* sV = reinterpret_cast<Op*>(smem + S::oV);
    Op* sW = reinterpret_cast<Op*>(smem + S::oW);
    Op* sVp = reinterpret_cast<Op*>(smem + S::oVp);
    Op* sVh = reinterpret_cast<Op*>(smem + S::oVh);
    Op* sX = reinterpret_cast<Op*>(smem + S::oX);
    Op* sTW = reinterpret_cast<Op*>(smem + S::oTW);
    Op* sTU = reinterpret_cast<Op*>(smem + S::oTU);
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
    constexpr bool kOut = KIND == K_OUT;
    constexpr bool kU = KIND != K_TRANS;

    // ---- entering state into registers (X rows 16w.., all 128 columns) and smem
    float X[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = 16 * w + gq + 8 * h, c = 8 * n + 2 * tq;
            float a = 0.f, b = 0.f;
            if (x0) {
                const float2 v2 = *reinterpret_cast<const float2*>(x0 + r * VD + c);
                a = v2.x;
                b = v2.y;
            } else if (KIND == K_TRANS) {
                a = (r == c) ? 1.f : 0.f;
                b = (r == c + 1) ? 1.f : 0.f;
            }
            X[n][2 * h] = a;
            X[n][2 * h + 1] = b;
        }
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int r = 16 * w + gq, c = 8 * n + 2 * tq;
        st2(sX + r * LDK + c, X[n][0], X[n][1]);
        st2(sX + (r + 8) * LDK + c, X[n][2], X[n][3]);
    }

    // warp tiling of the C x 128 products: RB row blocks, WPR warps per row block
    constexpr int RB = C / 16, WPR = 8 / RB, COLS = 128 / WPR, NTC = COLS / 8;
    const int m0 = 16 * (w % RB), n0 = COLS * (w / RB);
    // warp tiling of [K;Q] K^T
    constexpr int ROWSK = kOut ? 2 * C : C;
    constexpr int RBk = ROWSK / 16, WPRk = 8 / RBk, COLSk = C / WPRk, NTk = COLSk / 8;
    static_assert(8 % RB == 0 && 8 % RBk == 0 && NTk >= 1, "warp tiling");
    const int mk0 = 16 * (w % RBk), nk0 = COLSk * (w / RBk);

    const int64_t qk_stride = int64_t(Hqk) * KD, v_stride = int64_t(Hv) * VD;
    const Op* qbase = reinterpret_cast<const Op*>(P.q) + qh * KD;
    const Op* kbase = reinterpret_cast<const Op*>(P.k) + qh * KD;
    const Op* vbase = reinterpret_cast<const Op*>(P.v) + j * VD;
    Op* obase = reinterpret_cast<Op*>(P.o) + j * VD;

    for (int ch = cb; ch < ce; ++ch) {
        const int64_t tc = t0 + int64_t(ch) * C;
        const int c = int((t1 - tc) < int64_t(C) ? (t1 - tc) : int64_t(C));

        if (KIND == K_HIST || (KIND == K_OUT && P.hist)) {  // entering state, for the backward
            Op* hp = reinterpret_cast<Op*>(P.hist) + (hist_base + ch) * Hv * (KD * VD) +
                     int64_t(j) * (KD * VD);
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int r = 16 * w + gq, cc = 8 * n + 2 * tq;
                st2(hp + r * VD + cc, X[n][0], X[n][1]);
                st2(hp + (r + 8) * VD + cc, X[n][2], X[n][3]);
            }
        }

        // ---- loads
        load_tile<Op, C>(sK, LDK, kbase + tc * qk_stride, qk_stride, c);
        if (kOut) load_tile<Op, C>(sQ, LDK, qbase + tc * qk_stride, qk_stride, c);
        if (kU) load_tile<Op, C>(sV, LDK, vbase + tc * v_stride, v_stride, c);
        for (int i = tid; i < C; i += NTHREADS) {
            const bool ok = i < c;
            sGam[i] = ok ? P.g[(tc + i) * Hv + j] : 0.f;
            sBeta[i] = ok ? P.beta[(tc + i) * Hv + j] : 0.f;
        }
        __syncthreads();

        // ---- gates (warp 0): inclusive cumsum, e^gamma, e^{gamma_C - gamma}
        if (w == 0) {
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

        // ---- K K^T (and Q K^T) into fp32 scratch
        {
            float acc[NTk][4];
            zero_acc(acc);
            const bool qrows = mk0 >= C;
            warp_mma<NTk, false, true>(acc, qrows ? sQ : sK, LDK, sK, LDK, qrows ? mk0 - C : mk0,
                                       nk0, KD);
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

        // ---- A (strictly lower, in place) and P (lower incl. diagonal)
        for (int idx = tid; idx < C * C; idx += NTHREADS) {
            const int i = idx / C, jj = idx % C;
            const float d = expf(sGam[i] - sGam[jj]);
            sA[i * LDF + jj] = (i > jj) ? sBeta[i] * d * sA[i * LDF + jj] : 0.f;
            if (kOut) sP[i * LDC + jj] = from_f<Op>((i >= jj) ? d * sT[i * LDF + jj] : 0.f);
        }
        __syncthreads();

        // ---- T = (I + A)^-1: diagonal 16x16 blocks by substitution (lane = column)
        constexpr int NB = C / 16;
        if (w < NB && lane < 16) {
            const int b0 = 16 * w, col = lane;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(sA[(b0 + r) * LDF + b0 + m], x[m], acc);
                x[r] = (r == col) ? 1.f : -acc;
                if (r < col) x[r] = 0.f;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(b0 + r) * LDF + b0 + col] = x[r];
        }
        __syncthreads();
        // off-diagonal blocks, one block sub-diagonal at a time:
        //   T_IJ = -T_II * sum_{M=J}^{I-1} A_IM T_MJ
#pragma unroll 1
        for (int d = 1; d < NB; ++d) {
            const int nblk = NB - d;
            for (int e = tid; e < nblk * 256; e += NTHREADS) {
                const int J = e >> 8, r = (e >> 4) & 15, cc = e & 15, I = J + d;
                float acc = 0.f;
                for (int M = J; M < I; ++M) {
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        acc = fmaf(sA[(16 * I + r) * LDF + 16 * M + m],
                                   sT[(16 * M + m) * LDF + 16 * J + cc], acc);
                }
                sTmp[(J * 16 + r) * 17 + cc] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 256; e += NTHREADS) {
                const int J = e >> 8, r = (e >> 4) & 15, cc = e & 15, I = J + d;
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    if (m <= r)
                        acc = fmaf(sT[(16 * I + r) * LDF + 16 * I + m], sTmp[(J * 16 + m) * 17 + cc],
                                   acc);
                sT[(16 * I + r) * LDF + 16 * J + cc] = -acc;
            }
            __syncthreads();
        }

        // ---- -T diag(beta e) and T diag(beta) as MMA operands (and gamma, T when asked)
        const bool lowlevel = KIND == K_OUT && (P.a_out || P.gam_out);
        for (int idx = tid; idx < C * C; idx += NTHREADS) {
            const int i = idx / C, jj = idx % C;
            const float t = (jj <= i) ? sT[i * LDF + jj] : 0.f;
            sTW[i * LDC + jj] = from_f<Op>(-t * sBeta[jj] * sE[jj]);
            if (kU) sTU[i * LDC + jj] = from_f<Op>(t * sBeta[jj]);
            if (lowlevel && i < c) {
                if (P.a_out) reinterpret_cast<Op*>(P.a_out)[((tc + i) * Hv + j) * C + jj] = from_f<Op>(t);
                if (P.gam_out && jj == 0) P.gam_out[(tc + i) * Hv + j] = sGam[i];
            }
        }
        __syncthreads();

        // ---- -W = (-T diag(beta e)) K  -> smem;  U = (T diag(beta)) V -> registers
        float vacc[NTC][4];
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
        zero_acc(vacc);
        if (kU) warp_mma<NTC, false, false>(vacc, sTU, LDC, sV, LDK, m0, n0, C);
        __syncthreads();

        // ---- V' = U - W X
        warp_mma<NTC, false, false>(vacc, sW, LDK, sX, LDK, m0, n0, KD);
#pragma unroll
        for (int n = 0; n < NTC; ++n) {
            const int cc = n0 + 8 * n + 2 * tq;
            const int r0 = m0 + gq, r1 = m0 + gq + 8;
            st2(sVp + r0 * LDK + cc, vacc[n][0], vacc[n][1]);
            st2(sVp + r1 * LDK + cc, vacc[n][2], vacc[n][3]);
            st2(sVh + r0 * LDK + cc, vacc[n][0] * sKd[r0], vacc[n][1] * sKd[r0]);
            st2(sVh + r1 * LDK + cc, vacc[n][2] * sKd[r1], vacc[n][3] * sKd[r1]);
        }

        // ---- O = scale (diag(e) Q X + P V')
        float oacc[NTC][4];
        if (kOut) {
            zero_acc(oacc);
            warp_mma<NTC, false, false>(oacc, sQ, LDK, sX, LDK, m0, n0, KD);
            const float e0 = sE[m0 + gq], e1 = sE[m0 + gq + 8];
#pragma unroll
            for (int n = 0; n < NTC; ++n) {
                oacc[n][0] *= e0;
                oacc[n][1] *= e0;
                oacc[n][2] *= e1;
                oacc[n][3] *= e1;
            }
        }
        __syncthreads();
        if (kOut) {
            warp_mma<NTC, false, false>(oacc, sP, LDC, sVp, LDK, m0, n0, C);
            const float sc = P.scale;
#pragma unroll
            for (int n = 0; n < NTC; ++n) {
                const int cc = n0 + 8 * n + 2 * tq;
                const int r0 = m0 + gq, r1 = m0 + gq + 8;
                if (r0 < c) st2(obase + (tc + r0) * v_stride + cc, sc * oacc[n][0], sc * oacc[n][1]);
                if (r1 < c) st2(obase + (tc + r1) * v_stride + cc, sc * oacc[n][2], sc * oacc[n][3]);
            }
        }

        // ---- X <- e^{gamma_C} X + K^T diag(e^{gamma_C - gamma}) V'
        {
            const float eC = sE[C - 1];
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                X[n][0] *= eC;
                X[n][1] *= eC;
                X[n][2] *= eC;
                X[n][3] *= eC;
            }
            warp_mma<16, true, false>(X, sK, LDK, sVh, LDK, 16 * w, 0, C);
        }
        __syncthreads();
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const int r = 16 * w + gq, cc = 8 * n + 2 * tq;
            st2(sX + r * LDK + cc, X[n][0], X[n][1]);
            st2(sX + (r + 8) * LDK + cc, X[n][2], X[n][3]);
        }
        // the next chunk's loads are followed by a barrier before sX is read
    }

    if (x_out) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const int r = 16 * w + gq, cc = 8 * n + 2 * tq;
            if (KIND == K_TRANS) {  // segment transitions are stored transposed (M^T)
                x_out[cc * VD + r] = X[n][0];
                x_out[(cc + 1) * VD + r] = X[n][1];
                x_out[cc * VD + r + 8] = X[n][2];
                x_out[(cc + 1) * VD + r + 8] = X[n][3];
            } else {
                *reinterpret_cast<float2*>(x_out + r * VD + cc) = make_float2(X[n][0], X[n][1]);
                *reinterpret_cast<float2*>(x_out + (r + 8) * VD + cc) = make_float2(X[n][2], X[n][3]);
            }
        }
    }
}

constexpr int64_t KV = int64_t(KD) * VD;

// Phase A.  Exact mode: blockIdx.z = 0 computes S_j (the state after segment j from a zero
// state; from h0 for j = 0) into hin[g+1]; blockIdx.z = 1 computes M_j (j >= 1) into
// mbuf[g].  Warm-up mode: the state entering segment j >= 1, scanned from a zero state over
// the `warmup` chunks before it (exactly, from h0, when the window reaches chunk 0).
template <typename Op, int C>
__global__ void __launch_bounds__(NTHREADS, 1) k_phase_a(Problem P) {
    extern __shared__ __align__(128) char smem[];
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) return;
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_bounds(P, s, t0, t1);
    const int nt = int((t1 - t0 + C - 1) / C);
    const float* h0 = P.h0 ? P.h0 + (int64_t(s) * P.Hv + j) * KV : nullptr;
    if (P.cp == CP_EXACT) {
        if (lj >= nseg - 1) return;
        const int cb = lj * P.L, ce = min(cb + P.L, nt);
        if (blockIdx.z == 0) {
            scan_chunks<Op, C, K_STATE>(P, smem, s, j, t0, t1, cb, ce, lj == 0 ? h0 : nullptr,
                                        P.hin + (int64_t(gseg + 1) * P.Hv + j) * KV, 0);
        } else {
            if (lj == 0) return;
            scan_chunks<Op, C, K_TRANS>(P, smem, s, j, t0, t1, cb, ce, nullptr,
                                        P.mbuf + (int64_t(gseg) * P.Hv + j) * KV, 0);
        }
    } else {
        if (lj == 0 || blockIdx.z != 0) return;
        const int cb = lj * P.L, w0 = cb - P.warmup;
        scan_chunks<Op, C, K_STATE>(P, smem, s, j, t0, t1, max(w0, 0), cb, w0 <= 0 ? h0 : nullptr,
                                    P.hin + (int64_t(gseg) * P.Hv + j) * KV, 0);
    }
}

// Phase C: every segment from its entering state; writes O (K_OUT) or the entering state
// of every chunk (K_HIST, the backward's recompute), and the final state.
template <typename Op, int C, int KIND>
__global__ void __launch_bounds__(NTHREADS, 1) k_phase_c(Problem P) {
    extern __shared__ __align__(128) char smem[];
    const int gseg = blockIdx.x, j = blockIdx.y;
    const int2 sj = plan_seg(P.plan, gseg);
    const int s = sj.x, lj = sj.y;
    if (s < 0 || s >= P.N) return;
    const int nseg = plan_seg_off(P.plan, s + 1) - plan_seg_off(P.plan, s);
    int64_t t0, t1;
    seq_bounds(P, s, t0, t1);
    const int nt = int((t1 - t0 + C - 1) / C);
    const int cb = lj * P.L, ce = min(cb + P.L, nt);
    const float* x0 = (lj == 0) ? (P.h0 ? P.h0 + (int64_t(s) * P.Hv + j) * KV : nullptr)
                                : P.hin + (int64_t(gseg) * P.Hv + j) * KV;
    float* x_out = (lj == nseg - 1 && P.ht) ? P.ht + (int64_t(s) * P.Hv + j) * KV : nullptr;
    const int64_t hb = plan_chunk_off(P.plan, s);
    scan_chunks<Op, C, KIND>(P, smem, s, j, t0, t1, cb, ce, x0, x_out, hb);
}

// Fix-up: hin[g0+j+1] = M_j hin[g0+j] + S_j for j = 1..nseg-2, serially.  The transitions
// are stored transposed (M^T); each arrives in shared memory by a bulk copy issued one step
// ahead (two buffers).  Thread t accumulates a 4-row x 8-column block over a slice of the
// inner index: one 16-byte load of M^T and two broadcast loads of the state per 16 packed
// (two-lane) FMAs; the slices' partial blocks meet in shared memory.  S_j of the next step is
// read into registers one step early.  fp32.  Measured on GB300 at 8 columns per CTA a step
// takes ~2.8k cycles, most of it shared-memory traffic: the 64 KB transition tile, the
// broadcast state loads and the 32 KB of partial blocks written and read back.
#ifdef GDN_TRACE
__device__ unsigned long long g_fix_trace[64][4];  // debug builds: SM clock per fix-up step
#define FTRACE(k, e)                                                                            \
    do {                                                                                        \
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0 && (k) < 64) \
            g_fix_trace[k][e] = clock64();                                                      \
    } while (0)
#else
#define FTRACE(k, e) \
    do {             \
    } while (0)
#endif
constexpr int FIX_NB = 2, FIX_T = 256;
// Shared memory of a fix-up CTA with CG groups of 8 state columns: FIX_NB transition tiles, the
// k-slice partial blocks (8 warps x 32 lanes x 32 floats whatever CG is) and the CTA's
// columns of x.
constexpr int fix_smem(int CG) { return FIX_NB * KD * KD * 4 + 8 * 32 * 32 * 4 + KD * 8 * CG * 4 + 64; }
// REV = false: the forward, hin[g0+lj+1] = M_lj hin[g0+lj] + S_lj for lj = 1..nseg-2, reading
// M^T (the transposed store).  REV = true: the backward, dhb[g0+lj] = M_lj^T dhb[g0+lj+1] +
// dhb[g0+lj] for lj = nseg-2..1, reading M (the untransposed store).  In both the shared
// tile holds A^T for the step's matrix A, and xbuf[g] is read as S and overwritten in place.
// A CTA owns W = 8 CG columns of one (sequence, v-head) chain.  Its 8 warps split the
// contraction into KS = 8 / CG slices; a thread accumulates a 4-row x 8-column block of one
// column group over its slice, and the slices are summed through shared memory.  Few chains
// take CG = 1 (short steps, many CTAs per chain); many chains take a wider CG so that all
// chains run in one wave and each transition tile is read by fewer CTAs.
// dec (null = every step composes): the decay-bounded exact mode's per-(segment, v-head)
// flag; a step whose segment has dec >= 0 has a negligible transition, so its result is S
// itself (already in xbuf) and the step neither loads its transition nor computes.
template <bool REV, int CG>
__global__ void __launch_bounds__(FIX_T) k_fixup(const PlanDev plan, const float* mats, float* xbuf,
                                                 int Hv, int* err, const int* dec) {
    constexpr int W = 8 * CG, KS = 8 / CG, MS = KD / KS;
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    extern __shared__ __align__(128) unsigned char fsm[];
    float* Ms = reinterpret_cast<float*>(fsm);                                // FIX_NB x 128 x 128
    float* red = reinterpret_cast<float*>(fsm + FIX_NB * KD * KD * 4);        // 8 x 32 x 32
    float* xs = reinterpret_cast<float*>(fsm + FIX_NB * KD * KD * 4 + 8 * 32 * 32 * 4);  // 128 x W
    uint64_t* bar = reinterpret_cast<uint64_t*>(fsm + FIX_NB * KD * KD * 4 + 8 * 32 * 32 * 4 + KD * W * 4);
    const int s = blockIdx.x, j = blockIdx.y, cb = blockIdx.z * W;
    const int g0 = plan_seg_off(plan, s), nseg = plan_seg_off(plan, s + 1) - g0;
    if (nseg <= 2) return;
    const int last = nseg - 2;  // steps 1..last
    const int t = threadIdx.x, rg = t & 31, ks = (t >> 5) / CG, cg = (t >> 5) % CG;
    const int orow = t >> 1, oc = (t & 1) * 4;  // each thread finishes 4 columns of orow per group
    auto seg_of = [&](int q) { return REV ? nseg - 2 - q : 1 + q; };  // step q -> segment lj
    auto mt = [&](int q) { return mats + (int64_t(g0 + seg_of(q)) * Hv + j) * KV; };
    // x entering step q, and the S / result slot of step q
    auto xin = [&](int q) { return REV ? g0 + seg_of(q) + 1 : g0 + seg_of(q); };
    auto xout = [&](int q) { return REV ? g0 + seg_of(q) : g0 + seg_of(q) + 1; };
    auto hp = [&](int g, int c) {
        return reinterpret_cast<float4*>(xbuf + (int64_t(g) * Hv + j) * KV + orow * VD + cb + 8 * c + oc);
    };
    // the first step at or after q whose transition is not negligible (last: none)
    auto next_active = [&](int q) {
        if (!dec) return q;
        while (q < last && dec[int64_t(g0 + seg_of(q)) * Hv + j] >= 0) ++q;
        return q;
    };
    // the first composing step, found by all threads at once (one flag load each)
    __shared__ int s_first;
    if (t == 0) s_first = dec ? last : 0;
    __syncthreads();
    if (dec)
        for (int q = t; q < last; q += FIX_T)
            if (dec[int64_t(g0 + seg_of(q)) * Hv + j] < 0) atomicMin(&s_first, q);
    __syncthreads();
    const int q0 = s_first;
    if (q0 >= last) return;  // every result is its S, already in place
    if (t == 0) {
        for (int b = 0; b < FIX_NB; ++b) tc::mbar_init(&bar[b], 1);
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (t == 0) {
        tc::mbar_expect_tx(&bar[0], KD * KD * 4);
        tc::bulk_load(Ms, mt(q0), KD * KD * 4, &bar[0]);
    }
    float4 snext[CG];
#pragma unroll
    for (int c = 0; c < CG; ++c) {
        *reinterpret_cast<float4*>(&xs[orow * W + 8 * c + oc]) = *hp(xin(q0), c);
        snext[c] = *hp(xout(q0), c);
    }
    bool ok = true;
    int uses[FIX_NB] = {0, 0};  // completed loads per buffer (mbarrier phase parity)
    int b = 0;
    for (int q = q0; q < last;) {
        const int qn = next_active(q + 1);
        if (t == 0 && qn < last) {  // into the other buffer (its last step is done with it)
            tc::mbar_expect_tx(&bar[b ^ 1], KD * KD * 4);
            tc::bulk_load(Ms + (b ^ 1) * KD * KD, mt(qn), KD * KD * 4, &bar[b ^ 1]);
        }
        FTRACE(q + 1, 0);
        ok = ok && tc::mbar_wait(&bar[b], uses[b] & 1);
        ++uses[b];
        FTRACE(q + 1, 1);
        __syncthreads();  // also orders the previous step's xs update
        FTRACE(q + 1, 2);
        float4 sj[CG];
#pragma unroll
        for (int c = 0; c < CG; ++c) {
            sj[c] = snext[c];
            if (qn < last) snext[c] = *hp(xout(qn), c);
        }
        const float* M = Ms + b * KD * KD;
        // acc[r][p]: row r, columns (2p, 2p + 1) as a packed pair (one packed FMA per pair)
        uint64_t acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int p2 = 0; p2 < 4; ++p2) acc[r][p2] = 0ull;
#pragma unroll 8
        for (int m = MS * ks; m < MS * ks + MS; ++m) {
            const float4 a = *reinterpret_cast<const float4*>(M + m * KD + 4 * rg);
            const ulonglong2 x0 = *reinterpret_cast<const ulonglong2*>(&xs[m * W + 8 * cg]);
            const ulonglong2 x1 = *reinterpret_cast<const ulonglong2*>(&xs[m * W + 8 * cg + 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint64_t ar = tc::dup2(av[r]);
                acc[r][0] = tc::ffma2(ar, x0.x, acc[r][0]);
                acc[r][1] = tc::ffma2(ar, x0.y, acc[r][1]);
                acc[r][2] = tc::ffma2(ar, x1.x, acc[r][2]);
                acc[r][3] = tc::ffma2(ar, x1.y, acc[r][3]);
            }
        }
        // partial block -> red[ks][rg][cg][32], 16-byte pieces rotated by rg against bank
        // conflicts
        float* rp = red + ((ks * 32 + rg) * CG + cg) * 32;
#pragma unroll
        for (int pq = 0; pq < 8; ++pq) {
            const int r = pq >> 1, c2 = (pq & 1) * 2;
            *reinterpret_cast<ulonglong2*>(rp + ((pq ^ (rg & 7)) << 2)) =
                make_ulonglong2(acc[r][c2], acc[r][c2 + 1]);
        }
        FTRACE(q + 1, 3);
        __syncthreads();  // partial blocks visible; everyone is done with xs and buffer b
        {
            const int org = orow >> 2, pq = ((orow & 3) << 1) | (oc >> 2);
#pragma unroll
            for (int c = 0; c < CG; ++c) {
                float4 o = sj[c];
#pragma unroll
                for (int k2 = 0; k2 < KS; ++k2) {
                    const float4 p = *reinterpret_cast<const float4*>(
                        red + ((k2 * 32 + org) * CG + c) * 32 + ((pq ^ (org & 7)) << 2));
                    o.x += p.x;
                    o.y += p.y;
                    o.z += p.z;
                    o.w += p.w;
                }
                *hp(xout(q), c) = o;
                // x entering the next composing step: this result when it follows at once,
                // else the S that the negligible steps in between left in place (the last
                // of them is the entering slot of step qn)
                *reinterpret_cast<float4*>(&xs[orow * W + 8 * c + oc]) =
                    (qn == q + 1 || qn >= last) ? o : *hp(xin(qn), c);
            }
        }
        q = qn;
        b ^= 1;
    }
    if (!ok && t == 0 && err) atomicOr(err, 1 << 30);
}

// Column groups per fix-up CTA: the narrowest that puts every chain of the launch in one wave
// at one CTA per SM (the shared memory allows no more).
int fixup_groups(int chains) {
    const int sms = sm_count();
    for (int cg = 1; cg < 8; cg *= 2)
        if (int64_t(chains) * (VD / (8 * cg)) <= sms) return cg;
    return 8;
}

template <bool REV>
static void launch_fixup_cg(int N, int Hv, const PlanDev& plan, const float* mats, float* xbuf,
                            int* err, bool pdl, cudaStream_t st, const int* dec) {
    auto run = [&](auto kern, int cg) {
        const int smem = fix_smem(cg);
        smem_attr(kern, smem);
        const dim3 grid(N, Hv, VD / (8 * cg));
        if (pdl) launch_pdl(kern, grid, dim3(FIX_T), smem, st, plan, mats, xbuf, Hv, err, dec);
        else kern<<<grid, FIX_T, smem, st>>>(plan, mats, xbuf, Hv, err, dec);
    };
    switch (fixup_groups(N * Hv)) {
        case 1: run(k_fixup<REV, 1>, 1); break;
        case 2: run(k_fixup<REV, 2>, 2); break;
        case 4: run(k_fixup<REV, 4>, 4); break;
        default: run(k_fixup<REV, 8>, 8); break;
    }
}

// Work decomposition on the device from the device cu_seqlens (same rule as the host).
__global__ void k_plan(const int* cu, int N, int T, int C, int L, int total_segs, int2* seg,
                       int* seg_off, int* chunk_off, int* err) {
    tc::pdl_launch_dependents();
    if (err && threadIdx.x == 0) *err = 0;  // the call's error word starts clear
    for (int i = threadIdx.x; i < total_segs; i += blockDim.x) seg[i] = make_int2(-1, -1);
    __syncthreads();
    if (threadIdx.x != 0) return;
    int acc_s = 0, acc_c = 0;
    for (int s = 0; s < N; ++s) {
        const int len = cu ? cu[s + 1] - cu[s] : T;
        const int nt = (max(len, 0) + C - 1) / C;
        const int ns = max(1, (nt + L - 1) / L);
        seg_off[s] = acc_s;
        chunk_off[s] = acc_c;
        for (int q = 0; q < ns; ++q)
            if (acc_s + q < total_segs) seg[acc_s + q] = make_int2(s, q);
        acc_s += ns;
        acc_c += nt;
    }
    seg_off[N] = min(acc_s, total_segs);
    chunk_off[N] = acc_c;
}

// One thread waits (bounded) on an mbarrier that nothing completes; on giving up it sets its
// bit in the error word.  No other memory is touched.
__global__ void k_debug_wait(int* err, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_fence_init();
        if (!tc::mbar_wait(&bar, 0, limit_ns)) atomicOr(err, 1 << 25);
    }
}

cudaError_t launch_debug_wait(int* err, int limit_us, cudaStream_t st) {
    k_debug_wait<<<1, 32, 0, st>>>(err, 1000ull * unsigned(limit_us));
    return cudaGetLastError();
}

void launch_plan(const Problem& P, int C, cudaStream_t st) {
    timing_begin("fwd_plan", st);
    k_plan<<<1, 256, 0, st>>>(P.cu, P.N, P.T, C, P.L, P.total_segs, P.plan.seg, P.plan.seg_off,
                              P.plan.chunk_off, P.err);
    timing_end(st);
}

void launch_fixup(const Problem& P, cudaStream_t st) {
    timing_begin("fwd_fixup", st);
    launch_fixup_cg<false>(P.N, P.Hv, P.plan, P.mbuf, P.hin, P.err, true, st, P.dec);
    timing_end(st);
}

void launch_bwd_fixup_tc(const BwdProblem& B, cudaStream_t st) {
    const Problem& P = B.f;
    launch_fixup_cg<true>(P.N, P.Hv, P.plan, P.mbuf_t, B.dhb, P.err, true, st, P.dec);
}

template <typename Op, int C>
static cudaError_t launch_fwd_t(const Problem& P, bool hist, cudaStream_t st) {
    using S = FwdSmem<Op, C>;
    const int smem = int(S::bytes);
    cudaError_t e;
    e = cudaFuncSetAttribute(k_phase_a<Op, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_phase_c<Op, C, K_OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_phase_c<Op, C, K_HIST>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;

    launch_plan(P, C, st);
    if (P.cp != CP_NONE) {
        dim3 ga(P.total_segs, P.Hv, P.cp == CP_EXACT ? 2 : 1);
        timing_begin("fwd_phase_a", st);
        k_phase_a<Op, C><<<ga, NTHREADS, smem, st>>>(P);
        timing_end(st);
        if (P.cp == CP_EXACT) launch_fixup(P, st);
    }
    dim3 gc(P.total_segs, P.Hv);
    timing_begin(hist ? "fwd_recompute_states" : "fwd_phase_c", st);
    if (hist)
        k_phase_c<Op, C, K_HIST><<<gc, NTHREADS, smem, st>>>(P);
    else
        k_phase_c<Op, C, K_OUT><<<gc, NTHREADS, smem, st>>>(P);
    timing_end(st);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const Problem& P, int dtype, bool hist, cudaStream_t st) {
    // bf16 problems run on the tensor-core kernels (launch_fwd_tc); this path is the fp32
    // test mode
    if (dtype != 1) return cudaErrorInvalidValue;
    return launch_fwd_t<float, 32>(P, hist, st);
}

int fwd_chunk_size(int dtype) { return dtype == 0 ? 64 : 32; }

}  // namespace gdn

#ifdef GDN_TRACE
extern "C" int gdn_debug_fix_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, gdn::g_fix_trace, sizeof(gdn::g_fix_trace)));
}
#endif
