// Chunk-local preparation, fully parallel over (chunk, v-head), for the tensor-core scan.
//
// Per chunk of 64 tokens (FlashQLA pages, agentlenshq "GDN chunked prefill optimisation":
// the chunk-local W/U preparation): gamma = in-chunk cumsum of g, then
//     [KK; QK] = [K; Q] K^T                        (tcgen05, fp32 accumulation in TMEM)
//     A  = diag(beta) (KK * Dm),  P = QK * D         (D_ij = exp(gamma_i - gamma_j), i >= j)
//     T  = (I + A)^-1                                (fp32: substitution + TF32 block products)
//     TU = T diag(beta),  W' = -T diag(beta e) K     (W' = -W of the pages' WY form; tcgen05)
// K and Q arrive by TMA; W' and TU leave by bulk copies from shared-memory tiles already in
// the 128-byte-swizzled layout the scan's tensor-core operands use, P and T (for the backward)
// by 16-byte stores of the same image from registers.  (P staged for a bulk copy instead cost
// the inverse a wait for the copy's reads; TU written by 16-byte stores instead made the
// preparation slower.)  Rows past the end of a sequence hold whatever tokens follow (finite); beta = g = 0 there makes T's rows and the
// columns of TU and W' for them exactly zero, and P's rows for them are written as zeros (the
// backward's dO^T P must not see them).
#include <cuda.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc05.cuh"

namespace gdn {
namespace {

using namespace tc;

#ifdef GDN_TRACE
__device__ unsigned long long g_prep_trace[8 * 9];  // debug builds: SM clock at phase ends
#ifndef GDN_PTRACE_X
#define GDN_PTRACE_X 0
#endif
// per v-head slot (the CTA-level events go to slot 8)
#define PTRACE_H(h, e)                                                                          \
    do {                                                                                        \
        if (blockIdx.x == GDN_PTRACE_X && blockIdx.y == 0 && threadIdx.x == 0 && (h) < 9)       \
            g_prep_trace[(h) * 8 + (e)] = clock64();                                            \
    } while (0)
#define PTRACE(e) PTRACE_H(hh, e)
#else
#define PTRACE_H(h, e) \
    do {               \
    } while (0)
#define PTRACE(e) \
    do {          \
    } while (0)
#endif

// 8 warps: warp w reads TMEM lanes [32 (w % 4), +32); the row-per-thread phases (A and P,
// W' staging) split a row's 64 columns between warps w and w + 4, the item loops (gates in,
// TU / TW staging) spread over all 256 threads, and the inverse runs on warps 0-3.  At 64
// registers per thread four CTAs (32 warps) fit an SM, as four CTAs of 4 warps did: each CTA's
// row phases take half the time.
constexpr int PT = 256;  // threads
constexpr int TU4 = 64 * 8 / PT;  // (row, 8-column chunk) items per thread of the TU / TW staging
constexpr int CH = 64;

// The 64 x 64 lower-triangular A and T are kept as their ten nonzero 16 x 16 blocks (row
// stride BLD), block (I, M), I >= M, at index I (I + 1) / 2 + M.
constexpr int BLD = 20, BLKF = 16 * BLD;  // floats per block row / per block
__device__ __forceinline__ int tri(int I, int M) { return I * (I + 1) / 2 + M; }

// One CTA per (chunk, q/k head, slice of at most GMAX v-heads of its group): K and Q are
// loaded and [K;Q] K^T formed once, then each v-head's gating, inverse and W' follow in turn.
// Shared memory (from a 1024-aligned base), small enough for four CTAs per SM.  Once
// [K;Q] K^T is in TMEM the two Q halves of the operand tile hold A's blocks (six, then four),
// and after the inverse the TU staging tile and the TW operand tile; the whole [K;Q] tile
// finally stages W'.
struct PrepSmem {
    static constexpr uint32_t oKQ = 0;                    // 2 x 16 KB: rows 0-63 K, 64-127 Q
    static constexpr uint32_t oQ0 = 8192, oQ1 = 24576;    // the Q halves
    static constexpr uint32_t oT = 32768;                 // T: 10 blocks (12.5 KB)
    static constexpr uint32_t oTmp = oT + 10 * BLKF * 4;  // 4 x 16 x 20 fp32
    static constexpr uint32_t oGam = oTmp + 4 * 16 * 20 * 4;
    static constexpr uint32_t oE = oGam + CH * 4, oEi = oE + CH * 4, oBeta = oEi + CH * 4,
                              oBe = oBeta + CH * 4, oFlag = oBe + CH * 4, oBar = oFlag + 16,
                              oSlot = oBar + 3 * 8;
    static constexpr int GMAX = 8;                        // v-heads per CTA (q/k group slice)
    static constexpr uint32_t oGin = oSlot + 16;          // g, beta of those heads: [GMAX][2][64]
    static constexpr uint32_t bytes = oGin + GMAX * 2 * CH * 4 + 1024;  // + alignment slack
    static_assert(6 * BLKF * 4 <= 8192 && 4 * BLKF * 4 <= 8192, "A blocks fit the Q halves");
};

__global__ void __launch_bounds__(PT, 4) k_prep(Problem P, const __grid_constant__ TcMaps maps) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using S = PrepSmem;
    float* sT = reinterpret_cast<float*>(smem + S::oT);
    auto ablk = [&](int b) {
        return reinterpret_cast<float*>(smem + (b < 6 ? S::oQ0 + b * BLKF * 4 : S::oQ1 + (b - 6) * BLKF * 4));
    };
    auto tblk = [&](int b) { return sT + b * BLKF; };
    float* sTmp = reinterpret_cast<float*>(smem + S::oTmp);
    float* sGam = reinterpret_cast<float*>(smem + S::oGam);
    float* sE = reinterpret_cast<float*>(smem + S::oE);
    float* sEi = reinterpret_cast<float*>(smem + S::oEi);
    float* sBeta = reinterpret_cast<float*>(smem + S::oBeta);
    float* sNbe = reinterpret_cast<float*>(smem + S::oBe);  // -beta e
    int* sFlag = reinterpret_cast<int*>(smem + S::oFlag);
    float* sPart = reinterpret_cast<float*>(smem + S::oFlag + 8);  // two partial sums
    float* sGin = reinterpret_cast<float*>(smem + S::oGin);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);  // load, [K;Q]K^T, W'
    uint32_t* slot = reinterpret_cast<uint32_t*>(smem + S::oSlot);

    pdl_launch_dependents();
    pdl_wait();
#ifndef GDN_CHECK
    // no planner kernel ran before this one (equal-length batch): the call's error word starts
    // clear here (a kernel of this call reports into it only after a bounded wait of seconds)
    if (P.plan.uni_ns > 0 && P.err && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *P.err = 0;
#endif
    const int gch = blockIdx.x;
    if (gch >= plan_chunk_off(P.plan, P.N)) return;
    const int G = P.Hv / P.Hqk;
    const int hpc = P.prep_heads;                         // v-heads per CTA (<= GMAX)
    const int nsl = (G + hpc - 1) / hpc;                  // slices of a q/k group
    const int qh = blockIdx.y / nsl, j0 = qh * G + (blockIdx.y % nsl) * hpc;
    const int nh = min(hpc, qh * G + G - j0);             // v-heads of this CTA
    int lo = 0, hi = P.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (plan_chunk_off(P.plan, mid) <= gch) lo = mid;
        else hi = mid - 1;
    }
    const int s = lo;
    const int ch = gch - plan_chunk_off(P.plan, s);
    int64_t t0, t1;
    if (P.cu) {
        t0 = P.cu[s];
        t1 = P.cu[s + 1];
    } else {
        t0 = int64_t(s) * P.T;
        t1 = t0 + P.T;
    }
    const int64_t tc = t0 + int64_t(ch) * CH;
    if (tc >= t1) return;
    const int c = int((t1 - tc) < int64_t(CH) ? (t1 - tc) : int64_t(CH));
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const uint32_t kq = smem_addr(smem + S::oKQ);
    int* err = P.err;
    const int64_t T_all = P.cu ? int64_t(P.T) : int64_t(P.N) * P.T;  // tokens (store extents)
    const bool store_t = P.prep_stride >= PREP_BWD_BYTES;  // T in the record (backward)
    const bool want_t = store_t || P.a_out != nullptr;

    if (tid == 0) {
        for (int b = 0; b < 3; ++b) mbar_init(&bars[b], 1);
        mbar_fence_init();
    }
    if (w == 0) tmem_alloc(slot, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *slot;
    PTRACE_H(8, 0);
    if (tid == 0) {
        mbar_expect_tx(&bars[0], 32768);
        tma_load_3d(smem + S::oKQ, &maps.k, &bars[0], 0, qh, int(tc));
        tma_load_3d(smem + S::oKQ + 16384, &maps.k, &bars[0], 64, qh, int(tc));
        tma_load_3d(smem + S::oKQ + 8192, &maps.q, &bars[0], 0, qh, int(tc));
        tma_load_3d(smem + S::oKQ + 16384 + 8192, &maps.q, &bars[0], 64, qh, int(tc));
    }
    // g and beta of every v-head of this CTA (rows past the sequence end 0)
    for (int idx = tid; idx < nh * CH; idx += PT) {
        const int hh = idx / CH, r = idx % CH;
        const bool ok = r < c;
        sGin[(hh * 2) * CH + r] = ok ? P.g[(tc + r) * P.Hv + j0 + hh] : 0.f;
        sGin[(hh * 2 + 1) * CH + r] = ok ? P.beta[(tc + r) * P.Hv + j0 + hh] : 0.f;
    }
    if (tid == 0) {
        // [KK; QK] = [K; Q] K^T into TMEM columns [0, 64), shared by the v-heads
        bool ok = mbar_wait(&bars[0], 0);
        if (ok) {
            constexpr uint32_t ID1 = make_idesc(128, 64, 0, 0);
            const uint64_t d = make_desc(kq, 0, 1024);
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const uint32_t off = (st >> 2) * 16384 + (st & 3) * 32;
                mma_bf16(tm, d + (off >> 4), d + (off >> 4), ID1, st > 0);
            }
        } else if (err) {
            atomicOr(err, 1 << 29);
        }
        commit(&bars[1]);
    }
    __syncthreads();  // g, beta staged
    {
        const bool ok = warp_uniform_wait(&bars[1], 0);
        if (!ok && lane == 0 && err) atomicOr(err, 1 << 28);
    }
    fence_after_sync();

    float kn = 0.f;  // threads of warps 0-1: |k_i|^2 of their row of KK^T (from the first head)
#pragma unroll 1
    for (int hh = 0; hh < nh; ++hh) {
        const int j = j0 + hh;
        PTRACE(0);
        unsigned char* rec = static_cast<unsigned char*>(P.prep) + (int64_t(gch) * P.Hv + j) * P.prep_stride;
        if (w == 0) {  // in-chunk gates of this v-head
            const float gv[2] = {sGin[(hh * 2) * CH + 2 * lane], sGin[(hh * 2) * CH + 2 * lane + 1]};
            const float bv[2] = {sGin[(hh * 2 + 1) * CH + 2 * lane], sGin[(hh * 2 + 1) * CH + 2 * lane + 1]};
            const float run0 = gv[0], run1 = gv[0] + gv[1];
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
                sGam[r] = gm[u];
                sE[r] = e;
                sEi[r] = expf(-gm[u]);
                sBeta[r] = bv[u];
                sNbe[r] = -(bv[u] * e);
                if (P.gam_out && r < c && in_range((tc + r) * P.Hv + j, T_all * P.Hv, err))
                    P.gam_out[(tc + r) * P.Hv + j] = gm[u];
            }
            if (lane == 0) *sFlag = (last < -80.f || !(last == last)) ? 1 : 0;
        }
        // the previous head's W' stores have read their staging tiles (waited for here, after
        // this head's gates, rather than at the end of that head: the A/P phase reuses them)
        if (tid == 0 && hh > 0) bulk_wait_read0();
        __syncthreads();  // gates visible; the previous head's staging has been read
        PTRACE(1);

        // A (rows of KK) and P (rows of QK): thread = one row of the stacked product, warp w
        // its half w / 4 of the 64 columns
        {
            const bool pw = *sFlag != 0;
            const int wq = w & 3;
            const bool qrows = wq >= 2;
            const int i = 32 * (wq & 1) + lane;
            const float gi = sGam[i], ei = sE[i], bi = sBeta[i];
            unsigned char* pt = rec + PREP_P;  // P's record image (bf16, swizzled rows)
#pragma unroll 1
            for (int q16 = 0; q16 < 2; ++q16) {  // 16 columns at a time (register budget)
                const int c0 = 32 * (w >> 2) + 16 * q16;
                float raw[16];
                tmem_ld16(tm + (uint32_t(32 * wq) << 16) + c0, raw);
                tmem_ld_wait();
                if (!qrows && hh == 0 && (c0 >> 4) == (i >> 4)) {  // the diagonal: |k_i|^2, once
#pragma unroll
                    for (int u = 0; u < 16; ++u) kn = (u == (i & 15)) ? raw[u] : kn;
                }
                // with rc the row's factor (beta_i e_i for A, e_i for P), element j is
                // rc e^{-gamma_j} raw_j: two packed products per pair of columns; at extreme
                // decay (pw) e^{gamma_i - gamma_j} is formed directly instead
                const uint64_t rc2 = dup2(qrows ? ei : bi * ei);
                if (!qrows) {
                    const int I = i >> 4, r = i & 15, M = c0 >> 4;
                    if (M <= I) {  // blocks above the diagonal are not stored
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const int jb = c0 + 4 * j4;
                            float x[4];
                            if (pw) {
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    x[u] = bi * expf(gi - sGam[jb + u]) * raw[4 * j4 + u];
                            } else {
                                const ulonglong2 ev = *reinterpret_cast<const ulonglong2*>(sEi + jb);
                                unpk2(fmul2(fmul2(rc2, ev.x), pk2(raw[4 * j4], raw[4 * j4 + 1])), x[0], x[1]);
                                unpk2(fmul2(fmul2(rc2, ev.y), pk2(raw[4 * j4 + 2], raw[4 * j4 + 3])), x[2], x[3]);
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) x[u] = jb + u < i ? x[u] : 0.f;
                            *reinterpret_cast<float4*>(ablk(tri(I, M)) + r * BLD + (jb & 15)) =
                                make_float4(x[0], x[1], x[2], x[3]);
                        }
                    }
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 2; ++c4) {
                        const int c8 = (c0 >> 3) + c4;
                        float x[8];
                        if (pw) {
#pragma unroll
                            for (int u = 0; u < 8; ++u) x[u] = expf(gi - sGam[8 * c8 + u]) * raw[8 * c4 + u];
                        } else {
                            const ulonglong2 e0 = *reinterpret_cast<const ulonglong2*>(sEi + 8 * c8);
                            const ulonglong2 e1 = *reinterpret_cast<const ulonglong2*>(sEi + 8 * c8 + 4);
                            const uint64_t evs[4] = {e0.x, e0.y, e1.x, e1.y};
#pragma unroll
                            for (int u2 = 0; u2 < 4; ++u2)
                                unpk2(fmul2(fmul2(rc2, evs[u2]), pk2(raw[8 * c4 + 2 * u2], raw[8 * c4 + 2 * u2 + 1])),
                                      x[2 * u2], x[2 * u2 + 1]);
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) x[u] = (8 * c8 + u <= i && i < c) ? x[u] : 0.f;
                        uint4 q4;
                        q4.x = pack_bf16(x[0], x[1]);
                        q4.y = pack_bf16(x[2], x[3]);
                        q4.z = pack_bf16(x[4], x[5]);
                        q4.w = pack_bf16(x[6], x[7]);
                        *reinterpret_cast<uint4*>(pt + i * 128 + ((c8 ^ (i & 7)) << 4)) = q4;
                    }
                }
            }
            if (!qrows && P.logb && (w >> 2) == (wq & 1)) {  // warps 0 and 5 hold |k_i|^2
                // log of a bound on the 2-norm of this chunk's state transition: per token
                // exp(g) (I - beta k k^T), whose norm is exp(g) max(1, |1 - beta |k|^2|); the
                // 1e-3 |beta |k|^2| term covers the rounding of |k|^2.  Row i's term, summed
                // over the warp, then over the two warps (rows 0-31, 32-63) below
                float term = 0.f;
                if (i < c) {
                    const float t = bi * kn;
                    const float a = fabsf(1.f - t) + 1e-3f * fabsf(t);
                    term = sGin[(hh * 2) * CH + i] + logf(fmaxf(1.f, a));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) term += __shfl_xor_sync(0xffffffffu, term, off);
                if (lane == 0) sPart[wq & 1] = term;
            }
        }
        __syncthreads();
        PTRACE(2);
        if (tid == 32 && P.logb) P.logb[int64_t(gch) * P.Hv + j] = sPart[0] + sPart[1];

        // T = (I + A)^-1: diagonal blocks by substitution (warp q < 4, lane = column) ...
        if (w < 4 && lane < 16) {
            const int col = lane;
            const float* ab = ablk(tri(w, w));
            float* tb = tblk(tri(w, w));
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) {
                    if (m & 1) a1 = fmaf(ab[r * BLD + m], x[m], a1);
                    else a0 = fmaf(ab[r * BLD + m], x[m], a0);
                }
                x[r] = (r == col) ? 1.f : (r < col ? 0.f : -(a0 + a1));
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) tb[r * BLD + col] = x[r];
        }
        __syncthreads();
        // ... then the off-diagonal blocks on TF32 tiles, by halves: with T_AA, T_BB the inverses
        // of the two 32 x 32 diagonal halves, T_BA = -T_BB (A_BA T_AA).  Three passes of at most
        // two 16 x 16 products per warp; scratch blocks S0..S3 in sTmp.
        {
            auto mm = [&](float (&acc)[2][4], const float* Am, const float* Bm) {  // acc += Am Bm
#pragma unroll
                for (int kk = 0; kk < 16; kk += 8) {
                    const float* ar = Am + gq * BLD + kk + tq;
                    const uint32_t a0 = f2tf32(ar[0]), a1 = f2tf32(ar[8 * BLD]), a2 = f2tf32(ar[4]),
                                   a3 = f2tf32(ar[8 * BLD + 4]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float* br = Bm + (kk + tq) * BLD + 8 * nt + gq;
                        mma_tf32(acc[nt], a0, a1, a2, a3, f2tf32(br[0]), f2tf32(br[4 * BLD]));
                    }
                }
            };
            auto put = [&](float* D, const float (&acc)[2][4], float sg) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float* tr = D + gq * BLD + 8 * nt + 2 * tq;
                    tr[0] = sg * acc[nt][0];
                    tr[1] = sg * acc[nt][1];
                    tr[8 * BLD] = sg * acc[nt][2];
                    tr[8 * BLD + 1] = sg * acc[nt][3];
                }
            };
            auto slot = [&](int q) { return sTmp + q * (16 * BLD); };
            float acc[2][4];
            auto zero = [&]() {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            };
            // pass 1: T10 = -T11 (A10 T00), T32 = -T33 (A32 T22); Y21 = A21 T11, Y31 = A31 T11
            zero();
            if (w == 0 || w == 1) {
                const int lo = 2 * w;  // 0 or 2
                mm(acc, ablk(tri(lo + 1, lo)), tblk(tri(lo, lo)));
                put(slot(w), acc, 1.f);
                __syncwarp();
                zero();
                mm(acc, tblk(tri(lo + 1, lo + 1)), slot(w));
                put(tblk(tri(lo + 1, lo)), acc, -1.f);
            } else if (w < 4) {
                mm(acc, ablk(tri(w, 1)), tblk(tri(1, 1)));
                put(slot(w), acc, 1.f);
            }
            __syncthreads();
            // pass 2: Y20 = A20 T00 + A21 T10 (S0), Y30 = A30 T00 + A31 T10 (S1);
            // T21 = -T22 Y21, T31 = -(T32 Y21 + T33 Y31)
            zero();
            if (w == 0 || w == 1) {
                mm(acc, ablk(tri(w + 2, 0)), tblk(tri(0, 0)));
                mm(acc, ablk(tri(w + 2, 1)), tblk(tri(1, 0)));
                __syncwarp();
                put(slot(w), acc, 1.f);
            } else if (w == 2) {
                mm(acc, tblk(tri(2, 2)), slot(2));
                put(tblk(tri(2, 1)), acc, -1.f);
            } else if (w == 3) {
                mm(acc, tblk(tri(3, 2)), slot(2));
                mm(acc, tblk(tri(3, 3)), slot(3));
                put(tblk(tri(3, 1)), acc, -1.f);
            }
            __syncthreads();
            // pass 3: T20 = -T22 Y20, T30 = -(T32 Y20 + T33 Y30)
            if (w == 0) {
                zero();
                mm(acc, tblk(tri(2, 2)), slot(0));
                put(tblk(tri(2, 0)), acc, -1.f);
            } else if (w == 1) {
                zero();
                mm(acc, tblk(tri(3, 2)), slot(0));
                mm(acc, tblk(tri(3, 3)), slot(1));
                put(tblk(tri(3, 0)), acc, -1.f);
            }
            __syncthreads();
        }
        PTRACE(3);
        // TU = T diag(beta) and TW = -T diag(beta e) as swizzled bf16 tiles over the dead A
        // blocks: TU leaves by a bulk copy, TW is the B operand of W'^T = K^T TW^T
        // item it -> row r = it % 64 (consecutive lanes take consecutive rows of one block:
        // conflict-free reads with the block row stride, and the swizzled stores spread over
        // all banks), 8-column chunk c8 = it / 64 (warp-uniform: broadcast gate loads)
        for (int it = tid; it < CH * 8; it += PT) {
            const int r = it & 63, c8 = it >> 6;
            // T is exactly zero above its diagonal (the substitution writes those zeros and the
            // blocks above it are not read), so the products need no mask: two packed products
            // per pair of columns
            ulonglong2 t0 = make_ulonglong2(0ull, 0ull), t1 = t0;
            if ((c8 >> 1) <= (r >> 4)) {
                const float* tp = tblk(tri(r >> 4, c8 >> 1)) + (r & 15) * BLD + (c8 & 1) * 8;
                t0 = *reinterpret_cast<const ulonglong2*>(tp);
                t1 = *reinterpret_cast<const ulonglong2*>(tp + 4);
            }
            const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(sBeta + 8 * c8);
            const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(sBeta + 8 * c8 + 4);
            const ulonglong2 n0 = *reinterpret_cast<const ulonglong2*>(sNbe + 8 * c8);
            const ulonglong2 n1 = *reinterpret_cast<const ulonglong2*>(sNbe + 8 * c8 + 4);
            float xu[8], xw[8];
            unpk2(fmul2(t0.x, b0.x), xu[0], xu[1]);
            unpk2(fmul2(t0.y, b0.y), xu[2], xu[3]);
            unpk2(fmul2(t1.x, b1.x), xu[4], xu[5]);
            unpk2(fmul2(t1.y, b1.y), xu[6], xu[7]);
            unpk2(fmul2(t0.x, n0.x), xw[0], xw[1]);
            unpk2(fmul2(t0.y, n0.y), xw[2], xw[3]);
            unpk2(fmul2(t1.x, n1.x), xw[4], xw[5]);
            unpk2(fmul2(t1.y, n1.y), xw[6], xw[7]);
            uint4 a, b;
            a.x = pack_bf16(xu[0], xu[1]);
            a.y = pack_bf16(xu[2], xu[3]);
            a.z = pack_bf16(xu[4], xu[5]);
            a.w = pack_bf16(xu[6], xu[7]);
            b.x = pack_bf16(xw[0], xw[1]);
            b.y = pack_bf16(xw[2], xw[3]);
            b.z = pack_bf16(xw[4], xw[5]);
            b.w = pack_bf16(xw[6], xw[7]);
            const uint32_t off = r * 128 + ((c8 ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(smem + S::oQ0 + off) = a;  // TU staging
            *reinterpret_cast<uint4*>(smem + S::oQ1 + off) = b;  // TW operand tile
        }
        fence_proxy_async_smem();
        __syncthreads();
        PTRACE(4);
        if (tid == 0) {
            // W'^T [dk][i] = K^T TW^T into TMEM columns [64, 128), then TU's record copy
            constexpr uint32_t ID2 = make_idesc(128, 64, 1, 0);
            const uint64_t da = make_desc(kq, 16384, 1024);
            const uint64_t db = make_desc(smem_addr(smem + S::oQ1), 0, 1024);
            fence_after_sync();
#pragma unroll
            for (int st = 0; st < 4; ++st) mma_bf16(tm + 64, da + (st * 2048 >> 4), db + (st * 32 >> 4), ID2, st > 0);
            commit(&bars[2]);
            bulk_store(rec + PREP_TU, smem + S::oQ0, 8192);
            bulk_commit();
        }
        // T itself for the backward (the record's swizzled bf16 image) and for the low-level
        // output: 16-byte stores straight from the fp32 blocks while the W' product runs
        if (want_t) {
#pragma unroll
            for (int u4 = 0; u4 < TU4; ++u4) {
                const int it = tid + PT * u4, r = it & 63, c8 = it >> 6;  // as the staging above
                float t8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) t8[u] = 0.f;
                if ((c8 >> 1) <= (r >> 4)) {
                    const float* tp = tblk(tri(r >> 4, c8 >> 1)) + (r & 15) * BLD + (c8 & 1) * 8;
#pragma unroll
                    for (int u = 0; u < 8; ++u) t8[u] = (8 * c8 + u <= r) ? tp[u] : 0.f;
                }
                uint4 q4;
                q4.x = pack_bf16(t8[0], t8[1]);
                q4.y = pack_bf16(t8[2], t8[3]);
                q4.z = pack_bf16(t8[4], t8[5]);
                q4.w = pack_bf16(t8[6], t8[7]);
                if (store_t) *reinterpret_cast<uint4*>(rec + PREP_T + r * 128 + ((c8 ^ (r & 7)) << 4)) = q4;
                if (P.a_out && r < c &&  // token tc + r: its row of T, 64 bf16 columns
                    in_range(((tc + r) * P.Hv + j) * CH + 8 * c8 + 7, T_all * P.Hv * CH, err))
                    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(P.a_out) +
                                              ((tc + r) * P.Hv + j) * CH + 8 * c8) = q4;
            }
        }
        {
            const bool ok = warp_uniform_wait(&bars[2], hh & 1);
            if (!ok && lane == 0 && err) atomicOr(err, 1 << 27);
        }
        if (tid == 0) bulk_wait_read0();  // TU's staging has been read: W' may take it
        __syncthreads();
        PTRACE(5);
        fence_after_sync();
        {
            // thread = key row dk, warp w its half w / 4 of the 64 tokens; W' row i, column dk
            // goes to its K-major staging block (columns 0-63 over the TU staging, 64-127 over
            // the consumed TW tile)
            const int dk = tid & 127;
            const uint32_t base = smem_addr(smem + ((dk >> 6) ? S::oQ1 : S::oQ0)) + (dk & 7) * 2;
            const int cch = (dk & 63) >> 3;
#pragma unroll 1
            for (int q16 = 0; q16 < 2; ++q16) {
                const int i0 = 32 * (w >> 2) + 16 * q16;
                float d[16];
                tmem_ld16(tm + (uint32_t(32 * (w & 3)) << 16) + 64 + i0, d);
                tmem_ld_wait();
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    const int i = i0 + ii;
                    sts16(base + i * 128 + ((cch ^ (i & 7)) << 4), __bfloat16_as_ushort(__float2bfloat16_rn(d[ii])));
                }
            }
            fence_proxy_async_smem();
        }
        fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            bulk_store(rec + PREP_W, smem + S::oQ0, 8192);
            bulk_store(rec + PREP_W + 8192, smem + S::oQ1, 8192);
            bulk_commit();
            PTRACE(6);
            PTRACE(7);
        }
    }
    if (tid == 0) bulk_wait_read0();  // the last head's stores have read their tiles
    __syncthreads();
    if (w == 0) {
        fence_after_sync();
        tmem_dealloc(tm, 128);
    }
}

}  // namespace

void launch_prep(const Problem& P, const TcMaps& maps, cudaStream_t st) {
    if (P.total_chunks <= 0) return;
    smem_attr(k_prep, int(PrepSmem::bytes));
    // a CTA prepares the v-heads of (a slice of) one q/k group in turn, sharing K, Q and
    // [K;Q] K^T; a launch too small to fill the SMs several times over gives each CTA one
    // v-head instead, so that the heads run side by side
    const int G = P.Hv / P.Hqk;
    Problem Q = P;
    Q.prep_heads = int64_t(P.total_chunks) * P.Hqk >= 2 * int64_t(sm_count()) ? std::min(G, PrepSmem::GMAX) : 1;
    const int nsl = (G + Q.prep_heads - 1) / Q.prep_heads;
    timing_begin("fwd_prep", st);
    launch_pdl(k_prep, dim3(P.total_chunks, P.Hqk * nsl), dim3(PT), PrepSmem::bytes, st, Q, maps);
    timing_end(st);
}

}  // namespace gdn

#ifdef GDN_TRACE
extern "C" int gdn_debug_prep_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, gdn::g_prep_trace, sizeof(gdn::g_prep_trace)));
}
#endif
