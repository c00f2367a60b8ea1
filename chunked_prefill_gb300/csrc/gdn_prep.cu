// Chunk-local preparation, fully parallel over (chunk, v-head), for the tensor-core scan.
//
// Per chunk of 64 tokens (FlashQLA pages, agentlenshq "GDN chunked prefill optimisation":
// the chunk-local W/U preparation): gamma = in-chunk cumsum of g, then
//     KK = K K^T, QK = Q K^T                        (bf16 mma.sync, fp32 accumulation)
//     A  = diag(beta) (KK * Dm),  P = QK * D         (D_ij = exp(gamma_i - gamma_j), i >= j)
//     T  = (I + A)^-1                                (fp32: substitution + TF32 block products)
//     TU = T diag(beta),  W' = -T diag(beta e) K     (W' = -W of the pages' WY form)
// W', TU and P leave as bf16 tiles already in the 128-byte-swizzled layout the scan's
// tensor-core operands use, so the scan moves them with plain bulk copies.  Rows and columns
// past the end of a sequence come out zero (g = beta = 0 and zero K/Q rows there).
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc05.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int PT = 128;  // threads
constexpr int CH = 64;
constexpr int LDK = KD + 8;  // bf16 operand rows
constexpr int LDA = 68;      // fp32 scratch rows
constexpr int LDW = 72;      // bf16 TW rows

// The fp32 A and T scratch reuse the K and Q tiles once [K;Q] K^T is in registers (small
// footprint: five CTAs per SM hide each other's latency).
struct PrepSmem {
    static constexpr size_t TILE = size_t(CH) * LDK * 2;
    static constexpr size_t oK = 0, oQ = oK + TILE, oA = oK, oT = oQ,
                            oTmp = oQ + TILE, oGam = oTmp + 4 * 16 * 20 * 4,
                            oE = oGam + CH * 4, oEi = oE + CH * 4, oBeta = oEi + CH * 4,
                            oBe = oBeta + CH * 4, oFlag = oBe + CH * 4;
    static constexpr size_t bytes = oFlag + 16;
    static_assert(size_t(CH) * LDA * 4 <= TILE, "fp32 scratch fits a bf16 tile");
    static_assert(size_t(CH) * LDW * 2 <= TILE && 16384 <= TILE, "TW and the W' staging fit a tile");
};

__device__ __forceinline__ void st_chunk8g(unsigned char* tile, int r, int ch, const float* x) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]);
    u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]);
    u.w = pack_bf16(x[6], x[7]);
    *reinterpret_cast<uint4*>(tile + r * 128 + ((ch ^ (r & 7)) << 4)) = u;
}

__global__ void __launch_bounds__(PT, 5) k_prep(Problem P) {
    extern __shared__ __align__(128) char smem[];
    using S = PrepSmem;
    __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smem + S::oK);
    __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem + S::oQ);
    float* sA = reinterpret_cast<float*>(smem + S::oA);
    float* sT = reinterpret_cast<float*>(smem + S::oT);
    float* sTmp = reinterpret_cast<float*>(smem + S::oTmp);
    float* sGam = reinterpret_cast<float*>(smem + S::oGam);
    float* sE = reinterpret_cast<float*>(smem + S::oE);
    float* sEi = reinterpret_cast<float*>(smem + S::oEi);
    float* sBeta = reinterpret_cast<float*>(smem + S::oBeta);
    float* sBe = reinterpret_cast<float*>(smem + S::oBe);
    int* sFlag = reinterpret_cast<int*>(smem + S::oFlag);

    const int gch = blockIdx.x, j = blockIdx.y;
    int lo = 0, hi = P.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.plan.chunk_off[mid] <= gch) lo = mid;
        else hi = mid - 1;
    }
    const int s = lo;
    if (gch >= P.plan.chunk_off[P.N]) return;
    const int ch = gch - P.plan.chunk_off[s];
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
    const int G = P.Hv / P.Hqk, qh = j / G;
    const int64_t qk_stride = int64_t(P.Hqk) * KD;
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(P.k) + qh * KD + tc * qk_stride;
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(P.q) + qh * KD + tc * qk_stride;

    for (int idx = tid; idx < CH * 16; idx += PT) {
        const int r = idx >> 4, cv = idx & 15;
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (r < c) {
            a = *reinterpret_cast<const uint4*>(kb + r * qk_stride + cv * 8);
            b = *reinterpret_cast<const uint4*>(qb + r * qk_stride + cv * 8);
        }
        *reinterpret_cast<uint4*>(sK + r * LDK + cv * 8) = a;
        *reinterpret_cast<uint4*>(sQ + r * LDK + cv * 8) = b;
    }
    if (w == 0) {
        float gv[2], bv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = 2 * lane + u;
            gv[u] = r < c ? P.g[(tc + r) * P.Hv + j] : 0.f;
            bv[u] = r < c ? P.beta[(tc + r) * P.Hv + j] : 0.f;
        }
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
            sBe[r] = bv[u] * e;
        }
        if (lane == 0) *sFlag = (last < -80.f || !(last == last)) ? 1 : 0;
    }
    __syncthreads();

    // [K;Q] K^T: warp w owns rows 32w..32w+31 of the stacked 128 x 64 product
    {
        const bool qrows = w >= 2;
        const __nv_bfloat16* Ab = qrows ? sQ : sK;
        const int rb = 32 * (w & 1);
        float acc0[8][4], acc1[8][4];
        zero_acc(acc0);
        zero_acc(acc1);
        warp_mma<8, false, true>(acc0, Ab, LDK, sK, LDK, rb, 0, KD);
        warp_mma<8, false, true>(acc1, Ab, LDK, sK, LDK, rb + 16, 0, KD);
        __syncthreads();  // K and Q tiles consumed: A and T may overwrite them
        const bool pw = *sFlag != 0;
        float* sP32 = sT;  // P in fp32 until it leaves; T overwrites it afterwards
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float(&acc)[8][4] = half ? acc1 : acc0;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = rb + 16 * half + gq + 8 * hh;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int jj = 8 * n + 2 * tq + u;
                        const float v = acc[n][2 * hh + u];
                        const float d = pw ? expf(sGam[i] - sGam[jj]) : sE[i] * sEi[jj];
                        if (!qrows) sA[i * LDA + jj] = (i > jj) ? sBeta[i] * d * v : 0.f;
                        else sP32[i * LDA + jj] = (i >= jj) ? d * v : 0.f;
                    }
                }
            }
        }
    }
    __syncthreads();
    // P leaves as a pre-swizzled bf16 tile: eight threads per 128-byte row
    {
        unsigned char* ptile = static_cast<unsigned char*>(P.prep) +
                               (int64_t(gch) * P.Hv + j) * PREP_TILE_BYTES + PREP_P;
        for (int it = tid; it < CH * 8; it += PT) {
            const int r = it >> 3, c8 = it & 7;
            const float4 a = *reinterpret_cast<const float4*>(sT + r * LDA + 8 * c8);
            const float4 b = *reinterpret_cast<const float4*>(sT + r * LDA + 8 * c8 + 4);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            st_chunk8g(ptile, r, c8, x);
        }
    }
    __syncthreads();

    // T = (I + A)^-1: diagonal blocks by substitution (warp q, lane = column) ...
    if (lane < 16) {
        const int b0 = 16 * w, col = lane;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) {
                if (m & 1) a1 = fmaf(sA[(b0 + r) * LDA + b0 + m], x[m], a1);
                else a0 = fmaf(sA[(b0 + r) * LDA + b0 + m], x[m], a0);
            }
            x[r] = (r == col) ? 1.f : (r < col ? 0.f : -(a0 + a1));
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(b0 + r) * LDA + b0 + col] = x[r];
    }
    __syncthreads();
    // ... then the off-diagonal blocks on TF32 tiles, one block sub-diagonal per step
    {
        float* xs = sTmp + w * (16 * 20);
#pragma unroll 1
        for (int dd = 1; dd < 4; ++dd) {
            const int J = w, I = w + dd;
            if (I < 4) {
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                for (int M = J; M < I; ++M) {
#pragma unroll
                    for (int kk = 0; kk < 16; kk += 8) {
                        const float* ar = sA + (16 * I + gq) * LDA + 16 * M + kk + tq;
                        const uint32_t a0 = f2tf32(ar[0]), a1 = f2tf32(ar[8 * LDA]),
                                       a2 = f2tf32(ar[4]), a3 = f2tf32(ar[8 * LDA + 4]);
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const float* br = sT + (16 * M + kk + tq) * LDA + 16 * J + 8 * nt + gq;
                            mma_tf32(acc[nt], a0, a1, a2, a3, f2tf32(br[0]), f2tf32(br[4 * LDA]));
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    xs[gq * 20 + 8 * nt + 2 * tq] = acc[nt][0];
                    xs[gq * 20 + 8 * nt + 2 * tq + 1] = acc[nt][1];
                    xs[(gq + 8) * 20 + 8 * nt + 2 * tq] = acc[nt][2];
                    xs[(gq + 8) * 20 + 8 * nt + 2 * tq + 1] = acc[nt][3];
                }
                __syncwarp();
                float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < 16; kk += 8) {
                    const float* ar = sT + (16 * I + gq) * LDA + 16 * I + kk + tq;
                    const uint32_t a0 = f2tf32(ar[0]), a1 = f2tf32(ar[8 * LDA]),
                                   a2 = f2tf32(ar[4]), a3 = f2tf32(ar[8 * LDA + 4]);
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float* br = xs + (kk + tq) * 20 + 8 * nt + gq;
                        mma_tf32(acc2[nt], a0, a1, a2, a3, f2tf32(br[0]), f2tf32(br[4 * 20]));
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    float* tr = sT + (16 * I + gq) * LDA + 16 * J + 8 * nt + 2 * tq;
                    tr[0] = -acc2[nt][0];
                    tr[1] = -acc2[nt][1];
                    tr[8 * LDA] = -acc2[nt][2];
                    tr[8 * LDA + 1] = -acc2[nt][3];
                }
                __syncwarp();
            }
            __syncthreads();
        }
    }
    // TU = T diag(beta) leaves as a swizzled bf16 tile (eight threads per 128-byte row);
    // TW = -T diag(beta e) goes to shared memory (bf16, row stride LDW) over the dead A
    unsigned char* rec = static_cast<unsigned char*>(P.prep) + (int64_t(gch) * P.Hv + j) * PREP_TILE_BYTES;
    __nv_bfloat16* sTW = reinterpret_cast<__nv_bfloat16*>(smem + S::oK);
    for (int it = tid; it < CH * 8; it += PT) {
        const int r = it >> 3, c8 = it & 7;
        const float4 t0 = *reinterpret_cast<const float4*>(sT + r * LDA + 8 * c8);
        const float4 t1 = *reinterpret_cast<const float4*>(sT + r * LDA + 8 * c8 + 4);
        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        float xu[8], xw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = 8 * c8 + u;
            xu[u] = c <= r ? tv[u] * sBeta[c] : 0.f;
            xw[u] = c <= r ? -tv[u] * sBe[c] : 0.f;
        }
        st_chunk8g(rec + PREP_TU, r, c8, xu);
        uint4 w4;
        w4.x = pack_bf16(xw[0], xw[1]);
        w4.y = pack_bf16(xw[2], xw[3]);
        w4.z = pack_bf16(xw[4], xw[5]);
        w4.w = pack_bf16(xw[6], xw[7]);
        *reinterpret_cast<uint4*>(sTW + r * LDW + 8 * c8) = w4;
    }
    __syncthreads();  // T is dead: K comes back (from L2) over it
    __nv_bfloat16* sK2 = reinterpret_cast<__nv_bfloat16*>(smem + S::oT);
    for (int idx = tid; idx < CH * 16; idx += PT) {
        const int r = idx >> 4, cv = idx & 15;
        uint4 a = make_uint4(0, 0, 0, 0);
        if (r < c) a = *reinterpret_cast<const uint4*>(kb + r * qk_stride + cv * 8);
        *reinterpret_cast<uint4*>(sK2 + r * LDK + cv * 8) = a;
    }
    __syncthreads();
    // W' = TW K (64 x 128): warp w owns rows 16w..16w+15; TW is lower triangular, so only the
    // first 16(w+1) inner indices contribute
    float acc[16][4];
    zero_acc(acc);
    warp_mma<16, false, false>(acc, sTW, LDW, sK2, LDK, 16 * w, 0, 16 * (w + 1));
    __syncthreads();  // TW consumed: the staging tile overwrites it
    {
        unsigned char* stg = reinterpret_cast<unsigned char*>(smem + S::oK);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = 16 * w + gq + 8 * hh;
                const uint32_t v2 = pack_bf16(acc[n][2 * hh], acc[n][2 * hh + 1]);
                *reinterpret_cast<uint32_t*>(stg + (n >> 3) * 8192 + i * 128 + (((n & 7) ^ (i & 7)) << 4) +
                                             4 * tq) = v2;
            }
        }
    }
    __syncthreads();
    for (int it = tid; it < 16384 / 16; it += PT)
        reinterpret_cast<uint4*>(rec + PREP_W)[it] = reinterpret_cast<const uint4*>(smem + S::oK)[it];
}

}  // namespace

void launch_prep(const Problem& P, cudaStream_t st) {
    if (P.total_chunks <= 0) return;
    cudaFuncSetAttribute(k_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, int(PrepSmem::bytes));
    timing_begin("fwd_prep", st);
    k_prep<<<dim3(P.total_chunks, P.Hv), PT, PrepSmem::bytes, st>>>(P);
    timing_end(st);
}

}  // namespace gdn
