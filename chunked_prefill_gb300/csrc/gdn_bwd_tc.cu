// Local gradients of the chunked gated delta rule backward on the 5th-generation tensor cores
// (bf16 operands in shared memory, fp32 accumulators in tensor memory).
//
// The algebra is the one at the top of gdn_bwd.cu (FlashQLA pages, agentlenshq "backward pass"
// paragraph).  One persistent CTA per SM walks the (chunk, v-head) items.  Per item the inputs
// are the chunk's tiles K, Q, V, dO (TMA), its record from the forward preparation (W', TU =
// T diag(beta), P, T: bulk copies of 128-byte-swizzled images), the state h entering the chunk
// and the gradient dh of the state leaving it (TMA).  Every product is a 128-row tcgen05
// product with N = 64:
//
//   * products with a 128-wide side (key dk or value v) are formed TRANSPOSED, that side on the
//     128 tensor-memory lanes and the chunk's 64 tokens on the columns (slots of 64 columns;
//     v, a, u, z name s0, s1, s6, s7 on even items and s6, s7, s0, s1 on odd ones):
//       v   V'^T = V^T TU^T + h^T W'^T                   a   dO^T P        s2  dh^T K^T
//           (dV'^T = scale a + s2 diag(kd))
//       s3  (dO h^T)^T = h dO^T                          s5  (V' dh^T)^T = dh V'^T
//       a   dW^T = -(h dV'^T)                            u   dYU^T = dV'^T T
//       z   (dQk K)^T = K^T dQk^T                        v   (dQk^T Q)^T = Q^T dQk, later
//       a   dYW^T = dW^T T                                   + ((dB + dB^T) K)^T
//   * the 64 x 64 products use lanes 0-63 of a 128-row product (the A rows past 64 read the
//     neighbouring tile; those lanes are never read):
//       s4  K K^T     v  dP = dO V'^T     u / s2  dW K^T, dV' V^T     s3  Z = dT T^T
//       s2  T^T Z
//
// Intermediate operands return to shared memory as bf16 128-byte-swizzled tiles with one
// tensor-memory lane per tile row (V'^T, dV'^T, dW^T: 128 rows of 64 tokens; dQk, dT, Z,
// dB + dB^T: 64 x 64), and the next products read them K-major or MN-major as their roles
// need.  Per-token sums over the 128-wide side (the dgamma and dbeta terms) are butterfly
// transposes across the 32 lanes of a warp, then a fixed-order sum over the four lane
// quarters (deterministic).
//
// 16 warps share every epilogue step (warp w: lanes 32 (w % 4) .. + 31, 16 of the 64
// columns); the 64-row steps fall to the warps of lane quarters 0 and 1, and the others take
// the <dh, h> sum and the per-token pre-sums meanwhile.  One thread, lane 0 of warp 2 (no share
// in the 64-row steps), requests every copy and issues every product: a tcgen05.mma issue
// waits for the tensor pipe, so the issuing warp loses the execution time of what it issues.
// While an item's later products run, the next item's tiles are requested into the regions
// the remaining products no longer read (K and Q alternate between two regions so that the
// next K lands while the last product still reads this K), and its first products are issued
// into the slots this item no longer uses.  Every wait on an mbarrier is bounded; on a timeout
// the CTA records an error word, lets its copies and products drain (again bounded) and leaves.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc05.cuh"

namespace gdn {
namespace {

using namespace tc;

#ifdef GDN_TRACE
__device__ unsigned long long g_tcl_trace[48];  // debug builds: SM clock at the steps of one item of CTA 0
#define TTRACE(e)                                                                                \
    do {                                                                                         \
        if (blockIdx.x == 0 && threadIdx.x == 0 && n == 2 && (e) >= 0 && (e) < 20) g_tcl_trace[e] = clock64(); \
    } while (0)
#define ITRACE(e)                                                                                \
    do {                                                                                         \
        if (blockIdx.x == 0 && n == 2 && (e) >= 0 && (e) < 16) g_tcl_trace[20 + (e)] = clock64(); \
    } while (0)
#else
#define ITRACE(e) \
    do {          \
    } while (0)
#define TTRACE(e) \
    do {          \
    } while (0)
#endif

constexpr int LT = 512;   // 16 warps; warp w reads tensor-memory lanes [32 (w % 4), +32),
                          // columns [16 (w / 4), +16) of a 64-column accumulator
constexpr int LCH = 64;   // chunk

// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t L_K = 0;         // K   [64 tok][128 dk]   two 8 KB column blocks
constexpr uint32_t L_Q = 16384;     // Q
constexpr uint32_t L_V = 32768;     // V   [64 tok][128 v]
constexpr uint32_t L_DO = 49152;    // dO; from the dW product on dW^T [128 dk][64 tok]
constexpr uint32_t L_W = 65536;     // W' (record); from the V' product on V'^T [128 v][64 tok]
constexpr uint32_t L_TU = 81920;    // TU  [64 i][64 j]  (record)
constexpr uint32_t L_P = 90112;     // P   (record)
constexpr uint32_t L_T = 98304;     // T   (record)
constexpr uint32_t L_DT = 106496;   // dT [64 i][64 j]; later dB + dB^T
constexpr uint32_t L_QK = 114688;   // dQk [64 i][64 j]; later Z
constexpr uint32_t L_DV = 122880;   // dV'^T [128 v][64 tok]
constexpr uint32_t L_H = 139264;    // h  [128 dk][128 v]  two 16 KB column blocks
constexpr uint32_t L_DH = 172032;   // dh
constexpr uint32_t L_STG = 204800;  // dB fp32 [64][64], 16-byte chunks XOR-swizzled by row
constexpr uint32_t L_SM = 221184;   // small arrays (floats)
constexpr int F_GAM = 0, F_E = 64, F_KD = 128, F_BETA = 192, F_BE = 256;
constexpr int F_PPR = 320;   // [4][64]  row sums of dP * P (by column group)
constexpr int F_PPC = 576;   // [2][64]  column sums of dP * P (by lane quarter 0, 1)
constexpr int F_PQ = 704;    // [4][64]  <Q_i, (dO h^T)_i>    (by lane quarter)
constexpr int F_PR = 960;    // [4][64]  <K_i, (V' dh^T)_i>
constexpr int F_PTW = 1216;  // [4][64]  <K_i, dYW_i>
constexpr int F_PTU = 1472;  // [4][64]  <V_i, dYU_i>
constexpr int F_PAR = 1728;  // [4][64]  row sums of dA * A (by column group)
constexpr int F_PAC = 1984;  // [2][64]  column sums of dA * A
constexpr int F_PRS = 2112;  // [4][64]  row sums of dA * (Dm * Bm)
constexpr int F_RED = 2368;  // [16]     <dh, h> by warp
constexpr int F_EI = 2384;   // [64]     exp(-gamma)
constexpr int F_PW = 2448;   // (int)    1: exp(gamma_i - gamma_j) formed directly (extreme decay)
constexpr int F_END = 2452;
constexpr uint32_t L_BAR = L_SM + F_END * 4;
// copies landed (B_*); products done (M_*: M_1 dO^T P, M_10 dh^T K^T, M_2 h dO^T, M_11 K K^T,
// committed by whichever thread issued them)
enum LocBar { B_K = 0, B_Q, B_V, B_DO, B_W, B_TU, B_P, B_T, B_H, B_DH, NLD,
              M_0 = NLD, M_1, M_2, M_3, M_4, M_5, M_6, M_7, M_8, M_9, M_10, M_11, M_DRAIN, NBAR };
// The thread that requests every copy and issues every product: lane 0 of warp 2, which has no
// share in the 64-row epilogues, so that the next item's first products (issued there) cost
// no epilogue time.
constexpr int ISS = 64;
constexpr uint32_t L_SLOT = L_BAR + NBAR * 8;  // TMEM base address, error word
constexpr uint32_t L_END = L_SLOT + 16;
constexpr uint32_t LOC_SMEM = L_END + 1024;    // + alignment slack
static_assert(L_BAR % 8 == 0, "mbarrier alignment");
static_assert(LOC_SMEM <= 232448, "shared memory budget");

// tensor-memory slots of 64 columns
constexpr uint32_t SL0 = 0, SL1 = 64, SL2 = 128, SL3 = 192, SL4 = 256, SL5 = 320, SL6 = 384, SL7 = 448;

// M = 128, N = 64 instruction descriptors by (A major, B major): K = K-major, M = MN-major
constexpr uint32_t ID_KK = make_idesc(128, 64, 0, 0);
constexpr uint32_t ID_KM = make_idesc(128, 64, 0, 1);
constexpr uint32_t ID_MK = make_idesc(128, 64, 1, 0);
constexpr uint32_t ID_MM = make_idesc(128, 64, 1, 1);

// K step s (16 elements) of a K-major SW128 tile of R rows (64-column blocks at R * 128 bytes)
__device__ __forceinline__ uint64_t dK_(uint32_t base, uint32_t R, int s) {
    return make_desc(base + uint32_t(s >> 2) * R * 128u + uint32_t(s & 3) * 32u, 0, 1024);
}
// K step s (16 rows) of an MN-major SW128 tile (rows along K; 64-wide M/N blocks at lbo)
__device__ __forceinline__ uint64_t dM_(uint32_t base, uint32_t lbo, int s) {
    return make_desc(base + uint32_t(s) * 2048u, lbo, 1024);
}

__device__ __forceinline__ unsigned char* loc_smem() {
    extern __shared__ __align__(1024) unsigned char loc_raw[];
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(loc_raw) + 1023) & ~uintptr_t(1023));
}

// row r, columns [c0, c0 + 16) (c0 a multiple of 16) of a 64-column SW128 tile, as bf16
__device__ __forceinline__ void st_row16(uint32_t tile, int r, int c0, const float (&x)[16]) {
    const uint32_t row = tile + uint32_t(r) * 128u;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint32_t ch = uint32_t(((c0 >> 3) + u) ^ (r & 7));
        uint4 q;
        q.x = pack_bf16(x[8 * u], x[8 * u + 1]);
        q.y = pack_bf16(x[8 * u + 2], x[8 * u + 3]);
        q.z = pack_bf16(x[8 * u + 4], x[8 * u + 5]);
        q.w = pack_bf16(x[8 * u + 6], x[8 * u + 7]);
        sts128(row + ch * 16u, q);
    }
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// the same row segment read back as fp32
__device__ __forceinline__ void ld_row16(uint32_t tile, int r, int c0, float (&x)[16]) {
    const uint32_t row = tile + uint32_t(r) * 128u;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint32_t ch = uint32_t(((c0 >> 3) + u) ^ (r & 7));
        const uint4 q = lds128(row + ch * 16u);
        x[8 * u] = bf_lo(q.x);
        x[8 * u + 1] = bf_hi(q.x);
        x[8 * u + 2] = bf_lo(q.y);
        x[8 * u + 3] = bf_hi(q.y);
        x[8 * u + 4] = bf_lo(q.z);
        x[8 * u + 5] = bf_hi(q.z);
        x[8 * u + 6] = bf_lo(q.w);
        x[8 * u + 7] = bf_hi(q.w);
    }
}
// rows c0 .. c0 + 15 (c0 a multiple of 16) of column col of a [64][128] SW128 tile: the
// swizzled chunk of row c0 + ii depends on ii % 8 only, so eight bases serve the sixteen loads
__device__ __forceinline__ void ld_col16(uint32_t tile, int c0, int col, float (&x)[16]) {
    const uint32_t b0 = tile + uint32_t(col >> 6) * 8192u + uint32_t(c0) * 128u + uint32_t(col & 7) * 2u;
    const uint32_t ck = uint32_t((col & 63) >> 3);
    uint32_t bm[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) bm[m] = b0 + ((ck ^ uint32_t(m)) << 4);
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
        unsigned short h;
        asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(h) : "r"(bm[ii & 7] + uint32_t(ii) * 128u) : "memory");
        x[ii] = __uint_as_float(uint32_t(h) << 16);
    }
}

// Column sums over the 32 lanes of the warp of 16 values per lane (butterfly transpose):
// lanes 2m and 2m + 1 return the sum over all lanes of v[m].  v is clobbered.
__device__ __forceinline__ float lane_colsum16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
        const bool up = (lane & (2 * s)) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = up ? v[i] : v[i + s];
            const float keep = up ? v[i + s] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * s);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Paths that few items take, kept out of line so that the code every item runs stays compact
// (the kernel's code is larger than an SM's instruction cache; instruction-fetch stalls were
// the one stall that differed between otherwise identical runs).
struct F16 {
    float v[16];
};
// D_ij = exp(gamma_i - gamma_j) for the 16 columns from gam16, formed directly (a chunk whose
// decay is too steep for the products of exponentials)
__device__ __noinline__ F16 decay_row_direct(float gi, const float* gam16) {
    F16 r;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) r.v[jj] = expf(gi - gam16[jj]);
    return r;
}
// rows [0, n) of a 16-row column segment of a token-major bf16 gradient: element ii at
// col[ii * stride] (index idx0 + ii * stride of lim), for a chunk cut by the sequence end
__device__ __noinline__ void st_col_bf16(__nv_bfloat16* col, int64_t stride, F16 x, int n, int64_t idx0,
                                         int64_t lim, int* err) {
#pragma unroll 1
    for (int ii = 0; ii < 16; ++ii)
        if (ii < n && in_range(idx0 + ii * stride, lim, err)) col[ii * stride] = __float2bfloat16_rn(x.v[ii]);
}

// lane 0 waits (bounded, polling: a parked lane wakes too late for these waits, which are on
// the item's critical path), the result is broadcast to the warp
__device__ __forceinline__ bool lwait(uint64_t* bars, int b, uint32_t par, int* errflag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) {
        ok = mbar_wait_spin(&bars[b], par);
        if (!ok) atomicOr(errflag, 1 << b);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    return ok;
}
// single-thread wait (the issuer)
__device__ __forceinline__ bool twait(uint64_t* bars, int b, uint32_t par, int* errflag) {
    if (mbar_wait_spin(&bars[b], par)) return true;
    atomicOr(errflag, 1 << b);
    return false;
}

struct LocMaps {
    CUtensorMap k, q, v, dO, h, dh;
    CUtensorMap dv, dq, dk;  // outputs (dq, dk: bf16 ones only, G = 1)
};

// byte offset of element (row t, column col) of a [64][128] bf16 tile in the 128-byte-swizzled
// image a TMA box of 64 columns uses (two 8 KB column blocks)
__device__ __forceinline__ uint32_t out_tile_off(int t, int col) {
    return uint32_t(col >> 6) * 8192u + uint32_t(t) * 128u + (uint32_t(((col & 63) >> 3) ^ (t & 7)) << 4) +
           uint32_t(col & 7) * 2u;
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

struct Item {
    int gch, j, qh, c;
    int64_t tc;
};

// PART: several v-heads share a q/k head, so dq and dk go to the fp32 per-v-head partials
// (B.dqp, B.dkp) that a later kernel reduces
template <bool PART>
__global__ void __launch_bounds__(LT, 1) k_tc_bwd_local(BwdProblem B, const __grid_constant__ LocMaps maps,
                                                        int64_t items) {
    pdl_launch_dependents();
    unsigned char* sm = loc_smem();
    const Problem& P = B.f;
    float* sF = reinterpret_cast<float*>(sm + L_SM);
    float* sGam = sF + F_GAM;
    float* sE = sF + F_E;
    float* sKd = sF + F_KD;
    float* sBeta = sF + F_BETA;
    float* sBe = sF + F_BE;
    float* sEi = sF + F_EI;
    int* sPw = reinterpret_cast<int*>(sF + F_PW);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L_BAR);
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + L_SLOT);
    int* errflag = reinterpret_cast<int*>(sm + L_SLOT + 4);

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int q4 = w & 3, cg = w >> 2, c16 = 16 * cg;  // lane quarter, column group
    const uint32_t lb = uint32_t(32 * q4) << 16;
    const int Hv = P.Hv, Hqk = P.Hqk, G = Hv / Hqk;
    const float sc = P.scale;
    const int64_t qk_stride = int64_t(Hqk) * KD, v_stride = int64_t(Hv) * VD;
    const int64_t T_all = P.cu ? int64_t(P.T) : int64_t(P.N) * P.T;  // tokens (store extents)
    const uint32_t base = smem_addr(sm);
    const uint32_t aV = base + L_V, aDO = base + L_DO, aW = base + L_W, aTU = base + L_TU, aP = base + L_P,
                   aT = base + L_T, aDT = base + L_DT, aQK = base + L_QK, aDV = base + L_DV, aH = base + L_H,
                   aDH = base + L_DH, aSTG = base + L_STG;

    if (tid == 0) {
        for (int b = 0; b < NBAR; ++b) mbar_init(&bars[b], 1);
        *errflag = 0;
        mbar_fence_init();
    }
    if (w == 0) tmem_alloc(slot, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tm = *slot;
    pdl_wait();  // (the set-up above reads nothing an earlier kernel writes)

    auto locate = [&](int64_t item, Item& x) -> bool {
        const int gch = int(item / Hv);
        x.gch = gch;
        x.j = int(item % Hv);
        x.qh = x.j / G;
        if (gch >= plan_chunk_off(P.plan, P.N)) return false;
        int lo = 0, hi = P.N - 1;  // chunk -> sequence by binary search
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (plan_chunk_off(P.plan, mid) <= gch) lo = mid;
            else hi = mid - 1;
        }
        int64_t t0, t1;
        seq_bounds(P, lo, t0, t1);
        x.tc = t0 + int64_t(gch - plan_chunk_off(P.plan, lo)) * LCH;
        if (x.tc >= t1) return false;
        x.c = int((t1 - x.tc) < int64_t(LCH) ? (t1 - x.tc) : int64_t(LCH));
        return true;
    };

    // Tensor-memory slots of an item: an odd item swaps {s0, s1} with {s6, s7}, so that the next
    // item's first products can go to the slots this item no longer uses while its last product
    // and the dK epilogue still hold s0, s1 (or s6, s7) and s5.  K and Q trade shared-memory
    // regions the same way (K of an even item in the K region), so that the next item's K can
    // land while the last product still reads this item's K.
    auto slot_v = [](uint32_t par) { return par ? SL6 : SL0; };
    auto slot_a = [](uint32_t par) { return par ? SL7 : SL1; };
    auto slot_u = [](uint32_t par) { return par ? SL0 : SL6; };
    auto slot_z = [](uint32_t par) { return par ? SL1 : SL7; };
    auto kreg_of = [](uint32_t par) { return par ? L_Q : L_K; };
    auto qreg_of = [](uint32_t par) { return par ? L_K : L_Q; };

    // ---- copies and products (thread ISS only); ldn counts the phases requested on each load barrier
    int ldn[NLD];
#pragma unroll
    for (int b = 0; b < NLD; ++b) ldn[b] = 0;
    auto rec_of = [&](const Item& x) {
        return static_cast<const unsigned char*>(P.prep) + (int64_t(x.gch) * Hv + x.j) * P.prep_stride;
    };
    auto req_rows = [&](int b, uint32_t off, const CUtensorMap* m, int head, int64_t tcx) {
        mbar_expect_tx(&bars[b], 16384);
        tma_load_3d(sm + off, m, &bars[b], 0, head, int(tcx));
        tma_load_3d(sm + off + 8192, m, &bars[b], 64, head, int(tcx));
        ++ldn[b];
    };
    auto req_rec = [&](int b, uint32_t off, const Item& x, int roff, uint32_t bytes) {
        mbar_expect_tx(&bars[b], bytes);
        bulk_load(sm + off, rec_of(x) + roff, bytes, &bars[b]);
        ++ldn[b];
    };
    auto req_state = [&](int b, uint32_t off, const CUtensorMap* m, const Item& x) {
        const int row = (x.gch * Hv + x.j) * 128;
        mbar_expect_tx(&bars[b], 32768);
        tma_load_2d(sm + off, m, &bars[b], 0, row);
        tma_load_2d(sm + off + 16384, m, &bars[b], 64, row);
        ++ldn[b];
    };
    auto req_K = [&](const Item& x, uint32_t off) { req_rows(B_K, off, &maps.k, x.qh, x.tc); };
    auto req_Q = [&](const Item& x, uint32_t off) { req_rows(B_Q, off, &maps.q, x.qh, x.tc); };
    auto req_V = [&](const Item& x) { req_rows(B_V, L_V, &maps.v, x.j, x.tc); };
    auto req_DO = [&](const Item& x) { req_rows(B_DO, L_DO, &maps.dO, x.j, x.tc); };
    auto req_W = [&](const Item& x) { req_rec(B_W, L_W, x, PREP_W, 16384); };
    auto req_TU = [&](const Item& x) { req_rec(B_TU, L_TU, x, PREP_TU, 8192); };
    auto req_P = [&](const Item& x) { req_rec(B_P, L_P, x, PREP_P, 8192); };
    auto req_T = [&](const Item& x) { req_rec(B_T, L_T, x, PREP_T, 8192); };
    auto req_H = [&](const Item& x) { req_state(B_H, L_H, &maps.h, x); };
    auto req_DH = [&](const Item& x) { req_state(B_DH, L_DH, &maps.dh, x); };
    // the first products of an item in two groups: V'^T, dO^T P, h dO^T (need V, TU, W', h, dO,
    // P) and dh^T K^T, K K^T (need dh, K)
    auto issue_A = [&](uint32_t xpar) {
        const uint32_t s_v = slot_v(xpar), s_a = slot_a(xpar);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16(tm + s_v, dM_(aV, 8192, s), dK_(aTU, 64, s), ID_MK, s > 0);
#pragma unroll
        for (int s = 0; s < 8; ++s) mma_bf16(tm + s_v, dM_(aH, 16384, s), dK_(aW, 64, s), ID_MK, 1u);
        commit(&bars[M_0]);
#pragma unroll
        for (int s = 0; s < 4; ++s) mma_bf16(tm + s_a, dM_(aDO, 8192, s), dM_(aP, 8192, s), ID_MM, s > 0);
        commit(&bars[M_1]);
#pragma unroll
        for (int s = 0; s < 8; ++s) mma_bf16(tm + SL3, dK_(aH, 128, s), dK_(aDO, 64, s), ID_KK, s > 0);
        commit(&bars[M_2]);
    };
    auto issue_B = [&](uint32_t xpar) {
        const uint32_t xK = base + kreg_of(xpar);
#pragma unroll
        for (int s = 0; s < 8; ++s) mma_bf16(tm + SL2, dM_(aDH, 16384, s), dK_(xK, 64, s), ID_MK, s > 0);
        commit(&bars[M_10]);
#pragma unroll
        for (int s = 0; s < 8; ++s) mma_bf16(tm + SL4, dK_(xK, 64, s), dK_(xK, 64, s), ID_KK, s > 0);
        commit(&bars[M_11]);
    };
    // (issuer) copies of the next item landed within limit_ns (polling; no error when not)
    auto landed = [&](uint32_t npar, bool group_a, uint64_t limit_ns) -> bool {
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            const bool in = group_a ? (mbar_test(&bars[B_V], npar) && mbar_test(&bars[B_TU], npar) &&
                                       mbar_test(&bars[B_W], npar) && mbar_test(&bars[B_H], npar) &&
                                       mbar_test(&bars[B_DO], npar) && mbar_test(&bars[B_P], npar))
                                    : (mbar_test(&bars[B_DH], npar) && mbar_test(&bars[B_K], npar));
            if (in) return true;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    };

    bool pre = false;             // (issuer) the current item's tiles were requested during the previous one
    bool eA = false, eB = false;  // (issuer) its first product groups were issued during the previous one
    float ngv[2] = {0.f, 0.f}, nbv[2] = {0.f, 0.f};  // (warp 0) the next item's g, beta
    bool have_ng = false;
    bool failed = false;
    bool carry_ok = true;  // the previous item's last step (its failure is acted on at the next barrier)
    uint32_t n = 0;      // items done (parity of every barrier phase)
#pragma unroll 1
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        Item cur, nxt;
        if (!locate(item, cur)) {
            pre = false;
            eA = eB = false;
            have_ng = false;
            continue;
        }
        const bool has_next = item + gridDim.x < items && locate(item + gridDim.x, nxt);
        const uint32_t par = n & 1;
        TTRACE(0);
        const uint32_t sv = slot_v(par), sa = slot_a(par), su = slot_u(par), sz = slot_z(par);
        const uint32_t kreg = kreg_of(par), qreg = qreg_of(par);
        const uint32_t aK = base + kreg, aQ = base + qreg;
        const int j = cur.j, qh = cur.qh, c = cur.c;
        const int64_t tc = cur.tc;
        // a full chunk's dv (and with G = 1 its dq, dk) leave as tile stores of staged images:
        // dv and dk through the dB staging region, dq through the dV' region (both free then);
        // thread 0 issues each store after the barrier that follows its staging and waits for
        // its reads before the barrier that precedes the region's next writer
        const bool tile_out = c == LCH;
        bool ok = true;
        bool nA = false, nB = false;  // (issuer) the next item's groups issued during this one
        if (tid == ISS && !pre) {
            req_K(cur, kreg);
            req_V(cur);
            req_W(cur);
            req_TU(cur);
            req_H(cur);
            req_DO(cur);
            req_P(cur);
            req_DH(cur);
            req_Q(cur, qreg);
            req_T(cur);
        }

        // ---- gates (warp 0); rows past the sequence end: g = beta = 0
        if (w == 0) {
            float gv[2], bv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                const bool in = r < c;
                gv[u] = have_ng ? ngv[u] : (in ? P.g[(tc + r) * Hv + j] : 0.f);
                bv[u] = have_ng ? nbv[u] : (in ? P.beta[(tc + r) * Hv + j] : 0.f);
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
                sKd[r] = expf(last - gm[u]);
                sBeta[r] = bv[u];
                sBe[r] = bv[u] * e;
                sEi[r] = expf(-gm[u]);
            }
            if (lane == 0) *sPw = (last < -80.f || !(last == last)) ? 1 : 0;
        }
        // a chunk cut by the sequence end: the rows past it belong to the next sequence (or
        // are the fill past the tensor end); zero them in K, Q, V, dO
        if (c < LCH) {
            ok = lwait(bars, B_K, par, errflag) && lwait(bars, B_Q, par, errflag) &&
                 lwait(bars, B_V, par, errflag) && lwait(bars, B_DO, par, errflag);
            if (ok) {
                const int nz = (LCH - c) * 16;  // 16-byte chunks per tile
                const uint4 z = make_uint4(0, 0, 0, 0);
                for (int idx = tid; idx < 4 * nz; idx += LT) {
                    const int t = idx / nz, rem = idx % nz;
                    const int r = c + (rem >> 4), blk = (rem >> 3) & 1, ch = rem & 7;
                    sts128(base + uint32_t(t) * 16384u + uint32_t(blk) * 8192u + uint32_t(r) * 128u +
                               uint32_t(ch) * 16u,
                           z);
                }
                fence_proxy_async_smem();
            }
        }
        if (__syncthreads_or(!ok || !carry_ok)) { failed = true; break; }
        TTRACE(1);

        // ---- first products (those the previous item did not issue)
        if (tid == ISS) {
            ITRACE(0);
            fence_after_sync();
            if (!eA) {
                ok = twait(bars, B_V, par, errflag) && twait(bars, B_TU, par, errflag) &&
                     twait(bars, B_W, par, errflag) && twait(bars, B_H, par, errflag) &&
                     twait(bars, B_DO, par, errflag) && twait(bars, B_P, par, errflag);
                if (ok) {
                    issue_A(par);
                } else {
                    commit(&bars[M_0]);
                    commit(&bars[M_1]);
                    commit(&bars[M_2]);
                }
            }
            if (!eB) {
                ok = ok && twait(bars, B_DH, par, errflag) && twait(bars, B_K, par, errflag);
                if (ok) {
                    issue_B(par);
                } else {
                    commit(&bars[M_10]);
                    commit(&bars[M_11]);
                }
            }
            ITRACE(1);
        }
        __syncwarp();

        // V'^T -> bf16 tile (in the W' region)
        ok = lwait(bars, M_0, par, errflag) && ok;
        TTRACE(2);
        fence_after_sync();
        {
            float x[16];
            tmem_ld16(tm + lb + sv + c16, x);
            tmem_ld_wait();
            st_row16(aW, 32 * q4 + lane, c16, x);
        }
        if (tid == 0) bulk_wait_read0();  // the previous item's dq and dk stores have read their images
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(3);
        if (tid == ISS) {
            ITRACE(2);
            fence_after_sync();
            // dP = dO V'^T (lanes 0-63), (V' dh^T)^T = dh V'^T
#pragma unroll
            for (int s = 0; s < 8; ++s) mma_bf16(tm + sv, dK_(aDO, 64, s), dM_(aW, 16384, s), ID_KM, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) mma_bf16(tm + SL5, dK_(aDH, 128, s), dM_(aW, 16384, s), ID_KM, s > 0);
            commit(&bars[M_3]);
            ITRACE(3);
        }
        __syncwarp();

        // dV'^T = scale dO^T P + dh^T K^T diag(kd) -> bf16 tile
        ok = lwait(bars, M_1, par, errflag) && lwait(bars, M_10, par, errflag) && ok;
        TTRACE(4);
        fence_after_sync();
        {
            float a[16], b[16];
            tmem_ld16(tm + lb + sa + c16, a);
            tmem_ld16(tm + lb + SL2 + c16, b);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                const float4 kd = *reinterpret_cast<const float4*>(sKd + c16 + i);
                a[i] = sc * a[i] + kd.x * b[i];
                a[i + 1] = sc * a[i + 1] + kd.y * b[i + 1];
                a[i + 2] = sc * a[i + 2] + kd.z * b[i + 2];
                a[i + 3] = sc * a[i + 3] + kd.w * b[i + 3];
            }
            st_row16(aDV, 32 * q4 + lane, c16, a);
        }
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(5);
        if (tid == ISS) {
            ITRACE(4);
            fence_after_sync();
            ok = twait(bars, B_T, par, errflag);
            if (ok) {
                // dW^T = -(h dV'^T), dV' V^T (lanes 0-63), dYU^T = dV'^T T
#pragma unroll
                for (int s = 0; s < 8; ++s) mma_bf16(tm + sa, dK_(aH, 128, s), dM_(aDV, 16384, s), ID_KM, s > 0);
#pragma unroll
                for (int s = 0; s < 8; ++s) mma_bf16(tm + SL2, dM_(aDV, 16384, s), dK_(aV, 64, s), ID_MK, s > 0);
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tm + su, dK_(aDV, 128, s), dM_(aT, 8192, s), ID_KM, s > 0);
            }
            commit(&bars[M_4]);
            ITRACE(5);
        }
        __syncwarp();

        // dP (lanes 0-63): dgamma terms of dP * P, dQk = dP * D -> bf16 tile;
        // r_i = kd_i <K_i, (V' dh^T)_i> partial sums
        ok = lwait(bars, M_3, par, errflag) && lwait(bars, B_P, par, errflag) &&
             lwait(bars, B_K, par, errflag) && ok;
        TTRACE(6);
        fence_after_sync();
        if (q4 < 2) {
            const int i = 32 * q4 + lane;
            float x[16], pr[16];
            tmem_ld16(tm + lb + sv + c16, x);
            ld_row16(aP, i, c16, pr);
            tmem_ld_wait();
            const float gi = sGam[i], ei = sE[i];
            float dm[16];  // D_ij = exp(gamma_i - gamma_j)
            if (*sPw) {
                const F16 r = decay_row_direct(gi, sGam + c16);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) dm[jj] = r.v[jj];
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; jj += 4) {
                    const float4 e4 = *reinterpret_cast<const float4*>(sEi + c16 + jj);
                    dm[jj] = ei * e4.x;
                    dm[jj + 1] = ei * e4.y;
                    dm[jj + 2] = ei * e4.z;
                    dm[jj + 3] = ei * e4.w;
                }
            }
            float rs = 0.f;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int jx = c16 + jj;
                const bool on = i >= jx;
                const float v = on ? sc * x[jj] : 0.f;
                const float pp = v * pr[jj];
                rs += pp;
                pr[jj] = pp;
                x[jj] = on ? v * dm[jj] : 0.f;
            }
            sF[F_PPR + 64 * cg + i] = rs;
            const float cs = lane_colsum16(pr);
            if (!(lane & 1)) sF[F_PPC + 64 * q4 + c16 + (lane >> 1)] = cs;
            st_row16(aQK, i, c16, x);
        }
        {
            const int k = 32 * q4 + lane;
            float y[16];
            tmem_ld16(tm + lb + SL5 + c16, y);
            tmem_ld_wait();
            float kc[16];
            ld_col16(aK, c16, k, kc);
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) y[ii] *= kc[ii];
            const float cs = lane_colsum16(y);
            if (!(lane & 1)) sF[F_PR + 64 * q4 + c16 + (lane >> 1)] = cs;
        }
        if (q4 >= 2 && w != ISS / 32) {
            // <dh, h> over the two state tiles (identical swizzled layouts), by the warps without
            // a share in the 64-row epilogue other than the issuer's
            const int t2 = 32 * ((w >> 2) * 2 + (q4 - 2) - 1) + lane;  // 0 .. 223
            ok = lwait(bars, B_H, par, errflag) && lwait(bars, B_DH, par, errflag) && ok;
            float hd = 0.f;
#pragma unroll 1
            for (int u = t2; u < 2048; u += 224) {
                const uint32_t off = uint32_t(u) * 16u;
                const uint4 a = lds128(aH + off), b = lds128(aDH + off);
                hd += bf_lo(a.x) * bf_lo(b.x) + bf_hi(a.x) * bf_hi(b.x) + bf_lo(a.y) * bf_lo(b.y) +
                      bf_hi(a.y) * bf_hi(b.y) + bf_lo(a.z) * bf_lo(b.z) + bf_hi(a.z) * bf_hi(b.z) +
                      bf_lo(a.w) * bf_lo(b.w) + bf_hi(a.w) * bf_hi(b.w);
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, off);
            if (lane == 0) sF[F_RED + (t2 >> 5)] = hd;  // warps 0 .. 6 of this group
        }
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(7);
        if (tid == ISS) {
            ITRACE(6);
            fence_after_sync();
            // (dQk K)^T = K^T dQk^T, (dQk^T Q)^T = Q^T dQk
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tm + sz, dM_(aK, 8192, s), dK_(aQK, 64, s), ID_MK, s > 0);
            ok = twait(bars, B_Q, par, errflag);
            if (ok) {
#pragma unroll
                for (int s = 0; s < 4; ++s) mma_bf16(tm + sv, dM_(aQ, 8192, s), dM_(aQK, 8192, s), ID_MM, s > 0);
            }
            commit(&bars[M_5]);
            if (has_next) {  // W' (now V'^T), TU, P and dh are no longer read
                req_W(nxt);
                req_TU(nxt);
                req_P(nxt);
                req_DH(nxt);
            }
            ITRACE(7);
        }
        __syncwarp();

        // dW^T -> bf16 tile (in the dO region); dV = diag(beta) dYU, <V_i, dYU_i>
        ok = lwait(bars, M_4, par, errflag) && lwait(bars, B_V, par, errflag) && ok;
        TTRACE(8);
        fence_after_sync();
        {
            float x[16], y[16];
            tmem_ld16(tm + lb + sa + c16, x);
            tmem_ld16(tm + lb + su + c16, y);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = -x[i];
            st_row16(aDO, 32 * q4 + lane, c16, x);
            const int v = 32 * q4 + lane;
            float vc[16];
            ld_col16(aV, c16, v, vc);
            if (tile_out) {  // staged for the tile store (the dB staging region is free here)
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    sts16(aSTG + out_tile_off(c16 + ii, v),
                          __bfloat16_as_ushort(__float2bfloat16_rn(sBeta[c16 + ii] * y[ii])));
                    y[ii] *= vc[ii];
                }
            } else {
                F16 o;
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    o.v[ii] = sBeta[c16 + ii] * y[ii];
                    y[ii] *= vc[ii];
                }
                st_col_bf16(reinterpret_cast<__nv_bfloat16*>(B.dv) + int64_t(j) * VD + v + (tc + c16) * v_stride,
                            v_stride, o, c - c16, int64_t(j) * VD + v + (tc + c16) * v_stride, T_all * v_stride, P.err);
            }
            const float cs = lane_colsum16(y);
            if (!(lane & 1)) sF[F_PTU + 64 * q4 + c16 + (lane >> 1)] = cs;
        }
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(9);
        if (tid == 0 && tile_out) {
            tma_store_3d(&maps.dv, sm + L_STG, 0, j, int(tc));
            tma_store_3d(&maps.dv, sm + L_STG + 8192, 64, j, int(tc));
            bulk_commit();
        }
        if (tid == ISS) {
            ITRACE(8);
            fence_after_sync();
            // dW K^T (lanes 0-63), dYW^T = dW^T T
#pragma unroll
            for (int s = 0; s < 8; ++s) mma_bf16(tm + su, dM_(aDO, 16384, s), dK_(aK, 64, s), ID_MK, s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tm + sa, dK_(aDO, 128, s), dM_(aT, 8192, s), ID_KM, s > 0);
            commit(&bars[M_6]);
            if (has_next) {  // h and V are no longer read
                req_H(nxt);
                req_V(nxt);
            }
            ITRACE(9);
        }
        __syncwarp();

        // dQ = scale diag(e) dO h^T + dQk K; <Q_i, (dO h^T)_i>
        ok = lwait(bars, M_5, par, errflag) && lwait(bars, M_2, par, errflag) &&
             lwait(bars, B_Q, par, errflag) && ok;
        TTRACE(10);
        fence_after_sync();
        {
            float a[16], b[16];
            tmem_ld16(tm + lb + SL3 + c16, a);
            tmem_ld16(tm + lb + sz + c16, b);
            tmem_ld_wait();
            const int k = 32 * q4 + lane;
            if (PART) {
                float* dq = B.dqp + int64_t(j) * KD + k;
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    const int cx = c16 + ii;
                    if (cx < c && in_range(int64_t(j) * KD + k + (tc + cx) * Hv * KD, T_all * Hv * KD, P.err))
                        dq[(tc + cx) * Hv * KD] = sc * sE[cx] * a[ii] + b[ii];
                }
            } else if (tile_out) {  // staged in the dV' region (its last products have completed)
#pragma unroll
                for (int ii = 0; ii < 16; ++ii)
                    sts16(aDV + out_tile_off(c16 + ii, k),
                          __bfloat16_as_ushort(__float2bfloat16_rn(sc * sE[c16 + ii] * a[ii] + b[ii])));
                fence_proxy_async_smem();
            } else {
                F16 o;
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) o.v[ii] = sc * sE[c16 + ii] * a[ii] + b[ii];
                st_col_bf16(reinterpret_cast<__nv_bfloat16*>(B.dq) + int64_t(qh) * KD + k + (tc + c16) * qk_stride,
                            qk_stride, o, c - c16, int64_t(qh) * KD + k + (tc + c16) * qk_stride, T_all * qk_stride,
                            P.err);
            }
            float qc[16];
            ld_col16(aQ, c16, k, qc);
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) a[ii] *= qc[ii];
            const float cs = lane_colsum16(a);
            if (!(lane & 1)) sF[F_PQ + 64 * q4 + c16 + (lane >> 1)] = cs;
        }

        // dT = (dW K^T) diag(beta e) + (dV' V^T) diag(beta) (lanes 0-63) -> bf16 tile;
        // <K_i, dYW_i>
        ok = lwait(bars, M_6, par, errflag) && ok;
        TTRACE(11);
        fence_after_sync();
        if (tid == ISS && ok && has_next) req_DO(nxt);  // the dW products are done: next dO
        if (q4 < 2) {
            const int i = 32 * q4 + lane;
            float d1[16], d2[16];
            tmem_ld16(tm + lb + su + c16, d1);
            tmem_ld16(tm + lb + SL2 + c16, d2);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 16; jj += 4) {
                const float4 be = *reinterpret_cast<const float4*>(sBe + c16 + jj);
                const float4 bb = *reinterpret_cast<const float4*>(sBeta + c16 + jj);
                d1[jj] = be.x * d1[jj] + bb.x * d2[jj];
                d1[jj + 1] = be.y * d1[jj + 1] + bb.y * d2[jj + 1];
                d1[jj + 2] = be.z * d1[jj + 2] + bb.z * d2[jj + 2];
                d1[jj + 3] = be.w * d1[jj + 3] + bb.w * d2[jj + 3];
            }
            st_row16(aDT, i, c16, d1);
        }
        {
            const int k = 32 * q4 + lane;
            float z[16];
            tmem_ld16(tm + lb + sa + c16, z);
            tmem_ld_wait();
            float kc[16];
            ld_col16(aK, c16, k, kc);
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) z[ii] *= kc[ii];
            const float cs = lane_colsum16(z);
            if (!(lane & 1)) sF[F_PTW + 64 * q4 + c16 + (lane >> 1)] = cs;
        }
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(12);
        if (tid == 0 && tile_out && !PART) {
            tma_store_3d(&maps.dq, sm + L_DV, 0, qh, int(tc));
            tma_store_3d(&maps.dq, sm + L_DV + 8192, 64, qh, int(tc));
            bulk_commit();
        }
        if (tid == ISS) {
            ITRACE(10);
            fence_after_sync();
            // Z = dT T^T (lanes 0-63)
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tm + SL3, dK_(aDT, 64, s), dK_(aT, 64, s), ID_KK, s > 0);
            commit(&bars[M_7]);
            if (has_next) req_K(nxt, qreg);  // Q is no longer read: next K into its region
            ITRACE(11);
        }
        __syncwarp();

        // Z -> bf16 tile (in the dQk region)
        ok = lwait(bars, M_7, par, errflag) && ok;
        TTRACE(13);
        fence_after_sync();
        if (q4 < 2) {
            float x[16];
            tmem_ld16(tm + lb + SL3 + c16, x);
            tmem_ld_wait();
            st_row16(aQK, 32 * q4 + lane, c16, x);
        }
        if (tid == 0) bulk_wait_read0();  // dv's tile store has read the staging region
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(14);
        if (tid == ISS) {
            ITRACE(12);
            fence_after_sync();
            // T^T Z (lanes 0-63)
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tm + SL2, dM_(aT, 8192, s), dM_(aQK, 8192, s), ID_MM, s > 0);
            commit(&bars[M_8]);
            // the next item's first group while the 64-row epilogues run (its warp has no share in
            // them): slots s6/s7 (or s0/s1) and s3 are free
            if (has_next && nxt.c == LCH && landed(par ^ 1u, true, 1500)) {
                issue_A(par ^ 1u);
                nA = true;
            }
            ITRACE(13);
        }
        __syncwarp();

        // dA = strictly-lower(-T^T Z), its dgamma / dbeta terms with A = diag(beta) (Dm * Bm),
        // dB = diag(beta) (dA * Dm) -> fp32 staging -> dB + dB^T as a bf16 tile (dT region)
        ok = lwait(bars, M_8, par, errflag) && lwait(bars, M_11, par, errflag) && ok;
        TTRACE(15);
        fence_after_sync();
        if (q4 < 2) {
            const int i = 32 * q4 + lane;
            float da[16], bm[16];
            tmem_ld16(tm + lb + SL2 + c16, da);
            tmem_ld16(tm + lb + SL4 + c16, bm);
            tmem_ld_wait();
            const float gi = sGam[i], bi = sBeta[i], ei = sE[i];
            float dm[16];  // D_ij = exp(gamma_i - gamma_j)
            if (*sPw) {
                const F16 r = decay_row_direct(gi, sGam + c16);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) dm[jj] = r.v[jj];
            } else {
#pragma unroll
                for (int jj = 0; jj < 16; jj += 4) {
                    const float4 e4 = *reinterpret_cast<const float4*>(sEi + c16 + jj);
                    dm[jj] = ei * e4.x;
                    dm[jj + 1] = ei * e4.y;
                    dm[jj + 2] = ei * e4.z;
                    dm[jj + 3] = ei * e4.w;
                }
            }
            float rs = 0.f, ra = 0.f;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int jx = c16 + jj;
                const bool strict = i > jx;
                const float D = strict ? dm[jj] : 0.f;
                const float dav = strict ? -da[jj] : 0.f;
                const float fdb = D * bm[jj];
                rs += dav * fdb;
                const float aa = dav * bi * fdb;
                ra += aa;
                da[jj] = bi * dav * D;
                bm[jj] = aa;
            }
            sF[F_PRS + 64 * cg + i] = rs;
            sF[F_PAR + 64 * cg + i] = ra;
            const float cs = lane_colsum16(bm);
            if (!(lane & 1)) sF[F_PAC + 64 * q4 + c16 + (lane >> 1)] = cs;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t ch = uint32_t((4 * cg + u) ^ (i & 15));
                sts128(aSTG + uint32_t(i) * 256u + ch * 16u,
                       make_uint4(__float_as_uint(da[4 * u]), __float_as_uint(da[4 * u + 1]),
                                  __float_as_uint(da[4 * u + 2]), __float_as_uint(da[4 * u + 3])));
            }
            named_sync(2, LT / 2);  // the warps of lane quarters 0 and 1
            float s2[16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t ch = uint32_t((4 * cg + u) ^ (i & 15));
                const float4 own = lds128f(aSTG + uint32_t(i) * 256u + ch * 16u);
                s2[4 * u] = own.x;
                s2[4 * u + 1] = own.y;
                s2[4 * u + 2] = own.z;
                s2[4 * u + 3] = own.w;
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int jx = c16 + jj;
                s2[jj] += lds32f(aSTG + uint32_t(jx) * 256u + (uint32_t((i >> 2) ^ (jx & 15)) << 4) +
                                 uint32_t(i & 3) * 4u);
            }
            st_row16(aDT, i, c16, s2);
        } else if (w == 6 || w == 7) {
            // every per-token term but those of dA, in place (thread i reads its own entries
            // before writing them): F_PQ[i] dgamma so far, F_PQ[64 + i] dbeta so far,
            // F_PQ[128 + i] r_i; F_RED[8] = <dh, h>
            const int i = tid - 192;
            float pq = 0.f, pr = 0.f, ptw = 0.f, ptu = 0.f, ppr = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                pq += sF[F_PQ + 64 * q + i];
                pr += sF[F_PR + 64 * q + i];
                ptw += sF[F_PTW + 64 * q + i];
                ptu += sF[F_PTU + 64 * q + i];
                ppr += sF[F_PPR + 64 * q + i];
            }
            const float ri = sKd[i] * pr;
            sF[F_PQ + i] = ppr - (sF[F_PPC + i] + sF[F_PPC + 64 + i]) + sc * sE[i] * pq - ri + sBe[i] * ptw;
            sF[F_PQ + 64 + i] = sE[i] * ptw + ptu;
            sF[F_PQ + 128 + i] = ri;
            if (i == 0) {
                float hd = 0.f;
#pragma unroll
                for (int q = 0; q < 7; ++q) hd += sF[F_RED + q];
                sF[F_RED + 8] = hd;
            }
        }
        fence_proxy_async_smem();
        fence_before_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        TTRACE(16);
        if (tid == ISS) {
            ITRACE(14);
            fence_after_sync();
            // ((dB + dB^T) K)^T = K^T (dB + dB^T) onto (dQk^T Q)^T
#pragma unroll
            for (int s = 0; s < 4; ++s) mma_bf16(tm + sv, dM_(aK, 8192, s), dM_(aDT, 8192, s), ID_MM, 1u);
            commit(&bars[M_9]);
            if (has_next) req_T(nxt);  // T is no longer read
            ITRACE(15);
        }
        __syncwarp();

        // dK = dQk^T Q + (dB + dB^T) K + diag(kd) (V' dh^T) + diag(beta e) dYW
        ok = lwait(bars, M_9, par, errflag) && ok;
        TTRACE(17);
        fence_after_sync();
        if (tid == ISS && ok && has_next) req_Q(nxt, kreg);  // the last product has read K
        have_ng = false;
        if (w == 0 && has_next) {  // the next item's gates, in flight during the epilogue
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                const bool in = r < nxt.c;
                ngv[u] = in ? P.g[(nxt.tc + r) * Hv + nxt.j] : 0.f;
                nbv[u] = in ? P.beta[(nxt.tc + r) * Hv + nxt.j] : 0.f;
            }
            have_ng = true;
        }
        {
            float x[16], y[16], z[16];
            tmem_ld16(tm + lb + sv + c16, x);
            tmem_ld16(tm + lb + SL5 + c16, y);
            tmem_ld16(tm + lb + sa + c16, z);
            tmem_ld_wait();
            const int k = 32 * q4 + lane;
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                const int cx = c16 + ii;
                x[ii] += sKd[cx] * y[ii] + sBe[cx] * z[ii];
            }
            if (PART) {
                float* dk = B.dkp + int64_t(j) * KD + k;
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    const int cx = c16 + ii;
                    if (cx < c && in_range(int64_t(j) * KD + k + (tc + cx) * Hv * KD, T_all * Hv * KD, P.err))
                        dk[(tc + cx) * Hv * KD] = x[ii];
                }
            } else if (tile_out) {  // staged in the dB staging region (the dA step is done with it)
#pragma unroll
                for (int ii = 0; ii < 16; ++ii)
                    sts16(aSTG + out_tile_off(c16 + ii, k), __bfloat16_as_ushort(__float2bfloat16_rn(x[ii])));
                fence_proxy_async_smem();
            } else {
                F16 o;
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) o.v[ii] = x[ii];
                st_col_bf16(reinterpret_cast<__nv_bfloat16*>(B.dk) + int64_t(qh) * KD + k + (tc + c16) * qk_stride,
                            qk_stride, o, c - c16, int64_t(qh) * KD + k + (tc + c16) * qk_stride, T_all * qk_stride,
                            P.err);
            }
        }
        // per-token totals (warp 0, rows 2 lane and 2 lane + 1), then dg = reverse in-chunk
        // cumsum of dgamma, and dbeta
        if (w == 0) {
            float dgv[2], dbv[2], rr = 0.f;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = 2 * lane + u;
                float par4 = 0.f, prs = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    par4 += sF[F_PAR + 64 * q + i];
                    prs += sF[F_PRS + 64 * q + i];
                }
                rr += sF[F_PQ + 128 + i];
                dgv[u] = sF[F_PQ + i] + par4 - (sF[F_PAC + i] + sF[F_PAC + 64 + i]);
                dbv[u] = sF[F_PQ + 64 + i] + prs;
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) rr += __shfl_xor_sync(0xffffffffu, rr, off);
            if (lane == 31) dgv[1] += rr + sE[LCH - 1] * sF[F_RED + 8];
            const float v1 = dgv[1], v0 = dgv[0] + dgv[1];
            float tot = v0;  // suffix scan over lanes (from the top)
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, tot, off);
                if (lane + off < 32) tot += y;
            }
            const float excl = tot - v0;
            const float vals[2] = {v0 + excl, v1 + excl};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int r = 2 * lane + u;
                if (r < c && in_range((tc + r) * Hv + j, T_all * Hv, P.err)) {
                    B.dg[(tc + r) * Hv + j] = vals[u];
                    B.dbeta[(tc + r) * Hv + j] = dbv[u];
                }
            }
        }
        // end of the item: the issuer's warp only signals its arrival (its dK share is done) and
        // issues the next item's second group (s2 and s4 were read by the dA epilogue) while
        // the others finish; the next item's first barrier takes it in again
        fence_before_sync();
        if (w == ISS / 32) {
            named_arrive(3, LT);
            if (tid == ISS && nA && landed(par ^ 1u, false, 0)) {
                issue_B(par ^ 1u);
                nB = true;
            }
            __syncwarp();
        } else {
            named_sync(3, LT);
            if (tid == 0 && tile_out && !PART) {
                tma_store_3d(&maps.dk, sm + L_STG, 0, qh, int(tc));
                tma_store_3d(&maps.dk, sm + L_STG + 8192, 64, qh, int(tc));
                bulk_commit();
            }
        }
        carry_ok = ok;
        TTRACE(18);
        pre = has_next;
        eA = nA;
        eB = nB;
        ++n;
    }

    if (tid == 0) bulk_wait0();  // the last tile stores have completed
    if (!failed && __syncthreads_or(!carry_ok)) failed = true;
    if (failed && tid == ISS) {
        // let the copies in flight land and the products drain before the CTA leaves
#pragma unroll
        for (int b = 0; b < NLD; ++b)
            if (ldn[b] > 0) mbar_wait(&bars[b], uint32_t(ldn[b] - 1) & 1u);
        commit(&bars[M_DRAIN]);
        mbar_wait(&bars[M_DRAIN], 0);
        if (P.err) atomicOr(P.err, *errflag | (1 << 26));
    }
    fence_before_sync();
    __syncthreads();
    if (w == 0) {
        fence_after_sync();
        tmem_dealloc(tm, 512);
    }
}

}  // namespace

#ifdef GDN_TRACE
extern "C" int gdn_debug_tcl_trace(unsigned long long* out) {
    return int(cudaMemcpyFromSymbol(out, g_tcl_trace, sizeof(g_tcl_trace)));
}
#endif

cudaError_t launch_bwd_local_tc(const BwdProblem& B, int64_t T_total, cudaStream_t st) {
    const Problem& P = B.f;
    if (P.total_chunks <= 0) return cudaSuccess;
    // the chunk records must carry T, and the states of every chunk must be there
    if (P.prep_stride < PREP_BWD_BYTES || !P.prep || !P.hist || !B.dhist) return cudaErrorInvalidValue;
    LocMaps maps;
    const int64_t rows = int64_t(P.total_chunks) * P.Hv * KD;
    // the per-chunk state rows are addressed by 32-bit TMA coordinates
    if (rows > int64_t(0x7fffffff) - KD) return cudaErrorNotSupported;
    if (!make_map(&maps.k, P.k, P.Hqk, T_total) || !make_map(&maps.q, P.q, P.Hqk, T_total) ||
        !make_map(&maps.v, P.v, P.Hv, T_total) || !make_map(&maps.dO, B.dO, P.Hv, T_total) ||
        !make_rows_map(&maps.h, P.hist, rows) || !make_rows_map(&maps.dh, B.dhist, rows) ||
        !make_map(&maps.dv, B.dv, P.Hv, T_total) || (!B.dqp && !make_map(&maps.dq, B.dq, P.Hqk, T_total)) ||
        (!B.dkp && !make_map(&maps.dk, B.dk, P.Hqk, T_total)))
        return cudaErrorInvalidValue;
    const bool part = B.dqp != nullptr;  // (B.dkp with it: both when Hv != Hqk)
    if (part != (B.dkp != nullptr)) return cudaErrorInvalidValue;
    cudaError_t e = part ? smem_attr(k_tc_bwd_local<true>, int(LOC_SMEM)) : smem_attr(k_tc_bwd_local<false>, int(LOC_SMEM));
    if (e != cudaSuccess) return e;
    const int64_t items = int64_t(P.total_chunks) * P.Hv;
    const int grid = int(items < int64_t(sm_count()) ? items : int64_t(sm_count()));  // persistent
    return part ? launch_pdl(k_tc_bwd_local<true>, dim3(grid), dim3(LT), LOC_SMEM, st, B, maps, items)
                : launch_pdl(k_tc_bwd_local<false>, dim3(grid), dim3(LT), LOC_SMEM, st, B, maps, items);
}

}  // namespace gdn
