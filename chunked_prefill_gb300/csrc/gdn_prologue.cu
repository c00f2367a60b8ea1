// Fused prologue of the gated delta rule: the activations that turn a layer's raw
// projections into the method's inputs, in one pass over HBM, and their reverse mode.
//
// The FlashQLA pages take q, k, g and beta as given (agentlenshq "GDN chunked prefill
// optimisation": g is a log-decay, beta a write strength, q and k unit-norm keys of the
// delta rule) and do not say how a model forms them.  This file takes the plainest reading
// consistent with those roles:
//   q = q_raw / sqrt(|q_raw|^2 + eps),  k likewise (eps = 1e-6; per token and q/k head)
//   g = -exp(A_log[j]) * softplus(a + dt_bias[j])     (g <= 0; per token and v-head j)
//   beta = sigmoid(b)                                  (0 < beta < 1)
// Reverse mode, with n = sqrt(|x|^2 + eps) and y = x / n:
//   dx = (dy - y <y, dy>) / n
//   da = dg * (-exp(A_log)) * sigmoid(a + dt_bias);  ddt_bias = sum_t da
//   dA_log = sum_t dg * g;  db = dbeta * beta (1 - beta)
// The two sums over tokens are taken in a fixed order (partial sums over fixed token ranges,
// then a fixed-shape tree over the ranges), so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_internal.h"

namespace gdn {
namespace {

constexpr float PRO_EPS = 1e-6f;
constexpr int PRO_T = 256;         // threads per block
constexpr int PRO_SPLITS = 1024;   // partial sums per head in the backward reduction

__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// 4 consecutive elements of a 128-wide row per lane
template <typename Op> struct Vec4;
template <> struct Vec4<float> {
    static __device__ __forceinline__ void load(const float* p, float (&x)[4]) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    static __device__ __forceinline__ void store(float* p, const float (&x)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};
template <> struct Vec4<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[4]) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[4]) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 v;
        v.x = *reinterpret_cast<const uint32_t*>(&a);
        v.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = v;
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Rows: one warp per (token, q/k head) row pair (the q row and the k row), RPW pairs in
// flight per warp.  Gates: the remaining work of the grid-stride loop, one element per thread.
template <typename Op, int RPW>
__global__ void __launch_bounds__(PRO_T) k_prologue_fwd(const Op* qr, const Op* kr, Op* q, Op* k,
                                                        int64_t rows, const float* a, const float* b,
                                                        const float* A_log, const float* dt_bias,
                                                        float* g, float* beta, int64_t gates, int Hv) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * PRO_T + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * PRO_T) >> 5;
    for (int64_t r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
        float xq[RPW][4], xk[RPW][4];
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
            if (r0 + u < rows) {
                Vec4<Op>::load(qr + (r0 + u) * 128 + 4 * lane, xq[u]);
                Vec4<Op>::load(kr + (r0 + u) * 128 + 4 * lane, xk[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
            if (r0 + u >= rows) break;
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sq = fmaf(xq[u][e], xq[u][e], sq);
                sk = fmaf(xk[u][e], xk[u][e], sk);
            }
            const float iq = rsqrtf(warp_sum(sq) + PRO_EPS), ik = rsqrtf(warp_sum(sk) + PRO_EPS);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                xq[u][e] *= iq;
                xk[u][e] *= ik;
            }
            Vec4<Op>::store(q + (r0 + u) * 128 + 4 * lane, xq[u]);
            Vec4<Op>::store(k + (r0 + u) * 128 + 4 * lane, xk[u]);
        }
    }
    const int64_t tid = int64_t(blockIdx.x) * PRO_T + threadIdx.x, nth = int64_t(gridDim.x) * PRO_T;
    for (int64_t i = tid; i < gates; i += nth) {
        const int j = int(i % Hv);
        g[i] = -expf(A_log[j]) * softplus_f(a[i] + dt_bias[j]);
        beta[i] = sigmoid_f(b[i]);
    }
}

template <typename Op, int RPW>
__global__ void __launch_bounds__(PRO_T) k_prologue_bwd(const Op* qr, const Op* kr, const Op* dq, const Op* dk,
                                                        Op* dqr, Op* dkr, int64_t rows, const float* a,
                                                        const float* b, const float* A_log,
                                                        const float* dt_bias, const float* dg,
                                                        const float* dbeta, float* da, float* db,
                                                        int64_t gates, int Hv) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t(blockIdx.x) * PRO_T + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t(gridDim.x) * PRO_T) >> 5;
    for (int64_t r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
        // every load of the iteration in flight before the first reduction
        float x[RPW][2][4], d[RPW][2][4];
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
            if (r0 + u < rows) {
                const int64_t o = (r0 + u) * 128 + 4 * lane;
                Vec4<Op>::load(qr + o, x[u][0]);
                Vec4<Op>::load(kr + o, x[u][1]);
                Vec4<Op>::load(dq + o, d[u][0]);
                Vec4<Op>::load(dk + o, d[u][1]);
            }
        }
#pragma unroll
        for (int u = 0; u < RPW; ++u) {
            const int64_t r = r0 + u;
            if (r >= rows) break;
#pragma unroll
            for (int which = 0; which < 2; ++which) {
                float s = 0.f, t = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    s = fmaf(x[u][which][e], x[u][which][e], s);
                    t = fmaf(x[u][which][e], d[u][which][e], t);
                }
                const float in = rsqrtf(warp_sum(s) + PRO_EPS);
                const float ydy = warp_sum(t) * in;  // <y, dy>
                float o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) o4[e] = (d[u][which][e] - x[u][which][e] * in * ydy) * in;
                Vec4<Op>::store((which ? dkr : dqr) + r * 128 + 4 * lane, o4);
            }
        }
    }
    const int64_t tid = int64_t(blockIdx.x) * PRO_T + threadIdx.x, nth = int64_t(gridDim.x) * PRO_T;
    for (int64_t i = tid; i < gates; i += nth) {
        const int j = int(i % Hv);
        da[i] = -dg[i] * expf(A_log[j]) * sigmoid_f(a[i] + dt_bias[j]);
        const float bt = sigmoid_f(b[i]);
        db[i] = dbeta[i] * bt * (1.f - bt);
    }
}

// Per (split, head) partial sums of dA_log = sum_t dg g and ddt_bias = sum_t da over the
// split's contiguous token range, in a fixed order.  Heads are taken in tiles of HT =
// min(Hv, 256); a tile is read as R = 256 / HT consecutive token rows per step (coalesced),
// thread t accumulating head t % HT of row t / HT, and the R row partials of each head are
// then added in row order.
__global__ void __launch_bounds__(PRO_T) k_prologue_part(const float* a, const float* A_log,
                                                         const float* dt_bias, const float* dg,
                                                         const float* da, int64_t T_total, int Hv,
                                                         float* part) {
    __shared__ float red[2][PRO_T];
    const int sp = blockIdx.x, tid = threadIdx.x;
    const int64_t per = (T_total + PRO_SPLITS - 1) / PRO_SPLITS;
    const int64_t t0 = per * sp, t1 = t0 + per < T_total ? t0 + per : T_total;
    const int HT = Hv < PRO_T ? Hv : PRO_T, R = PRO_T / HT;
    for (int jb = 0; jb < Hv; jb += HT) {
        const int r = tid / HT, j = jb + tid % HT;
        float sA = 0.f, sB = 0.f;
        if (r < R && j < Hv) {
            const float ea = expf(A_log[j]), bias = dt_bias[j];
#pragma unroll 4
            for (int64_t t = t0 + r; t < t1; t += R) {
                const int64_t i = t * Hv + j;
                sA = fmaf(dg[i], -ea * softplus_f(a[i] + bias), sA);
                sB += da[i];
            }
        }
        red[0][tid] = sA;
        red[1][tid] = sB;
        __syncthreads();
        if (tid < HT && jb + tid < Hv) {
            float uA = 0.f, uB = 0.f;
            for (int q = 0; q < R; ++q) {
                uA += red[0][q * HT + tid];
                uB += red[1][q * HT + tid];
            }
            part[(int64_t(sp) * Hv + jb + tid) * 2] = uA;
            part[(int64_t(sp) * Hv + jb + tid) * 2 + 1] = uB;
        }
        __syncthreads();
    }
}

// One block per head: thread s holds split s, then a fixed-shape tree over the splits.
__global__ void __launch_bounds__(PRO_SPLITS) k_prologue_sum(const float* part, int Hv, float* dA_log,
                                                             float* ddt_bias) {
    __shared__ float red[2][PRO_SPLITS];
    const int j = blockIdx.x, sp = threadIdx.x;
    red[0][sp] = part[(int64_t(sp) * Hv + j) * 2];
    red[1][sp] = part[(int64_t(sp) * Hv + j) * 2 + 1];
    __syncthreads();
    for (int o = PRO_SPLITS / 2; o > 0; o >>= 1) {
        if (sp < o) {
            red[0][sp] += red[0][sp + o];
            red[1][sp] += red[1][sp + o];
        }
        __syncthreads();
    }
    if (sp == 0) {
        dA_log[j] = red[0][0];
        ddt_bias[j] = red[1][0];
    }
}

int pro_blocks(int64_t rows, int64_t gates, int rpw) {
    const int64_t want = (rows + rpw * (PRO_T / 32) - 1) / (rpw * (PRO_T / 32));
    const int64_t want_g = (gates + PRO_T - 1) / PRO_T;
    const int64_t cap = int64_t(sm_count()) * 8;  // 8 resident blocks of 256 threads per SM
    int64_t n = want > want_g ? want : want_g;
    if (n > cap) n = cap;
    return int(n < 1 ? 1 : n);
}

}  // namespace

size_t prologue_bwd_workspace(int Hv) { return size_t(Hv) * PRO_SPLITS * 2 * sizeof(float); }

cudaError_t launch_prologue_fwd(const PrologueArgs& A, cudaStream_t st) {
    constexpr int RPW = 2;
    const int nb = pro_blocks(A.rows, A.gates, RPW);
    timing_begin("prologue_fwd", st);
    if (A.dtype == 0)
        k_prologue_fwd<__nv_bfloat16, RPW><<<nb, PRO_T, 0, st>>>(
            static_cast<const __nv_bfloat16*>(A.q_raw), static_cast<const __nv_bfloat16*>(A.k_raw),
            static_cast<__nv_bfloat16*>(A.q), static_cast<__nv_bfloat16*>(A.k), A.rows, A.a, A.b,
            A.A_log, A.dt_bias, A.g, A.beta, A.gates, A.Hv);
    else
        k_prologue_fwd<float, RPW><<<nb, PRO_T, 0, st>>>(
            static_cast<const float*>(A.q_raw), static_cast<const float*>(A.k_raw),
            static_cast<float*>(A.q), static_cast<float*>(A.k), A.rows, A.a, A.b, A.A_log,
            A.dt_bias, A.g, A.beta, A.gates, A.Hv);
    timing_end(st);
    return cudaGetLastError();
}

cudaError_t launch_prologue_bwd(const PrologueArgs& A, cudaStream_t st) {
    constexpr int RPW = 2;
    const int nb = pro_blocks(A.rows, A.gates, RPW);
    timing_begin("prologue_bwd", st);
    if (A.dtype == 0)
        k_prologue_bwd<__nv_bfloat16, RPW><<<nb, PRO_T, 0, st>>>(
            static_cast<const __nv_bfloat16*>(A.q_raw), static_cast<const __nv_bfloat16*>(A.k_raw),
            static_cast<const __nv_bfloat16*>(A.dq), static_cast<const __nv_bfloat16*>(A.dk),
            static_cast<__nv_bfloat16*>(A.dq_raw), static_cast<__nv_bfloat16*>(A.dk_raw), A.rows,
            A.a, A.b, A.A_log, A.dt_bias, A.dg, A.dbeta, A.da, A.db, A.gates, A.Hv);
    else
        k_prologue_bwd<float, RPW><<<nb, PRO_T, 0, st>>>(
            static_cast<const float*>(A.q_raw), static_cast<const float*>(A.k_raw),
            static_cast<const float*>(A.dq), static_cast<const float*>(A.dk),
            static_cast<float*>(A.dq_raw), static_cast<float*>(A.dk_raw), A.rows, A.a, A.b,
            A.A_log, A.dt_bias, A.dg, A.dbeta, A.da, A.db, A.gates, A.Hv);
    timing_end(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    timing_begin("prologue_bwd_sum", st);
    k_prologue_part<<<PRO_SPLITS, PRO_T, 0, st>>>(A.a, A.A_log, A.dt_bias, A.dg, A.da,
                                                               A.gates / A.Hv, A.Hv, A.part);
    k_prologue_sum<<<A.Hv, PRO_SPLITS, 0, st>>>(A.part, A.Hv, A.dA_log, A.ddt_bias);
    timing_end(st);
    return cudaGetLastError();
}

}  // namespace gdn
