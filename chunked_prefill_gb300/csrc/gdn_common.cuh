// Shared device helpers of the GDN kernels: bf16 / fp32 conversions and the fp32 warp-tile
// product of the CUDA-core kernels that serve the fp32 test mode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int KD = 128;  // key dim
constexpr int VD = 128;  // value dim

// Checked builds (compiled with -DGDN_CHECK): an output store first tests its element index
// against the extent of the tensor it writes; an index outside [0, n) sets ERR_BOUNDS in the
// call's error word and the store is skipped.  Release builds compile the test away.
constexpr int ERR_BOUNDS = int(0x80000000u);
#ifdef GDN_CHECK
__device__ __forceinline__ bool in_range(int64_t i, int64_t n, int* err) {
    if (i >= 0 && i < n) return true;
    if (err) atomicOr(err, ERR_BOUNDS);
    return false;
}
#else
__device__ __forceinline__ bool in_range(int64_t, int64_t, int*) { return true; }
#endif

template <typename Op> struct OpTraits;
template <> struct OpTraits<__nv_bfloat16> {
    static constexpr int PAD = 8;  // 16 bytes: ldmatrix rows land on distinct banks
};
template <> struct OpTraits<float> {
    static constexpr int PAD = 4;
};

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
template <typename Op> __device__ __forceinline__ Op from_f(float x);
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }

// store two consecutive values
__device__ __forceinline__ void st2(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ void st2(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
}

// Warp tile product acc[n] += A[m0:m0+16, 0:kdim] * B[0:kdim, n0+8n : n0+8n+8], n < NT, on
// the CUDA cores (the fp32 test-mode kernels):
//   A(m,k) = A_COL ? A[k*lda + m] : A[m*lda + k]
//   B(k,n) = B_NK  ? B[n*ldb + k] : B[k*ldb + n]
// Accumulator layout (that of the m16n8 tensor-core fragment, so the callers' epilogues index
// it the same way): lane = 4*g + t holds
//   acc[n][0] = (m0+g,   n0+8n+2t), acc[n][1] = (m0+g,   n0+8n+2t+1),
//   acc[n][2] = (m0+g+8, n0+8n+2t), acc[n][3] = (m0+g+8, n0+8n+2t+1).
template <int NT, bool A_COL, bool B_NK>
__device__ __forceinline__ void warp_mma(float (&acc)[NT][4], const float* A, int lda,
                                         const float* B, int ldb, int m0, int n0, int kdim) {
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    for (int k = 0; k < kdim; ++k) {
        const float alo = A_COL ? A[k * lda + m0 + g] : A[(m0 + g) * lda + k];
        const float ahi = A_COL ? A[k * lda + m0 + g + 8] : A[(m0 + g + 8) * lda + k];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int c = n0 + n * 8 + 2 * t;
            const float b0 = B_NK ? B[c * ldb + k] : B[k * ldb + c];
            const float b1 = B_NK ? B[(c + 1) * ldb + k] : B[k * ldb + c + 1];
            acc[n][0] = fmaf(alo, b0, acc[n][0]);
            acc[n][1] = fmaf(alo, b1, acc[n][1]);
            acc[n][2] = fmaf(ahi, b0, acc[n][2]);
            acc[n][3] = fmaf(ahi, b1, acc[n][3]);
        }
    }
}

template <int NT>
__device__ __forceinline__ void zero_acc(float (&acc)[NT][4]) {
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
}

}  // namespace gdn
