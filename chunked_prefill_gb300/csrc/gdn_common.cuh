// Shared device helpers of the GDN kernels: warp-level tensor-core tiles (mma.sync
// m16n8k16 bf16 -> fp32) with ldmatrix operand loads, and an fp32 SIMT twin with the same
// accumulator layout for the fp32 test mode.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int KD = 128;  // key dim
constexpr int VD = 128;  // value dim

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t& r0, uint32_t& r1, const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(p)));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Warp tile product acc[n] += A[m0:m0+16, 0:kdim] * B[0:kdim, n0+8n : n0+8n+8], n < NT.
//   A(m,k) = A_COL ? A[k*lda + m] : A[m*lda + k]
//   B(k,n) = B_NK  ? B[n*ldb + k] : B[k*ldb + n]
// Accumulator layout (the mma.sync m16n8 C layout): lane = 4*g + t holds
//   acc[n][0] = (m0+g,   n0+8n+2t), acc[n][1] = (m0+g,   n0+8n+2t+1),
//   acc[n][2] = (m0+g+8, n0+8n+2t), acc[n][3] = (m0+g+8, n0+8n+2t+1).
template <int NT, bool A_COL, bool B_NK>
__device__ __forceinline__ void warp_mma(float (&acc)[NT][4], const __nv_bfloat16* A, int lda,
                                         const __nv_bfloat16* B, int ldb, int m0, int n0,
                                         int kdim) {
    const int lane = threadIdx.x & 31;
    const int r8 = lane & 7, b1 = (lane >> 3) & 1, b2 = lane >> 4;
#pragma unroll 2
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        uint32_t a[4];
        if (!A_COL)
            ldsm_x4(a, A + (m0 + r8 + b1 * 8) * lda + k0 + b2 * 8);
        else
            ldsm_x4_t(a, A + (k0 + r8 + b2 * 8) * lda + m0 + b1 * 8);
#pragma unroll
        for (int n = 0; n + 1 < NT; n += 2) {
            uint32_t b[4];
            if (B_NK)
                ldsm_x4(b, B + (n0 + n * 8 + r8 + b2 * 8) * ldb + k0 + b1 * 8);
            else
                ldsm_x4_t(b, B + (k0 + r8 + b1 * 8) * ldb + n0 + n * 8 + b2 * 8);
            mma_bf16(acc[n], a, b[0], b[1]);
            mma_bf16(acc[n + 1], a, b[2], b[3]);
        }
        if (NT & 1) {
            constexpr int n = NT - 1;
            uint32_t x0, x1;
            if (B_NK)
                ldsm_x2(x0, x1, B + (n0 + n * 8 + r8) * ldb + k0 + b1 * 8);
            else
                ldsm_x2_t(x0, x1, B + (k0 + r8 + b1 * 8) * ldb + n0 + n * 8);
            mma_bf16(acc[n], a, x0, x1);
        }
    }
}

// fp32 SIMT twin with the identical accumulator layout (fp32 test mode).
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

// 16-byte asynchronous global -> shared copy (zero fill when !valid; src must still be a
// valid address), committed and awaited in groups by the issuing thread
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(sdst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(gsrc), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

}  // namespace gdn
