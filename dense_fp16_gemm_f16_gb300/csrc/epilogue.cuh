// epilogue.cuh -- element types and the fused output transform.
//
// The kernels run for fp16 or bf16 operands (same tcgen05 kind::f16 MMA with
// an fp32 accumulator; only the operand format bits of the instruction
// descriptor differ) and write D in the operand type, rounded to nearest even.
//
// The optional fused epilogue computes, in fp32 and before that single
// rounding,   D = act(alpha * (A B^T) + beta * C + bias[n])
// -- the scaled update C = alpha A B + beta C of the GEMM blog post (section
// 2.1) with the bias and activation fusion it recommends (section 5.4), and
// the "epilogue fusion" the Croqtile tutorial credits cuBLAS with in its
// comparison section.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

namespace gemm_gb300 {

struct EpiParams {
    float alpha;
    float beta;
    const void* C;      // [M][N] like D, or nullptr
    const void* bias;   // [N], or nullptr
    int32_t act;        // 0 none, 1 relu
    int32_t on;         // 0: plain D = A B^T (the other fields are ignored)
};

template <class T>
struct Elem;

template <>
struct Elem<__half> {
    static constexpr uint32_t kFormat = 0;   // instruction-descriptor A/B format: f16
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        const __half2 x = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&x);
    }
    __device__ __forceinline__ static __half from_float(float v) { return __float2half_rn(v); }
    __device__ __forceinline__ static float lo(uint32_t w) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
    }
    __device__ __forceinline__ static float hi(uint32_t w) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
    }
    __device__ __forceinline__ static float to_float(__half v) { return __half2float(v); }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr uint32_t kFormat = 1;   // instruction-descriptor A/B format: bf16
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        const __nv_bfloat162 x = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&x);
    }
    __device__ __forceinline__ static __nv_bfloat16 from_float(float v) { return __float2bfloat16_rn(v); }
    // a bf16 value is the top 16 bits of the fp32 with the same value
    __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
    __device__ __forceinline__ static float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
};

// Applies the fused transform to 8 consecutive columns [col, col + 8) of one
// output row; col is a multiple of 8 (N % 8 == 0 keeps the 16-byte loads in
// bounds and aligned).  Rows at or past M read no C.
template <class T>
__device__ __forceinline__ void epi_apply8(const EpiParams& e, float (&x)[8], int64_t row, int64_t col,
                                           int64_t M, int64_t N) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] *= e.alpha;
    if (e.C != nullptr && e.beta != 0.0f && row < M) {
        const uint4 c = *reinterpret_cast<const uint4*>(static_cast<const T*>(e.C) + row * N + col);
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] += e.beta * Elem<T>::lo(w[i]);
            x[2 * i + 1] += e.beta * Elem<T>::hi(w[i]);
        }
    }
    if (e.bias != nullptr) {
        const uint4 b = *reinterpret_cast<const uint4*>(static_cast<const T*>(e.bias) + col);
        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] += Elem<T>::lo(w[i]);
            x[2 * i + 1] += Elem<T>::hi(w[i]);
        }
    }
    if (e.act == 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = x[i] < 0.0f ? 0.0f : x[i];   // relu; NaN and -0 pass
    }
}

// The same transform for one element (the small-M kernel writes D one
// element at a time).
template <class T>
__device__ __forceinline__ float epi_apply1(const EpiParams& e, float x, int64_t row, int64_t col, int64_t N) {
    x *= e.alpha;
    if (e.C != nullptr && e.beta != 0.0f) x += e.beta * Elem<T>::to_float(static_cast<const T*>(e.C)[row * N + col]);
    if (e.bias != nullptr) x += Elem<T>::to_float(static_cast<const T*>(e.bias)[col]);
    if (e.act == 1) x = x < 0.0f ? 0.0f : x;
    return x;
}

}  // namespace gemm_gb300
