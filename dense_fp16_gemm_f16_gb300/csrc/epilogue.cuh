// epilogue.cuh -- element types and the fused output transform.
//
// The kernels run for fp16 or bf16 operands (tcgen05 kind::f16) and for
// E4M3 or E5M2 operands (kind::f8f6f4), always with an fp32 accumulator; the
// operand format is a field of the instruction descriptor.  D is written in
// the operand type for 16-bit operands and in bf16 for 8-bit ones, rounded to
// nearest even.
//
// The optional fused epilogue computes, in fp32 and before that single
// rounding,   D = act(alpha * s[n] * (A B^T) + beta * C + bias[n])
// -- the scaled update C = alpha A B + beta C of the GEMM blog post (section
// 2.1) with the bias and activation fusion it recommends (section 5.4), and
// the "epilogue fusion" the Croqtile tutorial credits cuBLAS with in its
// comparison section.  s[n] is an optional fp32 scale per output column: the
// per-channel weight scale of the blog post's 8-bit quantisation (section
// 4.2), with the per-tensor activation scale folded into alpha.
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
    const float* scale_n;  // [N] fp32, or nullptr
    int32_t act;        // 0 none, 1 relu
    int32_t on;         // 0: plain D = A B^T (the other fields are ignored)
};

template <class T>
struct Elem;

template <>
struct Elem<__half> {
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

// The 8 C values at [row][col, col + 8) as one 16-byte load (zero when C is
// not read or the row is past M).  col is a multiple of 8 (N % 8 == 0 keeps
// the load in bounds and aligned).  Issued ahead of its use, its latency
// hides behind the TMEM reads.
template <class T>
__device__ __forceinline__ uint4 epi_load_c8(const EpiParams& e, int64_t row, int64_t col, int64_t M, int64_t N) {
    if (e.C == nullptr || e.beta == 0.0f || row >= M) return make_uint4(0u, 0u, 0u, 0u);
    return *reinterpret_cast<const uint4*>(static_cast<const T*>(e.C) + row * N + col);
}

// Applies the fused transform to 8 consecutive columns [col, col + 8) of one
// output row, given that row's C values from epi_load_c8.
template <class T>
__device__ __forceinline__ void epi_apply8_c(const EpiParams& e, float (&x)[8], uint4 c, int64_t col) {
    if (e.scale_n != nullptr) {
        const float4 s0 = *reinterpret_cast<const float4*>(e.scale_n + col);
        const float4 s1 = *reinterpret_cast<const float4*>(e.scale_n + col + 4);
        const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= e.alpha * s[i];
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= e.alpha;
    }
    if (e.C != nullptr && e.beta != 0.0f) {
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

// The per-column scale and bias of the 64 columns [col0, col0 + 64) that a
// warp of the tiled epilogue writes: lane l fetches columns col0 + 2l and
// col0 + 2l + 1 with one coalesced access per vector.  The tiled epilogue
// fetches them for a whole unit before it waits for the unit's accumulator,
// and stages each chunk's values in shared memory, from where every lane reads
// them as broadcasts (epi_apply8_s).  Measured on GB300 against the other ways
// tried, for a 256-column tile: fetching them per 8-column group after the TMEM
// reads put a global-memory round trip on every group (9.2 us per tile);
// handing them out by warp shuffles cost ~3000 cycles per 64-column chunk
// (8 us); the plain epilogue takes 3.4 us.
template <class T>
struct EpiCols64 {
    float2 s;     // alpha * scale_n of the two columns (alpha when there is no scale_n)
    uint32_t b;   // bias of the two columns, packed (0 when there is none)
    __device__ __forceinline__ void load(const EpiParams& e, int64_t col0, int lane, int64_t N) {
        const int64_t c = col0 + 2 * lane;
        const bool in = c < N;   // N % 8 == 0: both columns are in or both out
        s = make_float2(e.alpha, e.alpha);
        if (e.scale_n != nullptr && in) {
            const float2 v = *reinterpret_cast<const float2*>(e.scale_n + c);
            s = make_float2(e.alpha * v.x, e.alpha * v.y);
        }
        b = (e.bias != nullptr && in) ? *reinterpret_cast<const uint32_t*>(static_cast<const T*>(e.bias) + c) : 0u;
    }
    // this lane's share into the warp's staging area: 64 fp32 factors, then 64 bias values
    __device__ __forceinline__ void stage(uint8_t* area, int lane) const {
        reinterpret_cast<float2*>(area)[lane] = s;
        reinterpret_cast<uint32_t*>(area + 256)[lane] = b;
    }
};

// epi_apply8_c for the 8 columns [8j, 8j + 8) of a warp's 64-column chunk,
// with the chunk's factors alpha * s[n] and bias staged by EpiCols64::stage
// (`area`) and its C values from epi_load_c8 (used only when use_c).
template <class T>
__device__ __forceinline__ void epi_apply8_s(const EpiParams& e, float (&x)[8], uint4 c, bool use_c,
                                             const uint8_t* area, int j) {
    {
        const float4 s0 = reinterpret_cast<const float4*>(area)[2 * j];
        const float4 s1 = reinterpret_cast<const float4*>(area)[2 * j + 1];
        const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] *= sc[i];
    }
    if (use_c) {
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] += e.beta * Elem<T>::lo(w[i]);
            x[2 * i + 1] += e.beta * Elem<T>::hi(w[i]);
        }
    }
    if (e.bias != nullptr) {
        const uint4 bv = reinterpret_cast<const uint4*>(area + 256)[j];
        const uint32_t w[4] = {bv.x, bv.y, bv.z, bv.w};
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
    x *= e.scale_n != nullptr ? e.alpha * e.scale_n[col] : e.alpha;
    if (e.C != nullptr && e.beta != 0.0f) x += e.beta * Elem<T>::to_float(static_cast<const T*>(e.C)[row * N + col]);
    if (e.bias != nullptr) x += Elem<T>::to_float(static_cast<const T*>(e.bias)[col]);
    if (e.act == 1) x = x < 0.0f ? 0.0f : x;
    return x;
}

// The per-column part of the transform for one output column n (alpha *
// s[n] and the bias), fetched ahead of use; apply() is epi_apply1 with them.
template <class T>
struct EpiColumnFactors {
    float a = 1.0f;   // alpha * s[n]
    float b = 0.0f;   // bias[n]
    __device__ __forceinline__ void load(const EpiParams& e, int64_t n) {
        a = e.scale_n != nullptr ? e.alpha * e.scale_n[n] : e.alpha;
        b = e.bias != nullptr ? Elem<T>::to_float(static_cast<const T*>(e.bias)[n]) : 0.0f;
    }
    __device__ __forceinline__ float apply(const EpiParams& e, float x, int64_t row, int64_t col, int64_t N) const {
        x *= a;
        if (e.C != nullptr && e.beta != 0.0f) x += e.beta * Elem<T>::to_float(static_cast<const T*>(e.C)[row * N + col]);
        if (e.bias != nullptr) x += b;
        if (e.act == 1) x = x < 0.0f ? 0.0f : x;
        return x;
    }
};

// One output column n of the small-M kernel (rows 0..MN-1): the C values and
// the bias are fetched with independent loads before any output is written,
// so their latencies overlap (and an in-place C == D is read before it is
// overwritten).  apply() is epi_apply1 on the fetched values.
// The C values stay in their 16-bit form, two to a register.
template <class T, int MN>
struct EpiColumn {
    uint32_t c[(MN + 1) / 2];
    float b;
    float a;   // alpha * s[n]
    __device__ __forceinline__ void load(const EpiParams& e, int64_t n, int64_t M, int64_t N) {
        const bool use_c = e.C != nullptr && e.beta != 0.0f;
        const uint16_t* C = static_cast<const uint16_t*>(e.C);
#pragma unroll
        for (int i = 0; i < (MN + 1) / 2; ++i) c[i] = 0u;
#pragma unroll
        for (int m = 0; m < MN; ++m)
            if (use_c && m < M) c[m >> 1] |= static_cast<uint32_t>(C[m * N + n]) << (16 * (m & 1));
        b = e.bias != nullptr ? Elem<T>::to_float(static_cast<const T*>(e.bias)[n]) : 0.0f;
        a = e.scale_n != nullptr ? e.alpha * e.scale_n[n] : e.alpha;
    }
    __device__ __forceinline__ float apply(const EpiParams& e, float x, int m) const {
        x *= a;
        if (e.C != nullptr && e.beta != 0.0f)
            x += e.beta * ((m & 1) ? Elem<T>::hi(c[m >> 1]) : Elem<T>::lo(c[m >> 1]));
        if (e.bias != nullptr) x += b;
        if (e.act == 1) x = x < 0.0f ? 0.0f : x;
        return x;
    }
};

}  // namespace gemm_gb300
