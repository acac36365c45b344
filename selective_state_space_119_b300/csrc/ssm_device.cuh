// ssm_device.cuh -- device helpers shared by the libssm kernels (sm_103a).
//
// Element access for the two I/O types, the exponential and the two
// activations the selective scan uses:
//   softplus(v) = log(1 + e^v)   on delta ("Mamba: State Space Models Challenge
//                                 Transformers", "Mamba's Innovation: Selection";
//                                 "State Space Models and Mamba", "Mamba:
//                                 Selective State Spaces")
//   silu(z)     = z / (1 + e^-z)  the output gate (same section, y * silu(z))
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the SFU (PTX ex2.approx.ftz.f32). exp(dt * A) is evaluated as
// 2^(dt * (A * log2 e)), with A * log2 e formed once per channel.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLn2 = 0.6931471805599453f;

// log2(x) with the SFU (PTX lg2.approx.ftz.f32).
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = log(1 + e^v) with two SFU operations. w = e^v; for w < 2^-7
// the rounding of 1 + w would dominate log(1 + w), so the Taylor series
// w - w^2/2 + w^3/3 - w^4/4 is used there (truncation error below w^5/5,
// under 2^-28 relative). Above v = 20, log(1 + e^v) equals v to within e^-20.
__device__ __forceinline__ float softplus(float v) {
    const float w = ex2(v * kLog2e);
    const float series = w * fmaf(w, fmaf(w, fmaf(w, -0.25f, 1.f / 3.f), -0.5f), 1.f);
    const float logged = lg2(1.f + w) * kLn2;
    const float r = w < 0.0078125f ? series : logged;
    return v > 20.f ? v : r;
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z). For z < -88, e^-z overflows to
// inf and the quotient is -0, the correctly signed limit.
__device__ __forceinline__ float silu(float z) {
    return __fdividef(z, 1.f + __expf(-z));
}

// ---------------------------------------------------------------------------
// I/O element types: fp32 or bf16 storage, fp32 arithmetic.
// ---------------------------------------------------------------------------
template <typename T> struct IO;

template <> struct IO<float> {
    __device__ __forceinline__ static float ld(const float* p) { return __ldg(p); }
    __device__ __forceinline__ static void st(float* p, float v) { *p = v; }
};

template <> struct IO<__nv_bfloat16> {
    __device__ __forceinline__ static float ld(const __nv_bfloat16* p) {
        return __bfloat162float(__ldg(p));
    }
    __device__ __forceinline__ static void st(__nv_bfloat16* p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

// CPT consecutive channels of one token, loaded/stored as one vector
// (CPT * sizeof(T) bytes; the caller guarantees that alignment).
template <typename T, int CPT> struct Vec;

template <int CPT> struct Vec<float, CPT> {
    static_assert(CPT == 1 || CPT == 2 || CPT == 4, "fp32 vector width");
    __device__ __forceinline__ static void ld(const float* p, float (&v)[CPT]) {
        if constexpr (CPT == 1) {
            v[0] = __ldg(p);
        } else if constexpr (CPT == 2) {
            const float2 u = __ldg(reinterpret_cast<const float2*>(p));
            v[0] = u.x; v[1] = u.y;
        } else {
            const float4 u = __ldg(reinterpret_cast<const float4*>(p));
            v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        }
    }
    // shared-memory pair access (CPT == 2)
    __device__ __forceinline__ static void lds(const float* p, float (&v)[CPT]) {
        static_assert(CPT == 2, "pairs");
        const float2 u = *reinterpret_cast<const float2*>(p);
        v[0] = u.x; v[1] = u.y;
    }
    __device__ __forceinline__ static void sts(float* p, const float (&v)[CPT]) {
        static_assert(CPT == 2, "pairs");
        *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    }
    __device__ __forceinline__ static void st(float* p, const float (&v)[CPT]) {
        if constexpr (CPT == 1) {
            *p = v[0];
        } else if constexpr (CPT == 2) {
            *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
        } else {
            *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
};

template <int CPT> struct Vec<__nv_bfloat16, CPT> {
    static_assert(CPT == 1 || CPT == 2 || CPT == 4 || CPT == 8, "bf16 vector width");
    __device__ __forceinline__ static void unpack(uint32_t w, float& lo, float& hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
        return *reinterpret_cast<const uint32_t*>(&b);
    }
    __device__ __forceinline__ static void ld(const __nv_bfloat16* p, float (&v)[CPT]) {
        if constexpr (CPT == 1) {
            v[0] = __bfloat162float(__ldg(p));
        } else if constexpr (CPT == 2) {
            unpack(__ldg(reinterpret_cast<const unsigned int*>(p)), v[0], v[1]);
        } else if constexpr (CPT == 4) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
            unpack(u.x, v[0], v[1]); unpack(u.y, v[2], v[3]);
        } else {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
            unpack(u.x, v[0], v[1]); unpack(u.y, v[2], v[3]);
            unpack(u.z, v[4], v[5]); unpack(u.w, v[6], v[7]);
        }
    }
    // shared-memory pair access (CPT == 2)
    __device__ __forceinline__ static void lds(const __nv_bfloat16* p, float (&v)[CPT]) {
        static_assert(CPT == 2, "pairs");
        unpack(*reinterpret_cast<const uint32_t*>(p), v[0], v[1]);
    }
    __device__ __forceinline__ static void sts(__nv_bfloat16* p, const float (&v)[CPT]) {
        static_assert(CPT == 2, "pairs");
        *reinterpret_cast<uint32_t*>(p) = pack(v[0], v[1]);
    }
    __device__ __forceinline__ static void st(__nv_bfloat16* p, const float (&v)[CPT]) {
        if constexpr (CPT == 1) {
            *p = __float2bfloat16_rn(v[0]);
        } else if constexpr (CPT == 2) {
            *reinterpret_cast<unsigned int*>(p) = pack(v[0], v[1]);
        } else if constexpr (CPT == 4) {
            *reinterpret_cast<uint2*>(p) = make_uint2(pack(v[0], v[1]), pack(v[2], v[3]));
        } else {
            *reinterpret_cast<uint4*>(p) = make_uint4(pack(v[0], v[1]), pack(v[2], v[3]),
                                                      pack(v[4], v[5]), pack(v[6], v[7]));
        }
    }
};

}  // namespace ssm
