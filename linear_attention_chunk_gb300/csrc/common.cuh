// common.cuh -- small device helpers shared by the libgla kernels.
//
// Decay powers follow the Simple GLA recurrence of "Beyond the KV cache:
// Training and serving i14's Laplace 3B linear attention model on AWS
// Trainium2 with native PyTorch" (section "i14 and the Laplace 3B
// architecture", paragraph "GLA mixer"): lambda = exp(log_lambda), and a
// power lambda^n is taken directly for every n >= 0 that the chunked form
// needs -- never as a quotient lambda^i / lambda^j, which overflows for
// small lambda (lambda = 0.5 gives 2^128 at n = -128).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gla {

// Device status word bits (see gla_check()).
enum : unsigned int {
    kDevTimeout = 1u << 0,   // an mbarrier / flag wait gave up
    kDevBadState = 1u << 1,  // an internal consistency check failed
};

// log2(lambda) from the natural log, in double once per CTA.
__device__ __forceinline__ float log2_of_decay(float log_lambda) {
    return (float)((double)log_lambda * 1.4426950408889634073599246810019);
}

// lambda^n for integer n >= 0; lambda^0 = 1 even when lambda = 0
// (log2 lambda = -inf). Negative n is never asked for.
__device__ __forceinline__ float decay_pow(float log2_lambda, int n) {
    return n == 0 ? 1.0f : exp2f((float)n * log2_lambda);
}

template <typename T> struct Elem;

template <> struct Elem<float> {
    static __device__ __forceinline__ float load(const float *p) { return *p; }
    static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};

template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two bf16 products in one instruction (round to nearest).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
    __nv_bfloat162 z = __hmul2(x, y);
    return *reinterpret_cast<uint32_t *>(&z);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

}  // namespace gla
