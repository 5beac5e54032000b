// epilogue.cu -- the per-head epilogue of the Simple GLA mixer, from the
// "GLA mixer" paragraph of "Beyond the KV cache: Training and serving i14's
// Laplace 3B linear attention model on AWS Trainium2 with native PyTorch"
// (its equations did not survive extraction; the reading):
//     u = o + sigmoid(q . (a * k)) v       self-augmentation, a = aug_balance of the head
//     y = w * u / sqrt(mean(u^2) + eps)    Head RMSNorm over the head's dv channels
//     z = y * g * sigmoid(g)               the SiLU(g) output gate
// per (token, head). A stream over o, q, k, v, g in and z out (1,920 bytes
// per head-token at bf16, dk = 96, dv = 192): one warp per (token, head),
// 16-byte loads for the bf16 96 x 192 shape (lanes striding over channels
// otherwise); the two reductions are warp shuffles. The fp32 validation
// path keeps exact sigmoids; the bf16 path uses the fast forms.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace gla {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + __expf(-x)); }

// DK, DV: compile-time channel counts (0: take them from the parameters).
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(32 * kWarps) mixer_epilogue_kernel(EpilogueParams p) {
    const size_t row = (size_t)blockIdx.x * kWarps + threadIdx.x / 32;   // token * H + head
    const int lane = threadIdx.x % 32;
    if (row >= (size_t)p.NT * p.H) return;
    const int h = (int)(row % (size_t)p.H);
    const int dk = DK ? DK : p.dk, dv = DV ? DV : p.dv;
    const T *q = static_cast<const T *>(p.q) + row * dk;
    const T *k = static_cast<const T *>(p.k) + row * dk;
    const T *o = static_cast<const T *>(p.o) + row * dv;
    const T *v = static_cast<const T *>(p.v) + row * dv;
    const T *g = static_cast<const T *>(p.g) + row * dv;
    T *z = static_cast<T *>(p.z) + row * dv;
    const float *a = p.aug ? p.aug + (size_t)h * dk : nullptr;
    const float *w = p.norm_w ? p.norm_w + (size_t)h * dv : nullptr;

    float dot = 0.f;
    if (a) {
#pragma unroll 4
        for (int i = lane; i < dk; i += 32) dot += Elem<T>::load(q + i) * a[i] * Elem<T>::load(k + i);
    }
    const float gate = sigmoidf_(warp_sum(dot));

    constexpr int kMaxPer = 8;   // dv <= 256
    float u[kMaxPer];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < kMaxPer; ++m) {
        const int c = lane + 32 * m;
        u[m] = 0.f;
        if (c < dv) {
            u[m] = fmaf(gate, Elem<T>::load(v + c), Elem<T>::load(o + c));
            ss = fmaf(u[m], u[m], ss);
        }
    }
    const float r = rsqrtf(warp_sum(ss) / (float)dv + p.eps);
#pragma unroll
    for (int m = 0; m < kMaxPer; ++m) {
        const int c = lane + 32 * m;
        if (c < dv) {
            const float gc = Elem<T>::load(g + c);
            Elem<T>::store(z + c, u[m] * r * (w ? w[c] : 1.f) * gc * sigmoidf_(gc));
        }
    }
}

// bf16, dk = 96, dv = 192: one warp per row with 16-byte accesses; lane l < 24
// owns channels 8l..8l+7 of o, v, g, z and lane l < 12 dims 8l..8l+7 of q, k.
// At bf16 output precision the gate's SiLU takes the tanh form,
// g sigmoid(g) = (g/2)(1 + tanh(g/2)): one special-function op per channel.
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(32 * kWarps) mixer_epilogue_bf16_kernel(EpilogueParams p) {
    const size_t row = (size_t)blockIdx.x * kWarps + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= (size_t)p.NT * p.H) return;
    const int h = (int)(row % (size_t)p.H);
    uint4 ov = make_uint4(0, 0, 0, 0), vv = ov, gv = ov, qv = ov, kv = ov;
    if (lane < 24) {
        ov = __ldcs(static_cast<const uint4 *>(p.o) + row * 24 + lane);
        vv = __ldcs(static_cast<const uint4 *>(p.v) + row * 24 + lane);
        gv = __ldcs(static_cast<const uint4 *>(p.g) + row * 24 + lane);
    }
    if (lane < 12 && p.aug) {
        qv = __ldcs(static_cast<const uint4 *>(p.q) + row * 12 + lane);
        kv = __ldcs(static_cast<const uint4 *>(p.k) + row * 12 + lane);
    }
    float dot = 0.f;
    if (lane < 12 && p.aug) {
        const float4 *a4 = reinterpret_cast<const float4 *>(p.aug + (size_t)h * 96 + 8 * lane);
        const float4 a0 = __ldg(a4), a1 = __ldg(a4 + 1);
        const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 qf = unpack_bf16x2(qw[e]), kf = unpack_bf16x2(kw[e]);
            dot = fmaf(qf.x * a[2 * e], kf.x, dot);
            dot = fmaf(qf.y * a[2 * e + 1], kf.y, dot);
        }
    }
    const float gate = __fdividef(1.f, 1.f + __expf(-warp_sum(dot)));
    float u[8];
    float ss = 0.f;
    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 of = unpack_bf16x2(ow[e]), vf = unpack_bf16x2(vw[e]);
        u[2 * e] = fmaf(gate, vf.x, of.x);
        u[2 * e + 1] = fmaf(gate, vf.y, of.y);
        ss = fmaf(u[2 * e], u[2 * e], fmaf(u[2 * e + 1], u[2 * e + 1], ss));
    }
    const float r = rsqrtf(warp_sum(ss) * (1.f / 192.f) + p.eps);
    if (lane < 24) {
        float w[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
        if (p.norm_w) {
            const float4 *w4 = reinterpret_cast<const float4 *>(p.norm_w + (size_t)h * 192 + 8 * lane);
            const float4 w0 = __ldg(w4), w1 = __ldg(w4 + 1);
            w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
            w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
        }
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t zw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 gf = unpack_bf16x2(gw[e]);
            const float h0 = 0.5f * gf.x, h1 = 0.5f * gf.y;
            const float s0 = fmaf(h0, tanh_fast(h0), h0), s1 = fmaf(h1, tanh_fast(h1), h1);   // SiLU(g)
            zw[e] = pack_bf16x2(u[2 * e] * r * w[2 * e] * s0, u[2 * e + 1] * r * w[2 * e + 1] * s1);
        }
        __stcs(static_cast<uint4 *>(p.z) + row * 24 + lane, make_uint4(zw[0], zw[1], zw[2], zw[3]));
    }
}

template <typename T>
cudaError_t epilogue_impl(const EpilogueParams &p, cudaStream_t s, int *launches) {
    const size_t rows = (size_t)p.NT * p.H;
    if (rows == 0) return cudaSuccess;
    const size_t blocks = (rows + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffull) return cudaErrorInvalidValue;
    if (std::is_same<T, __nv_bfloat16>::value && p.dk == 96 && p.dv == 192)
        mixer_epilogue_bf16_kernel<<<(unsigned)blocks, 32 * kWarps, 0, s>>>(p);
    else if (p.dk == 96 && p.dv == 192)
        mixer_epilogue_kernel<T, 96, 192><<<(unsigned)blocks, 32 * kWarps, 0, s>>>(p);
    else
        mixer_epilogue_kernel<T, 0, 0><<<(unsigned)blocks, 32 * kWarps, 0, s>>>(p);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mixer_epilogue(const EpilogueParams &p, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? epilogue_impl<__nv_bfloat16>(p, s, launches) : epilogue_impl<float>(p, s, launches);
}

}  // namespace gla
