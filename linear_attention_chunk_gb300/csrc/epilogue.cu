// epilogue.cu -- the per-head epilogue of the Simple GLA mixer, from the
// "GLA mixer" paragraph of "Beyond the KV cache: Training and serving i14's
// Laplace 3B linear attention model on AWS Trainium2 with native PyTorch"
// (its equations did not survive extraction; the reading):
//     u = o + sigmoid(q . (a * k)) v       self-augmentation, a = aug_balance of the head
//     y = w * u / sqrt(mean(u^2) + eps)    Head RMSNorm over the head's dv channels
//     z = y * g * sigmoid(g)               the SiLU(g) output gate
// per (token, head). A stream over o, q, k, v, g in and z out (1,920 bytes
// per head-token at bf16, dk = 96, dv = 192): a half-warp per (token, head)
// with contiguous vector accesses for the bf16 96 x 192 shape (a warp per
// row, lanes striding over channels, otherwise); the two reductions are
// shuffles. The fp32 validation
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

// bf16, dk = 96, dv = 192: two rows per warp, a half-warp (16 lanes) per
// row, so no lane idles. Lane l of a half owns channels 8l..8l+7 (16 bytes)
// and 128+4l..128+4l+3 (8 bytes) of o, v, g, z, and dims 4l..4l+3 and
// 64+2l, 64+2l+1 of q, k: every access is a contiguous run across the half.
// At bf16 output precision the gate's SiLU takes the tanh form,
// g sigmoid(g) = (g/2)(1 + tanh(g/2)): one special-function op per channel.
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float half_sum(float x) {   // over the 16 lanes of a half-warp
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// kFromU: the rows of p.o already hold u (the forward added the
// self-augmentation); only the normalisation, the norm weight and the gate
// are applied, and p.o may be p.z (in place: each lane reads the channels it
// then writes).
template <bool kFromU>
__global__ void __launch_bounds__(32 * kWarps) mixer_epilogue_bf16_kernel(EpilogueParams p) {
    const size_t rows = (size_t)p.NT * p.H;
    const size_t row = ((size_t)blockIdx.x * kWarps + threadIdx.x / 32) * 2 + (threadIdx.x / 16) % 2;
    const int l = threadIdx.x % 16;
    if (row - (row & 1) >= rows) return;          // both rows of this warp are past the end
    const bool live = row < rows;                 // the odd row of an odd total is not
    const size_t r = live ? row : row - 1;        // (it mirrors its partner and stores nothing)
    const int h = (int)(r % (size_t)p.H);
    const unsigned char *ob = static_cast<const unsigned char *>(p.o) + r * 384;
    const unsigned char *gb = static_cast<const unsigned char *>(p.g) + r * 384;
    const uint4 o16 = __ldcs(reinterpret_cast<const uint4 *>(ob) + l);
    const uint4 g16 = __ldcs(reinterpret_cast<const uint4 *>(gb) + l);
    const uint2 o8 = __ldcs(reinterpret_cast<const uint2 *>(ob + 256) + l);
    const uint2 g8 = __ldcs(reinterpret_cast<const uint2 *>(gb + 256) + l);
    uint4 v16 = make_uint4(0, 0, 0, 0);
    uint2 v8 = make_uint2(0, 0);
    if constexpr (!kFromU) {
        const unsigned char *vb = static_cast<const unsigned char *>(p.v) + r * 384;
        v16 = __ldcs(reinterpret_cast<const uint4 *>(vb) + l);
        v8 = __ldcs(reinterpret_cast<const uint2 *>(vb + 256) + l);
    }
    float dot = 0.f;
    if (!kFromU && p.aug) {
        const unsigned char *qb = static_cast<const unsigned char *>(p.q) + r * 192;
        const unsigned char *kb = static_cast<const unsigned char *>(p.k) + r * 192;
        const uint2 q8 = __ldcs(reinterpret_cast<const uint2 *>(qb) + l);
        const uint2 k8 = __ldcs(reinterpret_cast<const uint2 *>(kb) + l);
        const uint32_t q4 = __ldcs(reinterpret_cast<const unsigned int *>(qb + 128) + l);
        const uint32_t k4 = __ldcs(reinterpret_cast<const unsigned int *>(kb + 128) + l);
        const float *a = p.aug + (size_t)h * 96;
        const float4 a4 = __ldg(reinterpret_cast<const float4 *>(a) + l);
        const float2 a2 = __ldg(reinterpret_cast<const float2 *>(a + 64) + l);
        const float2 qa = unpack_bf16x2(q8.x), qb2 = unpack_bf16x2(q8.y), qc = unpack_bf16x2(q4);
        const float2 ka = unpack_bf16x2(k8.x), kb2 = unpack_bf16x2(k8.y), kc = unpack_bf16x2(k4);
        dot = fmaf(qa.x * a4.x, ka.x, dot);
        dot = fmaf(qa.y * a4.y, ka.y, dot);
        dot = fmaf(qb2.x * a4.z, kb2.x, dot);
        dot = fmaf(qb2.y * a4.w, kb2.y, dot);
        dot = fmaf(qc.x * a2.x, kc.x, dot);
        dot = fmaf(qc.y * a2.y, kc.y, dot);
    }
    const float gate = kFromU ? 0.f : __fdividef(1.f, 1.f + __expf(-half_sum(dot)));
    const uint32_t ow[6] = {o16.x, o16.y, o16.z, o16.w, o8.x, o8.y};
    const uint32_t vw[6] = {v16.x, v16.y, v16.z, v16.w, v8.x, v8.y};
    float u[12];
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 6; ++e) {
        const float2 of = unpack_bf16x2(ow[e]), vf = unpack_bf16x2(vw[e]);
        u[2 * e] = fmaf(gate, vf.x, of.x);
        u[2 * e + 1] = fmaf(gate, vf.y, of.y);
        ss = fmaf(u[2 * e], u[2 * e], fmaf(u[2 * e + 1], u[2 * e + 1], ss));
    }
    const float rinv = rsqrtf(half_sum(ss) * (1.f / 192.f) + p.eps);
    float w[12];
#pragma unroll
    for (int e = 0; e < 12; ++e) w[e] = rinv;
    if (p.norm_w) {
        const float *wr = p.norm_w + (size_t)h * 192;
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(wr) + 2 * l);
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(wr) + 2 * l + 1);
        const float4 w2 = __ldg(reinterpret_cast<const float4 *>(wr + 128) + l);
        const float wv[12] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w, w2.x, w2.y, w2.z, w2.w};
#pragma unroll
        for (int e = 0; e < 12; ++e) w[e] *= wv[e];
    }
    const uint32_t gw[6] = {g16.x, g16.y, g16.z, g16.w, g8.x, g8.y};
    uint32_t zw[6];
#pragma unroll
    for (int e = 0; e < 6; ++e) {
        const float2 gf = unpack_bf16x2(gw[e]);
        const float h0 = 0.5f * gf.x, h1 = 0.5f * gf.y;
        zw[e] = pack_bf16x2(u[2 * e] * w[2 * e] * fmaf(h0, tanh_fast(h0), h0),
                            u[2 * e + 1] * w[2 * e + 1] * fmaf(h1, tanh_fast(h1), h1));
    }
    if (live) {
        unsigned char *zb = static_cast<unsigned char *>(p.z) + r * 384;
        __stcs(reinterpret_cast<uint4 *>(zb) + l, make_uint4(zw[0], zw[1], zw[2], zw[3]));
        __stcs(reinterpret_cast<uint2 *>(zb + 256) + l, make_uint2(zw[4], zw[5]));
    }
}

template <typename T>
cudaError_t epilogue_impl(const EpilogueParams &p, cudaStream_t s, int *launches) {
    const size_t rows = (size_t)p.NT * p.H;
    if (rows == 0) return cudaSuccess;
    const size_t blocks = (rows + kWarps - 1) / kWarps;
    if (blocks > 0x7fffffffull) return cudaErrorInvalidValue;
    if (std::is_same<T, __nv_bfloat16>::value && p.dk == 96 && p.dv == 192)
        mixer_epilogue_bf16_kernel<false><<<(unsigned)((rows + 2 * kWarps - 1) / (2 * kWarps)), 32 * kWarps, 0, s>>>(p);
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

cudaError_t launch_mixer_finish(const EpilogueParams &p, cudaStream_t s, int *launches) {
    if (p.dk != 96 || p.dv != 192) return cudaErrorInvalidValue;
    const size_t rows = (size_t)p.NT * p.H;
    if (rows == 0) return cudaSuccess;
    const size_t blocks = (rows + 2 * kWarps - 1) / (2 * kWarps);
    if (blocks > 0x7fffffffull) return cudaErrorInvalidValue;
    mixer_epilogue_bf16_kernel<true><<<(unsigned)blocks, 32 * kWarps, 0, s>>>(p);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
