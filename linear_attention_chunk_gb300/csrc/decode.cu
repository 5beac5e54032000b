// decode.cu -- the single-token recurrent step of the Simple GLA mixer, the
// serving path of "Beyond the KV cache: Training and serving i14's Laplace
// 3B linear attention model on AWS Trainium2 with native PyTorch" (section
// "Inference optimization on Trainium2": the recurrent state lives in one
// fixed page per sequence; work per generated token is constant). Per
// (sequence n, head h), with the update and readout of the "GLA mixer"
// paragraph:
//     S <- lambda * S + k v^T     (fp32, in place)
//     o  = scale * S^T q          (after the update)
//
// The step is a pure stream over S: 73,728 B read and 73,728 B written per
// (n, h) at dk = 96, dv = 192, against 0.5 FLOP per byte -- HBM bound on any
// GPU. The fast path gives each (n, h) one CTA of 192 threads: thread t owns
// four adjacent state columns (one float4) of every fourth row, so a warp
// reads 512 contiguous bytes per load and every thread has 24 independent
// 16-byte loads in flight before it computes. Column partial sums of S^T q
// are reduced across the four row groups in shared memory.
#include "common.cuh"
#include "kernels.h"

namespace gla {
namespace {

constexpr int kDk = 96, kDv = 192;
constexpr int kColGroups = kDv / 4;               // 48 float4 column groups
constexpr int kRowGroups = 4;
constexpr int kRowsPerThread = kDk / kRowGroups;  // 24
constexpr int kThreads96 = kColGroups * kRowGroups;  // 192

template <typename T>
__global__ void __launch_bounds__(kThreads96) decode_96x192_kernel(DecodeParams p) {
    const size_t unit = blockIdx.x;                 // n * H + h
    const int h = (int)(unit % (size_t)p.H);
    const int tid = threadIdx.x;
    const int cg = tid % kColGroups, rg = tid / kColGroups;
    __shared__ float qs[kDk], ks[kDk];
    __shared__ float4 red[kRowGroups][kColGroups];

    float4 *S4 = reinterpret_cast<float4 *>(p.S + unit * (size_t)(kDk * kDv));
    float4 s[kRowsPerThread];
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) s[m] = __ldcs(S4 + (rg + kRowGroups * m) * kColGroups + cg);

    const T *q = static_cast<const T *>(p.q) + unit * kDk;
    const T *k = static_cast<const T *>(p.k) + unit * kDk;
    const T *v = static_cast<const T *>(p.v) + unit * kDv + 4 * cg;
    if (tid < kDk) {
        qs[tid] = Elem<T>::load(q + tid);
        ks[tid] = Elem<T>::load(k + tid);
    }
    const float v0 = Elem<T>::load(v), v1 = Elem<T>::load(v + 1), v2 = Elem<T>::load(v + 2),
                v3 = Elem<T>::load(v + 3);
    const float lam = expf(p.log_lambda[h]);
    __syncthreads();

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
        const int r = rg + kRowGroups * m;
        const float kr = ks[r], qr = qs[r];
        float4 x = s[m];
        x.x = fmaf(lam, x.x, kr * v0);
        x.y = fmaf(lam, x.y, kr * v1);
        x.z = fmaf(lam, x.z, kr * v2);
        x.w = fmaf(lam, x.w, kr * v3);
        acc.x = fmaf(x.x, qr, acc.x);
        acc.y = fmaf(x.y, qr, acc.y);
        acc.z = fmaf(x.z, qr, acc.z);
        acc.w = fmaf(x.w, qr, acc.w);
        __stcs(S4 + r * kColGroups + cg, x);
    }
    red[rg][cg] = acc;
    __syncthreads();
    if (tid < kColGroups) {
        float4 t = red[0][tid];
#pragma unroll
        for (int g = 1; g < kRowGroups; ++g) {
            t.x += red[g][tid].x; t.y += red[g][tid].y; t.z += red[g][tid].z; t.w += red[g][tid].w;
        }
        T *o = static_cast<T *>(p.o) + unit * kDv + 4 * tid;
        Elem<T>::store(o + 0, p.scale * t.x);
        Elem<T>::store(o + 1, p.scale * t.y);
        Elem<T>::store(o + 2, p.scale * t.z);
        Elem<T>::store(o + 3, p.scale * t.w);
    }
}

// Any dk, dv: one CTA per (n, h), threads stride over state columns.
template <typename T>
__global__ void __launch_bounds__(128) decode_generic_kernel(DecodeParams p) {
    const size_t unit = blockIdx.x;
    const int h = (int)(unit % (size_t)p.H);
    const int dk = p.dk, dv = p.dv;
    const T *q = static_cast<const T *>(p.q) + unit * dk;
    const T *k = static_cast<const T *>(p.k) + unit * dk;
    const T *v = static_cast<const T *>(p.v) + unit * dv;
    T *o = static_cast<T *>(p.o) + unit * dv;
    float *S = p.S + unit * (size_t)dk * dv;
    const float lam = expf(p.log_lambda[h]);
    for (int c = threadIdx.x; c < dv; c += blockDim.x) {
        const float vc = Elem<T>::load(v + c);
        float acc = 0.f;
        for (int a = 0; a < dk; ++a) {
            float x = fmaf(lam, S[(size_t)a * dv + c], Elem<T>::load(k + a) * vc);
            S[(size_t)a * dv + c] = x;
            acc = fmaf(x, Elem<T>::load(q + a), acc);
        }
        Elem<T>::store(o + c, p.scale * acc);
    }
}

template <typename T>
cudaError_t decode_impl(const DecodeParams &p, cudaStream_t s, int *launches) {
    const size_t units = (size_t)p.N * p.H;
    if (units == 0) return cudaSuccess;
    if (units > 0x7fffffffull) return cudaErrorInvalidValue;
    if (p.dk == kDk && p.dv == kDv)
        decode_96x192_kernel<T><<<(unsigned)units, kThreads96, 0, s>>>(p);
    else
        decode_generic_kernel<T><<<(unsigned)units, 128, 0, s>>>(p);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? decode_impl<__nv_bfloat16>(p, s, launches) : decode_impl<float>(p, s, launches);
}

}  // namespace gla
