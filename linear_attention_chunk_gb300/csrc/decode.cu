// decode.cu -- the single-token recurrent step of the Simple GLA mixer, the
// serving path of "Beyond the KV cache: Training and serving i14's Laplace
// 3B linear attention model on AWS Trainium2 with native PyTorch" (section
// "Inference optimization on Trainium2": the recurrent state lives in one
// fixed page per sequence; work per generated token is constant). Per
// (sequence n, head h), with the update and readout of the "GLA mixer"
// paragraph:
//     S <- lambda * S + k v^T     (fp32, in place)
//     o  = scale * S^T q          (after the update)
// lambda = exp(log_lambda[h]), or exp(log_decay[n, h]) for the per-token
// (data-dependent) decay of the gated variant.
//
// The step is a pure stream over S: 73,728 B read and 73,728 B written per
// (n, h) at dk = 96, dv = 192, against 0.5 FLOP per byte -- HBM bound on any
// GPU. The fast path gives each (n, h) one CTA of 192 threads: thread t owns
// four adjacent state columns (one float4) of every fourth row, so a warp
// reads 512 contiguous bytes per load and every thread has 24 independent
// 16-byte loads in flight before it computes. Column partial sums of S^T q
// are reduced across the four row groups in shared memory.
//
// With the mixer epilogue (kEpi) the step writes z = Head RMSNorm(o +
// sigmoid(q.(a*k)) v) * SiLU(g) instead of o (the reading of the "GLA mixer"
// paragraph used by epilogue.cu): the gate's dot product and the row's mean
// square are reduced in the same CTA, so o never leaves the chip.
#include "common.cuh"
#include "kernels.h"

namespace gla {
namespace {

constexpr int kDk = 96, kDv = 192;
constexpr int kColGroups = kDv / 4;               // 48 float4 column groups
constexpr int kRowGroups = 4;
constexpr int kRowsPerThread = kDk / kRowGroups;  // 24
constexpr int kThreads96 = kColGroups * kRowGroups;  // 192

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + __expf(-x)); }

template <typename T, bool kEpi>
__global__ void __launch_bounds__(kThreads96) decode_96x192_kernel(DecodeParams p) {
    const size_t unit = blockIdx.x;                 // n * H + h
    const int h = (int)(unit % (size_t)p.H);
    const int tid = threadIdx.x;
    const int cg = tid % kColGroups, rg = tid / kColGroups;
    __shared__ float qs[kDk], ks[kDk];
    __shared__ float4 red[kRowGroups][kColGroups];
    __shared__ float gate_s, ss_s[2];

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
    const float lam = expf(p.log_decay ? p.log_decay[unit] : p.log_lambda[h]);
    __syncthreads();
    if constexpr (kEpi) {
        if (tid < 32) {   // the self-augmentation gate sigmoid(q . (a * k)) of this (n, h)
            float dot = 0.f;
            if (p.aug) {
#pragma unroll
                for (int i = tid; i < kDk; i += 32) dot += qs[i] * p.aug[h * kDk + i] * ks[i];
            }
            dot = warp_sum(dot);
            if (tid == 0) gate_s = sigmoidf_(dot);
        }
    }

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
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < kColGroups) {
        t = red[0][tid];
#pragma unroll
        for (int g = 1; g < kRowGroups; ++g) {
            t.x += red[g][tid].x; t.y += red[g][tid].y; t.z += red[g][tid].z; t.w += red[g][tid].w;
        }
    }
    T *o = static_cast<T *>(p.o) + unit * kDv + 4 * tid;
    if constexpr (!kEpi) {
        if (tid < kColGroups) {
            Elem<T>::store(o + 0, p.scale * t.x);
            Elem<T>::store(o + 1, p.scale * t.y);
            Elem<T>::store(o + 2, p.scale * t.z);
            Elem<T>::store(o + 3, p.scale * t.w);
        }
    } else {
        // u = o + gate v; z = w u / sqrt(mean(u^2) + eps) * SiLU(g), written to p.o
        const float gate = gate_s;
        float u[4] = {0.f, 0.f, 0.f, 0.f}, part = 0.f;
        if (tid < kColGroups) {
            u[0] = fmaf(gate, v0, p.scale * t.x);
            u[1] = fmaf(gate, v1, p.scale * t.y);
            u[2] = fmaf(gate, v2, p.scale * t.z);
            u[3] = fmaf(gate, v3, p.scale * t.w);
            part = u[0] * u[0] + u[1] * u[1] + u[2] * u[2] + u[3] * u[3];
        }
        part = warp_sum(part);                       // the 48 owners are warps 0 and 1
        if (tid == 0 || tid == 32) ss_s[tid / 32] = part;
        __syncthreads();
        const float r = rsqrtf((ss_s[0] + ss_s[1]) / (float)kDv + p.eps);
        if (tid < kColGroups) {
            const T *g = static_cast<const T *>(p.g) + unit * kDv + 4 * tid;
            const float *w = p.norm_w ? p.norm_w + h * kDv + 4 * tid : nullptr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float gj = Elem<T>::load(g + j);
                Elem<T>::store(o + j, u[j] * r * (w ? w[j] : 1.f) * gj * sigmoidf_(gj));
            }
        }
    }
}

// Any dk <= 128, dv <= 256: one CTA of 128 threads per (n, h), threads
// stride over state columns (at most two columns each).
template <typename T, bool kEpi>
__global__ void __launch_bounds__(128) decode_generic_kernel(DecodeParams p) {
    const size_t unit = blockIdx.x;
    const int h = (int)(unit % (size_t)p.H);
    const int dk = p.dk, dv = p.dv;
    const T *q = static_cast<const T *>(p.q) + unit * dk;
    const T *k = static_cast<const T *>(p.k) + unit * dk;
    const T *v = static_cast<const T *>(p.v) + unit * dv;
    T *o = static_cast<T *>(p.o) + unit * dv;
    float *S = p.S + unit * (size_t)dk * dv;
    const float lam = expf(p.log_decay ? p.log_decay[unit] : p.log_lambda[h]);
    __shared__ float red[4];
    float u[2] = {0.f, 0.f};
    for (int m = 0; m < 2; ++m) {
        const int c = threadIdx.x + 128 * m;
        if (c >= dv) break;
        const float vc = Elem<T>::load(v + c);
        float acc = 0.f;
        for (int a = 0; a < dk; ++a) {
            float x = fmaf(lam, S[(size_t)a * dv + c], Elem<T>::load(k + a) * vc);
            S[(size_t)a * dv + c] = x;
            acc = fmaf(x, Elem<T>::load(q + a), acc);
        }
        u[m] = p.scale * acc;
        if constexpr (!kEpi) Elem<T>::store(o + c, u[m]);
    }
    if constexpr (kEpi) {
        // block sums over the 4 warps: the gate's dot product, then the mean square
        auto block_sum = [&](float x) {
            x = warp_sum(x);
            __syncthreads();
            if (threadIdx.x % 32 == 0) red[threadIdx.x / 32] = x;
            __syncthreads();
            return red[0] + red[1] + red[2] + red[3];
        };
        float dot = 0.f;
        if (p.aug)
            for (int i = threadIdx.x; i < dk; i += 128)
                dot += Elem<T>::load(q + i) * p.aug[(size_t)h * dk + i] * Elem<T>::load(k + i);
        const float gate = sigmoidf_(block_sum(dot));
        float part = 0.f;
        for (int m = 0; m < 2; ++m) {
            const int c = threadIdx.x + 128 * m;
            if (c < dv) {
                u[m] = fmaf(gate, Elem<T>::load(v + c), u[m]);
                part = fmaf(u[m], u[m], part);
            }
        }
        const float r = rsqrtf(block_sum(part) / (float)dv + p.eps);
        const T *g = static_cast<const T *>(p.g) + unit * dv;
        for (int m = 0; m < 2; ++m) {
            const int c = threadIdx.x + 128 * m;
            if (c < dv) {
                const float gc = Elem<T>::load(g + c);
                Elem<T>::store(o + c, u[m] * r * (p.norm_w ? p.norm_w[(size_t)h * dv + c] : 1.f) * gc *
                                          sigmoidf_(gc));
            }
        }
    }
}

template <typename T>
cudaError_t decode_impl(const DecodeParams &p, cudaStream_t s, int *launches) {
    const size_t units = (size_t)p.N * p.H;
    if (units == 0) return cudaSuccess;
    if (units > 0x7fffffffull) return cudaErrorInvalidValue;
    const bool epi = p.g != nullptr;
    if (p.dk == kDk && p.dv == kDv) {
        if (epi) decode_96x192_kernel<T, true><<<(unsigned)units, kThreads96, 0, s>>>(p);
        else decode_96x192_kernel<T, false><<<(unsigned)units, kThreads96, 0, s>>>(p);
    } else {
        if (epi) decode_generic_kernel<T, true><<<(unsigned)units, 128, 0, s>>>(p);
        else decode_generic_kernel<T, false><<<(unsigned)units, 128, 0, s>>>(p);
    }
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? decode_impl<__nv_bfloat16>(p, s, launches) : decode_impl<float>(p, s, launches);
}

}  // namespace gla
