// fwd_full.cu -- launches of the one-CTA-per-(b, h) chunk kernel (its body
// and design in fwd_full.cuh): the forward, plain or segmented.
#include "fwd_full.cuh"

namespace gla {
namespace {

using namespace fullhead;

template <bool kRev, int kC>
__global__ void __launch_bounds__(kThreads, 1)
    gla_fwd_full_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const FullArgs a) {
    full_body<kRev, kC>(tm_q, tm_k, tm_v, tm_o, a, (int)blockIdx.x);
}

}  // namespace

cudaError_t launch_fwd_full_tc(const FwdParams &p, float *S_in, int nseg, int seg_chunks, cudaStream_t s,
                               int *launches) {
    if (p.dk != kDk || p.dv != kDv || p.g) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mo;
    cudaError_t e;
    if ((e = make_token_map(&mq, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mk, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, p.o, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    FullArgs a{p.log_lambda, S_in ? S_in : p.h0, p.hT, p.scale, 1.f, 1.f, p.T, p.H, nck, nseg,
               nseg > 1 ? seg_chunks : nck, p.B * p.H, nseg > 1 ? (size_t)p.B * p.H * kDk * kDv : 0, p.status};
    auto kernel = p.chunk == 128 ? gla_fwd_full_kernel<false, 128> : gla_fwd_full_kernel<false, 64>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    kernel<<<(unsigned)(p.B * p.H * nseg), kThreads, kSmemBytes, s>>>(mq, mk, mv, mo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
