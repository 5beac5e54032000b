// fwd_full.cu -- launches of the one-CTA-per-(b, h) chunk kernel (its body
// and design in fwd_full.cuh): the forward, plain or segmented, with the
// per-head or the per-token decay, the variable-length prefill into a state
// pool, and the per-token decay's dv.
#include "fwd_full.cuh"

namespace gla {
namespace {

using namespace fullhead;

template <bool kRev, int kC, bool kGate, bool kVar = false, bool kEpi = false>
__global__ void __launch_bounds__(kThreads, 1)
    gla_fwd_full_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const FullArgs a) {
    full_body<kRev, kC, kGate, kVar, kEpi>(tm_q, tm_k, tm_v, tm_o, a, (int)blockIdx.x);
}

}  // namespace

cudaError_t launch_fwd_full_tc(const FwdParams &p, float *S_in, int nseg, int seg_chunks, cudaStream_t s,
                               int *launches, const EpilogueParams *epi) {
    if (p.dk != kDk || p.dv != kDv || (epi && (p.g || p.chunk != 128))) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mo;
    cudaError_t e;
    if ((e = make_token_map(&mq, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mk, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, p.o, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    FullArgs a{p.log_lambda, S_in ? S_in : p.h0, p.hT, p.scale, 1.f, 1.f, p.T, p.H, nck, nseg,
               nseg > 1 ? seg_chunks : nck, p.B * p.H, nseg > 1 ? (size_t)p.B * p.H * kDk * kDv : 0, p.status, p.g,
               nullptr, nullptr, 0, nullptr, epi ? epi->aug : nullptr};
    auto kernel = epi ? gla_fwd_full_kernel<false, 128, false, false, true>
                : p.g ? (p.chunk == 128 ? gla_fwd_full_kernel<false, 128, true> : gla_fwd_full_kernel<false, 64, true>)
                      : (p.chunk == 128 ? gla_fwd_full_kernel<false, 128, false>
                                        : gla_fwd_full_kernel<false, 64, false>);
    const uint32_t smem = p.chunk == 128 ? Layout<128>::kSmemBytes : Layout<64>::kSmemBytes;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<(unsigned)(p.B * p.H * nseg), kThreads, smem, s>>>(mq, mk, mv, mo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

// dv and dh0 of the per-token decay's backward: the recurrence in reverse time
// with rows = k, columns = q, values = dO; state = (state gradient) / scale,
// seeded by dhT / scale and written out times the scale as dh0.
cudaError_t launch_bwd_dv_full_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv || !p.g) return cudaErrorInvalidValue;
    CUtensorMap mrow, mcol, mval, mout;
    cudaError_t e;
    if ((e = make_token_map(&mrow, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mcol, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mval, p.do_, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mout, p.dv_out, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    FullArgs a{p.log_lambda, p.dhT, p.dh0, p.scale, 1.f / p.scale, p.scale, p.T, p.H, nck, 1, nck, p.B * p.H, 0,
               p.status, p.g, nullptr, nullptr, 0, nullptr, nullptr};
    auto kernel = p.chunk == 128 ? gla_fwd_full_kernel<true, 128, true> : gla_fwd_full_kernel<true, 64, true>;
    const uint32_t smem = p.chunk == 128 ? Layout<128>::kSmemBytes : Layout<64>::kSmemBytes;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<(unsigned)(p.B * p.H), kThreads, smem, s>>>(mrow, mcol, mval, mout, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

// Variable-length forward: one CTA per (sequence, head) over the packed
// [1, total_T, H, d] tensors; states read from and written back to the pool.
cudaError_t launch_fwd_varlen_full_tc(const VarlenParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mo;
    cudaError_t e;
    if ((e = make_token_map(&mq, p.q, 1, p.total_T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mk, p.k, 1, p.total_T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, 1, p.total_T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, p.o, 1, p.total_T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    // nck and seg_chunks are per sequence (set in the kernel); one segment
    const FullArgs a{p.log_lambda, p.pool, p.pool, p.scale, 1.f, 1.f, p.total_T, p.H, 0, 1, 0, p.nseq * p.H, 0,
                     p.status, p.g, p.cu_seqlens, p.slots, p.n_slots, static_cast<__nv_bfloat16 *>(p.o), nullptr};
    auto kernel = p.g ? (p.chunk == 128 ? gla_fwd_full_kernel<false, 128, true, true>
                                        : gla_fwd_full_kernel<false, 64, true, true>)
                      : (p.chunk == 128 ? gla_fwd_full_kernel<false, 128, false, true>
                                        : gla_fwd_full_kernel<false, 64, false, true>);
    const uint32_t smem = p.chunk == 128 ? Layout<128>::kSmemBytes : Layout<64>::kSmemBytes;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    kernel<<<(unsigned)(p.nseq * p.H), kThreads, smem, s>>>(mq, mk, mv, mo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
