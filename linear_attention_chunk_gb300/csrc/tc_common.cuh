// tc_common.cuh -- device helpers shared by the tensor-core chunk kernels:
// row-wise work on 64-byte-swizzled shared-memory tiles, the decay-masked
// score block written to TMEM as bf16 pairs, and the bounded group waits.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace gla {
namespace tc {

using namespace ptx;

constexpr uint32_t kBlk = 128 * 64;                  // [128 rows][32 bf16] block = 8 KB
constexpr uint32_t kGroupThreads = 128;

// Multiply row `row` of NB (3 or 6) 64-byte-swizzled blocks at blk0 (stride
// kBlk) in place by w, six 16-byte chunks at a time (loads first, then
// stores, so the loads overlap). The 64-byte swizzle only permutes a row's
// chunks, so a row is scaled as it lies; chunks are visited in swizzled
// order so that the 32 rows a warp touches at once fall in distinct banks.
template <int NB>
__device__ __forceinline__ void scale_rows(unsigned char *blk0, uint32_t row, float w) {
    const uint32_t w2 = pack_bf16x2(w, w);
#pragma unroll
    for (int h6 = 0; h6 < 4 * NB; h6 += 6) {
        uint4 v[6];
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int k = h6 + i;
            v[i] = *reinterpret_cast<const uint4 *>(blk0 + (k >> 2) * kBlk + sw64_offset(row, (uint32_t)(k & 3)));
        }
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            v[i].x = mul_bf16x2(v[i].x, w2);
            v[i].y = mul_bf16x2(v[i].y, w2);
            v[i].z = mul_bf16x2(v[i].z, w2);
            v[i].w = mul_bf16x2(v[i].w, w2);
        }
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int k = h6 + i;
            *reinterpret_cast<uint4 *>(blk0 + (k >> 2) * kBlk + sw64_offset(row, (uint32_t)(k & 3))) = v[i];
        }
    }
}

// Row `row` of NB 64-byte-swizzled blocks at src, times w, into the same row
// of the blocks at dst (both with stride kBlk).
template <int NB>
__device__ __forceinline__ void scale_rows_to(const unsigned char *src, unsigned char *dst, uint32_t row, float w) {
    const uint32_t w2 = pack_bf16x2(w, w);
#pragma unroll
    for (int h6 = 0; h6 < 4 * NB; h6 += 6) {
        uint4 v[6];
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int k = h6 + i;
            v[i] = *reinterpret_cast<const uint4 *>(src + (k >> 2) * kBlk + sw64_offset(row, (uint32_t)(k & 3)));
        }
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            v[i].x = mul_bf16x2(v[i].x, w2);
            v[i].y = mul_bf16x2(v[i].y, w2);
            v[i].z = mul_bf16x2(v[i].z, w2);
            v[i].w = mul_bf16x2(v[i].w, w2);
        }
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int k = h6 + i;
            *reinterpret_cast<uint4 *>(dst + (k >> 2) * kBlk + sw64_offset(row, (uint32_t)(k & 3))) = v[i];
        }
    }
}

// Write 32 fp32 values (raw bits, times mul) as bf16 into row `row` of a
// 64-byte-swizzled block.
__device__ __forceinline__ void write_row_sw64_bits(unsigned char *blk, uint32_t row, const uint32_t (&r)[32],
                                                    float mul) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = pack_bf16x2(__uint_as_float(r[8 * c + 2 * e]) * mul, __uint_as_float(r[8 * c + 2 * e + 1]) * mul);
        *reinterpret_cast<uint4 *>(blk + sw64_offset(row, c)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Write 32 fp32 values as bf16 into row `row` of a 64-byte-swizzled block.
__device__ __forceinline__ void write_row_sw64(unsigned char *blk, uint32_t row, const float (&x)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4 *>(blk + sw64_offset(row, c)) =
            make_uint4(pack_bf16x2(x[8 * c + 0], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                       pack_bf16x2(x[8 * c + 4], x[8 * c + 5]), pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
}

// Packed decay pairs for P, as bf16x2 (low half = column j, high half =
// column j+1), stored at index u + kPairBias for u = -kPairBias..128:
//   forward  pp[u] = (lambda^u, lambda^(u-1)),  u = i - j: columns j, j+1 sit
//            at exponents u, u-1;
//   reverse  pr[u] = (lambda^(u-1), lambda^u),  u = j - i + 1: columns j, j+1
//            sit at exponents u-1, u.
// A negative exponent is the masked side of the diagonal and holds zero, so
// the diagonal block needs no separate mask.
constexpr int kPairBias = 32, kPairLen = 128 + kPairBias + 1;

__device__ __forceinline__ void fill_pair_tables(uint32_t *pp, uint32_t *pr, float l2, int tid, int nthr) {
    for (int i = tid; i < kPairLen; i += nthr) {
        const int u = i - kPairBias;
        const float w = u >= 0 ? decay_pow(l2, u) : 0.f, w1 = u >= 1 ? decay_pow(l2, u - 1) : 0.f;
        pp[i] = pack_bf16x2(w, w1);
        pr[i] = pack_bf16x2(w1, w);
    }
}

// 32 fp32 scores (raw bits, as loaded from TMEM) rounded to 16 bf16 pairs,
// in place in the first 16 entries.
__device__ __forceinline__ void pack_scores(uint32_t (&r)[32]) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) r[e >> 1] = pack_bf16x2(__uint_as_float(r[e]), __uint_as_float(r[e + 1]));
}

// One 32-column block of P for TMEM lane row i, block columns j0..j0+31
// (n0 = i - j0 in both directions), from the scores packed by pack_scores
// (x[0..15]), written as 16 bf16 pairs at taddr: each pair is multiplied by
// its bf16 decay pair in one packed instruction. Only blocks on the kept side
// of the diagonal come here, so every index stays inside the table.
template <bool kRev>
__device__ __forceinline__ void build_p_block(uint32_t (&x)[32], int n0, uint32_t taddr, const uint32_t *pp,
                                              const uint32_t *pr) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const int u = kRev ? e - n0 + 1 : n0 - e;       // table index of columns (e, e+1)
        x[e >> 1] = mul_bf16x2(x[e >> 1], kRev ? pr[u + kPairBias] : pp[u + kPairBias]);
    }
    tmem_st_16cols(taddr, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
}

// Calls f(ks) for the n = C / 16 token steps of a chunk (4 or 8), fully
// unrolled: an MMA issued from a loop with a run-time trip count costs about
// twice the issue time of one whose descriptors are formed from constants.
template <typename F>
__device__ __forceinline__ void for_token_steps(int n, F &&f) {
    if (n == 8) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) f(ks);
    } else {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) f(ks);
    }
}

// One elected thread of a 128-thread group waits on an mbarrier; the verdict
// is published through a two-slot flag so every thread of the group takes
// the same branch after the group's named barrier.
__device__ __forceinline__ bool group_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl,
                                           volatile int *decision, uint32_t gt, uint32_t named, uint32_t &k) {
    if (gt == 0) decision[k & 1] = mbar_wait(bar, parity, ctl) ? 0 : 1;
    named_sync(named, kGroupThreads);
    return decision[(k++) & 1] == 0;
}

__device__ __forceinline__ bool lane0_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl, int lane) {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(bar, parity, ctl) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

}  // namespace tc
}  // namespace gla
