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
// kStride, kBlk by default) in place by w, six 16-byte chunks at a time (loads
// first, then stores, so the loads overlap). The 64-byte swizzle only permutes
// a row's chunks, so a row is scaled as it lies; chunks are visited in
// swizzled order so that the 32 rows a warp touches at once fall in distinct
// banks.
template <int NB, uint32_t kStride = kBlk>
__device__ __forceinline__ void scale_rows(unsigned char *blk0, uint32_t row, float w) {
    const uint32_t w2 = pack_bf16x2(w, w);
#pragma unroll
    for (int h6 = 0; h6 < 4 * NB; h6 += 6) {
        uint4 v[6];
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int k = h6 + i;
            v[i] = *reinterpret_cast<const uint4 *>(blk0 + (k >> 2) * kStride + sw64_offset(row, (uint32_t)(k & 3)));
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
            *reinterpret_cast<uint4 *>(blk0 + (k >> 2) * kStride + sw64_offset(row, (uint32_t)(k & 3))) = v[i];
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

// ------------------------------------------------------------ gated mode
// The per-token decay of the gated form, S_t = exp(g_t) S_{t-1} + k_t v_t^T:
// every power of a fixed decay becomes the decay of a run of tokens, exp of a
// sum of g inside the chunk.
// A log-decay at or below this clears the state: exp(-80) is below fp32's
// normal range.
constexpr float kResetLogDecay = -80.f;
constexpr float kLog2e = 1.4426950408889634f;

// 2^x for x <= 0 by the hardware approximation (relative error about 2^-22;
// results below fp32's normal range flush to 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Running sums over the C tokens of a chunk, lane l holding tokens 4l..4l+3
// of gate values x[0..3] (natural-log decays; 0 past the chunk's end): the
// log2-decay of tokens 0..t without the clearing gates, gl[t], and the
// position of the last clearing gate among them, zc[t] (-1 if none), for
// t < 128. The decay of tokens j+1..i is then 2^(gl[i] - gl[j]) when
// zc[i] <= j, and 0 otherwise. Also each token's own decay factor, af[t] =
// exp(x) (0 for a clearing gate).
__device__ __forceinline__ void gate_scan_store(const float (&x)[4], int lane, float *gl, int *zc, float *af) {
    float ls[4];
    int lz[4];
    float s = 0.f;
    int z = -1;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (x[r] > kResetLogDecay)
            s += x[r] * kLog2e;
        else
            z = 4 * lane + r;
        ls[r] = s;
        lz[r] = z;
    }
    float si = s;
    int zi = z;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float ys = __shfl_up_sync(0xffffffffu, si, d);
        const int yz = __shfl_up_sync(0xffffffffu, zi, d);
        if (lane >= d) {
            si += ys;
            zi = max(zi, yz);
        }
    }
    const float es = si - s;   // exclusive: the lanes below
    const int ez = __shfl_up_sync(0xffffffffu, zi, 1);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        gl[4 * lane + r] = es + ls[r];
        zc[4 * lane + r] = lz[r] >= 0 ? lz[r] : (lane > 0 ? ez : -1);
    }
    float a[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) a[r] = x[r] > kResetLogDecay ? ex2_approx(x[r] * kLog2e) : 0.f;
    *reinterpret_cast<float4 *>(af + 4 * lane) = make_float4(a[0], a[1], a[2], a[3]);
}

// Gated, forward direction: one 32-column block of P for TMEM lane row i,
// columns j0..j0+31 (j <= i), from the fp32 scores x (raw bits): P_ij =
// A_ij d_ij with d_ij the decay of tokens j+1..i, written as 16 bf16 pairs at
// taddr. The weights
// are walked from the block's right end leftwards, d_i,j-1 = d_ij af[j]: a
// clearing gate's factor 0 zeroes every column left of it. Off the diagonal
// the walk starts from d0 = d_i,j0+31 (one exponential per row, dl = 32); in
// the diagonal block (d0 = 0, dl = i - j0) it starts at the row's own column
// with 1, and the columns right of it stay 0. One copy of this code serves
// every block: the kernel's roles share the instruction cache.
__device__ __forceinline__ void build_p_block_gated(uint32_t (&x)[32], int dl, int j0, float d0, const float *af,
                                                    uint32_t taddr) {
    float d = d0;
#pragma unroll
    for (int m = 7; m >= 0; --m) {
        const float4 a4 = *reinterpret_cast<const float4 *>(af + j0 + 4 * m);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int r = 3; r >= 0; --r) {
            const int e = 4 * m + r;
            d = e == dl ? 1.f : d;
            x[e] = __float_as_uint(__uint_as_float(x[e]) * d);
            d *= av[r];
        }
    }
#pragma unroll
    for (int e = 0; e < 32; e += 2) x[e >> 1] = pack_bf16x2(__uint_as_float(x[e]), __uint_as_float(x[e + 1]));
    tmem_st_16cols(taddr, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
}


// Gated, reverse direction: one 32-column block for TMEM lane row j, columns
// i0..i0+31 (i >= j), P_ji = X_ji d_ji with d_ji the decay of tokens j+1..i,
// written as 16 bf16 pairs at taddr. The weights are walked from the block's
// left end rightwards, d_j,i+1 = d_ji af[i+1]: a clearing gate's factor 0
// zeroes every column right of it. Off the diagonal the walk starts from d0 =
// d_j,i0 (one exponential per row, dl = -1); in the diagonal block (d0 = 0,
// dl = j - i0) it starts at the row's own column with 1, and the columns left
// of it stay 0.
__device__ __forceinline__ void build_p_block_gated_rev(uint32_t (&x)[32], int dl, int i0, float d0,
                                                        const float *af, uint32_t taddr) {
    float d = d0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float4 a4 = *reinterpret_cast<const float4 *>(af + i0 + 4 * m);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int e = 4 * m + r;
            if (e > 0) d *= av[r];
            d = e == dl ? 1.f : d;
            x[e] = __float_as_uint(__uint_as_float(x[e]) * d);
        }
    }
#pragma unroll
    for (int e = 0; e < 32; e += 2) x[e >> 1] = pack_bf16x2(__uint_as_float(x[e]), __uint_as_float(x[e + 1]));
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
