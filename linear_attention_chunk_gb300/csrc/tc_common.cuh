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
            uint32_t *u = reinterpret_cast<uint32_t *>(&v[i]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 f = unpack_bf16x2(u[e]);
                u[e] = pack_bf16x2(f.x * w, f.y * w);
            }
        }
#pragma unroll
        for (int i = 0; i < 6; ++i) {
            const int k = h6 + i;
            *reinterpret_cast<uint4 *>(blk0 + (k >> 2) * kBlk + sw64_offset(row, (uint32_t)(k & 3))) = v[i];
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

// One 32-column block of P for one row, packed to bf16 pairs in TMEM.
// Forward: x_j * lambda^(i - j), kept for j <= i; n0 = i - j0.
// Reverse: x_j * lambda^(j - i), kept for j >= i; n0 = i - j0 as well.
// Only the diagonal block needs the mask.
template <bool kRev>
__device__ __forceinline__ void build_p_block(const uint32_t (&r)[32], int n0, bool diagonal, uint32_t taddr,
                                              const float *pw) {
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const int d0 = kRev ? e - n0 : n0 - e;          // exponent of column e
        const int d1 = kRev ? e + 1 - n0 : n0 - e - 1;  // exponent of column e + 1
        float x0, x1;
        if (!diagonal) {
            x0 = __uint_as_float(r[e]) * pw[d0];
            x1 = __uint_as_float(r[e + 1]) * pw[d1];
        } else {
            x0 = d0 >= 0 ? __uint_as_float(r[e]) * pw[max(d0, 0)] : 0.f;
            x1 = d1 >= 0 ? __uint_as_float(r[e + 1]) * pw[max(d1, 0)] : 0.f;
        }
        pk[e >> 1] = pack_bf16x2(x0, x1);
    }
    tmem_st_16cols(taddr, pk);
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
