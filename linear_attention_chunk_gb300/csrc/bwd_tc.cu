// bwd_tc.cu -- dq and dk of the chunked Simple GLA backward on the tcgen05
// tensor core, sm_103a.
//
// The backward of "Beyond the KV cache: Training and serving i14's Laplace
// 3B linear attention model on AWS Trainium2 with native PyTorch" ("Engineering
// challenges", "Challenge 3: Backward-pass unrolling for a sequential
// recurrence": the gradient passes through every serial state update of the
// chunked form of "Challenge 1"). Per chunk of Cc tokens (0-based i, j):
//   dq_i = s ( lambda^(i+1) S_prev do_i + sum_{j<=i} lambda^(i-j) (do_i.v_j) k_j )
//   dk_j = s sum_{i>=j} lambda^(i-j) (do_i.v_j) q_i + lambda^(Cc-1-j) G v_j
// with S_prev the forward state entering the chunk (S <- lambda^Cc S + sum_j
// lambda^(Cc-1-j) k_j v_j^T, from h0) and G the state gradient leaving it
// (G <- lambda^Cc G + s sum_i lambda^(i+1) q_i do_i^T, from dhT, last chunk
// first).
//
// Both are the chunked recurrence with the roles of the key and value
// dimensions exchanged: a 192-wide score contraction, a 96-wide output and a
// 96 x 192 state. One kernel serves both:
//   dq (forward in time): rows "A" = do, columns "B" = v, values "C" = k,
//                         state S, readout weight lambda^(i+1);
//   dk (reverse in time): rows "A" = v, columns "B" = do, values "C" = q,
//                         state G / s, readout weight lambda^(Cc-1-j).
// Per chunk:
//   score  X  = A B^T                 (K = 192; TMEM [0,128))
//   P      = bf16(X .* D) in place over X (columns [0,64))
//   inter  O1 = A S_prev^T            (K = 192, N = 96; S_prev as a bf16 smem copy)
//   state  S += (w .* C)^T B          (M = 96 padded to 128, N = 192)
//   intra  O2 = P C                   (K = C tokens, N = 96)
//   out    = s (O2 + w_row O1)        -> bf16 -> TMA store
// The row weight of the state update (lambda^(Cc-1-j) forward, lambda^(i+1)
// reverse) goes on the small C tile: a scaled copy C~ = w .* C is made as soon
// as C lands, so A and B are read only by the tensor core.
// One CTA per (b, h), one buffer per tile, each refilled as soon as its
// readers are done: A after the inter MMA, B after the state MMA, C after the
// intra MMA (and the copy). The MMA issuer is a non-blocking event loop.
// Warps: 0 TMA, 1 TMEM + MMA, 2-5 make C~, 6-9 build P, 10-13 state hand-off
// and output epilogue.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tmap.h"

namespace gla {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kDk = 96, kDv = 192;
constexpr int kThreads = 448;
constexpr uint32_t kBarScale = 1, kBarP = 2, kBarE = 3;

constexpr uint32_t kOffA = 0;                       // [C][192]: 6 blocks
constexpr uint32_t kOffB = 6 * kBlk;                // [C][192]: 6 blocks
constexpr uint32_t kOffC = 12 * kBlk;               // [C][96]: 3 blocks
constexpr uint32_t kOffCt = 15 * kBlk;              // C~ = w .* C: 3 blocks + 1 zero block (M pad)
constexpr uint32_t kSbBlk = kDk * 64;               // [96 rows][32 bf16] = 6 KB
constexpr uint32_t kOffSb = 19 * kBlk;              // S_prev copy: 6 blocks of 96 rows
constexpr uint32_t kOffOut = kOffSb + 6 * kSbBlk;   // output staging: 3 blocks
constexpr uint32_t kOffPw = kOffOut + 3 * kBlk;
enum { BAR_FULLAB, BAR_FULLC, BAR_AFREE, BAR_BFREE, BAR_CFREE, BAR_SCORE, BAR_CTREADY, BAR_PREADY, BAR_SBREADY,
       BAR_SFULL, BAR_OFULL, BAR_OEMPTY, BAR_DONE, kNumBars };
constexpr uint32_t kOffPair = kOffPw + 132 * 4;     // pp, pr: packed decay pairs
constexpr uint32_t kOffBar = kOffPair + 2 * 164 * 4;
static_assert(kPairLen <= 164, "pair table stride");
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemUsed = kOffMisc + 32;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512, kColX = 0, kColO2 = 128, kColO1 = 224, kColS = 320;

struct TrArgs {
    const float *log_lambda;
    const float *s0;       // initial state [B,H,96,192] (times init_mul), or NULL
    float scale, init_mul;
    int T, H, C, nck;
    unsigned int *status;
};

template <bool kRev>
__global__ void __launch_bounds__(kThreads, 1)
    gla_bwd_tr_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_o,
                      const TrArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int C = a.C, T = a.T, nck = a.nck;
    const int ksteps_tok = C / 16;

    float *pw = reinterpret_cast<float *>(sm + kOffPw);
    uint32_t *pp = reinterpret_cast<uint32_t *>(sm + kOffPair);
    uint32_t *pr = pp + 164;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    volatile int *dec = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);   // [3][2]
    const WaitCtl ctl{abort_flag, a.status};
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };
    auto natural = [&](int c) { return kRev ? nck - 1 - c : c; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 6; ++i) dec[i] = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
        prefetch_tmap(&tm_c);
        prefetch_tmap(&tm_o);
    }
    {
        const float l2 = log2_of_decay(a.log_lambda[h]);
        for (int n = threadIdx.x; n < 132; n += kThreads) pw[n] = n <= 128 ? decay_pow(l2, n) : 0.f;
        fill_pair_tables(pp, pr, l2, threadIdx.x, kThreads);
    }
    // Zero what TMA never writes: the M-padding block of C~, and for C = 64 the
    // rows 64..127 of every tile block (C~ rows there are made from zero C rows).
    for (uint32_t i = threadIdx.x; i < kBlk / 16; i += kThreads)
        *reinterpret_cast<uint4 *>(sm + kOffCt + 3 * kBlk + i * 16) = make_uint4(0, 0, 0, 0);
    if (C < 128) {
        const uint32_t lo = (uint32_t)C * 64, per_blk = (kBlk - lo) / 16;
        for (uint32_t i = threadIdx.x; i < 15 * per_blk; i += kThreads) {
            const uint32_t blk = i / per_blk, o = lo + (i % per_blk) * 16;
            *reinterpret_cast<uint4 *>(sm + blk * kBlk + o) = make_uint4(0, 0, 0, 0);   // A, B, C blocks
        }
    }
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        // A of chunk c once the inter MMA of c-1 has completed, B once the state
        // MMA of c-1 has (it follows the score and inter MMAs), C once the intra
        // MMA of c-1 (and the copy C~) has.
        const uint32_t tx_ab = 12u * (uint32_t)C * 64u, tx_c = 3u * (uint32_t)C * 64u;
        int nab = 0, nc = 0;   // chunks whose A and B / C loads were issued
        for (int c = 0; c < nck; ++c) {
            const uint32_t ph = (uint32_t)(c - 1) & 1u;   // phase parity of chunk c-1
            const int t0 = natural(c) * C;
            if (c >= 1 && !lane0_wait(bar(BAR_AFREE), ph, ctl, lane)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(BAR_FULLAB), tx_ab);
#pragma unroll
                for (int j = 0; j < 6; ++j) tma_load_4d(base + kOffA + j * kBlk, &tm_a, bar(BAR_FULLAB), 32 * j, h, t0, b);
            }
            __syncwarp();
            nab = c + 1;
            if (c >= 1 && !lane0_wait(bar(BAR_BFREE), ph, ctl, lane)) break;
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < 6; ++j) tma_load_4d(base + kOffB + j * kBlk, &tm_b, bar(BAR_FULLAB), 32 * j, h, t0, b);
            }
            __syncwarp();
            if (c >= 1 && !lane0_wait(bar(BAR_CFREE), ph, ctl, lane)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(BAR_FULLC), tx_c);
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(base + kOffC + j * kBlk, &tm_c, bar(BAR_FULLC), 32 * j, h, t0, b);
            }
            __syncwarp();
            nc = c + 1;
        }
        // Drain: the last loads issued must have landed before the CTA exits (a
        // chunk left half-issued by an abort waits out the 1 ms limit).
        if (lane == 0) {
            if (nab >= 1) mbar_wait_drain(bar(BAR_FULLAB), (uint32_t)(nab - 1) & 1u, 1000000ull);
            if (nc >= 1) mbar_wait_drain(bar(BAR_FULLC), (uint32_t)(nc - 1) & 1u, 1000000ull);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        // Four events per chunk c, each in chunk order, issued as soon as ready:
        //   X(c)   score       tiles A, B landed; O2(c-1) complete (P(c-1) read)
        //   O1(c)  inter       after X(c); S_prev copy ready; O1/O2 drained
        //   ST(c)  state       after O1(c) (so the hand-off that rewrites the
        //                      S_prev copy follows O1's completion); C~ ready
        //   O2(c)  intra       after ST(c); P built
        if (lane == 0) {
            const uint32_t idX = idesc_bf16(128, C, false, false);
            const uint32_t id96 = idesc_bf16(128, kDk, false, false);     // O1: A K-major, S_prev^T K-major
            const uint32_t idO2 = idesc_bf16(128, kDk, false, true);      // O2: P (TMEM), C MN-major
            const uint32_t idS = idesc_bf16(128, kDv, true, true);        // S: C~^T MN-major, B MN-major
            int qx = 0, q1 = 0, qs = 0, q2 = 0;
            uint64_t t_idle = globaltimer_ns();
            uint32_t spins = 0;
            while (q2 < nck) {
                bool progress = false;
                if (qx < nck && qx == q2 && mbar_test(bar(BAR_FULLAB), (uint32_t)qx & 1u) &&
                    (qx == 0 || mbar_test(bar(BAR_OFULL), (uint32_t)(qx - 1) & 1u))) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 12; ++ks) {
                        const uint32_t off = (uint32_t)(ks >> 1) * kBlk + (uint32_t)(ks & 1) * 32;
                        mma_bf16_ss(tmem + kColX, smem_desc(base + kOffA + off, 16, 512, 4),
                                    smem_desc(base + kOffB + off, 16, 512, 4), idX, ks > 0);
                    }
                    mma_commit(bar(BAR_SCORE));
                    ++qx;
                    progress = true;
                }
                if (q1 < qx && mbar_test(bar(BAR_SBREADY), (uint32_t)q1 & 1u) &&
                    (q1 == 0 || mbar_test(bar(BAR_OEMPTY), (uint32_t)(q1 - 1) & 1u))) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 12; ++ks) {
                        const uint32_t off = (uint32_t)(ks >> 1) * kBlk + (uint32_t)(ks & 1) * 32;
                        const uint32_t soff = (uint32_t)(ks >> 1) * kSbBlk + (uint32_t)(ks & 1) * 32;
                        mma_bf16_ss(tmem + kColO1, smem_desc(base + kOffA + off, 16, 512, 4),
                                    smem_desc(base + kOffSb + soff, 16, 512, 4), id96, ks > 0);
                    }
                    mma_commit(bar(BAR_AFREE));
                    ++q1;
                    progress = true;
                }
                if (qs < q1 && mbar_test(bar(BAR_CTREADY), (uint32_t)qs & 1u)) {
                    tc_fence_after();
                    for_token_steps(ksteps_tok, [&](int ks) {
                        mma_bf16_ss(tmem + kColS, smem_desc(base + kOffCt + (uint32_t)ks * 1024, kBlk, 512, 4),
                                    smem_desc(base + kOffB + (uint32_t)ks * 1024, kBlk, 512, 4), idS, 1);
                    });
                    mma_commit(bar(BAR_SFULL));
                    mma_commit(bar(BAR_BFREE));   // B is read by the score and the state MMAs
                    ++qs;
                    progress = true;
                }
                if (q2 < qs && mbar_test(bar(BAR_PREADY), (uint32_t)q2 & 1u)) {
                    tc_fence_after();
                    for_token_steps(ksteps_tok, [&](int ks) {
                        mma_bf16_ts(tmem + kColO2, tmem + kColX + 8u * (uint32_t)ks,
                                    smem_desc(base + kOffC + (uint32_t)ks * 1024, kBlk, 512, 4), idO2, ks > 0);
                    });
                    mma_commit(bar(BAR_OFULL));
                    mma_commit(bar(BAR_CFREE));
                    ++q2;
                    progress = true;
                }
                if (progress) {
                    t_idle = globaltimer_ns();
                    spins = 0;
                } else if ((++spins & 255u) == 0) {
                    if (*abort_flag) break;
                    if (globaltimer_ns() - t_idle > kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicOr(a.status, kDevTimeout);
                        break;
                    }
                }
            }
            // Every MMA issued must be complete before TMEM is released.
            mma_commit(bar(BAR_DONE));
        }
        __syncwarp();
        lane0_wait(bar(BAR_DONE), 0, ctl, lane);
    } else if (warp < 6) {
        // ------------------------ warps 2-5: C~ = w .* C, the state-update operand
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 64;
        uint32_t kw = 0;
        for (int c = 0; c < nck; ++c) {
            const int Cc = min(C, T - natural(c) * C);
            if (!group_wait(bar(BAR_FULLC), (uint32_t)c & 1u, ctl, dec, gt, kBarScale, kw)) break;
            // C~ is a single buffer: the state MMA of chunk c-1 must have read it.
            if (c >= 1 && !group_wait(bar(BAR_SFULL), (uint32_t)(c - 1) & 1u, ctl, dec, gt, kBarScale, kw)) break;
            const float w = kRev ? pw[row + 1] : (row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f);
            scale_rows_to<3>(sm + kOffC, sm + kOffCt, row, w);
            fence_proxy_async_smem();
            named_sync(kBarScale, kGroupThreads);
            if (gt == 0) mbar_arrive(bar(BAR_CTREADY));
        }
    } else if (warp < 10) {
        // --------------------------------------- warps 6-9: P in place over X
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 192;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        const int nblk = C / 32;
        const int diag = (int)quad;
        uint32_t kw = 0;
        for (int c = 0; c < nck; ++c) {
            if (!group_wait(bar(BAR_SCORE), c & 1, ctl, dec + 2, gt, kBarP, kw)) break;
            tc_fence_after();
            // Blocks in increasing order: P block bk lands in columns [16bk, 16bk+16),
            // inside score block bk/2, which this warp has already read (or never needs).
#pragma unroll 1
            for (int bk = 0; bk < nblk; ++bk) {
                const bool keep = kRev ? (bk >= diag) : (bk <= diag);
                if (keep) {
                    uint32_t r[32];
                    tmem_ld_32cols(tl + kColX + 32u * bk, r);
                    tmem_ld_wait();
                    pack_scores(r);
                    build_p_block<kRev>(r, (int)row - 32 * bk, tl + kColX + 16u * bk, pp, pr);
                } else {
                    uint32_t z[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) z[e] = 0u;
                    tmem_st_16cols(tl + kColX + 16u * bk, z);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            named_sync(kBarP, kGroupThreads);
            if (gt == 0) mbar_arrive(bar(BAR_PREADY));
        }
    } else {
        // ------------------------------- warps 10-13: state hand-off, output
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 320;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        uint32_t kw = 0;
        // Initial state: copy = bf16(s0), TMEM S = lambda^C0 * s0 (C0: first chunk processed).
        {
            const float w0 = pw[kRev ? T - (nck - 1) * C : min(C, T)];
            if (quad < 3) {
                const float *src = a.s0 ? a.s0 + (((size_t)b * a.H + h) * kDk + row) * kDv : nullptr;
#pragma unroll 1
                for (int blk = 0; blk < 6; ++blk) {
                    uint32_t r[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float4 v4 = src ? *reinterpret_cast<const float4 *>(src + blk * 32 + e)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                        r[e] = __float_as_uint(v4.x * a.init_mul);
                        r[e + 1] = __float_as_uint(v4.y * a.init_mul);
                        r[e + 2] = __float_as_uint(v4.z * a.init_mul);
                        r[e + 3] = __float_as_uint(v4.w * a.init_mul);
                    }
                    write_row_sw64_bits(sm + kOffSb + blk * kSbBlk, row, r, 1.f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * w0);
                    tmem_st_32cols(tl + kColS + blk * 32, r);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarE, kGroupThreads);
            if (gt == 0) mbar_arrive(bar(BAR_SBREADY));
        }
        for (int c = 0; c < nck; ++c) {
            const int nc = natural(c);
            const int t0 = nc * C;
            const int Cc = min(C, T - t0);
            const bool last = (c == nck - 1);
            if (!group_wait(bar(BAR_SFULL), c & 1, ctl, dec + 4, gt, kBarE, kw)) break;
            tc_fence_after();
            if (!last && quad < 3) {
                const float wn = kRev ? pw[C] : pw[min(C, T - t0 - C)];
#pragma unroll 1
                for (int blk = 0; blk < 6; ++blk) {
                    uint32_t r[32];
                    tmem_ld_32cols(tl + kColS + blk * 32, r);
                    tmem_ld_wait();
                    write_row_sw64_bits(sm + kOffSb + blk * kSbBlk, row, r, 1.f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * wn);
                    tmem_st_32cols(tl + kColS + blk * 32, r);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarE, kGroupThreads);
            if (gt == 0 && !last) mbar_arrive(bar(BAR_SBREADY));

            if (!group_wait(bar(BAR_OFULL), c & 1, ctl, dec + 4, gt, kBarE, kw)) break;
            tc_fence_after();
            if (gt == 0) tma_store_wait_read_all();
            named_sync(kBarE, kGroupThreads);
            {
                const float wr = kRev ? (row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f) : pw[row + 1];
#pragma unroll 1
                for (int blk = 0; blk < 3; ++blk) {
                    uint32_t r2[32], r1[32];
                    tmem_ld_32cols(tl + kColO2 + blk * 32, r2);
                    tmem_ld_32cols(tl + kColO1 + blk * 32, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r2[e] = __float_as_uint(fmaf(wr, __uint_as_float(r1[e]), __uint_as_float(r2[e])));
                    write_row_sw64_bits(sm + kOffOut + blk * kBlk, row, r2, a.scale);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_sync(kBarE, kGroupThreads);
            if (gt == 0) {
                mbar_arrive(bar(BAR_OEMPTY));
#pragma unroll
                for (int blk = 0; blk < 3; ++blk) tma_store_4d(&tm_o, base + kOffOut + blk * kBlk, 32 * blk, h, t0, b);
                tma_store_commit();
            }
        }
        if (gt == 0) tma_store_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <bool kRev>
cudaError_t launch_tr(const void *A, const void *Bt, const void *Ct, void *out, const float *s0, float init_mul,
                      const BwdParams &p, cudaStream_t s, int *launches) {
    CUtensorMap ma, mb, mc, mo;
    cudaError_t e;
    if ((e = make_token_map(&ma, A, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mb, Bt, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mc, Ct, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, out, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gla_bwd_tr_kernel<kRev>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    TrArgs a{p.log_lambda, s0, p.scale, init_mul, p.T, p.H, p.chunk, (p.T + p.chunk - 1) / p.chunk, p.status};
    gla_bwd_tr_kernel<kRev><<<(unsigned)(p.B * p.H), kThreads, kSmemBytes, s>>>(ma, mb, mc, mo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace

// dq: rows do, columns v, values k, state S from h0, forward in time.
cudaError_t launch_bwd_dq_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv) return cudaErrorInvalidValue;
    return launch_tr<false>(p.do_, p.v, p.k, p.dq_out, p.h0, 1.f, p, s, launches);
}

// dk: rows v, columns do, values q, state G / s from dhT / s, reverse in time.
cudaError_t launch_bwd_dk_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv) return cudaErrorInvalidValue;
    return launch_tr<true>(p.v, p.do_, p.q, p.dk_out, p.dhT, 1.f / p.scale, p, s, launches);
}

}  // namespace gla
