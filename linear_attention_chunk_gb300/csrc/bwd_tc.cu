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
// intra MMA (and the copy). The B and C refills each close a chain of the
// chunk period, so all three tiles of the next chunk are prefetched into L2
// a chunk ahead. The MMA issuer is a non-blocking event loop.
// Warps: 0 TMA, 1 TMEM + MMA, 2-5 make C~, 6-9 build P, 10-13 state hand-off
// and output epilogue.
//
// Gated mode (kGate, the per-token decay S_t = exp(g_t) S_{t-1} + k_t v_t^T):
// each lambda power becomes the decay of a run of tokens of the chunk,
// lambda^(i-j) -> exp(G_i - G_j), lambda^(i+1) -> exp(G_i), lambda^(Cc-1-j)
// -> exp(G_last - G_j), lambda^Cc -> exp(G_last), G the running sum of g. The
// first warp of each group (C~, P, epilogue) loads its chunk's gates one
// chunk ahead and scans them into the group's own shared-memory arrays, so
// no group waits on another for them. P's weights are walked along the
// per-token factors exp(g) (leftwards for dq, rightwards for dk). The
// epilogue group also saves the bf16 copy of the state entering every chunk
// (S_prev for dq, G / s for dk) to a workspace slot per (b, h, chunk), from
// which the gate gradient is formed (dg_tc.cu).
#include <cuda.h>

#include "common.cuh"
#include "fwd_full.cuh"
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
// Gated mode: the gate arrays of the C~ group, the P group and (double
// buffered) the epilogue group: [128] float running log2-decays, [128] int
// last clearing positions, [128] float factors exp(g) each.
constexpr uint32_t kGateArr = 128 * 12;
constexpr uint32_t kOffGate = (kSmemUsed + 15) & ~15u;
constexpr uint32_t kSmemBytesGated = kSmemBytes + 4 * kGateArr + 16;
static_assert(kSmemBytesGated <= 232448, "shared memory budget (gated)");
// One saved state copy: 6 blocks of [96 rows][32 bf16], as held in shared memory.
constexpr uint32_t kStateCopyBytes = 6 * kSbBlk;

constexpr uint32_t kTmemCols = 512, kColX = 0, kColO2 = 128, kColO1 = 224, kColS = 320;

struct TrArgs {
    const float *log_lambda;
    const float *s0;       // initial state [B,H,96,192] (times init_mul), or NULL
    float scale, init_mul;
    int T, H, C, nck;
    unsigned int *status;
    // Gated mode: per-token log-decays [B, T, H], and the state copies'
    // workspace, kStateCopyBytes per (b, h, chunk) in natural chunk order.
    const float *g;
    unsigned char *saved;
};

// The kernel body for the chain (b, h) = (unit / H, unit % H), run by warps
// 0-13; a launch of more threads (the paired dk / dv launch below) leaves the
// rest without a role.
template <bool kRev, bool kGate>
__device__ __forceinline__ void tr_body(const CUtensorMap &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_c,
                                        const CUtensorMap &tm_o, const TrArgs &a, int unit) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int b = unit / a.H, h = unit % a.H;
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
    // Gated mode: this lane's four gates (tokens 4 lane .. 4 lane + 3) of
    // chunk c in processing order, 0 past the sequence's end or the last chunk.
    auto load_gates = [&](int c, float (&x)[4]) {
        const int t0 = natural(c) * C, cc = c < nck ? min(C, T - t0) : 0;
        const float *gh = a.g + (size_t)b * T * a.H + h;
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = 4 * lane + r < cc ? gh[(size_t)(t0 + 4 * lane + r) * a.H] : 0.f;
    };
    // Gated mode: group `grp`'s gate arrays (0: C~, 1: P, 2 and 3: epilogue).
    auto gate_arrays = [&](int grp, float *&gl, int *&zc, float *&af) {
        unsigned char *g0 = sm + kOffGate + (uint32_t)grp * kGateArr;
        gl = reinterpret_cast<float *>(g0);
        zc = reinterpret_cast<int *>(g0 + 512);
        af = reinterpret_cast<float *>(g0 + 1024);
    };

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
    if (threadIdx.x < kThreads) {
        if constexpr (!kGate) {   // the gated mode has no per-head decay (log_lambda is NULL)
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
                // The next chunk's tiles into L2, about a chunk ahead of their loads.
                if (c + 1 < nck) {
                    const int t1 = natural(c + 1) * C;
#pragma unroll
                    for (int j = 0; j < 6; ++j) tma_prefetch_4d(&tm_a, 32 * j, h, t1, b);
#pragma unroll
                    for (int j = 0; j < 6; ++j) tma_prefetch_4d(&tm_b, 32 * j, h, t1, b);
#pragma unroll
                    for (int j = 0; j < 3; ++j) tma_prefetch_4d(&tm_c, 32 * j, h, t1, b);
                }
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
        float *Gl, *Af;
        int *Zc;
        gate_arrays(0, Gl, Zc, Af);
        float gpre[4];
        if (kGate && gt < 32) load_gates(0, gpre);
        for (int c = 0; c < nck; ++c) {
            const int Cc = min(C, T - natural(c) * C);
            // gated: scan this chunk's gates (the group's barrier in the wait publishes them)
            if (kGate && gt < 32) {
                gate_scan_store(gpre, lane, Gl, Zc, Af);
                load_gates(c + 1, gpre);
            }
            if (!group_wait(bar(BAR_FULLC), (uint32_t)c & 1u, ctl, dec, gt, kBarScale, kw)) break;
            // C~ is a single buffer: the state MMA of chunk c-1 must have read it.
            if (c >= 1 && !group_wait(bar(BAR_SFULL), (uint32_t)(c - 1) & 1u, ctl, dec, gt, kBarScale, kw)) break;
            float w;
            if constexpr (kGate)   // dk: decay of tokens 0..i; dq: decay of tokens j+1..Cc-1
                w = kRev ? (Zc[row] < 0 ? exp2f(Gl[row]) : 0.f)
                         : (row < (uint32_t)Cc && Zc[Cc - 1] <= (int)row ? exp2f(Gl[Cc - 1] - Gl[row]) : 0.f);
            else
                w = kRev ? pw[row + 1] : (row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f);
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
        float *Gl, *Af;
        int *Zc;
        gate_arrays(1, Gl, Zc, Af);
        float gpre[4];
        if (kGate && gt < 32) load_gates(0, gpre);
        for (int c = 0; c < nck; ++c) {
            if (kGate && gt < 32) {
                gate_scan_store(gpre, lane, Gl, Zc, Af);
                load_gates(c + 1, gpre);
            }
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
                    if constexpr (kGate) {
                        const bool dg = bk == diag;
                        const float gi = Gl[row];
                        if constexpr (kRev) {
                            // row j, columns i >= j: walked rightwards from the block's first column
                            const int il = 32 * bk;
                            const float d0 = dg || Zc[il] > (int)row ? 0.f : ex2_approx(Gl[il] - gi);
                            tmem_ld_wait();
                            build_p_block_gated_rev(r, dg ? lane : -1, il, d0, Af, tl + kColX + 16u * bk);
                        } else {
                            // row i, columns j <= i: walked leftwards from the block's last column
                            const int jr = 32 * bk + 31;
                            const float d0 = dg || Zc[row] > jr ? 0.f : ex2_approx(gi - Gl[jr]);
                            tmem_ld_wait();
                            build_p_block_gated(r, dg ? lane : 32, 32 * bk, d0, Af, tl + kColX + 16u * bk);
                        }
                    } else {
                        tmem_ld_wait();
                        pack_scores(r);
                        build_p_block<kRev>(r, (int)row - 32 * bk, tl + kColX + 16u * bk, pp, pr);
                    }
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
    } else if (warp < 14) {
        // ------------------------------- warps 10-13: state hand-off, output
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 320;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        uint32_t kw = 0;
        // Gated mode: the group's gate arrays for chunks of even / odd processing
        // index; chunk c+1 is scanned at the start of iteration c.
        float *Gls[2], *Afs[2];
        int *Zcs[2];
        gate_arrays(2, Gls[0], Zcs[0], Afs[0]);
        gate_arrays(3, Gls[1], Zcs[1], Afs[1]);
        // decay of the whole chunk whose arrays sit in slot `sl`, Cc tokens long
        auto chunk_decay = [&](int sl, int Cc) { return Zcs[sl][Cc - 1] < 0 ? exp2f(Gls[sl][Cc - 1]) : 0.f; };
        // where the state copy entering chunk c (processing order) is saved
        auto saved_slot = [&](int c) {
            return a.saved + ((size_t)(b * a.H + h) * nck + natural(c)) * kStateCopyBytes;
        };
        float gpre[4];
        if constexpr (kGate) {
            if (gt < 32) {
                load_gates(0, gpre);
                gate_scan_store(gpre, lane, Gls[0], Zcs[0], Afs[0]);
                load_gates(1, gpre);
            }
            named_sync(kBarE, kGroupThreads);
        }
        // Initial state: copy = bf16(s0), TMEM S = lambda^C0 * s0 (C0: first chunk processed).
        {
            const float w0 = kGate ? chunk_decay(0, min(C, T - natural(0) * C))
                                   : pw[kRev ? T - (nck - 1) * C : min(C, T)];
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
            if (kGate && gt == 0) {
                bulk_store(saved_slot(0), base + kOffSb, kStateCopyBytes);
                tma_store_commit();
            }
        }
        for (int c = 0; c < nck; ++c) {
            const int nc = natural(c);
            const int t0 = nc * C;
            const int Cc = min(C, T - t0);
            const bool last = (c == nck - 1);
            if constexpr (kGate) {
                if (gt < 32) {
                    gate_scan_store(gpre, lane, Gls[(c + 1) & 1], Zcs[(c + 1) & 1], Afs[(c + 1) & 1]);
                    load_gates(c + 2, gpre);
                }
                // The saved copy of the state must be read out before the hand-off
                // rewrites it. The bulk groups in flight are the previous copy's and
                // the previous chunk's output (which reads the staging buffer, not the
                // copy): wait for all but the most recent, the output, except before
                // the first chunk, when the initial copy's is the only one.
                if (gt == 0) {
                    if (c == 0)
                        tma_store_wait_read_all();
                    else
                        tma_store_wait_read_1();
                }
            }
            if (!group_wait(bar(BAR_SFULL), c & 1, ctl, dec + 4, gt, kBarE, kw)) break;
            tc_fence_after();
            if (!last && quad < 3) {
                const float wn = kGate ? chunk_decay((c + 1) & 1, min(C, T - natural(c + 1) * C))
                                       : (kRev ? pw[C] : pw[min(C, T - t0 - C)]);
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
            if (kGate && gt == 0 && !last) {
                bulk_store(saved_slot(c + 1), base + kOffSb, kStateCopyBytes);
                tma_store_commit();
            }

            if (!group_wait(bar(BAR_OFULL), c & 1, ctl, dec + 4, gt, kBarE, kw)) break;
            tc_fence_after();
            // The staging buffer's previous store must be read out; in gated mode the
            // state copy's store, committed after it, may stay in flight.
            if (gt == 0) {
                if (kGate && !last)
                    tma_store_wait_read_1();
                else
                    tma_store_wait_read_all();
            }
            named_sync(kBarE, kGroupThreads);
            {
                float wr;
                if constexpr (kGate) {   // dk: decay of tokens j+1..Cc-1; dq: decay of tokens 0..i
                    const float *Gl = Gls[c & 1];
                    const int *Zc = Zcs[c & 1];
                    wr = kRev ? (row < (uint32_t)Cc && Zc[Cc - 1] <= (int)row ? exp2f(Gl[Cc - 1] - Gl[row]) : 0.f)
                              : (Zc[row] < 0 ? exp2f(Gl[row]) : 0.f);
                } else {
                    wr = kRev ? (row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f) : pw[row + 1];
                }
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

template <bool kRev, bool kGate>
__global__ void __launch_bounds__(kThreads, 1)
    gla_bwd_tr_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_o,
                      const TrArgs a) {
    tr_body<kRev, kGate>(tm_a, tm_b, tm_c, tm_o, a, (int)blockIdx.x);
}

// dk and dv of the per-head decay in one launch. Each (b, h) has a dk CTA
// (this file's kernel in reverse time: rows v, columns do, values q) and a dv
// CTA (the one-CTA-per-head kernel of fwd_full.cuh in reverse time: rows k,
// columns q, values do). Both walk the chunks last to first. The CTAs come in
// groups of four, [dk u, dk u+1, dv u, dv u+1] for u = 2 g: CTAs that start
// together read each q and do tile close in time, so the second read is served
// from L2 and q and do leave DRAM once for both gradients. (With [dk u, dv u]
// side by side the launch measured 19 % slower: neighbouring SMs then run
// different code.) An odd B H ends in one group of two, [dk, dv].
constexpr int kPairThreads = 512;
static_assert(kPairThreads >= kThreads && kPairThreads == fullhead::kThreads, "paired launch width");
constexpr uint32_t kPairSmem = kSmemBytes > fullhead::kSmemBytesMax ? kSmemBytes : fullhead::kSmemBytesMax;

template <int kC>
__global__ void __launch_bounds__(kPairThreads, 1)
    gla_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_dk,
                      const __grid_constant__ CUtensorMap tm_row, const __grid_constant__ CUtensorMap tm_col,
                      const __grid_constant__ CUtensorMap tm_val, const __grid_constant__ CUtensorMap tm_dv,
                      const TrArgs ta, const fullhead::FullArgs fa) {
    const int BH = (int)(gridDim.x >> 1), g = (int)(blockIdx.x >> 2), r = (int)(blockIdx.x & 3);
    const bool full_group = 2 * g + 1 < BH;
    const int unit = full_group ? 2 * g + (r & 1) : 2 * g;
    const bool dv = full_group ? (r >> 1) != 0 : (r & 1) != 0;
    if (dv)
        fullhead::full_body<true, kC>(tm_row, tm_col, tm_val, tm_dv, fa, unit);
    else
        tr_body<true, false>(tm_a, tm_b, tm_c, tm_dk, ta, unit);
}

template <bool kRev, bool kGate>
cudaError_t launch_tr(const void *A, const void *Bt, const void *Ct, void *out, const float *s0, float init_mul,
                      const BwdParams &p, unsigned char *saved, cudaStream_t s, int *launches) {
    CUtensorMap ma, mb, mc, mo;
    cudaError_t e;
    if ((e = make_token_map(&ma, A, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mb, Bt, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mc, Ct, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, out, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    const uint32_t smem = kGate ? kSmemBytesGated : kSmemBytes;
    e = cudaFuncSetAttribute(gla_bwd_tr_kernel<kRev, kGate>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    TrArgs a{p.log_lambda, s0, p.scale, init_mul, p.T, p.H, p.chunk, (p.T + p.chunk - 1) / p.chunk, p.status,
             p.g, saved};
    gla_bwd_tr_kernel<kRev, kGate><<<(unsigned)(p.B * p.H), kThreads, smem, s>>>(ma, mb, mc, mo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace

size_t bwd_gated_tc_state_bytes(int B, int T, int H, int chunk) {
    const size_t nck = ((size_t)T + chunk - 1) / chunk;
    return 2 * (size_t)B * H * nck * kStateCopyBytes;
}

// The two halves of state copies, then the gate-gradient kernel's 16-byte
// work counter.
size_t bwd_gated_tc_workspace_size(int B, int T, int H, int chunk) {
    return bwd_gated_tc_state_bytes(B, T, H, chunk) + 16;
}

// dq: rows do, columns v, values k, state S from h0, forward in time. Gated:
// the state copy entering each chunk is saved in the first half of the workspace.
cudaError_t launch_bwd_dq_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv) return cudaErrorInvalidValue;
    if (p.g)
        return launch_tr<false, true>(p.do_, p.v, p.k, p.dq_out, p.h0, 1.f, p,
                                      static_cast<unsigned char *>(p.workspace), s, launches);
    return launch_tr<false, false>(p.do_, p.v, p.k, p.dq_out, p.h0, 1.f, p, nullptr, s, launches);
}

// dk: rows v, columns do, values q, state G / s from dhT / s, reverse in time.
// Gated: the state copy entering each chunk (G / s) is saved in the second half.
cudaError_t launch_bwd_dk_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv) return cudaErrorInvalidValue;
    if (p.g)
        return launch_tr<true, true>(p.v, p.do_, p.q, p.dk_out, p.dhT, 1.f / p.scale, p,
                                     static_cast<unsigned char *>(p.workspace) +
                                         bwd_gated_tc_state_bytes(p.B, p.T, p.H, p.chunk) / 2,
                                     s, launches);
    return launch_tr<true, false>(p.v, p.do_, p.q, p.dk_out, p.dhT, 1.f / p.scale, p, nullptr, s, launches);
}

// dk, dv and dh0 of the per-head decay: one launch of 2 B H CTAs (see
// gla_bwd_kv_kernel). dk: state G / s from dhT / s; dv: the same state,
// written out times s as dh0.
cudaError_t launch_bwd_kv_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv || p.g) return cudaErrorInvalidValue;
    CUtensorMap ma, mb, mc, mdk, mrow, mcol, mval, mdv;
    cudaError_t e;
    if ((e = make_token_map(&ma, p.v, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mb, p.do_, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mc, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mdk, p.dk_out, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mrow, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mcol, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mval, p.do_, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mdv, p.dv_out, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    const TrArgs ta{p.log_lambda, p.dhT, p.scale, 1.f / p.scale, p.T, p.H, p.chunk, nck, p.status, nullptr, nullptr};
    const fullhead::FullArgs fa{p.log_lambda, p.dhT, p.dh0, p.scale, 1.f / p.scale, p.scale, p.T, p.H, nck, 1, nck,
                                p.B * p.H, 0, p.status, nullptr, nullptr, nullptr, 0, nullptr, nullptr};
    auto kernel = p.chunk == 128 ? gla_bwd_kv_kernel<128> : gla_bwd_kv_kernel<64>;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmem)) != cudaSuccess)
        return e;
    kernel<<<(unsigned)(2 * p.B * p.H), kPairThreads, kPairSmem, s>>>(ma, mb, mc, mdk, mrow, mcol, mval, mdv, ta, fa);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
