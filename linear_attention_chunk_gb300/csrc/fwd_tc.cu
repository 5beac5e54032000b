// fwd_tc.cu -- chunked Simple GLA forward on the 5th-generation tensor core
// (tcgen05 MMA with TMEM accumulators, TMA-staged bf16 tiles), sm_103a.
//
// The chunked form of "Beyond the KV cache: Training and serving i14's
// Laplace 3B linear attention model on AWS Trainium2 with native PyTorch",
// section "Engineering challenges", "Challenge 1" (equations "Chunked GLA
// intra-chunk output" and "Chunked GLA state update", Figure 3). For a chunk
// of Cc valid tokens entering with state S_prev (0-based i, j inside it):
//   P     = (Q K^T) .* D,   D_ij = lambda^(i-j) for j <= i, else 0
//   O     = scale * ( P V + diag(lambda^(i+1)) Q S_prev )
//   S_new = lambda^Cc S_prev + (diag(lambda^(Cc-1-j)) K)^T V
// Only the state chain is serial; everything inside a chunk is a dense
// contraction.
//
// Work split: one CTA per (b, h, half of dv). Each CTA walks the chunks of
// its sequence in order and keeps its 96 x 96 slice of the fp32 state in
// TMEM for the whole sequence. Sibling CTAs (the two dv halves of one head)
// are adjacent in the grid, so the second read of q and k hits L2. With two
// CTAs per chain, this kernel serves calls with few (sequence, head) chains
// (two CTAs per chain still within one wave), whose chunk period it
// shortens; the one-CTA-per-chain kernel (fwd_full.cuh) serves the rest.
//
// Warp roles (448 threads):
//   warp 0      TMA producer: Q, K, V tiles of chunk c into stage c%2
//   warp 1      TMEM owner and MMA issuer (a non-blocking event loop)
//   warps 2-9   "P group", two warps per TMEM lane quadrant:
//                 sub-group 0 (warps 2-5) scales K in place by lambda^(Cc-1-j)
//                 and signals it at once, then builds the even 32-column
//                 blocks of P = bf16(A .* D);
//                 sub-group 1 (warps 6-9) writes Q~ = diag(lambda^(i+1)) Q into
//                 TMEM and builds the odd blocks of P.
//               P is built with packed bf16x2 multiplies by a table of decay
//               pairs whose zero entries mask the diagonal block. Blocks of P
//               on the masked side of the diagonal are zero and written once.
//   warps 10-13 "E group": the state hand-off (bf16 copy of S for the next
//               chunk's Q~ S, S <- lambda^C' S in TMEM, hT at the end) and the
//               output epilogue (O * scale -> bf16 -> smem -> TMA store)
//
// Gated mode (kGate, a per-token log-decay g in place of log lambda): every
// power of lambda becomes the decay of a run of tokens. The first warp of
// each P sub-group loads its chunk's gates one chunk ahead and scans them
// into running log2-sums, last-clear positions and per-token factors exp(g);
// P's weights are walked along the factors block by block, and sub-group 0
// publishes the chunk's total decay for the E group's rescale of the state.
// The hot per-block loops run one copy of their code: the roles share the
// instruction cache, and the gated kernel was bound by instruction fetch.
//
// TMEM (512 columns): R0, R1 = [0,128), [128,256) hold A = Q K^T of chunk c
// in R[c%2], then that chunk's O (first 96 columns); S = [256,352) fp32;
// P = [352,416) bf16 pairs (A operand of P V); Q~ = [416,464) bf16 pairs (A
// operand of Q~ S_prev). P and Q~ are single buffers, rewritten only after
// the previous chunk's output MMAs have completed.
// The issuer runs three kinds of events per chunk c as soon as their inputs
// are ready (in chunk order within each kind):
//   QK(c)    MMA1  R[c%2]  = Q K^T                (tiles landed, R[c%2] free)
//   ST(c)    MMA4  S      += K~^T V   -> state    (K~ scaled, S rescaled)
//   OUT(c)   MMA2  R[c%2]  = Q~ S_prev
//            MMA3  R[c%2] += P V      -> output   (P built, Q~ scaled)
// with ST(c) before OUT(c); ST(c+1) may run ahead of OUT(c). The serial
// chain per chunk is ST + the state hand-off; P and the output run beside it.
//
// Shared-memory operand layouts (64-byte swizzle, 32-column blocks of
// 128 rows x 64 B): Q, K, V tiles [token][d] are K-major for Q K^T and
// Q~ S and MN-major for the state update (K~^T as A; the fourth dk block of
// K is a zero block, padding dk = 96 to M = 128) and for P V (V as B); the
// bf16 S_prev copy [dk][dv] is an MN-major B operand (96-row blocks,
// double-buffered so the hand-off of chunk c can run while MMA2(c) still
// waits for P).
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

constexpr int kDk = 96, kDv = 192, kDvHalf = 96;
constexpr int kThreads = 448;
constexpr uint32_t kBarP0 = 1, kBarP1 = 2, kBarE = 3;  // named barriers of the three 128-thread groups

constexpr uint32_t kStageQ = 0;                      // 3 blocks
constexpr uint32_t kStageK = 3 * kBlk;               // 4 blocks (the 4th stays zero: dk pad to 128)
constexpr uint32_t kStageV = 7 * kBlk;               // 3 blocks (this CTA's 96 dv columns)
constexpr uint32_t kStageBytes = 10 * kBlk;          // 80 KB
constexpr uint32_t kSbBlk = kDk * 64;                // [96 rows][32 bf16] = 6 KB
constexpr uint32_t kSbBytes = 3 * kSbBlk;
constexpr uint32_t kOffSb = 2 * kStageBytes;         // two S_prev copies
constexpr uint32_t kOffOut = kOffSb + 2 * kSbBytes;  // output staging, 3 blocks
constexpr uint32_t kOffPw = kOffOut + 3 * kBlk;      // lambda^n, n = 0..128 (+pad)
enum { BAR_FULL0, BAR_FULL1, BAR_FULLV0, BAR_FULLV1, BAR_EMPTY0, BAR_EMPTY1, BAR_QK0, BAR_QK1, BAR_KREADY0, BAR_KREADY1,
       BAR_PREADY0, BAR_PREADY1, BAR_SBREADY, BAR_SFULL, BAR_OFULL0, BAR_OFULL1, BAR_OEMPTY0, BAR_OEMPTY1,
       BAR_KFREE0, BAR_KFREE1, BAR_DONE, BAR_GDEC0, BAR_GDEC1, kNumBars };
constexpr uint32_t kOffPair = kOffPw + 132 * 4;     // pp, pr: packed decay pairs
constexpr uint32_t kOffBar = kOffPair + 2 * 164 * 4;
static_assert(kPairLen <= 164, "pair table stride");
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort, 3 x 2 decision slots
constexpr uint32_t kSmemUsed = kOffMisc + 32;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;    // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
// Gated mode: each P sub-group's running sums of the chunk's log2-decays,
// positions of the last state-clearing gate and per-token decay factors,
// [128] float + [128] int + [128] float per sub-group.
constexpr uint32_t kGateSub = 128 * 12;
// ... then two floats: the decay of chunk c in slot c % 2, published by P
// sub-group 0 (BAR_GDEC) for the E group's rescale of the state.
constexpr uint32_t kOffGate = (kSmemUsed + 15) & ~15u, kGateBytes = 2 * kGateSub + 32;
static_assert(kOffGate % 16 == 0, "the decay factors are read as float4");
constexpr uint32_t kSmemBytesGated = kSmemBytes + kGateBytes;
static_assert(kSmemBytesGated <= 232448, "shared memory budget (gated)");
constexpr uint32_t kTmemCols = 512, kColR = 0, kColS = 256, kColP = 352, kColQ = 416;

struct FwdTcArgs {
    const float *log_lambda;
    const float *h0;       // initial state (times init_mul), or NULL
    float *hT;             // final state (times final_mul), or NULL
    float scale;
    float init_mul, final_mul;
    int T, H, C, nck;
    // Sequence segmentation (forward only): the grid covers nseg segments of
    // seg_chunks chunks; segment g starts from h0 + g * h0_seg_stride and only
    // the last segment writes hT. nseg = 1 means one chain per (b, h).
    int nseg, seg_chunks, BH;
    size_t h0_seg_stride;
    unsigned int *status;
    // Variable-length mode (kVar): BH = nseq * H; sequence n holds tokens
    // [cu_seqlens[n], cu_seqlens[n+1]) of the packed [1, T, H, d] tensors, and
    // its state lives in slot slots[n] (n if NULL) of h0 = hT, a [n_slots, H,
    // dk, dv] pool, read at the start and overwritten at the end.
    const int *cu_seqlens;
    const int *slots;
    int n_slots;
    __nv_bfloat16 *o;      // the output, for the masked store of a sequence's last partial chunk
    // Gated mode: per-token log-decays [B, T, H] (natural log) replacing the
    // per-head decay.
    const float *g;
};

// The forward pass (the backward's reverse-time runs use the one-CTA-per-head
// kernel of fwd_full.cuh).
//
// kGate: the per-token decay of the gated form, S_t = exp(g_t) S_{t-1} +
// k_t v_t^T. The lambda powers become decays of token runs: lambda^(i-j) ->
// exp(G_i - G_j), lambda^(i+1) -> exp(G_i), lambda^(Cc-1-j) -> exp(G_last -
// G_j), lambda^Cc -> exp(G_last), G the running sum of the chunk's g. A gate
// at or below kResetLogDecay clears the state: G skips it, and the position
// of the last such gate, kept beside G, gives any run that holds one the
// weight 0.
template <int kC, bool kVar, bool kGate = false>
__global__ void __launch_bounds__(kThreads, 1)
    gla_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const FwdTcArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array by pointer
    // arithmetic so that accesses through it stay shared-memory accesses.
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = blockIdx.x & 1;
    const int seg = (blockIdx.x >> 1) / a.BH;
    const int bh = (blockIdx.x >> 1) % a.BH;
    constexpr int C = kC;   // chunk length, 64 or 128: token loops are unrolled
    const int h = bh % a.H;
    // b: batch index of the states; bt, tok0: token coordinates of the sequence
    int b = bh / a.H, bt = b, tok0 = 0, T = a.T, nck_seq = a.nck;
    if constexpr (kVar) {
        const int n = b, beg = a.cu_seqlens[n], end = a.cu_seqlens[n + 1];
        const int slot = a.slots ? a.slots[n] : n;
        if (beg < 0 || end < beg || end > a.T || slot < 0 || slot >= a.n_slots) {
            if (threadIdx.x == 0) atomicOr(a.status, kDevBadState);
            return;
        }
        if (end == beg) return;   // empty sequence: its state stays as it is
        b = slot;
        bt = 0;
        tok0 = beg;
        T = end - beg;
        nck_seq = (T + C - 1) / C;
    }
    const int cbeg = seg * a.seg_chunks;                          // first chunk of this segment
    const int nck = min(kVar ? nck_seq : a.seg_chunks, nck_seq - cbeg);   // chunks of this CTA
    const bool last_seg = seg == a.nseg - 1;
    const float *h0 = a.h0 ? a.h0 + (size_t)seg * a.h0_seg_stride : nullptr;
    constexpr int ksteps_tok = C / 16;
    // Gated mode: this lane's four gate values (tokens 4 lane .. 4 lane + 3)
    // of chunk c of this CTA, 0 past the sequence's end or the last chunk.
    // Callers load one chunk ahead of use.
    auto load_gates = [&](int c, float (&x)[4]) {
        const int lane4 = 4 * (int)(threadIdx.x & 31);
        const float *gh = a.g + ((size_t)bt * a.T + tok0) * a.H + h;
        const int t0 = (cbeg + c) * C, cc = c < nck ? min(C, T - t0) : 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = lane4 + r < cc ? gh[(size_t)(t0 + lane4 + r) * a.H] : 0.f;
    };

    float *pw = reinterpret_cast<float *>(sm + kOffPw);
    uint32_t *pp = reinterpret_cast<uint32_t *>(sm + kOffPair);
    uint32_t *pr = pp + 164;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    volatile int *dec = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);   // [3][2]
    const WaitCtl ctl{abort_flag, a.status};
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 6; ++i) dec[i] = 0;
        for (int i = 0; i < kNumBars; ++i)
            mbar_init(bar(i), (i == BAR_PREADY0 || i == BAR_PREADY1) ? 2u : 1u);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    if constexpr (!kGate) {   // the gated mode has no per-head decay (log_lambda is NULL)
        const float l2 = log2_of_decay(a.log_lambda[h]);
        for (int n = threadIdx.x; n < 132; n += kThreads) pw[n] = n <= 128 ? decay_pow(l2, n) : 0.f;
        fill_pair_tables(pp, pr, l2, threadIdx.x, kThreads);
    }
    // Zero what TMA never writes: the dk padding block of K (both stages),
    // and for C = 64 the rows 64..127 of every Q, K, V block.
    for (uint32_t i = threadIdx.x; i < 2 * (kBlk / 16); i += kThreads) {
        const uint32_t s = i / (kBlk / 16), o = (i % (kBlk / 16)) * 16;
        st_shared_v4(base + s * kStageBytes + kStageK + 3 * kBlk + o, 0, 0, 0, 0);
    }
    if constexpr (C < 128) {
        const uint32_t lo = (uint32_t)C * 64, per_blk = (kBlk - lo) / 16;
        for (uint32_t i = threadIdx.x; i < 2 * 10 * per_blk; i += kThreads) {
            const uint32_t blk = i / per_blk, o = lo + (i % per_blk) * 16;
            st_shared_v4(base + blk * kBlk + o, 0, 0, 0, 0);   // blocks 0..19 = both stages
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
        // Each tile of stage s is refilled as soon as chunk c-2 is done with it:
        // Q once Q~(c-2) is in TMEM (P ready), K once the state update of c-2
        // has completed, V once the output MMAs of c-2 have completed.
        const uint32_t tx_qk = 6u * (uint32_t)C * 64u, tx_v = 3u * (uint32_t)C * 64u;
        int nq = 0, nv = 0;   // chunks whose Q (and K) / V loads were issued
        for (int c = 0; c < nck; ++c) {
            const int s = c & 1;
            const uint32_t ph = ((c >> 1) - 1) & 1;   // phase parity of chunk c-2
            const uint32_t st = base + (uint32_t)s * kStageBytes;
            const uint32_t fb = bar(BAR_FULL0 + s), fv = bar(BAR_FULLV0 + s);
            const int t0 = (cbeg + c) * C;
            if (c >= 2 && !lane0_wait(bar(BAR_PREADY0 + s), ph, ctl, lane)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, tx_qk);
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(st + kStageQ + j * kBlk, &tm_q, fb, 32 * j, h, tok0 + t0, bt);
            }
            __syncwarp();
            nq = c + 1;
            if (c >= 2 && !lane0_wait(bar(BAR_KFREE0 + s), ph, ctl, lane)) break;
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(st + kStageK + j * kBlk, &tm_k, fb, 32 * j, h, tok0 + t0, bt);
            }
            __syncwarp();
            if (c >= 2 && !lane0_wait(bar(BAR_EMPTY0 + s), ph, ctl, lane)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(fv, tx_v);
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    tma_load_4d(st + kStageV + j * kBlk, &tm_v, fv, kDvHalf * half + 32 * j, h, tok0 + t0, bt);
            }
            __syncwarp();
            nv = c + 1;
        }
        // Drain: every load issued must have landed before the CTA exits (a
        // chunk left half-issued by an abort waits out the 1 ms limit).
        if (lane == 0) {
            for (int c = (nq >= 2 ? nq - 2 : 0); c < nq; ++c)
                mbar_wait_drain(bar(BAR_FULL0 + (c & 1)), (c >> 1) & 1, 1000000ull);
            for (int c = (nv >= 2 ? nv - 2 : 0); c < nv; ++c)
                mbar_wait_drain(bar(BAR_FULLV0 + (c & 1)), (c >> 1) & 1, 1000000ull);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------- MMA issuer (event loop)
        if (lane == 0) {
            const uint32_t idA = idesc_bf16(128, C, false, false);
            const uint32_t idO = idesc_bf16(128, kDvHalf, false, true);
            const uint32_t idS = idesc_bf16(128, kDvHalf, true, true);
            int q1 = 0, q4 = 0, q23 = 0;   // next chunk of each event kind
            uint64_t t_idle = globaltimer_ns();
            uint32_t spins = 0;
            while (q23 < nck) {
                bool progress = false;
                // ST(c): S += K~^T V once K~ is scaled and S rescaled. It may run ahead
                // of OUT(c-1): the hand-off that follows it rewrites the S_prev copy
                // OUT(c-1) reads only after the epilogue group has seen OUT(c-1) complete.
                if (q4 < q1) {
                    const int c = q4, s = c & 1;
                    if (mbar_test(bar(BAR_KREADY0 + s), (c >> 1) & 1) && mbar_test(bar(BAR_SBREADY), c & 1) &&
                        mbar_test(bar(BAR_FULLV0 + s), (c >> 1) & 1)) {
                        tc_fence_after();
                        const uint32_t st = base + (uint32_t)s * kStageBytes;
#pragma unroll
                        for (int ks = 0; ks < ksteps_tok; ++ks)
                            mma_bf16_ss(tmem + kColS, smem_desc(st + kStageK + (uint32_t)ks * 1024, kBlk, 512, 4),
                                        smem_desc(st + kStageV + (uint32_t)ks * 1024, kBlk, 512, 4), idS, 1);
                        mma_commit(bar(BAR_SFULL));
                        mma_commit(bar(BAR_KFREE0 + s));
                        ++q4;
                        progress = true;
                    }
                }
                // QK(c): tiles landed and R[c%2] released by the epilogue of chunk c-2
                if (q1 < nck) {
                    const int c = q1, s = c & 1;
                    if (mbar_test(bar(BAR_FULL0 + s), (c >> 1) & 1) &&
                        (c < 2 || mbar_test(bar(BAR_OEMPTY0 + s), ((c - 2) >> 1) & 1))) {
                        tc_fence_after();
                        const uint32_t st = base + (uint32_t)s * kStageBytes;
#pragma unroll
                        for (int ks = 0; ks < 6; ++ks) {
                            const uint32_t off = (uint32_t)(ks >> 1) * kBlk + (uint32_t)(ks & 1) * 32;
                            mma_bf16_ss(tmem + kColR + 128u * s, smem_desc(st + kStageQ + off, 16, 512, 4),
                                        smem_desc(st + kStageK + off, 16, 512, 4), idA, ks > 0);
                        }
                        mma_commit(bar(BAR_QK0 + s));
                        ++q1;
                        progress = true;
                    }
                }
                // OUT(c): O = Q~ S_prev + P V once P is built and Q~ scaled
                if (q23 < q4) {
                    const int c = q23, s = c & 1;
                    if (mbar_test(bar(BAR_PREADY0 + s), (c >> 1) & 1)) {
                        tc_fence_after();
                        const uint32_t st = base + (uint32_t)s * kStageBytes;
                        const uint32_t dR = tmem + kColR + 128u * s;
                        const uint32_t sb = base + kOffSb + (uint32_t)s * kSbBytes;
#pragma unroll
                        for (int ks = 0; ks < 6; ++ks)
                            mma_bf16_ts(dR, tmem + kColQ + 8u * (uint32_t)ks,
                                        smem_desc(sb + (uint32_t)ks * 1024, kSbBlk, 512, 4), idO, ks > 0);
#pragma unroll
                        for (int ks = 0; ks < ksteps_tok; ++ks)
                            mma_bf16_ts(dR, tmem + kColP + 8u * (uint32_t)ks,
                                        smem_desc(st + kStageV + (uint32_t)ks * 1024, kBlk, 512, 4), idO, 1);
                        mma_commit(bar(BAR_OFULL0 + s));
                        mma_commit(bar(BAR_EMPTY0 + s));
                        ++q23;
                        progress = true;
                    }
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
    } else if (warp < 10) {
        // ------------------------------------------------- P group (2..9)
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t sub = (uint32_t)(warp - 2) >> 2;            // 0: K + even blocks, 1: Q + odd blocks
        const uint32_t row = quad * 32 + (uint32_t)lane;          // TMEM lane = token row
        const uint32_t gt = (uint32_t)threadIdx.x - 64 - 128 * sub;  // 0..127 within the sub-group
        const uint32_t named = sub ? kBarP1 : kBarP0;
        volatile int *mydec = dec + 2 * sub;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        const int nblk = C / 32;
        const int diag = (int)quad;                               // block holding this warp's diagonal
        uint32_t kw = 0;
        // P blocks above the diagonal are zero for every chunk: write them once.
        {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
            for (int blk = (int)sub; blk < 4; blk += 2) {
                if (blk <= diag) continue;
                tmem_st_16cols(tl + kColP + 16u * blk, z);
            }
            tmem_st_wait();
        }
        // Gated mode: the sub-group's running sums; its first warp scans each
        // chunk's gates, loaded one chunk ahead into registers.
        float *Gl = reinterpret_cast<float *>(sm + kOffGate + sub * kGateSub);
        int *Zc = reinterpret_cast<int *>(sm + kOffGate + sub * kGateSub + 512);
        float *Af = reinterpret_cast<float *>(sm + kOffGate + sub * kGateSub + 1024);
        float gpre[4];
        if constexpr (kGate) {
            if (gt < 32) load_gates(0, gpre);
        }
        for (int c = 0; c < nck; ++c) {
            const int s = c & 1;
            const int Cc = min(C, T - (cbeg + c) * C);
            if constexpr (kGate) {
                // Every thread of the sub-group is past chunk c-1's reads (the
                // barrier before its P-ready signal); the named barrier in the
                // wait below publishes these sums to the sub-group.
                if (gt < 32) {
                    gate_scan_store(gpre, (int)gt, Gl, Zc, Af);
                    load_gates(c + 1, gpre);
                    if (sub == 0) {
                        // the chunk's decay for the E group's rescale of the state
                        __syncwarp();
                        if (gt == 0) {
                            float *slot = reinterpret_cast<float *>(sm + kOffGate + 2 * kGateSub) + s;
                            *slot = Zc[Cc - 1] < 0 ? exp2f(Gl[Cc - 1]) : 0.f;
                            mbar_arrive(bar(BAR_GDEC0 + s));
                        }
                    }
                }
            }
            if (!group_wait(bar(BAR_QK0 + s), (c >> 1) & 1, ctl, mydec, gt, named, kw)) break;
            tc_fence_after();
            if (sub == 0) {
                // K~ = diag(w) K with w = lambda^(Cc-1-j) (zero past the end of the
                // sequence); signalled at once.
                float wk;
                if constexpr (kGate)   // the decay of tokens j+1..Cc-1
                    wk = row < (uint32_t)Cc && Zc[Cc - 1] <= (int)row ? exp2f(Gl[Cc - 1] - Gl[row]) : 0.f;
                else
                    wk = row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f;
                scale_rows<3>(sm + (uint32_t)s * kStageBytes + kStageK, row, wk);
                fence_proxy_async_smem();
                named_sync(named, kGroupThreads);
                if (gt == 0) mbar_arrive(bar(BAR_KREADY0 + s));
            }
            // P and Q~ live in single TMEM buffers: the previous chunk's output
            // MMAs (their only readers) must have completed before they change.
            if (c >= 1 && !group_wait(bar(BAR_OFULL0 + (s ^ 1)), ((c - 1) >> 1) & 1, ctl, mydec, gt, named, kw))
                break;
            tc_fence_after();
            if (sub == 1) {
                // Q~ = diag(lambda^(i+1)) Q into TMEM as the A operand of Q~ S_prev:
                // lane = token row, column c = dk pair (2c, 2c+1).
                float wq;
                if constexpr (kGate)   // the decay of the chunk's tokens 0..i
                    wq = Zc[row] < 0 ? exp2f(Gl[row]) : 0.f;
                else
                    wq = pw[row + 1];
                const uint32_t wq2 = pack_bf16x2(wq, wq);
                const unsigned char *qt = sm + (uint32_t)s * kStageBytes + kStageQ;
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    uint32_t pk[16];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(qt + j * kBlk + sw64_offset(row, cc));
                        pk[4 * cc + 0] = mul_bf16x2(v.x, wq2);
                        pk[4 * cc + 1] = mul_bf16x2(v.y, wq2);
                        pk[4 * cc + 2] = mul_bf16x2(v.z, wq2);
                        pk[4 * cc + 3] = mul_bf16x2(v.w, wq2);
                    }
                    tmem_st_16cols(tl + kColQ + 16u * j, pk);
                }
            }
            // P = bf16((Q K^T) .* D) for this sub-group's blocks on the kept side of the
            // diagonal (at most two per warp), one block at a time through one copy of the code.
            // Tokens past the end of a ragged chunk have zero q and k, so A is zero there.
            {
                const int b0 = (int)sub, b1 = (int)sub + 2;
                const bool has0 = b0 < nblk && b0 <= diag;
                const bool has1 = b1 < nblk && b1 <= diag;
                if constexpr (kGate) {
                    const float gi = Gl[row];
                    const int zi = Zc[row];
#pragma unroll 1
                    for (int blk = b0; blk <= b1; blk += 2) {
                        if (blk == b0 ? !has0 : !has1) continue;
                        uint32_t x[32];
                        tmem_ld_32cols(tl + kColR + 128u * s + 32u * blk, x);
                        const bool dg = blk == diag;
                        const int jr = 32 * blk + 31;   // the block's last column
                        const float d0 = dg || zi > jr ? 0.f : ex2_approx(gi - Gl[jr]);
                        tmem_ld_wait();
                        build_p_block_gated(x, dg ? lane : 32, 32 * blk, d0, Af, tl + kColP + 16u * blk);
                    }
                } else {
#pragma unroll 1
                    for (int blk = b0; blk <= b1; blk += 2) {
                        if (blk == b0 ? !has0 : !has1) continue;
                        uint32_t x[32];
                        tmem_ld_32cols(tl + kColR + 128u * s + 32u * blk, x);
                        tmem_ld_wait();
                        pack_scores(x);
                        build_p_block<false>(x, (int)row - 32 * blk, tl + kColP + 16u * blk, pp, pr);
                    }
                }
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(named, kGroupThreads);
            if (gt == 0) mbar_arrive(bar(BAR_PREADY0 + s));
        }
    } else {
        // ------------------------------------------------- E group (10..13)
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 320;           // 0..127
        volatile int *mydec = dec + 4;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        uint32_t kw = 0;
        // Initial state: S_prev copy 0 = bf16(h0 slice), TMEM S = lambda^C0 * h0,
        // with C0 the length of the first chunk processed.
        // gated mode: chunk decays published by P sub-group 0, slot c % 2
        const volatile float *dslot = reinterpret_cast<const volatile float *>(sm + kOffGate + 2 * kGateSub);
        {
            float w0 = 1.f;
            if constexpr (kGate) {
                if (group_wait(bar(BAR_GDEC0), 0, ctl, mydec, gt, kBarE, kw)) w0 = dslot[0];
            } else {
                w0 = pw[min(C, T - cbeg * C)];
            }
            if (quad < 3) {
                const float *src =
                    h0 ? h0 + (((size_t)b * a.H + h) * kDk + row) * kDv + kDvHalf * half : nullptr;
#pragma unroll
                for (int blk = 0; blk < 3; ++blk) {
                    float x[32];
                    uint32_t r[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float4 v4 = src ? *reinterpret_cast<const float4 *>(src + blk * 32 + e)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                        x[e] = v4.x * a.init_mul; x[e + 1] = v4.y * a.init_mul;
                        x[e + 2] = v4.z * a.init_mul; x[e + 3] = v4.w * a.init_mul;
                    }
                    write_row_sw64(sm + kOffSb + blk * kSbBlk, row, x);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(x[e] * w0);
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
            const int s = c & 1;
            const int t0 = (cbeg + c) * C;
            // State hand-off (rows 0..95 = quadrants 0..2).
            if (!group_wait(bar(BAR_SFULL), c & 1, ctl, mydec, gt, kBarE, kw)) break;
            tc_fence_after();
            const bool last = (c == nck - 1);
            float wgate = 1.f;   // gated mode: the decay of chunk c+1
            if constexpr (kGate) {
                if (!last) {
                    const int cn = c + 1;
                    if (!group_wait(bar(BAR_GDEC0 + (cn & 1)), (cn >> 1) & 1, ctl, mydec, gt, kBarE, kw)) break;
                    wgate = dslot[cn & 1];
                }
            }
            if (quad < 3) {
                // rescale by lambda^(length of the next chunk processed)
                const float wn = last ? 1.f : (kGate ? wgate : pw[min(C, T - t0 - C)]);
                unsigned char *sb_next = sm + kOffSb + (uint32_t)(s ^ 1) * kSbBytes;
                float *dst = (last && last_seg && a.hT)
                                 ? a.hT + (((size_t)b * a.H + h) * kDk + row) * kDv + kDvHalf * half
                                 : nullptr;
                // Three 32-column blocks through one copy of the code at C = 128 (the
                // roles share the instruction cache).
                auto handle = [&](uint32_t (&r)[32], int blk) {
                    if (last) {
                        if (dst) {
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                *reinterpret_cast<float4 *>(dst + blk * 32 + e) = make_float4(
                                    __uint_as_float(r[e]) * a.final_mul, __uint_as_float(r[e + 1]) * a.final_mul,
                                    __uint_as_float(r[e + 2]) * a.final_mul, __uint_as_float(r[e + 3]) * a.final_mul);
                        }
                    } else {
                        write_row_sw64_bits(sb_next + blk * kSbBlk, row, r, 1.f);
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * wn);
                        tmem_st_32cols(tl + kColS + blk * 32, r);
                    }
                };
                if constexpr (C < 128) {
                    // short chunks: the hand-off is a larger share of the chunk's
                    // period, so the next block's TMEM load overlaps this one's work
                    uint32_t ra[32], rb[32];
                    tmem_ld_32cols(tl + kColS, ra);
                    tmem_ld_wait();
                    tmem_ld_32cols(tl + kColS + 32, rb);
                    handle(ra, 0);
                    tmem_ld_wait();
                    tmem_ld_32cols(tl + kColS + 64, ra);
                    handle(rb, 1);
                    tmem_ld_wait();
                    handle(ra, 2);
                } else {
#pragma unroll 1
                    for (int blk = 0; blk < 3; ++blk) {
                        uint32_t r[32];
                        tmem_ld_32cols(tl + kColS + 32u * blk, r);
                        tmem_ld_wait();
                        handle(r, blk);
                    }
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarE, kGroupThreads);
            if (gt == 0 && !last) mbar_arrive(bar(BAR_SBREADY));

            // Output tile: O * scale -> bf16 -> staging -> TMA store. A partial last
            // chunk of a packed variable-length sequence is stored row by row
            // instead: its tile would overlap the next sequence's rows.
            if (!group_wait(bar(BAR_OFULL0 + s), (c >> 1) & 1, ctl, mydec, gt, kBarE, kw)) break;
            tc_fence_after();
            const bool rowwise = kVar && T - t0 < C;
            if (!rowwise) {
                if (gt == 0) tma_store_wait_read_all();   // staging free (store of chunk c-1 read it)
                named_sync(kBarE, kGroupThreads);
            }
            {
                const uint32_t src = tl + kColR + 128u * s;
                __nv_bfloat16 *orow =
                    kVar ? a.o + ((size_t)(tok0 + t0 + (int)row) * a.H + h) * kDv + kDvHalf * half : nullptr;
                const bool row_in = (int)row < T - t0;
                auto handle = [&](const uint32_t (&r)[32], int blk) {
                    if (!rowwise) {
                        write_row_sw64_bits(sm + kOffOut + blk * kBlk, row, r, a.scale);
                    } else if (row_in) {
#pragma unroll
                        for (int e = 0; e < 32; e += 8)
                            *reinterpret_cast<uint4 *>(orow + 32 * blk + e) = make_uint4(
                                pack_bf16x2(__uint_as_float(r[e]) * a.scale, __uint_as_float(r[e + 1]) * a.scale),
                                pack_bf16x2(__uint_as_float(r[e + 2]) * a.scale, __uint_as_float(r[e + 3]) * a.scale),
                                pack_bf16x2(__uint_as_float(r[e + 4]) * a.scale, __uint_as_float(r[e + 5]) * a.scale),
                                pack_bf16x2(__uint_as_float(r[e + 6]) * a.scale, __uint_as_float(r[e + 7]) * a.scale));
                    }
                };
                if constexpr (C < 128) {
                    uint32_t ra[32], rb[32];
                    tmem_ld_32cols(src, ra);
                    tmem_ld_wait();
                    tmem_ld_32cols(src + 32, rb);
                    handle(ra, 0);
                    tmem_ld_wait();
                    tmem_ld_32cols(src + 64, ra);
                    handle(rb, 1);
                    tmem_ld_wait();
                    handle(ra, 2);
                } else {
#pragma unroll 1
                    for (int blk = 0; blk < 3; ++blk) {
                        uint32_t r[32];
                        tmem_ld_32cols(src + 32u * blk, r);
                        tmem_ld_wait();
                        handle(r, blk);
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_sync(kBarE, kGroupThreads);
            if (gt == 0) {
                mbar_arrive(bar(BAR_OEMPTY0 + s));
                if (!rowwise) {
#pragma unroll
                    for (int blk = 0; blk < 3; ++blk)
                        tma_store_4d(&tm_o, base + kOffOut + blk * kBlk, kDvHalf * half + 32 * blk, h, tok0 + t0, bt);
                    tma_store_commit();
                }
            }
        }
        if (gt == 0) tma_store_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// One launch of the dv-half chunk kernel: `qm`, `km` are [B,T,H,96] maps,
// `vm` and `om` [B,T,H,192] maps (box height = chunk).
template <bool kGate>
cudaError_t launch_chunk_kernel(const CUtensorMap &qm, const CUtensorMap &km, const CUtensorMap &vm,
                                const CUtensorMap &om, const FwdTcArgs &a, int B, cudaStream_t s, int *launches) {
    auto kernel = a.C == 128 ? gla_fwd_tc_kernel<128, false, kGate> : gla_fwd_tc_kernel<64, false, kGate>;
    const uint32_t smem = kGate ? kSmemBytesGated : kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<(unsigned)(B * a.H * 2), kThreads, smem, s>>>(qm, km, vm, om, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

// The forward with two CTAs per (b, h) chain, one per half of the value
// columns: for few chains, whose chunk period the halved state shortens.
cudaError_t launch_fwd_half_tc(const FwdParams &p, cudaStream_t s, int *launches) {
    CUtensorMap mq, mk, mv, mo;
    cudaError_t e;
    if ((e = make_token_map(&mq, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mk, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, p.o, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    const FwdTcArgs a{p.log_lambda, p.h0, p.hT, p.scale, 1.f, 1.f, p.T, p.H, p.chunk, nck, 1, nck, p.B * p.H, 0,
                      p.status, nullptr, nullptr, 0, nullptr, p.g};
    return p.g ? launch_chunk_kernel<true>(mq, mk, mv, mo, a, p.B, s, launches)
               : launch_chunk_kernel<false>(mq, mk, mv, mo, a, p.B, s, launches);
}

}  // namespace

size_t fwd_tc_workspace_size(int B, int T, int H, int chunk, bool gated) {
    return seg_workspace_bytes(B, H, plan_segments(B, T, H, chunk), gated);
}

cudaError_t launch_fwd_tc(const FwdParams &p, cudaStream_t s, int *launches, const EpilogueParams *epi) {
    if (p.dk != kDk || p.dv != kDv || (epi && p.g)) return cudaErrorInvalidValue;
    // One CTA holds the whole state of a (b, h) chain. Few chains and a long
    // sequence: split each sequence into segments that run in parallel, when
    // the caller gave the workspace for it. Few chains otherwise (two CTAs per
    // chain still within one wave): two CTAs per chain, each half the state.
    const SegPlan plan = plan_segments(p.B, p.T, p.H, p.chunk);
    const bool segmented =
        plan.nseg > 1 && p.workspace && p.workspace_bytes >= seg_workspace_bytes(p.B, p.H, plan, p.g != nullptr);
    const bool half = !segmented && 2L * p.B * p.H <= device_sm_count();
    // The mixer epilogue's normalisation rides in the one-CTA-per-chain
    // kernel's output stage at C = 128, the rest follows as a light pass;
    // otherwise the whole epilogue follows the forward as its own launch.
    const bool fused = epi && !half && p.chunk == 128;
    cudaError_t e;
    if (half) {
        e = launch_fwd_half_tc(p, s, launches);
    } else if (!segmented) {
        e = launch_fwd_full_tc(p, nullptr, 1, 0, s, launches, fused ? epi : nullptr);
    } else {
        float *S_in = nullptr;
        e = launch_seg_prologue(p, plan, &S_in, s, launches);
        if (e == cudaSuccess)
            e = launch_fwd_full_tc(p, S_in, plan.nseg, plan.seg_chunks, s, launches, fused ? epi : nullptr);
    }
    if (e == cudaSuccess && epi)
        e = fused ? launch_mixer_finish(*epi, s, launches) : launch_mixer_epilogue(*epi, true, s, launches);
    return e;
}

// Variable-length forward over the packed [1, total_T, H, d] tensors; states
// in the pool.
cudaError_t launch_fwd_varlen_tc(const VarlenParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv) return cudaErrorInvalidValue;
    // More chains than half the SMs: one CTA per (sequence, head) holds the
    // whole state; fewer: two per chain, each half the state.
    if (2L * p.nseq * p.H > device_sm_count()) return launch_fwd_varlen_full_tc(p, s, launches);
    CUtensorMap mq, mk, mv, mo;
    cudaError_t e;
    if ((e = make_token_map(&mq, p.q, 1, p.total_T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mk, p.k, 1, p.total_T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, 1, p.total_T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mo, p.o, 1, p.total_T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    FwdTcArgs a{p.log_lambda, p.pool, p.pool, p.scale, 1.f, 1.f, p.total_T, p.H, p.chunk, 0, 1, 0, p.nseq * p.H, 0,
                p.status, p.cu_seqlens, p.slots, p.n_slots, static_cast<__nv_bfloat16 *>(p.o), p.g};
    // gated: per-token log-decays [total_T, H] packed like q
    auto kernel = p.g ? (p.chunk == 128 ? gla_fwd_tc_kernel<128, true, true> : gla_fwd_tc_kernel<64, true, true>)
                      : (p.chunk == 128 ? gla_fwd_tc_kernel<128, true> : gla_fwd_tc_kernel<64, true>);
    const uint32_t smem = p.g ? kSmemBytesGated : kSmemBytes;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    kernel<<<(unsigned)(p.nseq * p.H * 2), kThreads, smem, s>>>(mq, mk, mv, mo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
