// fwd_full.cuh -- the chunked Simple GLA forward with one CTA per (b, h): the
// whole 96 x 192 state in one CTA, on the 5th-generation tensor core
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
//
// The dv-half kernel (fwd_tc.cu) gives each head two CTAs, which each form
// Q K^T and P for their half of the value columns: a layer of 128 heads is
// 256 CTAs, 1.7 waves of one CTA per SM on 152 SMs, the second wave leaving
// 48 SMs idle. Here one CTA holds the whole state (192 TMEM columns), so
// such a layer is one wave of 128 CTAs and Q K^T is formed once per head.
// Fitting the whole head into one SM's TMEM and shared memory:
//   TMEM (512 columns): AP = [0, 128) holds A = Q K^T (C columns), then P
//     built in place over it (bf16 pairs in columns [0, C/2)) and Q~ =
//     diag(lambda^(i+1)) Q (columns [64, 112)), the A operands of the output
//     MMAs; O = [128, 320) the output accumulator; S = [320, 512) the fp32
//     state, rows 0..95.
//   Shared memory (the Layout below): Q in one buffer; K and V in two
//     stages; one bf16 copy of S_prev (the B operand of Q~ S_prev); the
//     output of chunk c staged in the V slot of its own stage once the state
//     and output MMAs have read V. At C = 64 the tiles take half the bytes,
//     and two S_prev copies and two output buffers take the room (kDual).
//   One P-group warp per TMEM lane quadrant owns its 32 token rows, so P
//     can overwrite the score columns that warp has already read. At C = 64
//     the score, P, Q~ and output tiles are M = 64 (lanes 0-15 of each
//     quadrant).
// Warps (16, 512 threads; a warp reaches the TMEM lanes of quadrant warp % 4):
//   15          TMA producer
//   3           TMEM owner and MMA issuer (a non-blocking event loop)
//   4-7         P group: its rows of Q to registers as soon as Q lands (Q's
//               single buffer is then free once QK has read it; the producer
//               has already prefetched the next tile into L2), K~ =
//               diag(lambda^(Cc-1-j)) K in place (signalled at once), P =
//               bf16(A .* D) by packed bf16x2 multiplies with a table of decay
//               pairs whose zeros mask the diagonal block, then Q~ into TMEM
//   8-11        E group: output epilogue (O * scale -> bf16 -> V slot -> TMA store)
//   12-14, 0-2  H group (quadrants 0-2, the state's 96 rows; the first three
//               warps take column blocks 0-2, the last three 3-5): the state
//               hand-off (bf16 copy of S for the next chunk's Q~ S, S <-
//               lambda^C' S) and hT
// Per chunk c the MMA issuer runs, in order, as soon as their inputs are ready:
//   QK(c)   A = Q K^T               (tiles landed; OUT(c-1) complete: AP free)
//   ST(c)   S += K~^T V             (K~ scaled; hand-off of c-1 done)
//   OUT(c)  O = Q~ S_prev + P V     (P, Q~ in TMEM; epilogue of c-1 has read O)
// The hand-off of chunk c follows ST(c) and (with one S_prev copy) OUT(c).
// Modes (template flags of full_body): reverse time (the backward's dv), the
// per-token decay, and the packed variable-length prefill into a state pool;
// a segmented long sequence runs one CTA per (segment, b, h).
//
// The kernel body is a device function so that one launch can run it beside
// another body on a neighbouring CTA (the backward's dk and dv, bwd_tc.cu).
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tc_common.cuh"
#include "tmap.h"

namespace gla {
namespace fullhead {
namespace {

using namespace ptx;
using namespace tc;

constexpr int kDk = 96, kDv = 192;
constexpr int kThreads = 512;
constexpr uint32_t kBarP = 1, kBarE = 2, kBarH = 3;   // named barriers of the three groups
constexpr uint32_t kHThreads = 192;

constexpr uint32_t kSbBlk = kDk * 64;                // S_prev copy: [96 rows][32 bf16] blocks, 6 KB
constexpr uint32_t kSbBytes = 6 * kSbBlk;            // 36 KB
enum { BAR_FULLQ, BAR_FULLK0, BAR_FULLK1, BAR_FULLV0, BAR_FULLV1, BAR_QFREE, BAR_KFREE0, BAR_KFREE1, BAR_VFREE0,
       BAR_VFREE1, BAR_QKDONE, BAR_KREADY, BAR_PREADY, BAR_SBREADY, BAR_SFULL, BAR_OFULL, BAR_OEMPTY, BAR_DONE,
       kNumBars };
static_assert(kPairLen <= 164, "pair table stride");
constexpr uint32_t kGateArr = 128 * 12;

// Shared-memory layout for chunk length kC. Token tiles are blocks of
// [kC rows][32 bf16] (kC * 64 bytes, 64-byte swizzle): Q 3 blocks; two stages
// of K (3 blocks) then V (6 blocks), so K~^T's fourth (pad) M block reads V's
// first; the S_prev copy. At kC = 64 the tiles take half the bytes, and the
// room holds a second S_prev copy and two output staging buffers, so that
// neither the state hand-off nor the V slot waits for the output (kDual).
template <int kC>
struct Layout {
    static constexpr bool kDual = kC == 64;
    static constexpr uint32_t kB = (uint32_t)kC * 64;          // one tile block
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffStage = 3 * kB;
    static constexpr uint32_t kStK = 0, kStV = 3 * kB;
    static constexpr uint32_t kStageBytes = 9 * kB;
    static constexpr uint32_t kOffSb = kOffStage + 2 * kStageBytes;
    static constexpr uint32_t kNSb = kDual ? 2 : 1;
    static constexpr uint32_t kOutBytes = 6 * kB;              // kDual: output staging, two buffers
    static constexpr uint32_t kOffOut = kOffSb + kNSb * kSbBytes;
    static constexpr uint32_t kOffPw = kOffOut + (kDual ? 2 * kOutBytes : 0);   // lambda^n, n = 0..128 (+pad)
    static constexpr uint32_t kOffPair = kOffPw + 132 * 4;     // pp, pr: packed decay pairs
    static constexpr uint32_t kOffBar = kOffPair + 2 * 164 * 4;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;   // tmem base, abort flag, 3 x 2 decision slots
    // Per-token decay: the H group's two chunk-decay slots, and the P group's
    // gate arrays for the chunk in hand ([128] running log2-decays, [128] last
    // clearing positions, [128] per-token factors exp(g)).
    static constexpr uint32_t kOffHDec = kOffMisc + 32;
    static constexpr uint32_t kOffGate = kOffHDec + 16;
    // The mixer epilogue's normalisation (kEpi): the head's aug row [96] and the
    // self-augmentation gates of two chunks [2][128].
    static constexpr uint32_t kOffEpi = kOffGate + kGateArr;
    static constexpr uint32_t kSmemUsed = kOffEpi + (96 + 256) * 4;
    static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;   // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kOffEpi % 16 == 0, "the aug row is read as float4");
    static_assert(kOffStage % 1024 == 0 && kStageBytes % 1024 == 0 && kOffSb % 1024 == 0 && kOffOut % 1024 == 0,
                  "tile alignment");
};
constexpr uint32_t kSmemBytesMax =
    Layout<128>::kSmemBytes > Layout<64>::kSmemBytes ? Layout<128>::kSmemBytes : Layout<64>::kSmemBytes;

constexpr uint32_t kTmemCols = 512, kColAP = 0, kColQt = 64, kColO = 128, kColS = 320;

struct FullArgs {
    const float *log_lambda;
    const float *h0;       // initial state [B,H,96,192] (times init_mul), or NULL
    float *hT;             // final state (times final_mul), or NULL
    float scale, init_mul, final_mul;
    int T, H, nck;
    // Sequence segmentation: the grid covers nseg segments of seg_chunks
    // chunks; segment g starts from h0 + g * h0_seg_stride and only the last
    // segment writes hT. nseg = 1: one chain per (b, h).
    int nseg, seg_chunks, BH;
    size_t h0_seg_stride;
    unsigned int *status;
    const float *g;        // per-token log-decays [B, T, H] (the gated form), or NULL
    // Variable-length mode (kVar): BH = nseq * H; sequence n holds tokens
    // cu_seqlens[n] .. cu_seqlens[n+1] of the packed [1, T, H, d] tensors and
    // its state in pool slot slots[n] (or n) of h0 == hT; a partial last chunk
    // is stored row by row to o (its tile would overlap the next sequence).
    const int *cu_seqlens, *slots;
    int n_slots;
    __nv_bfloat16 *o;
    // The mixer epilogue's self-augmentation (kEpi): the output rows become
    // u = o + sigmoid(q . (aug * k)) v, aug [H, 96] fp32 or NULL (zero); the
    // RMS normalisation, the norm weight and the gate follow in a second pass.
    const float *aug;
};

// One elected thread of an n-thread group waits; the verdict is published
// through a two-slot flag so every thread of the group takes the same branch
// after the group's named barrier.
__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, const WaitCtl &ctl, volatile int *decision,
                                      uint32_t gt, uint32_t named, uint32_t nthreads, uint32_t &k) {
    if (gt == 0) decision[k & 1] = mbar_wait(bar, parity, ctl) ? 0 : 1;
    named_sync(named, nthreads);
    return decision[(k++) & 1] == 0;
}

// Gated mode: the decay of a whole chunk from one warp's gates (four per lane,
// 0 past the chunk's end): 0 if any gate clears the state, else 2^(the sum of
// the log2-decays).
__device__ __forceinline__ float chunk_decay_warp(const float (&x)[4]) {
    float s = 0.f;
    int clr = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (x[r] > kResetLogDecay)
            s += x[r] * kLog2e;
        else
            clr = 1;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, d);
        clr |= __shfl_xor_sync(0xffffffffu, clr, d);
    }
    return clr ? 0.f : exp2f(s);
}

// kRev = false: the forward pass. kRev = true: the same chunked recurrence
// run backwards in time, which is how the backward pass obtains dv and dh0:
// rows are k tokens, columns q tokens, values dO, the mask keeps col >= row
// with lambda^(col-row), the row weights swap (lambda^(Cc-1-j) on the
// readout, lambda^(i+1) on the state update), chunks run last to first, and
// the state is the state gradient divided by the scale.
// kGate: the per-token decay of the gated form, S_t = exp(g_t) S_{t-1} +
// k_t v_t^T, in place of lambda: every power of lambda becomes the decay of a
// run of the chunk's tokens, lambda^(i-j) -> exp(G_i - G_j), lambda^(i+1) ->
// exp(G_i), lambda^(Cc-1-j) -> exp(G_last - G_j), lambda^Cc -> exp(G_last),
// with G the running sum of g over the chunk; a gate at or below the clearing
// threshold zeroes every decay across it. The P group's first warp scans each
// chunk's gates into shared arrays (loaded one chunk ahead), and P's weights
// are walked along the factors exp(g); the H group's first warp reduces each
// chunk's gates to its total decay for the state's rescale, one chunk ahead.
// `blk` is the CTA's unit: segment blk / BH of chain (b, h) = blk % BH.
// kEpi (forward, per-head decay, C = 128): each output row leaves with the
// self-augmentation added, u = o + sigmoid(q . (aug * k)) v over the head's
// 192 channels. The P group forms the row's gate from its q row (in
// registers) and its k row (before K is scaled); the E group forms u from O
// (TMEM) and v (the V slot it stages u into) in its one pass over the row.
template <bool kRev, int kC, bool kGate = false, bool kVar = false, bool kEpi = false>
__device__ __forceinline__ void full_body(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                          const CUtensorMap &tm_o, const FullArgs &a, int blk) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    constexpr int C = kC;   // chunk length, 64 or 128
    using L = Layout<kC>;
    constexpr bool kDual = L::kDual;
    constexpr uint32_t kB = L::kB, kOffQ = L::kOffQ, kOffStage = L::kOffStage, kStK = L::kStK, kStV = L::kStV;
    constexpr uint32_t kStageBytes = L::kStageBytes, kOffSb = L::kOffSb, kOffOut = L::kOffOut, kOffPw = L::kOffPw;
    constexpr uint32_t kOffPair = L::kOffPair, kOffBar = L::kOffBar, kOffMisc = L::kOffMisc, kOffHDec = L::kOffHDec;
    constexpr uint32_t kOffGate = L::kOffGate;
    static_assert(!kEpi || (!kRev && !kGate && !kVar && kC == 128), "the fused normalisation is a forward at C = 128");
    float *ep_aug = reinterpret_cast<float *>(sm + L::kOffEpi);   // [96], then the gates [2][128]
    float *ep_sig = ep_aug + 96;
    // Token rows of the score, P, Q~ and output tiles: M = C. An M = 64 tile
    // holds row i in TMEM lane 32 (i / 16) + i % 16 (lanes 0-15 of each
    // quadrant), as accumulator and as the A operand read from TMEM.
    constexpr int kM = C;
    constexpr int ksteps_tok = C / 16;
    static_assert(!kVar || !kRev, "variable-length mode is a forward");
    const int seg = blk / a.BH, bh = blk % a.BH;
    const int h = bh % a.H;
    // b: the state's index; bt, tokb: the batch and first-token coordinates of
    // the sequence in the token tensors; T: its length
    int b = bh / a.H, bt = b, tokb = 0, T = a.T, nck_seq = a.nck;
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
        tokb = beg;
        T = end - beg;
        nck_seq = (T + kC - 1) / kC;
    }
    const int cbeg = seg * a.seg_chunks;                 // first chunk of this segment
    const int nck = kVar ? nck_seq : min(a.seg_chunks, nck_seq - cbeg);   // chunks of this CTA
    const bool last_seg = seg == a.nseg - 1;
    const float *h0 = a.h0 ? a.h0 + (size_t)seg * a.h0_seg_stride : nullptr;
    auto tok0 = [&](int c) { return (kRev ? nck - 1 - c : cbeg + c) * C; };
    auto clen = [&](int c) { return min(C, T - tok0(c)); };
    // Gated mode: this lane's four gates (tokens 4 lane .. 4 lane + 3) of chunk
    // c in processing order, 0 past the sequence's end or the CTA's last chunk.
    auto load_gates = [&](int c, float (&x)[4]) {
        const int t0 = c < nck ? tok0(c) : 0, cc = c < nck ? clen(c) : 0;
        const float *gh = a.g + ((size_t)bt * a.T + tokb + t0) * a.H + h;
#pragma unroll
        for (int r = 0; r < 4; ++r) x[r] = 4 * lane + r < cc ? gh[(size_t)(4 * lane + r) * a.H] : 0.f;
    };

    float *pw = reinterpret_cast<float *>(sm + kOffPw);
    uint32_t *pp = reinterpret_cast<uint32_t *>(sm + kOffPair);
    uint32_t *pr = pp + 164;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    volatile int *dec = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);   // [3][2]
    const WaitCtl ctl{abort_flag, a.status};
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };
    auto stage = [&](int c) { return base + kOffStage + (uint32_t)(c & 1) * kStageBytes; };

    const uint32_t tx3 = 3u * (uint32_t)C * 64u, tx6 = 6u * (uint32_t)C * 64u;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 6; ++i) dec[i] = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), i == BAR_QFREE ? 2u : 1u);
        fence_mbar_init();
        fence_proxy_async_smem();
        // The per-head decay's first K, Q and V loads go out now, under the setup
        // below (decay tables, TMEM allocation); the producer issues the rest (all
        // of them with the per-token decay, whose forward measured slower this way).
        if (!kGate && nck > 0) {
            const uint32_t st = stage(0);
            const int t0 = tok0(0);
            mbar_arrive_expect_tx(bar(BAR_FULLK0), tx3);
#pragma unroll
            for (int j = 0; j < 3; ++j) tma_load_4d(st + kStK + j * kB, &tm_k, bar(BAR_FULLK0), 32 * j, h, tokb + t0, bt);
            mbar_arrive_expect_tx(bar(BAR_FULLQ), tx3);
#pragma unroll
            for (int j = 0; j < 3; ++j) tma_load_4d(base + kOffQ + j * kB, &tm_q, bar(BAR_FULLQ), 32 * j, h, tokb + t0, bt);
            mbar_arrive_expect_tx(bar(BAR_FULLV0), tx6);
#pragma unroll
            for (int j = 0; j < 6; ++j) tma_load_4d(st + kStV + j * kB, &tm_v, bar(BAR_FULLV0), 32 * j, h, tokb + t0, bt);
        }
        prefetch_tmap(&tm_o);
    }
    if constexpr (!kGate) {   // the gated form has no per-head decay (log_lambda is NULL)
        const float l2 = log2_of_decay(a.log_lambda[h]);
        for (int n = threadIdx.x; n < 132; n += kThreads) pw[n] = n <= 128 ? decay_pow(l2, n) : 0.f;
        fill_pair_tables(pp, pr, l2, threadIdx.x, kThreads);
    }
    if constexpr (kEpi)
        for (int n = threadIdx.x; n < 96; n += kThreads) ep_aug[n] = a.aug ? a.aug[h * 96 + n] : 0.f;
    if (warp == 3) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 15) {
        // ------------------------------------------------------- TMA producer
        // K(c) into stage c % 2 once ST(c-2) has completed; Q(c) once QK(c-1)
        // has completed and Q~(c-1) is in TMEM; V(c) into stage c % 2 once the
        // output of chunk c-2, staged in that slot, has been read out. With the
        // per-head decay chunk 0's loads went out with the barriers' initialisation.
        int nq = 0, nk = 0, nv = 0;   // chunks whose Q / K / V loads were issued
        for (int c = 0; c < nck; ++c) {
            const int s = c & 1;
            const uint32_t st = stage(c);
            const int t0 = tok0(c);
            const uint32_t ph2 = (uint32_t)((c >> 1) - 1) & 1u;   // phase parity of chunk c-2
            if (c >= 2 && !lane0_wait(bar(BAR_KFREE0 + s), ph2, ctl, lane)) break;
            if (lane == 0 && (kGate || c > 0)) {
                mbar_arrive_expect_tx(bar(BAR_FULLK0 + s), tx3);
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(st + kStK + j * kB, &tm_k, bar(BAR_FULLK0 + s), 32 * j, h, tokb + t0, bt);
            }
            __syncwarp();
            nk = c + 1;
            if (c >= 1 && !lane0_wait(bar(BAR_QFREE), (uint32_t)(c - 1) & 1u, ctl, lane)) break;
            if (lane == 0) {
                if (kGate || c > 0) {
                    mbar_arrive_expect_tx(bar(BAR_FULLQ), tx3);
#pragma unroll
                    for (int j = 0; j < 3; ++j)
                        tma_load_4d(base + kOffQ + j * kB, &tm_q, bar(BAR_FULLQ), 32 * j, h, tokb + t0, bt);
                }
                // Q has one buffer: bring the next chunk's tile into L2 now, so that its
                // load, which waits for this one to be consumed, is served from L2.
                if (c + 1 < nck)
#pragma unroll
                    for (int j = 0; j < 3; ++j) tma_prefetch_4d(&tm_q, 32 * j, h, tokb + tok0(c + 1), bt);
            }
            __syncwarp();
            nq = c + 1;
            if (c >= 2 && !lane0_wait(bar(BAR_VFREE0 + s), ph2, ctl, lane)) break;
            if (lane == 0) {
                if (kGate || c > 0) {
                    mbar_arrive_expect_tx(bar(BAR_FULLV0 + s), tx6);
#pragma unroll
                    for (int j = 0; j < 6; ++j)
                        tma_load_4d(st + kStV + j * kB, &tm_v, bar(BAR_FULLV0 + s), 32 * j, h, tokb + t0, bt);
                }
                // V(c+1)'s slot frees only once the output of chunk c-1 has been stored from
                // it; bring that tile into L2 now, so that its load is served from L2 (the
                // per-head decay's forward: measured 62.5 -> 60.6 us on the layer shape; the
                // reverse and gated modes measured 0.5-1.5 % slower with it).
                if (!kRev && !kGate && c + 1 < nck)
#pragma unroll
                    for (int j = 0; j < 6; ++j) tma_prefetch_4d(&tm_v, 32 * j, h, tokb + tok0(c + 1), bt);
            }
            __syncwarp();
            nv = c + 1;
        }
        // Drain: every load issued must have landed before the CTA exits.
        if (lane == 0) {
            if (nq >= 1) mbar_wait_drain(bar(BAR_FULLQ), (uint32_t)(nq - 1) & 1u, 1000000ull);
            for (int c = (nk >= 2 ? nk - 2 : 0); c < nk; ++c)
                mbar_wait_drain(bar(BAR_FULLK0 + (c & 1)), (uint32_t)(c >> 1) & 1u, 1000000ull);
            for (int c = (nv >= 2 ? nv - 2 : 0); c < nv; ++c)
                mbar_wait_drain(bar(BAR_FULLV0 + (c & 1)), (uint32_t)(c >> 1) & 1u, 1000000ull);
        }
        __syncwarp();
    } else if (warp == 3) {
        // ----------------------------------------------- MMA issuer (event loop)
        if (lane == 0) {
            const uint32_t idA = idesc_bf16(kM, C, false, false);     // Q K^T: both K-major
            const uint32_t idS = idesc_bf16(128, kDv, true, true);    // K~^T V: both MN-major
            const uint32_t idO = idesc_bf16(kM, kDv, false, true);    // Q~ S, P V: A in TMEM, B MN-major
            int qk = 0, stt = 0, out = 0;   // next chunk of each event kind
            uint64_t t_idle = globaltimer_ns();
            uint32_t spins = 0;
            while (out < nck) {
                bool progress = false;
                // QK(c): the AP region is free once OUT(c-1) has completed
                if (qk < nck && qk == out) {
                    const int c = qk;
                    if (mbar_test(bar(BAR_FULLQ), (uint32_t)c & 1u) &&
                        mbar_test(bar(BAR_FULLK0 + (c & 1)), (uint32_t)(c >> 1) & 1u) &&
                        (c == 0 || mbar_test(bar(BAR_OFULL), (uint32_t)(c - 1) & 1u))) {
                        tc_fence_after();
                        const uint32_t st = stage(c);
#pragma unroll
                        for (int ks = 0; ks < 6; ++ks) {
                            const uint32_t off = (uint32_t)(ks >> 1) * kB + (uint32_t)(ks & 1) * 32;
                            mma_bf16_ss(tmem + kColAP, smem_desc(base + kOffQ + off, 16, 512, 4),
                                        smem_desc(st + kStK + off, 16, 512, 4), idA, ks > 0);
                        }
                        mma_commit(bar(BAR_QKDONE));
                        mma_commit(bar(BAR_QFREE));
                        ++qk;
                        progress = true;
                    }
                }
                // ST(c): S += K~^T V once K~ is scaled and S rescaled (hand-off of c-1)
                if (stt < qk) {
                    const int c = stt;
                    if (mbar_test(bar(BAR_KREADY), (uint32_t)c & 1u) &&
                        mbar_test(bar(BAR_FULLV0 + (c & 1)), (uint32_t)(c >> 1) & 1u) &&
                        mbar_test(bar(BAR_SBREADY), (uint32_t)c & 1u)) {
                        tc_fence_after();
                        const uint32_t st = stage(c);
#pragma unroll
                        for (int ks = 0; ks < ksteps_tok; ++ks)
                            mma_bf16_ss(tmem + kColS, smem_desc(st + kStK + (uint32_t)ks * 1024, kB, 512, 4),
                                        smem_desc(st + kStV + (uint32_t)ks * 1024, kB, 512, 4), idS, 1);
                        mma_commit(bar(BAR_SFULL));
                        mma_commit(bar(BAR_KFREE0 + (c & 1)));
                        ++stt;
                        progress = true;
                    }
                }
                // OUT(c): O = Q~ S_prev + P V once P and Q~ are built and O has been read out
                if (out < stt) {
                    const int c = out;
                    if (mbar_test(bar(BAR_PREADY), (uint32_t)c & 1u) &&
                        (c == 0 || mbar_test(bar(BAR_OEMPTY), (uint32_t)(c - 1) & 1u))) {
                        tc_fence_after();
                        const uint32_t stv = stage(c) + kStV;
                        const uint32_t sb_prev = base + kOffSb + (kDual ? (uint32_t)(c & 1) * kSbBytes : 0u);
#pragma unroll
                        for (int ks = 0; ks < 6; ++ks)
                            mma_bf16_ts(tmem + kColO, tmem + kColQt + 8u * (uint32_t)ks,
                                        smem_desc(sb_prev + (uint32_t)ks * 1024, kSbBlk, 512, 4), idO, ks > 0);
#pragma unroll
                        for (int ks = 0; ks < ksteps_tok; ++ks)
                            mma_bf16_ts(tmem + kColO, tmem + kColAP + 8u * (uint32_t)ks,
                                        smem_desc(stv + (uint32_t)ks * 1024, kB, 512, 4), idO, 1);
                        mma_commit(bar(BAR_OFULL));
                        ++out;
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
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------- P group (4..7)
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;          // K row scaled by this thread
        // the token row in this thread's TMEM lane (M = 64: lanes 16-31 hold none and
        // repeat the row of lane - 16, into TMEM lanes no MMA reads)
        const uint32_t trow = kM == 128 ? row : quad * 16 + ((uint32_t)lane & 15u);
        const int dblk = (int)trow / 32;                          // the diagonal P block
        const uint32_t gt = (uint32_t)threadIdx.x - 128;         // 0..127
        const uint32_t tl = tmem + ((quad * 32) << 16);
        constexpr int nblk = C / 32;
        uint32_t kw = 0;
        // gated: the group's gate arrays, scanned by its first warp one chunk at a time
        float *Gl = reinterpret_cast<float *>(sm + kOffGate);
        int *Zc = reinterpret_cast<int *>(sm + kOffGate + 512);
        float *Af = reinterpret_cast<float *>(sm + kOffGate + 1024);
        float gpre[4];
        if (kGate && gt < 32) load_gates(0, gpre);
        for (int c = 0; c < nck; ++c) {
            const int Cc = clen(c);
            if (kGate && gt < 32) {
                // every thread of the group is past chunk c-1's reads of the arrays (the
                // barrier before its P-ready signal); the barrier in the wait below
                // publishes the new ones
                gate_scan_store(gpre, lane, Gl, Zc, Af);
                load_gates(c + 1, gpre);
            }
            // Q has one buffer: as soon as it lands, this thread's row of it goes to
            // registers, and the tile is free once QK(c), its other reader, is done.
            if (!gwait(bar(BAR_FULLQ), (uint32_t)c & 1u, ctl, dec, gt, kBarP, 128, kw)) break;
            uint4 qrow[12];
#pragma unroll
            for (int j = 0; j < 3; ++j)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    qrow[4 * j + cc] = ld_shared_v4(base + kOffQ + j * kB + sw64_offset(trow, (uint32_t)cc));
            named_sync(kBarP, 128);
            if (gt == 0) mbar_arrive(bar(BAR_QFREE));
            if (!gwait(bar(BAR_QKDONE), (uint32_t)c & 1u, ctl, dec, gt, kBarP, 128, kw)) break;
            tc_fence_after();
            // K~ = diag(lambda^(Cc-1-j)) K in place (zero past the end), or lambda^(i+1)
            // in reverse; signalled at once.
            {
                float wk;
                if constexpr (kGate && kRev)   // the decay of the chunk's tokens 0..i
                    wk = Zc[row] < 0 ? exp2f(Gl[row]) : 0.f;
                else if constexpr (kGate)      // the decay of tokens j+1..Cc-1
                    wk = row < (uint32_t)Cc && Zc[Cc - 1] <= (int)row ? exp2f(Gl[Cc - 1] - Gl[row]) : 0.f;
                else
                    wk = kRev ? pw[row + 1] : (row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f);
                if constexpr (kEpi) {
                    // The row's self-augmentation gate from q (registers) and the k row,
                    // read once: the dot product is taken before the row is scaled.
                    const uint32_t kb = stage(c) + kStK;
                    const uint32_t w2 = pack_bf16x2(wk, wk);
                    float dot = 0.f;
#pragma unroll
                    for (int j = 0; j < 3; ++j)
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            const uint32_t addr = kb + j * kB + sw64_offset(row, (uint32_t)cc);
                            uint4 kv = ld_shared_v4(addr);
                            const uint32_t kw4[4] = {kv.x, kv.y, kv.z, kv.w};
                            const uint4 qv = qrow[4 * j + cc];
                            const uint32_t qw4[4] = {qv.x, qv.y, qv.z, qv.w};
                            const float4 a0 = *reinterpret_cast<const float4 *>(ep_aug + 32 * j + 8 * cc);
                            const float4 a1 = *reinterpret_cast<const float4 *>(ep_aug + 32 * j + 8 * cc + 4);
                            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 qf = unpack_bf16x2(qw4[e]), kf = unpack_bf16x2(kw4[e]);
                                dot = fmaf(qf.x * av[2 * e], kf.x, dot);
                                dot = fmaf(qf.y * av[2 * e + 1], kf.y, dot);
                            }
                            kv.x = mul_bf16x2(kv.x, w2);
                            kv.y = mul_bf16x2(kv.y, w2);
                            kv.z = mul_bf16x2(kv.z, w2);
                            kv.w = mul_bf16x2(kv.w, w2);
                            st_shared_v4(addr, kv.x, kv.y, kv.z, kv.w);
                        }
                    ep_sig[(c & 1) * 128 + row] = 1.f / (1.f + __expf(-dot));
                } else if (row < (uint32_t)C) {
                    scale_rows<3, kB>(sm + (stage(c) - base) + kStK, row, wk);
                }
            }
            fence_proxy_async_smem();
            named_sync(kBarP, 128);
            if (gt == 0) mbar_arrive(bar(BAR_KREADY));
            // P = bf16((Q K^T) .* D) in place over A. Blocks in increasing order:
            // P block bk lands in columns [16 bk, 16 bk + 16), inside score block
            // bk / 2, which this warp has already read (or never needs). Blocks on
            // the masked side of the diagonal (above it forward, below it in
            // reverse) are written as zeros.
#pragma unroll 1
            for (int bk = 0; bk < nblk; ++bk) {
                if (kRev ? bk >= dblk : bk <= dblk) {
                    uint32_t x[32];
                    tmem_ld_32cols(tl + kColAP + 32u * bk, x);
                    if constexpr (kGate) {
                        const bool dg = bk == dblk;
                        const float gi = Gl[trow];
                        if constexpr (kRev) {
                            // row j, columns i >= j: walked rightwards from the block's first column
                            const int il = 32 * bk;
                            const float d0 = dg || Zc[il] > (int)trow ? 0.f : ex2_approx(Gl[il] - gi);
                            tmem_ld_wait();
                            build_p_block_gated_rev(x, dg ? (int)trow - il : -1, il, d0, Af, tl + kColAP + 16u * bk);
                        } else {
                            // row i, columns j <= i: walked leftwards from the block's last column
                            const int jr = 32 * bk + 31;
                            const float d0 = dg || Zc[trow] > jr ? 0.f : ex2_approx(gi - Gl[jr]);
                            tmem_ld_wait();
                            build_p_block_gated(x, dg ? (int)trow - 32 * bk : 32, 32 * bk, d0, Af,
                                                tl + kColAP + 16u * bk);
                        }
                    } else {
                        tmem_ld_wait();
                        pack_scores(x);
                        build_p_block<kRev>(x, (int)trow - 32 * bk, tl + kColAP + 16u * bk, pp, pr);
                    }
                } else {
                    uint32_t z[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) z[e] = 0u;
                    tmem_st_16cols(tl + kColAP + 16u * bk, z);
                }
            }
            // Q~ = diag(lambda^(i+1)) Q into columns [64, 112), the A operand of
            // Q~ S_prev: lane = token row, column = dk pair, from the row kept in
            // registers. This warp's score columns there (C = 128) were read above.
            {
                // lambda^(i+1); lambda^(Cc-1-j) in reverse (zero past the end)
                float wq;
                if constexpr (kGate && kRev)   // the decay of tokens j+1..Cc-1
                    wq = trow < (uint32_t)Cc && Zc[Cc - 1] <= (int)trow ? exp2f(Gl[Cc - 1] - Gl[trow]) : 0.f;
                else if constexpr (kGate)      // the decay of the chunk's tokens 0..i
                    wq = Zc[trow] < 0 ? exp2f(Gl[trow]) : 0.f;
                else
                    wq = kRev ? (trow < (uint32_t)Cc ? pw[Cc - 1 - (int)trow] : 0.f) : pw[trow + 1];
                const uint32_t wq2 = pack_bf16x2(wq, wq);
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    uint32_t pk[16];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 v = qrow[4 * j + cc];
                        pk[4 * cc + 0] = mul_bf16x2(v.x, wq2);
                        pk[4 * cc + 1] = mul_bf16x2(v.y, wq2);
                        pk[4 * cc + 2] = mul_bf16x2(v.z, wq2);
                        pk[4 * cc + 3] = mul_bf16x2(v.w, wq2);
                    }
                    tmem_st_16cols(tl + kColQt + 16u * j, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            named_sync(kBarP, 128);
            if (gt == 0) mbar_arrive(bar(BAR_PREADY));
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------- E group (8..11)
        const uint32_t quad = (uint32_t)(warp & 3);
        // the output row in this thread's TMEM lane (M = 64: lanes 0-15 of the quadrant)
        const uint32_t row = kM == 128 ? quad * 32 + (uint32_t)lane : quad * 16 + (uint32_t)lane;
        const bool has_row = kM == 128 || lane < 16;
        const uint32_t gt = (uint32_t)threadIdx.x - 256;         // 0..127
        const uint32_t tl = tmem + ((quad * 32) << 16);
        uint32_t kw = 0;
        for (int c = 0; c < nck; ++c) {
            if (!gwait(bar(BAR_OFULL), (uint32_t)c & 1u, ctl, dec + 2, gt, kBarE, 128, kw)) break;
            tc_fence_after();
            // Stage in V(c)'s slot: ST(c) and OUT(c), its readers, have completed.
            // kDual: in output buffer c % 2 instead, so V(c)'s slot is free at once,
            // once the store from that buffer two chunks ago has been read out.
            const uint32_t stg = kDual ? base + kOffOut + (uint32_t)(c & 1) * L::kOutBytes : stage(c) + kStV;
            if constexpr (kDual) {
                if (gt == 0) {
                    mbar_arrive(bar(BAR_VFREE0 + (c & 1)));
                    tma_store_wait_read_1();
                }
                named_sync(kBarE, 128);
            }
            const int t0 = tok0(c);
            // a packed sequence's partial last chunk: rows straight to o
            const bool rowwise = kVar && clen(c) < C;
            __nv_bfloat16 *orow = kVar ? a.o + ((size_t)(tokb + t0 + (int)row) * a.H + h) * kDv : nullptr;
            const bool row_out = has_row && (int)row < clen(c);
            auto put = [&](const uint32_t (&r)[32], int blk) {
                if (!rowwise) {
                    if (has_row) write_row_sw64_bits(sm + (stg - base) + blk * kB, row, r, a.scale);
                } else if (row_out) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        *reinterpret_cast<uint4 *>(orow + 32 * blk + e) = make_uint4(
                            pack_bf16x2(__uint_as_float(r[e]) * a.scale, __uint_as_float(r[e + 1]) * a.scale),
                            pack_bf16x2(__uint_as_float(r[e + 2]) * a.scale, __uint_as_float(r[e + 3]) * a.scale),
                            pack_bf16x2(__uint_as_float(r[e + 4]) * a.scale, __uint_as_float(r[e + 5]) * a.scale),
                            pack_bf16x2(__uint_as_float(r[e + 6]) * a.scale, __uint_as_float(r[e + 7]) * a.scale));
                }
            };
            if constexpr (kEpi) {
                // u = o * scale + sigma * v over this row's v in the V slot (each
                // thread owns its row), the next block's TMEM load in flight while
                // this one is formed and staged.
                const float sg = ep_sig[(c & 1) * 128 + row];
                auto put_u = [&](uint32_t (&r)[32], int blk) {
                    const uint32_t vrow = stg + blk * kB;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 vv = ld_shared_v4(vrow + sw64_offset(row, (uint32_t)cc));
                        const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 vf = unpack_bf16x2(vw[e]);
                            const int m = 8 * cc + 2 * e;
                            r[m] = __float_as_uint(fmaf(sg, vf.x, __uint_as_float(r[m]) * a.scale));
                            r[m + 1] = __float_as_uint(fmaf(sg, vf.y, __uint_as_float(r[m + 1]) * a.scale));
                        }
                    }
                    write_row_sw64_bits(sm + (stg - base) + blk * kB, row, r, 1.f);
                };
                uint32_t ra[32], rb[32];
                tmem_ld_32cols(tl + kColO, ra);
#pragma unroll 1
                for (int bp = 0; bp < 3; ++bp) {
                    const int blk = 2 * bp;
                    tmem_ld_wait();
                    tmem_ld_32cols(tl + kColO + 32u * (blk + 1), rb);
                    put_u(ra, blk);
                    tmem_ld_wait();
                    if (bp < 2) tmem_ld_32cols(tl + kColO + 32u * (blk + 2), ra);
                    put_u(rb, blk + 1);
                }
            } else {
                // Six 32-column blocks, the next block's TMEM load in flight while
                // this one is converted and staged.
                uint32_t ra[32], rb[32];
                tmem_ld_32cols(tl + kColO, ra);
#pragma unroll 1
                for (int bp = 0; bp < 3; ++bp) {
                    const int blk = 2 * bp;
                    tmem_ld_wait();
                    tmem_ld_32cols(tl + kColO + 32u * (blk + 1), rb);
                    put(ra, blk);
                    tmem_ld_wait();
                    if (bp < 2) tmem_ld_32cols(tl + kColO + 32u * (blk + 2), ra);
                    put(rb, blk + 1);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_sync(kBarE, 128);
            if (gt == 0) {
                mbar_arrive(bar(BAR_OEMPTY));
                if (!rowwise) {
#pragma unroll
                    for (int blk = 0; blk < 6; ++blk) tma_store_4d(&tm_o, stg + blk * kB, 32 * blk, h, tokb + t0, bt);
                    tma_store_commit();
                    if (!kDual) tma_store_wait_read_all();
                }
                if (!kDual) mbar_arrive(bar(BAR_VFREE0 + (c & 1)));
            }
        }
        if (gt == 0) tma_store_wait_all();
    } else {
        // ------------------- H group (warps 12-14 and 0-2: rows 0..95, two column halves)
        const uint32_t quad = (uint32_t)(warp & 3);               // 0, 1, 2
        const uint32_t row = quad * 32 + (uint32_t)lane;          // state row (dk index)
        const int half = warp >= 12 ? 0 : 1;                      // column blocks 3 half .. 3 half + 2
        const uint32_t gt = (uint32_t)half * 96u + row;           // 0..191
        const uint32_t tl = tmem + ((quad * 32) << 16);
        const int blk0 = 3 * half;
        uint32_t kw = 0;
        // gated: chunk decays, reduced by the group's first warp one chunk ahead
        volatile float *hdec = reinterpret_cast<volatile float *>(sm + kOffHDec);
        float hpre[4];
        if (kGate && gt < 32) {
            load_gates(0, hpre);
            const float d = chunk_decay_warp(hpre);
            if (lane == 0) hdec[0] = d;
            load_gates(1, hpre);
        }
        if constexpr (kGate) named_sync(kBarH, kHThreads);
        // Initial state: copy = bf16(h0), TMEM S = lambda^C0 h0 (C0: the first chunk's length).
        {
            const float w0 = kGate ? hdec[0] : pw[clen(0)];
            const float *src = h0 ? h0 + (((size_t)b * a.H + h) * kDk + row) * kDv : nullptr;
#pragma unroll 1
            for (int blk = blk0; blk < blk0 + 3; ++blk) {
                float x[32];
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 v4 = src ? *reinterpret_cast<const float4 *>(src + blk * 32 + e)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[e] = v4.x * a.init_mul;
                    x[e + 1] = v4.y * a.init_mul;
                    x[e + 2] = v4.z * a.init_mul;
                    x[e + 3] = v4.w * a.init_mul;
                }
                write_row_sw64(sm + kOffSb + blk * kSbBlk, row, x);
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(x[e] * w0);
                tmem_st_32cols(tl + kColS + 32u * blk, r);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarH, kHThreads);
            if (gt == 0) mbar_arrive(bar(BAR_SBREADY));
        }
        bool hT_staged = false;
        for (int c = 0; c < nck; ++c) {
            const bool last = c == nck - 1;
            const bool write_hT = last && last_seg && a.hT;
            if (kGate && gt < 32) {
                // the decay of chunk c+1 (published by the barrier in the wait below)
                const float d = chunk_decay_warp(hpre);
                if (lane == 0) hdec[(c + 1) & 1] = d;
                load_gates(c + 2, hpre);
            }
            if (!gwait(bar(BAR_SFULL), (uint32_t)c & 1u, ctl, dec + 4, gt, kBarH, kHThreads, kw)) break;
            // the copy is single: OUT(c) must have read it before it changes
            // (kDual: two copies, and OUT(c-1), the last reader of the one rewritten
            // now, completed before ST(c) was issued)
            if (!kDual && !gwait(bar(BAR_OFULL), (uint32_t)c & 1u, ctl, dec + 4, gt, kBarH, kHThreads, kw)) break;
            // hT goes out as one 73,728-byte bulk store, staged row-major in the other
            // stage's K and V slots (72 KB, contiguous), free once the output of chunk
            // c-1, staged in that V slot, has been read out (K's last reader, ST(c-1),
            // is long complete).
            if (write_hT && c >= 1 &&
                !gwait(bar(BAR_VFREE0 + ((c - 1) & 1)), (uint32_t)((c - 1) >> 1) & 1u, ctl, dec + 4, gt, kBarH,
                       kHThreads, kw))
                break;
            tc_fence_after();
            const float wn = last ? 1.f : (kGate ? hdec[(c + 1) & 1] : pw[clen(c + 1)]);
            // the staging row of hT (fp32, 768 bytes): the stage not holding chunk c
            // (kDual: its 36 KB hold rows 0-47, the S_prev copy OUT(c) does not
            // read rows 48-95)
            const uint32_t sb_next = kOffSb + (kDual ? (uint32_t)((c + 1) & 1) * kSbBytes : 0u);
            unsigned char *hrow = !write_hT ? nullptr
                                  : (!kDual || row < 48) ? sm + (stage(c + 1) - base) + row * (kDv * 4)
                                                         : sm + sb_next + (row - 48) * (kDv * 4);
            // Three 32-column blocks, the next block's TMEM load in flight while
            // this one is copied and rescaled.
            auto handle = [&](uint32_t (&r)[32], int blk) {
                if (last) {
                    if (hrow) {
                        // (once per sequence: the bank conflicts of rows 768 bytes apart are
                        // cheaper than the per-thread global stores they replace)
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a.final_mul);
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            st_shared_v4(smem_u32(hrow + (blk * 32 + e) * 4), r[e], r[e + 1], r[e + 2], r[e + 3]);
                    }
                } else {
                    write_row_sw64_bits(sm + sb_next + blk * kSbBlk, row, r, 1.f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * wn);
                    tmem_st_32cols(tl + kColS + 32u * blk, r);
                }
            };
            {
                uint32_t ra[32], rb[32];
                tmem_ld_32cols(tl + kColS + 32u * blk0, ra);
                tmem_ld_wait();
                tmem_ld_32cols(tl + kColS + 32u * (blk0 + 1), rb);
                handle(ra, blk0);
                tmem_ld_wait();
                tmem_ld_32cols(tl + kColS + 32u * (blk0 + 2), ra);
                handle(rb, blk0 + 1);
                tmem_ld_wait();
                handle(ra, blk0 + 2);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            named_sync(kBarH, kHThreads);
            if (gt == 0 && !last) mbar_arrive(bar(BAR_SBREADY));
            if (gt == 0 && write_hT) {
                float *hdst = a.hT + ((size_t)b * a.H + h) * kDk * kDv;
                if constexpr (kDual) {
                    bulk_store(hdst, stage(c + 1), 48 * kDv * 4);
                    bulk_store(hdst + 48 * kDv, base + sb_next, 48 * kDv * 4);
                } else {
                    bulk_store(hdst, stage(c + 1), kDk * kDv * 4);
                }
                tma_store_commit();
                hT_staged = true;
            }
        }
        if (hT_staged) tma_store_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 3) tmem_dealloc(tmem, kTmemCols);
}


}  // namespace
}  // namespace fullhead
}  // namespace gla
