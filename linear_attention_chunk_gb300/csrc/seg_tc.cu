// seg_tc.cu -- sequence segmentation of the chunked forward for long
// sequences with few (b, h) pairs.
//
// The chunk-state recurrence of "Beyond the KV cache: Training and serving
// i14's Laplace 3B linear attention model on AWS Trainium2 with native
// PyTorch" ("Challenge 1", "Chunked GLA state update": S <- lambda^C S +
// sum_j lambda^(C-1-j) k_j v_j^T) is linear in S, so the state entering a
// segment of L tokens is the state entering the previous segment decayed by
// lambda^L plus that segment's own contribution from a zero state. Three
// launches, all on the caller's stream:
//   1. gla_seg_state_kernel: per (b, h, segment but the last) the segment's
//      local end state dS_g from zero (k and v only);
//   2. gla_seg_scan_kernel: S_in(0) = h0, S_in(g) = lambda^L(g-1) S_in(g-1) + dS_(g-1);
//   3. the forward kernel on every segment at once, each from S_in(g).
// This reads k and v of all but the last segment twice (up to 1,728 instead
// of 1,152 bytes per head-token) in exchange for B*H*2*G CTAs instead of B*H*2.
// Workspace: dS and S_in, each [G][B][H][96][192] fp32.
//
// With a per-token decay (the gated form, g [B,T,H]) the segment's decay
// lambda^L becomes D(g) = exp(sum of the segment's g), 0 when one of its
// gates clears the state, and the row weight of K the decay of the tokens
// after it in the segment. The state pass also writes D(g) ([G][B][H] fp32,
// after S_in in the workspace) for the scan.
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
constexpr int kStates = kDk * kDv;                  // floats per (b, h) state
constexpr int kThreads = 192;
constexpr int kStages = 3;
// K's three dk blocks, then V's six. The state MMA runs at M = 128 over dk =
// 96: its fourth M block reads V's first block in place of a zero pad. Those
// products land only in TMEM lanes 96..127, which nothing reads, and without
// the pad three stages fit.
constexpr uint32_t kStageK = 0;                     // 3 blocks
constexpr uint32_t kStageV = 3 * kBlk;              // 6 blocks: all 192 dv columns
constexpr uint32_t kStageBytes = 9 * kBlk;          // 72 KB
enum { BAR_FULL0 = 0, BAR_EMPTY0 = kStages, BAR_KREADY0 = 2 * kStages, BAR_SFULL = 3 * kStages, BAR_DONE,
       kNumBars };
constexpr uint32_t kOffBar = kStages * kStageBytes;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
// gated: the chunk's running log2-decays [128], then 4 + 4 reduction slots
constexpr uint32_t kOffGate = kOffMisc + 32;
constexpr uint32_t kSmemBytes = kOffGate + 128 * 4 + 32 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 256;                 // the 192-column state
constexpr uint32_t kBarK = 1;

struct SegArgs {
    const float *log_lambda;
    float *dS;             // [G][B][H][96][192]
    int H, C, seg_chunks, BH;
    unsigned int *status;
    const float *g;        // gated: per-token log-decays [B, T, H], else NULL
    int T;
    float *dseg;           // gated: the segments' decays D [G][B][H]
};

// A log-decay at or below this clears the state (exp(-80) is below fp32's
// normal range).
constexpr float kResetLogDecay = -80.f;
constexpr float kLog2e = 1.4426950408889634f;

// dS of segment g < G-1 of sequence (b, h): its end state from a zero start,
//   dS = sum_i lambda^((n-1-i) C) sum_j lambda^(C-1-j) k_ij v_ij^T
// over its n = seg_chunks chunks i (all full: only the last segment holds
// the sequence's end, and its dS is never needed). The decay of the later
// chunks is folded into the row weight of K, lambda^((n-1-i) C + C-1-j), so
// the state accumulates in TMEM over the whole segment with no rescale
// between chunks: a streaming K~^T V reduction (M = 96 run as 128, N = 192)
// through a three-stage ring, one CTA per (segment, b, h).
// Warps: 0 TMA, 1 TMEM + MMA, 2-5 row weights on K and the final dS store.
// kGate: the row weight of token j is the decay of the segment's tokens after
// j, 2^(A_end - A_j) with A the running sum of log2-decays from the segment's
// start (0 when a clearing gate lies after j), and the segment's decay D is
// written out for the scan.
template <bool kGate>
__global__ void __launch_bounds__(kThreads, 1)
    gla_seg_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const SegArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int seg = blockIdx.x / a.BH;
    const int bh = blockIdx.x % a.BH;
    const int b = bh / a.H, h = bh % a.H;
    const int C = a.C;
    const int cbeg = seg * a.seg_chunks;
    const int n = a.seg_chunks;
    const int ksteps_tok = C / 16;

    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    volatile int *dec = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);
    const WaitCtl ctl{abort_flag, a.status};
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 2; ++i) dec[i] = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
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
        const uint32_t tx = 9u * (uint32_t)C * 64u;
        int issued = 0;
        for (int c = 0; c < n; ++c) {
            const int s = c % kStages;
            if (c >= kStages && !lane0_wait(bar(BAR_EMPTY0 + s), ((c / kStages) - 1) & 1, ctl, lane)) break;
            if (lane == 0) {
                const uint32_t st = base + (uint32_t)s * kStageBytes;
                const uint32_t fb = bar(BAR_FULL0 + s);
                mbar_arrive_expect_tx(fb, tx);
                const int t0 = (cbeg + c) * C;
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(st + kStageK + j * kBlk, &tm_k, fb, 32 * j, h, t0, b);
#pragma unroll
                for (int j = 0; j < 6; ++j) tma_load_4d(st + kStageV + j * kBlk, &tm_v, fb, 32 * j, h, t0, b);
            }
            __syncwarp();
            issued = c + 1;
        }
        // Drain: the last loads issued must have landed before the CTA exits.
        if (lane == 0)
            for (int c = max(issued - kStages, 0); c < issued; ++c)
                mbar_wait_drain(bar(BAR_FULL0 + c % kStages), (c / kStages) & 1, 1000000ull);
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------- MMA issuer
        const uint32_t idS = idesc_bf16(128, kDv, true, true);
        for (int c = 0; c < n; ++c) {
            const int s = c % kStages;
            if (!lane0_wait(bar(BAR_KREADY0 + s), (c / kStages) & 1, ctl, lane)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = base + (uint32_t)s * kStageBytes;
                for_token_steps(ksteps_tok, [&](int ks) {
                    mma_bf16_ss(tmem, smem_desc(st + kStageK + (uint32_t)ks * 1024, kBlk, 512, 4),
                                smem_desc(st + kStageV + (uint32_t)ks * 1024, kBlk, 512, 4), idS,
                                (c > 0 || ks > 0) ? 1u : 0u);
                });
                mma_commit(bar(BAR_EMPTY0 + s));
            }
            __syncwarp();
        }
        if (lane == 0) mma_commit(bar(BAR_SFULL));   // the segment's state is complete
        __syncwarp();
    } else {
        // ------------------------ warps 2-5: K~ rows, then dS out of TMEM
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 64;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        const float l2 = kGate ? 0.f : log2_of_decay(a.log_lambda[h]);
        uint32_t kw = 0;
        bool ok = true;
        // Gated: the segment's total log2-decay and its last clearing position,
        // then a running sum carried from chunk to chunk.
        float *gl = reinterpret_cast<float *>(sm + kOffGate);
        float *red = gl + 128;
        int *redz = reinterpret_cast<int *>(red + 4);
        const float *gh = kGate ? a.g + ((size_t)b * a.T + (size_t)cbeg * C) * a.H + h : nullptr;
        float a_end = 0.f, a_before = 0.f;
        int z_end = -1;
        if constexpr (kGate) {
            float part = 0.f;
            int zp = -1;
            for (int t = (int)gt; t < n * C; t += kGroupThreads) {
                const float x = gh[(size_t)t * a.H];
                if (x > kResetLogDecay)
                    part += x * kLog2e;
                else
                    zp = t;
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                part += __shfl_xor_sync(0xffffffffu, part, d);
                zp = max(zp, __shfl_xor_sync(0xffffffffu, zp, d));
            }
            if (lane == 0) {
                red[quad] = part;
                redz[quad] = zp;
            }
            named_sync(kBarK, kGroupThreads);
            a_end = red[0] + red[1] + red[2] + red[3];
            z_end = max(max(redz[0], redz[1]), max(redz[2], redz[3]));
            if (gt == 0) a.dseg[(size_t)seg * a.BH + bh] = z_end < 0 ? exp2f(a_end) : 0.f;
        }
        for (int c = 0; c < n; ++c) {
            const int s = c % kStages;
            if (!group_wait(bar(BAR_FULL0 + s), (c / kStages) & 1, ctl, dec, gt, kBarK, kw)) {
                ok = false;
                break;
            }
            float wk;
            if constexpr (kGate) {
                // the chunk's running sums: one warp scans its 128 gates
                if (gt < 32) {
                    float x[4], ls[4], sacc = 0.f;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int t = 4 * (int)gt + r;
                        x[r] = t < C ? gh[(size_t)(c * C + t) * a.H] : 0.f;
                        if (x[r] > kResetLogDecay) sacc += x[r] * kLog2e;
                        ls[r] = sacc;
                    }
                    float si = sacc;
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, si, d);
                        if ((int)gt >= d) si += y;
                    }
#pragma unroll
                    for (int r = 0; r < 4; ++r) gl[4 * gt + r] = si - sacc + ls[r];
                }
                named_sync(kBarK, kGroupThreads);
                const int pos = c * C + (int)row;   // position in the segment
                wk = row < (uint32_t)C && z_end <= pos ? exp2f(a_end - (a_before + gl[row])) : 0.f;
                a_before += gl[C - 1];
            } else {
                // rows past the chunk (C = 64) are never read by the MMA; keep them finite
                wk = row < (uint32_t)C ? decay_pow(l2, (n - 1 - c) * C + C - 1 - (int)row) : 0.f;
            }
            scale_rows<3>(sm + (uint32_t)s * kStageBytes + kStageK, row, wk);
            fence_proxy_async_smem();
            named_sync(kBarK, kGroupThreads);   // also: every thread is done with gl
            if (gt == 0) mbar_arrive(bar(BAR_KREADY0 + s));
        }
        if (ok && group_wait(bar(BAR_SFULL), 0, ctl, dec, gt, kBarK, kw)) {
            tc_fence_after();
            if (quad < 3) {
                float *dst = a.dS + (((size_t)seg * a.BH + bh) * kDk + row) * kDv;
#pragma unroll 1
                for (int blk = 0; blk < 6; ++blk) {
                    uint32_t r[32];
                    tmem_ld_32cols(tl + blk * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + blk * 32 + e) =
                            make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                                        __uint_as_float(r[e + 3]));
                }
            }
        }
    }
    // Every MMA issued must be complete before TMEM is released.
    if (warp == 1) {
        if (lane == 0) mma_commit(bar(BAR_DONE));
        __syncwarp();
        lane0_wait(bar(BAR_DONE), 0, ctl, lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// S_in(0) = h0 (or 0); S_in(g) = lambda^L S_in(g-1) + dS(g-1), L = seg_chunks * C
// (gated: D(g-1) in place of lambda^L).
// One CTA per (b, h, slice of 1024 state entries); each thread carries one
// float4 through the G segments.
constexpr int kScanSlice = 1024;
static_assert(kStates % kScanSlice == 0 && kScanSlice == 4 * 256, "scan slices");
__global__ void __launch_bounds__(256) gla_seg_scan_kernel(const float *log_lambda, const float *h0,
                                                           const float *dS, float *S_in, int G, int H, int BH,
                                                           int seg_tokens, const float *dseg) {
    const int bh = blockIdx.x / (kStates / kScanSlice), slice = blockIdx.x % (kStates / kScanSlice);
    const int h = bh % H;
    const float wL = dseg ? 0.f : decay_pow(log2_of_decay(log_lambda[h]), seg_tokens);
    const size_t off = (size_t)bh * kStates + (size_t)slice * kScanSlice + 4 * threadIdx.x;
    float4 s = h0 ? *reinterpret_cast<const float4 *>(h0 + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < G; ++g) {
        *reinterpret_cast<float4 *>(S_in + (size_t)g * BH * kStates + off) = s;
        if (g + 1 < G) {
            const float4 x = *reinterpret_cast<const float4 *>(dS + (size_t)g * BH * kStates + off);
            const float w = dseg ? dseg[(size_t)g * BH + bh] : wL;
            s = make_float4(fmaf(w, s.x, x.x), fmaf(w, s.y, x.y), fmaf(w, s.z, x.z), fmaf(w, s.w, x.w));
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

}  // namespace

int device_sm_count() { return sm_count(); }

SegPlan plan_segments(int B, int T, int H, int chunk) {
    SegPlan p{1, 0};
    const int nck = (T + chunk - 1) / chunk;
    p.seg_chunks = nck;
    const long units = 2L * B * H;
    const int sms = sm_count();
    if (units <= 0 || units >= sms || nck < 16) return p;
    int G = (int)((2L * sms) / units);
    G = min(G, nck / 8);
    if (G < 2) return p;
    p.seg_chunks = (nck + G - 1) / G;
    if (chunk == 64) p.seg_chunks += p.seg_chunks & 1;   // the state pass then runs 128-token tiles
    p.nseg = (nck + p.seg_chunks - 1) / p.seg_chunks;
    if (p.nseg < 2) p.seg_chunks = nck;
    return p;
}

size_t seg_workspace_bytes(int B, int H, const SegPlan &p, bool gated) {
    if (p.nseg <= 1) return 0;
    return 2 * (size_t)p.nseg * B * H * kStates * sizeof(float) +
           (gated ? (((size_t)p.nseg * B * H * sizeof(float) + 255) & ~(size_t)255) : 0);
}

cudaError_t launch_seg_prologue(const FwdParams &p, const SegPlan &plan, float **S_in, cudaStream_t s,
                                int *launches) {
    float *dS = static_cast<float *>(p.workspace);
    *S_in = dS + (size_t)plan.nseg * p.B * p.H * kStates;
    // A segment's state does not depend on the chunk length (each token's weight
    // is the decay of the segment's tokens after it): with 64-token chunks the
    // pass runs over 128-token tiles when a segment holds an even number of chunks.
    const bool wide = p.chunk == 64 && plan.seg_chunks % 2 == 0;
    const int tile = wide ? 128 : p.chunk, tiles = wide ? plan.seg_chunks / 2 : plan.seg_chunks;
    CUtensorMap mk, mv;
    cudaError_t e;
    if ((e = make_token_map(&mk, p.k, p.B, p.T, p.H, kDk, tile)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, p.B, p.T, p.H, kDv, tile)) != cudaSuccess) return e;
    auto kernel = p.g ? gla_seg_state_kernel<true> : gla_seg_state_kernel<false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    float *dseg = p.g ? *S_in + (size_t)plan.nseg * p.B * p.H * kStates : nullptr;
    SegArgs a{p.log_lambda, dS, p.H, tile, tiles, p.B * p.H, p.status, p.g, p.T, dseg};
    // The last segment's own contribution is never needed: G-1 segments per sequence.
    kernel<<<(unsigned)(p.B * p.H * (plan.nseg - 1)), kThreads, kSmemBytes, s>>>(mk, mv, a);
    if (launches) ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    gla_seg_scan_kernel<<<(unsigned)(p.B * p.H * (kStates / kScanSlice)), 256, 0, s>>>(
        p.log_lambda, p.h0, dS, *S_in, plan.nseg, p.H, p.B * p.H, plan.seg_chunks * p.chunk, dseg);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
