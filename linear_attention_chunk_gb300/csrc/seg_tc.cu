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
//   1. gla_seg_state_kernel: per (b, h, dv half, segment) the segment's local
//      end state dS_g from zero (the state-update chain alone, k and v only);
//   2. gla_seg_scan_kernel: S_in(0) = h0, S_in(g) = lambda^L(g-1) S_in(g-1) + dS_(g-1);
//   3. the forward kernel on every segment at once, each from S_in(g).
// This reads k and v twice (1,728 instead of 1,152 bytes per head-token) in
// exchange for B*H*2*G CTAs instead of B*H*2.
// Workspace: dS and S_in, each [G][B][H][96][192] fp32.
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
constexpr int kStates = kDk * kDv;                  // floats per (b, h) state
constexpr int kThreads = 320;
constexpr int kStages = 3;
constexpr uint32_t kStageK = 0;                     // 4 blocks (the 4th stays zero: dk pad to 128)
constexpr uint32_t kStageV = 4 * kBlk;              // 3 blocks
constexpr uint32_t kStageBytes = 7 * kBlk;          // 56 KB
constexpr uint32_t kOffPw = kStages * kStageBytes;
enum { BAR_FULL0 = 0, BAR_EMPTY0 = kStages, BAR_KREADY0 = 2 * kStages, BAR_SREADY = 3 * kStages, BAR_SFULL,
       BAR_DONE, kNumBars };
constexpr uint32_t kOffBar = kOffPw + 132 * 4;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 32 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kBarK = 1, kBarE = 2;

struct SegArgs {
    const float *log_lambda;
    float *dS;             // [G][B][H][96][192]
    int T, H, C, nck, seg_chunks, BH;
    unsigned int *status;
};

__global__ void __launch_bounds__(kThreads, 1)
    gla_seg_state_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const SegArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = blockIdx.x & 1;
    const int seg = (blockIdx.x >> 1) / a.BH;
    const int bh = (blockIdx.x >> 1) % a.BH;
    const int b = bh / a.H, h = bh % a.H;
    const int C = a.C, T = a.T;
    const int cbeg = seg * a.seg_chunks;
    const int nck = min(a.seg_chunks, a.nck - cbeg);
    const int ksteps_tok = C / 16;

    float *pw = reinterpret_cast<float *>(sm + kOffPw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    volatile int *dec = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);
    const WaitCtl ctl{abort_flag, a.status};
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < 4; ++i) dec[i] = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    {
        const float l2 = log2_of_decay(a.log_lambda[h]);
        for (int n = threadIdx.x; n < 132; n += kThreads) pw[n] = n <= 128 ? decay_pow(l2, n) : 0.f;
    }
    for (uint32_t i = threadIdx.x; i < kStages * (kBlk / 16); i += kThreads) {
        const uint32_t s = i / (kBlk / 16), o = (i % (kBlk / 16)) * 16;
        *reinterpret_cast<uint4 *>(sm + s * kStageBytes + kStageK + 3 * kBlk + o) = make_uint4(0, 0, 0, 0);
    }
    if (C < 128) {
        const uint32_t lo = (uint32_t)C * 64, per_blk = (kBlk - lo) / 16;
        for (uint32_t i = threadIdx.x; i < kStages * 7 * per_blk; i += kThreads) {
            const uint32_t blk = i / per_blk, o = lo + (i % per_blk) * 16;
            *reinterpret_cast<uint4 *>(sm + blk * kBlk + o) = make_uint4(0, 0, 0, 0);
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
        const uint32_t tx = 6u * (uint32_t)C * 64u;
        int issued = 0;
        for (int c = 0; c < nck; ++c) {
            const int s = c % kStages;
            if (c >= kStages && !lane0_wait(bar(BAR_EMPTY0 + s), ((c / kStages) - 1) & 1, ctl, lane)) break;
            if (lane == 0) {
                const uint32_t st = base + (uint32_t)s * kStageBytes;
                const uint32_t fb = bar(BAR_FULL0 + s);
                mbar_arrive_expect_tx(fb, tx);
                const int t0 = (cbeg + c) * C;
#pragma unroll
                for (int j = 0; j < 3; ++j) {
                    tma_load_4d(st + kStageK + j * kBlk, &tm_k, fb, 32 * j, h, t0, b);
                    tma_load_4d(st + kStageV + j * kBlk, &tm_v, fb, kDvHalf * half + 32 * j, h, t0, b);
                }
            }
            __syncwarp();
            issued = c + 1;
        }
        for (int c = max(issued - kStages, 0); c < issued; ++c)
            lane0_wait(bar(BAR_FULL0 + c % kStages), (c / kStages) & 1, ctl, lane);
    } else if (warp == 1) {
        const uint32_t idS = idesc_bf16(128, kDvHalf, true, true);
        for (int c = 0; c < nck; ++c) {
            const int s = c % kStages;
            if (!lane0_wait(bar(BAR_FULL0 + s), (c / kStages) & 1, ctl, lane)) break;
            if (!lane0_wait(bar(BAR_KREADY0 + s), (c / kStages) & 1, ctl, lane)) break;
            if (!lane0_wait(bar(BAR_SREADY), c & 1, ctl, lane)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = base + (uint32_t)s * kStageBytes;
                for_token_steps(ksteps_tok, [&](int ks) {
                    mma_bf16_ss(tmem, smem_desc(st + kStageK + (uint32_t)ks * 1024, kBlk, 512, 4),
                                smem_desc(st + kStageV + (uint32_t)ks * 1024, kBlk, 512, 4), idS,
                                (c > 0 || ks > 0) ? 1u : 0u);
                });
                mma_commit(bar(BAR_SFULL));
                mma_commit(bar(BAR_EMPTY0 + s));
            }
            __syncwarp();
        }
        if (lane == 0) mma_commit(bar(BAR_DONE));
        __syncwarp();
        lane0_wait(bar(BAR_DONE), 0, ctl, lane);
    } else if (warp < 6) {
        // K~ = diag(lambda^(Cc-1-j)) K, once the tiles landed
        const uint32_t row = (uint32_t)(warp & 3) * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 64;
        uint32_t kw = 0;
        for (int c = 0; c < nck; ++c) {
            const int s = c % kStages;
            const int Cc = min(C, T - (cbeg + c) * C);
            if (!group_wait(bar(BAR_FULL0 + s), (c / kStages) & 1, ctl, dec, gt, kBarK, kw)) break;
            const float wk = row < (uint32_t)Cc ? pw[Cc - 1 - (int)row] : 0.f;
            scale_rows<3>(sm + (uint32_t)s * kStageBytes + kStageK, row, wk);
            fence_proxy_async_smem();
            named_sync(kBarK, kGroupThreads);
            if (gt == 0) mbar_arrive(bar(BAR_KREADY0 + s));
        }
    } else {
        // S <- lambda^(next chunk's length) S between chunks; dS out at the end
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t gt = (uint32_t)threadIdx.x - 192;
        const uint32_t tl = tmem + ((quad * 32) << 16);
        uint32_t kw = 0;
        named_sync(kBarE, kGroupThreads);
        if (gt == 0) mbar_arrive(bar(BAR_SREADY));           // chunk 0 starts from zero
        for (int c = 0; c < nck; ++c) {
            const bool last = (c == nck - 1);
            if (!group_wait(bar(BAR_SFULL), c & 1, ctl, dec + 2, gt, kBarE, kw)) break;
            tc_fence_after();
            if (quad < 3) {
                const float wn = last ? 1.f : pw[min(C, T - (cbeg + c + 1) * C)];
                float *dst = a.dS + (((size_t)seg * a.BH + bh) * kDk + row) * kDv + kDvHalf * half;
#pragma unroll
                for (int blk = 0; blk < 3; ++blk) {
                    uint32_t r[32];
                    tmem_ld_32cols(tl + blk * 32, r);
                    tmem_ld_wait();
                    if (last) {
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4 *>(dst + blk * 32 + e) =
                                make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                            __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * wn);
                        tmem_st_32cols(tl + blk * 32, r);
                    }
                }
                tmem_st_wait();
            }
            tc_fence_before();
            named_sync(kBarE, kGroupThreads);
            if (gt == 0 && !last) mbar_arrive(bar(BAR_SREADY));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// S_in(0) = h0 (or 0); S_in(g) = lambda^L S_in(g-1) + dS(g-1), L = seg_chunks * C.
// One CTA per (b, h); each thread carries 18 float4 of the 96 x 192 state.
__global__ void __launch_bounds__(256) gla_seg_scan_kernel(const float *log_lambda, const float *h0,
                                                           const float *dS, float *S_in, int G, int H, int BH,
                                                           int seg_tokens) {
    const int bh = blockIdx.x, h = bh % H;
    const float wL = decay_pow(log2_of_decay(log_lambda[h]), seg_tokens);
    constexpr int kVec = kStates / 4 / 256;   // 18
    float4 s[kVec];
    const float4 *src = h0 ? reinterpret_cast<const float4 *>(h0 + (size_t)bh * kStates) : nullptr;
#pragma unroll
    for (int m = 0; m < kVec; ++m) s[m] = src ? src[threadIdx.x + 256 * m] : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < G; ++g) {
        float4 *out = reinterpret_cast<float4 *>(S_in + ((size_t)g * BH + bh) * kStates);
#pragma unroll
        for (int m = 0; m < kVec; ++m) out[threadIdx.x + 256 * m] = s[m];
        if (g + 1 < G) {
            const float4 *d = reinterpret_cast<const float4 *>(dS + ((size_t)g * BH + bh) * kStates);
#pragma unroll
            for (int m = 0; m < kVec; ++m) {
                const float4 x = d[threadIdx.x + 256 * m];
                s[m] = make_float4(fmaf(wL, s[m].x, x.x), fmaf(wL, s[m].y, x.y), fmaf(wL, s[m].z, x.z),
                                   fmaf(wL, s[m].w, x.w));
            }
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 148;
    }
    return n;
}

}  // namespace

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
    p.nseg = (nck + p.seg_chunks - 1) / p.seg_chunks;
    return p;
}

size_t seg_workspace_bytes(int B, int H, const SegPlan &p) {
    if (p.nseg <= 1) return 0;
    return 2 * (size_t)p.nseg * B * H * kStates * sizeof(float);
}

cudaError_t launch_seg_prologue(const FwdParams &p, const SegPlan &plan, float **S_in, cudaStream_t s,
                                int *launches) {
    float *dS = static_cast<float *>(p.workspace);
    *S_in = dS + (size_t)plan.nseg * p.B * p.H * kStates;
    CUtensorMap mk, mv;
    cudaError_t e;
    if ((e = make_token_map(&mk, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gla_seg_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    SegArgs a{p.log_lambda, dS, p.T, p.H, p.chunk, nck, plan.seg_chunks, p.B * p.H, p.status};
    // The last segment's own contribution is never needed; its CTAs still run (cheap) to keep the grid simple.
    gla_seg_state_kernel<<<(unsigned)(2 * p.B * p.H * plan.nseg), kThreads, kSmemBytes, s>>>(mk, mv, a);
    if (launches) ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    gla_seg_scan_kernel<<<(unsigned)(p.B * p.H), 256, 0, s>>>(p.log_lambda, p.h0, dS, *S_in, plan.nseg, p.H,
                                                                p.B * p.H, plan.seg_chunks * p.chunk);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
