// dg_tc.cu -- the gate gradient of the per-token decay form, formed chunk by
// chunk on the tcgen05 tensor core, sm_103a.
//
// The gated form S_t = exp(g_t) S_{t-1} + k_t v_t^T, o_t = s S_t^T q_t is the
// data-dependent counterpart of the per-head decay of the "GLA mixer" of
// "Beyond the KV cache: Training and serving i14's Laplace 3B linear attention
// model on AWS Trainium2 with native PyTorch" (the pages run the mixer through
// the fused GLA chunk kernel family, "Challenge 1", and train through every
// serial update, "Challenge 3"). With G_t = dL/dS_t, the gradient of a gate is
//   dg_t = exp(g_t) <G_t, S_{t-1}>.
// Inside a chunk of Cc tokens (0-based i, j, t) that enters with state S_prev
// and whose last state receives the gradient G_out from later tokens (and
// dhT), with D(x..y) the decay of the chunk's tokens x..y (1 for an empty
// run), this splits exactly into four parts:
//   dg_t = sum_{i >= t > j} M_ij + sum_{i >= t} r_i + sum_{j < t} e_j + z
//   M_ij = s D(j+1..i) (q_i.k_j) (do_i.v_j)      for j < i
//   r_i  = s D(0..i) q_i^T S_prev do_i
//   e_j  = D(j+1..Cc-1) k_j^T G_out v_j
//   z    = D(0..Cc-1) <G_out, S_prev>
// Each part is a product of decays (all <= 1) and the data, local to the
// chunk. The identity dg_t = sum_{r >= t} (q_r.dq_r - k_r.dk_r), by contrast,
// sums a difference over the whole rest of the sequence and loses 1-3 % of
// max |dg| to the bf16 rounding of its operands.
//
// S_prev and G_out / s are the bf16 state copies that the dq and dk kernels
// save for every chunk (bwd_tc.cu). The rectangle sum is formed from the
// column and row sums of M: sum_{i >= t > j} M_ij = sum_{u < t} (col_u -
// row_u) with col_u = sum_{i > u} M_iu and row_u = sum_{j < u} M_uj; that
// difference cancels only inside one chunk, in fp32, from the fp32 score
// accumulators.
//
// The chunks are independent, there is no state chain: one persistent CTA
// per SM takes (b, h, chunk) units from a counter in the workspace until
// none are left. Warp 0 loads (TMA tiles of q, k, v, do; 1-D bulk copies of
// the two saved states), warp 1 owns TMEM and issues four MMAs: the scores
// A = Q K^T and X = dO V^T (N = C), and R1 = dO S_prev^T and E1 = V
// (G_out/s)^T (N = 96), so that r_i = s D(0..i) q_i.R1_i and e_j =
// s D(j+1..Cc-1) k_j.E1_j. Warps 2-9 hold one token row per thread, two warps
// per TMEM lane quadrant (warps 2-5 and 6-9). As soon as a unit's tiles land
// they take their q (first warp of a pair) or k row (second) into registers
// and the z sum from the two copies; once its MMAs are complete, shared
// memory is handed back and the next unit's loads overlap the rest, which
// reads only TMEM: r and e, and M with the decays walked along the per-token
// factors, the first of each pair the even 32-column blocks of M, the second
// the odd ones; each block's column sums come from a transposing warp
// reduction. Warps 2-5 then add up the row's parts, run the two scans and
// write dg; the next unit's MMAs wait only for TMEM.
#include <cuda.h>

#include <algorithm>

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
constexpr int kThreads = 320;
constexpr uint32_t kBarCompute = 1;                  // named barrier of the eight compute warps
constexpr uint32_t kBarRows = 2;                     // named barrier of the first four (the scans)
constexpr uint32_t kComputeThreads = 256;
constexpr uint32_t kSbBlk = kDk * 64;                // saved state copy: [96 rows][32 bf16] blocks
constexpr uint32_t kStateCopyBytes = 6 * kSbBlk;
constexpr uint32_t kOffQ = 0, kOffK = 3 * kBlk, kOffV = 6 * kBlk, kOffDo = 12 * kBlk;
constexpr uint32_t kOffS = 18 * kBlk, kOffG = kOffS + kStateCopyBytes;
constexpr uint32_t kOffGate = kOffG + kStateCopyBytes;   // Gl [128] f32, Zc [128] i32, Af [128] f32
constexpr uint32_t kOffCol = kOffGate + 128 * 12;         // [4][128] column sums of M per warp
constexpr uint32_t kOffRed = kOffCol + 4 * 128 * 4;       // [3][4] per-warp totals of the scans
constexpr uint32_t kOffXch = kOffRed + 64;                 // [128] e_j, [128] partial row sums, [8] z parts
constexpr uint32_t kOffBar = kOffXch + (2 * 128 + 8) * 4;
// LOAD: a unit's tiles landed (or the end marker); MMA: its products are in
// TMEM; SMEM: the compute warps are done with its tiles (after MMA); TMEM:
// they are done with its products.
enum { BAR_LOAD, BAR_MMA, BAR_SMEM, BAR_TMEM, kNumBars };
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;     // tmem base, abort flag, 2 verdicts, 2 unit slots
constexpr uint32_t kSmemUsed = kOffMisc + 32;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffS % 1024 == 0 && kOffG % 1024 == 0, "the saved copies keep their 64-byte swizzle phase");
static_assert(kOffGate % 16 == 0, "the decay factors are read as float4");

constexpr uint32_t kTmemCols = 512, kColA = 0, kColX = 128, kColR = 256, kColE = 352;

struct DgArgs {
    const float *g;                    // [B, T, H] log-decays
    const unsigned char *saved_s;      // S_prev copy per (b, h, chunk)
    const unsigned char *saved_g;      // G_out / s copy per (b, h, chunk)
    float *dg;                         // [B, T, H]
    unsigned int *next_unit;           // work counter, zero at launch
    float scale;
    int T, H, C, nck, nunits;
    unsigned int *status;
};

// Lane l of a warp holding 32 values each returns the sum over the warp's
// lanes of value l (a transposing reduction: 31 shuffles).
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
    for (int sft = 16; sft >= 1; sft >>= 1) {
        const bool up = (lane & sft) != 0;
#pragma unroll
        for (int i = 0; i < sft; ++i) {
            const float send = up ? v[i] : v[i + sft];
            const float keep = up ? v[i + sft] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
        }
    }
    return v[0];
}

// One compute thread waits on an mbarrier; the verdict goes through a
// two-slot flag so that all eight compute warps take the same branch after
// their named barrier.
__device__ __forceinline__ bool compute_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl,
                                             volatile int *decision, uint32_t ct, uint32_t &k) {
    if (ct == 0) decision[k & 1] = mbar_wait(bar, parity, ctl) ? 0 : 1;
    named_sync(kBarCompute, kComputeThreads);
    return decision[(k++) & 1] == 0;
}

// Dot product of 32 fp32 values (raw bits, from TMEM) with 32 bf16 held as
// four 16-byte vectors.
__device__ __forceinline__ float dot_row_regs(const uint32_t (&x)[32], const uint4 *r) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {r[c].x, r[c].y, r[c].z, r[c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16x2(w[e]);
            acc = fmaf(f.x, __uint_as_float(x[8 * c + 2 * e]), acc);
            acc = fmaf(f.y, __uint_as_float(x[8 * c + 2 * e + 1]), acc);
        }
    }
    return acc;
}

__global__ void __launch_bounds__(kThreads, 1)
    gla_dg_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const DgArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_u32(sm);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int C = a.C;

    float *Gl = reinterpret_cast<float *>(sm + kOffGate);
    int *Zc = reinterpret_cast<int *>(sm + kOffGate + 512);
    float *Af = reinterpret_cast<float *>(sm + kOffGate + 1024);
    float *colp = reinterpret_cast<float *>(sm + kOffCol);
    float *red = reinterpret_cast<float *>(sm + kOffRed);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kOffMisc + 4);
    volatile int *decision = reinterpret_cast<volatile int *>(sm + kOffMisc + 8);   // [2]
    volatile int *unit_slot = reinterpret_cast<volatile int *>(sm + kOffMisc + 16); // [2]: unit, or -1 at the end
    const WaitCtl ctl{abort_flag, a.status};
    auto bar = [&](int i) { return base + kOffBar + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
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
        // ------------------------------------------------------------- loads
        if (lane == 0) {
            const uint32_t fb = bar(BAR_LOAD);
            uint32_t issued = 0;
            bool failed = false;
            int u = (int)atomicAdd(a.next_unit, 1u);   // the ticket is taken ahead of the wait
            for (uint32_t k = 0;; ++k) {
                // Unit k - 1's tiles are free once its MMAs are complete and the
                // compute warps have read their rows and the z sum.
                if (k > 0 && !mbar_wait(bar(BAR_SMEM), (k - 1) & 1u, ctl)) {
                    failed = true;
                    break;
                }
                if (u >= a.nunits) {
                    unit_slot[k & 1] = -1;
                    mbar_arrive(fb);   // completes the phase with no bytes: the end marker
                    break;
                }
                unit_slot[k & 1] = u;
                const int nc = u % a.nck, bh = u / a.nck;
                const int b = bh / a.H, h = bh % a.H, t0 = nc * C;
                const size_t slot = ((size_t)bh * a.nck + nc) * kStateCopyBytes;
                mbar_arrive_expect_tx(fb, 18u * (uint32_t)C * 64u + 2u * kStateCopyBytes);
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(base + kOffQ + j * kBlk, &tm_q, fb, 32 * j, h, t0, b);
#pragma unroll
                for (int j = 0; j < 3; ++j) tma_load_4d(base + kOffK + j * kBlk, &tm_k, fb, 32 * j, h, t0, b);
#pragma unroll
                for (int j = 0; j < 6; ++j) tma_load_4d(base + kOffV + j * kBlk, &tm_v, fb, 32 * j, h, t0, b);
#pragma unroll
                for (int j = 0; j < 6; ++j) tma_load_4d(base + kOffDo + j * kBlk, &tm_do, fb, 32 * j, h, t0, b);
                bulk_load(base + kOffS, a.saved_s + slot, kStateCopyBytes, fb);
                bulk_load(base + kOffG, a.saved_g + slot, kStateCopyBytes, fb);
                ++issued;
                u = (int)atomicAdd(a.next_unit, 1u);
            }
            // On the error path the last copies may still be in flight: they must
            // land before the CTA exits. (On the normal path the compute warps
            // have consumed every unit's tiles before the end marker.)
            if (failed && issued > 0) mbar_wait_drain(fb, (issued - 1) & 1u, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMAs
        if (lane == 0) {
            uint32_t committed = 0;
            const uint32_t idS = idesc_bf16(128, C, false, false);     // scores: both K-major
            const uint32_t id96 = idesc_bf16(128, kDk, false, false);  // state products: copy K-major
            for (uint32_t k = 0;; ++k) {
                if (!mbar_wait(bar(BAR_LOAD), k & 1u, ctl)) break;
                if (unit_slot[k & 1] < 0) break;
                // the compute warps are done with unit k - 1's products
                if (k > 0 && !mbar_wait(bar(BAR_TMEM), (k - 1) & 1u, ctl)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 6; ++ks) {
                    const uint32_t off = (uint32_t)(ks >> 1) * kBlk + (uint32_t)(ks & 1) * 32;
                    mma_bf16_ss(tmem + kColA, smem_desc(base + kOffQ + off, 16, 512, 4),
                                smem_desc(base + kOffK + off, 16, 512, 4), idS, ks > 0);
                }
#pragma unroll
                for (int ks = 0; ks < 12; ++ks) {
                    const uint32_t off = (uint32_t)(ks >> 1) * kBlk + (uint32_t)(ks & 1) * 32;
                    const uint32_t soff = (uint32_t)(ks >> 1) * kSbBlk + (uint32_t)(ks & 1) * 32;
                    mma_bf16_ss(tmem + kColX, smem_desc(base + kOffDo + off, 16, 512, 4),
                                smem_desc(base + kOffV + off, 16, 512, 4), idS, ks > 0);
                    mma_bf16_ss(tmem + kColR, smem_desc(base + kOffDo + off, 16, 512, 4),
                                smem_desc(base + kOffS + soff, 16, 512, 4), id96, ks > 0);
                    mma_bf16_ss(tmem + kColE, smem_desc(base + kOffV + off, 16, 512, 4),
                                smem_desc(base + kOffG + soff, 16, 512, 4), id96, ks > 0);
                }
                mma_commit(bar(BAR_MMA));
                ++committed;
            }
            // The MMAs issued must be complete before TMEM is released.
            if (committed > 0) mbar_wait_drain(bar(BAR_MMA), (committed - 1) & 1u, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ------------------------- warps 2-9: one token row each, two warps per row
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t sub = (uint32_t)(warp - 2) >> 2;           // 0: warps 2-5, 1: warps 6-9
        const uint32_t row = quad * 32 + (uint32_t)lane;
        const uint32_t ct = (uint32_t)threadIdx.x - 64;          // 0..255
        const uint32_t tl = tmem + ((quad * 32) << 16);
        const int nblk = C / 32;
        const float s = a.scale;
        float *xe = reinterpret_cast<float *>(sm + kOffXch);     // e_j of each row
        float *xrow = xe + 128;                                   // the second warp's part of each row sum
        float *xz = xrow + 128;                                   // per-warp parts of z
        uint32_t kw = 0;
        for (uint32_t k = 0;; ++k) {
            // Every compute thread takes the same branch: one waits, all read the verdict.
            if (!compute_wait(bar(BAR_LOAD), k & 1u, ctl, decision, ct, kw)) break;
            const int u = unit_slot[k & 1];
            if (u < 0) break;
            const int nc = u % a.nck, bh = u / a.nck;
            const int b = bh / a.H, h = bh % a.H, t0 = nc * C, Cc = min(C, a.T - t0);
            const bool in = (int)row < Cc;
            // The chunk's gates (the first warp): issued now, scanned after the reads below.
            float gx[4];
            if (ct < 32) {
                const float *gh = a.g + ((size_t)b * a.T + t0) * a.H + h;
#pragma unroll
                for (int r = 0; r < 4; ++r) gx[r] = 4 * lane + r < Cc ? gh[(size_t)(4 * lane + r) * a.H] : 0.f;
            }
            // <G_out / s, S_prev> over this thread's share of the two copies (same layout)
            float zpart = 0.f;
            for (uint32_t i = ct; i < kStateCopyBytes / 16; i += kComputeThreads) {
                const uint4 us = ld_shared_v4(base + kOffS + i * 16), ug = ld_shared_v4(base + kOffG + i * 16);
                const uint32_t ws[4] = {us.x, us.y, us.z, us.w}, wg[4] = {ug.x, ug.y, ug.z, ug.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 fs = unpack_bf16x2(ws[e]), fg = unpack_bf16x2(wg[e]);
                    zpart = fmaf(fs.x, fg.x, zpart);
                    zpart = fmaf(fs.y, fg.y, zpart);
                }
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) zpart += __shfl_xor_sync(0xffffffffu, zpart, d);
            if (lane == 0) xz[sub * 4 + quad] = zpart;
            // This thread's q (first warp of a pair) or k row (second), for r or e.
            uint4 rr[12];
            {
                const uint32_t tile = base + (sub == 0 ? kOffQ : kOffK);
#pragma unroll
                for (int blk = 0; blk < 3; ++blk)
#pragma unroll
                    for (int c = 0; c < 4; ++c) rr[4 * blk + c] = ld_shared_v4(tile + blk * kBlk + sw64_offset(row, (uint32_t)c));
            }
            if (ct < 32) gate_scan_store(gx, lane, Gl, Zc, Af);
            // The barrier inside also orders the reads above before the hand-back of
            // shared memory, and the gate arrays before their readers.
            if (!compute_wait(bar(BAR_MMA), k & 1u, ctl, decision, ct, kw)) break;
            if (ct == 0) mbar_arrive(bar(BAR_SMEM));
            tc_fence_after();
            const float gi = Gl[row];
            const int zi = Zc[row];
            const int last = Cc - 1;
            // r_i = s D(0..i) q_i.R1_i (first warp of the pair), e_j = s D(j+1..Cc-1)
            // k_j.E1_j (second)
            float dot = 0.f;
            {
                const uint32_t col0 = tl + (sub == 0 ? kColR : kColE);
                uint32_t x0[32], x1[32];
                tmem_ld_32cols(col0, x0);
                tmem_ld_32cols(col0 + 32u, x1);
                tmem_ld_wait();
                dot = dot_row_regs(x0, &rr[0]) + dot_row_regs(x1, &rr[4]);
                tmem_ld_32cols(col0 + 64u, x0);
                tmem_ld_wait();
                dot += dot_row_regs(x0, &rr[8]);
            }
            const float r_i = sub == 0 && in && zi < 0 ? s * exp2f(gi) * dot : 0.f;
            if (sub == 1) xe[row] = in && Zc[last] <= (int)row ? s * exp2f(Gl[last] - gi) * dot : 0.f;
            // M row i = row: blocks of 32 columns j < i (this warp's half of them),
            // weights D(j+1..i) walked leftwards from each block's last column (the
            // diagonal block from the row's own column, which is excluded).
            float rowsum = 0.f;
#pragma unroll 1
            for (int bj = (int)sub; bj < nblk; bj += 2) {
                float m[32];
                if (bj <= (int)quad) {
                    uint32_t xa[32], xx[32];
                    tmem_ld_32cols(tl + kColA + 32u * bj, xa);
                    tmem_ld_32cols(tl + kColX + 32u * bj, xx);
                    const bool dgb = bj == (int)quad;
                    const int jr = 32 * bj + 31;
                    const int dl = dgb ? lane : 32;
                    float d = dgb || zi > jr ? 0.f : ex2_approx(gi - Gl[jr]);
                    tmem_ld_wait();
#pragma unroll
                    for (int mm = 7; mm >= 0; --mm) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(Af + 32 * bj + 4 * mm);
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int r = 3; r >= 0; --r) {
                            const int e = 4 * mm + r;
                            d = e == dl ? 1.f : d;
                            const float v = s * d * __uint_as_float(xa[e]) * __uint_as_float(xx[e]);
                            m[e] = in && e != dl ? v : 0.f;
                            d *= av[r];
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) rowsum += m[e];
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) m[e] = 0.f;
                }
                colp[quad * 128 + 32 * bj + lane] = warp_transpose_sum(m, lane);
            }
            if (sub == 1) xrow[row] = rowsum;
            tc_fence_before();
            named_sync(kBarCompute, kComputeThreads);
            if (ct == 0) mbar_arrive(bar(BAR_TMEM));   // the next unit's MMAs may overwrite TMEM
            if (sub == 0) {
                // Scans over the chunk's rows: w_u = col_u - row_u + e_u (exclusive
                // prefix), r_i (inclusive suffix); z over the block.
                float col = 0.f;
                for (int qd = 0; qd < 4; ++qd) col += colp[qd * 128 + row];
                const float w = in ? col - (rowsum + xrow[row]) + xe[row] : 0.f;
                float wi = w, rs = r_i;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const float yw = __shfl_up_sync(0xffffffffu, wi, d);
                    const float yr = __shfl_down_sync(0xffffffffu, rs, d);
                    if (lane >= d) wi += yw;
                    if (lane + d < 32) rs += yr;
                }
                if (lane == 31) red[quad] = wi;          // warp totals of w
                if (lane == 0) red[4 + quad] = rs;       // warp totals of r
                named_sync(kBarRows, 128);
                float wpre = 0.f, rsuf = 0.f, z = 0.f;
                for (int qd = 0; qd < 4; ++qd) {
                    if (qd < (int)quad) wpre += red[qd];
                    if (qd > (int)quad) rsuf += red[4 + qd];
                }
                for (int k8 = 0; k8 < 8; ++k8) z += xz[k8];
                const float dchunk = Zc[last] < 0 ? exp2f(Gl[last]) : 0.f;
                float dg = s * dchunk * z + (wpre + wi - w) + (rsuf + rs);
                if (in) {
                    const size_t gidx = ((size_t)b * a.T + t0 + row) * a.H + h;
                    if (!(a.g[gidx] > kResetLogDecay)) dg = 0.f;   // a clearing gate: exp(g) = 0
                    a.dg[gidx] = dg;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_bwd_dg_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    if (p.dk != kDk || p.dv != kDv || !p.g || !p.dg) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv, mdo;
    cudaError_t e;
    if ((e = make_token_map(&mq, p.q, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mk, p.k, p.B, p.T, p.H, kDk, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mv, p.v, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    if ((e = make_token_map(&mdo, p.do_, p.B, p.T, p.H, kDv, p.chunk)) != cudaSuccess) return e;
    const int nck = (p.T + p.chunk - 1) / p.chunk;
    const size_t nunits = (size_t)p.B * p.H * nck;
    if (nunits == 0) return cudaSuccess;
    if (nunits > 0x7fffffffu - 1024u) return cudaErrorInvalidValue;   // the work counter's range
    unsigned char *ws = static_cast<unsigned char *>(p.workspace);
    const size_t half = bwd_gated_tc_state_bytes(p.B, p.T, p.H, p.chunk) / 2;
    unsigned int *counter = reinterpret_cast<unsigned int *>(ws + 2 * half);
    if ((e = cudaMemsetAsync(counter, 0, sizeof(unsigned int), s)) != cudaSuccess) return e;
    DgArgs a{p.g, ws, ws + half, p.dg, counter, p.scale, p.T, p.H, p.chunk, nck, (int)nunits, p.status};
    e = cudaFuncSetAttribute(gla_dg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)std::min<size_t>(nunits, (size_t)device_sm_count());
    gla_dg_kernel<<<grid, kThreads, kSmemBytes, s>>>(mq, mk, mv, mdo, a);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
