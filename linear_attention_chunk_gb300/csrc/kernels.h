// kernels.h -- internal launch interface between the C ABI (gla_abi.cu) and
// the kernel translation units. Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gla {

struct FwdParams {
    const void *q, *k, *v;
    const float *log_lambda;
    const float *h0;
    float scale;
    int B, T, H, dk, dv, chunk;
    void *o;
    float *hT;
    void *workspace;
    size_t workspace_bytes;
    unsigned int *status;  // device status word
    // Per-token log-decay [B, T, H] (the gated forward), replacing log_lambda;
    // NULL for the fixed per-head decay.
    const float *g;
};

struct BwdParams {
    const void *q, *k, *v;
    const float *log_lambda;
    const float *h0;
    float scale;
    const void *do_;
    const float *dhT;
    int B, T, H, dk, dv, chunk;
    void *dq_out, *dk_out, *dv_out;
    float *dh0;
    void *workspace;
    size_t workspace_bytes;
    unsigned int *status;
    // Gated backward: per-token log-decays [B, T, H] replacing log_lambda, and
    // the gate gradient dg [B, T, H] fp32 (written).
    const float *g;
    float *dg;
};

struct VarlenParams {
    const void *q, *k, *v;      // packed [total_T, H, d]
    const float *log_lambda;
    float scale;
    const int *cu_seqlens;      // [nseq + 1], device
    const int *slots;           // [nseq], device, or NULL
    float *pool;                // [n_slots, H, dk, dv] fp32 states
    int n_slots, nseq, total_T, H, dk, dv, chunk;
    void *o;                    // packed [total_T, H, dv]
    unsigned int *status;
    const float *g;             // gated: per-token log-decays [total_T, H], or NULL
};

struct DecodeParams {
    const void *q, *k, *v;
    const float *log_lambda;
    float *S;
    float scale;
    int N, H, dk, dv;
    void *o;                 // o, or z when g is given
    unsigned int *status;
    // mixer epilogue (g != NULL): aug [H, dk] (NULL: 0), norm_w [H, dv] (NULL: 1)
    const void *g;
    const float *aug, *norm_w;
    float eps;
    // Per-(sequence, head) log-decay [N, H] replacing log_lambda, or NULL.
    const float *log_decay;
};

// The mixer epilogue over [NT, H, d] rows (epilogue.cu).
struct EpilogueParams {
    const void *o, *q, *k, *v, *g;
    const float *aug, *norm_w;
    float eps;
    int NT, H, dk, dv;
    void *z;
};
cudaError_t launch_mixer_epilogue(const EpilogueParams &p, bool bf16, cudaStream_t s, int *launches);
// The rest of the epilogue over rows of p.o that already hold u = o +
// sigmoid(q . (aug * k)) v (bf16, dk = 96, dv = 192; p.o may be p.z): the
// RMS normalisation, the norm weight and SiLU(g), into p.z.
cudaError_t launch_mixer_finish(const EpilogueParams &p, cudaStream_t s, int *launches);

// The causal depthwise Conv1d (width 4) with SiLU (conv.cu). Batched: nseq
// sequences of T tokens, window n at win_in / win_out + n*4*D (either may be
// NULL). Varlen: cu_seqlens / slots on the device, the window pool
// [n_slots, 4, D] at win_in == win_out. Step: one token per sequence,
// window [nseq, 4, D] at win_out, in place.
struct ConvParams {
    const void *x;
    const float *w, *b;          // [D, 4], [D] or NULL
    const int *cu_seqlens, *slots;
    const float *win_in;
    float *win_out;
    int n_slots, nseq;
    long NT;                     // tokens in x
    int T, D;
    void *y;
    unsigned int *status;
};
// Diagnostic: make the bounded device waits run out (selftest.cu).
cudaError_t launch_selftest_wait(unsigned int *status, uint64_t limit_ns, int *result, cudaStream_t s,
                                 int *launches);
cudaError_t launch_conv_fwd(const ConvParams &p, bool varlen, bool bf16, cudaStream_t s, int *launches);
cudaError_t launch_conv_step(const ConvParams &p, bool bf16, cudaStream_t s, int *launches);

// SIMT kernels (any dk <= 128, dv <= 256; fp32 or bf16 elements).
cudaError_t launch_fwd_simt(const FwdParams &p, bool bf16, cudaStream_t s, int *launches);
cudaError_t launch_bwd_simt(const BwdParams &p, bool bf16, cudaStream_t s, int *launches);

// Decode step (bandwidth kernel; dk=96/dv=192 fast path, generic otherwise).
cudaError_t launch_decode(const DecodeParams &p, bool bf16, cudaStream_t s, int *launches);

// hT = h0 (or 0) for an empty sequence.
cudaError_t launch_copy_state(const float *src, float *dst, size_t n, cudaStream_t s, int *launches);

// tcgen05 / TMA tensor-core kernels (bf16, dk = 96, dv = 192). The forward
// runs on the one-CTA-per-(b, h) kernel, segmented when the plan and the
// workspace allow, and on the dv-half kernel (two CTAs per chain) when few
// chains run unsegmented; the variable-length prefill likewise by its
// number of (sequence, head) chains.
// epi (or NULL): the mixer epilogue over the output, z in place of o: its
// self-augmentation fused into the one-CTA-per-chain kernel's output stage
// at C = 128 and the rest in launch_mixer_finish, else one launch of
// launch_mixer_epilogue after the forward.
cudaError_t launch_fwd_tc(const FwdParams &p, cudaStream_t s, int *launches, const EpilogueParams *epi = nullptr);
// The forward with one CTA per (b, h) holding the whole state (fwd_full.cu);
// S_in (or NULL: p.h0) holds each segment's initial state when nseg > 1.
// epi (or NULL): the mixer epilogue's self-augmentation fused into the
// output stage (per-head decay, chunk 128): rows leave as u = o +
// sigmoid(q . (aug * k)) v, for launch_mixer_finish to normalise them and
// apply the norm weight and the SiLU gate.
cudaError_t launch_fwd_full_tc(const FwdParams &p, float *S_in, int nseg, int seg_chunks, cudaStream_t s,
                               int *launches, const EpilogueParams *epi = nullptr);
// dv and dh0 of the per-token decay's backward on the one-CTA-per-(b, h)
// kernel in reverse time (p.g required).
cudaError_t launch_bwd_dv_full_tc(const BwdParams &p, cudaStream_t s, int *launches);
// Variable-length forward with the states in a pool (bf16, dk = 96, dv = 192).
cudaError_t launch_fwd_varlen_tc(const VarlenParams &p, cudaStream_t s, int *launches);
// The same on the one-CTA-per-(sequence, head) kernel (fwd_full.cu).
cudaError_t launch_fwd_varlen_full_tc(const VarlenParams &p, cudaStream_t s, int *launches);
cudaError_t launch_bwd_tc(const BwdParams &p, cudaStream_t s, int *launches);
// dq and dk: the transposed-shape chunk kernel (192-wide scores, 96-wide outputs).
cudaError_t launch_bwd_dq_tc(const BwdParams &p, cudaStream_t s, int *launches);
cudaError_t launch_bwd_dk_tc(const BwdParams &p, cudaStream_t s, int *launches);
// dk, dv and dh0 of the per-head decay in one launch: the dk and the dv chain
// of each (b, h) on neighbouring CTAs, so q and do are read from DRAM once.
cudaError_t launch_bwd_kv_tc(const BwdParams &p, cudaStream_t s, int *launches);
// The gated backward (p.g, p.dg set): dq, dk, dv, dh0 by the three chunk
// kernels in gated mode, the dq and dk kernels saving the bf16 state copy of
// every chunk in the workspace, then dg from those copies (dg_tc.cu).
cudaError_t launch_bwd_gated_tc(const BwdParams &p, cudaStream_t s, int *launches);
cudaError_t launch_bwd_dg_tc(const BwdParams &p, cudaStream_t s, int *launches);
// Workspace of the gated backward: two bf16 96 x 192 state copies per
// (b, h, chunk), in the layout the chunk kernels keep them in shared memory
// (bwd_gated_tc_state_bytes), then a 16-byte work counter of the dg kernel.
size_t bwd_gated_tc_state_bytes(int B, int T, int H, int chunk);
size_t bwd_gated_tc_workspace_size(int B, int T, int H, int chunk);
size_t fwd_tc_workspace_size(int B, int T, int H, int chunk, bool gated = false);

// Sequence segmentation of the forward (seg_tc.cu): a plan, its workspace,
// and the two launches that produce each segment's initial state.
struct SegPlan {
    int nseg;        // 1: no segmentation
    int seg_chunks;  // chunks per segment (the last may be shorter)
};
SegPlan plan_segments(int B, int T, int H, int chunk);
// The current device's SM count (152 if it cannot be read).
int device_sm_count();
size_t seg_workspace_bytes(int B, int H, const SegPlan &p, bool gated = false);
cudaError_t launch_seg_prologue(const FwdParams &p, const SegPlan &plan, float **S_in, cudaStream_t s,
                                int *launches);
size_t bwd_tc_workspace_size(int B, int T, int H, int chunk);

// Per-thread error detail, set by the launchers on failure.
void set_error_detail(const char *fmt, ...);
// Clears this thread's error detail and launch count (the start of a call).
void reset_call_state();

}  // namespace gla
