/*
 * gla.h -- C ABI of libgla, the Simple Gated Linear Attention (Simple GLA)
 * mixer for NVIDIA GB300 (sm_103a).
 *
 * Source of the operation: "Beyond the KV cache: Training and serving i14's
 * Laplace 3B linear attention model on AWS Trainium2 with native PyTorch".
 *   - Section "i14 and the Laplace 3B architecture", paragraph "GLA mixer"
 *     ("GLA recurrent-state update equation", "GLA state-readout equation"):
 *     each head h keeps a dk x dv matrix state (96 x 192 in the model),
 *     decayed by a fixed per-head factor lambda_h and written by the rank-1
 *     outer product k_t v_t^T; the query reads the state out.
 *   - Section "Engineering challenges", "Challenge 1" ("Chunked GLA
 *     intra-chunk output", "Chunked GLA state update", Figure 3): the
 *     chunked form -- masked linear attention inside a chunk plus the
 *     running state, the state advanced by lambda^C; only the state chain
 *     is serial.
 *   - "Challenge 3: Backward-pass unrolling for a sequential recurrence":
 *     the backward passes through every serial state update.
 *   - "Inference optimization on Trainium2": one fixed state page per
 *     sequence, constant work per generated token.
 *
 * What is computed (0-based token t, per batch row b and head h, with
 * lambda = exp(log_lambda[h]) and lambda^0 = 1 even for lambda = 0):
 *     S_{-1} = h0  (zero when h0 is NULL)
 *     S_t    = lambda * S_{t-1} + k_t v_t^T          (dk x dv, fp32)
 *     o_t    = scale * S_t^T q_t                     (readout after the update)
 *     hT     = S_{T-1}                               (unscaled)
 * The scale multiplies the readout only.
 *
 * Layouts (row-major, contiguous, token-major as a fused per-token QKV
 * projection emits them):
 *     q, k, do, dq, dk   [B, T, H, dk]
 *     v, o, dv           [B, T, H, dv]
 *     h0, hT, dhT, dh0   [B, H, dk, dv]  fp32, dv fastest
 *     decode q, k        [N, H, dk];  v, o [N, H, dv];  S_inout [N, H, dk, dv] fp32
 *     log_lambda         [H] fp32, natural log of the decay (<= 0, -inf allowed)
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers (cudaMalloc'd or equivalent), owned by the
 *     caller; the library never frees or retains them. They must be 16-byte
 *     aligned. Input and output buffers must not alias, except that decode
 *     updates S_inout in place.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL means the legacy default stream). Argument errors are detected on
 *     the host and returned before anything is launched.
 *   - The library allocates no device memory. Scratch, when a path needs
 *     it, is the caller's `workspace`.
 *   - `dtype` selects the element type of q, k, v, o, do, dq, dk, dv
 *     (GLA_BF16: bf16 bit patterns; GLA_FP32: float). States are fp32 in
 *     both modes. GLA_BF16 requires dk = 96, dv = 192 (the tensor-core path);
 *     GLA_FP32 is the validation mode and accepts 1 <= dk <= 128, 1 <= dv <= 256.
 *   - `chunk` is the chunk length C, 64 or 128. T need not be a multiple of
 *     C: the last chunk is ragged. Results do not depend on C beyond rounding.
 *   - B, H, N may be 0 (nothing is launched); T may be 0 for the forward
 *     (then hT = h0, or zero).
 *   - Device-side failures (a wait that timed out) are recorded in a device
 *     status word; gla_check() synchronises the stream and reports them.
 */
#ifndef LIBGLA_GLA_H
#define LIBGLA_GLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GLA_OK = 0,
    GLA_ERR_INVALID_ARG = 1,   /* null or misaligned pointer, bad size, overflow */
    GLA_ERR_UNSUPPORTED = 2,   /* shape or mode this build does not implement   */
    GLA_ERR_CUDA = 3,          /* a CUDA runtime call failed (see gla_last_error) */
    GLA_ERR_TIMEOUT = 4,       /* a device-side wait gave up (reported by gla_check) */
    GLA_ERR_WORKSPACE = 5      /* workspace smaller than the *_workspace_size query */
} gla_status;

typedef enum {
    GLA_BF16 = 0,
    GLA_FP32 = 1
} gla_dtype;

/*
 * gla_chunk_fwd -- chunked forward ("Challenge 1": intra-chunk masked linear
 * attention plus the running state; the state advanced by lambda^C).
 *
 *   q, k [B,T,H,dk], v [B,T,H,dv] (dtype), log_lambda [H] fp32,
 *   h0 [B,H,dk,dv] fp32 or NULL (zero initial state), scale (readout factor),
 *   chunk 64 or 128, o [B,T,H,dv] (dtype, written), hT [B,H,dk,dv] fp32 or
 *   NULL (final state not wanted), workspace/workspace_bytes: optional device
 *   scratch. With at least gla_chunk_fwd_workspace_size() bytes the library
 *   may split long sequences into segments processed in parallel (same
 *   result up to rounding); with less (or NULL) it runs one serial chain per
 *   (b, h). Never fails for lack of workspace.
 */
gla_status gla_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *log_lambda, const float *h0, float scale,
                         int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                         void *o, float *hT,
                         void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace that let gla_chunk_fwd use sequence segmentation for
 * this shape (0 when the shape has enough (b, h) pairs to fill the GPU). */
size_t gla_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                    gla_dtype dtype);

/*
 * gla_chunk_fwd_noalloc -- gla_chunk_fwd for callers that cannot allocate
 * device memory. The method's description has no counterpart to this entry
 * point: it exists for the library's users, not for the mixer's math.
 *
 * Who needs it: code that runs the forward where a cudaMalloc is not
 * allowed -- a plugin whose host framework owns all device memory through
 * its own pool, or a serving loop that must neither stall the device
 * (cudaMalloc can synchronise it) nor fail with out-of-memory mid-step.
 * gla_chunk_fwd asks for a workspace when it splits long sequences into
 * segments; this entry point instead uses a fixed scratch array of
 * GLA_NOALLOC_SCRATCH_BYTES (24 MiB) that the library reserves in each
 * device's memory when it is loaded there, and holds until the process
 * exits. It never calls cudaMalloc, cudaFree or any allocating routine.
 *
 * Arguments, layouts and results are those of gla_chunk_fwd (without the
 * workspace). The segment plan needs at most 2 x SMs x dk x dv x 4 bytes
 * (22.4 MB on the GB300's 152 SMs), so the array covers every shape on a GPU
 * with up to 170 SMs. Should a plan ever need more, the call runs the
 * unsegmented forward (one chain per (b, h), as gla_chunk_fwd does without a
 * workspace): slower on few long sequences, the same result, still no
 * allocation.
 *
 * - The first call on a device that needs scratch looks up the array's
 *   device address (cudaGetSymbolAddress). Make that first call before any
 *   stream capture.
 * - Every call on a device shares the one array and leaves the last call's
 *   contents in it; each call writes every scratch byte it reads, so nothing
 *   has to be cleared between calls.
 * - Calls that overlap on the GPU (on different streams, or from different
 *   host threads without ordering) race on the array: order them.
 */
#define GLA_NOALLOC_SCRATCH_BYTES (24u << 20)
gla_status gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *log_lambda, const float *h0, float scale,
                                 int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                                 void *o, float *hT, void *stream);

/*
 * gla_chunk_fwd_varlen -- the chunked forward over sequences of different
 * lengths packed one after another, each entering from and leaving its state
 * in a state pool shared with gla_decode_step. This is the prefill of a
 * serving loop: requests arrive with prompts of any length, are prefilled
 * together, and continue with decode steps on the same pool (the pages keep
 * each sequence's state in a fixed-size page, "Inference optimization on
 * Trainium2"). The recurrence is that of gla_chunk_fwd.
 *
 *   q, k [total_T, H, dk], v [total_T, H, dv] (bf16), packed: sequence n holds
 *   tokens [cu_seqlens[n], cu_seqlens[n+1]); log_lambda [H] fp32; scale;
 *   cu_seqlens [nseq + 1] int32 in device memory, cu_seqlens[0] = 0,
 *   non-decreasing, cu_seqlens[nseq] <= total_T; slots [nseq] int32 in device
 *   memory or NULL (sequence n uses slot n); state_pool [n_slots, H, dk, dv]
 *   fp32, updated in place: slot slots[n] is read as the initial state of
 *   sequence n and overwritten with its final state (a new sequence's slot
 *   must hold zeros, or the state to continue from); o [total_T, H, dv] bf16
 *   (written for every token of every sequence). chunk 64 or 128; dk = 96,
 *   dv = 192, dtype GLA_BF16 only.
 * - Slots of one call must be distinct. A sequence of length 0 leaves its
 *   slot untouched.
 * - cu_seqlens and slots are device data the host does not read: a bad entry
 *   (a decreasing offset, an offset past total_T, a slot outside
 *   [0, n_slots)) skips that sequence on the device and sets a bit that the
 *   next gla_check() reports as GLA_ERR_INVALID_ARG.
 * - Tokens of different sequences never mix: the last partial chunk of a
 *   sequence masks the next sequence's rows and stores its outputs row by row.
 */
gla_status gla_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *log_lambda,
                                float scale, const int *cu_seqlens, const int *slots, float *state_pool,
                                int n_slots, int nseq, int total_T, int H, int dk, int dv, int chunk,
                                gla_dtype dtype, void *o, void *stream);

/*
 * gla_chunk_fwd_varlen_gated -- gla_chunk_fwd_varlen with a per-token decay
 * (the gated form of gla_chunk_fwd_gated): g [total_T, H] fp32, the
 * natural-log decay of each packed token and head, in place of log_lambda.
 * Everything else, including the device-side checks of cu_seqlens and
 * slots, as gla_chunk_fwd_varlen; the serving steps that follow are
 * gla_decode_step_gated on the same pool.
 */
gla_status gla_chunk_fwd_varlen_gated(const void *q, const void *k, const void *v, const float *g,
                                      float scale, const int *cu_seqlens, const int *slots, float *state_pool,
                                      int n_slots, int nseq, int total_T, int H, int dk, int dv, int chunk,
                                      gla_dtype dtype, void *o, void *stream);

/*
 * gla_chunk_bwd -- gradients of L = sum_t <do_t, o_t> + <dhT, hT> through
 * the chunked forward ("Challenge 3": through every serial state update).
 * lambda is fixed (not learned), so there is no gradient for log_lambda.
 *
 *   q, k, v, log_lambda, h0, scale, B..dtype as for gla_chunk_fwd,
 *   do [B,T,H,dv] (dtype), dhT [B,H,dk,dv] fp32 or NULL (zero),
 *   dq, dk_ [B,T,H,dk], dv_ [B,T,H,dv] (dtype, written),
 *   dh0 [B,H,dk,dv] fp32 or NULL (not wanted),
 *   workspace: at least gla_chunk_bwd_workspace_size() bytes (may be 0).
 * GLA_BF16 runs two tensor-core launches side by side: dk and dv (with dh0)
 * in one launch on `stream`, dq on a helper stream that the call forks from
 * `stream` and joins back with events (created once per host thread and
 * device); GLA_FP32 the validation kernels. CUDA maps streams onto a limited number of
 * hardware queues (8 by default); setting CUDA_DEVICE_MAX_CONNECTIONS to 32
 * before the first CUDA call keeps them from sharing one.
 */
gla_status gla_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *log_lambda, const float *h0, float scale,
                         const void *do_, const float *dhT,
                         int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                         void *dq, void *dk_, void *dv_, float *dh0,
                         void *workspace, size_t workspace_bytes, void *stream);

size_t gla_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                    gla_dtype dtype);

/*
 * gla_chunk_fwd_gated -- the chunked forward with a per-token decay: the
 * gated form of the same mixer, in which the fixed per-head decay becomes
 * a decay per token and head (flash-linear-attention's chunk_simple_gla,
 * whose fused kernel "Challenge 1" names, takes it as its gate input g;
 * with g constant over tokens it is gla_chunk_fwd):
 *     S_t = exp(g_t) S_{t-1} + k_t v_t^T,   o_t = scale * S_t^T q_t
 *   g [B,T,H] fp32: natural-log decay of each token and head, <= 0. -inf
 *   (or any value <= -80, whose exp is below fp32's normal range) clears
 *   the state. Positive values are outside the contract: the chunk weights
 *   rely on decays <= 1.
 *   Everything else as gla_chunk_fwd (q, k, v, h0, o, hT, chunk, dtype,
 *   workspace): with at least gla_chunk_fwd_gated_workspace_size() bytes a
 *   long sequence is split into segments that run in parallel, each
 *   segment's decay the exp of its summed g. GLA_BF16 runs the tensor-core
 *   kernel; GLA_FP32 the validation kernel (one chain per (b, h)).
 */
gla_status gla_chunk_fwd_gated(const void *q, const void *k, const void *v,
                               const float *g, const float *h0, float scale,
                               int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                               void *o, float *hT,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace that let gla_chunk_fwd_gated split long sequences into
 * segments (the segment states and decays; 0 when no split pays). */
size_t gla_chunk_fwd_gated_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                          gla_dtype dtype);

/*
 * gla_decode_step_gated -- one recurrent step with a per-token decay:
 *     S <- exp(g[n,h]) S + k v^T (in place),   o = scale * S^T q
 *   g [N,H] fp32, the log-decay of this step's token per sequence and head
 *   (<= 0; -inf clears the state). Otherwise as gla_decode_step.
 */
gla_status gla_decode_step_gated(const void *q, const void *k, const void *v, const float *g,
                                 float *S_inout, float scale, int N, int H, int dk, int dv,
                                 gla_dtype dtype, void *o, void *stream);

/*
 * gla_chunk_bwd_gated -- gradients of L = sum_t <do_t, o_t> + <dhT, hT>
 * through the gated form of gla_chunk_fwd_gated, the gates' own included:
 *     G_t = dL/dS_t (through every later state update),
 *     dq_t = scale S_t do_t,   dk_t = G_t v_t,   dv_t = G_t^T k_t,
 *     dh0 = exp(g_0) G_0,      dg_t = exp(g_t) <G_t, S_{t-1}>   (S_{-1} = h0)
 * ("Challenge 3": the backward passes through every serial state update of
 * the chunked form of "Challenge 1"; the gate enters each update as its decay).
 *   q, k, v, g, h0, scale, do, dhT, dq, dk_, dv_, dh0 as gla_chunk_bwd, with
 *   g [B,T,H] fp32 (as gla_chunk_fwd_gated) in place of log_lambda;
 *   dg [B,T,H] fp32 (written; 0 for a clearing gate). With g_t = ln lambda_h
 *   for every token, the sum of dg over (b, t) is the gradient of a learned
 *   per-head log lambda_h.
 *   workspace: at least gla_chunk_bwd_gated_workspace_size() bytes (required
 *   when T > 0). It receives the state entering every chunk and the state
 *   gradient leaving it, from which dg is formed chunk by chunk.
 * GLA_BF16 runs four tensor-core launches (dq, dk, dv side by side, dq and
 * dk on helper streams forked from `stream` and joined back as in
 * gla_chunk_bwd, then dg after a 4-byte memset of its work counter in the
 * workspace); GLA_FP32 the validation kernels.
 */
gla_status gla_chunk_bwd_gated(const void *q, const void *k, const void *v, const float *g,
                               const float *h0, float scale, const void *do_, const float *dhT,
                               int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                               void *dq, void *dk_, void *dv_, float *dh0, float *dg,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace gla_chunk_bwd_gated needs: two states per (b, h, chunk)
 * (bf16: 2 x B x H x ceil(T / chunk) x 36,864 bytes and a 16-byte work
 * counter; fp32: 2 x B x H x ceil(T / chunk) x dk x dv x 4 bytes). */
size_t gla_chunk_bwd_gated_workspace_size(int B, int T, int H, int dk, int dv, int chunk,
                                          gla_dtype dtype);

/*
 * gla_decode_step -- one recurrent step per (sequence n, head h), the
 * serving path ("Inference optimization on Trainium2": the state lives in a
 * fixed page per sequence):
 *     S <- lambda * S + k v^T   (in place, fp32)
 *     o  = scale * S^T q        (after the update)
 *
 *   q, k [N,H,dk], v [N,H,dv] (dtype), log_lambda [H], S_inout [N,H,dk,dv]
 *   fp32 (read and written), o [N,H,dv] (dtype, written).
 */
gla_status gla_decode_step(const void *q, const void *k, const void *v,
                           const float *log_lambda, float *S_inout, float scale,
                           int N, int H, int dk, int dv, gla_dtype dtype,
                           void *o, void *stream);

/*
 * The mixer epilogue, per (token or sequence, head): the reading of the
 * "GLA mixer" paragraph, whose equations did not survive extraction:
 *     u = o + sigmoid(q . (aug_h * k)) v     self-augmentation (aug_balance;
 *                                            aug_h = 0 is a half-strength skip)
 *     y = norm_w_h * u / sqrt(mean(u^2) + eps)   Head RMSNorm over the dv channels
 *                                            (each head normalised on its own;
 *                                            the pages group heads into decay
 *                                            tiers without saying how)
 *     z = y * g * sigmoid(g)                 the SiLU(g) gate of the fused projection
 * aug [H, dk] fp32 or NULL (zero), norm_w [H, dv] fp32 or NULL (one), eps >= 0.
 * W_out, the projection that follows, is a dense GEMM outside this library.
 *
 * gla_mixer_epilogue: over rows [NT, H, *] (NT = B*T tokens, or N sequences):
 *   o, v, g, z [NT, H, dv], q, k [NT, H, dk], all of `dtype` (GLA_BF16 or
 *   GLA_FP32); dk <= 1024, dv <= 256. z may not alias the inputs.
 * gla_decode_step_mixer: gla_decode_step followed by the epilogue in the same
 *   kernel (o never reaches memory); g [N, H, dv] of `dtype`, z [N, H, dv].
 */
/* gla_chunk_fwd_mixer: gla_chunk_fwd followed by the epilogue, z in place of
 *   o: g [B,T,H,dv] bf16, z [B,T,H,dv] bf16, hT and the workspace as for
 *   gla_chunk_fwd. GLA_BF16 only (dk = 96, dv = 192). The forward's launches
 *   and one more, with no scratch memory: at chunk 128 on the one-CTA-per-
 *   (b, h) kernel the forward's output stage adds the self-augmentation and
 *   writes u into z, and a second pass normalises each row of z in place and
 *   multiplies it by norm_w and SiLU(g); otherwise the forward writes o into
 *   z and the epilogue rewrites each row of z in place.
 *   z may not alias q, k, v or g.
 */
gla_status gla_chunk_fwd_mixer(const void *q, const void *k, const void *v, const void *g, const float *log_lambda,
                               const float *h0, float scale, const float *aug, const float *norm_w, float eps, int B,
                               int T, int H, int dk, int dv, int chunk, gla_dtype dtype, void *z, float *hT,
                               void *workspace, size_t workspace_bytes, void *stream);
gla_status gla_mixer_epilogue(const void *o, const void *q, const void *k, const void *v, const void *g,
                              const float *aug, const float *norm_w, float eps, int NT, int H, int dk, int dv,
                              gla_dtype dtype, void *z, void *stream);
gla_status gla_decode_step_mixer(const void *q, const void *k, const void *v, const float *log_lambda,
                                 float *S_inout, float scale, const void *g, const float *aug,
                                 const float *norm_w, float eps, int N, int H, int dk, int dv, gla_dtype dtype,
                                 void *z, void *stream);

/*
 * The causal depthwise Conv1d of width 4 with SiLU that filters the token
 * stream in front of the mixer ("i14 and the Laplace 3B architecture",
 * paragraph "Normalisation and convolution"; no equation survives, the
 * reading), per channel c:
 *     y_t[c] = SiLU( sum_{i=0..3} w[c][i] x_{t-3+i}[c] + b[c] )
 * Inputs before a call's first token come from the sequence's conv window:
 * its last four inputs so far, fp32, [4, D] rows oldest first (zeros for a
 * new sequence; the oldest row is carried, never multiplied). Four fp32 rows
 * of D = 3072 per layer are the part of the 29.5 MB per-sequence state that
 * is not the mixer's.
 *   w [D, 4] fp32 (tap 3 multiplies the current token), b [D] fp32 or NULL
 *   (zero); x, y rows of D channels of `dtype` (GLA_BF16 or GLA_FP32); D a
 *   multiple of 8 (bf16) or 4 (fp32). y may not overlap x or a window.
 *
 * gla_conv1d_fwd: x, y [B, T, D]; win_in [B, 4, D] fp32 or NULL (zeros);
 *   win_out [B, 4, D] fp32 or NULL (not wanted), the windows after the call.
 *   win_in == win_out updates the windows in place (any other overlap is
 *   undefined). T = 0 copies win_in to win_out.
 * gla_conv1d_varlen: sequences packed as for gla_chunk_fwd_varlen (x, y
 *   [total_T, D]; cu_seqlens [nseq + 1] and slots [nseq] or NULL in device
 *   memory, with the same error behaviour: a bad entry skips the sequence and
 *   the next gla_check() reports GLA_ERR_INVALID_ARG); win_pool
 *   [n_slots, 4, D] fp32 holds each slot's window before the call and gets
 *   the window after it (a sequence of length 0 leaves its slot untouched).
 *   Tokens past cu_seqlens[nseq] get no output.
 * gla_conv1d_step: one new token per sequence (the serving step): x, y
 *   [N, D]; win [N, 4, D] fp32, read and updated in place (shifted by one
 *   row, the new input last).
 * Each call launches one kernel for y and, when a window is written by a
 * call over several tokens, one small kernel after it for the windows.
 */
gla_status gla_conv1d_fwd(const void *x, const float *w, const float *b, const float *win_in, int B, int T, int D,
                          gla_dtype dtype, void *y, float *win_out, void *stream);
gla_status gla_conv1d_varlen(const void *x, const float *w, const float *b, const int *cu_seqlens,
                             const int *slots, float *win_pool, int n_slots, int nseq, int total_T, int D,
                             gla_dtype dtype, void *y, void *stream);
gla_status gla_conv1d_step(const void *x, const float *w, const float *b, float *win, int N, int D,
                           gla_dtype dtype, void *y, void *stream);

/*
 * gla_selftest_wait_timeout -- diagnostic of the device-side failure
 * detection, with no fault and no hang: one kernel waits on two mbarriers
 * that nothing completes. The first wait gives up after limit_us (1 to
 * 1,000,000) and flags a timeout; the second, with the kernels' own 2 s
 * limit, must leave as soon as it sees that flag. result: 3 ints in device
 * memory (16-byte aligned): [0], [1] = 1 if the wait completed, 0 if it gave
 * up; [2] = microseconds the second wait lasted. The next gla_check()
 * reports GLA_ERR_TIMEOUT and clears the status word.
 */
gla_status gla_selftest_wait_timeout(unsigned int limit_us, int *result, void *stream);

/* Synchronise `stream` and report: GLA_ERR_CUDA if the stream or an earlier
 * launch failed, GLA_ERR_TIMEOUT if a device-side wait gave up since the last
 * gla_check (the status word is cleared on read), else GLA_OK. */
gla_status gla_check(void *stream);

/* Static, human-readable name of a status code. */
const char *gla_status_string(gla_status status);

/* Detail of the last error raised on this host thread (empty if none). */
const char *gla_last_error(void);

/* Number of kernels the last gla_chunk_fwd / gla_chunk_bwd / gla_decode_step
 * call on this host thread launched (0 after an argument error). */
int gla_last_launch_count(void);

/* Library version, e.g. "libgla 0.1.0 sm_103a". */
const char *gla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBGLA_GLA_H */
