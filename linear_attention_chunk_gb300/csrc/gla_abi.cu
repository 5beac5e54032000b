// gla_abi.cu -- the C ABI of libgla (declared in include/gla.h): host-side
// argument validation, the device status word, and dispatch to the kernels.
//
// The operations are those of "Beyond the KV cache: Training and serving
// i14's Laplace 3B linear attention model on AWS Trainium2 with native
// PyTorch": the Simple GLA recurrence of the "GLA mixer" paragraph, its
// chunked form ("Challenge 1"), its backward through the serial state chain
// ("Challenge 3") and the serving step ("Inference optimization on
// Trainium2"). Every argument error is caught here, before any launch.
#include <cuda_runtime.h>

#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "gla.h"
#include "common.cuh"
#include "kernels.h"

namespace gla {

// One status word per device that loads the library; kernels set bits in it
// (kDevTimeout, ...) and gla_check() reads and clears it.
static __device__ unsigned int g_status_word;

namespace {

thread_local char t_err[512] = {0};
thread_local int t_launches = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int *g_status_ptr[kMaxDevices] = {nullptr};

gla_status fail(gla_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return st;
}

gla_status cuda_fail(cudaError_t e, const char *where) {
    return fail(GLA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of this device's status word (looked up once per device).
gla_status status_word(unsigned int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GLA_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        g_status_ptr[dev] = static_cast<unsigned int *>(ptr);
    }
    *out = g_status_ptr[dev];
    return GLA_OK;
}

// Common shape checks of the chunk entry points.
gla_status check_chunk_shape(int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype) {
    if (dtype != GLA_BF16 && dtype != GLA_FP32) return fail(GLA_ERR_INVALID_ARG, "dtype %d is not GLA_BF16/GLA_FP32", (int)dtype);
    if (B < 0 || T < 0 || H < 0) return fail(GLA_ERR_INVALID_ARG, "negative size B=%d T=%d H=%d", B, T, H);
    if (dk <= 0 || dv <= 0) return fail(GLA_ERR_INVALID_ARG, "dk=%d dv=%d must be positive", dk, dv);
    if (chunk != 64 && chunk != 128) return fail(GLA_ERR_UNSUPPORTED, "chunk %d is not 64 or 128", chunk);
    if (dtype == GLA_BF16 && (dk != 96 || dv != 192))
        return fail(GLA_ERR_UNSUPPORTED, "GLA_BF16 needs dk=96, dv=192 (got %d, %d)", dk, dv);
    if (dtype == GLA_FP32 && (dk > 128 || dv > 256))
        return fail(GLA_ERR_UNSUPPORTED, "GLA_FP32 needs dk <= 128, dv <= 256 (got %d, %d)", dk, dv);
    const long double elems = (long double)B * T * H * (dk > dv ? dk : dv);
    if (elems > (long double)(1ull << 40)) return fail(GLA_ERR_INVALID_ARG, "tensor too large (%Lg elements)", elems);
    if ((long double)B * H > 2147483647.0L) return fail(GLA_ERR_INVALID_ARG, "B*H too large");
    return GLA_OK;
}

#define REQUIRE_PTR(p, name)                                                              \
    do {                                                                                  \
        if (!(p)) return fail(GLA_ERR_INVALID_ARG, "%s is NULL", name);                   \
        if (!aligned16(p)) return fail(GLA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

#define OPTIONAL_PTR(p, name)                                                             \
    do {                                                                                  \
        if ((p) && !aligned16(p)) return fail(GLA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
    } while (0)

// Shape checks of the Conv1d entry points (B sequences of T tokens of D channels).
gla_status check_conv_shape(int B, int T, int D, gla_dtype dtype) {
    if (dtype != GLA_BF16 && dtype != GLA_FP32) return fail(GLA_ERR_INVALID_ARG, "dtype %d is not GLA_BF16/GLA_FP32", (int)dtype);
    if (B < 0 || T < 0) return fail(GLA_ERR_INVALID_ARG, "negative size B=%d T=%d", B, T);
    const int vec = dtype == GLA_BF16 ? 8 : 4;
    if (D <= 0 || D % vec != 0) return fail(GLA_ERR_UNSUPPORTED, "D=%d must be a positive multiple of %d", D, vec);
    if ((long double)B * T * D > (long double)(1ull << 40)) return fail(GLA_ERR_INVALID_ARG, "tensor too large");
    return GLA_OK;
}

// The decode step with or without the mixer epilogue (g == NULL: plain o).
gla_status decode_common(const void *q, const void *k, const void *v, const float *log_lambda, float *S_inout,
                         float scale, const void *g, const float *aug, const float *norm_w, float eps, int N,
                         int H, int dk, int dv, gla_dtype dtype, void *o, void *stream, const char *name,
                         const float *log_decay = nullptr) {
    t_err[0] = 0;
    t_launches = 0;
    if (dtype != GLA_BF16 && dtype != GLA_FP32) return fail(GLA_ERR_INVALID_ARG, "dtype %d invalid", (int)dtype);
    if (N < 0 || H < 0) return fail(GLA_ERR_INVALID_ARG, "negative size N=%d H=%d", N, H);
    if (dk <= 0 || dv <= 0) return fail(GLA_ERR_INVALID_ARG, "dk=%d dv=%d must be positive", dk, dv);
    if (dtype == GLA_BF16 && (dk != 96 || dv != 192))
        return fail(GLA_ERR_UNSUPPORTED, "GLA_BF16 needs dk=96, dv=192 (got %d, %d)", dk, dv);
    if (dtype == GLA_FP32 && (dk > 128 || dv > 256))
        return fail(GLA_ERR_UNSUPPORTED, "GLA_FP32 needs dk <= 128, dv <= 256 (got %d, %d)", dk, dv);
    if ((long double)N * H > 2147483647.0L) return fail(GLA_ERR_INVALID_ARG, "N*H too large");
    if (!(eps >= 0.f)) return fail(GLA_ERR_INVALID_ARG, "eps must be >= 0");
    OPTIONAL_PTR(aug, "aug");
    OPTIONAL_PTR(norm_w, "norm_w");
    if (N == 0 || H == 0) return GLA_OK;
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    if (log_decay) {
        REQUIRE_PTR(log_decay, "g");
    } else {
        REQUIRE_PTR(log_lambda, "log_lambda");
    }
    REQUIRE_PTR(S_inout, "S_inout");
    REQUIRE_PTR(o, name);
    unsigned int *status = nullptr;
    gla_status st = status_word(&status);
    if (st != GLA_OK) return st;
    DecodeParams p{q, k, v, log_lambda, S_inout, scale, N, H, dk, dv, o, status, g, aug, norm_w, eps, log_decay};
    int launches = 0;
    cudaError_t e = launch_decode(p, dtype == GLA_BF16, static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "decode launch");
}


}  // namespace

void set_error_detail(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
}

void reset_call_state() {
    t_err[0] = 0;
    t_launches = 0;
}

}  // namespace gla

using namespace gla;

extern "C" {

gla_status gla_chunk_fwd(const void *q, const void *k, const void *v, const float *log_lambda,
                         const float *h0, float scale, int B, int T, int H, int dk, int dv, int chunk,
                         gla_dtype dtype, void *o, float *hT, void *workspace, size_t workspace_bytes,
                         void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_chunk_shape(B, T, H, dk, dv, chunk, dtype);
    if (st != GLA_OK) return st;
    OPTIONAL_PTR(h0, "h0");
    OPTIONAL_PTR(hT, "hT");
    OPTIONAL_PTR(workspace, "workspace");
    if (B == 0 || H == 0) return GLA_OK;
    REQUIRE_PTR(log_lambda, "log_lambda");
    if (T > 0) {
        REQUIRE_PTR(q, "q");
        REQUIRE_PTR(k, "k");
        REQUIRE_PTR(v, "v");
        REQUIRE_PTR(o, "o");
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    cudaError_t e;
    if (T == 0) {
        e = launch_copy_state(h0, hT, (size_t)B * H * dk * dv, s, &launches);
        t_launches = launches;
        return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_fwd(T=0)");
    }
    FwdParams p{q, k, v, log_lambda, h0, scale, B, T, H, dk, dv, chunk, o, hT,
                workspace, workspace ? workspace_bytes : 0, status};
    if (dtype == GLA_BF16)
        e = launch_fwd_tc(p, s, &launches);
    else
        e = launch_fwd_simt(p, false, s, &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_fwd launch");
}

gla_status gla_chunk_fwd_gated(const void *q, const void *k, const void *v, const float *g, const float *h0,
                               float scale, int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                               void *o, float *hT, void *workspace, size_t workspace_bytes, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_chunk_shape(B, T, H, dk, dv, chunk, dtype);
    if (st != GLA_OK) return st;
    OPTIONAL_PTR(h0, "h0");
    OPTIONAL_PTR(hT, "hT");
    OPTIONAL_PTR(workspace, "workspace");
    if (B == 0 || H == 0) return GLA_OK;
    if (T > 0) {
        REQUIRE_PTR(q, "q");
        REQUIRE_PTR(k, "k");
        REQUIRE_PTR(v, "v");
        REQUIRE_PTR(g, "g");
        REQUIRE_PTR(o, "o");
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    cudaError_t e;
    if (T == 0) {
        e = launch_copy_state(h0, hT, (size_t)B * H * dk * dv, s, &launches);
        t_launches = launches;
        return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_fwd_gated(T=0)");
    }
    FwdParams p{q, k, v, nullptr, h0, scale, B, T, H, dk, dv, chunk, o, hT,
                workspace, workspace ? workspace_bytes : 0, status, g};
    if (dtype == GLA_BF16)
        e = launch_fwd_tc(p, s, &launches);
    else
        e = launch_fwd_simt(p, false, s, &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_fwd_gated launch");
}

size_t gla_chunk_fwd_gated_workspace_size(int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype) {
    if (check_chunk_shape(B, T, H, dk, dv, chunk, dtype) != GLA_OK) return 0;
    if (dtype != GLA_BF16) return 0;
    return fwd_tc_workspace_size(B, T, H, chunk, true);
}

gla_status gla_decode_step_gated(const void *q, const void *k, const void *v, const float *g, float *S_inout,
                                 float scale, int N, int H, int dk, int dv, gla_dtype dtype, void *o, void *stream) {
    if (N > 0 && H > 0 && !g) return fail(GLA_ERR_INVALID_ARG, "g is NULL");
    return decode_common(q, k, v, nullptr, S_inout, scale, nullptr, nullptr, nullptr, 0.f, N, H, dk, dv, dtype, o,
                         stream, "o", g);
}

gla_status gla_chunk_fwd_mixer(const void *q, const void *k, const void *v, const void *g, const float *log_lambda,
                               const float *h0, float scale, const float *aug, const float *norm_w, float eps, int B,
                               int T, int H, int dk, int dv, int chunk, gla_dtype dtype, void *z, float *hT,
                               void *workspace, size_t workspace_bytes, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_chunk_shape(B, T, H, dk, dv, chunk, dtype);
    if (st != GLA_OK) return st;
    if (dtype != GLA_BF16) return fail(GLA_ERR_UNSUPPORTED, "gla_chunk_fwd_mixer supports GLA_BF16 only");
    if (!(eps >= 0.f)) return fail(GLA_ERR_INVALID_ARG, "eps must be >= 0");
    OPTIONAL_PTR(h0, "h0");
    OPTIONAL_PTR(hT, "hT");
    OPTIONAL_PTR(aug, "aug");
    OPTIONAL_PTR(norm_w, "norm_w");
    OPTIONAL_PTR(workspace, "workspace");
    if (B == 0 || H == 0) return GLA_OK;
    if ((long double)B * T > 2147483647.0L || (long double)B * T * H > 2147483647.0L * 8.0L)
        return fail(GLA_ERR_INVALID_ARG, "B*T or B*T*H too large");
    REQUIRE_PTR(log_lambda, "log_lambda");
    if (T > 0) {
        REQUIRE_PTR(q, "q");
        REQUIRE_PTR(k, "k");
        REQUIRE_PTR(v, "v");
        REQUIRE_PTR(g, "g");
        REQUIRE_PTR(z, "z");
        if (z == q || z == k || z == v || z == g) return fail(GLA_ERR_INVALID_ARG, "z may not alias an input");
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    cudaError_t e;
    if (T == 0) {
        e = launch_copy_state(h0, hT, (size_t)B * H * dk * dv, s, &launches);
        t_launches = launches;
        return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_fwd_mixer(T=0)");
    }
    // The forward writes into z's buffer either the normalised rows, which a
    // second pass multiplies by the norm weight and the SiLU gate (one CTA per
    // chain at chunk 128), or o, which the epilogue then rewrites row by row
    // in place (a warp reads all of a row's inputs before storing it).
    FwdParams p{q, k, v, log_lambda, h0, scale, B, T, H, dk, dv, chunk, z, hT,
                workspace, workspace ? workspace_bytes : 0, status};
    const EpilogueParams ep{z, q, k, v, g, aug, norm_w, eps, B * T, H, dk, dv, z};
    e = launch_fwd_tc(p, s, &launches, &ep);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_fwd_mixer launch");
}

size_t gla_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype) {
    if (check_chunk_shape(B, T, H, dk, dv, chunk, dtype) != GLA_OK) return 0;
    if (dtype != GLA_BF16) return 0;
    return fwd_tc_workspace_size(B, T, H, chunk);
}

gla_status gla_chunk_bwd(const void *q, const void *k, const void *v, const float *log_lambda,
                         const float *h0, float scale, const void *do_, const float *dhT, int B, int T,
                         int H, int dk, int dv, int chunk, gla_dtype dtype, void *dq, void *dk_, void *dv_,
                         float *dh0, void *workspace, size_t workspace_bytes, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_chunk_shape(B, T, H, dk, dv, chunk, dtype);
    if (st != GLA_OK) return st;
    OPTIONAL_PTR(h0, "h0");
    OPTIONAL_PTR(dhT, "dhT");
    OPTIONAL_PTR(dh0, "dh0");
    OPTIONAL_PTR(workspace, "workspace");
    if (B == 0 || H == 0) return GLA_OK;
    REQUIRE_PTR(log_lambda, "log_lambda");
    const size_t need = gla_chunk_bwd_workspace_size(B, T, H, dk, dv, chunk, dtype);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(GLA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (T > 0) {
        REQUIRE_PTR(q, "q");
        REQUIRE_PTR(k, "k");
        REQUIRE_PTR(v, "v");
        REQUIRE_PTR(do_, "do");
        REQUIRE_PTR(dq, "dq");
        REQUIRE_PTR(dk_, "dk");
        REQUIRE_PTR(dv_, "dv");
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    cudaError_t e;
    if (T == 0) {
        // No tokens: dh0 = dhT (the state passes through untouched).
        e = launch_copy_state(dhT, dh0, (size_t)B * H * dk * dv, s, &launches);
        t_launches = launches;
        return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_bwd(T=0)");
    }
    BwdParams p{q, k, v, log_lambda, h0, scale, do_, dhT, B, T, H, dk, dv, chunk, dq, dk_, dv_, dh0,
                workspace, workspace ? workspace_bytes : 0, status};
    if (dtype == GLA_BF16)
        e = launch_bwd_tc(p, s, &launches);
    else
        e = launch_bwd_simt(p, false, s, &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_bwd launch");
}

size_t gla_chunk_bwd_gated_workspace_size(int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype) {
    if (check_chunk_shape(B, T, H, dk, dv, chunk, dtype) != GLA_OK) return 0;
    if (dtype == GLA_BF16) return bwd_gated_tc_workspace_size(B, T, H, chunk);
    const size_t nck = ((size_t)T + chunk - 1) / chunk;
    return 2 * (size_t)B * H * nck * dk * dv * sizeof(float);
}

gla_status gla_chunk_bwd_gated(const void *q, const void *k, const void *v, const float *g, const float *h0,
                               float scale, const void *do_, const float *dhT, int B, int T, int H, int dk, int dv,
                               int chunk, gla_dtype dtype, void *dq, void *dk_, void *dv_, float *dh0, float *dg,
                               void *workspace, size_t workspace_bytes, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_chunk_shape(B, T, H, dk, dv, chunk, dtype);
    if (st != GLA_OK) return st;
    OPTIONAL_PTR(h0, "h0");
    OPTIONAL_PTR(dhT, "dhT");
    OPTIONAL_PTR(dh0, "dh0");
    OPTIONAL_PTR(workspace, "workspace");
    if (B == 0 || H == 0) return GLA_OK;
    if ((long double)B * H * ((T + (long double)chunk - 1) / chunk) > 2147483647.0L)
        return fail(GLA_ERR_INVALID_ARG, "B*H*chunks too large");
    if (dtype == GLA_FP32 && (T + chunk - 1) / chunk > 65535)
        return fail(GLA_ERR_UNSUPPORTED, "GLA_FP32 gated backward needs at most 65535 chunks");
    if (T > 0) {
        REQUIRE_PTR(q, "q");
        REQUIRE_PTR(k, "k");
        REQUIRE_PTR(v, "v");
        REQUIRE_PTR(g, "g");
        REQUIRE_PTR(do_, "do");
        REQUIRE_PTR(dq, "dq");
        REQUIRE_PTR(dk_, "dk");
        REQUIRE_PTR(dv_, "dv");
        REQUIRE_PTR(dg, "dg");
        const size_t need = gla_chunk_bwd_gated_workspace_size(B, T, H, dk, dv, chunk, dtype);
        if (workspace == nullptr || workspace_bytes < need)
            return fail(GLA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                        workspace ? workspace_bytes : (size_t)0);
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int launches = 0;
    cudaError_t e;
    if (T == 0) {
        // No tokens: dh0 = dhT (the state passes through untouched); no gates.
        e = launch_copy_state(dhT, dh0, (size_t)B * H * dk * dv, s, &launches);
        t_launches = launches;
        return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_bwd_gated(T=0)");
    }
    BwdParams p{q, k, v, nullptr, h0, scale, do_, dhT, B, T, H, dk, dv, chunk, dq, dk_, dv_, dh0,
                workspace, workspace_bytes, status, g, dg};
    if (dtype == GLA_BF16)
        e = launch_bwd_gated_tc(p, s, &launches);
    else
        e = launch_bwd_simt(p, false, s, &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_chunk_bwd_gated launch");
}

static gla_status varlen_common(const void *q, const void *k, const void *v, const float *log_lambda, const float *g,
                                float scale,
                                const int *cu_seqlens, const int *slots, float *state_pool, int n_slots, int nseq,
                                int total_T, int H, int dk, int dv, int chunk, gla_dtype dtype, void *o,
                                void *stream, const char *name) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_chunk_shape(1, total_T, H, dk, dv, chunk, dtype);
    if (st != GLA_OK) return st;
    if (dtype != GLA_BF16) return fail(GLA_ERR_UNSUPPORTED, "%s supports GLA_BF16 only", name);
    if (nseq < 0 || n_slots < 0) return fail(GLA_ERR_INVALID_ARG, "negative nseq=%d or n_slots=%d", nseq, n_slots);
    if ((long double)nseq * H * 2 > 2147483647.0L) return fail(GLA_ERR_INVALID_ARG, "nseq*H too large");
    OPTIONAL_PTR(slots, "slots");
    if (nseq == 0 || H == 0) return GLA_OK;
    if (g) {
        REQUIRE_PTR(g, "g");
    } else {
        REQUIRE_PTR(log_lambda, "log_lambda");
    }
    REQUIRE_PTR(cu_seqlens, "cu_seqlens");
    REQUIRE_PTR(state_pool, "state_pool");
    if (!slots && n_slots < nseq)
        return fail(GLA_ERR_INVALID_ARG, "without slots the pool needs nseq=%d slots, has %d", nseq, n_slots);
    if (total_T > 0) {
        REQUIRE_PTR(q, "q");
        REQUIRE_PTR(k, "k");
        REQUIRE_PTR(v, "v");
        REQUIRE_PTR(o, "o");
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    if (total_T == 0) return GLA_OK;   // every sequence is empty: no state changes
    VarlenParams p{q, k, v, log_lambda, scale, cu_seqlens, slots, state_pool, n_slots, nseq, total_T, H, dk, dv,
                   chunk, o, status, g};
    int launches = 0;
    const cudaError_t e = launch_fwd_varlen_tc(p, static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, name);
}

gla_status gla_chunk_fwd_varlen(const void *q, const void *k, const void *v, const float *log_lambda, float scale,
                                const int *cu_seqlens, const int *slots, float *state_pool, int n_slots, int nseq,
                                int total_T, int H, int dk, int dv, int chunk, gla_dtype dtype, void *o,
                                void *stream) {
    return varlen_common(q, k, v, log_lambda, nullptr, scale, cu_seqlens, slots, state_pool, n_slots, nseq, total_T, H,
                         dk, dv, chunk, dtype, o, stream, "gla_chunk_fwd_varlen");
}

gla_status gla_chunk_fwd_varlen_gated(const void *q, const void *k, const void *v, const float *g, float scale,
                                      const int *cu_seqlens, const int *slots, float *state_pool, int n_slots,
                                      int nseq, int total_T, int H, int dk, int dv, int chunk, gla_dtype dtype,
                                      void *o, void *stream) {
    if (nseq > 0 && H > 0 && total_T > 0 && !g) return fail(GLA_ERR_INVALID_ARG, "g is NULL");
    return varlen_common(q, k, v, nullptr, g, scale, cu_seqlens, slots, state_pool, n_slots, nseq, total_T, H, dk,
                         dv, chunk, dtype, o, stream, "gla_chunk_fwd_varlen_gated");
}

size_t gla_chunk_bwd_workspace_size(int B, int T, int H, int dk, int dv, int chunk, gla_dtype dtype) {
    if (check_chunk_shape(B, T, H, dk, dv, chunk, dtype) != GLA_OK) return 0;
    if (dtype != GLA_BF16) return 0;
    return bwd_tc_workspace_size(B, T, H, chunk);
}

gla_status gla_decode_step(const void *q, const void *k, const void *v, const float *log_lambda,
                           float *S_inout, float scale, int N, int H, int dk, int dv, gla_dtype dtype,
                           void *o, void *stream) {
    return decode_common(q, k, v, log_lambda, S_inout, scale, nullptr, nullptr, nullptr, 0.f, N, H, dk, dv, dtype,
                         o, stream, "o");
}

gla_status gla_decode_step_mixer(const void *q, const void *k, const void *v, const float *log_lambda,
                                 float *S_inout, float scale, const void *g, const float *aug,
                                 const float *norm_w, float eps, int N, int H, int dk, int dv, gla_dtype dtype,
                                 void *z, void *stream) {
    if (N > 0 && H > 0) {
        if (!g) return fail(GLA_ERR_INVALID_ARG, "g is NULL");
        if (!aligned16(g)) return fail(GLA_ERR_INVALID_ARG, "g is not 16-byte aligned");
    }
    return decode_common(q, k, v, log_lambda, S_inout, scale, g, aug, norm_w, eps, N, H, dk, dv, dtype, z, stream,
                         "z");
}

gla_status gla_mixer_epilogue(const void *o, const void *q, const void *k, const void *v, const void *g,
                              const float *aug, const float *norm_w, float eps, int NT, int H, int dk, int dv,
                              gla_dtype dtype, void *z, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    if (dtype != GLA_BF16 && dtype != GLA_FP32) return fail(GLA_ERR_INVALID_ARG, "dtype %d invalid", (int)dtype);
    if (NT < 0 || H < 0) return fail(GLA_ERR_INVALID_ARG, "negative size NT=%d H=%d", NT, H);
    if (dk <= 0 || dv <= 0) return fail(GLA_ERR_INVALID_ARG, "dk=%d dv=%d must be positive", dk, dv);
    if (dk > 1024 || dv > 256) return fail(GLA_ERR_UNSUPPORTED, "needs dk <= 1024, dv <= 256 (got %d, %d)", dk, dv);
    if ((long double)NT * H > 2147483647.0L * 8.0L) return fail(GLA_ERR_INVALID_ARG, "NT*H too large");
    if (!(eps >= 0.f)) return fail(GLA_ERR_INVALID_ARG, "eps must be >= 0");
    OPTIONAL_PTR(aug, "aug");
    OPTIONAL_PTR(norm_w, "norm_w");
    if (NT == 0 || H == 0) return GLA_OK;
    REQUIRE_PTR(o, "o");
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(g, "g");
    REQUIRE_PTR(z, "z");
    EpilogueParams p{o, q, k, v, g, aug, norm_w, eps, NT, H, dk, dv, z};
    int launches = 0;
    cudaError_t e = launch_mixer_epilogue(p, dtype == GLA_BF16, static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_mixer_epilogue launch");
}

gla_status gla_conv1d_fwd(const void *x, const float *w, const float *b, const float *win_in, int B, int T, int D,
                          gla_dtype dtype, void *y, float *win_out, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_conv_shape(B, T, D, dtype);
    if (st != GLA_OK) return st;
    OPTIONAL_PTR(b, "b");
    OPTIONAL_PTR(win_in, "win_in");
    OPTIONAL_PTR(win_out, "win_out");
    if (B == 0 || (T == 0 && !win_out)) return GLA_OK;
    REQUIRE_PTR(w, "w");
    if (T > 0) {
        REQUIRE_PTR(x, "x");
        REQUIRE_PTR(y, "y");
        if (x == y) return fail(GLA_ERR_INVALID_ARG, "y may not alias x");
    }
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    ConvParams p{x, w, b, nullptr, nullptr, win_in, win_out, B, B, (long)B * T, T, D, y, status};
    int launches = 0;
    const cudaError_t e = launch_conv_fwd(p, false, dtype == GLA_BF16, static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_conv1d_fwd launch");
}

gla_status gla_conv1d_varlen(const void *x, const float *w, const float *b, const int *cu_seqlens,
                             const int *slots, float *win_pool, int n_slots, int nseq, int total_T, int D,
                             gla_dtype dtype, void *y, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_conv_shape(1, total_T, D, dtype);
    if (st != GLA_OK) return st;
    if (nseq < 0 || n_slots < 0) return fail(GLA_ERR_INVALID_ARG, "negative nseq=%d or n_slots=%d", nseq, n_slots);
    OPTIONAL_PTR(b, "b");
    OPTIONAL_PTR(slots, "slots");
    if (nseq == 0) return GLA_OK;
    if (!slots && n_slots < nseq)
        return fail(GLA_ERR_INVALID_ARG, "without slots the pool needs nseq=%d slots, has %d", nseq, n_slots);
    REQUIRE_PTR(w, "w");
    REQUIRE_PTR(cu_seqlens, "cu_seqlens");
    REQUIRE_PTR(win_pool, "win_pool");
    if (total_T == 0) return GLA_OK;   // every sequence is empty: no window changes
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(y, "y");
    if (x == y) return fail(GLA_ERR_INVALID_ARG, "y may not alias x");
    unsigned int *status = nullptr;
    if ((st = status_word(&status)) != GLA_OK) return st;
    ConvParams p{x, w, b, cu_seqlens, slots, win_pool, win_pool, n_slots, nseq, (long)total_T, 0, D, y, status};
    int launches = 0;
    const cudaError_t e = launch_conv_fwd(p, true, dtype == GLA_BF16, static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_conv1d_varlen launch");
}

gla_status gla_conv1d_step(const void *x, const float *w, const float *b, float *win, int N, int D,
                           gla_dtype dtype, void *y, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    gla_status st = check_conv_shape(N, 1, D, dtype);
    if (st != GLA_OK) return st;
    OPTIONAL_PTR(b, "b");
    if (N == 0) return GLA_OK;
    REQUIRE_PTR(x, "x");
    REQUIRE_PTR(w, "w");
    REQUIRE_PTR(win, "win");
    REQUIRE_PTR(y, "y");
    if (x == y) return fail(GLA_ERR_INVALID_ARG, "y may not alias x");
    ConvParams p{x, w, b, nullptr, nullptr, win, win, N, N, (long)N, 1, D, y, nullptr};
    int launches = 0;
    const cudaError_t e = launch_conv_step(p, dtype == GLA_BF16, static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_conv1d_step launch");
}

gla_status gla_selftest_wait_timeout(unsigned int limit_us, int *result, void *stream) {
    t_err[0] = 0;
    t_launches = 0;
    if (limit_us == 0 || limit_us > 1000000u) return fail(GLA_ERR_INVALID_ARG, "limit_us must be in 1..1000000");
    REQUIRE_PTR(result, "result");
    unsigned int *status = nullptr;
    gla_status st = status_word(&status);
    if (st != GLA_OK) return st;
    int launches = 0;
    const cudaError_t e = launch_selftest_wait(status, (uint64_t)limit_us * 1000u, result,
                                               static_cast<cudaStream_t>(stream), &launches);
    t_launches = launches;
    return e == cudaSuccess ? GLA_OK : cuda_fail(e, "gla_selftest_wait_timeout launch");
}

gla_status gla_check(void *stream) {
    t_err[0] = 0;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "earlier launch");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
        if (word & kDevTimeout) return fail(GLA_ERR_TIMEOUT, "a device-side wait timed out (status 0x%x)", word);
        if (word & kDevBadState)
            return fail(GLA_ERR_INVALID_ARG, "a sequence had a bad cu_seqlens or slots entry and was skipped "
                                             "(status 0x%x)", word);
        return fail(GLA_ERR_CUDA, "device reported an internal error (status 0x%x)", word);
    }
    return GLA_OK;
}

const char *gla_status_string(gla_status status) {
    switch (status) {
    case GLA_OK: return "GLA_OK";
    case GLA_ERR_INVALID_ARG: return "GLA_ERR_INVALID_ARG";
    case GLA_ERR_UNSUPPORTED: return "GLA_ERR_UNSUPPORTED";
    case GLA_ERR_CUDA: return "GLA_ERR_CUDA";
    case GLA_ERR_TIMEOUT: return "GLA_ERR_TIMEOUT";
    case GLA_ERR_WORKSPACE: return "GLA_ERR_WORKSPACE";
    }
    return "GLA_ERR_UNKNOWN";
}

const char *gla_last_error(void) { return t_err; }

int gla_last_launch_count(void) { return t_launches; }

const char *gla_version(void) { return "libgla 0.1.0 sm_103a"; }

}  // extern "C"
