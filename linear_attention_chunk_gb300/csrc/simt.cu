// simt.cu -- plain FFMA (SIMT) kernels of the chunked Simple GLA forward and
// backward, for the fp32 validation mode and for any dk <= 128, dv <= 256.
//
// The chunked form is the one of "Beyond the KV cache: Training and serving
// i14's Laplace 3B linear attention model on AWS Trainium2 with native
// PyTorch", section "Engineering challenges", "Challenge 1" (equations
// "Chunked GLA intra-chunk output" and "Chunked GLA state update", Figure 3).
// For a chunk of Cc valid tokens entering with state S_prev (0-based i, j):
//   o_i   = scale * ( lambda^(i+1) S_prev^T q_i + sum_{j<=i} lambda^(i-j) (q_i.k_j) v_j )
//   S_new = lambda^Cc S_prev + sum_{j<Cc} lambda^(Cc-1-j) k_j v_j^T
// The backward ("Challenge 3": through every serial state update) is split
// into three independent chains per (b, h):
//   chunk order   : dq_i = scale*( lambda^(i+1) S_prev do_i + sum_{j<=i} lambda^(i-j)(do_i.v_j) k_j )
//   reverse order : G (gradient of the state leaving the chunk), starting at dhT:
//                   dk_j = scale*sum_{i>=j} lambda^(i-j)(do_i.v_j) q_i + lambda^(Cc-1-j) G v_j
//                   dv_j = scale*sum_{i>=j} lambda^(i-j)(q_i.k_j) do_i + lambda^(Cc-1-j) G^T k_j
//                   G   <- lambda^Cc G + scale*sum_i lambda^(i+1) q_i do_i^T,  dh0 = final G.
// Each CTA owns one (b, h) and a slice of the state's columns (forward, dv
// slice) or rows (dq and dk chains, dk slice); fp32 throughout.
//
// The forward also takes a per-token log-decay g [B,T,H] in place of the
// per-head one (the gated form: S_t = exp(g_t) S_{t-1} + k_t v_t^T). Every
// lambda power then becomes the decay of a run of tokens, exp of a sum of
// g: lambda^(i-j) -> exp(G_i - G_j), lambda^(i+1) -> exp(G_i), with G the
// running sum of g inside the chunk. A gate at or below kResetLogDecay
// (-inf included) clears the state; G skips it and a count of such gates
// runs beside G, so that a run holding one gets weight 0 and runs on either
// side keep finite sums.
#include "common.cuh"
#include "kernels.h"

namespace gla {
namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 32;   // state columns (or rows) per CTA
// exp(-80) is below fp32's normal range: such a gate clears the state.
constexpr float kResetLogDecay = -80.f;

__device__ __forceinline__ size_t tok_off(int b, int t, int h, int T, int H, int d) {
    return (((size_t)b * T + t) * H + h) * (size_t)d;
}

// pw[n] = lambda^n for n = 0..C
__device__ __forceinline__ void fill_powers(float *pw, int C, float l2) {
    for (int n = threadIdx.x; n <= C; n += blockDim.x) pw[n] = decay_pow(l2, n);
}

template <typename T>
__device__ __forceinline__ float dot_rows(const T *a, const T *b, int d) {
    float acc = 0.f;
    for (int x = 0; x < d; ++x) acc = fmaf(Elem<T>::load(a + x), Elem<T>::load(b + x), acc);
    return acc;
}

// Decays inside a chunk for the backward kernels: the decay of tokens
// j+1..i (-1 <= j <= i), lambda^(i-j) for the fixed per-head decay, or from
// the chunk's scanned gates (log2 running sums Gl, clearing-gate counts Rc)
// for the per-token one.
struct ChunkDecay {
    const float *pw;
    const float *Gl;
    const int *Rc;
    bool gated;
    __device__ __forceinline__ float operator()(int j, int i) const {
        if (!gated) return pw[i - j];
        if (j < 0) return Rc[i] == 0 ? exp2f(Gl[i]) : 0.f;
        return Rc[i] == Rc[j] ? exp2f(Gl[i] - Gl[j]) : 0.f;
    }
};

// Thread 0 scans tokens t0..t0+Cc-1 of (b, h)'s gates into Gl, Rc; the
// caller synchronises.
__device__ __forceinline__ void scan_gates(const float *g, int b, int t0, int Cc, int h, int Tn, int H, float *Gl,
                                           int *Rc) {
    if (threadIdx.x != 0) return;
    float acc = 0.f;
    int r = 0;
    for (int i = 0; i < Cc; ++i) {
        const float gi = g[((size_t)b * Tn + t0 + i) * H + h];
        if (gi > kResetLogDecay)
            acc += (float)((double)gi * 1.4426950408889634073599246810019);
        else
            ++r;
        Gl[i] = acc;
        Rc[i] = r;
    }
}

// ------------------------------------------------------------------ forward
template <typename T>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(FwdParams p) {
    extern __shared__ float sm[];
    const int C = p.chunk, dk = p.dk, dv = p.dv, H = p.H, Tn = p.T;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int c0 = blockIdx.y * kSlice;
    const int nc = min(kSlice, dv - c0);
    float *S = sm;                       // [dk][kSlice]
    float *P = S + dk * kSlice;          // [C][C]
    float *Vs = P + C * C;               // [C][kSlice]
    float *pw = Vs + C * kSlice;         // [C+1]
    float *Gl = pw + C + 1;              // [C] gated: log2 of the decay of tokens 0..i of the chunk
    int *Rc = reinterpret_cast<int *>(Gl + C);   // [C] gated: clearing gates among tokens 0..i
    const bool gated = p.g != nullptr;
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    T *o = static_cast<T *>(p.o);
    if (!gated) fill_powers(pw, C, log2_of_decay(p.log_lambda[h]));
    const size_t sbase = ((size_t)b * H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * nc; idx += blockDim.x) {
        int a = idx / nc, c = idx % nc;
        S[a * kSlice + c] = p.h0 ? p.h0[sbase + (size_t)a * dv + c0 + c] : 0.f;
    }
    __syncthreads();
    // Decay of the chunk's tokens j+1..i (-1 <= j <= i), lambda^(i-j) for the
    // fixed per-head decay.
    auto decay = [&](int j, int i) -> float {
        if (!gated) return pw[i - j];
        if (j < 0) return Rc[i] == 0 ? exp2f(Gl[i]) : 0.f;
        return Rc[i] == Rc[j] ? exp2f(Gl[i] - Gl[j]) : 0.f;
    };
    for (int t0 = 0; t0 < Tn; t0 += C) {
        const int Cc = min(C, Tn - t0);
        if (gated) {
            if (threadIdx.x == 0) {
                float acc = 0.f;
                int r = 0;
                for (int i = 0; i < Cc; ++i) {
                    const float gi = p.g[((size_t)b * Tn + t0 + i) * H + h];
                    if (gi > kResetLogDecay)
                        acc += (float)((double)gi * 1.4426950408889634073599246810019);
                    else
                        ++r;
                    Gl[i] = acc;
                    Rc[i] = r;
                }
            }
            __syncthreads();
        }
        for (int idx = threadIdx.x; idx < Cc * Cc; idx += blockDim.x) {
            int i = idx / Cc, j = idx % Cc;
            float val = 0.f;
            if (j <= i)
                val = dot_rows(q + tok_off(b, t0 + i, h, Tn, H, dk), k + tok_off(b, t0 + j, h, Tn, H, dk), dk) *
                      decay(j, i);
            P[i * C + j] = val;
        }
        for (int idx = threadIdx.x; idx < Cc * nc; idx += blockDim.x) {
            int j = idx / nc, c = idx % nc;
            Vs[j * kSlice + c] = Elem<T>::load(v + tok_off(b, t0 + j, h, Tn, H, dv) + c0 + c);
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < Cc * nc; idx += blockDim.x) {
            int i = idx / nc, c = idx % nc;
            const T *qi = q + tok_off(b, t0 + i, h, Tn, H, dk);
            float inter = 0.f;
            for (int a = 0; a < dk; ++a) inter = fmaf(Elem<T>::load(qi + a), S[a * kSlice + c], inter);
            float intra = 0.f;
            for (int j = 0; j <= i; ++j) intra = fmaf(P[i * C + j], Vs[j * kSlice + c], intra);
            Elem<T>::store(o + tok_off(b, t0 + i, h, Tn, H, dv) + c0 + c, p.scale * fmaf(decay(-1, i), inter, intra));
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < dk * nc; idx += blockDim.x) {
            int a = idx / nc, c = idx % nc;
            float acc = decay(-1, Cc - 1) * S[a * kSlice + c];
            for (int j = 0; j < Cc; ++j)
                acc = fmaf(decay(j, Cc - 1) * Elem<T>::load(k + tok_off(b, t0 + j, h, Tn, H, dk) + a),
                           Vs[j * kSlice + c], acc);
            S[a * kSlice + c] = acc;
        }
        __syncthreads();
    }
    if (p.hT)
        for (int idx = threadIdx.x; idx < dk * nc; idx += blockDim.x) {
            int a = idx / nc, c = idx % nc;
            p.hT[sbase + (size_t)a * dv + c0 + c] = S[a * kSlice + c];
        }
}

// -------------------------------------------------- backward, chunk order: dq
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dq_simt_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int C = p.chunk, dk = p.dk, dv = p.dv, H = p.H, Tn = p.T;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int a0 = blockIdx.y * kSlice;
    const int na = min(kSlice, dk - a0);
    float *S = sm;                 // [kSlice][dv]   rows a0.. of the state
    float *Dm = S + kSlice * dv;   // [C][C]
    float *pw = Dm + C * C;        // [C+1]
    float *Gl = pw + C + 1;        // [C] gated: scanned gates of the chunk
    int *Rc = reinterpret_cast<int *>(Gl + C);
    const bool gated = p.g != nullptr;
    const ChunkDecay dec{pw, Gl, Rc, gated};
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *dO = static_cast<const T *>(p.do_);
    T *dq = static_cast<T *>(p.dq_out);
    if (!gated) fill_powers(pw, C, log2_of_decay(p.log_lambda[h]));
    const size_t sbase = ((size_t)b * H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
        int a = idx / dv, c = idx % dv;
        S[a * dv + c] = p.h0 ? p.h0[sbase + (size_t)(a0 + a) * dv + c] : 0.f;
    }
    __syncthreads();
    const int nck = (Tn + C - 1) / C;
    for (int t0 = 0; t0 < Tn; t0 += C) {
        const int Cc = min(C, Tn - t0);
        if (gated) {
            scan_gates(p.g, b, t0, Cc, h, Tn, H, Gl, Rc);
            // the gate gradient's input: the state entering this chunk
            float *saved = static_cast<float *>(p.workspace) + (((size_t)b * H + h) * nck + t0 / C) * dk * dv;
            for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
                int a = idx / dv, c = idx % dv;
                saved[(size_t)(a0 + a) * dv + c] = S[a * dv + c];
            }
            __syncthreads();
        }
        for (int idx = threadIdx.x; idx < Cc * Cc; idx += blockDim.x) {
            int i = idx / Cc, j = idx % Cc;
            float val = 0.f;
            if (j <= i)
                val = dot_rows(dO + tok_off(b, t0 + i, h, Tn, H, dv), v + tok_off(b, t0 + j, h, Tn, H, dv), dv) *
                      dec(j, i);
            Dm[i * C + j] = val;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < Cc * na; idx += blockDim.x) {
            int i = idx / na, a = idx % na;
            const T *doi = dO + tok_off(b, t0 + i, h, Tn, H, dv);
            float inter = 0.f;
            for (int c = 0; c < dv; ++c) inter = fmaf(S[a * dv + c], Elem<T>::load(doi + c), inter);
            float intra = 0.f;
            for (int j = 0; j <= i; ++j)
                intra = fmaf(Dm[i * C + j], Elem<T>::load(k + tok_off(b, t0 + j, h, Tn, H, dk) + a0 + a), intra);
            Elem<T>::store(dq + tok_off(b, t0 + i, h, Tn, H, dk) + a0 + a, p.scale * fmaf(dec(-1, i), inter, intra));
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
            int a = idx / dv, c = idx % dv;
            float acc = dec(-1, Cc - 1) * S[a * dv + c];
            for (int j = 0; j < Cc; ++j)
                acc = fmaf(dec(j, Cc - 1) * Elem<T>::load(k + tok_off(b, t0 + j, h, Tn, H, dk) + a0 + a),
                           Elem<T>::load(v + tok_off(b, t0 + j, h, Tn, H, dv) + c), acc);
            S[a * dv + c] = acc;
        }
        __syncthreads();
    }
}

// ------------------------------------------ backward, reverse order: dk, dh0
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dk_simt_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int C = p.chunk, dk = p.dk, dv = p.dv, H = p.H, Tn = p.T;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int a0 = blockIdx.y * kSlice;
    const int na = min(kSlice, dk - a0);
    float *G = sm;                 // [kSlice][dv]
    float *Dm = G + kSlice * dv;   // [C][C]
    float *pw = Dm + C * C;
    float *Gl = pw + C + 1;        // [C] gated: scanned gates of the chunk
    int *Rc = reinterpret_cast<int *>(Gl + C);
    const bool gated = p.g != nullptr;
    const ChunkDecay dec{pw, Gl, Rc, gated};
    const T *q = static_cast<const T *>(p.q);
    const T *v = static_cast<const T *>(p.v);
    const T *dO = static_cast<const T *>(p.do_);
    T *dk_out = static_cast<T *>(p.dk_out);
    if (!gated) fill_powers(pw, C, log2_of_decay(p.log_lambda[h]));
    const size_t sbase = ((size_t)b * H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
        int a = idx / dv, c = idx % dv;
        G[a * dv + c] = p.dhT ? p.dhT[sbase + (size_t)(a0 + a) * dv + c] : 0.f;
    }
    __syncthreads();
    const int nck = (Tn + C - 1) / C;
    for (int ci = nck - 1; ci >= 0; --ci) {
        const int t0 = ci * C, Cc = min(C, Tn - t0);
        if (gated) {
            scan_gates(p.g, b, t0, Cc, h, Tn, H, Gl, Rc);
            // the gate gradient's input: the state gradient leaving this chunk
            float *saved = static_cast<float *>(p.workspace) + ((size_t)p.B * H * nck) * dk * dv +
                           (((size_t)b * H + h) * nck + ci) * dk * dv;
            for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
                int a = idx / dv, c = idx % dv;
                saved[(size_t)(a0 + a) * dv + c] = G[a * dv + c];
            }
            __syncthreads();
        }
        for (int idx = threadIdx.x; idx < Cc * Cc; idx += blockDim.x) {
            int i = idx / Cc, j = idx % Cc;
            float val = 0.f;
            if (j <= i)
                val = dot_rows(dO + tok_off(b, t0 + i, h, Tn, H, dv), v + tok_off(b, t0 + j, h, Tn, H, dv), dv) *
                      dec(j, i);
            Dm[i * C + j] = val;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < Cc * na; idx += blockDim.x) {
            int j = idx / na, a = idx % na;
            const T *vj = v + tok_off(b, t0 + j, h, Tn, H, dv);
            float inter = 0.f;
            for (int c = 0; c < dv; ++c) inter = fmaf(G[a * dv + c], Elem<T>::load(vj + c), inter);
            float intra = 0.f;
            for (int i = j; i < Cc; ++i)
                intra = fmaf(Dm[i * C + j], Elem<T>::load(q + tok_off(b, t0 + i, h, Tn, H, dk) + a0 + a), intra);
            Elem<T>::store(dk_out + tok_off(b, t0 + j, h, Tn, H, dk) + a0 + a,
                           fmaf(p.scale, intra, dec(j, Cc - 1) * inter));
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
            int a = idx / dv, c = idx % dv;
            float acc = 0.f;
            for (int i = 0; i < Cc; ++i)
                acc = fmaf(dec(-1, i) * Elem<T>::load(q + tok_off(b, t0 + i, h, Tn, H, dk) + a0 + a),
                           Elem<T>::load(dO + tok_off(b, t0 + i, h, Tn, H, dv) + c), acc);
            G[a * dv + c] = fmaf(dec(-1, Cc - 1), G[a * dv + c], p.scale * acc);
        }
        __syncthreads();
    }
    if (p.dh0)
        for (int idx = threadIdx.x; idx < na * dv; idx += blockDim.x) {
            int a = idx / dv, c = idx % dv;
            p.dh0[sbase + (size_t)(a0 + a) * dv + c] = G[a * dv + c];
        }
}

// ------------------------------------------------ backward, reverse order: dv
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dv_simt_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int C = p.chunk, dk = p.dk, dv = p.dv, H = p.H, Tn = p.T;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int c0 = blockIdx.y * kSlice;
    const int nc = min(kSlice, dv - c0);
    float *G = sm;                 // [dk][kSlice]
    float *Am = G + dk * kSlice;   // [C][C]
    float *pw = Am + C * C;
    float *Gl = pw + C + 1;        // [C] gated: scanned gates of the chunk
    int *Rc = reinterpret_cast<int *>(Gl + C);
    const bool gated = p.g != nullptr;
    const ChunkDecay dec{pw, Gl, Rc, gated};
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *dO = static_cast<const T *>(p.do_);
    T *dv_out = static_cast<T *>(p.dv_out);
    if (!gated) fill_powers(pw, C, log2_of_decay(p.log_lambda[h]));
    const size_t sbase = ((size_t)b * H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * nc; idx += blockDim.x) {
        int a = idx / nc, c = idx % nc;
        G[a * kSlice + c] = p.dhT ? p.dhT[sbase + (size_t)a * dv + c0 + c] : 0.f;
    }
    __syncthreads();
    const int nck = (Tn + C - 1) / C;
    for (int ci = nck - 1; ci >= 0; --ci) {
        const int t0 = ci * C, Cc = min(C, Tn - t0);
        if (gated) {
            scan_gates(p.g, b, t0, Cc, h, Tn, H, Gl, Rc);
            __syncthreads();
        }
        for (int idx = threadIdx.x; idx < Cc * Cc; idx += blockDim.x) {
            int i = idx / Cc, j = idx % Cc;
            float val = 0.f;
            if (j <= i)
                val = dot_rows(q + tok_off(b, t0 + i, h, Tn, H, dk), k + tok_off(b, t0 + j, h, Tn, H, dk), dk) *
                      dec(j, i);
            Am[i * C + j] = val;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < Cc * nc; idx += blockDim.x) {
            int j = idx / nc, c = idx % nc;
            const T *kj = k + tok_off(b, t0 + j, h, Tn, H, dk);
            float inter = 0.f;
            for (int a = 0; a < dk; ++a) inter = fmaf(G[a * kSlice + c], Elem<T>::load(kj + a), inter);
            float intra = 0.f;
            for (int i = j; i < Cc; ++i)
                intra = fmaf(Am[i * C + j], Elem<T>::load(dO + tok_off(b, t0 + i, h, Tn, H, dv) + c0 + c), intra);
            Elem<T>::store(dv_out + tok_off(b, t0 + j, h, Tn, H, dv) + c0 + c,
                           fmaf(p.scale, intra, dec(j, Cc - 1) * inter));
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < dk * nc; idx += blockDim.x) {
            int a = idx / nc, c = idx % nc;
            float acc = 0.f;
            for (int i = 0; i < Cc; ++i)
                acc = fmaf(dec(-1, i) * Elem<T>::load(q + tok_off(b, t0 + i, h, Tn, H, dk) + a),
                           Elem<T>::load(dO + tok_off(b, t0 + i, h, Tn, H, dv) + c0 + c), acc);
            G[a * kSlice + c] = fmaf(dec(-1, Cc - 1), G[a * kSlice + c], p.scale * acc);
        }
        __syncthreads();
    }
}

// ------------------------------------------- backward, the gate gradient dg
// One CTA per (b, h, chunk), from the states the dq and dk kernels saved:
// S_prev entering the chunk and G_out leaving it. With D(x..y) the decay of
// the chunk's tokens x..y (0-based t, i, j inside the chunk),
//   dg_t = sum_{i >= t > j} s D(j+1..i) (q_i.k_j)(do_i.v_j)
//        + sum_{i >= t} s D(0..i) q_i^T S_prev do_i
//        + sum_{j < t} D(j+1..Cc-1) k_j^T G_out v_j + D(0..Cc-1) <G_out, S_prev>,
// which is exp(g_t) <G_t, S_{t-1}> with G_t and S_{t-1} expanded inside the
// chunk; every sum is taken as written.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_dg_simt_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int C = p.chunk, dk = p.dk, dv = p.dv, H = p.H, Tn = p.T;
    const int b = blockIdx.x / H, h = blockIdx.x % H, ci = blockIdx.y;
    const int t0 = ci * C, Cc = min(C, Tn - t0), nck = (Tn + C - 1) / C;
    float *M = sm;                                  // [C][C]: s D(j+1..i)(q_i.k_j)(do_i.v_j), j < i
    float *Gl = M + C * C;                          // [C]
    int *Rc = reinterpret_cast<int *>(Gl + C);      // [C]
    float *r = reinterpret_cast<float *>(Rc + C);   // [C]
    float *e = r + C;                               // [C]
    float *red = e + C;                             // [kThreads]
    const ChunkDecay dec{nullptr, Gl, Rc, true};
    const T *q = static_cast<const T *>(p.q);
    const T *k = static_cast<const T *>(p.k);
    const T *v = static_cast<const T *>(p.v);
    const T *dO = static_cast<const T *>(p.do_);
    const size_t nstate = (size_t)dk * dv;
    const float *S = static_cast<const float *>(p.workspace) + (((size_t)b * H + h) * nck + ci) * nstate;
    const float *G = S + (size_t)p.B * H * nck * nstate;
    scan_gates(p.g, b, t0, Cc, h, Tn, H, Gl, Rc);
    __syncthreads();
    for (int i = threadIdx.x; i < Cc; i += blockDim.x) {
        const T *qi = q + tok_off(b, t0 + i, h, Tn, H, dk), *ki = k + tok_off(b, t0 + i, h, Tn, H, dk);
        const T *vi = v + tok_off(b, t0 + i, h, Tn, H, dv), *doi = dO + tok_off(b, t0 + i, h, Tn, H, dv);
        float rq = 0.f, ek = 0.f;
        for (int a = 0; a < dk; ++a) {
            float sd = 0.f, gv = 0.f;
            for (int c = 0; c < dv; ++c) {
                sd = fmaf(S[(size_t)a * dv + c], Elem<T>::load(doi + c), sd);
                gv = fmaf(G[(size_t)a * dv + c], Elem<T>::load(vi + c), gv);
            }
            rq = fmaf(Elem<T>::load(qi + a), sd, rq);
            ek = fmaf(Elem<T>::load(ki + a), gv, ek);
        }
        r[i] = p.scale * dec(-1, i) * rq;
        e[i] = dec(i, Cc - 1) * ek;
        for (int j = 0; j < Cc; ++j)
            M[i * C + j] = j < i ? p.scale * dec(j, i) *
                                       dot_rows(qi, k + tok_off(b, t0 + j, h, Tn, H, dk), dk) *
                                       dot_rows(doi, v + tok_off(b, t0 + j, h, Tn, H, dv), dv)
                                 : 0.f;
    }
    float zp = 0.f;
    for (size_t x = threadIdx.x; x < nstate; x += blockDim.x) zp = fmaf(S[x], G[x], zp);
    red[threadIdx.x] = zp;
    __syncthreads();
    float z = 0.f;
    for (int x = 0; x < (int)blockDim.x; ++x) z += red[x];
    z *= dec(-1, Cc - 1);
    for (int t = threadIdx.x; t < Cc; t += blockDim.x) {
        float acc = z;
        for (int i = t; i < Cc; ++i) {
            acc += r[i];
            for (int j = 0; j < t; ++j) acc += M[i * C + j];
        }
        for (int j = 0; j < t; ++j) acc += e[j];
        const size_t gidx = ((size_t)b * Tn + t0 + t) * H + h;
        p.dg[gidx] = p.g[gidx] > kResetLogDecay ? acc : 0.f;   // a clearing gate: exp(g) = 0
    }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T>
cudaError_t fwd_simt_impl(const FwdParams &p, cudaStream_t s, int *launches) {
    const size_t smem = sizeof(float) * ((size_t)p.dk * kSlice + (size_t)p.chunk * p.chunk +
                                         (size_t)p.chunk * kSlice + p.chunk + 1 + 2 * (size_t)p.chunk);
    cudaError_t e = set_smem(fwd_simt_kernel<T>, smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.B * p.H), (unsigned)((p.dv + kSlice - 1) / kSlice));
    fwd_simt_kernel<T><<<grid, kThreads, smem, s>>>(p);
    if (launches) ++*launches;
    return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_simt_impl(const BwdParams &p, cudaStream_t s, int *launches) {
    // + [C] gate sums and [C] clearing counts (gated mode)
    const size_t sm_rows = sizeof(float) * ((size_t)kSlice * p.dv + (size_t)p.chunk * p.chunk + 3 * p.chunk + 1);
    const size_t sm_cols = sizeof(float) * ((size_t)p.dk * kSlice + (size_t)p.chunk * p.chunk + 3 * p.chunk + 1);
    const size_t sm_dg = sizeof(float) * ((size_t)p.chunk * p.chunk + 4 * p.chunk + kThreads);
    cudaError_t e;
    if ((e = set_smem(bwd_dq_simt_kernel<T>, sm_rows)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_dk_simt_kernel<T>, sm_rows)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_dv_simt_kernel<T>, sm_cols)) != cudaSuccess) return e;
    if (p.g && (e = set_smem(bwd_dg_simt_kernel<T>, sm_dg)) != cudaSuccess) return e;
    const unsigned bh = (unsigned)(p.B * p.H);
    dim3 grid_rows(bh, (unsigned)((p.dk + kSlice - 1) / kSlice));
    dim3 grid_cols(bh, (unsigned)((p.dv + kSlice - 1) / kSlice));
    if (p.dq_out) {
        bwd_dq_simt_kernel<T><<<grid_rows, kThreads, sm_rows, s>>>(p);
        if (launches) ++*launches;
    }
    if (p.dk_out || p.dh0) {
        bwd_dk_simt_kernel<T><<<grid_rows, kThreads, sm_rows, s>>>(p);
        if (launches) ++*launches;
    }
    if (p.dv_out) {
        bwd_dv_simt_kernel<T><<<grid_cols, kThreads, sm_cols, s>>>(p);
        if (launches) ++*launches;
    }
    if (p.g && p.dg) {   // gated: after dq and dk, whose saved states it reads (same stream)
        dim3 grid_dg(bh, (unsigned)((p.T + p.chunk - 1) / p.chunk));
        bwd_dg_simt_kernel<T><<<grid_dg, kThreads, sm_dg, s>>>(p);
        if (launches) ++*launches;
    }
    return cudaGetLastError();
}

__global__ void copy_state_kernel(const float *src, float *dst, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : 0.f;
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdParams &p, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? fwd_simt_impl<__nv_bfloat16>(p, s, launches) : fwd_simt_impl<float>(p, s, launches);
}

cudaError_t launch_bwd_simt(const BwdParams &p, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? bwd_simt_impl<__nv_bfloat16>(p, s, launches) : bwd_simt_impl<float>(p, s, launches);
}

cudaError_t launch_copy_state(const float *src, float *dst, size_t n, cudaStream_t s, int *launches) {
    if (n == 0 || dst == nullptr) return cudaSuccess;
    unsigned blocks = (unsigned)((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    copy_state_kernel<<<blocks, 256, 0, s>>>(src, dst, n);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace gla
