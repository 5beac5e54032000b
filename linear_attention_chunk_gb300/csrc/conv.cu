// conv.cu -- the causal depthwise Conv1d (width 4) with SiLU in front of the
// mixer, from "Beyond the KV cache: Training and serving i14's Laplace 3B
// linear attention model on AWS Trainium2 with native PyTorch", section "i14
// and the Laplace 3B architecture", paragraph "Normalisation and
// convolution" (no equation survives; the reading), per channel c:
//     y_t[c] = SiLU( sum_{i=0..3} w[c][i] x_{t-3+i}[c] + b[c] ),
// where inputs before a sequence's first token in this call come from its
// conv window: the sequence's last four inputs so far, fp32, oldest first.
//
// The op streams x in and y out (2 x D x sizeof(T) bytes per token) and is
// HBM-bound. The main kernel is persistent, one CTA per SM, each with one
// contiguous range of tokens: a producer warp moves whole rows of x into a
// 6-stage shared-memory ring with 1-D bulk copies (about 24 KB per stage,
// one copy per stage, completion on an mbarrier; 144 KB in flight per SM),
// and each consumer thread owns one vector of channels for the whole range, so the previous three inputs stay in its registers
// and only a sequence's first token in the range reads history from memory.
// Arithmetic is on fp32 pairs (the packed f32x2 FMA of sm_100 and later);
// at bf16 the SiLU is 0.5a(1 + tanh(a/2)) with the hardware tanh (one
// special-function op per element), at fp32 a / (1 + e^-a). A stage that
// lies inside one sequence (the common case) is computed branch-free, all
// its rows at once.
//
// Windows: a CTA range never starts on the second or third token of a
// sequence, so the CTA holding a sequence's first token is the only reader
// of its old window, and each thread rewrites its own channels of that
// window right after reading them -- in place is safe with no second pass.
// Rows up to 6 KB (D <= 3072 at bf16) use 8-byte channel vectors (four
// channels per thread, 24 consumer warps at D = 3072) for latency hiding,
// rows up to 7.5 KB 16-byte vectors; wider rows take a plain kernel (a
// thread per 16-byte vector and tile of 16 tokens, loads issued up front)
// followed by a small window kernel. The serving step is a thread per four
// channels of one sequence.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace gla {
namespace {

using namespace ptx;

constexpr int kTaps = 4;
constexpr int kTile = 16;       // tokens per thread (plain kernel)
constexpr int kThreads = 128;   // channel vectors per CTA (plain, window and step kernels)


// ----------------------------------------------------------- fp32 pairs
using f2 = uint64_t;   // two fp32 lanes (lo = even channel, hi = odd channel)

__device__ __forceinline__ f2 f2_bits(uint32_t lo, uint32_t hi) {
    f2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void f2_split(f2 v, uint32_t &lo, uint32_t &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float tanh_fast(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// VB bytes of T (a thread's channel vector: VB = 16 or 8) as W = VB/4
// 32-bit words, and as P fp32 channel pairs.
template <int VB> struct VecT;
template <> struct VecT<16> { using type = uint4; };
template <> struct VecT<8> { using type = uint2; };

template <int VB>
__device__ __forceinline__ void vec_words(const typename VecT<VB>::type &u, uint32_t (&w)[VB / 4]) {
    if constexpr (VB == 16) {
        w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else {
        w[0] = u.x; w[1] = u.y;
    }
}
template <int VB>
__device__ __forceinline__ typename VecT<VB>::type words_vec(const uint32_t (&w)[VB / 4]) {
    if constexpr (VB == 16) return make_uint4(w[0], w[1], w[2], w[3]);
    else return make_uint2(w[0], w[1]);
}

template <typename T, int VB> constexpr int pairs_of() { return VB / (int)sizeof(T) / 2; }

template <typename T, int VB>
__device__ __forceinline__ void unpack_pairs(const typename VecT<VB>::type &u, f2 (&p)[pairs_of<T, VB>()]) {
    uint32_t w[VB / 4];
    vec_words<VB>(u, w);
    if constexpr (std::is_same<T, float>::value) {
#pragma unroll
        for (int e = 0; e < VB / 8; ++e) p[e] = f2_bits(w[2 * e], w[2 * e + 1]);
    } else {   // bf16 -> fp32 is a 16-bit shift
#pragma unroll
        for (int e = 0; e < VB / 4; ++e) p[e] = f2_bits(w[e] << 16, w[e] & 0xffff0000u);
    }
}

// y pairs -> VB bytes of T (bf16 rounds to nearest even).
template <typename T, int VB>
__device__ __forceinline__ typename VecT<VB>::type pack_pairs(const f2 (&p)[pairs_of<T, VB>()]) {
    constexpr int P = pairs_of<T, VB>();
    uint32_t w[VB / 4];
#pragma unroll
    for (int e = 0; e < P; ++e) {
        uint32_t lo, hi;
        f2_split(p[e], lo, hi);
        if constexpr (std::is_same<T, float>::value) {
            w[2 * e] = lo;
            w[2 * e + 1] = hi;
        } else {
            w[e] = pack_bf16x2(__uint_as_float(lo), __uint_as_float(hi));
        }
    }
    return words_vec<VB>(w);
}

template <typename T, int VB>
__device__ __forceinline__ typename VecT<VB>::type ld_vec(const T *p) {
    return __ldg(reinterpret_cast<const typename VecT<VB>::type *>(p));
}

// fp32 pairs in memory (windows, bias): 16-byte accesses, 8-byte for an odd pair.
template <int P>
__device__ __forceinline__ void load_pairs(const float *p, f2 (&f)[P]) {
#pragma unroll
    for (int e = 0; e + 1 < P; e += 2) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p + 2 * e);
        f[e] = f2_bits(u.x, u.y);
        f[e + 1] = f2_bits(u.z, u.w);
    }
    if (P % 2) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p + 2 * (P - 1));
        f[P - 1] = f2_bits(u.x, u.y);
    }
}

template <int P>
__device__ __forceinline__ void store_pairs(float *p, const f2 (&f)[P]) {
#pragma unroll
    for (int e = 0; e + 1 < P; e += 2) {
        uint32_t a, b, c, d;
        f2_split(f[e], a, b);
        f2_split(f[e + 1], c, d);
        *reinterpret_cast<uint4 *>(p + 2 * e) = make_uint4(a, b, c, d);
    }
    if (P % 2) {
        uint32_t a, b;
        f2_split(f[P - 1], a, b);
        *reinterpret_cast<uint2 *>(p + 2 * (P - 1)) = make_uint2(a, b);
    }
}

// Taps and bias of one thread's channels c0 .. c0+2P-1 (w is [D, 4]). At
// bf16 they are held halved (exact: a power of two), so the accumulation
// gives a/2, the argument the tanh form of SiLU needs.
template <typename T, int P>
struct Taps {
    f2 w[kTaps][P], b[P];
    __device__ __forceinline__ void load(const float *wp, const float *bp, int c0) {
        const float k = std::is_same<T, float>::value ? 1.f : 0.5f;
#pragma unroll
        for (int e = 0; e < P; ++e) {
            const float4 u = __ldg(reinterpret_cast<const float4 *>(wp) + c0 + 2 * e);
            const float4 v = __ldg(reinterpret_cast<const float4 *>(wp) + c0 + 2 * e + 1);
            w[0][e] = f2_bits(__float_as_uint(k * u.x), __float_as_uint(k * v.x));
            w[1][e] = f2_bits(__float_as_uint(k * u.y), __float_as_uint(k * v.y));
            w[2][e] = f2_bits(__float_as_uint(k * u.z), __float_as_uint(k * v.z));
            w[3][e] = f2_bits(__float_as_uint(k * u.w), __float_as_uint(k * v.w));
            b[e] = 0;
        }
        if (bp) {
            load_pairs<P>(bp + c0, b);
            if (!std::is_same<T, float>::value)
#pragma unroll
                for (int e = 0; e < P; ++e) b[e] = mul2(b[e], f2_bits(0x3f000000u, 0x3f000000u));
        }
    }
};

// y = SiLU(w0 h0 + w1 h1 + w2 h2 + w3 x + b) for one channel pair.
template <typename T, int P>
__device__ __forceinline__ f2 conv_pair(const Taps<T, P> &tp, int e, f2 h0, f2 h1, f2 h2, f2 x) {
    f2 a = fma2(tp.w[0][e], h0, tp.b[e]);
    a = fma2(tp.w[1][e], h1, a);
    a = fma2(tp.w[2][e], h2, a);
    a = fma2(tp.w[3][e], x, a);
    uint32_t lo, hi;
    f2_split(a, lo, hi);
    if constexpr (std::is_same<T, float>::value) {
        const float l = __uint_as_float(lo), u = __uint_as_float(hi);
        // for a -> -inf the divisor overflows to inf and the result is -0, the limit
        return f2_bits(__float_as_uint(__fdividef(l, 1.f + __expf(-l))),
                       __float_as_uint(__fdividef(u, 1.f + __expf(-u))));
    } else {   // a holds a/2: y = a/2 (1 + tanh(a/2))
        const f2 t = f2_bits(__float_as_uint(tanh_fast(__uint_as_float(lo))),
                             __float_as_uint(tanh_fast(__uint_as_float(hi))));
        return fma2(a, t, a);
    }
}

template <typename T, int P>
__device__ __forceinline__ void conv_point(const Taps<T, P> &tp, const f2 (&h)[3][P], const f2 (&x)[P], f2 (&y)[P]) {
#pragma unroll
    for (int e = 0; e < P; ++e) y[e] = conv_pair<T, P>(tp, e, h[0][e], h[1][e], h[2][e], x[e]);
}

// The sequence holding token t: start s, end e, window row 0 of its slot
// before the call (nullptr: a zero window) and after it (nullptr: not
// written). Returns false when t is in no sequence (past the last one, or
// the offsets around it are bad: then the status bit is set).
template <bool kVar>
__device__ __forceinline__ bool locate(const ConvParams &p, long t, long &s, long &e, const float *&win_in,
                                       float *&win_out) {
    if (!kVar) {
        const long n = t / p.T;
        s = n * p.T;
        e = s + p.T;
        win_in = p.win_in ? p.win_in + (size_t)n * kTaps * p.D : nullptr;
        win_out = p.win_out ? p.win_out + (size_t)n * kTaps * p.D : nullptr;
        return true;
    }
    // the largest n in [0, nseq] with cu[n] <= t (offsets assumed non-decreasing)
    int lo = 0, hi = p.nseq;
    if (p.cu_seqlens[0] > t) return false;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (p.cu_seqlens[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    if (lo == p.nseq) return false;   // past the last sequence: no output
    s = p.cu_seqlens[lo];
    e = p.cu_seqlens[lo + 1];
    const int slot = p.slots ? p.slots[lo] : lo;
    if (s < 0 || e <= t || e > p.NT || slot < 0 || slot >= p.n_slots) {
        atomicOr(p.status, kDevBadState);
        return false;
    }
    win_in = p.win_in + (size_t)slot * kTaps * p.D;
    win_out = p.win_out + (size_t)slot * kTaps * p.D;
    return true;
}

// History of token t (positions t-3, t-2, t-1) for channels c0..: from x
// inside the sequence, from the window before it. x points at channel c0.
template <typename T, int VB>
__device__ __forceinline__ void load_history(const T *x, size_t D, long t, long s, const float *win, int c0,
                                             f2 (&h)[3][pairs_of<T, VB>()]) {
    constexpr int P = pairs_of<T, VB>();
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const long src = t - 3 + j;
        if (src >= s) {
            unpack_pairs<T, VB>(ld_vec<T, VB>(x + (size_t)src * D), h[j]);
        } else if (win) {
            load_pairs<P>(win + (size_t)(kTaps - (s - src)) * D + c0, h[j]);
        } else {
#pragma unroll
            for (int e = 0; e < P; ++e) h[j][e] = 0;
        }
    }
}

// ------------------------------------------------------- streaming kernel
constexpr int kStages = 6;
constexpr uint32_t kStageTarget = 24 * 1024;   // bytes of x per ring stage

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// First token of CTA c's range: an even split of the tokens, moved off the
// second and third token of a sequence (to the fourth, or the sequence's
// end) so that a sequence's old window is read by one CTA only.
template <bool kVar>
__device__ __forceinline__ long range_start(const ConvParams &p, long c, long G) {
    if (c <= 0) return 0;
    if (c >= G) return p.NT;
    long t = p.NT * c / G;
    long s, e;
    const float *wi;
    float *wo;
    if (locate<kVar>(p, t, s, e, wi, wo) && t - s > 0 && t - s < 3) t = min(s + 3, e);
    return t;
}

// Consumer threads per CTA by vector width: 8-byte vectors give twice the
// warps (latency hiding) on rows up to 6 KB; 16-byte vectors cover rows up
// to 7.5 KB. One more warp produces.
template <int VB> constexpr int stream_max_vecs() { return VB == 8 ? 768 : 480; }

// Warps 0..nw-1 consume (thread g owns channel vector g), warp nw produces;
// tiles of R rows (R = 2 or 4, unrolled) from the CTA's range start.
template <typename T, bool kVar, int R, int VB>
__global__ void __launch_bounds__(stream_max_vecs<VB>() + 32, 1) conv_stream_kernel(const ConvParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int V = VB / (int)sizeof(T), P = V / 2;
    using Vec = typename VecT<VB>::type;
    const int groups = p.D / V;
    const int nw = (groups + 31) / 32;
    const uint32_t rowbytes = (uint32_t)p.D * (uint32_t)sizeof(T);
    const uint32_t stage_bytes = (uint32_t)R * rowbytes;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t base = smem_u32(smem);
    const uint32_t bar_full = base + kStages * stage_bytes;   // rowbytes is a multiple of 16
    const uint32_t bar_empty = bar_full + 8 * kStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kStages * stage_bytes + 16 * kStages);
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, nw);
        }
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{abort_flag, p.status};
    const size_t D = (size_t)p.D;
    const long tb = range_start<kVar>(p, blockIdx.x, gridDim.x);
    const long te = range_start<kVar>(p, (long)blockIdx.x + 1, gridDim.x);
    const long ntiles = te > tb ? (te - tb + R - 1) / R : 0;

    if (kVar) {   // offsets no token leads to are checked too (a bad one only sets the status bit)
        for (long n = (long)blockIdx.x * blockDim.x + threadIdx.x; n < p.nseq; n += (long)gridDim.x * blockDim.x) {
            const int s = p.cu_seqlens[n], e = p.cu_seqlens[n + 1];
            const int slot = p.slots ? p.slots[n] : (int)n;
            if (s < 0 || e < s || e > p.NT || slot < 0 || slot >= p.n_slots) atomicOr(p.status, kDevBadState);
        }
    }

    if (warp == nw) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            long issued = 0;
            for (long i = 0; i < ntiles; ++i) {
                const int s = (int)(i % kStages);
                if (i >= kStages && !mbar_wait(bar_empty + 8 * s, (uint32_t)((i / kStages) - 1) & 1u, ctl)) break;
                const long t0 = tb + i * R;
                const uint32_t bytes = (uint32_t)min((long)R, te - t0) * rowbytes;
                mbar_arrive_expect_tx(bar_full + 8 * s, bytes);
                bulk_load(base + (uint32_t)s * stage_bytes, static_cast<const T *>(p.x) + (size_t)t0 * D, bytes,
                          bar_full + 8 * s);
                issued = i + 1;
            }
            // the copies in flight land before the CTA exits, also after an abort
            for (long j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
                mbar_wait_drain(bar_full + 8 * (uint32_t)(j % kStages), (uint32_t)(j / kStages) & 1u, 1000000ull);
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int g = threadIdx.x;
    const bool active = g < groups;
    const int c0 = (active ? g : 0) * V;
    const T *x = static_cast<const T *>(p.x) + c0;
    T *y = static_cast<T *>(p.y) + c0;
    Taps<T, P> tp;
    tp.load(p.w, p.b, c0);

    f2 h[3][P] = {};   // inputs at t-3, t-2, t-1
    long s_beg = 0, s_end = -1;
    for (long i = 0; i < ntiles; ++i) {
        const int s = (int)(i % kStages);
        if (!mbar_wait(bar_full + 8 * s, (uint32_t)(i / kStages) & 1u, ctl)) break;
        const long t0 = tb + i * R;
        const int rows = (int)min((long)R, te - t0);
        // plain shared loads: the wait above (a memory clobber) orders them
        const unsigned char *stage = smem + (size_t)s * stage_bytes + (size_t)c0 * sizeof(T);
        if (rows == R && t0 + R <= s_end) {
            // the whole stage lies in the current sequence: all R rows at once
            f2 hx[R + 3][P];   // inputs t0-3 .. t0+R-1
#pragma unroll
            for (int e = 0; e < P; ++e) {
                hx[0][e] = h[0][e];
                hx[1][e] = h[1][e];
                hx[2][e] = h[2][e];
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
                unpack_pairs<T, VB>(*reinterpret_cast<const Vec *>(stage + (size_t)r * rowbytes), hx[r + 3]);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                f2 out[P];
#pragma unroll
                for (int e = 0; e < P; ++e)
                    out[e] = conv_pair<T, P>(tp, e, hx[r][e], hx[r + 1][e], hx[r + 2][e], hx[r + 3][e]);
                if (active) *reinterpret_cast<Vec *>(y + (size_t)(t0 + r) * D) = pack_pairs<T, VB>(out);
            }
#pragma unroll
            for (int e = 0; e < P; ++e) {
                h[0][e] = hx[R][e];
                h[1][e] = hx[R + 1][e];
                h[2][e] = hx[R + 2][e];
            }
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r >= rows) break;
                const long t = t0 + r;
                if (t >= s_end) {
                    const float *wi;
                    float *wo;
                    if (!locate<kVar>(p, t, s_beg, s_end, wi, wo)) {
                        s_end = t + 1;   // look again at the next token
                        continue;
                    }
                    load_history<T, VB>(x, D, t, s_beg, wi, c0, h);
                    if (t == s_beg && wo && active) {
                        // this thread's channels of the window after the call: input
                        // e-4+k from x inside the sequence, else old row k + len (= h[k + len - 1])
                        const long len = s_end - s_beg;
#pragma unroll
                        for (int k = 0; k < kTaps; ++k) {
                            const long xs = s_end - kTaps + k;
                            f2 row[P];
                            if (xs >= s_beg) {
                                unpack_pairs<T, VB>(ld_vec<T, VB>(x + (size_t)xs * D), row);
                            } else {
                                const int j = (int)(k + len - 1);   // 0..2 here
#pragma unroll
                                for (int e = 0; e < P; ++e) row[e] = j == 0 ? h[0][e] : j == 1 ? h[1][e] : h[2][e];
                            }
                            store_pairs<P>(wo + (size_t)k * D + c0, row);
                        }
                    }
                }
                f2 xv[P], out[P];
                unpack_pairs<T, VB>(*reinterpret_cast<const Vec *>(stage + (size_t)r * rowbytes), xv);
                conv_point<T, P>(tp, h, xv, out);
#pragma unroll
                for (int e = 0; e < P; ++e) {
                    h[0][e] = h[1][e];
                    h[1][e] = h[2][e];
                    h[2][e] = xv[e];
                }
                if (active) *reinterpret_cast<Vec *>(y + (size_t)t * D) = pack_pairs<T, VB>(out);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
}

// ---------------------------------------------------------- plain kernel
// y for one tile of TILE tokens x one VB-byte channel vector per thread, all
// the tile's row loads (and the three rows before it) issued up front. The
// windows are then written by conv_window_kernel in a second launch.
template <typename T, bool kVar, int VB, int TILE>
__global__ void __launch_bounds__(kThreads) conv_fwd_kernel(const ConvParams p) {
    constexpr int V = VB / (int)sizeof(T), P = V / 2;
    using Vec = typename VecT<VB>::type;
    const int groups = p.D / V;
    const int ncb = (groups + kThreads - 1) / kThreads;
    const long tile = blockIdx.x / ncb;
    const int g = (int)(blockIdx.x % ncb) * kThreads + threadIdx.x;
    if (g >= groups) return;
    const int c0 = g * V;
    const size_t D = (size_t)p.D;
    const long t0 = tile * TILE;
    const long t1 = min(t0 + TILE, (long)p.NT);
    const T *x = static_cast<const T *>(p.x) + c0;
    T *y = static_cast<T *>(p.y) + c0;

    Vec xr[TILE], xh[3];
#pragma unroll
    for (int j = 0; j < 3; ++j)
        if (t0 - 3 + j >= 0) xh[j] = ld_vec<T, VB>(x + (size_t)(t0 - 3 + j) * D);
#pragma unroll
    for (int i = 0; i < TILE; ++i)
        if (t0 + i < t1) xr[i] = ld_vec<T, VB>(x + (size_t)(t0 + i) * D);
    Taps<T, P> tp;
    tp.load(p.w, p.b, c0);

    f2 h[3][P] = {};
    long s = 0, e = -1;
#pragma unroll
    for (int i = 0; i < TILE; ++i) {
        const long t = t0 + i;
        if (t >= t1) break;
        if (t >= e) {
            const float *wi;
            float *wo;
            if (!locate<kVar>(p, t, s, e, wi, wo)) {
                e = t + 1;
                continue;
            }
            if (i == 0 && t0 - 3 >= s) {   // the tile's first token, its history inside the sequence
#pragma unroll
                for (int j = 0; j < 3; ++j) unpack_pairs<T, VB>(xh[j], h[j]);
            } else {
                load_history<T, VB>(x, D, t, s, wi, c0, h);
            }
        }
        f2 xv[P], out[P];
        unpack_pairs<T, VB>(xr[i], xv);
        conv_point<T, P>(tp, h, xv, out);
#pragma unroll
        for (int k = 0; k < P; ++k) {
            h[0][k] = h[1][k];
            h[1][k] = h[2][k];
            h[2][k] = xv[k];
        }
        *reinterpret_cast<Vec *>(y + (size_t)t * D) = pack_pairs<T, VB>(out);
    }
}

// The window after the call, per (sequence, channel vector), for the plain
// kernel and for T = 0: row r holds the input at position e-4+r, from x
// when it lies in this call, else from the window before (row r + length).
template <typename T, bool kVar>
__global__ void __launch_bounds__(kThreads) conv_window_kernel(const ConvParams p) {
    constexpr int V = 16 / (int)sizeof(T), P = V / 2;
    const int ncb = (p.D / V + kThreads - 1) / kThreads;
    const int n = blockIdx.x / ncb;
    const int g = (int)(blockIdx.x % ncb) * kThreads + threadIdx.x;
    if (g >= p.D / V) return;
    const int c0 = g * V;
    const size_t D = (size_t)p.D;
    long s, e;
    const float *win_in;
    float *win_out;
    if (kVar) {
        s = p.cu_seqlens[n];
        e = p.cu_seqlens[n + 1];
        const int slot = p.slots ? p.slots[n] : n;
        if (s < 0 || e < s || e > p.NT || slot < 0 || slot >= p.n_slots) {
            atomicOr(p.status, kDevBadState);
            return;
        }
        if (e == s) return;   // an empty sequence leaves its slot untouched
        win_in = p.win_in + (size_t)slot * kTaps * D;
        win_out = p.win_out + (size_t)slot * kTaps * D;
    } else {
        s = (long)n * p.T;
        e = s + p.T;
        win_in = p.win_in ? p.win_in + (size_t)n * kTaps * D : nullptr;
        win_out = p.win_out + (size_t)n * kTaps * D;
    }
    const long len = e - s;
    f2 old[kTaps][P];
#pragma unroll
    for (int r = 0; r < kTaps; ++r) {
        if (win_in && r + len < kTaps) load_pairs<P>(win_in + (size_t)(r + len) * D + c0, old[r]);
        else
#pragma unroll
            for (int k = 0; k < P; ++k) old[r][k] = 0;
    }
    const T *x = static_cast<const T *>(p.x) + c0;
#pragma unroll
    for (int r = 0; r < kTaps; ++r) {
        const long src = e - kTaps + r;
        if (src >= s) {
            f2 f[P];
            unpack_pairs<T, 16>(ld_vec<T, 16>(x + (size_t)src * D), f);
            store_pairs<P>(win_out + (size_t)r * D + c0, f);
        } else {
            store_pairs<P>(win_out + (size_t)r * D + c0, old[r]);
        }
    }
}

// One token per sequence n: the window gives the three previous inputs; it
// shifts by one row and takes the new input, in place. A thread owns four
// channels (two pairs: one 16-byte access per window row), which keeps the
// registers low enough for 48 resident warps per SM: the step is a latency-
// bound gather of 7 rows per sequence.
template <typename T> constexpr int step_vb() { return std::is_same<T, float>::value ? 16 : 8; }

template <typename T>
__global__ void __launch_bounds__(kThreads) conv_step_kernel(const ConvParams p) {
    constexpr int VB = step_vb<T>(), V = VB / (int)sizeof(T), P = V / 2;
    using Vec = typename VecT<VB>::type;
    const int ncb = (p.D / V + kThreads - 1) / kThreads;
    const int n = blockIdx.x / ncb;
    const int g = (int)(blockIdx.x % ncb) * kThreads + threadIdx.x;
    if (g >= p.D / V) return;
    const int c0 = g * V;
    const size_t D = (size_t)p.D;
    float *win = p.win_out + (size_t)n * kTaps * D + c0;
    f2 h[3][P], xv[P], out[P];
#pragma unroll
    for (int j = 0; j < 3; ++j) load_pairs<P>(win + (size_t)(j + 1) * D, h[j]);
    unpack_pairs<T, VB>(ld_vec<T, VB>(static_cast<const T *>(p.x) + (size_t)n * D + c0), xv);
    Taps<T, P> tp;
    tp.load(p.w, p.b, c0);
    conv_point<T, P>(tp, h, xv, out);
    *reinterpret_cast<Vec *>(static_cast<T *>(p.y) + (size_t)n * D + c0) = pack_pairs<T, VB>(out);
#pragma unroll
    for (int j = 0; j < 3; ++j) store_pairs<P>(win + (size_t)j * D, h[j]);
    store_pairs<P>(win + (size_t)3 * D, xv);
}

template <typename T, int VB>
cudaError_t launch_stream(const ConvParams &p, bool var, cudaStream_t st) {
    const int groups = p.D * (int)sizeof(T) / VB;
    const uint32_t rowbytes = (uint32_t)p.D * (uint32_t)sizeof(T);   // <= 7.5 KB
    const int R = kStageTarget / rowbytes >= 4 ? 4 : 2;
    const size_t smem = (size_t)kStages * R * rowbytes + 16 * kStages + 16;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long ntiles = (p.NT + R - 1) / R;
    const unsigned grid = (unsigned)min(ntiles, (long)sms);
    const unsigned threads = (unsigned)(((groups + 31) / 32 + 1) * 32);
    void (*kernel)(const ConvParams);
    if (R == 4) kernel = var ? conv_stream_kernel<T, true, 4, VB> : conv_stream_kernel<T, false, 4, VB>;
    else kernel = var ? conv_stream_kernel<T, true, 2, VB> : conv_stream_kernel<T, false, 2, VB>;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    kernel<<<grid, threads, smem, st>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t conv_fwd_impl(const ConvParams &p, bool var, cudaStream_t st, int *launches) {
    constexpr int V = 16 / (int)sizeof(T);
    const int groups = p.D / V;
    const unsigned ncb = (unsigned)((groups + kThreads - 1) / kThreads);
    cudaError_t e;
    if (p.NT > 0 && 2 * groups <= stream_max_vecs<8>()) {
        if (launches) ++*launches;
        return launch_stream<T, 8>(p, var, st);   // the windows are written by the same kernel
    }
    if (p.NT > 0 && groups <= stream_max_vecs<16>()) {
        if (launches) ++*launches;
        return launch_stream<T, 16>(p, var, st);
    }
    if (p.NT > 0) {
        const size_t blocks = (size_t)((p.NT + kTile - 1) / kTile) * ncb;
        if (blocks > 0x7fffffffull) return cudaErrorInvalidValue;
        if (var) conv_fwd_kernel<T, true, 16, kTile><<<(unsigned)blocks, kThreads, 0, st>>>(p);
        else conv_fwd_kernel<T, false, 16, kTile><<<(unsigned)blocks, kThreads, 0, st>>>(p);
        if (launches) ++*launches;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (p.win_out && p.nseq > 0) {
        const size_t blocks = (size_t)p.nseq * ncb;
        if (blocks > 0x7fffffffull) return cudaErrorInvalidValue;
        if (var) conv_window_kernel<T, true><<<(unsigned)blocks, kThreads, 0, st>>>(p);
        else conv_window_kernel<T, false><<<(unsigned)blocks, kThreads, 0, st>>>(p);
        if (launches) ++*launches;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t conv_step_impl(const ConvParams &p, cudaStream_t st, int *launches) {
    constexpr int V = step_vb<T>() / (int)sizeof(T);
    const size_t blocks = (size_t)p.nseq * ((p.D / V + kThreads - 1) / kThreads);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffull) return cudaErrorInvalidValue;
    conv_step_kernel<T><<<(unsigned)blocks, kThreads, 0, st>>>(p);
    if (launches) ++*launches;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv_fwd(const ConvParams &p, bool varlen, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? conv_fwd_impl<__nv_bfloat16>(p, varlen, s, launches) : conv_fwd_impl<float>(p, varlen, s, launches);
}

cudaError_t launch_conv_step(const ConvParams &p, bool bf16, cudaStream_t s, int *launches) {
    return bf16 ? conv_step_impl<__nv_bfloat16>(p, s, launches) : conv_step_impl<float>(p, s, launches);
}

}  // namespace gla
