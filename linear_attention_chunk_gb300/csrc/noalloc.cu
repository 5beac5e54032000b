// noalloc.cu -- gla_chunk_fwd_noalloc: the chunked forward for callers that
// cannot allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc: an
// inference plugin whose host framework owns every byte of device memory
// through its own pool, or a serving loop that must not stall the device
// (cudaMalloc can synchronise it) or fail with out-of-memory in the middle
// of a step. gla_chunk_fwd asks such callers for a workspace when it splits
// a long sequence into segments; this entry point needs none. Its scratch is
// a fixed array in the library's own device memory, reserved when the
// library is loaded on a device and held until the process exits.
//
// This entry point has no counterpart in the method's description; it only
// changes where the segmentation scratch lives.
#include <cuda_runtime.h>

#include <mutex>

#include "gla.h"
#include "kernels.h"

namespace {

// Scratch of the segmented forward: per-segment local end states and
// per-segment initial states, 2 x segments x B x H x dk x dv x 4 bytes. The
// segment plan splits only when B x H x 2 CTAs leave the GPU under-filled,
// and keeps segments x B x H at or below the SM count, so the scratch is at
// most 2 x SMs x 73,728 bytes: 22.4 MB on the GB300's 152 SMs, and within
// this 24 MiB array on any GPU with up to 170 SMs.
constexpr size_t kNoallocScratchBytes = 24u << 20;   // 24 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of this device's scratch array, looked up once per device
// (the host-side symbol is only a stand-in and must never reach a kernel).
gla_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        gla::set_error_detail("gla_chunk_fwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return GLA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        gla::set_error_detail("gla_chunk_fwd_noalloc: device index %d out of range", dev);
        return GLA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            gla::set_error_detail("gla_chunk_fwd_noalloc: cudaGetSymbolAddress(scratch): %s",
                                  cudaGetErrorString(e));
            return GLA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GLA_OK;
}

}  // namespace

extern "C" gla_status gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const float *log_lambda, const float *h0, float scale, int B,
                                            int T, int H, int dk, int dv, int chunk, gla_dtype dtype, void *o,
                                            float *hT, void *stream) {
    // No launch has happened yet: a failure below reports none.
    gla::reset_call_state();
    const size_t need = gla_chunk_fwd_workspace_size(B, T, H, dk, dv, chunk, dtype);
    // A segment plan larger than the array (only possible on a GPU with more
    // than 170 SMs) falls back to one chain per (b, h), which needs no
    // scratch: slower, but the same result, and still no allocation.
    void *scratch = nullptr;
    if (need > 0 && need <= kNoallocScratchBytes) {
        const gla_status st = scratch_address(&scratch);
        if (st != GLA_OK) return st;
    }
    return gla_chunk_fwd(q, k, v, log_lambda, h0, scale, B, T, H, dk, dv, chunk, dtype, o, hT, scratch,
                         scratch ? kNoallocScratchBytes : 0, stream);
}
