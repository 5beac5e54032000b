// bwd_dispatch.cu -- bf16 backward dispatch.
// The per-head decay: two tensor-core launches.
//   dk, dv, dh0: one launch pairing, for each (b, h), the transposed-shape
//                chunk kernel in reverse time (dk) with the one-CTA-per-head
//                chunk kernel in reverse time (dv, dh0) on neighbouring CTAs,
//                so that q and do leave DRAM once for both (bwd_tc.cu)
//   dq:          the transposed-shape chunk kernel, forward in time (bwd_tc.cu)
// The per-token decay: dq, dk (bwd_tc.cu) and dv, dh0 (the one-CTA-per-head
// chunk kernel in reverse time, fwd_full.cu) as three launches, then the gate
// gradient after dq and dk (dg_tc.cu).
// The launches are independent and run concurrently, on the caller's stream
// and on helper streams forked from it and joined back to it with events:
// each launch alone ends in a partial wave of CTAs; side by side, one
// kernel's CTAs fill the SMs the others leave idle (415.8 -> 374.9 us for the
// training workload when the backward was three launches). Fork and join are
// event records and waits, so the call stays asynchronous and can be
// captured in a CUDA graph. The helper streams and events are created once
// per host thread and device, and kept.
#include "kernels.h"

namespace gla {
namespace {

constexpr int kMaxDev = 64;

struct Fork {
    cudaStream_t aux[2] = {nullptr, nullptr};
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
};

cudaError_t fork_for_device(Fork **out) {
    thread_local Fork forks[kMaxDev];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    Fork &f = forks[dev];
    if (!f.aux[0]) {
        for (int i = 0; i < 2; ++i)
            if ((e = cudaStreamCreateWithFlags(&f.aux[i], cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (int i = 0; i < 3; ++i)
            if ((e = cudaEventCreateWithFlags(&f.ev[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &f;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    Fork *f = nullptr;
    cudaError_t e = fork_for_device(&f);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(f->ev[0], s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(f->aux[0], f->ev[0], 0)) != cudaSuccess) return e;
    cudaError_t el = launch_bwd_kv_tc(p, s, launches);
    if (el == cudaSuccess) el = launch_bwd_dq_tc(p, f->aux[0], launches);
    // Join whatever was launched before reporting, so the caller's stream
    // never runs ahead of work still in flight on the helper stream.
    if ((e = cudaEventRecord(f->ev[1], f->aux[0])) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, f->ev[1], 0)) != cudaSuccess) return e;
    return el;
}

// The gated backward: the same three launches in gated mode, dq and dk each
// saving the state copy entering every chunk in its half of the workspace,
// then the gate gradient from both sets of copies (after dq and dk, beside
// dv, on the first helper stream).
cudaError_t launch_bwd_gated_tc(const BwdParams &p, cudaStream_t s, int *launches) {
    Fork *f = nullptr;
    cudaError_t e = fork_for_device(&f);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventRecord(f->ev[0], s)) != cudaSuccess) return e;
    for (int i = 0; i < 2; ++i)
        if ((e = cudaStreamWaitEvent(f->aux[i], f->ev[0], 0)) != cudaSuccess) return e;
    cudaError_t el = launch_bwd_dq_tc(p, f->aux[0], launches);
    if (el == cudaSuccess) el = launch_bwd_dk_tc(p, f->aux[1], launches);
    if (el == cudaSuccess) el = launch_bwd_dv_full_tc(p, s, launches);
    if ((e = cudaEventRecord(f->ev[1], f->aux[1])) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(f->aux[0], f->ev[1], 0)) != cudaSuccess) return e;
    if (el == cudaSuccess) el = launch_bwd_dg_tc(p, f->aux[0], launches);
    // Join both helper streams before reporting (see launch_bwd_tc).
    if ((e = cudaEventRecord(f->ev[2], f->aux[0])) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, f->ev[2], 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, f->ev[1], 0)) != cudaSuccess) return e;
    return el;
}

size_t bwd_tc_workspace_size(int, int, int, int) { return 0; }

}  // namespace gla
