#!/usr/bin/env python3
"""Benchmark of libgla, the Simple GLA mixer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gla|reference]
                    [--mode all|fwd|fwd_bwd|decode|long|varlen|mixer|conv|gated] [--batch B] [--no-e2e]
                    [--no-cpu-baseline]

Prints ONE JSON line (rank 0). The headline `value` is the chunked forward
over the Laplace-layer workload (bf16, B=8, H=16, T=2048, dk=96, dv=192,
C=128: tokens/s = B*T per call over all heads). `modes` carries the same
measurement for the training forward+backward workload (B=16, tokens/s),
the serving decode workload (1,280 sequences x 16 heads x 24 distinct layer
states per step, seq-steps/s), the long-context prefill (T=65,536, chunk 128
and 64) and the variable-length serving prefill into the decode state pool
(64 prompts of 64..4,096 tokens), the mixer epilogue (fused into the
decode step, and standalone over the layer-forward output), the causal
Conv1d, and the forward with a per-token (data-dependent) decay on the
layer-forward shape, each with its own roofline.

Timing: W untimed warm-up steps, then exactly K steps between two
barrier + synchronize pairs, on the device with CUDA events recorded on the
stream the kernels run on; the max over ranks is taken. Every workload's
inputs exceed the 129 MB L2, so no flush is done between steps.
`--impl reference` times the double-precision CPU oracle instead (rank 0
only), on bounded samples of the same workloads.

Multi-GPU (torchrun): every rank runs its own copy of the workload on its
own GPU (independent batches, no collective on the data path); `value` is
the total over ranks divided by the slowest rank's time (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

# More hardware work queues than CUDA's default of 8, set before any CUDA
# context exists: the library's backward helper streams, the copy streams of
# the end-to-end legs and the compute stream must not share a queue, or their
# work serialises behind one another.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gla_gen as gen  # noqa: E402

METRIC = "Simple-GLA tokens/s (fwd, fwd+bwd), decode seq-steps/s; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

DK, DV, H = 96, 192, 16
STATE_BYTES = DK * DV * 4
CHUNK = 128


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def committed_traffic(kernel: str):
    """Per-launch DRAM traffic of `kernel` from its committed ncu summary, if
    the summary's recorded source hash still matches the kernel source."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", f"{kernel}.md")
    if not os.path.exists(prof):
        return None, None
    fields = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    srcs = [x.strip() for x in fields.get("source_files", "").split(",") if x.strip()]
    if not srcs or "traffic_bytes_per_launch" not in fields:
        return None, None
    try:
        h = hashlib.sha256()
        for src in srcs:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        digest = h.hexdigest()[:16]
    except OSError:
        return None, None
    if digest != fields.get("source_sha256_16"):
        return None, fields.get("workload")
    try:
        return float(fields["traffic_bytes_per_launch"]), fields.get("workload")
    except ValueError:
        return None, None


# ------------------------------------------------------------ algorithmic work
def fwd_work(B, T, with_h0, with_hT, C=CHUNK):
    """Bytes and tensor-core FLOPs of one gla_chunk_fwd call (bf16 q,k,v,o)."""
    ht = B * H * T
    bytes_ = ht * (2 * DK * 2 + 2 * DV * 2) + B * H * STATE_BYTES * (int(with_h0) + int(with_hT))
    flops_full = ht * (2 * C * DK + 2 * C * DV + 4 * DK * DV)
    flops_causal = ht * ((C + 1) * DK + (C + 1) * DV + 4 * DK * DV)
    return bytes_, flops_full, flops_causal


def bwd_work(B, T, with_h0, with_dhT, with_dh0, C=CHUNK):
    """Algorithmic bytes and tensor FLOPs of one gla_chunk_bwd call.
    Bytes: q, k, v, do read once and dq, dk, dv written once (1,920 B per
    head-token at bf16) plus the states. FLOPs, full tiles, per head-token:
    the two scores dO V^T (2 C dv, shared by dq and dk) and Q K^T (2 C dk),
    the three intra products dP K, dP^T Q (2 C dk each) and P^T dO (2 C dv),
    and five state-sized products (dO S^T, V G^T, K G, the recomputed K^T V
    and the gradient update Q^T dO; 2 dk dv each): 356,352 at C = 128. The
    launches issue more (each of the dq and dk kernels forms dO V^T):
    `issued` counts that."""
    ht = B * H * T
    bytes_ = ht * (4 * DK * 2 + 3 * DV * 2) + \
        B * H * STATE_BYTES * (int(with_h0) + int(with_dhT) + int(with_dh0))
    flops = ht * (2 * 2 * C * DV + 3 * 2 * C * DK + 5 * 2 * DK * DV)
    issued = flops + ht * 2 * C * DV
    return bytes_, flops, issued


def decode_work(N):
    per = 2 * STATE_BYTES + 2 * DK * 2 + 2 * DV * 2
    return N * H * per, N * H * 4 * DK * DV


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms in the background; summarised over a
    time window (the timed region)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.samples = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if bus_id:
            cmd.insert(1, f"--id={bus_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [p for (t, p) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not win:
            # a timed region shorter than the sampling period: nearest samples
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            win = [p for (_, p) in near]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(win[0][1]), "power_w_max": max((num(p[2]) or 0) for p in win),
                "samples": len(win), "reasons": reasons}


# -------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------ our kernels
def dev_tensor(x, dtype_str, device):
    import torch
    if dtype_str == "bf16":
        return torch.from_numpy(gen.bf16_bits(x).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


def time_steps(step_fns, K, W, dist, stream, graph=None):
    """Run W warm-up steps, then K timed steps between one pair of CUDA events
    on `stream` (an event between every step would add a gap of its own).
    With graph (the default, see --no-graph) one step's launches are captured
    once into a CUDA graph after the warm-up and the timed steps replay it: the
    same kernels on the same buffers, without per-launch host overhead.
    Returns (total_ms, per-step ms list, wall window, launches in timed region)."""
    import torch
    from linear_attention_chunk_gb300 import gla_check
    graph = GRAPH if graph is None else graph
    for _ in range(W):
        step_fns()
    gla_check()
    g = None
    per_step = 0
    if graph:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            per_step = step_fns()
        torch.cuda.synchronize()
        gla_check()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    launches = 0
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(K):
            if g is not None:
                g.replay()
                launches += per_step
            else:
                launches += step_fns()
        end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    dist.barrier()
    gla_check()
    total = start.elapsed_time(end)
    return total, [total / K] * K, (t0, t1), launches


GRAPH = True


def headline_config(world, B=8, T=2048):
    """The config of the headline line (the layer forward); the reference arm
    reports the same dict."""
    bytes_ = fwd_work(B, T, False, True)[0]
    return {"workload": f"layer_fwd_bf16_B{B}_H16_T{T}", "B": B, "T": T, "H": H, "dk": DK, "dv": DV,
            "chunk": CHUNK, "h0": "none", "hT": "written",
            "l2": f"inputs larger than L2 ({bytes_ / 1e6:.0f} MB per step), no flush",
            "parallelism": f"replicas x{world} (independent batches)"}


def bench_fwd(args, dist, device, stream, peaks, sampler):
    import torch
    import linear_attention_chunk_gb300 as gla
    B = args.batch or 8
    T = 2048
    c = gen.layer_fwd(seed=1, B=B, T=T)
    q, k, v = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v))
    ll = torch.from_numpy(c.log_lambda).to(device)
    o = torch.empty((B, T, H, DV), dtype=torch.bfloat16, device=device)
    hT = torch.empty((B, H, DK, DV), dtype=torch.float32, device=device)
    ws_n = gla.gla_chunk_fwd_workspace_size(B, T, H, DK, DV, CHUNK)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)

    def step():
        gla.gla_chunk_fwd(q, k, v, ll, None, c.scale, CHUNK, o=o, hT=hT, workspace=ws, stream=stream)
        return gla.gla_last_launch_count()

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    tokens = B * T * dist.world
    bytes_, fl_full, fl_causal = fwd_work(B, T, False, True)
    avg_ms = statistics.mean(per)
    ach_gbs = bytes_ / (avg_ms * 1e-3) / 1e9
    ach_tf = fl_full / (avg_ms * 1e-3) / 1e12
    traffic, traffic_wl = committed_traffic("gla_fwd_full")
    res = {
        "value": tokens * args.steps / (total * 1e-3), "unit": "tokens/s", "ms_per_step": total / args.steps,
        "config": headline_config(dist.world, B, T),
        "roofline": {"bound": "hbm", "achieved": ach_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "algorithmic_bytes_per_launch": bytes_, "avg_launch_ms": avg_ms,
                     "peak_source": peaks["source"]},
        "tensor": {"achieved": ach_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": ach_tf / peaks["bf16_tflops"], "flops_per_launch": fl_full,
                   "causal_flops_per_launch": fl_causal, "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    if not args.no_e2e:
        res["e2e"] = e2e_fwd(args, dist, device, stream, c, ll)
    del q, k, v, o, hT
    return res


def gated_case(B=8, T=2048):
    """The layer-forward shape with per-token log-decays of gated linear
    attention (log sigmoid(x)/16, x ~ N(0, 1)) in place of the per-head one."""
    c = gen.make_case(B, T, H, DK, DV, seed=1, normalise_k=True, chunk=CHUNK, gate="gla",
                      name=f"gated_fwd_bf16_B{B}_H16_T{T}")
    return c


def bench_gated(args, dist, device, stream, peaks, sampler):
    """The chunked forward with a per-token (data-dependent) decay,
    gla_chunk_fwd_gated, on the layer-forward shape."""
    import torch
    import linear_attention_chunk_gb300 as gla
    B = args.batch or 8
    T = 2048
    c = gated_case(B, T)
    q, k, v = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v))
    g = torch.from_numpy(c.extra["g"]).to(device)
    o = torch.empty((B, T, H, DV), dtype=torch.bfloat16, device=device)
    hT = torch.empty((B, H, DK, DV), dtype=torch.float32, device=device)

    def step():
        gla.gla_chunk_fwd_gated(q, k, v, g, None, c.scale, CHUNK, o=o, hT=hT, stream=stream)
        return gla.gla_last_launch_count()

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    bytes_, fl_full, fl_causal = fwd_work(B, T, False, True)
    bytes_ += B * T * H * 4                     # g, fp32 per token and head
    avg_ms = statistics.mean(per)
    traffic, _ = committed_traffic("gla_fwd_gated")   # per B=8 launch
    ach_gbs = bytes_ / (avg_ms * 1e-3) / 1e9
    ach_tf = fl_full / (avg_ms * 1e-3) / 1e12
    res = {
        "value": B * T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps,
        "config": {"workload": c.name, "B": B, "T": T, "H": H, "dk": DK, "dv": DV, "chunk": CHUNK,
                   "gates": "log sigmoid(x)/16, x ~ N(0,1), per token and head", "h0": "none", "hT": "written",
                   "l2": f"inputs larger than L2 ({bytes_ / 1e6:.0f} MB per step), no flush"},
        "roofline": {"bound": "hbm", "achieved": ach_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach_gbs / peaks["hbm_gbs"],
                     "traffic": traffic * B / 8 if traffic is not None else None,
                     "algorithmic_bytes_per_launch": bytes_, "avg_launch_ms": avg_ms,
                     "peak_source": peaks["source"]},
        "tensor": {"achieved": ach_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": ach_tf / peaks["bf16_tflops"], "flops_per_launch": fl_full,
                   "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    del q, k, v, g, o, hT
    res["long"] = bench_gated_long(args, dist, device, stream, peaks, sampler)
    res["bwd"] = bench_gated_bwd(args, dist, device, stream, peaks, sampler)
    return res


def bench_gated_bwd(args, dist, device, stream, peaks, sampler):
    """The backward with a per-token decay, gla_chunk_bwd_gated (dq, dk, dv,
    dh0 and the gate gradient dg), on the training shape (B=16, H=16,
    T=2048, chunk 128, h0 ~ N(0, 0.02)) with gated linear attention's gates."""
    import torch
    import linear_attention_chunk_gb300 as gla
    B, T = args.batch or 16, 2048
    c = gen.make_case(B, T, H, DK, DV, seed=2, normalise_k=True, h0_std=0.02, with_grad=True, chunk=CHUNK,
                      gate="gla", name=f"gated_bwd_bf16_B{B}_H16_T{T}")
    q, k, v, do = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v, c.do))
    g = torch.from_numpy(c.extra["g"]).to(device)
    h0 = torch.from_numpy(c.h0).to(device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dh0 = torch.empty_like(h0)
    dg = torch.empty_like(g)
    ws = torch.empty(gla.gla_chunk_bwd_gated_workspace_size(B, T, H, DK, DV, CHUNK), dtype=torch.uint8,
                     device=device)

    def step():
        gla.gla_chunk_bwd_gated(q, k, v, g, do, h0, None, c.scale, CHUNK, dq=dq, dk=dk, dv=dv, dh0=dh0, dg=dg,
                                workspace=ws, stream=stream)
        return gla.gla_last_launch_count()

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    bytes_ = bwd_work(B, T, True, False, True)[0] + B * T * H * 4 * 2     # + g in, dg out
    avg_ms = statistics.mean(per)
    ach = bytes_ / (avg_ms * 1e-3) / 1e9
    traffic, _ = committed_traffic("gla_chunk_bwd_gated")
    res = {
        "value": B * T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps,
        "config": {"workload": c.name, "B": B, "T": T, "H": H, "chunk": CHUNK, "h0": "N(0,0.02)", "dhT": "none",
                   "gates": "log sigmoid(x)/16, x ~ N(0,1), per token and head", "outputs": "dq, dk, dv, dh0, dg",
                   "l2": f"inputs larger than L2 ({bytes_ / 1e6:.0f} MB per call), no flush"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": traffic * B / 16 if traffic is not None else None,
                     "algorithmic_bytes_per_call": bytes_, "avg_call_ms": avg_ms,
                     "launches_per_call": launches // max(args.steps, 1), "peak_source": peaks["source"],
                     "note": "q, k, v, do, g in; dq, dk, dv, dg out (1,928 B per head-token) + h0, dh0; the saved "
                             "chunk states (2 x 288 B per head-token written and read) are not counted as work"},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    del q, k, v, do, g, h0, dq, dk, dv, dh0, dg, ws
    return res


def bench_gated_long(args, dist, device, stream, peaks, sampler):
    """The long-context prefill shape (B=1, H=16, T=65,536, chunk 128, h0 ~
    N(0, 0.1)) with per-token gates: split into segments whose decays are the
    exp of their summed gates. The single-chain time (workspace too small to
    split) is reported beside it."""
    import torch
    import linear_attention_chunk_gb300 as gla
    T = args.long_T or 65536
    c = gen.make_case(1, T, H, DK, DV, seed=4, normalise_k=False, h0_std=0.1, chunk=CHUNK, gate="gla",
                      name=f"gated_long_prefill_bf16_B1_H16_T{T}")
    q, k, v = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v))
    g = torch.from_numpy(c.extra["g"]).to(device)
    h0 = torch.from_numpy(c.h0).to(device)
    o = torch.empty((1, T, H, DV), dtype=torch.bfloat16, device=device)
    hT = torch.empty((1, H, DK, DV), dtype=torch.float32, device=device)
    out = {}
    for split in (True, False):
        n = gla.gla_chunk_fwd_gated_workspace_size(1, T, H, DK, DV, CHUNK) if split else 0
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=device)

        def step():
            gla.gla_chunk_fwd_gated(q, k, v, g, h0, c.scale, CHUNK, o=o, hT=hT, workspace=ws, stream=stream)
            return gla.gla_last_launch_count()

        total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
        total = dist.max(total)
        bytes_ = fwd_work(1, T, True, True)[0] + T * H * 4
        avg_ms = statistics.mean(per)
        ach = bytes_ / (avg_ms * 1e-3) / 1e9
        out[split] = {
            "value": T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
            "ms_per_step": total / args.steps,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes_per_call": bytes_,
                         "avg_call_ms": avg_ms, "launches_per_call": launches // max(args.steps, 1),
                         "peak_source": peaks["source"]},
            "gpu_launches": launches,
            "clocks": sampler.summary(*win) if sampler else None,
        }
    res = dict(out[True])
    res["config"] = {"workload": c.name, "B": 1, "T": T, "H": H, "chunk": CHUNK, "h0": "N(0,0.1)",
                     "gates": "log sigmoid(x)/16, x ~ N(0,1), per token and head"}
    res["single_chain"] = out[False]
    del q, k, v, g, o, hT, h0
    return res


def e2e_pipelined(args, dist, device, stream, host_in, host_out, compute):
    """Steps through the public API with host buffers, pipelined across steps:
    step i's inputs are copied host -> device on their own stream while step
    i-1 computes, and step i's outputs are read back on a third stream while
    step i+1 computes. Device inputs and outputs are double-buffered; every
    step's copies and kernels lie inside the timed region, which runs from
    the first copy in to the last copy out. compute(d_in, d_out, stream)
    launches one step on `stream` and returns its launch count."""
    import torch
    from linear_attention_chunk_gb300 import gla_check
    if device not in _COPY_STREAMS:   # created once: a fresh pair per call could land on busy queues
        _COPY_STREAMS[device] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    s_in, s_out = _COPY_STREAMS[device]
    d_in = [[torch.empty_like(h, device=device) for h in host_in] for _ in range(2)]
    d_out = [[torch.empty_like(h, device=device) for h in host_out] for _ in range(2)]
    ev = lambda: torch.cuda.Event()

    def run(n_steps, start=None, end=None):
        comp_done, out_done = [None, None], [None, None]
        launches = 0
        if start is not None:
            start.record(s_in)
        for i in range(n_steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if comp_done[b] is not None:
                    s_in.wait_event(comp_done[b])          # step i-2 is done reading these inputs
                for d, h in zip(d_in[b], host_in):
                    d.copy_(h, non_blocking=True)
                in_ready = ev()
                in_ready.record(s_in)
            stream.wait_event(in_ready)
            if out_done[b] is not None:
                stream.wait_event(out_done[b])             # step i-2's outputs have been read back
            with torch.cuda.stream(stream):
                launches += compute(d_in[b], d_out[b], stream)
                comp_done[b] = ev()
                comp_done[b].record(stream)
            s_out.wait_event(comp_done[b])
            with torch.cuda.stream(s_out):
                for h, d in zip(host_out, d_out[b]):
                    h.copy_(d, non_blocking=True)
                out_done[b] = ev()
                out_done[b].record(s_out)
        if end is not None:
            end.record(s_out)
        return launches

    run(max(args.warmup, 2))
    torch.cuda.synchronize()
    gla_check()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    run(args.steps, start, end)
    torch.cuda.synchronize()
    dist.barrier()
    gla_check()
    total = dist.max(start.elapsed_time(end))
    bi = sum(x.numel() * x.element_size() for x in host_in)
    bo = sum(x.numel() * x.element_size() for x in host_out)
    return total, bi, bo


_COPY_STREAMS = {}
E2E_OVERLAP = ("inputs copied in on their own stream while the previous step computes, outputs "
               "read back on a third stream while the next one computes (device buffers doubled)")


def copy_ceiling(args, dist, device, stream, host_in, host_out, units_per_step, unit, e2e_value):
    """The host-link bound of an e2e leg: the same harness and the same pinned
    host buffers (one copy per tensor, in and out every step), with no kernel
    in between. Returns the metric this allows and e2e's fraction of it."""
    total, bi, bo = e2e_pipelined(args, dist, device, stream, host_in, host_out, lambda d_in, d_out, st: 0)
    ceil = units_per_step * dist.world * args.steps / (total * 1e-3)
    return {"value": ceil, "unit": unit, "frac": e2e_value / ceil, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": total / args.steps,
            "what": "the same pipelined copies with no kernel: pinned host -> device in, device -> pinned host out"}


def e2e_fwd(args, dist, device, stream, c, ll):
    """Same metric through the public API with host buffers: every step
    copies q, k, v from pinned host memory, runs the forward, and reads o and
    hT back to pinned host memory (pipelined across steps)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    B, T = c.B, c.T
    pin = lambda x: torch.from_numpy(gen.bf16_bits(x).view(np.int16)).view(torch.bfloat16).pin_memory()
    host_in = [pin(c.q), pin(c.k), pin(c.v)]
    host_out = [torch.empty((B, T, H, DV), dtype=torch.bfloat16).pin_memory(),
                torch.empty((B, H, DK, DV), dtype=torch.float32).pin_memory()]

    def compute(d_in, d_out, st):
        q, k, v = d_in
        gla.gla_chunk_fwd(q, k, v, ll, None, c.scale, CHUNK, o=d_out[0], hT=d_out[1], stream=st)
        return gla.gla_last_launch_count()

    total, bi, bo = e2e_pipelined(args, dist, device, stream, host_in, host_out, compute)
    value = B * T * dist.world * args.steps / (total * 1e-3)
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "overlap": E2E_OVERLAP,
            "copy_ceiling": copy_ceiling(args, dist, device, stream, host_in, host_out, B * T, "tokens/s", value)}


def bench_fwd_bwd(args, dist, device, stream, peaks, sampler):
    """Training forward + backward (B=16, h0 ~ N(0, 0.02), dh0 written), and
    the backward alone on the same buffers (its own CUDA-event time)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    B, T = args.batch or 16, 2048
    c = gen.train_fwd_bwd(seed=2, B=B, T=T)
    q, k, v, do = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v, c.do))
    ll = torch.from_numpy(c.log_lambda).to(device)
    h0 = torch.from_numpy(c.h0).to(device)
    o = torch.empty((B, T, H, DV), dtype=torch.bfloat16, device=device)
    hT = torch.empty((B, H, DK, DV), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dh0 = torch.empty_like(h0)
    wsf = torch.empty(max(gla.gla_chunk_fwd_workspace_size(B, T, H, DK, DV, CHUNK), 16), dtype=torch.uint8, device=device)
    wsb = torch.empty(max(gla.gla_chunk_bwd_workspace_size(B, T, H, DK, DV, CHUNK), 16), dtype=torch.uint8, device=device)

    def bwd():
        gla.gla_chunk_bwd(q, k, v, ll, do, h0, None, c.scale, CHUNK, dq=dq, dk=dk, dv=dv, dh0=dh0,
                          workspace=wsb, stream=stream)
        return gla.gla_last_launch_count()

    def step():
        gla.gla_chunk_fwd(q, k, v, ll, h0, c.scale, CHUNK, o=o, hT=hT, workspace=wsf, stream=stream)
        return gla.gla_last_launch_count() + bwd()

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    fb, ff, _ = fwd_work(B, T, True, True)
    bb, bf, b_issued = bwd_work(B, T, True, False, True)
    avg_ms = statistics.mean(per)
    ach = (fb + bb) / (avg_ms * 1e-3) / 1e9
    ach_tf = (ff + bf) / (avg_ms * 1e-3) / 1e12
    l2 = f"inputs larger than L2 ({(fb + bb) / 1e6:.0f} MB per step), no flush"
    res = {
        "value": B * T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps,
        "config": {"workload": c.name, "B": B, "T": T, "H": H, "chunk": CHUNK, "h0": "N(0,0.02)", "dhT": "none",
                   "l2": l2},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes_per_step": fb + bb, "avg_step_ms": avg_ms, "peak_source": peaks["source"],
                     "bytes_per_head_token": "fwd 1,152 + bwd 1,920, plus states"},
        "tensor": {"achieved": ach_tf, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                   "frac": ach_tf / peaks["bf16_tflops_sustained"], "flops_per_step": ff + bf,
                   "flops_per_head_token": "fwd 147,456 + bwd 356,352 (full tiles)",
                   "issued_flops_per_step": ff + b_issued, "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }

    total, per, win, launches = time_steps(bwd, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    avg_ms = statistics.mean(per)
    ach = bb / (avg_ms * 1e-3) / 1e9
    ach_tf = bf / (avg_ms * 1e-3) / 1e12
    traffic, _ = committed_traffic("gla_chunk_bwd")   # dq + dk + dv launches of one B=16 call
    res["bwd"] = {
        "value": B * T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps,
        "config": {"workload": f"train_bwd_bf16_B{B}_H16_T{T}", "B": B, "T": T, "H": H, "chunk": CHUNK,
                   "h0": "N(0,0.02)", "dhT": "none", "dh0": "written",
                   "l2": f"inputs larger than L2 ({bb / 1e6:.0f} MB per call), no flush"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": traffic * B / 16 if traffic is not None else None,
                     "algorithmic_bytes_per_call": bb, "avg_call_ms": avg_ms,
                     "launches_per_call": launches // max(args.steps, 1), "peak_source": peaks["source"],
                     "note": "one call = the dq, dk and dv launches side by side on forked streams"},
        "tensor": {"achieved": ach_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                   "frac": ach_tf / peaks["bf16_tflops"], "flops_per_call": bf, "issued_flops_per_call": b_issued,
                   "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    return res


def bench_long(args, dist, device, stream, peaks, sampler):
    """Long-context prefill: B=1, H=16, T=65,536, nonzero h0, decay
    log-uniform in [0.9, 0.9999]; chunk 128 (value) and 64 (reported beside)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    T = args.long_T or 65536
    c = gen.long_prefill(seed=4, T=T, chunk=CHUNK)
    q, k, v = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v))
    ll = torch.from_numpy(c.log_lambda).to(device)
    h0 = torch.from_numpy(c.h0).to(device)
    o = torch.empty((1, T, H, DV), dtype=torch.bfloat16, device=device)
    hT = torch.empty((1, H, DK, DV), dtype=torch.float32, device=device)
    out = {}
    for C in (128, 64):
        ws = torch.empty(max(gla.gla_chunk_fwd_workspace_size(1, T, H, DK, DV, C), 16), dtype=torch.uint8,
                         device=device)

        def step():
            gla.gla_chunk_fwd(q, k, v, ll, h0, c.scale, C, o=o, hT=hT, workspace=ws, stream=stream)
            return gla.gla_last_launch_count()

        total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
        total = dist.max(total)
        bytes_, fl_full, _ = fwd_work(1, T, True, True, C=C)
        avg_ms = statistics.mean(per)
        ach = bytes_ / (avg_ms * 1e-3) / 1e9
        out[C] = {
            "value": T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
            "ms_per_step": total / args.steps,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "traffic": None,
                         "algorithmic_bytes_per_call": bytes_, "avg_call_ms": avg_ms,
                         "launches_per_call": launches // max(args.steps, 1),
                         "note": "one call = segment-state pass + scan + forward", "peak_source": peaks["source"]},
            "tensor": {"achieved": fl_full / (avg_ms * 1e-3) / 1e12, "peak": peaks["bf16_tflops"],
                       "unit": "TFLOP/s", "frac": fl_full / (avg_ms * 1e-3) / 1e12 / peaks["bf16_tflops"]},
            "gpu_launches": launches,
            "clocks": sampler.summary(*win) if sampler else None,
        }
    res = dict(out[128])
    res["config"] = {"workload": c.name, "B": 1, "T": T, "H": H, "chunk": 128, "h0": "N(0,0.1)",
                     "decay": "log-uniform [0.9, 0.9999]",
                     "l2": f"inputs larger than L2 ({fwd_work(1, T, True, True)[0] / 1e6:.0f} MB per step), no flush"}
    res["chunk64"] = out[64]
    return res


VARLEN_NSEQ, VARLEN_SLOTS = 64, 128


def varlen_case():
    """Serving prefill mix: 64 prompts, lengths log-uniform in [64, 4096]
    (seed 5), H = 16, states in a pool of 128 slots."""
    lengths = gen.serving_prefill_lengths(seed=5, nseq=VARLEN_NSEQ)
    return gen.make_varlen_case(lengths, H, seed=5, n_slots=VARLEN_SLOTS)


def bench_varlen(args, dist, device, stream, peaks, sampler):
    """Variable-length prefill into the decode state pool (gla_chunk_fwd_varlen)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    c = varlen_case()
    q, k, v = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v))
    ll = torch.from_numpy(c.log_lambda).to(device)
    cu = torch.from_numpy(c.cu_seqlens).to(device)
    slots = torch.from_numpy(c.slots).to(device)
    pool = torch.from_numpy(c.pool.astype(np.float32)).to(device)
    total = int(c.cu_seqlens[-1])
    o = torch.empty((total, H, DV), dtype=torch.bfloat16, device=device)

    def step():
        gla.gla_chunk_fwd_varlen(q, k, v, ll, cu, pool, slots, c.scale, CHUNK, o=o, stream=stream)
        return gla.gla_last_launch_count()

    tot, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    tot = dist.max(tot)
    bytes_ = total * H * (2 * DK * 2 + 2 * DV * 2) + VARLEN_NSEQ * H * STATE_BYTES * 2
    avg_ms = statistics.mean(per)
    ach = bytes_ / (avg_ms * 1e-3) / 1e9
    return {
        "value": total * dist.world * args.steps / (tot * 1e-3), "unit": "tokens/s",
        "ms_per_step": tot / args.steps,
        "config": {"workload": f"serving_prefill_varlen_bf16_N{VARLEN_NSEQ}_H{H}", "sequences": VARLEN_NSEQ,
                   "tokens": total, "lengths": "log-uniform [64, 4096], seed 5", "pool_slots": VARLEN_SLOTS,
                   "chunk": CHUNK,
                   "l2": f"inputs larger than L2 ({bytes_ / 1e6:.0f} MB per step), no flush"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes_per_launch": bytes_,
                     "avg_launch_ms": avg_ms, "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }


def bench_decode(args, dist, device, stream, peaks, sampler):
    import torch
    import linear_attention_chunk_gb300 as gla
    N, L = 1280, args.layers or 24
    g = torch.Generator(device=device)
    g.manual_seed(3)
    states = []
    for _ in range(L):
        S = torch.randn((N, H, DK, DV), generator=g, device=device, dtype=torch.float32)
        S.mul_(0.1)
        states.append(S)
    toks = []
    for layer in range(L):
        dc = gen.decode_tokens(N, H, DK, DV, seed=3 + 1000 * layer)
        toks.append(tuple(dev_tensor(x, "bf16", device) for x in (dc["q"], dc["k"], dc["v"])))
    ll = torch.from_numpy(gen.log_lambda_of(gen.decay_layer_schedule(H))).to(device)
    outs = [torch.empty((N, H, DV), dtype=torch.bfloat16, device=device) for _ in range(L)]
    scale = 1.0 / math.sqrt(DK)
    per_layer = []

    def step():
        n = 0
        for layer in range(L):
            q, k, v = toks[layer]
            gla.gla_decode_step(q, k, v, ll, states[layer], scale, o=outs[layer], stream=stream)
            n += gla.gla_last_launch_count()
        return n

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    bytes_, flops = decode_work(N)
    avg_launch_ms = statistics.mean(per) / L
    ach = bytes_ / (avg_launch_ms * 1e-3) / 1e9
    res = {
        "value": N * dist.world * args.steps / (total * 1e-3), "unit": "seq-steps/s",
        "ms_per_step": total / args.steps, "ms_per_layer_step": total / args.steps / L,
        "config": {"workload": f"serving_decode_bf16_N{N}_H16_L{L}", "N": N, "H": H, "layers": L,
                   "state": f"fp32 N(0,0.1), {L} distinct buffers, {L * N * H * STATE_BYTES / 1e9:.1f} GB",
                   "l2": f"{L} distinct 1.5 GB states per step, larger than L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": committed_traffic("gla_decode")[0],
                     "algorithmic_bytes_per_launch": bytes_, "avg_launch_ms": avg_launch_ms,
                     "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    if not args.no_e2e:
        res["e2e"] = e2e_decode(args, dist, device, stream, toks, states, ll, scale, N, L)
    del states
    return res


def bench_mixer(args, dist, device, stream, peaks, sampler):
    """The mixer epilogue (self-augmentation, Head RMSNorm, SiLU(g) gate):
    fused into the serving decode step (1,280 x 16 x 24 layer-steps), and the
    standalone kernel over the layer-forward output (8 x 2048 x 16)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    N, L = 1280, args.layers or 24
    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(3)
    states = []
    for _ in range(L):
        S = torch.randn((N, H, DK, DV), generator=gen_t, device=device, dtype=torch.float32)
        S.mul_(0.1)
        states.append(S)
    toks, gates = [], []
    for layer in range(L):
        dc = gen.decode_tokens(N, H, DK, DV, seed=3 + 1000 * layer)
        toks.append(tuple(dev_tensor(x, "bf16", device) for x in (dc["q"], dc["k"], dc["v"])))
        gates.append(torch.randn((N, H, DV), generator=gen_t, device=device).to(torch.bfloat16))
    ll = torch.from_numpy(gen.log_lambda_of(gen.decay_layer_schedule(H))).to(device)
    aug = (0.3 * torch.randn((H, DK), generator=gen_t, device=device)).contiguous()
    nw = (1.0 + 0.1 * torch.randn((H, DV), generator=gen_t, device=device)).contiguous()
    outs = [torch.empty((N, H, DV), dtype=torch.bfloat16, device=device) for _ in range(L)]
    scale = 1.0 / math.sqrt(DK)

    def step():
        n = 0
        for layer in range(L):
            q, k, v = toks[layer]
            gla.gla_decode_step_mixer(q, k, v, ll, states[layer], gates[layer], aug, nw, 1e-6, scale,
                                      z=outs[layer], stream=stream)
            n += gla.gla_last_launch_count()
        return n

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    bytes_, _ = decode_work(N)
    bytes_ += N * H * DV * 2                      # g
    avg_launch_ms = statistics.mean(per) / L
    ach = bytes_ / (avg_launch_ms * 1e-3) / 1e9
    dec = {
        "value": N * dist.world * args.steps / (total * 1e-3), "unit": "seq-steps/s",
        "ms_per_step": total / args.steps, "ms_per_layer_step": total / args.steps / L,
        "config": {"workload": f"serving_decode_mixer_bf16_N{N}_H16_L{L}", "N": N, "H": H, "layers": L,
                   "epilogue": "fused: self-augmentation, Head RMSNorm, SiLU(g)",
                   "l2": f"{L} distinct 1.5 GB states per step, larger than L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes_per_launch": bytes_,
                     "avg_launch_ms": avg_launch_ms, "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    del states, toks, gates, outs

    B, T = args.batch or 8, 2048
    rows = B * T * H
    shp = lambda d: (B, T, H, d)
    o = torch.randn(shp(DV), generator=gen_t, device=device).to(torch.bfloat16)
    v = torch.randn(shp(DV), generator=gen_t, device=device).to(torch.bfloat16)
    g = torch.randn(shp(DV), generator=gen_t, device=device).to(torch.bfloat16)
    q = torch.randn(shp(DK), generator=gen_t, device=device).to(torch.bfloat16)
    k = torch.randn(shp(DK), generator=gen_t, device=device).to(torch.bfloat16)
    z = torch.empty_like(o)

    def step2():
        gla.gla_mixer_epilogue(o, q, k, v, g, aug, nw, 1e-6, z=z, stream=stream)
        return gla.gla_last_launch_count()

    total, per, win, launches = time_steps(step2, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    bytes2 = rows * (3 * DV * 2 + 2 * DK * 2 + DV * 2)
    avg_ms = statistics.mean(per)
    ach2 = bytes2 / (avg_ms * 1e-3) / 1e9
    dec["standalone"] = {
        "value": B * T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps,
        "config": {"workload": f"mixer_epilogue_bf16_B{B}_H16_T{T}", "B": B, "T": T, "H": H,
                   "l2": f"inputs larger than L2 ({bytes2 / 1e6:.0f} MB per step), no flush"},
        "roofline": {"bound": "hbm", "achieved": ach2, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach2 / peaks["hbm_gbs"], "traffic": committed_traffic("mixer_epilogue")[0],
                     "algorithmic_bytes_per_launch": bytes2, "avg_launch_ms": avg_ms,
                     "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    del o, v, g, q, k, z

    # The layer forward with the epilogue (gla_chunk_fwd_mixer: the forward's
    # output stage writes u = o + sigmoid(q . (aug * k)) v into z, a second pass
    # normalises each row and applies the norm weight and the SiLU gate in place).
    c = gen.layer_fwd(seed=1, B=B, T=T)
    q, k, v = (dev_tensor(x, "bf16", device) for x in (c.q, c.k, c.v))
    ll = torch.from_numpy(c.log_lambda).to(device)
    g = torch.randn((B, T, H, DV), generator=gen_t, device=device).to(torch.bfloat16)
    z = torch.empty((B, T, H, DV), dtype=torch.bfloat16, device=device)
    hT = torch.empty((B, H, DK, DV), dtype=torch.float32, device=device)
    ws = torch.empty(max(gla.gla_chunk_fwd_workspace_size(B, T, H, DK, DV, CHUNK), 16), dtype=torch.uint8,
                     device=device)

    def step3():
        gla.gla_chunk_fwd_mixer(q, k, v, g, ll, None, c.scale, CHUNK, aug, nw, 1e-6, z=z, hT=hT, workspace=ws,
                                stream=stream)
        return gla.gla_last_launch_count()

    total, per, win, launches = time_steps(step3, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    # Algorithmic bytes of the call: q, k, v, g in, z out and hT. The two launches also move
    # the rows u once more (written by the forward, read back by the second pass):
    # reported beside it, not counted as work.
    bytes3 = B * T * H * (2 * DK * 2 + 3 * DV * 2) + B * H * STATE_BYTES
    bytes3_moved = bytes3 + B * T * H * (2 * DV * 2)
    avg_ms = statistics.mean(per)
    dec["fwd_mixer"] = {
        "value": B * T * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps,
        "config": {"workload": f"layer_fwd_mixer_bf16_B{B}_H16_T{T}_C{CHUNK}", "B": B, "T": T, "H": H,
                   "epilogue": "self-augmentation in the forward's output stage, then RMS norm, "
                               "norm weight and SiLU(g) in place over z (two launches)",
                   "l2": f"inputs larger than L2 ({bytes3 / 1e6:.0f} MB per step), no flush"},
        "roofline": {"bound": "hbm", "achieved": bytes3 / (avg_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": bytes3 / (avg_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": committed_traffic("mixer_fwd")[0], "algorithmic_bytes_per_call": bytes3,
                     "avg_call_ms": avg_ms,
                     "bytes_moved_by_both_launches": bytes3_moved, "peak_source": peaks["source"],
                     "note": "one call = the forward writing u = o + sigmoid(q.(aug*k)) v into z, "
                             "then z = u / rms(u) * norm_w * SiLU(g) in place"},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    return dec


def bench_conv(args, dist, device, stream, peaks, sampler):
    """The causal depthwise Conv1d (width 4) + SiLU in front of the mixer over
    the layer-forward token batch (8 x 2048 x 3072, four layers' distinct
    inputs per step), and its serving step (1,280 sequences x 24 layers,
    fp32 conv windows resident)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    D = gen.D_MODEL
    B, T, L = args.batch or 8, 2048, 4
    xs, ws, bs, wins, ys = [], [], [], [], []
    for layer in range(L):
        c = gen.make_conv_case(B, T, D, seed=40 + layer)
        xs.append(dev_tensor(c.x, "bf16", device))
        ws.append(torch.from_numpy(c.w).to(device))
        bs.append(torch.from_numpy(c.b).to(device))
        wins.append(torch.from_numpy(c.window).to(device))
        ys.append(torch.empty_like(xs[-1]))

    def step():
        n = 0
        for layer in range(L):
            gla.gla_conv1d_fwd(xs[layer], ws[layer], bs[layer], wins[layer], y=ys[layer], win_out=wins[layer],
                               stream=stream)
            n += gla.gla_last_launch_count()
        return n

    total, per, win, launches = time_steps(step, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    # x in, y out, the 3 window rows the first tokens read, the 4 rows written
    bytes_ = B * T * D * 2 * 2 + B * D * 4 * (3 + 4)
    avg_ms = statistics.mean(per) / L
    ach = bytes_ / (avg_ms * 1e-3) / 1e9
    res = {
        "value": B * T * L * dist.world * args.steps / (total * 1e-3), "unit": "tokens/s",
        "ms_per_step": total / args.steps, "ms_per_layer_step": total / args.steps / L,
        "config": {"workload": f"conv1d_k4_silu_bf16_B{B}_T{T}_D{D}_L{L}", "B": B, "T": T, "D": D, "layers": L,
                   "window": "fp32 [B,4,D] per layer, in place",
                   "l2": f"{L} distinct layer inputs per step ({L * B * T * D * 2 / 1e6:.0f} MB), larger than L2"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach / peaks["hbm_gbs"], "traffic": committed_traffic("conv_stream")[0],
                     "algorithmic_bytes_per_launch": bytes_, "avg_launch_ms": avg_ms,
                     "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    del xs, ys, wins

    N, L2 = 1280, args.layers or 24
    gen_t = torch.Generator(device=device)
    gen_t.manual_seed(44)
    wins = [torch.randn((N, 4, D), generator=gen_t, device=device) for _ in range(L2)]
    xs = [torch.randn((N, D), generator=gen_t, device=device).to(torch.bfloat16) for _ in range(L2)]
    ys = [torch.empty_like(x) for x in xs]

    def step2():
        n = 0
        for layer in range(L2):
            gla.gla_conv1d_step(xs[layer], ws[layer % L], bs[layer % L], wins[layer], y=ys[layer], stream=stream)
            n += gla.gla_last_launch_count()
        return n

    total, per, win, launches = time_steps(step2, args.steps, args.warmup, dist, stream)
    total = dist.max(total)
    bytes2 = N * D * (2 + 2 + 4 * 3 + 4 * 4)      # x, y, 3 window rows read, 4 written
    avg_ms = statistics.mean(per) / L2
    ach2 = bytes2 / (avg_ms * 1e-3) / 1e9
    res["step"] = {
        "value": N * dist.world * args.steps / (total * 1e-3), "unit": "seq-steps/s",
        "ms_per_step": total / args.steps, "ms_per_layer_step": total / args.steps / L2,
        "config": {"workload": f"conv1d_step_bf16_N{N}_D{D}_L{L2}", "N": N, "D": D, "layers": L2,
                   "l2": f"{L2} distinct {N * 4 * D * 4 / 1e6:.0f} MB windows per step, larger than L2"},
        "roofline": {"bound": "hbm", "achieved": ach2, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach2 / peaks["hbm_gbs"], "traffic": committed_traffic("conv_step")[0],
                     "algorithmic_bytes_per_launch": bytes2, "avg_launch_ms": avg_ms,
                     "peak_source": peaks["source"]},
        "gpu_launches": launches,
        "clocks": sampler.summary(*win) if sampler else None,
    }
    return res


def e2e_decode(args, dist, device, stream, toks, states, ll, scale, N, L):
    """Decode through the public API with host token buffers: per step the 24
    layers' q, k, v come from pinned host memory and the 24 outputs go back
    (pipelined across steps); the recurrent states stay resident on the
    device (the serving page)."""
    import torch
    import linear_attention_chunk_gb300 as gla
    host_in = [x.cpu().pin_memory() for t in toks for x in t]
    host_out = [torch.empty((N, H, DV), dtype=torch.bfloat16).pin_memory() for _ in range(L)]

    def compute(d_in, d_out, st):
        n = 0
        for layer in range(L):
            q, k, v = d_in[3 * layer:3 * layer + 3]
            gla.gla_decode_step(q, k, v, ll, states[layer], scale, o=d_out[layer], stream=st)
            n += gla.gla_last_launch_count()
        return n

    total, bi, bo = e2e_pipelined(args, dist, device, stream, host_in, host_out, compute)
    value = N * dist.world * args.steps / (total * 1e-3)
    return {"value": value, "unit": "seq-steps/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "overlap": E2E_OVERLAP,
            "copy_ceiling": copy_ceiling(args, dist, device, stream, host_in, host_out, N, "seq-steps/s", value)}


# ------------------------------------------------------------- CPU oracle
def oracle_fwd_sample(units, seed=1):
    """The oracle's recurrent forward over `units` (b, h) chains of the
    layer-forward workload (T=2048). Returns (seconds, tokens-equivalent, threads)."""
    import oracle
    B = max(1, math.ceil(units / H))
    c = gen.layer_fwd(seed=seed, B=B, T=2048)
    hs = min(units, H)
    q, k, v = c.q[:, :, :hs], c.k[:, :, :hs], c.v[:, :, :hs]
    ll = c.log_lambda[:hs]
    nthreads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.fwd_recurrent(q, k, v, ll, None, c.scale, nthreads=nthreads)
    dt = time.perf_counter() - t0
    head_tokens = B * hs * 2048
    return dt, head_tokens / H, nthreads, f"{B}x{hs} (b,h) chains of T=2048 (of 8x16)"


def oracle_gated_sample(units):
    """The oracle's gated recurrence over `units` (b, h) chains of the gated
    layer-forward workload (T=2048)."""
    import oracle
    B = max(1, math.ceil(units / H))
    c = gated_case(B, 2048)
    hs = min(units, H)
    sl = lambda x: x[:, :, :hs]
    nthreads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.fwd_gated(sl(c.q), sl(c.k), sl(c.v), c.extra["g"][:, :, :hs], None, c.scale, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, B * hs * 2048 / H, nthreads, f"{B}x{hs} (b,h) chains of T=2048 with per-token gates (of 8x16)"


def oracle_gated_bwd_sample(units):
    """The oracle's gated backward (O11, the gate gradient included) over
    `units` (b, h) chains of the gated training workload (T=2048)."""
    import oracle
    B = max(1, math.ceil(units / H))
    hs = min(units, H)
    c = gen.make_case(B, 2048, H, DK, DV, seed=2, normalise_k=True, h0_std=0.02, with_grad=True, chunk=CHUNK,
                      gate="gla")
    sl = lambda x: x[:, :, :hs]
    nthreads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.bwd_gated(sl(c.q), sl(c.k), sl(c.v), sl(c.extra["g"]), c.h0[:, :hs], c.scale, sl(c.do), None,
                     nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, B * hs * 2048 / H, nthreads, f"{B}x{hs} (b,h) chains of T=2048, gated backward (of 16x16)"


def oracle_bwd_sample(units, seed=2):
    import oracle
    B = max(1, math.ceil(units / H))
    c = gen.train_fwd_bwd(seed=seed, B=B, T=2048)
    hs = min(units, H)
    sl = lambda x: x[:, :, :hs]
    nthreads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.fwd_recurrent(sl(c.q), sl(c.k), sl(c.v), c.log_lambda[:hs], c.h0[:, :hs], c.scale, nthreads=nthreads)
    oracle.bwd(sl(c.q), sl(c.k), sl(c.v), c.log_lambda[:hs], c.h0[:, :hs], c.scale, sl(c.do), None,
               nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, B * hs * 2048 / H, nthreads, f"{B}x{hs} (b,h) chains of T=2048 fwd+bwd (of 16x16)"


def oracle_decode_sample(layers=1, N=640):
    import oracle
    nthreads = oracle.threads(0)
    dt = 0.0
    for layer in range(layers):
        dc = gen.decode_tokens(N, H, DK, DV, seed=3 + 1000 * layer)
        rng = np.random.default_rng(10_000 + layer)
        S = (rng.standard_normal((N, H, DK, DV), dtype=np.float32) * np.float32(0.1))
        t0 = time.perf_counter()
        oracle.decode(dc["q"], dc["k"], dc["v"], gen.log_lambda_of(gen.decay_layer_schedule(H)), S,
                      1.0 / math.sqrt(DK), nthreads=nthreads)
        dt += time.perf_counter() - t0
    # seq-steps: one token of one sequence through all 24 layers
    return dt, N * layers / 24.0, nthreads, f"{layers} of 24 layer-steps over N={N} (of 1,280) x 16 heads"


def cpu_baseline():
    dt, toks, nt, sample = oracle_fwd_sample(128)
    base = {"value": toks / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle", "sample": sample,
            "seconds": dt}
    modes = {}
    dt, toks, nt, sample = oracle_bwd_sample(128)
    modes["fwd_bwd"] = {"value": toks / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                        "sample": sample, "seconds": dt}
    dt, ss, nt, sample = oracle_decode_sample(2, 1280)
    modes["decode"] = {"value": ss / dt, "unit": "seq-steps/s", "cores": nt, "kind": "oracle",
                       "sample": sample, "seconds": dt}
    dt, toks, nt, sample = oracle_varlen_sample(8)
    modes["varlen"] = {"value": toks / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                       "sample": sample, "seconds": dt}
    dt, toks, nt, sample = oracle_conv_sample(8)
    modes["conv"] = {"value": toks / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                     "sample": sample, "seconds": dt}
    dt, toks, nt, sample = oracle_gated_sample(128)
    modes["gated"] = {"value": toks / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                      "sample": sample, "seconds": dt}
    dt, toks, nt, sample = oracle_gated_bwd_sample(64)
    modes["gated_bwd"] = {"value": toks / dt, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                          "sample": sample, "seconds": dt}
    return base, modes


def oracle_conv_sample(B):
    """The oracle's Conv1d over B of the 8 sequences of one layer input."""
    import oracle
    c = gen.make_conv_case(B, 2048, gen.D_MODEL, seed=40)
    nthreads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.conv1d(c.x, c.w, c.b, c.window, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, B * 2048, nthreads, f"{B} of 8 sequences x 2048 tokens x {gen.D_MODEL} channels, one layer"


def oracle_varlen_sample(nseq):
    """The oracle on the first nseq prompts of the serving prefill mix, all heads."""
    import oracle
    c = varlen_case()
    n = min(nseq, VARLEN_NSEQ)
    t0 = time.perf_counter()
    for i in range(n):
        a, b = int(c.cu_seqlens[i]), int(c.cu_seqlens[i + 1])
        oracle.fwd_recurrent(c.q[None, a:b], c.k[None, a:b], c.v[None, a:b], c.log_lambda,
                             c.pool[c.slots[i]][None].astype(np.float32), c.scale)
    dt = time.perf_counter() - t0
    toks = int(c.cu_seqlens[n])
    return dt, toks, os.cpu_count() or 1, f"{n} of {VARLEN_NSEQ} prompts ({toks} tokens) x {H} heads"


def run_reference(args, dist):
    """The reference arm: the double-precision oracle on the host cores."""
    if dist.rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_fwd_sample(16)
    total, toks = 0.0, 0.0
    for _ in range(args.steps):
        dt, tk, nt, sample = oracle_fwd_sample(16)
        total += dt
        toks += tk
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": headline_config(dist.world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                         "sample": f"per step: {sample}; tokens/s counts the sampled chains' tokens"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- main
def summary_line(key, res):
    """One human-readable line per mode (stderr), nested rows included."""
    def one(name, r):
        rf = r.get("roofline") or {}
        tn = r.get("tensor") or {}
        parts = [f"{name}: {r['value']:.4g} {r['unit']}", f"{r['ms_per_step']:.4f} ms/step"]
        if rf:
            parts.append(f"HBM {rf['achieved']:.0f} GB/s = {rf['frac']:.3f} of {rf['peak']:.0f}")
        if tn:
            parts.append(f"tensor {tn['achieved']:.0f} TFLOP/s = {tn['frac']:.3f} of {tn['peak']:.0f}")
        if r.get("e2e"):
            parts.append(f"e2e {r['e2e']['value']:.4g} {r['e2e']['unit']}")
        return "[bench] " + ", ".join(parts)
    lines = [one(key, res)]
    for sub in ("standalone", "fwd_mixer", "chunk64", "step", "long", "single_chain", "bwd"):
        if isinstance(res.get(sub), dict) and "value" in res[sub]:
            lines.append(one(f"{key}.{sub}", res[sub]))
            if isinstance(res[sub].get("single_chain"), dict):
                lines.append(one(f"{key}.{sub}.single_chain", res[sub]["single_chain"]))
    return "\n".join(lines)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gla", "reference"), default="gla")
    ap.add_argument("--mode", choices=("all", "fwd", "fwd_bwd", "bwd", "decode", "long", "varlen", "mixer", "conv",
                                       "gated"),
                    default="all")
    ap.add_argument("--batch", type=int, default=0, help="override B of the fwd / fwd_bwd workloads (profiling)")
    ap.add_argument("--layers", type=int, default=0, help="override the decode layer count (profiling)")
    ap.add_argument("--long-T", dest="long_T", type=int, default=0, help="override T of the long workload (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every timed step eagerly instead of replaying a captured CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 0)
    global GRAPH
    GRAPH = not args.no_graph

    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)

    import torch
    from linear_attention_chunk_gb300.build import build
    if dist.rank == 0 or not os.path.exists(os.path.join(ROOT, "linear_attention_chunk_gb300", "_lib", "libgla.so")):
        build()
    torch.cuda.set_device(dist.local_rank)
    dist.init("nccl")
    device = torch.device("cuda", dist.local_rank)
    stream = torch.cuda.Stream(device=device)
    peaks = load_peaks()
    bus = None
    try:
        props = torch.cuda.get_device_properties(device)
        bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
    except Exception:
        bus = None
    sampler = ClockSampler(bus)
    results = {}
    try:
        if args.mode in ("all", "fwd"):
            results["fwd"] = bench_fwd(args, dist, device, stream, peaks, sampler)
        if args.mode in ("all", "fwd_bwd", "bwd"):
            fb = bench_fwd_bwd(args, dist, device, stream, peaks, sampler)
            results["bwd"] = fb.pop("bwd")
            if args.mode != "bwd":
                results["fwd_bwd"] = fb
        if args.mode in ("all", "decode"):
            results["decode"] = bench_decode(args, dist, device, stream, peaks, sampler)
        if args.mode in ("all", "long"):
            results["long"] = bench_long(args, dist, device, stream, peaks, sampler)
        if args.mode in ("all", "varlen"):
            results["varlen"] = bench_varlen(args, dist, device, stream, peaks, sampler)
        if args.mode in ("all", "mixer"):
            results["mixer"] = bench_mixer(args, dist, device, stream, peaks, sampler)
        if args.mode in ("all", "conv"):
            results["conv"] = bench_conv(args, dist, device, stream, peaks, sampler)
        if args.mode in ("all", "gated"):
            results["gated"] = bench_gated(args, dist, device, stream, peaks, sampler)
    finally:
        sampler.stop()

    head_key = "fwd" if "fwd" in results else next(iter(results))
    head = results[head_key]
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the Laplace 3B mixer)",
        "config": dict(head["config"], parallelism=f"replicas x{dist.world} (independent batches)"),
        "roofline": head["roofline"],
        "tensor": head.get("tensor"),
        "e2e": head.get("e2e"),
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "modes": {k: v for k, v in results.items() if k != head_key},
        **{key: head[key] for key in ("standalone", "fwd_mixer", "chunk64", "step", "ms_per_layer_step", "long")
           if key in head},
        "peaks": peaks,
        "timing": {"events": "one CUDA event pair around the K timed steps, on the launch stream",
                   "steps": "replay of one step captured as a CUDA graph" if GRAPH else "eager launches",
                   "e2e": "eager launches through the API; every step's host copies inside the timed region, "
                          "overlapped with the neighbouring steps' kernels"},
    }
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        base, base_modes = cpu_baseline()
        line["cpu_baseline"] = base
        for k, v in base_modes.items():
            if k in line["modes"]:
                line["modes"][k]["cpu_baseline"] = v
        if "gated_bwd" in base_modes and "bwd" in line["modes"].get("gated", {}):
            line["modes"]["gated"]["bwd"]["cpu_baseline"] = base_modes["gated_bwd"]
    if dist.rank == 0:
        for key, res in results.items():
            log(summary_line(key, res))
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
