"""The library's calls inside a CUDA graph: they allocate nothing and never
synchronise, so a captured step replays to the same bits as the same calls
launched eagerly (forward with segmentation, the backward with its three
launches forked onto helper streams and joined back, decode with the fused
epilogue, the Conv1d prefill and serving step)."""
import numpy as np
import pytest

import gla_gen as gen
from gpu_util import case_to_dev, f32_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gla():
    import linear_attention_chunk_gb300 as m
    from linear_attention_chunk_gb300.build import build
    build()
    return m


def test_captured_step_replays_bit_exact(gla):
    import torch
    c = gen.make_case(1, 4096, 2, 96, 192, seed=700, lam_random=True, h0_std=0.1, with_grad=True)
    d = case_to_dev(c)
    ws = torch.empty(max(gla.gla_chunk_fwd_workspace_size(1, 4096, 2, 96, 192, 128), 16), dtype=torch.uint8,
                     device="cuda")
    dc = gen.make_decode_case(16, 4, 96, 192, seed=701)
    dq, dk, dvv, dll = to_dev(dc.q, "bf16"), to_dev(dc.k, "bf16"), to_dev(dc.v, "bf16"), f32_dev(dc.log_lambda)
    g = to_dev(gen.bf16_round(np.random.default_rng(702).normal(size=(16, 4, 192))), "bf16")
    cc = gen.make_conv_case(3, 50, 3072, seed=703)
    x, w, b = to_dev(cc.x, "bf16"), f32_dev(cc.w), f32_dev(cc.b)
    x1 = to_dev(gen.make_conv_case(3, 1, 3072, seed=704).x[:, 0], "bf16")

    def buffers():
        return dict(o=torch.empty_like(d["v"]), hT=torch.empty((1, 2, 96, 192), device="cuda"),
                    dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                    dh0=torch.empty((1, 2, 96, 192), device="cuda"),
                    S=f32_dev(dc.S), win=f32_dev(cc.window), z=torch.empty((16, 4, 192), dtype=torch.bfloat16,
                                                                           device="cuda"),
                    y=torch.empty_like(x), y1=torch.empty_like(x1))

    def step(bf, s):
        gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, 128, o=bf["o"], hT=bf["hT"],
                          workspace=ws, stream=s)
        gla.gla_chunk_bwd(d["q"], d["k"], d["v"], d["ll"], d["do"], d["h0"], d["dhT"], c.scale, 128, dq=bf["dq"],
                          dk=bf["dk"], dv=bf["dv"], dh0=bf["dh0"], stream=s)
        gla.gla_decode_step_mixer(dq, dk, dvv, dll, bf["S"], g, None, None, 1e-6, dc.scale, z=bf["z"], stream=s)
        gla.gla_conv1d_fwd(x, w, b, bf["win"], y=bf["y"], win_out=bf["win"], stream=s)
        gla.gla_conv1d_step(x1, w, b, bf["win"], y=bf["y1"], stream=s)

    s = torch.cuda.Stream()
    eager = buffers()
    with torch.cuda.stream(s):
        step(eager, s)
    torch.cuda.synchronize()
    gla.gla_check()
    graphed = buffers()
    with torch.cuda.stream(s):
        step(buffers(), s)            # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(graphed, s)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        graph.replay()
    torch.cuda.synchronize()
    gla.gla_check()
    for name in eager:
        assert torch.equal(eager[name], graphed[name]), name
