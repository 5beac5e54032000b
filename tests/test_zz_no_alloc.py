"""gla_chunk_fwd_noalloc: the forward for callers that may not allocate
device memory (for example a plugin whose host framework owns all device
memory through its own pool, or a serving loop that must not stall on
cudaMalloc). Its segmentation scratch is a fixed array inside the library
instead of a caller workspace.

The test calls it through the C ABI twice in a row, on a shape long enough
to be split into segments (so the array is really used) and with different
inputs each time (so contents left by the first call cannot leak into the
second). Each result must equal the ordinary entry point's bit for bit: the
same kernels run on the same inputs, only the scratch lives elsewhere. Each
is also checked against the double-precision oracle. This file is collected
last."""
import ctypes

import numpy as np
import pytest

import gla_gen as gen
import oracle
from gpu_util import TOL, case_to_dev, relerr, to_host

pytestmark = pytest.mark.gpu


def test_noalloc_forward_matches_workspace_forward_on_two_calls():
    import torch

    import linear_attention_chunk_gb300 as gla
    from linear_attention_chunk_gb300.build import build
    build()
    L = gla.lib()
    shapes = [(1, 8192, 4, 128, 201), (1, 5000, 2, 64, 202)]   # (B, T, H, chunk, seed)
    for B, T, H, C, seed in shapes:
        assert gla.gla_chunk_fwd_workspace_size(B, T, H, 96, 192, C) > 0   # segmented: scratch is used
        c = gen.make_case(B, T, H, 96, 192, seed=seed, dtype="bf16", lam_random=True, h0_std=0.1, chunk=C)
        d = case_to_dev(c)
        o_ws, h_ws = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], d["h0"], c.scale, C)
        o = torch.empty_like(o_ws)
        hT = torch.empty_like(h_ws)
        stream = torch.cuda.current_stream().cuda_stream
        st = L.gla_chunk_fwd_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                     d["ll"].data_ptr(), d["h0"].data_ptr(), ctypes.c_float(c.scale), B, T, H,
                                     96, 192, C, gla.GLA_BF16, o.data_ptr(), hT.data_ptr(), stream)
        assert st == gla.GLA_OK, L.gla_last_error().decode()
        assert L.gla_last_launch_count() == 3      # segment states, scan, forward
        gla.gla_check()
        assert torch.equal(o, o_ws)
        assert torch.equal(hT, h_ws)
        o_ref, h_ref = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, c.h0, c.scale)
        assert relerr(to_host(o), o_ref) <= TOL["bf16"]
        assert relerr(to_host(hT), h_ref) <= TOL["bf16"]
        assert np.isfinite(to_host(hT)).all()
