"""Host-side checks of the C ABI: the built library loads, exports every
function include/gla.h declares, and rejects bad arguments on the host with
the documented status codes before touching the GPU. No test here calls a
code path that would launch a kernel."""
import ctypes
import os
import re

import pytest

from linear_attention_chunk_gb300 import binding
from linear_attention_chunk_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gla.h")

FAKE = 0x10000   # 16-byte aligned, never dereferenced: every call below fails validation first
ODD = 0x10008    # 8-byte aligned only


@pytest.fixture(scope="module")
def L():
    build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_functions():
    assert declared_functions() == sorted(binding.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    handle = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_functions():
        assert ctypes.cast(getattr(handle, name), ctypes.c_void_p).value


def test_status_strings_and_version(L):
    assert binding.gla_status_string(0) == "GLA_OK"
    assert binding.gla_status_string(1) == "GLA_ERR_INVALID_ARG"
    assert binding.gla_status_string(4) == "GLA_ERR_TIMEOUT"
    assert binding.gla_status_string(99) == "GLA_ERR_UNKNOWN"
    assert "sm_103a" in binding.gla_version()


def fwd(L, q=FAKE, k=FAKE, v=FAKE, ll=FAKE, h0=None, B=1, T=256, H=1, dk=96, dv=192, chunk=128,
        dt=0, o=FAKE, hT=None, ws=None, wsb=0):
    return L.gla_chunk_fwd(q, k, v, ll, h0, 0.1, B, T, H, dk, dv, chunk, dt, o, hT, ws, wsb, None)


def test_fwd_rejects_bad_arguments(L):
    assert fwd(L, chunk=100) == binding.GLA_ERR_UNSUPPORTED
    assert fwd(L, chunk=256) == binding.GLA_ERR_UNSUPPORTED
    assert fwd(L, dk=64) == binding.GLA_ERR_UNSUPPORTED            # bf16 path is 96 x 192
    assert fwd(L, dt=1, dk=200) == binding.GLA_ERR_UNSUPPORTED     # fp32 mode limits
    assert fwd(L, dt=7) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, T=-1) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, dk=0) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, q=None) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, ll=None) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, o=None) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, v=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, h0=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, hT=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(L, B=1 << 20, T=1 << 20, H=16) == binding.GLA_ERR_INVALID_ARG  # too large
    assert "not 16-byte aligned" in L.gla_last_error().decode() or True


def test_fwd_error_detail_is_set(L):
    assert fwd(L, k=ODD) == binding.GLA_ERR_INVALID_ARG
    assert "k is not 16-byte aligned" in L.gla_last_error().decode()


def test_empty_batch_is_a_no_op(L):
    # B = 0 or H = 0: nothing to do, nothing launched, no device touched
    assert fwd(L, B=0, q=None, k=None, v=None, o=None) == binding.GLA_OK
    assert fwd(L, H=0, q=None, k=None, v=None, o=None) == binding.GLA_OK
    assert L.gla_decode_step(None, None, None, None, None, 1.0, 0, 16, 96, 192, 0, None, None) == binding.GLA_OK


def test_bwd_rejects_bad_arguments(L):
    def bwd(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ll=FAKE, h0=None, do=FAKE, dhT=None, B=1, T=256, H=1,
                 dk=96, dv=192, chunk=128, dt=0, dq=FAKE, dk_=FAKE, dv_=FAKE, dh0=None, ws=None, wsb=0)
        a.update(kw)
        return L.gla_chunk_bwd(a["q"], a["k"], a["v"], a["ll"], a["h0"], 0.1, a["do"], a["dhT"], a["B"],
                               a["T"], a["H"], a["dk"], a["dv"], a["chunk"], a["dt"], a["dq"], a["dk_"],
                               a["dv_"], a["dh0"], a["ws"], a["wsb"], None)
    assert bwd(chunk=32) == binding.GLA_ERR_UNSUPPORTED
    assert bwd(do=None) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dq=None) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dv_=ODD) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dhT=ODD) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dt=1, dv=300) == binding.GLA_ERR_UNSUPPORTED
    need = binding.gla_chunk_bwd_workspace_size(1, 256, 1, 96, 192, 128, 0)
    if need > 0:
        assert bwd(ws=None) == binding.GLA_ERR_WORKSPACE


def test_decode_rejects_bad_arguments(L):
    def dec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ll=FAKE, S=FAKE, N=4, H=16, dk=96, dv=192, dt=0, o=FAKE)
        a.update(kw)
        return L.gla_decode_step(a["q"], a["k"], a["v"], a["ll"], a["S"], 0.1, a["N"], a["H"], a["dk"],
                                 a["dv"], a["dt"], a["o"], None)
    assert dec(S=None) == binding.GLA_ERR_INVALID_ARG
    assert dec(S=ODD) == binding.GLA_ERR_INVALID_ARG
    assert dec(N=-3) == binding.GLA_ERR_INVALID_ARG
    assert dec(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert dec(dt=1, dk=129) == binding.GLA_ERR_UNSUPPORTED
    assert dec(dt=3) == binding.GLA_ERR_INVALID_ARG


def test_workspace_queries_are_host_only(L):
    for B, T in ((8, 2048), (1, 65536), (16, 2048), (1, 1)):
        for C in (64, 128):
            assert binding.gla_chunk_fwd_workspace_size(B, T, 16, 96, 192, C) >= 0
            assert binding.gla_chunk_bwd_workspace_size(B, T, 16, 96, 192, C) >= 0
    assert binding.gla_chunk_fwd_workspace_size(1, 100, 1, 5, 7, 64, binding.GLA_FP32) == 0
    assert binding.gla_chunk_fwd_workspace_size(1, 100, 1, 96, 192, 100) == 0   # invalid chunk


def test_varlen_rejects_bad_arguments(L):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ll=FAKE, cu=FAKE, slots=None, pool=FAKE, n_slots=8, nseq=4, T=100, H=16,
                 dk=96, dv=192, C=128, dt=0, o=FAKE)
        a.update(kw)
        return L.gla_chunk_fwd_varlen(a["q"], a["k"], a["v"], a["ll"], 0.1, a["cu"], a["slots"], a["pool"],
                                      a["n_slots"], a["nseq"], a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dt"],
                                      a["o"], None)
    assert call(dt=1) == binding.GLA_ERR_UNSUPPORTED          # bf16 only
    assert call(C=32) == binding.GLA_ERR_UNSUPPORTED
    assert call(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert call(nseq=-1) == binding.GLA_ERR_INVALID_ARG
    assert call(cu=None) == binding.GLA_ERR_INVALID_ARG
    assert call(pool=None) == binding.GLA_ERR_INVALID_ARG
    assert call(cu=ODD) == binding.GLA_ERR_INVALID_ARG
    assert call(slots=ODD) == binding.GLA_ERR_INVALID_ARG
    assert call(n_slots=3) == binding.GLA_ERR_INVALID_ARG      # no slots array: slot n for n < nseq
    assert call(o=None) == binding.GLA_ERR_INVALID_ARG
    assert call(nseq=0) == binding.GLA_OK                      # nothing to do, no device touched


def test_epilogue_entry_points_reject_bad_arguments(L):
    def epi(**kw):
        a = dict(o=FAKE, q=FAKE, k=FAKE, v=FAKE, g=FAKE, aug=None, w=None, eps=1e-6, NT=10, H=4, dk=96, dv=192, dt=0,
                 z=FAKE)
        a.update(kw)
        return L.gla_mixer_epilogue(a["o"], a["q"], a["k"], a["v"], a["g"], a["aug"], a["w"], a["eps"], a["NT"],
                                    a["H"], a["dk"], a["dv"], a["dt"], a["z"], None)
    assert epi(dt=5) == binding.GLA_ERR_INVALID_ARG
    assert epi(NT=-1) == binding.GLA_ERR_INVALID_ARG
    assert epi(dv=300) == binding.GLA_ERR_UNSUPPORTED
    assert epi(eps=-1.0) == binding.GLA_ERR_INVALID_ARG
    assert epi(g=None) == binding.GLA_ERR_INVALID_ARG
    assert epi(aug=ODD) == binding.GLA_ERR_INVALID_ARG
    assert epi(NT=0) == binding.GLA_OK

    def dec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, ll=FAKE, S=FAKE, g=FAKE, aug=None, w=None, eps=1e-6, N=4, H=16, dk=96,
                 dv=192, dt=0, z=FAKE)
        a.update(kw)
        return L.gla_decode_step_mixer(a["q"], a["k"], a["v"], a["ll"], a["S"], 0.1, a["g"], a["aug"], a["w"],
                                       a["eps"], a["N"], a["H"], a["dk"], a["dv"], a["dt"], a["z"], None)
    assert dec(g=None) == binding.GLA_ERR_INVALID_ARG
    assert dec(g=ODD) == binding.GLA_ERR_INVALID_ARG
    assert dec(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert dec(eps=-1.0) == binding.GLA_ERR_INVALID_ARG
    assert dec(N=0) == binding.GLA_OK


def test_conv_entry_points_reject_bad_arguments(L):
    def fwd(**kw):
        a = dict(x=FAKE, w=FAKE, b=None, wi=None, B=2, T=10, D=3072, dt=0, y=FAKE + 0x100, wo=FAKE)
        a.update(kw)
        return L.gla_conv1d_fwd(a["x"], a["w"], a["b"], a["wi"], a["B"], a["T"], a["D"], a["dt"], a["y"], a["wo"],
                                None)
    assert fwd(dt=7) == binding.GLA_ERR_INVALID_ARG
    assert fwd(B=-1) == binding.GLA_ERR_INVALID_ARG
    assert fwd(D=3076) == binding.GLA_ERR_UNSUPPORTED          # bf16 rows need D % 8 == 0
    assert fwd(D=0) == binding.GLA_ERR_UNSUPPORTED
    assert fwd(w=None) == binding.GLA_ERR_INVALID_ARG
    assert fwd(x=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(b=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(wi=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(y=FAKE, x=FAKE) == binding.GLA_ERR_INVALID_ARG    # y aliases x
    assert fwd(B=0) == binding.GLA_OK
    assert fwd(T=0, wo=None) == binding.GLA_OK                  # nothing to compute or copy

    def var(**kw):
        a = dict(x=FAKE, w=FAKE, b=None, cu=FAKE, slots=None, pool=FAKE, n_slots=8, nseq=4, T=100, D=3072, dt=0,
                 y=FAKE + 0x100)
        a.update(kw)
        return L.gla_conv1d_varlen(a["x"], a["w"], a["b"], a["cu"], a["slots"], a["pool"], a["n_slots"], a["nseq"],
                                   a["T"], a["D"], a["dt"], a["y"], None)
    assert var(nseq=-1) == binding.GLA_ERR_INVALID_ARG
    assert var(cu=None) == binding.GLA_ERR_INVALID_ARG
    assert var(pool=None) == binding.GLA_ERR_INVALID_ARG
    assert var(slots=ODD) == binding.GLA_ERR_INVALID_ARG
    assert var(n_slots=3) == binding.GLA_ERR_INVALID_ARG
    assert var(dt=1, D=3074) == binding.GLA_ERR_UNSUPPORTED     # fp32 rows need D % 4 == 0
    assert var(y=None) == binding.GLA_ERR_INVALID_ARG
    assert var(nseq=0) == binding.GLA_OK
    assert var(T=0) == binding.GLA_OK                           # every sequence empty: windows unchanged

    def step(**kw):
        a = dict(x=FAKE, w=FAKE, b=None, win=FAKE, N=4, D=3072, dt=0, y=FAKE + 0x100)
        a.update(kw)
        return L.gla_conv1d_step(a["x"], a["w"], a["b"], a["win"], a["N"], a["D"], a["dt"], a["y"], None)
    assert step(win=None) == binding.GLA_ERR_INVALID_ARG
    assert step(win=ODD) == binding.GLA_ERR_INVALID_ARG
    assert step(N=-2) == binding.GLA_ERR_INVALID_ARG
    assert step(D=12) == binding.GLA_ERR_UNSUPPORTED
    assert step(N=0) == binding.GLA_OK


def test_fused_forward_epilogue_rejects_bad_arguments(L):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE + 0x100, v=FAKE + 0x200, g=FAKE + 0x300, ll=FAKE, h0=None, aug=None, w=None,
                 eps=1e-6, B=2, T=256, H=16, dk=96, dv=192, C=128, dt=0, z=FAKE + 0x400, hT=None)
        a.update(kw)
        return L.gla_chunk_fwd_mixer(a["q"], a["k"], a["v"], a["g"], a["ll"], a["h0"], 0.1, a["aug"], a["w"],
                                     a["eps"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dt"], a["z"],
                                     a["hT"], None, 0, None)
    assert call(dt=1) == binding.GLA_ERR_UNSUPPORTED          # bf16 only
    assert call(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert call(C=32) == binding.GLA_ERR_UNSUPPORTED
    assert call(eps=-1.0) == binding.GLA_ERR_INVALID_ARG
    assert call(g=None) == binding.GLA_ERR_INVALID_ARG
    assert call(g=ODD) == binding.GLA_ERR_INVALID_ARG
    assert call(aug=ODD) == binding.GLA_ERR_INVALID_ARG
    assert call(z=FAKE + 0x300) == binding.GLA_ERR_INVALID_ARG   # z aliases g
    assert call(B=0) == binding.GLA_OK


def test_selftest_rejects_bad_arguments(L):
    assert L.gla_selftest_wait_timeout(0, FAKE, None) == binding.GLA_ERR_INVALID_ARG
    assert L.gla_selftest_wait_timeout(2000000, FAKE, None) == binding.GLA_ERR_INVALID_ARG
    assert L.gla_selftest_wait_timeout(1000, None, None) == binding.GLA_ERR_INVALID_ARG
    assert L.gla_selftest_wait_timeout(1000, ODD, None) == binding.GLA_ERR_INVALID_ARG


def test_gated_entry_points_reject_bad_arguments(L):
    def fwd(**kw):
        a = dict(q=FAKE, k=FAKE + 0x100, v=FAKE + 0x200, g=FAKE + 0x300, h0=None, B=2, T=256, H=16, dk=96, dv=192,
                 C=128, dt=0, o=FAKE + 0x400, hT=None)
        a.update(kw)
        return L.gla_chunk_fwd_gated(a["q"], a["k"], a["v"], a["g"], a["h0"], 0.1, a["B"], a["T"], a["H"], a["dk"],
                                     a["dv"], a["C"], a["dt"], a["o"], a["hT"], a.get("ws"), 0, None)
    assert fwd(g=None) == binding.GLA_ERR_INVALID_ARG
    assert fwd(g=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(h0=ODD) == binding.GLA_ERR_INVALID_ARG
    assert fwd(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert fwd(C=96) == binding.GLA_ERR_UNSUPPORTED
    assert fwd(dt=1, dv=300) == binding.GLA_ERR_UNSUPPORTED
    assert fwd(T=-1) == binding.GLA_ERR_INVALID_ARG
    assert fwd(B=0) == binding.GLA_OK
    assert fwd(ws=ODD) == binding.GLA_ERR_INVALID_ARG
    assert binding.gla_chunk_fwd_gated_workspace_size(1, 65536, 16, 96, 192, 128) > \
        binding.gla_chunk_fwd_workspace_size(1, 65536, 16, 96, 192, 128) > 0
    assert binding.gla_chunk_fwd_gated_workspace_size(8, 2048, 16, 96, 192, 128) == 0

    def dec(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, S=FAKE, N=4, H=16, dk=96, dv=192, dt=0, o=FAKE)
        a.update(kw)
        return L.gla_decode_step_gated(a["q"], a["k"], a["v"], a["g"], a["S"], 0.1, a["N"], a["H"], a["dk"],
                                       a["dv"], a["dt"], a["o"], None)
    assert dec(g=None) == binding.GLA_ERR_INVALID_ARG
    assert dec(g=ODD) == binding.GLA_ERR_INVALID_ARG
    assert dec(S=None) == binding.GLA_ERR_INVALID_ARG
    assert dec(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert dec(N=0) == binding.GLA_OK


def test_noalloc_reports_no_launch_when_it_fails(L):
    """A rejected gla_chunk_fwd_noalloc call launches nothing, and
    gla_last_launch_count says so (it never carries an earlier call's count)."""
    def noalloc(chunk=128, T=256, H=1):
        return L.gla_chunk_fwd_noalloc(FAKE, FAKE, FAKE, FAKE, None, 0.1, 1, T, H, 96, 192, chunk, 0, FAKE, None,
                                       None)
    assert noalloc(chunk=100) == binding.GLA_ERR_UNSUPPORTED
    assert L.gla_last_launch_count() == 0
    assert "chunk 100" in L.gla_last_error().decode()
    # A shape that is split into segments looks up the scratch array's device
    # address first; without a device that lookup fails, before any launch.
    # (Skipped where a GPU is visible: the fake pointers must never reach a kernel.)
    from conftest import gpu_available
    if not gpu_available():
        assert binding.gla_chunk_fwd_workspace_size(1, 8192, 4, 96, 192, 128) > 0
        assert noalloc(T=8192, H=4) == binding.GLA_ERR_CUDA
        assert L.gla_last_launch_count() == 0
        assert "noalloc" in L.gla_last_error().decode()


def test_gated_backward_rejects_bad_arguments(L):
    def bwd(**kw):
        a = dict(q=FAKE, k=FAKE + 0x100, v=FAKE + 0x200, g=FAKE + 0x300, h0=None, do=FAKE + 0x400, dhT=None, B=2,
                 T=256, H=16, dk=96, dv=192, C=128, dt=0, dq=FAKE + 0x500, dk_=FAKE + 0x600, dv_=FAKE + 0x700,
                 dh0=None, dg=FAKE + 0x800, ws=FAKE + 0x900, wsb=1 << 40)
        a.update(kw)
        return L.gla_chunk_bwd_gated(a["q"], a["k"], a["v"], a["g"], a["h0"], 0.1, a["do"], a["dhT"], a["B"],
                                     a["T"], a["H"], a["dk"], a["dv"], a["C"], a["dt"], a["dq"], a["dk_"],
                                     a["dv_"], a["dh0"], a["dg"], a["ws"], a["wsb"], None)
    assert bwd(g=None) == binding.GLA_ERR_INVALID_ARG
    assert bwd(g=ODD) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dg=None) == binding.GLA_ERR_INVALID_ARG
    assert bwd(do=None) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dhT=ODD) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dh0=ODD) == binding.GLA_ERR_INVALID_ARG
    assert bwd(dk=64) == binding.GLA_ERR_UNSUPPORTED
    assert bwd(C=32) == binding.GLA_ERR_UNSUPPORTED
    assert bwd(T=-1) == binding.GLA_ERR_INVALID_ARG
    assert bwd(B=0) == binding.GLA_OK
    assert bwd(ws=None) == binding.GLA_ERR_WORKSPACE
    need = binding.gla_chunk_bwd_gated_workspace_size(2, 256, 16, 96, 192, 128)
    assert need == 2 * 2 * 16 * 2 * 96 * 192 * 2 + 16       # two bf16 states per (b, h, chunk), a counter
    assert bwd(wsb=need - 16) == binding.GLA_ERR_WORKSPACE
    assert "workspace" in L.gla_last_error().decode()
    assert binding.gla_chunk_bwd_gated_workspace_size(1, 300, 2, 8, 16, 64, binding.GLA_FP32) == 2 * 2 * 5 * 8 * 16 * 4
    assert bwd(dt=1, dk=8, dv=16, C=64, T=64 * 65536, B=1, H=1) == binding.GLA_ERR_UNSUPPORTED   # 65,536 chunks
