"""libgla driven from plain C through include/gla.h: a C program
(tests/c_abi/gla_c_check.c), compiled with gcc and linked against
libgla.so and the CUDA runtime, runs the chunked forward and one decode step
on a stream of its own; its outputs are compared with the oracle. The CPU
test checks that the header compiles as C11 on its own."""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import gla_gen as gen
import oracle
from gpu_util import TOL, relerr

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_header_compiles_as_c11():
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    r = subprocess.run(["gcc", "-fsyntax-only", "-x", "c", "-std=c11", "-Wall", "-Wextra", "-Werror",
                        os.path.join(ROOT, "include", "gla.h")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_matches_oracle():
    from linear_attention_chunk_gb300.build import LIB, build
    build()
    B, T, H = 2, 300, 4
    c = gen.make_case(B, T, H, 96, 192, seed=800, dtype="bf16", normalise_k=True, chunk=128)
    dc = gen.decode_tokens(B, H, 96, 192, seed=801)
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "gla_c_check")
        r = subprocess.run(["gcc", "-std=c11", "-O2", "-I", os.path.join(ROOT, "include"), "-I",
                            os.path.join(CUDA, "include"), os.path.join(HERE, "c_abi", "gla_c_check.c"), "-o", exe,
                            "-L", os.path.dirname(LIB), "-lgla", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                            "-Wl,-rpath," + os.path.dirname(LIB), "-Wl,-rpath," + os.path.join(CUDA, "lib64")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        for name, x in (("q", c.q), ("k", c.k), ("v", c.v), ("dq", dc["q"]), ("dk", dc["k"]), ("dv", dc["v"])):
            gen.bf16_bits(x).tofile(os.path.join(d, name + ".bin"))
        c.log_lambda.astype(np.float32).tofile(os.path.join(d, "ll.bin"))
        np.array([c.scale], np.float32).tofile(os.path.join(d, "scale.bin"))
        r = subprocess.run([exe, d, str(B), str(T), str(H)], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stdout + r.stderr
        bf = lambda name, shape: gen.bf16_to_f32(np.fromfile(os.path.join(d, name), np.uint16)).reshape(shape)
        f32 = lambda name, shape: np.fromfile(os.path.join(d, name), np.float32).reshape(shape)
        o, hT = bf("o.bin", (B, T, H, 192)), f32("hT.bin", (B, H, 96, 192))
        od, S = bf("od.bin", (B, H, 192)), f32("S.bin", (B, H, 96, 192))
    ro, rhT = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    assert relerr(o, ro) <= TOL["bf16"] and relerr(hT, rhT) <= TOL["bf16"]
    rod, rS = oracle.decode(dc["q"], dc["k"], dc["v"], c.log_lambda, hT.astype(np.float64), c.scale)
    assert relerr(od, rod) <= TOL["bf16"] and relerr(S, rS) <= 1e-5
