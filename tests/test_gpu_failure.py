"""Device-side failure detection on the GPU, without a fault: the bounded
mbarrier waits that every tensor-core kernel uses are made to run out (a
barrier nothing completes), and the host sees GLA_ERR_TIMEOUT from gla_check.
The abort flag ends a sibling wait early, and the context stays usable."""
import time

import numpy as np
import pytest

import gla_gen as gen
import oracle
from gpu_util import TOL, case_to_dev, relerr, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gla():
    import linear_attention_chunk_gb300 as m
    from linear_attention_chunk_gb300.build import build
    build()
    return m


def test_wait_timeout_is_reported_and_the_context_survives(gla):
    gla.gla_check()                      # start from a clear status word
    t0 = time.time()
    r = gla.gla_selftest_wait_timeout(20000)   # the first wait gives up after 20 ms
    with pytest.raises(gla.GlaError) as ei:
        gla.gla_check()
    wall = time.time() - t0
    assert ei.value.status == gla.GLA_ERR_TIMEOUT
    completed0, completed1, waited1_us = r.cpu().tolist()
    assert completed0 == 0 and completed1 == 0
    assert 15000 <= waited1_us < 500000   # left on the abort flag, long before its own 2 s limit
    assert wall < 1.5
    gla.gla_check()                      # reading the status cleared it
    c = gen.make_case(1, 200, 2, 96, 192, seed=800, lam_random=True)
    d = case_to_dev(c)
    o, hT = gla.gla_chunk_fwd(d["q"], d["k"], d["v"], d["ll"], None, c.scale, 128)
    gla.gla_check()
    ro, rh = oracle.fwd_recurrent(c.q, c.k, c.v, c.log_lambda, None, c.scale)
    assert relerr(to_host(o), ro) <= TOL["bf16"]
    assert relerr(to_host(hT), rh) <= TOL["bf16"]
