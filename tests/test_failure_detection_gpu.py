"""Failure detection on the GPU without a fault: a kernel wait that runs out
(a barrier nothing completes, with a short limit) is reported through the
status word, the word is cleared by reading it, and the context stays
usable for the attention kernels afterwards.  The bounds check of the
checked build is exercised the same way: a check on an index one past its
range, which touches no memory."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


def test_timed_out_wait_is_reported_and_cleared():
    assert fa.device_status() == (fa.FA_OK, 0)
    fa.selftest_timeout(20000)  # 20 ms
    assert fa.device_status() == (fa.FA_ERR_TIMEOUT, fa.FA_SITE_SELFTEST)
    assert fa.device_status() == (fa.FA_OK, 0)
    fa.selftest_timeout(5000)
    with pytest.raises(fa.FaError) as e:
        fa.check_device_status()
    assert e.value.code == fa.FA_ERR_TIMEOUT


def test_context_usable_after_a_timeout():
    fa.selftest_timeout(10000)
    q, k, v, do = synth.draw(1, 2, 300, 128, seed=17)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=True)
    # The first error wins: the self test's record stays until it is read.
    assert fa.device_status() == (fa.FA_ERR_TIMEOUT, fa.FA_SITE_SELFTEST)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1 / math.sqrt(128))
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3
    fa.check_device_status()


def test_bounds_check_self_test():
    assert fa.device_status() == (fa.FA_OK, 0)
    fa.selftest_bounds()
    if fa.checks_enabled():
        assert fa.device_status() == (fa.FA_ERR_BOUNDS, fa.FA_SITE_SELFTEST_BOUNDS)
    assert fa.device_status() == (fa.FA_OK, 0)
