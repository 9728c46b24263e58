"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (a memory manager owns the device's memory, cudaMalloc's implicit
synchronisation is not acceptable, or no allocator is available).  It takes
its workspace from the library's fixed static scratch array.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test.  Two calls in a row, with
different shapes, are checked against fa_bwd with a caller workspace:
dQ within the backward tests' tolerance (max |dG| / max |G| <= 3e-2; dQ is
summed with atomics), dK and dV bit for bit.
"""
import ctypes
import math

import pytest
import torch

from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu

G_REL = 3e-2


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


def _case(B, H, N, d, causal, seed):
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in synth.draw(B, H, N, d, seed=seed))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    return q, k, v, o, do, lse, causal, scale


def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row():
    cases = [(2, 2, 300, 128, True, 1), (1, 3, 700, 64, False, 2)]
    for B, H, N, d, causal, seed in cases:
        q, k, v, o, do, lse, causal, scale = _case(B, H, N, d, causal, seed)
        ref = fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale)
        got = fa.bwd_noalloc(q, k, v, o, do, lse, causal=causal, scale=scale)
        fa.check_device_status()
        den = ref[0].float().abs().max().item()
        assert (got[0].float() - ref[0].float()).abs().max().item() <= G_REL * den
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])


def _largest_fitting_n(lib, d):
    """The largest N (one head) whose workspace fits the scratch array."""
    lim = fa.FA_NOALLOC_SCRATCH_BYTES
    n = 128
    while lib.fa_bwd_workspace_size(1, 1, n + 128, d) <= lim:
        n += 128
    assert lib.fa_bwd_workspace_size(1, 1, n, d) <= lim < lib.fa_bwd_workspace_size(1, 1, n + 1, d)
    return n


def test_noalloc_at_the_scratch_limit():
    """A workspace just under the limit (its last padded rows at the end of
    the array) matches fa_bwd; one row more is rejected."""
    lib = fa.load()
    d = 64
    N = _largest_fitting_n(lib, d)
    q, k, v, o, do, lse, causal, scale = _case(1, 1, N, d, False, 3)
    ref = fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale)
    got = fa.bwd_noalloc(q, k, v, o, do, lse, causal=causal, scale=scale)
    fa.check_device_status()
    den = ref[0].float().abs().max().item()
    assert (got[0].float() - ref[0].float()).abs().max().item() <= G_REL * den
    assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
    del q, k, v, o, do, lse, ref, got
    dev = torch.device("cuda")
    buf = torch.zeros(16, dtype=torch.bfloat16, device=dev)  # never touched
    p = buf.data_ptr()
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, N + 1, d, 0, ctypes.c_float(0.1),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_ERR_WORKSPACE
    # Argument errors come first, as fa_bwd reports them.
    rc = lib.fa_bwd_noalloc(p + 2, p, p, p, p, p, p, p, p, 1, 1, N + 1, d, 0, ctypes.c_float(0.1),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_ERR_ALIGN
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 1, N + 1, d, 2, ctypes.c_float(0.1),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_ERR_ARG
    assert torch.count_nonzero(buf) == 0


def test_noalloc_rejects_sizes_beyond_the_scratch():
    lib = fa.load()
    B, H, N, d = 1, 64, 8192, 128
    assert lib.fa_bwd_workspace_size(B, H, N, d) > (32 << 20)
    dev = torch.device("cuda")
    buf = torch.zeros(16, dtype=torch.bfloat16, device=dev)  # never touched
    p = buf.data_ptr()
    rc = lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0, ctypes.c_float(0.1),
                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_ERR_WORKSPACE
    assert torch.count_nonzero(buf) == 0
