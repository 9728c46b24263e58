"""The forward and backward passes captured into a CUDA graph and replayed.

The library keeps no host-side state between calls that a replay would
repeat wrongly: the backward's work-item counter lives in the caller's
workspace and is reset by its own prep kernel on every replay; under the
causal mask the forward's CTAs claim items from the capturing stream's
counter slot, which every launch (and so every replay) leaves at zero; the
staged O stores need no host state.  Shapes with more work items than SMs,
so the persistent paths (and the forward's staged O stores) run.
"""
import math

import pytest
import torch

from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_bwd_graph_replay_matches_eager(causal):
    B, H, N, d = 4, 16, 1024, 128
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in synth.draw(B, H, N, d, seed=31 + causal))
    scale = 1 / math.sqrt(d)
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)

    def step():
        fa.fwd(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
        fa.bwd(q, k, v, o, do, lse, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step()  # eager, on the stream the graph is captured on
    torch.cuda.current_stream(dev).wait_stream(s)
    fa.check_device_status(stream=s.cuda_stream)
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize(dev)
    fa.check_device_status()
    for name, a, b in zip(("o", "lse", "dk", "dv"), (o, lse, dk, dv), ref[:2] + ref[3:]):
        assert torch.equal(a, b), name
    # dQ is summed with atomics: equal up to the order of fp32 additions.
    assert (dq.float() - ref[2].float()).abs().max().item() < 1e-2
