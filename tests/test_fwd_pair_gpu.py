"""The CTA-pair forward kernel (tcgen05 cta_group::2; selected with
FA_FWD_PAIR=1 for square d = 128 shapes without a mask) against the fp64
oracle, and bit for bit against the default one-CTA kernel, whose softmax
code it shares.  The pair kernel runs in a child process, since the
library reads the switch once per process.

Tolerances as the other forward tests: O max |dO| <= 2e-2, mean <= 2e-3;
lse max |dlse| <= 1e-3.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (B, H, N, scale, seed): ragged N inside one 512-row item and across
# several, a row count that leaves a CTA of the pair without valid rows,
# negative and zero scales, and enough items for several per pair.
CASES = [
    (1, 1, 1, None, 1),
    (1, 2, 129, None, 2),
    (2, 3, 300, -0.3, 3),
    (1, 2, 640, 0.0, 4),
    (2, 2, 1000, None, 5),
    (4, 40, 1536, None, 6),
]

CHILD = r"""
import math, os, sys
sys.path.insert(0, sys.argv[1])
import torch
from io_aware_exact_02_gb300 import fa, synth
out = sys.argv[2]
cases = eval(sys.argv[3])
dev = torch.device("cuda")
for i, (B, H, N, scale, seed) in enumerate(cases):
    q, k, v, _ = synth.draw(B, H, N, 128, seed=seed, with_dout=False)
    s = 1.0 / math.sqrt(128) if scale is None else scale
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=False, scale=s)
    fa.check_device_status()
    torch.save({"o": o.cpu(), "lse": lse.cpu()}, os.path.join(out, "case%d.pt" % i))
"""


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


def test_pair_kernel_matches_oracle_and_the_one_cta_kernel(tmp_path):
    env = dict(os.environ, FA_FWD_PAIR="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(tmp_path), repr(CASES)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    dev = torch.device("cuda")
    for i, (B, H, N, scale, seed) in enumerate(CASES):
        got = torch.load(os.path.join(tmp_path, "case%d.pt" % i))
        q, k, v, _ = synth.draw(B, H, N, 128, seed=seed, with_dout=False)
        s = 1.0 / math.sqrt(128) if scale is None else scale
        o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=False, scale=s)
        fa.check_device_status()
        assert torch.equal(got["o"], o.cpu()) and torch.equal(got["lse"], lse.cpu()), (B, H, N)
        if B * H * N <= 4000:
            o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, s)
            do = np.abs(got["o"].float().numpy().astype(np.float64) - o_ref)
            dl = np.abs(got["lse"].numpy().astype(np.float64) - lse_ref)
            assert do.max() <= 2e-2 and do.mean() <= 2e-3, (B, H, N, do.max())
            assert dl.max() <= 1e-3, (B, H, N, dl.max())
