"""The forward pass's two kernels for non-causal d = 128: the CTA-pair kernel
(tcgen05 cta_group::2; opt-in) and the one-CTA kernel (the default), each
forced for every size by FA_FWD_PAIR=1 / 0 in a child process (the
library reads the switch once per process).  Both must agree bit for bit
(they share the softmax code and the products' summation order), and with
the fp64 oracle on the cases small enough for it.

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
from io_aware_exact_02_gb300 import build, fa

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (B, H, N, scale, seed): ragged N inside one 512-row item and across
# several, a row count that leaves a CTA of the pair without valid rows,
# negative and zero scales, several items per pair, and sizes on both sides
# of N = 2048.
CASES = [
    (1, 1, 1, None, 1),
    (1, 2, 129, None, 2),
    (2, 3, 300, -0.3, 3),
    (1, 2, 640, 0.0, 4),
    (2, 2, 1000, None, 5),
    (4, 40, 1536, None, 6),
    (2, 8, 2049, None, 7),
    (1, 4, 4500, 0.5, 8),
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


def _run_child(mode, out):
    os.makedirs(out, exist_ok=True)
    env = dict(os.environ, FA_FWD_PAIR=mode)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, out, repr(CASES)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]


def test_pair_and_one_cta_kernels_agree_and_match_the_oracle(tmp_path):
    pair_dir, one_dir = str(tmp_path / "pair"), str(tmp_path / "one")
    _run_child("1", pair_dir)
    _run_child("0", one_dir)
    from io_aware_exact_02_gb300 import synth
    for i, (B, H, N, scale, seed) in enumerate(CASES):
        a = torch.load(os.path.join(pair_dir, "case%d.pt" % i))
        b = torch.load(os.path.join(one_dir, "case%d.pt" % i))
        assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"]), (B, H, N)
        if B * H * N <= 20000:
            q, k, v, _ = synth.draw(B, H, N, 128, seed=seed, with_dout=False)
            s = 1.0 / math.sqrt(128) if scale is None else scale
            o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, s)
            do = np.abs(a["o"].float().numpy().astype(np.float64) - o_ref)
            dl = np.abs(a["lse"].numpy().astype(np.float64) - lse_ref)
            assert do.max() <= 2e-2 and do.mean() <= 2e-3, (B, H, N, do.max())
            assert dl.max() <= 1e-3, (B, H, N, dl.max())
