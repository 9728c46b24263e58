"""General forward pass on the GPU (fa_fwd_gqa through the C ABI) against
the fp64 oracle: grouped query heads packed into shared 128-row tiles (CMU
11-868 FlashAttention post, slide page 59), N_q != N_kv with the causal
mask aligned bottom-right, and split-KV decode merged by logsumexp (cs2680
Lecture 9 sec. 9.8).  Tolerances as for the square forward pass; rows that
see no key must give O = 0 and lse = -inf exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


def draw(B, Hq, Hkv, Nq, Nkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, Hq, Nq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, Hkv, Nkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, Hkv, Nkv, d), generator=g).to(torch.bfloat16)
    return q, k, v


def run(q, k, v, causal, scale, splits):
    dev = torch.device("cuda")
    o, lse = fa.fwd_gqa(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                        num_splits=splits)
    fa.check_device_status()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def compare(o, lse, o_ref, lse_ref, what):
    none = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), none), what
    assert np.all(o[none] == 0.0), what
    assert np.isfinite(o).all(), what
    do = np.abs(o - o_ref)
    assert do.max() <= O_MAX and do.mean() <= O_MEAN, (what, do.max(), do.mean())
    if (~none).any():
        assert np.abs(lse[~none] - lse_ref[~none]).max() <= LSE_MAX, what


CASES = [
    # B, Hq, Hkv, Nq, Nkv, d, causal, splits
    (2, 8, 2, 1, 1000, 128, False, 1),
    (2, 8, 2, 1, 1000, 128, True, 3),
    (2, 8, 2, 1, 1000, 128, False, 8),
    (1, 4, 4, 17, 300, 64, True, 2),
    (2, 16, 1, 4, 2049, 128, False, 5),
    (1, 8, 1, 40, 777, 64, True, 4),
    (1, 8, 2, 40, 40, 128, True, 1),
    (1, 2, 2, 3, 200, 64, False, 50),
    (1, 2, 1, 300, 100, 64, True, 1),
    (1, 2, 1, 300, 100, 128, True, 2),
    (3, 6, 3, 129, 4096, 128, True, 7),
    # more work items than SMs, so persistent CTAs take several each: decode
    # and short causal queries (items of equal cost), a non-causal prefill
    (8, 32, 8, 1, 4096, 128, True, 8),
    (16, 16, 4, 8, 3000, 128, True, 4),
    (8, 16, 4, 512, 512, 64, False, 1),
    # more than 32 splits: the combine reads the split lse values 32 at a
    # time and the split O rows eight at a time (ragged in both)
    (2, 8, 2, 1, 4700, 128, True, 37),
    (1, 4, 1, 2, 5000, 64, False, 64),
    # causal prefill with more items than SMs: persistent CTAs claim the
    # items (of unequal cost) from the work counter, with and without splits
    (8, 16, 4, 300, 300, 64, True, 1),
    (8, 16, 4, 260, 1000, 128, True, 2),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nkv,d,causal,splits", CASES)
def test_fwd_gqa_matches_oracle(B, Hq, Hkv, Nq, Nkv, d, causal, splits):
    q, k, v = draw(B, Hq, Hkv, Nq, Nkv, d, seed=Nq * 31 + Nkv + splits)
    scale = 1.0 / math.sqrt(d)
    o, lse = run(q, k, v, causal, scale, splits)
    o_ref, lse_ref = oracle.attn_fwd_gqa(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, (B, Hq, Hkv, Nq, Nkv, d, causal, splits))


def test_fwd_gqa_auto_splits_decode():
    B, Hq, Hkv, Nq, Nkv, d = 1, 8, 1, 1, 16384, 128
    q, k, v = draw(B, Hq, Hkv, Nq, Nkv, d, seed=3)
    splits = fa.fwd_gqa_splits(B, Hq, Hkv, Nq, Nkv, d)
    assert splits > 1
    o, lse = run(q, k, v, True, 0.1, None)
    o_ref, lse_ref = oracle.attn_fwd_gqa(q, k, v, True, 0.1)
    compare(o, lse, o_ref, lse_ref, "auto")


@pytest.mark.parametrize("B,H,N,d", [(2, 3, 700, 128), (8, 24, 1000, 128), (8, 24, 1000, 64)])
def test_square_general_path_equals_fa_fwd_bitwise(B, H, N, d):
    # The larger shapes have more items than SMs: persistent CTAs (claiming
    # the items from the work counter under the causal mask) in both paths.
    q, k, v, _ = synth.draw(B, H, N, d, seed=8, with_dout=False)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    for causal in (False, True):
        o1, l1 = fa.fwd(q, k, v, causal=causal)
        o2, l2 = fa.fwd_gqa(q, k, v, causal=causal, num_splits=1)
        fa.check_device_status()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_split_results_agree_across_split_counts():
    q, k, v = draw(1, 4, 2, 2, 3000, 128, seed=4)
    outs = [run(q, k, v, False, 0.09, s) for s in (1, 2, 6, 24)]
    for o, lse in outs[1:]:
        assert np.abs(o - outs[0][0]).max() < 1e-2
        assert np.abs(lse - outs[0][1]).max() < 1e-5


def test_fwd_gqa_errors():
    dev = torch.device("cuda")
    q = torch.zeros(1, 3, 4, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fwd_gqa(q, k, k)
    assert e.value.code == fa.FA_ERR_ARG
    q = torch.zeros(1, 4, 4, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fwd_gqa(q, k, k, num_splits=2, workspace=torch.zeros(16, dtype=torch.uint8, device=dev))
    assert e.value.code == fa.FA_ERR_WORKSPACE


# ------------------------------------------ full-size general workloads

def test_decode_workload_full_size():
    w = synth.DECODE
    q, k, v = synth.draw_gqa(w)
    o, lse = run(q, k, v, w.causal, w.softmax_scale, None)
    o_ref, lse_ref = oracle.attn_fwd_gqa(q, k, v, w.causal, w.softmax_scale)
    compare(o, lse, o_ref, lse_ref, w.name)


def test_gqa_prefill_workload_full_size_sampled():
    # The GPU runs the whole workload; the oracle checks batch 1 and the
    # query heads of two K/V heads (heads are independent).
    w = synth.GQA_PREFILL
    q, k, v = synth.draw_gqa(w)
    o, lse = run(q, k, v, w.causal, w.softmax_scale, None)
    G = w.Hq // w.Hkv
    for hk in (0, w.Hkv - 1):
        qs = q[1:2, hk * G:(hk + 1) * G]
        o_ref, lse_ref = oracle.attn_fwd_gqa(qs, k[1:2, hk:hk + 1], v[1:2, hk:hk + 1], w.causal,
                                             w.softmax_scale)
        compare(o[1:2, hk * G:(hk + 1) * G], lse[1:2, hk * G:(hk + 1) * G], o_ref, lse_ref,
                (w.name, hk))
