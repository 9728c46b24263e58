"""Block-sparse forward and backward on the GPU (through the C ABI) against
the fp64 oracle's block-sparse form.

Tolerances as for the dense passes (bf16 in/out, fp32 accumulation):
  O:   max |dO| <= 2e-2, mean |dO| <= 2e-3;  lse: max |dlse| <= 1e-3,
  dQ, dK, dV: max |G - G_ref| / max |G_ref| <= 3e-2.
Rows without a visible key must come out exactly as the oracle has them:
O = 0 and lse = -inf; keys no query sees get dK = dV = 0 exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX, G_REL = 2e-2, 2e-3, 1e-3, 3e-2


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


def dev(*ts):
    return tuple(t.to("cuda") for t in ts)


def run(q, k, v, do, mask, causal, scale):
    qd, kd, vd, dod = dev(q, k, v, do)
    md = mask.to("cuda")
    o, lse = fa.fwd_blocksparse(qd, kd, vd, md, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd_blocksparse(qd, kd, vd, o, dod, lse, md, causal=causal, scale=scale)
    fa.check_device_status()
    return [t.cpu() for t in (o, lse, dq, dk, dv)]


def check_fwd(o, lse, o_ref, lse_ref, what):
    o = o.float().numpy().astype(np.float64)
    lse = lse.numpy().astype(np.float64)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    assert np.all(o[empty] == 0.0), what
    assert np.isfinite(o).all(), what
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (what, err.max(), err.mean())
    if (~empty).any():
        assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= LSE_MAX, what


def unseen(mask, N, causal):
    """(rows without a visible key, keys no row sees) as boolean [N] arrays."""
    m = np.asarray(mask, dtype=bool)
    i = np.arange(N)
    vis = m[i[:, None] // 128, i[None, :] // 128]
    if causal:
        vis &= i[None, :] <= i[:, None]
    return ~vis.any(1), ~vis.any(0)


def check_bwd(grads, refs, what, mask, causal):
    N = refs[0].shape[-2]
    no_key, no_query = unseen(mask, N, causal)
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        g = g.float().numpy().astype(np.float64)
        assert np.isfinite(g).all(), (what, name)
        empty = no_key if name == "dq" else no_query
        assert np.all(g[..., empty, :] == 0.0) and np.all(r[..., empty, :] == 0.0), (what, name)
        den = np.abs(r).max()
        e = np.abs(g - r).max() / (den if den > 0 else 1.0)
        assert e <= G_REL, (what, name, e)


def masks_for(nb, seed):
    """A random mask with one empty query block and one empty key block."""
    m = synth.draw_block_mask(nb, 0.5, seed=seed, diagonal=False)
    if nb > 2:
        m[1, :] = 0
        m[:, nb - 2] = 0
    return m


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 640, 1000])
def test_blocksparse_matches_oracle(N, causal, d):
    B, H = 2, 2
    q, k, v, do = synth.draw(B, H, N, d, seed=3000 + N + d + causal)
    mask = masks_for(-(-N // 128), seed=N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = run(q, k, v, do, mask, causal, scale)
    what = "N=%d causal=%d d=%d" % (N, causal, d)
    o_ref, lse_ref = oracle.attn_fwd_blockmask(q, k, v, causal, scale, mask.numpy())
    check_fwd(o, lse, o_ref, lse_ref, what)
    refs = oracle.attn_bwd_blockmask(q, k, v, do, causal, scale, mask.numpy())
    check_bwd((dq, dk, dv), refs, what, mask, causal)


@pytest.mark.parametrize("density", [0.1, 0.9])
def test_blocksparse_densities_and_negative_scale(density):
    B, H, N, d = 1, 3, 1152, 128
    q, k, v, do = synth.draw(B, H, N, d, seed=41)
    mask = synth.draw_block_mask(9, density, seed=7)
    for causal in (False, True):
        o, lse, dq, dk, dv = run(q, k, v, do, mask, causal, -0.09)
        what = "density=%g causal=%d" % (density, causal)
        o_ref, lse_ref = oracle.attn_fwd_blockmask(q, k, v, causal, -0.09, mask.numpy())
        check_fwd(o, lse, o_ref, lse_ref, what)
        check_bwd((dq, dk, dv), oracle.attn_bwd_blockmask(q, k, v, do, causal, -0.09,
                                                          mask.numpy()), what, mask, causal)


def test_causal_upper_blocks_only_leave_rows_without_keys():
    # Under the causal mask a query block whose active blocks all lie above
    # the diagonal sees no key.
    B, H, N, d = 1, 2, 512, 64
    q, k, v, do = synth.draw(B, H, N, d, seed=12)
    mask = torch.zeros((4, 4), dtype=torch.uint8)
    mask[0, 2] = mask[0, 3] = 1  # query block 0: above the diagonal only
    mask[2, 0] = mask[2, 2] = 1
    mask[3, 1] = 1
    o, lse, dq, dk, dv = run(q, k, v, do, mask, True, 0.125)
    assert torch.all(torch.isneginf(lse[:, :, :128])) and torch.all(o[:, :, :256] == 0)
    o_ref, lse_ref = oracle.attn_fwd_blockmask(q, k, v, True, 0.125, mask.numpy())
    check_fwd(o, lse, o_ref, lse_ref, "upper only")
    check_bwd((dq, dk, dv), oracle.attn_bwd_blockmask(q, k, v, do, True, 0.125, mask.numpy()),
              "upper only", mask, True)


@pytest.mark.parametrize("causal", [False, True])
def test_all_ones_mask_is_the_dense_pass_bitwise(causal):
    B, H, N, d = 2, 2, 777, 128
    q, k, v, do = dev(*synth.draw(B, H, N, d, seed=5))
    mask = torch.ones((7, 7), dtype=torch.uint8, device="cuda")
    o1, l1 = fa.fwd_blocksparse(q, k, v, mask, causal=causal)
    o2, l2 = fa.fwd(q, k, v, causal=causal)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = fa.bwd_blocksparse(q, k, v, o1, do, l1, mask, causal=causal)
    g2 = fa.bwd(q, k, v, o2, do, l2, causal=causal)
    fa.check_device_status()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    # dQ is summed with fp32 atomics in either pass: equal up to their order.
    assert (g1[0].float() - g2[0].float()).abs().max().item() < 1e-2


def test_all_zero_mask():
    B, H, N, d = 1, 2, 300, 64
    q, k, v, do = dev(*synth.draw(B, H, N, d, seed=6))
    mask = torch.zeros((3, 3), dtype=torch.uint8, device="cuda")
    o, lse = fa.fwd_blocksparse(q, k, v, mask)
    dq, dk, dv = fa.bwd_blocksparse(q, k, v, o, do, lse, mask)
    fa.check_device_status()
    assert torch.all(torch.isneginf(lse)) and torch.count_nonzero(o) == 0
    for g in (dq, dk, dv):
        assert torch.count_nonzero(g) == 0


def test_bool_mask_and_bad_shape():
    q, k, v = dev(*synth.draw(1, 1, 256, 64, seed=8, with_dout=False)[:3])
    m = torch.tensor([[True, False], [True, True]], device="cuda")
    o1, l1 = fa.fwd_blocksparse(q, k, v, m)
    o2, l2 = fa.fwd_blocksparse(q, k, v, m.to(torch.uint8))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    with pytest.raises(ValueError):
        fa.fwd_blocksparse(q, k, v, torch.ones((3, 3), dtype=torch.uint8, device="cuda"))


# ------------------------------------------- full-size workload, sampled heads

def test_blocksparse_full_size_sampled_head():
    w = synth.BLOCKSPARSE
    q, k, v, do = synth.draw_workload(
        synth.Workload(w.name, w.B, w.H, w.N, w.d, w.causal))
    mask = synth.draw_block_mask(w.n_blocks, w.density, seed=0)
    o, lse, dq, dk, dv = run(q, k, v, do, mask, w.causal, w.softmax_scale)
    BH = w.B * w.H
    head = BH - 1

    def sel(t):
        return t.reshape(BH, *t.shape[2:])[head][None, None]

    o_ref, lse_ref = oracle.attn_fwd_blockmask(sel(q), sel(k), sel(v), w.causal,
                                               w.softmax_scale, mask.numpy())
    check_fwd(sel(o), sel(lse), o_ref, lse_ref, w.name)
    refs = oracle.attn_bwd_blockmask(sel(q), sel(k), sel(v), sel(do), w.causal, w.softmax_scale,
                                     mask.numpy())
    check_bwd((sel(dq), sel(dk), sel(dv)), refs, w.name, mask, w.causal)


def test_blocksparse_causal_large_sampled_head():
    B, H, N, d = 2, 8, 4096, 128
    q, k, v, do = synth.draw(B, H, N, d, seed=77)
    mask = synth.draw_block_mask(32, 0.4, seed=5)
    o, lse, dq, dk, dv = run(q, k, v, do, mask, True, 1 / math.sqrt(d))
    head = 11

    def sel(t):
        return t.reshape(B * H, *t.shape[2:])[head][None, None]

    o_ref, lse_ref = oracle.attn_fwd_blockmask(sel(q), sel(k), sel(v), True, 1 / math.sqrt(d),
                                               mask.numpy())
    check_fwd(sel(o), sel(lse), o_ref, lse_ref, "causal N4096")
    refs = oracle.attn_bwd_blockmask(sel(q), sel(k), sel(v), sel(do), True, 1 / math.sqrt(d),
                                     mask.numpy())
    check_bwd((sel(dq), sel(dk), sel(dv)), refs, "causal N4096", mask, True)


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_claimed_items_d64_sampled_heads(causal):
    # d = 64 with more work items (B*H*N/256 = 512) than SMs: the forward's
    # persistent CTAs claim the items, of uneven cost under the mask, from the
    # work counter.  Two sampled heads (one of them the last) against the
    # oracle's block-sparse form, forward and backward.
    B, H, N, d = 4, 16, 2048, 64
    q, k, v, do = synth.draw(B, H, N, d, seed=91 + causal)
    mask = synth.draw_block_mask(16, 0.3, seed=13 + causal)
    o, lse, dq, dk, dv = run(q, k, v, do, mask, causal, 1 / math.sqrt(d))
    for head in (5, B * H - 1):

        def sel(t):
            return t.reshape(B * H, *t.shape[2:])[head][None, None]

        o_ref, lse_ref = oracle.attn_fwd_blockmask(sel(q), sel(k), sel(v), causal,
                                                   1 / math.sqrt(d), mask.numpy())
        check_fwd(sel(o), sel(lse), o_ref, lse_ref, "d64 head %d" % head)
        refs = oracle.attn_bwd_blockmask(sel(q), sel(k), sel(v), sel(do), causal, 1 / math.sqrt(d),
                                         mask.numpy())
        check_bwd((sel(dq), sel(dk), sel(dv)), refs, "d64 head %d" % head, mask, causal)
