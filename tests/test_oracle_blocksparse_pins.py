"""Pins of the oracle's block-sparse form (the block-sparse extension of
FlashAttention named in cs2680 Lecture 9's reading guide): dense attention
with the scores of masked (query block, key block) pairs at -inf.  Checked
against torch's fp64 SDPA and autograd with the expanded element mask, the
dense and causal special cases, rows without keys, and central differences.
CPU only; small block sizes keep the cases tiny."""
import numpy as np
import pytest
import torch

import oracle


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def expand(bm, N, bs, causal):
    i = np.arange(N)
    m = bm[i[:, None] // bs, i[None, :] // bs].astype(bool)
    if causal:
        m &= i[None, :] <= i[:, None]
    return m


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_against_torch_sdpa_with_expanded_mask(causal, seed):
    B, H, N, d, bs, scale = 1, 2, 23, 5, 4, 0.6
    nb = -(-N // bs)
    bm = (np.random.default_rng(seed + 50).random((nb, nb)) < 0.55).astype(np.uint8)
    np.fill_diagonal(bm, 1)  # every row keeps at least its own block (and key)
    q, k, v, do = (rnd((B, H, N, d), seed * 10 + t) for t in range(4))
    o, lse = oracle.attn_fwd_blockmask(q, k, v, causal, scale, bm, bs)
    mask = torch.tensor(expand(bm, N, bs, causal))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    to.backward(torch.tensor(do))
    assert np.abs(o - to.detach().numpy()).max() < 1e-12
    s = scale * torch.einsum("bhid,bhjd->bhij", tq.detach(), tk.detach()).masked_fill(~mask, float("-inf"))
    assert np.abs(lse - torch.logsumexp(s, -1).numpy()).max() < 1e-12
    grads = oracle.attn_bwd_blockmask(q, k, v, do, causal, scale, bm, bs)
    for g, t in zip(grads, (tq, tk, tv)):
        assert np.abs(g - t.grad.numpy()).max() < 1e-11


def test_all_ones_is_dense_and_block_triangle_with_causal_is_causal():
    B, H, N, d, bs = 1, 2, 20, 4, 4
    nb = -(-N // bs)
    q, k, v, do = (rnd((B, H, N, d), 20 + t) for t in range(4))
    ones = np.ones((nb, nb), np.uint8)
    tri = np.tril(ones)
    for causal, bm in ((False, ones), (True, ones), (True, tri)):
        o, lse = oracle.attn_fwd_blockmask(q, k, v, causal, 0.5, bm, bs)
        o2, lse2 = oracle.attn_fwd(q, k, v, causal, 0.5)
        assert np.abs(o - o2).max() < 1e-14 and np.abs(lse - lse2).max() < 1e-14
        g = oracle.attn_bwd_blockmask(q, k, v, do, causal, 0.5, bm, bs)
        g2 = oracle.attn_bwd(q, k, v, do, causal, 0.5)
        for a, b in zip(g, g2):
            assert np.abs(a - b).max() < 1e-13


def test_rows_without_keys():
    B, H, N, d, bs = 1, 1, 12, 3, 4
    bm = np.ones((3, 3), np.uint8)
    bm[1, :] = 0  # query rows 4..7 see nothing
    q, k, v, do = (rnd((B, H, N, d), 30 + t) for t in range(4))
    o, lse = oracle.attn_fwd_blockmask(q, k, v, False, 1.0, bm, bs)
    assert np.all(o[0, 0, 4:8] == 0.0) and np.all(lse[0, 0, 4:8] == -np.inf)
    dq, dk, dv = oracle.attn_bwd_blockmask(q, k, v, do, False, 1.0, bm, bs)
    assert np.all(dq[0, 0, 4:8] == 0.0)
    # Those rows take no part in dK, dV: changing their q and dO changes nothing.
    q2, do2 = q.copy(), do.copy()
    q2[0, 0, 4:8] += 3.0
    do2[0, 0, 4:8] -= 1.0
    _, dk2, dv2 = oracle.attn_bwd_blockmask(q2, k, v, do2, False, 1.0, bm, bs)
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)


def test_backward_by_central_differences():
    B, H, N, d, bs = 1, 1, 7, 3, 2
    bm = np.array([[1, 0, 1, 0], [1, 1, 0, 0], [0, 1, 1, 1], [1, 0, 0, 1]], np.uint8)
    q, k, v, do = (rnd((B, H, N, d), 40 + t) for t in range(4))
    grads = oracle.attn_bwd_blockmask(q, k, v, do, True, 0.8, bm, bs)

    def loss(a, b, c):
        return float((oracle.attn_fwd_blockmask(a, b, c, True, 0.8, bm, bs)[0] * do).sum())

    h = 1e-6
    for which, grad in enumerate(grads):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            ap, am = [q.copy(), k.copy(), v.copy()], [q.copy(), k.copy(), v.copy()]
            ap[which][idx] += h
            am[which][idx] -= h
            num[idx] = (loss(*ap) - loss(*am)) / (2 * h)
        assert np.abs(num - grad).max() <= 1e-6 * max(np.abs(grad).max(), 1e-30)
