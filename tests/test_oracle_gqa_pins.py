"""Pins of the oracle's general form: grouped query heads (GQA/MQA, CMU
11-868 FlashAttention post, slide page 59), N_q != N_kv with the causal mask
aligned bottom-right, and the split-KV combine of cs2680 Lecture 9 sec. 9.8.
CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def bottom_right_mask(Nq, Nkv):
    i = np.arange(Nq)[:, None]
    j = np.arange(Nkv)[None, :]
    return j <= i + (Nkv - Nq)


@pytest.mark.parametrize("Hq,Hkv,Nq,Nkv,causal", [
    (4, 1, 5, 37, False), (4, 1, 5, 37, True), (8, 2, 1, 300, True), (6, 3, 17, 17, True),
    (2, 2, 40, 9, False), (4, 2, 33, 64, True)])
def test_against_torch_fp64_sdpa_gqa(Hq, Hkv, Nq, Nkv, causal):
    B, d, scale = 2, 8, 0.3
    q, k, v = rnd((B, Hq, Nq, d), 1), rnd((B, Hkv, Nkv, d), 2), rnd((B, Hkv, Nkv, d), 3)
    o, lse = oracle.attn_fwd_gqa(q, k, v, causal, scale)
    mask = torch.tensor(bottom_right_mask(Nq, Nkv)) if causal else None
    tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale,
                                                           enable_gqa=True).numpy()
    assert np.abs(o - ref).max() < 1e-12
    # lse from the definition, written with torch (an independent routine).
    s = scale * torch.einsum("bhid,bhjd->bhij", tq, tk.repeat_interleave(Hq // Hkv, dim=1))
    if causal:
        s = s.masked_fill(~mask, float("-inf"))
    assert np.abs(lse - torch.logsumexp(s, -1).numpy()).max() < 1e-12


def test_square_case_equals_the_square_oracle_on_repeated_heads():
    B, Hq, Hkv, N, d = 1, 6, 2, 45, 4
    q, k, v = rnd((B, Hq, N, d), 4), rnd((B, Hkv, N, d), 5), rnd((B, Hkv, N, d), 6)
    kr, vr = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
    for causal in (False, True):
        o, lse = oracle.attn_fwd_gqa(q, k, v, causal, 0.7)
        o2, lse2 = oracle.attn_fwd(q, kr, vr, causal, 0.7)
        assert np.abs(o - o2).max() < 1e-13 and np.abs(lse - lse2).max() < 1e-13


@pytest.mark.parametrize("cuts", [[20], [1, 2], [7, 8, 50], [33]])
def test_split_combine_identity(cuts):
    # Partial results over disjoint key ranges, merged by their lse, equal
    # the result over all keys (non-causal: each range is an ordinary
    # attention over its keys).
    B, Hq, Hkv, Nq, Nkv, d = 1, 4, 2, 3, 64, 8
    q, k, v = rnd((B, Hq, Nq, d), 7), rnd((B, Hkv, Nkv, d), 8), rnd((B, Hkv, Nkv, d), 9)
    edges = [0] + cuts + [Nkv]
    parts = [oracle.attn_fwd_gqa(q, k[:, :, a:b], v[:, :, a:b], False, 0.5)
             for a, b in zip(edges[:-1], edges[1:])]
    o_parts = np.stack([p[0] for p in parts])
    lse_parts = np.stack([p[1] for p in parts])
    o, lse = oracle.combine_splits(o_parts, lse_parts)
    o_full, lse_full = oracle.attn_fwd_gqa(q, k, v, False, 0.5)
    assert np.abs(o - o_full).max() < 1e-13 and np.abs(lse - lse_full).max() < 1e-13


def test_combine_of_two_parts_is_the_slide_12_identity():
    # With two parts, lse = ln(l1 + l2) and O = (l1/l2') O1 + (l2/l2') O2,
    # where l are the parts' denominators: the two-block formula.
    rng = np.random.default_rng(10)
    o1, o2 = rng.standard_normal((1, 5)), rng.standard_normal((1, 5))
    l1, l2 = 3.5, 0.25
    o, lse = oracle.combine_splits(np.stack([o1, o2]), np.log(np.array([[l1], [l2]])))
    assert abs(lse[0] - math.log(l1 + l2)) < 1e-15
    assert np.abs(o - (l1 / (l1 + l2)) * o1 - (l2 / (l1 + l2)) * o2).max() < 1e-15


def test_parts_without_keys_are_ignored():
    o_parts = np.stack([np.ones((2, 3)), np.full((2, 3), np.nan)])
    lse_parts = np.array([[0.3, -np.inf], [-np.inf, -np.inf]])
    o, lse = oracle.combine_splits(o_parts, lse_parts)
    assert np.allclose(o[0], 1.0) and lse[0] == 0.3
    assert np.all(o[1] == 0.0) and lse[1] == -np.inf


def test_decode_closed_forms():
    # One query row, scale 0: O is the mean of the visible values and lse is
    # ln(count); bottom-right causal with N_q = 1 sees every key.
    B, Hq, Hkv, Nkv, d = 2, 4, 1, 33, 6
    q, k, v = rnd((B, Hq, 1, d), 11), rnd((B, Hkv, Nkv, d), 12), rnd((B, Hkv, Nkv, d), 13)
    for causal in (False, True):
        o, lse = oracle.attn_fwd_gqa(q, k, v, causal, 0.0)
        assert np.abs(o - v.mean(2, keepdims=True)).max() < 1e-13
        assert np.abs(lse - math.log(Nkv)).max() < 1e-13


def test_rows_without_visible_keys():
    # N_q > N_kv with a bottom-right causal mask: the first N_q - N_kv query
    # rows see no key.
    B, H, Nq, Nkv, d = 1, 2, 10, 4, 3
    q, k, v = rnd((B, H, Nq, d), 14), rnd((B, H, Nkv, d), 15), rnd((B, H, Nkv, d), 16)
    o, lse = oracle.attn_fwd_gqa(q, k, v, True, 1.0)
    assert np.all(o[:, :, :Nq - Nkv] == 0.0) and np.all(lse[:, :, :Nq - Nkv] == -np.inf)
    assert np.all(np.isfinite(lse[:, :, Nq - Nkv:]))
    # The last N_kv rows form a square causal problem.
    o2, lse2 = oracle.attn_fwd(q[:, :, Nq - Nkv:], k, v, True, 1.0)
    assert np.abs(o[:, :, Nq - Nkv:] - o2).max() < 1e-13
