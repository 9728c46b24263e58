"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or the mathematics
fix: the two-block rescaling identity of the CMU 11-868 FlashAttention post
(slide page 12), the hand check l * e^m = sum e^x of cs2680 Lecture 9
(sec. 9.4), closed forms (constant scores, causal row 0, two keys; for the backward
pass: scale 0, causal row 0), invariants (row sums, permutation and shift
invariance; for the backward pass: sums of dV and dK, the bilinear identity
sum q . dQ = sum k . dK, the derivative in the scale), central finite
differences of the forward pass (for the backward pass), an independent
library routine
(torch's fp64 scaled_dot_product_attention and autograd), and the FLOP counts
the pages print.  All run on the CPU.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.txt")


def golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, val = line.split(None, 1)
                vals[key] = val.strip()
    return vals


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- two blocks

def _two_block_plain(s, v, split):
    """Slide page 12 of the CMU 11-868 post, no max subtraction:
    l1 = sum exp S1, O1 = A1 V1 / l1; l2 = l1 + sum exp S2,
    O2 = (l1 / l2) O1 + A2 V2 / l2."""
    s1, s2 = s[:, :split], s[:, split:]
    v1, v2 = v[:split], v[split:]
    a1, a2 = np.exp(s1), np.exp(s2)
    l1 = a1.sum(1, keepdims=True)
    o1 = a1 @ v1 / l1
    l2 = l1 + a2.sum(1, keepdims=True)
    return (l1 / l2) * o1 + a2 @ v2 / l2


def _two_block_running_max(s, v, split):
    """cs2680 Lecture 9 sec. 9.4: running max m, denominator l relative to m,
    accumulator O; the factor exp(m - m_new) corrects what was accumulated
    under the old maximum; divide by l once at the end."""
    m = np.full((s.shape[0], 1), -np.inf)
    l = np.zeros((s.shape[0], 1))
    o = np.zeros((s.shape[0], v.shape[1]))
    for lo, hi in ((0, split), (split, s.shape[1])):
        x = s[:, lo:hi]
        m_new = np.maximum(m, x.max(1, keepdims=True))
        alpha = np.exp(m - m_new)
        p = np.exp(x - m_new)
        l = alpha * l + p.sum(1, keepdims=True)
        o = alpha * o + p @ v[lo:hi]
        m = m_new
    return o / l, m[:, 0] + np.log(l[:, 0])


@pytest.mark.parametrize("seed,split", [(0, 5), (1, 1), (2, 17), (3, 31)])
def test_two_block_identity_matches_oracle(seed, split):
    N, d, scale = 32, 8, 0.7
    q, k, v = rnd((1, 1, N, d), seed), rnd((1, 1, N, d), seed + 100), rnd((1, 1, N, d), seed + 200)
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=scale)
    s = scale * (q[0, 0] @ k[0, 0].T)
    assert np.abs(_two_block_plain(s, v[0, 0], split) - o[0, 0]).max() < 1e-12
    o2, lse2 = _two_block_running_max(s, v[0, 0], split)
    assert np.abs(o2 - o[0, 0]).max() < 1e-12
    assert np.abs(lse2 - lse[0, 0]).max() < 1e-12


def test_two_block_identity_when_block_two_raises_the_max():
    # Block 2 holds a key aligned with every query, so the max grows there.
    N, d, scale = 16, 4, 1.0
    q = np.abs(rnd((1, 1, N, d), 7)) + 0.1
    k = rnd((1, 1, N, d), 8) * 0.1
    k[0, 0, 12] = 6.0
    v = rnd((1, 1, N, d), 9)
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=scale)
    s = scale * (q[0, 0] @ k[0, 0].T)
    assert (s[:, 8:].max(1) > s[:, :8].max(1) + 5).all()
    o2, lse2 = _two_block_running_max(s, v[0, 0], 8)
    assert np.abs(o2 - o[0, 0]).max() < 1e-12
    assert np.abs(lse2 - lse[0, 0]).max() < 1e-12


# ----------------------------------------------------- l * e^m = sum exp(x)

def test_hand_check_178_6():
    g = golden()
    scores = [float(x) for x in g["hand_check_scores_reconstructed"].split(",")]
    # Every query row is 1, so with scale 1 each row's scores are exactly the
    # reconstructed {1, 2, 3, 5}.
    k = np.array(scores).reshape(1, 1, -1, 1)
    N = k.shape[2]
    qN = np.ones((1, 1, N, 1))
    v = np.zeros((1, 1, N, 1))
    _, lse = oracle.attn_fwd(qN, k, v, causal=False, scale=1.0)
    m = max(scores)
    ell = sum(math.exp(x - m) for x in scores)
    assert abs(math.exp(lse[0, 0, 0]) - ell * math.exp(m)) < 1e-9
    assert round(math.exp(lse[0, 0, 0]), 1) == float(g["hand_check_sum_exp"])


def test_lse_is_log_sum_exp_of_scaled_scores():
    N, d, scale = 24, 6, 0.3
    q, k, v = rnd((2, 1, N, d), 1), rnd((2, 1, N, d), 2), rnd((2, 1, N, d), 3)
    for causal in (False, True):
        _, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
        for b in range(2):
            s = scale * (q[b, 0] @ k[b, 0].T)
            if causal:
                s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
            assert np.abs(np.exp(lse[b, 0]) - np.exp(s).sum(1)).max() < 1e-10 * np.exp(lse[b, 0]).max()


# ------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_A_sum_to_one_and_O_is_AV(causal):
    B, H, N, d = 2, 2, 20, 5
    q, k, v = rnd((B, H, N, d), 4), rnd((B, H, N, d), 5), rnd((B, H, N, d), 6)
    A = oracle.attn_probs(q, k, causal=causal, scale=0.8)
    assert np.abs(A.sum(-1) - 1.0).max() < 1e-12
    assert (A >= 0).all()
    if causal:
        assert np.all(A[..., np.triu_indices(N, 1)[0], np.triu_indices(N, 1)[1]] == 0.0)
    o, _ = oracle.attn_fwd(q, k, v, causal=causal, scale=0.8)
    assert np.abs(o - A @ v).max() < 1e-12


def test_constant_scores_give_mean_of_V():
    B, H, N, d = 1, 3, 33, 7
    q, k, v = rnd((B, H, N, d), 10), rnd((B, H, N, d), 11), rnd((B, H, N, d), 12)
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=0.0)
    assert np.abs(o - v.mean(2, keepdims=True)).max() < 1e-12
    assert np.abs(lse - math.log(N)).max() < 1e-12
    o, lse = oracle.attn_fwd(q, k, v, causal=True, scale=0.0)
    prefix = np.cumsum(v, 2) / np.arange(1, N + 1)[None, None, :, None]
    assert np.abs(o - prefix).max() < 1e-12
    assert np.abs(lse - np.log(np.arange(1, N + 1))[None, None, :]).max() < 1e-12


def test_causal_row_zero_is_V0():
    B, H, N, d = 2, 2, 9, 4
    q, k, v = rnd((B, H, N, d), 13), rnd((B, H, N, d), 14), rnd((B, H, N, d), 15)
    scale = 0.45
    o, lse = oracle.attn_fwd(q, k, v, causal=True, scale=scale)
    assert np.abs(o[:, :, 0] - v[:, :, 0]).max() < 1e-15
    assert np.abs(lse[:, :, 0] - scale * (q[:, :, 0] * k[:, :, 0]).sum(-1)).max() < 1e-12


def test_two_keys_closed_form():
    # d = 1, N = 2: the softmax of two scores is a logistic function.
    q = np.array([0.7, -1.3]).reshape(1, 1, 2, 1)
    k = np.array([1.5, -0.4]).reshape(1, 1, 2, 1)
    v = np.array([2.0, -3.0]).reshape(1, 1, 2, 1)
    scale = 1.1
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=scale)
    for i in range(2):
        s0, s1 = scale * q[0, 0, i, 0] * k[0, 0, 0, 0], scale * q[0, 0, i, 0] * k[0, 0, 1, 0]
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        assert abs(o[0, 0, i, 0] - (w0 * 2.0 + (1 - w0) * -3.0)) < 1e-14
        assert abs(lse[0, 0, i] - (s0 + math.log1p(math.exp(s1 - s0)))) < 1e-14


def test_joint_permutation_of_K_V_rows():
    B, H, N, d = 1, 2, 40, 8
    q, k, v = rnd((B, H, N, d), 16), rnd((B, H, N, d), 17), rnd((B, H, N, d), 18)
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=0.35)
    perm = np.random.default_rng(3).permutation(N)
    o2, lse2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.35)
    assert np.abs(o - o2).max() < 1e-12
    assert np.abs(lse - lse2).max() < 1e-12


@pytest.mark.parametrize("u_scale", [1.0, 1000.0])
def test_key_shift(u_scale):
    # k_j += u for every j adds scale * q_i . u to every score of row i: the
    # softmax is unchanged and lse moves by that amount.  u_scale = 1000
    # makes exp of the raw scores overflow, which the max subtraction absorbs.
    B, H, N, d = 1, 1, 30, 6
    q, k, v = rnd((B, H, N, d), 19), rnd((B, H, N, d), 20), rnd((B, H, N, d), 21)
    u = rnd((d,), 22) * u_scale
    scale = 0.5
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
        o2, lse2 = oracle.attn_fwd(q, k + u, v, causal=causal, scale=scale)
        shift = scale * (q[0, 0] @ u)
        assert np.all(np.isfinite(o2))
        assert np.abs(o - o2).max() < 1e-9
        assert np.abs(lse2[0, 0] - lse[0, 0] - shift).max() < 1e-9 * max(1.0, np.abs(shift).max())


def test_sampled_rows_match_full_forward():
    B, H, N, d = 2, 2, 50, 8
    q, k, v = rnd((B, H, N, d), 23), rnd((B, H, N, d), 24), rnd((B, H, N, d), 25)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=0.3)
        heads = np.array([0, 3, 1, 2, 3])
        rows = np.array([0, 49, 17, 1, 25])
        os_, ls_ = oracle.attn_fwd_rows(q, k, v, causal, 0.3, heads, rows)
        of = o.reshape(B * H, N, d)
        lf = lse.reshape(B * H, N)
        assert np.array_equal(os_, of[heads, rows])
        assert np.array_equal(ls_, lf[heads, rows])


# ------------------------------------------------ independent library routine

@pytest.mark.parametrize("causal", [False, True])
def test_against_torch_fp64_sdpa_and_autograd(causal):
    B, H, N, d = 2, 2, 37, 16
    q, k, v, do = (rnd((B, H, N, d), s) for s in (26, 27, 28, 29))
    scale = 0.25
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    to.backward(torch.tensor(do))
    o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
    assert np.abs(o - to.detach().numpy()).max() < 1e-12
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale)
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.abs(mine - ref.numpy()).max() < 1e-11


# ------------------------------------------------------ finite differences

@pytest.mark.parametrize("causal", [False, True])
def test_backward_by_central_differences(causal):
    B, H, N, d = 1, 1, 7, 3
    q, k, v, do = (rnd((B, H, N, d), s) for s in (30, 31, 32, 33))
    scale = 0.9
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, causal=causal, scale=scale)
        return float((o * do).sum())

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        rel = np.abs(num - grad).max() / max(np.abs(grad).max(), 1e-30)
        assert rel < 1e-6, (which, rel)


def test_backward_of_dV_is_A_transpose_dO():
    B, H, N, d = 1, 2, 11, 4
    q, k, v, do = (rnd((B, H, N, d), s) for s in (34, 35, 36, 37))
    for causal in (False, True):
        A = oracle.attn_probs(q, k, causal=causal, scale=0.6)
        _, _, dv = oracle.attn_bwd(q, k, v, do, causal=causal, scale=0.6)
        assert np.abs(dv - np.swapaxes(A, -1, -2) @ do).max() < 1e-12


# ------------------------------------- backward: closed forms, invariants
#
# With S = scale Q K^T (masked), P = softmax(S), O = P V and L = sum(dO * O):
# dV = P^T dO, dS = P o (dO V^T - D) with D_i = dO_i . O_i, dQ = scale dS K,
# dK = scale dS^T Q.  Each row of P sums to 1 and each row of dS sums to 0;
# the facts below follow from those two and from S being bilinear in Q, K.

def bwd_math_failures(lib=None):
    """Names of the backward's mathematical pins that the oracle (or the
    library ``lib``) fails; empty when it passes them all."""
    failed = []
    B, H, N, d = 1, 2, 9, 3
    q, k, v, do = (rnd((B, H, N, d), s) for s in (40, 41, 42, 43))
    scale = 0.8
    for causal in (False, True):
        tag = "_causal" if causal else ""
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale, lib=lib)
        # Rows of P sum to 1: sum_j dV_j = sum_i dO_i.
        if np.abs(dv.sum(2) - do.sum(2)).max() > 1e-12:
            failed.append("dv_sum" + tag)
        # Rows of dS sum to 0: sum_j dK_j = scale sum_i (sum_j dS_ij) q_i = 0.
        if np.abs(dk.sum(2)).max() > 1e-12:
            failed.append("dk_sum" + tag)
        # Bilinearity: sum_i q_i . dQ_i = sum_j k_j . dK_j (= sum_ij dS_ij S_ij).
        lhs, rhs = (q * dq).sum((2, 3)), (k * dk).sum((2, 3))
        if np.abs(lhs - rhs).max() > 1e-12:
            failed.append("qdq_kdk" + tag)
        # dL/dscale = sum_ij dS_ij S_ij / scale = sum_i q_i . dQ_i / scale,
        # against central differences of the forward pass in the scale.
        h = 1e-6
        lp = (oracle.attn_fwd(q, k, v, causal=causal, scale=scale + h, lib=lib)[0] * do).sum()
        lm = (oracle.attn_fwd(q, k, v, causal=causal, scale=scale - h, lib=lib)[0] * do).sum()
        if abs((lp - lm) / (2 * h) - lhs.sum() / scale) > 1e-6:
            failed.append("dscale" + tag)
        # Adding one vector u to every key shifts row i's scores by
        # scale q_i . u: P, O and every gradient stay the same.
        u = rnd((1, 1, 1, d), 44, 3.0)
        dq2, dk2, dv2 = oracle.attn_bwd(q, k + u, v, do, causal=causal, scale=scale, lib=lib)
        if max(np.abs(a - b).max() for a, b in ((dq, dq2), (dk, dk2), (dv, dv2))) > 1e-11:
            failed.append("key_shift" + tag)
        # Scale 0: P is uniform over the visible keys, so dQ = dK = 0 and
        # dV_j = sum over the rows i that see key j of dO_i / (keys row i sees).
        dq0, dk0, dv0 = oracle.attn_bwd(q, k, v, do, causal=causal, scale=0.0, lib=lib)
        counts = np.arange(1, N + 1) if causal else np.full(N, N)
        w = do / counts[None, None, :, None]
        want = np.cumsum(w[:, :, ::-1], axis=2)[:, :, ::-1] if causal else np.broadcast_to(
            w.sum(2, keepdims=True), dv0.shape)
        if np.abs(dv0 - want).max() > 1e-12 or np.abs(dq0).max() > 0 or np.abs(dk0).max() > 0:
            failed.append("scale0" + tag)
        if causal:
            # Row 0 sees only key 0: P_00 = 1, O_0 = v_0, so dS_00 = 0, dQ_0 = 0.
            if np.abs(dq[:, :, 0]).max() > 1e-13:
                failed.append("causal_dq_row0")
        else:
            # Reordering the keys (K and V rows together) reorders dK and dV
            # the same way and leaves dQ alone.
            perm = np.random.default_rng(45).permutation(N)
            dq3, dk3, dv3 = oracle.attn_bwd(q, k[:, :, perm], v[:, :, perm], do, causal=False,
                                            scale=scale, lib=lib)
            if (np.abs(dq3 - dq).max() > 1e-12 or np.abs(dk3 - dk[:, :, perm]).max() > 1e-12
                    or np.abs(dv3 - dv[:, :, perm]).max() > 1e-12):
                failed.append("key_permutation")
    return failed


def blockmask_bwd_math_failures(lib=None):
    """The same identities for the block-sparse backward pass: they hold
    under any mask (a row's visible keys are its whole softmax); a query
    row that sees no key has P = 0 and adds nothing to dV."""
    failed = []
    B, H, N, d, bs = 1, 2, 12, 3, 2
    q, k, v, do = (rnd((B, H, N, d), s) for s in (50, 51, 52, 53))
    scale = 0.7
    bm = np.array([[1, 0, 1, 0, 0, 1], [0, 0, 0, 0, 0, 0], [1, 1, 0, 0, 1, 0],
                   [0, 1, 1, 1, 0, 0], [0, 0, 0, 0, 1, 1], [1, 0, 0, 1, 0, 1]], np.uint8)
    for causal in (False, True):
        tag = "_causal" if causal else ""
        dq, dk, dv = oracle.attn_bwd_blockmask(q, k, v, do, causal, scale, bm, bs, lib=lib)
        _, lse = oracle.attn_fwd_blockmask(q, k, v, causal, scale, bm, bs, lib=lib)
        sees = np.isfinite(lse)[..., None]
        if np.abs(dv.sum(2) - (do * sees).sum(2)).max() > 1e-12:
            failed.append("bs_dv_sum" + tag)
        if np.abs(dk.sum(2)).max() > 1e-12:
            failed.append("bs_dk_sum" + tag)
        if np.abs((q * dq).sum((2, 3)) - (k * dk).sum((2, 3))).max() > 1e-12:
            failed.append("bs_qdq_kdk" + tag)
        u = rnd((1, 1, 1, d), 54, 3.0)
        g2 = oracle.attn_bwd_blockmask(q, k + u, v, do, causal, scale, bm, bs, lib=lib)
        if max(np.abs(a - b).max() for a, b in zip((dq, dk, dv), g2)) > 1e-11:
            failed.append("bs_key_shift" + tag)
    return failed


def test_backward_closed_forms_and_invariants():
    assert bwd_math_failures() == []


def test_blocksparse_backward_invariants():
    assert blockmask_bwd_math_failures() == []


# -------------------------------------------------------- FLOP counts

def test_flop_counts_match_the_pages():
    g = golden()
    rec = oracle.recompute_flops(4096, 128)
    assert rec == 2 * 4096 ** 2 * 128
    assert round(rec / 1e9, 2) == float(g["recompute_flops_S4096_d128"]) / 1e9
    # Fused intensity S/2: 4 S^2 d FLOPs over Q, K, V, O read/written once
    # (4 S d b bytes, b = 2).
    for S in (4096, 32768):
        fl = oracle.fwd_flops(1, 1, S, 128, causal=False)
        assert fl / (4 * S * 128 * 2) == float(g["fused_intensity_S%d" % S])
    # Unfused: the S x S scores are written, read, written, read: 4 S^2 b.
    fl = oracle.fwd_flops(1, 1, 4096, 128, causal=False)
    assert fl / (4 * 4096 ** 2 * 2) == float(g["unfused_intensity_d128"])
    assert oracle.fwd_flops(2, 3, 100, 64, causal=True) == 0.5 * 4 * 6 * 100 ** 2 * 64
