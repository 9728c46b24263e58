"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them.

Each mutation edits one expression of ``oracle/oracle.c`` (a dropped term, a
wrong sign or index, a transposed operand), builds the copy into a temporary
library and runs a battery of the pin checks against it: at least one check
must fail.  The unmodified source must pass the same battery.  CPU only.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "scores_drop_scale": ("        s[j] = scale * acc;\n    }\n    return len;",
                          "        s[j] = acc;\n    }\n    return len;"),
    "gqa_wrong_kv_head": ("const int64_t hk = h / G;", "const int64_t hk = h % Hkv;"),
    "gqa_causal_top_left": ("int64_t lim = i + Nkv - Nq + 1;", "int64_t lim = i + 1;"),
    "gqa_drop_scale": ("                s[j] = scale * acc;", "                s[j] = acc;"),
    "combine_unweighted": ("const double w = exp(lse_parts[t * R + r] - l);",
                           "const double w = 1.0 / (double)S;"),
    "combine_lse_no_max": ("const double l = m + log(sum);", "const double l = log(sum);"),
    "blockmask_transposed": ("return bm[(i / bs) * nb + j / bs] != 0;",
                             "return bm[(j / bs) * nb + i / bs] != 0;"),
    "blockmask_dk_drops_scale": ("        for (int64_t c = 0; c < d; ++c) dkj[c] *= scale;\n    }\n    free(lse);\n    free(D);\n    free(o);",
                                 "    }\n    free(lse);\n    free(D);\n    free(o);"),
    "lse_drop_max": ("return m + log(l);", "return log(l);"),
    "causal_off_by_one": ("return causal ? (i + 1 < N ? i + 1 : N) : N;",
                          "return causal ? (i < N ? i : N) : N;"),
    "out_uses_wrong_row": ("const double* vj = vh + j * d;\n        for (int64_t c = 0; c < d; ++c) o_row[c] += a * vj[c];",
                           "const double* vj = vh + (len - 1 - j) * d;\n        for (int64_t c = 0; c < d; ++c) o_row[c] += a * vj[c];"),
    "dS_wrong_sign": ("double ds = exp(s[j] - l) * (da[j] - Di);",
                      "double ds = exp(s[j] - l) * (da[j] + Di);"),
    "dQ_drop_scale": ("for (int64_t c = 0; c < d; ++c) dqi[c] *= scale;", ""),
    "dK_drop_scale": ("for (int64_t c = 0; c < d; ++c) dkj[c] *= scale;", ""),
    "dK_transposed_operand": ("dkj[c] += ds * qi[c];", "dkj[c] += ds * doi[c];"),
    "dV_uses_dS": ("dvj[c] += a * doi[c];", "dvj[c] += ds * doi[c];"),
    "D_drops_probability": ("Di += exp(s[j] - l) * acc;", "Di += acc;"),
    "bwd_causal_start": ("int64_t i0 = causal ? j : 0;", "int64_t i0 = causal ? j + 1 : 0;"),
    "e4m3_ties_to_odd": ("(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    "e4m3_subnormal_exponent": ("v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    "hadamard_no_sign": ("acc += odd ? -x[r * d + i] : x[r * d + i];", "acc += x[r * d + i];"),
    "fp8_rotate_q_only": ("oracle_hadamard(k, BH * N, d, kh);",
                          "for (int64_t i = 0; i < n; ++i) kh[i] = k[i];"),
    "fp8_scale_not_divided_by_d": ("hadamard ? scale / (double)d : scale", "scale"),
    "fp8_drop_descale": ("kd[i] = oracle_e4m3_decode(k8[i]) * (double)sk;",
                         "kd[i] = oracle_e4m3_decode(k8[i]);"),
    "fp8_inverse_scale": ("const float inv = 448.0f / amax;", "const float inv = amax / 448.0f;"),
}


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def battery(lib):
    """Names of the pin checks that fail for the oracle library ``lib``."""
    failed = []
    B, H, N, d = 1, 2, 9, 3
    q, k, v, do = (rnd((B, H, N, d), s) for s in (1, 2, 3, 4))
    scale = 0.8
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
        to.backward(torch.tensor(do))
        o, lse = oracle.attn_fwd(q, k, v, causal, scale, lib=lib)
        if np.abs(o - to.detach().numpy()).max() > 1e-12:
            failed.append("sdpa_O_%d" % causal)
        s = scale * np.einsum("bhid,bhjd->bhij", q, k)
        if causal:
            s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
        if np.abs(np.exp(lse) - np.exp(s).sum(-1)).max() > 1e-9:
            failed.append("lse_%d" % causal)
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale, lib=lib)
        for name, mine, ref in (("dq", dq, tq.grad), ("dk", dk, tk.grad), ("dv", dv, tv.grad)):
            if np.abs(mine - ref.numpy()).max() > 1e-11:
                failed.append("sdpa_%s_%d" % (name, causal))
        # central differences of L = sum(dO * O) along one random direction
        dirs = [rnd(q.shape, 10 + t) for t in range(3)]
        h = 1e-6
        for t, g in enumerate((dq, dk, dv)):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[t] += h * dirs[t]
            args_m[t] -= h * dirs[t]
            lp = (oracle.attn_fwd(*args_p, causal, scale, lib=lib)[0] * do).sum()
            lm = (oracle.attn_fwd(*args_m, causal, scale, lib=lib)[0] * do).sum()
            num = (lp - lm) / (2 * h)
            ana = (g * dirs[t]).sum()
            if abs(num - ana) > 1e-6 * max(1.0, abs(ana)):
                failed.append("fd_%d_%d" % (t, causal))
    o, lse = oracle.attn_fwd(q, k, v, True, scale, lib=lib)
    if np.abs(o[:, :, 0] - v[:, :, 0]).max() > 1e-15:
        failed.append("causal_row0")
    # general form: GQA + bottom-right causal against torch, and the combine
    Hq, Hkv, Nq, Nkv = 4, 2, 3, 11
    gq, gk, gv = rnd((1, Hq, Nq, d), 20), rnd((1, Hkv, Nkv, d), 21), rnd((1, Hkv, Nkv, d), 22)
    for causal in (False, True):
        i = np.arange(Nq)[:, None]
        j = np.arange(Nkv)[None, :]
        mask = torch.tensor(j <= i + Nkv - Nq) if causal else None
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(gq), torch.tensor(gk), torch.tensor(gv), attn_mask=mask, scale=scale,
            enable_gqa=True).numpy()
        go, _ = oracle.attn_fwd_gqa(gq, gk, gv, causal, scale, lib=lib)
        if np.abs(go - ref).max() > 1e-12:
            failed.append("gqa_sdpa_%d" % causal)
    parts = [oracle.attn_fwd_gqa(gq, gk[:, :, a:b], gv[:, :, a:b], False, scale, lib=lib)
             for a, b in ((0, 4), (4, 11))]
    co, clse = oracle.combine_splits(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]),
                                     lib=lib)
    fo, flse = oracle.attn_fwd_gqa(gq, gk, gv, False, scale, lib=lib)
    if np.abs(co - fo).max() > 1e-12 or np.abs(clse - flse).max() > 1e-12:
        failed.append("combine")
    # block-sparse form against torch with the expanded element mask
    bs, Nb = 2, 6
    bm = np.array([[1, 0, 1], [1, 1, 0], [0, 0, 1]], np.uint8)
    bq, bk, bv, bdo = (rnd((1, 1, Nb, d), 30 + t) for t in range(4))
    idx = np.arange(Nb)
    em = torch.tensor(bm[idx[:, None] // bs, idx[None, :] // bs].astype(bool))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (bq, bk, bv))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=em, scale=scale)
    to.backward(torch.tensor(bdo))
    bo, _ = oracle.attn_fwd_blockmask(bq, bk, bv, False, scale, bm, bs, lib=lib)
    if np.abs(bo - to.detach().numpy()).max() > 1e-12:
        failed.append("blockmask_fwd")
    bg = oracle.attn_bwd_blockmask(bq, bk, bv, bdo, False, scale, bm, bs, lib=lib)
    for name, g, t in zip("qkv", bg, (tq, tk, tv)):
        if np.abs(g - t.grad.numpy()).max() > 1e-11:
            failed.append("blockmask_d" + name)
    o, lse = oracle.attn_fwd(q, k, v, False, 0.0, lib=lib)
    if np.abs(o - v.mean(2, keepdims=True)).max() > 1e-12 or np.abs(lse - math.log(N)).max() > 1e-12:
        failed.append("scale0")
    failed += fp8_battery(lib)
    return failed


def fp8_battery(lib):
    """FP8 pins: the codec against torch, exact quantisation against exact
    attention with and without the rotation, and quantisation of a tensor
    whose scale is not 1."""
    failed = []
    c = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(c).view(torch.float8_e4m3fn).double().numpy()
    dec = oracle.e4m3_decode(c, lib=lib)
    ok = ~np.isnan(ref)
    if not np.array_equal(dec[ok], ref[ok]):
        failed.append("e4m3_decode")
    finite = ref[:0x7F]
    mids = (finite[:-1] + finite[1:]) / 2
    x = np.concatenate([mids, -mids, rnd(500, 40) * 30])
    x = x.astype(np.float32).astype(np.float64)
    tref = torch.tensor(x).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if not np.array_equal(oracle.e4m3_encode(x, lib=lib), tref):
        failed.append("e4m3_encode")
    d = 8
    if not np.array_equal(oracle.hadamard(np.eye(d), lib=lib) @ oracle.hadamard(np.eye(d), lib=lib),
                          d * np.eye(d)) or oracle.hadamard(np.eye(d), lib=lib)[1, 1] != -1:
        failed.append("hadamard")
    rng = np.random.default_rng(41)
    N8 = 12
    grid = finite[finite > 0]
    tq, tk, tv = (rng.choice(grid, size=(1, 1, N8, d)) * rng.choice([-1.0, 1.0], size=(1, 1, N8, d))
                  for _ in range(3))
    for t in (tq, tk, tv):
        t[0, 0, 0, 0] = 448.0
    f = 2.0 ** -4
    tq, tk, tv = tq * f, tk * f, tv * f
    q, k = oracle.hadamard(tq, lib=lib) / d, oracle.hadamard(tk, lib=lib) / d
    for had, (qq, kk) in ((True, (q, k)), (False, (tq, tk))):
        o8 = oracle.attn_fwd_fp8(qq, kk, tv, True, 0.3, had, lib=lib)[0]
        o, _ = oracle.attn_fwd(qq, kk, tv, True, 0.3, lib=lib)
        if np.abs(o8 - o).max() > 1e-9:
            failed.append("fp8_exact_%d" % had)
    codes, s = oracle.quantize_e4m3(tv, lib=lib)
    if s != np.float32(448.0 * f / 448.0) or not np.array_equal(
            oracle.e4m3_decode(codes, lib=lib) * s, tv):
        failed.append("quantize")
    return failed


def _build(src_text, tmp_path, name):
    c = tmp_path / (name + ".c")
    c.write_text(src_text)
    so = tmp_path / (name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", str(c), "-o", str(so), "-lm"],
                   check=True)
    return oracle.bind(str(so))


def test_unmodified_oracle_passes_battery():
    assert battery(oracle._load()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTATIONS[name]
    text = open(SRC).read()
    # The first occurrence is the mutated one (the square forms come first in
    # the file; later forms that repeat an expression have their own entries).
    assert text.count(before) >= 1, name
    lib = _build(text.replace(before, after, 1), tmp_path, name)
    assert battery(lib), "mutation %s passed every pin" % name


# The backward pass has no worked example on the pages; its closed forms and
# invariants (no library routine among them) must catch each planted
# backward mistake on their own.
BWD_MUTATIONS = ["dS_wrong_sign", "dQ_drop_scale", "dK_drop_scale", "dK_transposed_operand",
                 "dV_uses_dS", "D_drops_probability", "bwd_causal_start",
                 "blockmask_dk_drops_scale"]


@pytest.mark.parametrize("name", BWD_MUTATIONS)
def test_backward_mistake_fails_a_mathematical_pin(name, tmp_path):
    from test_oracle_pins import blockmask_bwd_math_failures, bwd_math_failures
    before, after = MUTATIONS[name]
    text = open(SRC).read()
    lib = _build(text.replace(before, after, 1), tmp_path, name)
    failed = bwd_math_failures(lib) + blockmask_bwd_math_failures(lib)
    assert failed, "mutation %s passed every mathematical backward pin" % name
