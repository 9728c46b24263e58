"""Pins of the oracle's FP8 form with incoherent processing (CMU 11-868
FlashAttention post, FA3 section, slide page 24): the E4M3 codec against
torch's float8_e4m3fn, the Hadamard matrix against scipy's, the rotation
identity (Q H)(K H)^T = d Q K^T on inputs whose quantisation is exact, and
the post's claim that the rotation lowers the quantisation error on data
with outliers.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_02_gb300 import synth


def test_decode_matches_torch_on_all_codes():
    c = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(c)
    ref = torch.tensor(c).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_encode_matches_torch_in_range_including_ties():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000) * np.exp2(rng.uniform(-12, 9, 200000))
    x = np.clip(x, -448, 448).astype(np.float32).astype(np.float64)
    finite = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (finite[:-1] + finite[1:]) / 2  # exact ties between neighbours
    x = np.concatenate([x, mids, -mids, finite, [0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -11]])
    mine = oracle.e4m3_encode(x)
    ref = torch.tensor(x).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_encode_saturates():
    assert list(oracle.e4m3_encode(np.array([448.0, 449.0, 1e6, -500.0, -448.0]))) == \
        [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


@pytest.mark.parametrize("d", [1, 2, 4, 8, 16, 32, 64, 128])
def test_hadamard_is_sylvester(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    h = oracle.hadamard(np.eye(d))
    assert np.array_equal(h, scipy_linalg.hadamard(d).astype(np.float64))
    assert np.array_equal(h @ h.T, d * np.eye(d))


def test_rotation_preserves_scores():
    rng = np.random.default_rng(1)
    x, y = rng.standard_normal((5, 64)), rng.standard_normal((7, 64))
    xh, yh = oracle.hadamard(x), oracle.hadamard(y)
    assert np.abs(xh @ yh.T - 64 * (x @ y.T)).max() < 1e-11


def grid_tensor(shape, rng, top=448.0):
    """Entries drawn from the finite E4M3 grid, with one entry = top."""
    finite = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    t = rng.choice(finite[finite <= top], size=shape) * rng.choice([-1.0, 1.0], size=shape)
    t.reshape(-1)[0] = top
    return t


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shift", [0, -5])
def test_exact_quantisation_reduces_to_exact_attention(causal, shift):
    # Q H, K H and V lie on the E4M3 grid times 2^shift with amax = 448 *
    # 2^shift, so quantisation is exact (descale 2^shift) and the FP8 form
    # must equal exact attention on Q, K, V: with the rotation the scores
    # are (Q H)(K H)^T / d = Q K^T.
    rng = np.random.default_rng(20 - shift)
    B, H, N, d = 1, 2, 40, 16
    f = 2.0 ** shift
    tq, tk = grid_tensor((B, H, N, d), rng) * f, grid_tensor((B, H, N, d), rng) * f
    v = grid_tensor((B, H, N, d), rng) * f
    q, k = oracle.hadamard(tq) / d, oracle.hadamard(tk) / d  # so that q H = tq
    for had, (qq, kk) in ((True, (q, k)), (False, (tq, tk))):
        o8, l8, q8, k8, v8, ds = oracle.attn_fwd_fp8(qq, kk, v, causal, 0.01, had)
        assert np.all(ds == np.float32(f))
        o, lse = oracle.attn_fwd(qq, kk, v, causal, 0.01)
        assert np.abs(o8 - o).max() < 1e-9 * np.abs(v).max()
        assert np.abs(l8 - lse).max() < 1e-9


def test_quantisation_round_trip_bound():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4096) * 3.0
    codes, s = oracle.quantize_e4m3(x)
    amax = np.abs(x).max()
    assert abs(s - amax / 448) <= 1e-6 * amax / 448
    back = oracle.e4m3_decode(codes) * s
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 in the normal range,
    # absolute error <= 2^-10 * s in the subnormal range.
    err = np.abs(back - x)
    assert np.all(err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-6))
    assert codes[np.argmax(np.abs(x))] & 0x7F == 0x7E


def test_scale_zero_gives_mean_of_dequantised_v():
    q, k, v = synth.draw_outliers(1, 2, 50, 32, seed=4)
    o, lse, _, _, v8, ds = oracle.attn_fwd_fp8(q, k, v, False, 0.0, True)
    vd = oracle.e4m3_decode(v8) * ds[2][:, :, None, None]
    assert np.abs(o - vd.mean(2, keepdims=True)).max() < 1e-12
    assert np.abs(lse - math.log(50)).max() < 1e-12


def test_hadamard_lowers_quantisation_error_on_outliers():
    # The post reports a 2.6x lower error on data with simulated outliers
    # (with FA3's block quantisation); with one scale per head the same
    # recipe gives about 1.8x here, so the pin asks for 1.5x.
    B, H, N, d = 1, 4, 512, 128
    q, k, v = synth.draw_outliers(B, H, N, d, seed=0)
    scale = 1 / math.sqrt(d)
    o, _ = oracle.attn_fwd(q, k, v, False, scale)
    rmse = []
    for had in (False, True):
        o8 = oracle.attn_fwd_fp8(q, k, v, False, scale, had)[0]
        rmse.append(math.sqrt(((o8 - o) ** 2).mean()))
    assert rmse[0] / rmse[1] >= 1.5, rmse
