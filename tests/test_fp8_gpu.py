"""FP8 forward pass with Hadamard incoherent processing on the GPU (through
the C ABI) against the oracle's FP8 form.

The quantiser writes bytes, so its codes are compared exactly where the
rounding decision is taken from the same fp32 value on both sides (no
rotation: x * (448 / amax) in fp32).  With the rotation the GPU's fp32
butterfly and the oracle's fp64 sum can round the rotated value apart by a
few fp32 ulps; a code may then be the neighbour of the oracle's, never
further.

Attention tolerance: the GPU rounds the probabilities to E4M3 (relative
error <= 2^-4) as the operand of O += P V, which the oracle does not, so
    max |O - O_oracle| <= 2^-4 * max |V_dequantised| + 2^-8 * max |O_oracle|
(the worst case with every rounding error aligned) and
    RMS |O - O_oracle| <= 2^-4 / sqrt(3) * RMS(V_dequantised),
the RMS of a relative rounding error spread evenly over +-2^-4, reached
when each row's softmax has one dominant key (diffuse rows average the
errors out far below it); lse does not see P's rounding:
    max |lse - lse_oracle| <= 1e-3 (no rotation), 2e-3 (rotation: neighbour
codes move single scores by up to 2^-4 of one product).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_02_gb300 import build, fa, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return fa.load()


def gpu_quantize(q, k, v, hadamard):
    B, H, N, d = q.shape
    dev = torch.device("cuda")
    ws = fa.fp8_quantize(q.to(dev), k.to(dev), v.to(dev), hadamard=hadamard)
    fa.check_device_status()
    off = fa.fp8_workspace_offsets(B, H, N, d)
    npad = -(-N // 128) * 128
    host = ws.cpu().numpy()
    n = B * H * N * d
    q8 = host[off[0]:off[0] + n].reshape(B, H, N, d)
    k8 = host[off[1]:off[1] + n].reshape(B, H, N, d)
    vt8 = host[off[2]:off[2] + B * H * d * npad].reshape(B, H, d, npad)
    amax = host[off[3]:off[3] + 12 * B * H].view(np.float32).reshape(3, B, H)
    return q8, k8, vt8, amax, ws


def code_steps(a, b):
    """Distance between E4M3 codes in steps along the number line."""
    def rank(c):
        c = c.astype(np.int64)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(rank(a) - rank(b))


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 300, 1000])
def test_quantiser_matches_oracle(N, hadamard):
    B, H, d = 2, 2, 128
    q, k, v = synth.draw_outliers(B, H, N, d, seed=N + hadamard)
    q8, k8, vt8, amax, _ = gpu_quantize(q, k, v, hadamard)
    _, _, oq8, ok8, ov8, ods = oracle.attn_fwd_fp8(q, k, v, False, 0.1, hadamard)
    # V is never rotated: exact codes, and the padding keys hold code 0.
    assert np.array_equal(vt8[..., :N], ov8.transpose(0, 1, 3, 2))
    assert np.all(vt8[..., N:] == 0)
    assert np.array_equal(amax[2] / np.float32(448), ods[2])
    for mine, ref, a, s in ((q8, oq8, amax[0], ods[0]), (k8, ok8, amax[1], ods[1])):
        if not hadamard:
            assert np.array_equal(mine, ref)
            assert np.array_equal(a / np.float32(448), s)
        else:
            assert np.all(np.abs(a / 448 - s) <= 1e-5 * s)
            steps = code_steps(mine, ref)
            assert steps.max() <= 1
            assert (steps == 0).mean() >= 0.99


def run_fp8(q, k, v, causal, scale, hadamard):
    dev = torch.device("cuda")
    o, lse = fa.fwd_fp8(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                        hadamard=hadamard)
    fa.check_device_status()
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check_attention(o, lse, ref, hadamard, what):
    o_ref, lse_ref, _, _, v8, ds = ref
    vd = oracle.e4m3_decode(v8) * ds[2][:, :, None, None].astype(np.float64)
    vmax, vrms = np.abs(vd).max(), math.sqrt((vd ** 2).mean())
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    assert err.max() <= 2.0 ** -4 * vmax + 2.0 ** -8 * np.abs(o_ref).max(), (what, err.max())
    assert math.sqrt((err ** 2).mean()) <= 2.0 ** -4 / math.sqrt(3) * vrms, \
        (what, math.sqrt((err ** 2).mean()))
    assert np.abs(lse - lse_ref).max() <= (2e-3 if hadamard else 1e-3), \
        (what, np.abs(lse - lse_ref).max())


@pytest.mark.parametrize("hadamard", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 256, 300, 1000])
def test_fp8_attention_matches_oracle(N, causal, hadamard):
    B, H, d = 2, 3, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=500 + N + causal, with_dout=False)
    scale = 1 / math.sqrt(d)
    o, lse = run_fp8(q, k, v, causal, scale, hadamard)
    ref = oracle.attn_fwd_fp8(q, k, v, causal, scale, hadamard)
    check_attention(o, lse, ref, hadamard, "N=%d causal=%d had=%d" % (N, causal, hadamard))


@pytest.mark.parametrize("scale", [0.0, -0.05, 0.3])
def test_fp8_other_scales(scale):
    q, k, v = synth.draw_outliers(1, 2, 333, 128, seed=9)
    for causal in (False, True):
        o, lse = run_fp8(q, k, v, causal, scale, True)
        ref = oracle.attn_fwd_fp8(q, k, v, causal, scale, True)
        check_attention(o, lse, ref, True, "scale=%g causal=%d" % (scale, causal))


def test_fp8_zero_inputs():
    z = torch.zeros(1, 1, 200, 128, dtype=torch.bfloat16)
    o, lse = run_fp8(z, z, z, False, 0.1, True)
    assert np.all(o == 0.0) and np.abs(lse - math.log(200)).max() < 1e-4


def test_hadamard_lowers_the_error_on_outliers():
    # The claim of the CMU post's slide page 24, on the GPU path: error of O
    # against exact attention on the bf16 inputs, with and without rotation.
    B, H, N, d = 1, 4, 1024, 128
    q, k, v = synth.draw_outliers(B, H, N, d, seed=0)
    scale = 1 / math.sqrt(d)
    o_exact, _ = oracle.attn_fwd(q, k, v, False, scale)
    rmse = []
    for had in (False, True):
        o, _ = run_fp8(q, k, v, False, scale, had)
        rmse.append(math.sqrt(((o - o_exact) ** 2).mean()))
    assert rmse[0] / rmse[1] >= 1.4, rmse


def test_quantised_entry_point_reuses_the_workspace():
    B, H, N, d = 1, 2, 640, 128
    q, k, v = (t.to("cuda") for t in synth.draw_outliers(B, H, N, d, seed=3))
    ws = fa.fp8_quantize(q, k, v, hadamard=True)
    o1, l1 = fa.fwd_fp8_quantized(ws, B, H, N, d, causal=True, hadamard=True)
    o2, l2 = fa.fwd_fp8(q, k, v, causal=True, hadamard=True)
    fa.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fp8_rejects_d64_and_small_workspace():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fwd_fp8(q, q, q)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED_D
    q = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(fa.fwd_fp8_workspace_size(1, 1, 128, 128) - 256, dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fwd_fp8(q, q, q, workspace=ws)
    assert e.value.code == fa.FA_ERR_WORKSPACE


# ------------------------------------------- full-size workload, sampled head

def test_fp8_full_size_sampled_head():
    B, H, N, d = 8, 16, 8192, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=0, with_dout=False)
    o, lse = run_fp8(q, k, v, False, 1 / math.sqrt(d), True)
    head = B * H - 1

    def sel(t):
        return t.reshape(B * H, N, *t.shape[3:])[head][None, None]

    ref = oracle.attn_fwd_fp8(sel(q), sel(k), sel(v), False, 1 / math.sqrt(d), True)
    check_attention(sel(o), sel(lse), ref, True, "B8 H16 N8192")


def test_fp8_causal_large_sampled_head():
    B, H, N, d = 2, 8, 8192, 128
    q, k, v = synth.draw_outliers(B, H, N, d, seed=21)
    o, lse = run_fp8(q, k, v, True, 1 / math.sqrt(d), True)
    head = 5

    def sel(t):
        return t.reshape(B * H, N, *t.shape[3:])[head][None, None]

    # Per-head scales: the oracle on one head sees the same amax as the GPU.
    ref = oracle.attn_fwd_fp8(sel(q), sel(k), sel(v), True, 1 / math.sqrt(d), True)
    check_attention(sel(o), sel(lse), ref, True, "causal B2 H8 N8192")
