"""Forward pass on the GPU (through the C ABI) against the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output):
  O:   max |dO| <= 2e-2 and mean |dO| <= 2e-3 over every element,
  lse: max |dlse| <= 1e-3 absolute.
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


def run_fwd(q, k, v, causal, scale):
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    fa.check_device_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def compare(o, lse, o_ref, lse_ref, what=""):
    do = np.abs(o.astype(np.float64) - o_ref)
    dl = np.abs(lse.astype(np.float64) - lse_ref)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    assert do.max() <= O_MAX, (what, do.max())
    assert do.mean() <= O_MEAN, (what, do.mean())
    assert dl.max() <= LSE_MAX, (what, dl.max())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 257, 300, 1000])
def test_fwd_matches_oracle_small(N, causal, d):
    B, H = 2, 3
    q, k, v, _ = synth.draw(B, H, N, d, seed=N + 7 * d + causal, with_dout=False)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, "N=%d causal=%d d=%d" % (N, causal, d))


def test_tiny_workload():
    w = synth.TINY
    q, k, v, _ = synth.draw_workload(w, with_dout=False)
    o, lse = run_fwd(q, k, v, w.causal, w.softmax_scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.softmax_scale)
    compare(o, lse, o_ref, lse_ref, "tiny")


@pytest.mark.parametrize("scale", [0.0, -0.2, 0.9, 2.0])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_scales(scale, causal):
    q, k, v, _ = synth.draw(1, 2, 333, 64, seed=11, with_dout=False)
    o, lse = run_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, "scale=%g" % scale)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_heavy_rows_force_rescaling(d):
    # 1% of K rows x8 (the long-context recipe) at a size the oracle runs in
    # full: the running maximum of many rows grows after the first tile, so
    # O is rescaled in tensor memory (at d = 64 without a mask after waiting
    # for the previous P V, which the S ring lets the next S overtake).
    q, k, v, _ = synth.draw(1, 4, 2048, d, seed=3, heavy_frac=0.01, with_dout=False)
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, causal, 1 / math.sqrt(d))
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1 / math.sqrt(d))
        compare(o, lse, o_ref, lse_ref, "heavy causal=%d d=%d" % (causal, d))


def test_fwd_heavy_rows_persistent_d64():
    # The same rescaling on persistent CTAs with O staged for TMA stores
    # (768 items on at most 152 CTAs): scale 0.5 and 3% of K rows x8 make
    # rescales frequent; sampled rows of the first, last and random heads.
    from io_aware_exact_02_gb300.synth import Workload
    w = Workload("heavy_d64", 8, 24, 1024, 64, False, heavy_frac=0.03, scale=0.5)
    q, k, v, _ = synth.draw_workload(w, seed=17, with_dout=False)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=False, scale=w.softmax_scale)
    fa.check_device_status()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    sampled_check(w, o, lse, q, k, v, n_heads=4, n_rows=48, seed=5, extra=late_items(w))


def test_fwd_deterministic_bitwise():
    q, k, v, _ = synth.draw(2, 2, 1111, 128, seed=5, with_dout=False)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, causal=True)
    fa.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_invariants_on_gpu():
    # No oracle: scale 0 gives the (prefix) mean of V and lse = ln(count);
    # a joint permutation of K and V rows leaves non-causal O unchanged.
    B, H, N, d = 1, 2, 700, 64
    q, k, v, _ = synth.draw(B, H, N, d, seed=9, with_dout=False)
    o, lse = run_fwd(q, k, v, False, 0.0)
    vm = v.double().mean(2, keepdim=True).numpy()
    assert np.abs(o - vm).max() < 1e-2
    assert np.abs(lse - math.log(N)).max() < 1e-4
    o, lse = run_fwd(q, k, v, True, 0.0)
    pref = (v.double().cumsum(2) / torch.arange(1, N + 1).double()[None, None, :, None]).numpy()
    assert np.abs(o - pref).max() < 2e-2
    assert np.abs(lse - np.log(np.arange(1, N + 1))[None, None]).max() < 1e-4
    o1, l1 = run_fwd(q, k, v, False, 0.125)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(1))
    o2, l2 = run_fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, 0.125)
    assert np.abs(o1 - o2).max() < 1e-2
    assert np.abs(l1 - l2).max() < 1e-4


def test_fwd_causal_row_zero_is_v0():
    q, k, v, _ = synth.draw(1, 3, 513, 128, seed=21, with_dout=False)
    o, lse = run_fwd(q, k, v, True, 0.3)
    assert np.abs(o[:, :, 0] - v[:, :, 0].float().numpy()).max() < 1e-6
    ref = 0.3 * (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1).numpy()
    assert np.abs(lse[:, :, 0] - ref).max() < 1e-4


def test_fwd_bad_arguments_raise():
    q, k, v, _ = synth.draw(1, 1, 64, 64, seed=1, with_dout=False)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    with pytest.raises(fa.FaError) as e:
        fa.fwd(q, k, v, scale=float("nan"))
    assert e.value.code == fa.FA_ERR_ARG
    big = torch.empty(1, 1, 64, 96, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fwd(big, big, big)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED_D


# ------------------------------------------- full-size workloads, sampled rows

FULL = [w.name for w in synth.ALL if w.name != "tiny"]


def late_items(w, n=2):
    """(head, first row) of the last n items of the forward's work list on
    this GPU's persistent grid: the items a CTA reaches last, after its
    barriers, rings and tensor memory have gone through every earlier
    item's phases."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sched = fa.fwd_schedule(w.B, w.H, w.N, w.causal, num_ctas=sms)
    return [(bh, pair * 256) for bh, pair, _, _ in sched[-n:]]


def sampled_check(w, o_dev, lse_dev, q, k, v, n_heads=3, n_rows=48, seed=0, extra=()):
    """Oracle rows of a few heads: random ones, the last head, and the heads
    of `extra` (head, first row) items with rows from those items' 256."""
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    heads = sorted(set(rng.choice(BH, size=min(n_heads, BH), replace=False).tolist()) | {BH - 1}
                   | {bh for bh, _ in extra})
    late_rows = [r0 + rng.choice(min(256, w.N - r0), size=min(6, w.N - r0), replace=False)
                 for _, r0 in extra if r0 < w.N]
    rows = np.unique(np.concatenate([rng.choice(w.N, size=n_rows, replace=False),
                                     [0, w.N - 1, min(w.N - 1, 128), min(w.N - 1, 255)]] +
                                    late_rows))
    qf = q.reshape(BH, w.N, w.d)[heads].unsqueeze(0)
    kf = k.reshape(BH, w.N, w.d)[heads].unsqueeze(0)
    vf = v.reshape(BH, w.N, w.d)[heads].unsqueeze(0)
    hh = np.repeat(np.arange(len(heads)), rows.size)
    rr = np.tile(rows, len(heads))
    o_ref, lse_ref = oracle.attn_fwd_rows(qf, kf, vf, w.causal, w.softmax_scale, hh, rr)
    o = o_dev.reshape(BH, w.N, w.d)[heads][:, rows].float().cpu().numpy().reshape(-1, w.d)
    lse = lse_dev.reshape(BH, w.N)[heads][:, rows].cpu().numpy().reshape(-1)
    compare(o, lse, o_ref, lse_ref, w.name)


@pytest.mark.parametrize("name", FULL)
def test_fwd_full_size_sampled(name):
    w = synth.by_name(name)
    q, k, v, _ = synth.draw_workload(w, with_dout=False)
    dev = torch.device("cuda")
    o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.softmax_scale)
    fa.check_device_status()
    assert torch.isfinite(lse).all()
    sampled_check(w, o, lse, q, k, v, extra=late_items(w))


@pytest.mark.parametrize("N,d,causal", [(1000, 128, 0), (1920, 128, 0), (3000, 64, 0), (257, 64, 0),
                                        (100, 128, 0), (129, 128, 0), (300, 128, 0), (64, 64, 0),
                                        (1000, 128, 1), (1000, 64, 1), (129, 128, 1), (300, 64, 1),
                                        (2000, 128, 1)])
def test_fwd_staged_stores_ragged(N, d, causal):
    # Grids with more items than SMs store O through the staging ring slots
    # with TMA (at d = 128 from the epilogue warpgroup): without a mask each
    # persistent CTA takes its items in snake order, under the causal mask
    # the CTAs claim items of unequal cost from the work counter.  The tail
    # tile of every head is partly past N (rows there must not be written),
    # and at N <= 128 every item's second Q tile has no rows at all.
    # Sampled rows of the first, last and random heads, including each
    # head's last rows.
    from io_aware_exact_02_gb300.synth import Workload
    w = Workload("staged_N%d_d%d_c%d" % (N, d, causal), 8, 24, N, d, bool(causal))
    q, k, v, _ = synth.draw_workload(w, seed=N + d, with_dout=False)
    dev = torch.device("cuda")
    # A guard band after O catches a store past the end of the tensor.
    o_buf = torch.full((w.B * w.H * N * d + 4096,), 7.0, dtype=torch.bfloat16, device=dev)
    o = o_buf[: w.B * w.H * N * d].view(w.B, w.H, N, d)
    lse = torch.empty((w.B, w.H, N), dtype=torch.float32, device=dev)
    fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal, scale=w.softmax_scale, out=o, lse=lse)
    fa.check_device_status()
    assert torch.all(o_buf[w.B * w.H * N * d:] == 7.0)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    sampled_check(w, o, lse, q, k, v, n_heads=4, n_rows=40, seed=N)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_claimed_items_repeat_bitwise(d):
    # Under the causal mask with more items than SMs, the persistent CTAs
    # claim items from the library's work counter for the stream, which
    # every launch must leave at zero.  Repeated calls on one stream, calls
    # on a second stream, a static (non-causal) call and a general-path call
    # in between, give the same bits every time; an item is computed by one
    # CTA whichever claims it.
    B, H, N = 8, 24, 1000
    q, k, v, _ = synth.draw(B, H, N, d, seed=70 + d, with_dout=False)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o0, l0 = fa.fwd(q, k, v, causal=True)
    runs = []
    for i in range(3):
        runs.append(fa.fwd(q, k, v, causal=True))
        fa.fwd(q, k, v, causal=False)
        fa.fwd_gqa(q, k, v, causal=True, num_splits=1)
    s2 = torch.cuda.Stream()
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s2):
        runs.append(fa.fwd(q, k, v, causal=True))
        runs.append(fa.fwd(q, k, v, causal=True))
    torch.cuda.current_stream().wait_stream(s2)
    torch.cuda.synchronize()
    fa.check_device_status()
    for o, l in runs:
        assert torch.equal(o, o0) and torch.equal(l, l0)
    w = synth.Workload("claimed_d%d" % d, B, H, N, d, True)
    sampled_check(w, o0, l0, q.cpu(), k.cpu(), v.cpu(), n_heads=3, n_rows=32, seed=d,
                  extra=late_items(w))


def test_fwd_claimed_items_concurrent_streams():
    # Masked forward passes in flight at once on two streams use two counter
    # slots and both give the serial result; so do calls on many more
    # streams in turn (each stream its own slot, each left at zero).
    B, H, N, d = 8, 16, 1024, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=81, with_dout=False)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o_ref, l_ref = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(24)]
    outs = []
    for s in streams[:2]:
        s.wait_stream(torch.cuda.current_stream())
    for s in streams[:2]:
        with torch.cuda.stream(s):
            outs.append(fa.fwd(q, k, v, causal=True))
    for s in streams[2:]:
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            outs.append(fa.fwd(q, k, v, causal=True))
        s.synchronize()
    torch.cuda.synchronize()
    fa.check_device_status()
    for o, l in outs:
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_fwd_claimed_items_per_thread_default_streams():
    # Two host threads launch masked forward passes on their own per-thread
    # default streams (one handle value, cudaStreamPerThread, for both): the
    # library tells the streams apart by their ids, so each gets its own
    # work-counter slot and both results equal the serial one bitwise.
    import ctypes
    import threading
    B, H, N, d = 8, 16, 1024, 128
    q, k, v, _ = synth.draw(B, H, N, d, seed=83, with_dout=False)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    o_ref, l_ref = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    outs = [(torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev))
            for _ in range(2)]
    rcs = [None, None]
    per_thread = ctypes.c_void_p(2)  # cudaStreamPerThread
    lib = fa.load()

    def run(i):
        torch.cuda.set_device(q.device)
        o, l = outs[i]
        rc = 0
        for _ in range(4):
            rc = rc or lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  l.data_ptr(), B, H, N, d, 1, ctypes.c_float(1 / math.sqrt(d)),
                                  per_thread)
        rcs[i] = rc

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    fa.check_device_status()
    assert rcs == [0, 0]
    for o, l in outs:
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_fwd_long_sequence_sampled_rows():
    # N = 65536 (512 key tiles per head) causal and not: sampled rows against
    # the oracle's row-wise definition.
    from io_aware_exact_02_gb300.synth import Workload
    for causal in (False, True):
        w = Workload("n64k_%d" % causal, 1, 2, 65536, 128, causal)
        q, k, v, _ = synth.draw_workload(w, seed=3, with_dout=False)
        dev = torch.device("cuda")
        o, lse = fa.fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=w.softmax_scale)
        fa.check_device_status()
        sampled_check(w, o, lse, q, k, v, n_heads=2, n_rows=24, seed=causal)
