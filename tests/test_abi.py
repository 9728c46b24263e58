"""The C-ABI library without a GPU: it loads, exports every symbol
include/fa.h declares, rejects bad arguments with its error codes before
touching a device, and its host-side scheduler follows the LPT rule."""
import ctypes
import os
import re

import pytest

from io_aware_exact_02_gb300 import build, fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_bound_symbols():
    assert declared_symbols() == sorted(fa.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.fa_version() == 1


def test_status_strings(lib):
    for code in (fa.FA_OK, fa.FA_ERR_ARG, fa.FA_ERR_UNSUPPORTED_D, fa.FA_ERR_ALIGN,
                 fa.FA_ERR_WORKSPACE, fa.FA_ERR_DEVICE, fa.FA_ERR_LAUNCH, fa.FA_ERR_TIMEOUT):
        s = lib.fa_status_string(code)
        assert s and s != b"unknown status"
    assert lib.fa_status_string(12345) == b"unknown status"


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced


def call_fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, causal=0,
             scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, causal, ctypes.c_float(scale), None)


def test_fwd_argument_errors_launch_nothing(lib):
    assert call_fwd(lib, q=None) == fa.FA_ERR_ARG
    assert call_fwd(lib, lse=None) == fa.FA_ERR_ARG
    assert call_fwd(lib, B=0) == fa.FA_ERR_ARG
    assert call_fwd(lib, H=-1) == fa.FA_ERR_ARG
    assert call_fwd(lib, N=0) == fa.FA_ERR_ARG
    assert call_fwd(lib, causal=2) == fa.FA_ERR_ARG
    assert call_fwd(lib, scale=float("nan")) == fa.FA_ERR_ARG
    assert call_fwd(lib, scale=float("inf")) == fa.FA_ERR_ARG
    assert call_fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED_D
    assert call_fwd(lib, d=256) == fa.FA_ERR_UNSUPPORTED_D
    assert call_fwd(lib, k=FAKE + 8) == fa.FA_ERR_ALIGN
    assert call_fwd(lib, lse=FAKE + 4) == fa.FA_ERR_ALIGN
    assert call_fwd(lib, B=1 << 16, H=1 << 16) == fa.FA_ERR_ARG


def test_bwd_argument_errors_launch_nothing(lib):
    ws = lib.fa_bwd_workspace_size(1, 1, 128, 64)

    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
                 B=1, H=1, N=128, d=64, causal=0, scale=0.125, ws=FAKE, wsb=ws)
        a.update(kw)
        return lib.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                          a["dv"], a["B"], a["H"], a["N"], a["d"], a["causal"],
                          ctypes.c_float(a["scale"]), a["ws"], a["wsb"], None)

    assert call(dv=None) == fa.FA_ERR_ARG
    assert call(N=0) == fa.FA_ERR_ARG
    assert call(d=80) == fa.FA_ERR_UNSUPPORTED_D
    assert call(do=FAKE + 2) == fa.FA_ERR_ALIGN
    assert call(ws=None) == fa.FA_ERR_WORKSPACE
    assert call(wsb=ws - 1) == fa.FA_ERR_WORKSPACE
    assert call(ws=FAKE + 16) == fa.FA_ERR_WORKSPACE

    def phases(mask, **kw):
        a = dict(q=FAKE, ws=FAKE, wsb=ws)
        a.update(kw)
        return lib.fa_bwd_phases(a["q"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128,
                                 64, 0, ctypes.c_float(0.125), a["ws"], a["wsb"], None, mask)

    # The phase mask is checked first; then the arguments as for fa_bwd.
    for mask in (0, 8, -1, 15):
        assert phases(mask) == fa.FA_ERR_ARG
    assert phases(2, q=None) == fa.FA_ERR_ARG
    assert phases(4, wsb=ws - 1) == fa.FA_ERR_WORKSPACE


def test_workspace_size(lib):
    # fp32 dQ accumulator over 128-row-padded rows plus two fp32 per row.
    def up(x):
        return (x + 255) // 256 * 256
    rows = 2 * 3 * 384
    # dQ accumulator, -D, -lse*log2(e), then a 256-byte slot for the counter
    assert lib.fa_bwd_workspace_size(2, 3, 300, 64) == up(rows * 64 * 4) + 2 * up(rows * 4) + 256
    assert lib.fa_bwd_workspace_size(1, 1, 128, 128) == 128 * 128 * 4 + 2 * 128 * 4 + 256
    assert lib.fa_bwd_workspace_size(1, 1, 1, 64) == 128 * 64 * 4 + 2 * 512 + 256
    assert lib.fa_bwd_workspace_size(1, 1, 0, 64) == 0
    assert lib.fa_bwd_workspace_size(1, 1, 128, 72) == 0


# ------------------------------------------------------------- scheduling

def greedy(costs, workers):
    """List scheduling: each item goes to the least-loaded worker, in order."""
    loads = [0] * workers
    for c in costs:
        w = loads.index(min(loads))
        loads[w] += c
    return loads


def golden_lpt():
    path = os.path.join(ROOT, "tests", "golden", "pages_numbers.txt")
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            key, val = line.split(None, 1)
            vals[key] = [int(x) for x in val.split(",")] if "," in val else val
    return vals["lpt_in_order"], vals["lpt_longest_first"]


def test_lpt_example_of_the_pages(lib):
    # Two batches of four causal query tiles costing 1, 2, 3, 4 key tiles,
    # three SMs: in order the SMs end with [9, 5, 6]; longest first gives
    # [7, 7, 6] (CMU 11-868 post, LPT paragraph).
    in_order, lpt = golden_lpt()
    costs = [1, 2, 3, 4, 1, 2, 3, 4]
    assert greedy(costs, 3) == in_order
    assert greedy(sorted(costs, reverse=True), 3) == lpt
    # The kernels' static persistent assignment reproduces the LPT loads on
    # the longest-first list.
    ordered = sorted(costs, reverse=True)
    workers = fa.snake_assign(len(ordered), 3)
    loads = [sum(c for c, w in zip(ordered, workers) if w == k) for k in range(3)]
    assert loads == lpt
    assert fa.snake_assign(7, 3) == [0, 1, 2, 2, 1, 0, 0]


@pytest.mark.parametrize("B,H,N,causal", [(1, 2, 1024, 1), (2, 5, 3000, 1), (3, 4, 700, 0),
                                          (1, 17, 4096, 1), (1, 1, 1, 0), (1, 1, 1024, 1),
                                          (1, 1, 1792, 1)])
def test_schedule_covers_every_item_once_longest_first(lib, B, H, N, causal):
    items = fa.fwd_schedule(B, H, N, causal, num_ctas=7)
    n_pairs = -(-N // 256)
    assert sorted((bh, p) for bh, p, _, _ in items) == [(bh, p) for bh in range(B * H)
                                                       for p in range(n_pairs)]
    if causal and len(items) > 7:
        # Claimed from the work counter at run time by 7 persistent CTAs.
        assert all(c == -1 for _, _, _, c in items)
    elif causal:
        # No more items than CTAs: item t on CTA t.
        assert [c for _, _, _, c in items] == list(range(len(items)))
    else:
        assert [c for _, _, _, c in items] == fa.snake_assign(len(items), min(len(items), 7))
    n_kv = -(-N // 128)
    for bh, p, c, _ in items:
        expect = (min(2 * p + 1, n_kv) + min(2 * p + 2, n_kv)) if causal else 2 * n_kv
        assert c == expect
    # Within each group of heads the costs never increase (LPT order), and the
    # order equals a stable longest-first sort of the group's items.
    group = 8 * n_pairs
    for g0 in range(0, len(items), group):
        chunk = items[g0:g0 + group]
        costs = [c for _, _, c, _ in chunk]
        assert costs == sorted(costs, reverse=True)
    if causal:
        loads_lpt = greedy([c for _, _, c, _ in items], 3)
        loads_fwd = greedy(sorted([c for _, _, c, _ in items]), 3)
        assert max(loads_lpt) <= max(loads_fwd)


def test_fwd_gqa_sizes_and_splits(lib):
    # No workspace with one effective split; otherwise per-split fp32 O and
    # lse of every packed row, each part rounded up to 256 bytes.
    assert lib.fa_fwd_gqa_workspace_size(2, 8, 2, 1, 1000, 128, 1) == 0
    rows = 2 * 2 * 4  # B * Hkv * (G * Nq)
    up = lambda x: (x + 255) // 256 * 256
    assert lib.fa_fwd_gqa_workspace_size(2, 8, 2, 1, 1000, 128, 3) == up(3 * rows * 128 * 4) + up(3 * rows * 4)
    # 1000 keys = 8 tiles: 50 requested splits become 8 (one tile each)
    assert lib.fa_fwd_gqa_workspace_size(1, 2, 2, 3, 1000, 64, 50) == up(8 * 6 * 64 * 4) + up(8 * 6 * 4)
    assert lib.fa_fwd_gqa_workspace_size(1, 3, 2, 3, 1000, 64, 2) == 0   # Hq not a multiple
    assert lib.fa_fwd_gqa_splits(8, 16, 16, 8192, 8192, 128, 0, 152) == 1
    # 64 items (B*Hkv) on 152 SMs: 7 splits fill 448/456 of three waves
    # (3 splits would leave 112 of 304 slots idle).
    assert lib.fa_fwd_gqa_splits(8, 32, 8, 1, 32768, 128, 1, 152) == 7
    # 256 items: 4 splits give 1024 of 1064 slots.
    assert lib.fa_fwd_gqa_splits(32, 32, 8, 1, 32768, 128, 1, 152) == 4
    # 1 item: at most 128 splits (128/152 of a wave); 116 is the first within 90%.
    assert lib.fa_fwd_gqa_splits(1, 8, 1, 1, 32768, 128, 1, 152) == 116
    assert lib.fa_fwd_gqa_splits(1, 8, 1, 1, 300, 128, 0, 152) == 1
    assert lib.fa_fwd_gqa_splits(1, 8, 1, 1, 300, 128, 0, 0) == fa.FA_ERR_ARG


def test_fwd_gqa_argument_errors_launch_nothing(lib):
    def call(**kw):
        a = dict(B=1, Hq=4, Hkv=2, Nq=3, Nkv=100, d=64, causal=0, splits=1, ws=None, wsb=0)
        a.update(kw)
        return lib.fa_fwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["Hq"], a["Hkv"], a["Nq"],
                              a["Nkv"], a["d"], a["causal"], ctypes.c_float(0.1), a["splits"],
                              a["ws"], a["wsb"], None)
    assert call(Hq=3) == fa.FA_ERR_ARG
    assert call(Hkv=0) == fa.FA_ERR_ARG
    assert call(Nkv=0) == fa.FA_ERR_ARG
    assert call(splits=0) == fa.FA_ERR_ARG
    assert call(d=80) == fa.FA_ERR_UNSUPPORTED_D
    assert call(splits=2, Nkv=1000) == fa.FA_ERR_WORKSPACE


def test_blocksparse_argument_errors_launch_nothing(lib):
    def fwd(mask=FAKE, **kw):
        a = dict(B=1, H=2, N=300, d=64, causal=0)
        a.update(kw)
        return lib.fa_fwd_blocksparse(FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["N"], a["d"],
                                      a["causal"], ctypes.c_float(0.1), mask, None)

    def bwd(mask=FAKE, **kw):
        a = dict(B=1, H=2, N=300, d=64, causal=0, ws=FAKE,
                 wsb=lib.fa_bwd_workspace_size(1, 2, 300, 64))
        a.update(kw)
        return lib.fa_bwd_blocksparse(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["B"],
                                      a["H"], a["N"], a["d"], a["causal"], ctypes.c_float(0.1),
                                      mask, a["ws"], a["wsb"], None)

    assert fwd(mask=None) == fa.FA_ERR_ARG
    assert bwd(mask=None) == fa.FA_ERR_ARG
    assert fwd(N=0) == fa.FA_ERR_ARG and bwd(N=0) == fa.FA_ERR_ARG
    assert fwd(causal=3) == fa.FA_ERR_ARG and bwd(causal=3) == fa.FA_ERR_ARG
    assert fwd(d=32) == fa.FA_ERR_UNSUPPORTED_D and bwd(d=32) == fa.FA_ERR_UNSUPPORTED_D
    assert bwd(wsb=16) == fa.FA_ERR_WORKSPACE
    # Valid arguments reach the device check (no GPU in a CPU-only run).
    if not torch_cuda_available():
        assert fwd() == fa.FA_ERR_DEVICE and bwd() == fa.FA_ERR_DEVICE


def torch_cuda_available():
    import torch
    return torch.cuda.is_available()


def test_fp8_sizes_and_argument_errors(lib):
    size = lib.fa_fwd_fp8_workspace_size(2, 3, 300, 128)
    off = (ctypes.c_size_t * 4)()
    assert lib.fa_fp8_workspace_offsets(2, 3, 300, 128, off) == fa.FA_OK
    qk = 2 * 3 * 300 * 128
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert list(off) == [0, up(qk), 2 * up(qk), 2 * up(qk) + up(2 * 3 * 128 * 384)]
    assert size == off[3] + up(3 * 6 * 4)
    assert lib.fa_fwd_fp8_workspace_size(1, 1, 128, 64) == 0
    assert lib.fa_fp8_workspace_offsets(1, 1, 128, 64, off) == fa.FA_ERR_UNSUPPORTED_D
    assert lib.fa_fp8_workspace_offsets(1, 1, 128, 128, None) == fa.FA_ERR_ARG

    def call(**kw):
        a = dict(B=1, H=1, N=128, d=128, causal=0, had=1, ws=FAKE,
                 wsb=lib.fa_fwd_fp8_workspace_size(1, 1, 128, 128))
        a.update(kw)
        return lib.fa_fwd_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, a["B"], a["H"], a["N"], a["d"],
                              a["causal"], ctypes.c_float(0.1), a["had"], a["ws"], a["wsb"], None)

    assert call(d=64) == fa.FA_ERR_UNSUPPORTED_D
    assert call(had=2) == fa.FA_ERR_ARG
    assert call(causal=5) == fa.FA_ERR_ARG
    assert call(ws=None) == fa.FA_ERR_WORKSPACE
    assert call(ws=FAKE + 128) == fa.FA_ERR_WORKSPACE
    assert call(wsb=100) == fa.FA_ERR_WORKSPACE
    assert lib.fa_fwd_fp8_quantized(FAKE, FAKE, 1, 1, 128, 128, 0, ctypes.c_float(0.1), 1, None,
                                    0, None) == fa.FA_ERR_WORKSPACE
    assert lib.fa_fp8_quantize(None, FAKE, FAKE, 1, 1, 128, 128, 1, FAKE, 1 << 20,
                               None) == fa.FA_ERR_ARG


def test_selftest_timeout_arguments(lib):
    assert lib.fa_selftest_timeout(0, None) == fa.FA_ERR_ARG
    assert lib.fa_selftest_timeout(1000001, None) == fa.FA_ERR_ARG
    if not torch_cuda_available():
        assert lib.fa_selftest_timeout(1000, None) == fa.FA_ERR_DEVICE


def test_noalloc_scratch_size_matches_the_header():
    import re
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "FA_NOALLOC_SCRATCH_BYTES not found"
    assert fa.FA_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_binding_rejects_tensors_on_another_device():
    # One call's tensors must share a device: the library resolves its
    # per-device state on the current device, which the binding sets to q's.
    import torch
    a = torch.empty(4, device="meta")
    b = torch.empty(4)
    with pytest.raises(ValueError, match="share a device"):
        fa._on_device(b, k=a)


def test_checks_compiled_out_of_the_default_build(lib):
    assert lib.fa_checks_enabled() == (1 if fa.CHECKED else 0)


def test_checked_build_compiles_and_reports_it():
    """The bounds-checked variant builds from the same sources (nvcc with
    -DFA_CHECKS) and exports the same symbols."""
    from io_aware_exact_02_gb300 import build
    path = build.build(checked=True)
    chk = fa.load(path)
    assert chk.fa_checks_enabled() == 1
    for name in declared_symbols():
        assert hasattr(chk, name), name
    assert chk.fa_status_string(fa.FA_ERR_BOUNDS) != b"unknown status"
