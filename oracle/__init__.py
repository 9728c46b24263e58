"""fp64 CPU oracle for exact attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The product path (the CUDA library and its Python binding)
never imports, links or calls it, and it shares no code with them.

The arithmetic lives in ``oracle.c`` (plain loops in fp64, OpenMP over
independent rows); this module builds it with gcc on first use and marshals
numpy arrays.  Every array is float64 with shape (B, H, N, d) (lse: (B, H, N)).

Readings of the pages that the oracle fixes (each one is also listed in the
design notes):
  * lse is the natural-log logsumexp of the *scaled* scores;
  * ``scale`` multiplies Q K^T before the softmax, any finite value;
  * causal masking is square and top-left: row i sees keys j <= i;
  * the backward pass is the textbook softmax Jacobian (the pages print no
    formula for it);
  * FP8 form: Q and K rotated by the Sylvester Hadamard matrix, one E4M3
    scale per head and tensor (amax / 448), codes rounded to nearest-even
    and saturated, the rounding decision taken in fp32, then exact
    attention over the dequantised tensors with scale / d.
The pages print no worked gradient example, so the backward pass is pinned
by the mathematics instead: central finite differences of the forward pass,
closed forms (scale 0, causal row 0) and invariants (sums of dV and dK, the
bilinear identity sum q . dQ = sum k . dK, the derivative in the scale, key
shift and permutation), which on their own catch every planted backward
mistake; and by an independent library routine (torch autograd).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP).  Returns the path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load an oracle shared library from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    i64, cint, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, i64, i64, i64, cint, dbl, dp, dp]
    lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, i64, i64, i64, cint, dbl,
                                         ip, ip, i64, dp, dp]
    lib.oracle_attn_probs.argtypes = [dp, dp, i64, i64, i64, cint, dbl, dp]
    lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, i64, i64, i64, cint, dbl,
                                    dp, dp, dp]
    lib.oracle_attn_fwd_gqa.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, i64, cint, dbl,
                                        dp, dp]
    lib.oracle_combine_splits.argtypes = [dp, dp, i64, i64, i64, dp, dp]
    u8p = ctypes.POINTER(ctypes.c_ubyte)
    lib.oracle_attn_fwd_blockmask.argtypes = [dp, dp, dp, i64, i64, i64, cint, dbl, u8p, i64,
                                              dp, dp]
    lib.oracle_attn_bwd_blockmask.argtypes = [dp, dp, dp, dp, i64, i64, i64, cint, dbl, u8p,
                                              i64, dp, dp, dp]
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_ubyte]
    lib.oracle_e4m3_decode.restype = dbl
    lib.oracle_e4m3_encode.argtypes = [dbl]
    lib.oracle_e4m3_encode.restype = ctypes.c_ubyte
    lib.oracle_e4m3_encode_array.argtypes = [dp, i64, u8p]
    lib.oracle_e4m3_decode_array.argtypes = [u8p, i64, dp]
    lib.oracle_hadamard.argtypes = [dp, i64, i64, dp]
    lib.oracle_quantize_e4m3.argtypes = [dp, i64, u8p]
    lib.oracle_quantize_e4m3.restype = ctypes.c_float
    fp = ctypes.POINTER(ctypes.c_float)
    lib.oracle_attn_fwd_fp8.argtypes = [dp, dp, dp, i64, i64, i64, cint, dbl, cint, dp, dp,
                                        u8p, u8p, u8p, fp]
    lib.oracle_fwd_flops.argtypes = [i64, i64, i64, cint]
    lib.oracle_fwd_flops.restype = dbl
    lib.oracle_recompute_flops.argtypes = [i64, i64]
    lib.oracle_recompute_flops.restype = dbl
    lib.oracle_num_threads.restype = cint
    lib.oracle_set_num_threads.argtypes = [cint]
    for f in (lib.oracle_attn_fwd, lib.oracle_attn_fwd_rows,
              lib.oracle_attn_probs, lib.oracle_attn_bwd,
              lib.oracle_attn_fwd_gqa, lib.oracle_combine_splits,
              lib.oracle_attn_fwd_blockmask, lib.oracle_attn_bwd_blockmask,
              lib.oracle_e4m3_encode_array, lib.oracle_e4m3_decode_array,
              lib.oracle_hadamard, lib.oracle_attn_fwd_fp8, lib.oracle_set_num_threads):
        f.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def _f64(x) -> np.ndarray:
    """Contiguous float64 numpy copy of x (numpy array or torch tensor)."""
    if hasattr(x, "detach"):  # torch tensor: bf16 -> fp32 -> fp64 is exact
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape4(q):
    if q.ndim != 4:
        raise ValueError("expected (B, H, N, d) arrays")
    return q.shape


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def attn_fwd(q, k, v, causal: bool, scale: float, lib=None):
    """O and lse of exact attention, fp64.  Returns (o (B,H,N,d), lse (B,H,N))."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    (lib or _load()).oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B * H, N, d, int(bool(causal)),
                            float(scale), _ptr(o), _ptr(lse))
    return o, lse


def attn_fwd_rows(q, k, v, causal: bool, scale: float, heads, rows):
    """O rows and lse for the selected flat heads (b*H + h) and rows only.

    Returns (o_sel (n, d), lse_sel (n,)).  For sampled checks of workloads too
    large for the full oracle.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    heads = np.ascontiguousarray(heads, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if heads.shape != rows.shape or heads.ndim != 1:
        raise ValueError("heads and rows must be 1-D and of equal length")
    if heads.size and (heads.min() < 0 or heads.max() >= B * H or rows.min() < 0
                       or rows.max() >= N):
        raise ValueError("head or row index out of range")
    n = heads.size
    o = np.zeros((n, d))
    lse = np.zeros((n,))
    ip = ctypes.POINTER(ctypes.c_int64)
    _load().oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B * H, N, d,
                                 int(bool(causal)), float(scale),
                                 heads.ctypes.data_as(ip), rows.ctypes.data_as(ip), n,
                                 _ptr(o), _ptr(lse))
    return o, lse


def attn_probs(q, k, causal: bool, scale: float, lib=None):
    """The attention matrix A = softmax(S), (B, H, N, N).  Small cases only."""
    q, k = _f64(q), _f64(k)
    B, H, N, d = _shape4(q)
    A = np.zeros((B, H, N, N))
    (lib or _load()).oracle_attn_probs(_ptr(q), _ptr(k), B * H, N, d, int(bool(causal)),
                              float(scale), _ptr(A))
    return A


def attn_bwd(q, k, v, dout, causal: bool, scale: float, lib=None):
    """dQ, dK, dV of L = sum(dout * O), fp64 textbook backward."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = _shape4(q)
    dq = np.zeros((B, H, N, d))
    dk = np.zeros((B, H, N, d))
    dv = np.zeros((B, H, N, d))
    (lib or _load()).oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B * H, N, d,
                            int(bool(causal)), float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def attn_fwd_gqa(q, k, v, causal: bool, scale: float, lib=None):
    """General forward: q (B, Hq, Nq, d), k and v (B, Hkv, Nkv, d), Hq a
    multiple of Hkv; causal is aligned bottom-right.  Returns (o, lse)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, d = _shape4(q)
    Bk, Hkv, Nkv, dk = _shape4(k)
    if Bk != B or dk != d or v.shape != k.shape or Hkv < 1 or Hq % Hkv:
        raise ValueError("incompatible q / k / v shapes")
    o = np.zeros((B, Hq, Nq, d))
    lse = np.zeros((B, Hq, Nq))
    (lib or _load()).oracle_attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d,
                                         int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    return o, lse


def combine_splits(o_parts, lse_parts, lib=None):
    """Merge partial (O_s, lse_s) over key ranges: o_parts (S, ..., d),
    lse_parts (S, ...).  Returns (o, lse) with the trailing shapes."""
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    S = o_parts.shape[0]
    d = o_parts.shape[-1]
    R = int(np.prod(o_parts.shape[1:-1]))
    o = np.zeros(o_parts.shape[1:])
    lse = np.zeros(lse_parts.shape[1:])
    (lib or _load()).oracle_combine_splits(_ptr(o_parts), _ptr(lse_parts), S, R, d, _ptr(o),
                                           _ptr(lse))
    return o, lse


def _blockmask(bm, N, bs):
    bm = np.ascontiguousarray(bm, dtype=np.uint8)
    nb = -(-N // bs)
    if bm.shape != (nb, nb):
        raise ValueError("block mask must be (%d, %d)" % (nb, nb))
    return bm, bm.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def attn_fwd_blockmask(q, k, v, causal: bool, scale: float, block_mask, block=128, lib=None):
    """Block-sparse forward: key j visible to query i iff
    block_mask[i // block, j // block] (and j <= i when causal)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    bm, bmp = _blockmask(block_mask, N, block)
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    (lib or _load()).oracle_attn_fwd_blockmask(_ptr(q), _ptr(k), _ptr(v), B * H, N, d,
                                               int(bool(causal)), float(scale), bmp, block,
                                               _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd_blockmask(q, k, v, dout, causal: bool, scale: float, block_mask, block=128,
                       lib=None):
    """dQ, dK, dV of the block-sparse forward."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = _shape4(q)
    bm, bmp = _blockmask(block_mask, N, block)
    dq, dk, dv = (np.zeros((B, H, N, d)) for _ in range(3))
    (lib or _load()).oracle_attn_bwd_blockmask(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B * H, N,
                                               d, int(bool(causal)), float(scale), bmp, block,
                                               _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def _u8p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte))


def e4m3_decode(codes, lib=None) -> np.ndarray:
    """Values (float64) of E4M3 codes (uint8, any shape)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(c.shape)
    (lib or _load()).oracle_e4m3_decode_array(_u8p(c), c.size, _ptr(out))
    return out


def e4m3_encode(x, lib=None) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, saturated to +-448) of float64 x."""
    x = _f64(x)
    out = np.zeros(x.shape, dtype=np.uint8)
    (lib or _load()).oracle_e4m3_encode_array(_ptr(x), x.size, _u8p(out))
    return out


def hadamard(x, lib=None) -> np.ndarray:
    """x H_d over the last axis (Sylvester Hadamard matrix, entries +-1)."""
    x = _f64(x)
    d = x.shape[-1]
    y = np.zeros(x.shape)
    (lib or _load()).oracle_hadamard(_ptr(x), x.size // d, d, _ptr(y))
    return y


def quantize_e4m3(x, lib=None):
    """One-scale E4M3 quantisation of all of x: (codes, descale)."""
    x = _f64(x)
    codes = np.zeros(x.shape, dtype=np.uint8)
    s = (lib or _load()).oracle_quantize_e4m3(_ptr(x), x.size, _u8p(codes))
    return codes, float(s)


def attn_fwd_fp8(q, k, v, causal: bool, scale: float, hadamard: bool, lib=None):
    """FP8 forward with optional Hadamard rotation of Q and K.

    Returns (o, lse, q8, k8, v8, descale): o (B,H,N,d) and lse (B,H,N) in
    float64; the E4M3 codes of the (rotated) Q, K and of V as (B,H,N,d)
    uint8; descale (3, B, H) float32, the per-head scales of Q, K, V."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    q8, k8, v8 = (np.zeros((B, H, N, d), dtype=np.uint8) for _ in range(3))
    ds = np.zeros((3, B, H), dtype=np.float32)
    (lib or _load()).oracle_attn_fwd_fp8(
        _ptr(q), _ptr(k), _ptr(v), B * H, N, d, int(bool(causal)), float(scale),
        int(bool(hadamard)), _ptr(o), _ptr(lse), _u8p(q8), _u8p(k8), _u8p(v8),
        ds.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return o, lse, q8, k8, v8, ds


def fwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """4 N^2 d per head for the two matmuls, halved when causal."""
    return float(_load().oracle_fwd_flops(B * H, N, d, int(bool(causal))))


def recompute_flops(N: int, d: int) -> float:
    """The backward pass's extra Q K^T per head: 2 N^2 d."""
    return float(_load().oracle_recompute_flops(N, d))
