"""ctypes binding of libfa.so (argument marshalling only).

Every function here passes raw device pointers, sizes and the current CUDA
stream to the C ABI declared in include/fa.h; all the arithmetic runs in the
library's CUDA kernels.  There is no fallback: if libfa.so is missing or
cannot be loaded, or a call returns an error code, a ``FaError`` is raised.

Tensors are torch tensors used as device buffers: q, k, v, o, dout, dq, dk,
dv are contiguous bf16 (B, H, N, d) on a CUDA device, lse is contiguous fp32
(B, H, N).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# FA_CHECKED=1 selects the bounds-checked build (python -m
# io_aware_exact_02_gb300.build --checked), whose kernels range-check every
# tile, mask and row index they compute.
CHECKED = os.environ.get("FA_CHECKED") == "1"
LIB_PATH = os.path.join(_HERE, "libfa_checked.so" if CHECKED else "libfa.so")

FA_OK = 0
FA_ERR_ARG = -1
FA_ERR_UNSUPPORTED_D = -2
FA_ERR_ALIGN = -3
FA_ERR_WORKSPACE = -4
FA_ERR_DEVICE = -5
FA_ERR_LAUNCH = -6
FA_ERR_TIMEOUT = -7
FA_ERR_BOUNDS = -8

# Size of the static scratch array fa_bwd_noalloc uses (FA_NOALLOC_SCRATCH_BYTES).
FA_NOALLOC_SCRATCH_BYTES = 32 << 20

# Every symbol include/fa.h declares, with (restype, argtypes).
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz,
                        _vp]),
    "fa_fwd_gqa_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "fa_fwd_gqa_splits": (_i, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "fa_bwd_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f,
                    _vp, _sz, _vp]),
    "fa_bwd_phases": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f,
                           _vp, _sz, _vp, _i]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f,
                            _vp]),
    "fa_fwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp]),
    "fa_bwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                _f, _vp, _vp, _sz, _vp]),
    "fa_fwd_fp8_workspace_size": (_sz, [_i, _i, _i, _i]),
    "fa_fp8_workspace_offsets": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]),
    "fa_fp8_quantize": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "fa_fwd_fp8_quantized": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_device_status": (_i, [_vp, _ip]),
    "fa_selftest_timeout": (_i, [_i, _vp]),
    "fa_checks_enabled": (_i, []),
    "fa_selftest_bounds": (_i, [_vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_fwd_schedule": (_i, [_i, _i, _i, _i, _i, _ip, _ip, _ip, _ip, _i]),
    "fa_snake_assign": (_i, [_i, _i, _ip]),
    "fa_version": (_i, []),
}


class FaError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__("%s failed: %s (%d)" % (fn, msg, code))
        self.code = code


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libfa.so (once) and declare its signatures.  Raises if missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise FaError("load", FA_ERR_DEVICE,
                          "%s is missing; build it with python -m io_aware_exact_02_gb300.build" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


def _check(fn: str, code: int):
    if code != FA_OK:
        raise FaError(fn, code, status_string(code))


def _stream_of(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check_qkv(name, t, shape, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s" % (name, dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _on_device(ref, **tensors):
    """Check that every given tensor is on ``ref``'s device and return a
    context manager that makes that device current for the call: the library
    looks up its per-device state (status word, SM count, tensor maps) on the
    current device, and tensor maps built there must address that device's
    memory."""
    for name, t in tensors.items():
        if t is not None and t.device != ref.device:
            raise ValueError("%s is on %s, expected %s (one call's tensors must share a device)"
                             % (name, t.device, ref.device))
    return torch.cuda.device(ref.device)


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """O, lse = attention(q, k, v).  Returns (o, lse) (allocated if not given)."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_qkv(name, t, (B, H, N, d))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv("out", out, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    with _on_device(q, k=k, v=v, out=out, lse=lse):
        rc = load().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, H, N, d, int(bool(causal)), ctypes.c_float(scale),
                           _stream_of(q))
    _check("fa_fwd", rc)
    return out, lse


def fwd_gqa_splits(B, Hq, Hkv, Nq, Nkv, d, causal=False, sm_count=None) -> int:
    """Key splits that fill the device's SMs (fa_fwd_gqa_splits)."""
    if sm_count is None:
        sm_count = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    n = load().fa_fwd_gqa_splits(B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)), int(sm_count))
    if n < 0:
        _check("fa_fwd_gqa_splits", n)
    return n


def fwd_gqa_workspace_size(B, Hq, Hkv, Nq, Nkv, d, num_splits) -> int:
    return int(load().fa_fwd_gqa_workspace_size(B, Hq, Hkv, Nq, Nkv, d, int(num_splits)))


def fwd_gqa(q, k, v, causal: bool = False, scale: float | None = None, num_splits=None,
            out=None, lse=None, workspace=None):
    """General forward: q (B, Hq, Nq, d), k and v (B, Hkv, Nkv, d), Hq a
    multiple of Hkv; causal aligned bottom-right; the keys cut into
    ``num_splits`` ranges (None: fa_fwd_gqa_splits).  Returns (o, lse)."""
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nkv, dk = k.shape
    scale = default_scale(d) if scale is None else float(scale)
    _check_qkv("q", q, (B, Hq, Nq, d))
    _check_qkv("k", k, (B, Hkv, Nkv, d))
    _check_qkv("v", v, (B, Hkv, Nkv, d))
    if num_splits is None:
        num_splits = fwd_gqa_splits(B, Hq, Hkv, Nq, Nkv, d, causal)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    _check_qkv("out", out, (B, Hq, Nq, d))
    _check_qkv("lse", lse, (B, Hq, Nq), torch.float32)
    need = fwd_gqa_workspace_size(B, Hq, Hkv, Nq, Nkv, d, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    with _on_device(q, k=k, v=v, out=out, lse=lse, workspace=workspace):
        rc = load().fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), B, Hq, Hkv, Nq, Nkv, d, int(bool(causal)),
                               ctypes.c_float(scale), int(num_splits), ws_ptr, ws_bytes,
                               _stream_of(q))
    _check("fa_fwd_gqa", rc)
    return out, lse


def bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
        dq=None, dk=None, dv=None, workspace=None, phases: int = 7):
    """dq, dk, dv of L = sum(dout * O).  Returns (dq, dk, dv).

    ``phases`` selects the backward kernels to run (bit 0 prep, bit 1 main,
    bit 2 dQ convert); the default runs all three, as fa_bwd does.
    """
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_qkv(name, t, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, (B, H, N, d))
    need = bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
            int(bool(causal)), ctypes.c_float(scale), workspace.data_ptr(), nbytes, _stream_of(q))
    with _on_device(q, k=k, v=v, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv,
                    workspace=workspace):
        if phases == 7:
            _check("fa_bwd", load().fa_bwd(*args))
        else:
            _check("fa_bwd_phases", load().fa_bwd_phases(*args, int(phases)))
    return dq, dk, dv


def bwd_noalloc(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
                dq=None, dk=None, dv=None):
    """fa_bwd without a caller workspace: the library's fixed scratch array is
    used instead (for callers that cannot allocate device memory).  Calls
    that overlap on the GPU race on that array.  Returns (dq, dk, dv)."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_qkv(name, t, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, (B, H, N, d))
    with _on_device(q, k=k, v=v, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv):
        rc = load().fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, N, d, int(bool(causal)),
                                   ctypes.c_float(scale), _stream_of(q))
    _check("fa_bwd_noalloc", rc)
    return dq, dk, dv


def _check_block_mask(block_mask, N, device):
    nt = (N + 127) // 128
    if not isinstance(block_mask, torch.Tensor) or block_mask.device != device:
        raise ValueError("block_mask must be a tensor on %s" % device)
    if block_mask.dtype not in (torch.uint8, torch.bool) or tuple(block_mask.shape) != (nt, nt):
        raise ValueError("block_mask must be uint8 or bool of shape (%d, %d)" % (nt, nt))
    if not block_mask.is_contiguous():
        raise ValueError("block_mask must be contiguous")


def fwd_blocksparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None,
                    out=None, lse=None):
    """Block-sparse forward: key block c is visible to query block r when
    block_mask[r, c] is nonzero; blocks are 128 rows.  Returns (o, lse)."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_qkv(name, t, (B, H, N, d))
    _check_block_mask(block_mask, N, q.device)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv("out", out, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    with _on_device(q, k=k, v=v, out=out, lse=lse):
        rc = load().fa_fwd_blocksparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse.data_ptr(), B, H, N, d, int(bool(causal)),
                                       ctypes.c_float(scale), block_mask.data_ptr(),
                                       _stream_of(q))
    _check("fa_fwd_blocksparse", rc)
    return out, lse


def bwd_blocksparse(q, k, v, o, dout, lse, block_mask, causal: bool = False,
                    scale: float | None = None, dq=None, dk=None, dv=None, workspace=None):
    """dq, dk, dv of the block-sparse forward.  Returns (dq, dk, dv)."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_qkv(name, t, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    _check_block_mask(block_mask, N, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, (B, H, N, d))
    if workspace is None:
        workspace = torch.empty(bwd_workspace_size(B, H, N, d), dtype=torch.uint8,
                                device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    with _on_device(q, k=k, v=v, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv,
                    workspace=workspace):
        rc = load().fa_bwd_blocksparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       dout.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                       int(bool(causal)), ctypes.c_float(scale),
                                       block_mask.data_ptr(), workspace.data_ptr(), nbytes,
                                       _stream_of(q))
    _check("fa_bwd_blocksparse", rc)
    return dq, dk, dv


def fwd_fp8_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_fwd_fp8_workspace_size(B, H, N, d))


def fp8_workspace_offsets(B: int, H: int, N: int, d: int):
    """Byte offsets of (q8, k8, vt8, amax) in the FP8 workspace."""
    off = (ctypes.c_size_t * 4)()
    _check("fa_fp8_workspace_offsets", load().fa_fp8_workspace_offsets(B, H, N, d, off))
    return tuple(int(x) for x in off)


def _fp8_workspace(workspace, B, H, N, d, device):
    need = fwd_fp8_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    return workspace, workspace.numel() * workspace.element_size()


def fp8_quantize(q, k, v, hadamard: bool = True, workspace=None):
    """Quantise bf16 q, k, v to the FP8 workspace (see fa_fp8_quantize).
    Returns the workspace (uint8 tensor)."""
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_qkv(name, t, (B, H, N, d))
    workspace, nbytes = _fp8_workspace(workspace, B, H, N, d, q.device)
    with _on_device(q, k=k, v=v, workspace=workspace):
        rc = load().fa_fp8_quantize(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, N, d,
                                    int(bool(hadamard)), workspace.data_ptr(), nbytes,
                                    _stream_of(q))
    _check("fa_fp8_quantize", rc)
    return workspace


def fwd_fp8_quantized(workspace, B, H, N, d, causal: bool = False, scale: float | None = None,
                      hadamard: bool = True, out=None, lse=None):
    """FP8 attention over a workspace written by fp8_quantize.  Returns (o, lse)."""
    scale = default_scale(d) if scale is None else float(scale)
    dev = workspace.device
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _check_qkv("out", out, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    with _on_device(workspace, out=out, lse=lse):
        rc = load().fa_fwd_fp8_quantized(out.data_ptr(), lse.data_ptr(), B, H, N, d,
                                         int(bool(causal)), ctypes.c_float(scale),
                                         int(bool(hadamard)), workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_of(out))
    _check("fa_fwd_fp8_quantized", rc)
    return out, lse


def fwd_fp8(q, k, v, causal: bool = False, scale: float | None = None, hadamard: bool = True,
            out=None, lse=None, workspace=None):
    """FP8 forward pass (quantise, then attention).  Returns (o, lse)."""
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_qkv(name, t, (B, H, N, d))
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_qkv("out", out, (B, H, N, d))
    _check_qkv("lse", lse, (B, H, N), torch.float32)
    workspace, nbytes = _fp8_workspace(workspace, B, H, N, d, q.device)
    with _on_device(q, k=k, v=v, out=out, lse=lse, workspace=workspace):
        rc = load().fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), B, H, N, d, int(bool(causal)),
                               ctypes.c_float(scale), int(bool(hadamard)), workspace.data_ptr(),
                               nbytes, _stream_of(q))
    _check("fa_fwd_fp8", rc)
    return out, lse


def device_status(stream=None):
    """Synchronise the stream; return (code, site) and clear the status word."""
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream if stream is None else stream)
    site = ctypes.c_int(0)
    code = load().fa_device_status(s, ctypes.byref(site))
    return int(code), int(site.value)


FA_SITE_SELFTEST = 901


def selftest_timeout(timeout_us: int = 20000):
    """Launch the failure-detection self test on the current stream (see
    fa_selftest_timeout); read the result with device_status()."""
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _check("fa_selftest_timeout", load().fa_selftest_timeout(int(timeout_us), s))


FA_SITE_SELFTEST_BOUNDS = 902


def checks_enabled() -> bool:
    """True for the bounds-checked build of the library."""
    return bool(load().fa_checks_enabled())


def selftest_bounds():
    """Launch the bounds-check self test on the current stream (see
    fa_selftest_bounds); read the result with device_status()."""
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _check("fa_selftest_bounds", load().fa_selftest_bounds(s))


def check_device_status(stream=None):
    code, site = device_status(stream)
    if code != FA_OK:
        raise FaError("kernel", code, status_string(code) + " (site %d)" % site)


def fwd_schedule(B: int, H: int, N: int, causal: bool, num_ctas: int = 152):
    """The forward kernel's work list: (bh, pair, cost, cta) per item, in list order
    (cta -1: claimed from the work counter at run time)."""
    lib = load()
    n = lib.fa_fwd_schedule(B, H, N, int(bool(causal)), int(num_ctas), None, None, None, None, 0)
    if n < 0:
        _check("fa_fwd_schedule", n)
    bh = (ctypes.c_int * n)()
    pr = (ctypes.c_int * n)()
    cost = (ctypes.c_int * n)()
    cta = (ctypes.c_int * n)()
    lib.fa_fwd_schedule(B, H, N, int(bool(causal)), int(num_ctas), bh, pr, cost, cta, n)
    return list(zip(bh, pr, cost, cta))


def snake_assign(n: int, workers: int):
    """The kernels' static assignment of n listed items to persistent workers."""
    out = (ctypes.c_int * max(n, 1))()
    _check("fa_snake_assign", load().fa_snake_assign(int(n), int(workers), out))
    return list(out)[:n]
