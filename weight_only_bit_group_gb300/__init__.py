"""Python binding of libwqgb300.so (group-wise low-bit weight quantization on GB300).

Argument marshalling only: every step of every operation runs in the CUDA
kernels behind the C ABI declared in ``include/wqgb300.h``.  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: if the
library is not built, importing works but the first call raises.

Functions mirror the C entry points and take/return torch tensors on the GPU:

    gptq_quantize_sym / gptq_quantize_asym(w, group=128, snr=True)
    gptq_dequantize(qweight, qzeros, scales, n, k, group, sym, out_dtype, layout)
    mxfp4_quantize(w, tie_mode, err=False) / mxfp4_dequantize(packed, e8m0, out_dtype)
    awq_search(w, a, alphas, max_rows=2048, tie_mode)
    uintx_quantize(w, nbits, group=64, err=False) / uintx_dequantize(...)
    quant_snr(w, deq, layout)

Every function accepts preallocated outputs (``out=``-style keyword arguments)
so timed loops allocate nothing.  Every tensor handed to the library -- input,
output or workspace -- is checked here for dtype, element count, contiguity and
device before the call, because the kernels size their reads and writes from the
shape arguments alone: a wrong buffer would otherwise be read or written past
its end.  Violations raise TypeError (dtype) or ValueError (the rest) and
nothing is launched.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

import torch

from ._build import LIB as _LIB_PATH

WQ_OK = 0
WQ_ERR_DEVICE_TIMEOUT = 8
WQ_DTYPE_F32 = 0
WQ_DTYPE_BF16 = 1
WQ_DTYPE_F16 = 2
WQ_LAYOUT_NK = 0
WQ_LAYOUT_KN = 1
WQ_TIE_HALF_EVEN = 0
WQ_TIE_PAGE_LITERAL = 1
WQ_OP_GPTQ_QUANTIZE = 0
WQ_OP_QUANT_SNR = 1
WQ_OP_AWQ_SEARCH = 2
WQ_OP_MXFP4_ERR = 3
WQ_OP_UINTX_ERR = 4

_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                       "wqgb300.h")
_lock = threading.Lock()
_lib = None


class WqError(RuntimeError):
    def __init__(self, status: int, name: str):
        msg = _lib.wq_status_string(status).decode()
        if status == 7:
            msg += ": " + _lib.wq_last_cuda_error().decode()
        super().__init__(f"{name} failed with status {status} ({msg})")
        self.status = status


def header_symbols() -> list[str]:
    """Names of the functions declared in include/wqgb300.h."""
    text = open(_HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**([a-z_0-9]+)\s*\(", text, flags=re.M)


def lib():
    """The loaded ctypes library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; "
                    "g.build()'` (nvcc, sm_103a) first; there is no CPU fallback")
            L = ctypes.CDLL(_LIB_PATH)
            P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            sig = {
                "wq_status_string": (ctypes.c_char_p, [I]),
                "wq_last_cuda_error": (ctypes.c_char_p, []),
                "wq_version": (ctypes.c_char_p, []),
                "wq_device_status": (I, []),
                "wq_workspace_bytes": (SZ, [I, I64, I64, I]),
                "gptq_quantize_sym": (I, [P, I64, I64, I, P, P, P, P, P, P, SZ, P]),
                "gptq_quantize_asym": (I, [P, I64, I64, I, P, P, P, P, P, P, SZ, P]),
                "gptq_dequantize": (I, [P, P, P, I64, I64, I, I, I, I, P, P]),
                "mxfp4_quantize": (I, [P, I64, I64, I, P, P, P]),
                "mxfp4_quantize_err": (I, [P, I64, I64, I, P, P, P, P, P, SZ, P]),
                "mxfp4_dequantize": (I, [P, P, I64, I64, I, P, P]),
                "awq_search": (I, [P, I64, I64, P, P, I, I, I, P, P, P, P, P, SZ, P]),
                "uintx_packed_bytes": (I64, [I64, I]),
                "uintx_quantize": (I, [P, I64, I64, I, I, P, P, P, P]),
                "uintx_quantize_err": (I, [P, I64, I64, I, I, P, P, P, P, P, P, SZ, P]),
                "uintx_dequantize": (I, [P, P, P, I64, I64, I, I, I, P, P]),
                "quant_snr": (I, [P, P, I, I, I64, I64, P, P, P, SZ, P]),
                "awq_fold": (I, [P, I64, I64, P, I, I, P, P]),
                "gptq_linear_workspace_bytes": (SZ, [I64, I64]),
                "gptq_linear": (I, [P, I64, P, P, P, I64, I64, I, I, I, P, P, SZ, P]),
                "mxfp4_linear": (I, [P, I64, P, P, I64, I64, I, P, P]),
                "gptq_gemm": (I, [P, I64, P, P, P, I64, I64, I, I, I, P, P]),
                "gptq_quantize_ex": (I, [P, I, I64, I64, I, I, P, P, P, P, P, P, SZ, P]),
                "mxfp4_quantize_ex": (I, [P, I, I64, I64, I, P, P, P]),
                "uintx_quantize_ex": (I, [P, I, I64, I64, I, I, P, P, P, P]),
                "uintx_dequantize_ex": (I, [P, P, I, P, I64, I64, I, I, P, P]),
                "uintx_gemm": (I, [P, I64, P, P, P, I64, I64, I, I, I, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, name: str):
    if status != WQ_OK:
        raise WqError(status, name)


# ------------------------------------------------------------------ argument checks
_OUT_DTYPES = {torch.float32: WQ_DTYPE_F32, torch.bfloat16: WQ_DTYPE_BF16}
_WIDE = {torch.float32: WQ_DTYPE_F32, torch.float16: WQ_DTYPE_F16}


def _names(dtypes) -> str:
    return " or ".join(str(d).replace("torch.", "") for d in dtypes)


def _arg(t, what: str, dtypes, numel=None, optional=False):
    """Check one tensor argument's dtype, element count and contiguity (`numel`
    None skips the count).  Devices are checked afterwards for all tensors of a
    call at once (_on_device), so that every other mistake is reported first."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{what} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor, got {type(t).__name__}")
    dts = dtypes if isinstance(dtypes, (tuple, list)) else (dtypes,)
    if t.dtype not in dts:
        raise TypeError(f"{what} must be {_names(dts)}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{what} must hold {numel} elements, got {t.numel()} (shape {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t


def _on_device(dev, **tensors):
    """Every tensor of the call is a CUDA tensor on `dev` (the last check before
    the library is called)."""
    for what, t in tensors.items():
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"{what} must be a CUDA tensor, got device {t.device}")
        if t.device != dev:
            raise ValueError(f"{what} is on {t.device}, expected {dev}")


def _matrix(t, what: str, dtypes):
    """A 2-D operand whose shape defines n, k."""
    _arg(t, what, dtypes)
    if t.dim() != 2:
        raise ValueError(f"{what} must be 2-D [n, k], got shape {tuple(t.shape)}")
    return t


def _out_code(dtype, what: str) -> int:
    if dtype not in _OUT_DTYPES:
        raise TypeError(f"{what}: the library writes float32 or bfloat16 outputs, not {dtype}")
    return _OUT_DTYPES[dtype]


def _out(t, what: str, dtype, shape, device):
    """A caller-supplied output buffer (checked) or a fresh one on `device`."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _arg(t, what, dtype, math.prod(shape))


def _ws(ws, nbytes: int, device):
    """A caller workspace (uint8, contiguous, at least nbytes) or a fresh one."""
    if ws is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    _arg(ws, "ws", torch.uint8)
    if ws.numel() < nbytes:
        raise ValueError(f"ws must hold at least {nbytes} bytes, got {ws.numel()}")
    return ws


def _layout(layout: str) -> int:
    if layout not in ("nk", "kn"):
        raise ValueError(f"layout must be 'nk' or 'kn', got {layout!r}")
    return WQ_LAYOUT_NK if layout == "nk" else WQ_LAYOUT_KN


def device_status() -> int:
    """Read and clear the device status word of the current device (wq_device_status):
    WQ_OK, or WQ_ERR_DEVICE_TIMEOUT if a bounded device-side wait ran out since the
    last read.  Synchronises with the legacy default stream."""
    return int(lib().wq_device_status())


def workspace_bytes(op: int, n: int, k: int, arg: int = 0) -> int:
    return int(lib().wq_workspace_bytes(op, n, k, arg))


def workspace(op: int, n: int, k: int, arg: int = 0, device="cuda") -> torch.Tensor:
    nbytes = max(workspace_bytes(op, n, k, arg), 256)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ GPTQ
def _gptq_quantize(name, w, group, snr, qweight, qzeros, scales, g_idx, snr_db, ws):
    _matrix(w, "w", (torch.bfloat16, torch.float16, torch.float32))
    wide = w.dtype != torch.bfloat16
    n, k = w.shape
    dev = w.device
    g = k // group if group > 0 else 0
    qweight = _out(qweight, "qweight", torch.int32, (k // 8, n), dev)
    qzeros = _out(qzeros, "qzeros", torch.int32, (g, n // 8), dev)
    scales = _out(scales, "scales", torch.float16, (g, n), dev)
    g_idx = _out(g_idx, "g_idx", torch.int32, (k,), dev)
    if snr:
        snr_db = _out(snr_db, "snr_db", torch.float64, (), dev)
        ws = _ws(ws, workspace_bytes(WQ_OP_GPTQ_QUANTIZE, n, k, group), dev)
    else:
        snr_db = None
        ws = None
    _on_device(dev, w=w, qweight=qweight, qzeros=qzeros, scales=scales, g_idx=g_idx, snr_db=snr_db, ws=ws)
    nws = 0 if ws is None else ws.numel()
    if wide:  # fp16 / fp32 weights: the binary32 path of gptq_quantize_ex
        st = lib().gptq_quantize_ex(_ptr(w), _WIDE[w.dtype], n, k, group, int(name == "gptq_quantize_sym"),
                                    _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), _ptr(snr_db),
                                    _ptr(ws), nws, _stream(dev))
    else:
        st = getattr(lib(), name)(_ptr(w), n, k, group, _ptr(qweight), _ptr(qzeros), _ptr(scales),
                                  _ptr(g_idx), _ptr(snr_db), _ptr(ws), nws, _stream(dev))
    _check(st, name)
    return {"qweight": qweight, "qzeros": qzeros, "scales": scales, "g_idx": g_idx,
            "snr_db": snr_db}


def gptq_quantize_sym(w, group=128, snr=True, *, qweight=None, qzeros=None, scales=None,
                      g_idx=None, snr_db=None, ws=None):
    """export_gptq_cpu.py quantize_sym on the GPU. w: bf16, fp16 or fp32 [N, K] CUDA tensor."""
    return _gptq_quantize("gptq_quantize_sym", w, group, snr, qweight, qzeros, scales, g_idx,
                          snr_db, ws)


def gptq_quantize_asym(w, group=128, snr=True, *, qweight=None, qzeros=None, scales=None,
                       g_idx=None, snr_db=None, ws=None):
    """export_gptq_cpu.py quantize_asym on the GPU. w: bf16, fp16 or fp32 [N, K] CUDA tensor."""
    return _gptq_quantize("gptq_quantize_asym", w, group, snr, qweight, qzeros, scales, g_idx,
                          snr_db, ws)


def _gptq_tensors(qweight, qzeros, scales, n, k, group, sym):
    """The packed GPTQ tensors of an [n, k] weight (qzeros may be None for sym)."""
    g = k // group if group > 0 else 0
    _arg(qweight, "qweight", torch.int32, (k // 8) * n)
    dev = qweight.device
    _arg(scales, "scales", torch.float16, g * n)
    _arg(qzeros, "qzeros", torch.int32, g * (n // 8), optional=bool(sym))
    return dev


def gptq_dequantize(qweight, qzeros, scales, n, k, group=128, sym=True,
                    out_dtype=torch.bfloat16, layout="nk", *, out=None):
    lay = _layout(layout)
    dt = _out_code(out_dtype, "gptq_dequantize")
    dev = _gptq_tensors(qweight, qzeros, scales, n, k, group, sym)
    out = _out(out, "out", out_dtype, (n, k) if lay == WQ_LAYOUT_NK else (k, n), dev)
    _on_device(dev, qweight=qweight, qzeros=qzeros, scales=scales, out=out)
    st = lib().gptq_dequantize(_ptr(qweight), _ptr(qzeros), _ptr(scales), n, k, group, int(sym),
                               dt, lay, _ptr(out), _stream(dev))
    _check(st, "gptq_dequantize")
    return out


# ------------------------------------------------------------------ MXFP4
def mxfp4_quantize(w, tie_mode=WQ_TIE_HALF_EVEN, *, packed=None, e8m0=None, err=False,
                   snr_db=None, rel_err=None, ws=None):
    """quantize_dflash_mxfp4.py quantize_mxfp4 on the GPU -> (packed u8 [N,K/2], e8m0 u8 [N,K/32]).
    w: bf16, fp16 or fp32 [N, K].  With err=True (bf16 weights) the reconstruction
    error of the same pass is returned too: (packed, e8m0, snr_db, rel_err), the
    scalars as 0-dim float64 tensors."""
    _matrix(w, "w", (torch.bfloat16, torch.float16, torch.float32))
    wide = w.dtype != torch.bfloat16
    n, k = w.shape
    dev = w.device
    packed = _out(packed, "packed", torch.uint8, (n, k // 2), dev)
    e8m0 = _out(e8m0, "e8m0", torch.uint8, (n, k // 32), dev)
    if err:
        if wide:
            raise TypeError("mxfp4_quantize(err=True) takes bf16 weights")
        snr_db = _out(snr_db, "snr_db", torch.float64, (), dev)
        rel_err = _out(rel_err, "rel_err", torch.float64, (), dev)
        ws = _ws(ws, workspace_bytes(WQ_OP_MXFP4_ERR, n, k, 0), dev)
        _on_device(dev, w=w, packed=packed, e8m0=e8m0, snr_db=snr_db, rel_err=rel_err, ws=ws)
        st = lib().mxfp4_quantize_err(_ptr(w), n, k, tie_mode, _ptr(packed), _ptr(e8m0), _ptr(snr_db),
                                      _ptr(rel_err), _ptr(ws), ws.numel(), _stream(dev))
        _check(st, "mxfp4_quantize_err")
        return packed, e8m0, snr_db, rel_err
    _on_device(dev, w=w, packed=packed, e8m0=e8m0)
    if wide:
        st = lib().mxfp4_quantize_ex(_ptr(w), _WIDE[w.dtype], n, k, tie_mode, _ptr(packed), _ptr(e8m0),
                                     _stream(dev))
    else:
        st = lib().mxfp4_quantize(_ptr(w), n, k, tie_mode, _ptr(packed), _ptr(e8m0), _stream(dev))
    _check(st, "mxfp4_quantize")
    return packed, e8m0


def mxfp4_dequantize(packed, e8m0, out_dtype=torch.float32, *, out=None):
    dt = _out_code(out_dtype, "mxfp4_dequantize")
    _matrix(packed, "packed", torch.uint8)
    n, k = packed.shape[0], packed.shape[1] * 2
    dev = packed.device
    _arg(e8m0, "e8m0", torch.uint8, n * (k // 32))
    out = _out(out, "out", out_dtype, (n, k), dev)
    _on_device(dev, packed=packed, e8m0=e8m0, out=out)
    st = lib().mxfp4_dequantize(_ptr(packed), _ptr(e8m0), n, k, dt, _ptr(out), _stream(dev))
    _check(st, "mxfp4_dequantize")
    return out


def awq_search(w, a, alphas, max_rows=2048, tie_mode=WQ_TIE_HALF_EVEN, *, best_s=None,
               best_idx=None, best_alpha=None, errs=None, ws=None):
    """quantize_dflash_mxfp4.py search_scale -> (best_s f32 [K], best_idx, best_alpha, errs f64)."""
    _matrix(w, "w", torch.bfloat16)
    n, k = w.shape
    dev = w.device
    _arg(a, "a", torch.float32, k)
    na = len(alphas)
    al = (ctypes.c_float * max(na, 1))(*[float(x) for x in alphas])
    best_s = _out(best_s, "best_s", torch.float32, (k,), dev)
    best_idx = _out(best_idx, "best_idx", torch.int32, (), dev)
    best_alpha = _out(best_alpha, "best_alpha", torch.float32, (), dev)
    errs = _out(errs, "errs", torch.float64, (na,), dev)
    ws = _ws(ws, workspace_bytes(WQ_OP_AWQ_SEARCH, n, k, na), dev)
    _on_device(dev, w=w, a=a, best_s=best_s, best_idx=best_idx, best_alpha=best_alpha, errs=errs, ws=ws)
    st = lib().awq_search(_ptr(w), n, k, _ptr(a), al, na, max_rows, tie_mode,
                          _ptr(best_s), _ptr(best_idx), _ptr(best_alpha), _ptr(errs), _ptr(ws),
                          ws.numel(), _stream(dev))
    _check(st, "awq_search")
    return best_s, best_idx, best_alpha, errs


# ------------------------------------------------------------------ uintx
def uintx_packed_bytes(numel: int, nbits: int) -> int:
    return int(lib().uintx_packed_bytes(numel, nbits))


def uintx_quantize(w, nbits, group=64, *, packed=None, scale=None, zp=None, err=False,
                   snr_db=None, rel_err=None, ws=None):
    """uintx_quant.py _quantize_impl + pack_uintx -> (packed u8, scale [N,K/g] in the weight's
    dtype, zp u8).  w: bf16, fp16 or fp32 [N, K]; the arithmetic runs in that dtype.
    With err=True (bf16 weights) the reconstruction error of the page's bf16
    dequantized weight is returned too: (packed, scale, zp, snr_db, rel_err)."""
    _matrix(w, "w", (torch.bfloat16, torch.float16, torch.float32))
    wide = w.dtype != torch.bfloat16
    n, k = w.shape
    dev = w.device
    g = k // group if group > 0 else 0
    nbytes = uintx_packed_bytes(n * k, nbits)
    packed = _out(packed, "packed", torch.uint8, (max(nbytes, 0),), dev)
    scale = _out(scale, "scale", w.dtype, (n, g), dev)
    zp = _out(zp, "zp", torch.uint8, (n, g), dev)
    if err:
        if wide:
            raise TypeError("uintx_quantize(err=True) takes bf16 weights")
        snr_db = _out(snr_db, "snr_db", torch.float64, (), dev)
        rel_err = _out(rel_err, "rel_err", torch.float64, (), dev)
        ws = _ws(ws, workspace_bytes(WQ_OP_UINTX_ERR, n, k, nbits), dev)
        _on_device(dev, w=w, packed=packed, scale=scale, zp=zp, snr_db=snr_db, rel_err=rel_err, ws=ws)
        st = lib().uintx_quantize_err(_ptr(w), n, k, nbits, group, _ptr(packed), _ptr(scale), _ptr(zp),
                                      _ptr(snr_db), _ptr(rel_err), _ptr(ws), ws.numel(), _stream(dev))
        _check(st, "uintx_quantize_err")
        return packed, scale, zp, snr_db, rel_err
    _on_device(dev, w=w, packed=packed, scale=scale, zp=zp)
    if wide:
        st = lib().uintx_quantize_ex(_ptr(w), _WIDE[w.dtype], n, k, nbits, group, _ptr(packed), _ptr(scale),
                                     _ptr(zp), _stream(dev))
    else:
        st = lib().uintx_quantize(_ptr(w), n, k, nbits, group, _ptr(packed), _ptr(scale), _ptr(zp),
                                  _stream(dev))
    _check(st, "uintx_quantize")
    return packed, scale, zp


def uintx_dequantize(packed, scale, zp, n, k, nbits, group=64, out_dtype=torch.bfloat16, *,
                     out=None):
    """_dequantize_native.  A bf16 scale gives bf16 (or its exact binary32 widening,
    out_dtype); an fp16 / fp32 scale computes and returns in that dtype."""
    g = k // group if group > 0 else 0
    _arg(scale, "scale", (torch.bfloat16, torch.float16, torch.float32), n * g)
    dev = scale.device
    nbytes = uintx_packed_bytes(n * k, nbits)
    _arg(packed, "packed", torch.uint8, max(nbytes, 0))
    _arg(zp, "zp", torch.uint8, n * g)
    if scale.dtype in _WIDE:
        out = _out(out, "out", scale.dtype, (n, k), dev)
        _on_device(dev, packed=packed, scale=scale, zp=zp, out=out)
        _check(lib().uintx_dequantize_ex(_ptr(packed), _ptr(scale), _WIDE[scale.dtype], _ptr(zp), n, k, nbits,
                                         group, _ptr(out), _stream(dev)), "uintx_dequantize_ex")
        return out
    dt = _out_code(out_dtype, "uintx_dequantize")
    out = _out(out, "out", out_dtype, (n, k), dev)
    _on_device(dev, packed=packed, scale=scale, zp=zp, out=out)
    st = lib().uintx_dequantize(_ptr(packed), _ptr(scale), _ptr(zp), n, k, nbits, group, dt,
                                _ptr(out), _stream(dev))
    _check(st, "uintx_dequantize")
    return out


# ------------------------------------------------------------------ consumers
def _acts(x, k=None):
    """Activations x: bf16 [m, k] (or [k] for one row) -> the 2-D view and m."""
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16:
        raise TypeError(f"x must be bfloat16, got {getattr(x, 'dtype', type(x))}")
    x2 = x.view(1, -1) if x.dim() == 1 else x
    if x2.dim() != 2:
        raise ValueError(f"x must be [m, k], got shape {tuple(x.shape)}")
    if k is not None and x2.shape[1] != k:
        raise ValueError(f"x has {x2.shape[1]} columns, the weight has k = {k}")
    _arg(x2, "x", torch.bfloat16)
    return x2, x2.shape[0]


def gptq_linear(x, qweight, qzeros, scales, n, k, group=128, sym=True, out_dtype=torch.float32,
                *, out=None, ws=None):
    """y = x deq(W)^T for a decode batch (x bf16 [m, k], 1 <= m <= 8) straight from
    the GPTQ tensors; y binary32 or bf16 [m, n]."""
    x2, m = _acts(x, k)
    dt = _out_code(out_dtype, "gptq_linear")
    _gptq_tensors(qweight, qzeros, scales, n, k, group, sym)
    dev = x2.device
    out = _out(out, "out", out_dtype, (m, n), dev)
    nbytes = int(lib().gptq_linear_workspace_bytes(m, n))
    if ws is None:  # zeroed once, as the ABI requires; reusable afterwards
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
    else:
        _ws(ws, nbytes, dev)
    _on_device(dev, x=x2, qweight=qweight, qzeros=qzeros, scales=scales, out=out, ws=ws)
    _check(lib().gptq_linear(_ptr(x2), m, _ptr(qweight), _ptr(qzeros), _ptr(scales), n, k, group,
                             int(sym), dt, _ptr(out), _ptr(ws), ws.numel(), _stream(dev)),
           "gptq_linear")
    return out


def gptq_gemm(x, qweight, qzeros, scales, n, k, group=128, sym=True, out_dtype=torch.float32,
              *, out=None):
    """y = x deq(W)^T on the tensor cores for prefill batches (x bf16 [m, k], any
    m >= 1) straight from the GPTQ tensors; y binary32 or bf16 [m, n]."""
    x2, m = _acts(x, k)
    dt = _out_code(out_dtype, "gptq_gemm")
    _gptq_tensors(qweight, qzeros, scales, n, k, group, sym)
    dev = x2.device
    out = _out(out, "out", out_dtype, (m, n), dev)
    _on_device(dev, x=x2, qweight=qweight, qzeros=qzeros, scales=scales, out=out)
    _check(lib().gptq_gemm(_ptr(x2), m, _ptr(qweight), _ptr(qzeros), _ptr(scales), n, k, group,
                           int(sym), dt, _ptr(out), _stream(dev)), "gptq_gemm")
    return out


def uintx_gemm(x, packed, scale, zp, n, k, nbits, group=64, out_dtype=torch.float32, *, out=None):
    """uintx_quant.py forward on the tensor cores: y = x deq(W)^T with deq the
    page's bf16 values (x bf16 [m, k], any m >= 1); y binary32 or bf16 [m, n]."""
    g = k // group if group > 0 else 0
    if isinstance(scale, torch.Tensor) and scale.dtype != torch.bfloat16:
        raise TypeError(f"scale must be bfloat16 (uintx_gemm takes the bf16 weights' scales), got {scale.dtype}")
    x2, m = _acts(x, k)
    _arg(scale, "scale", torch.bfloat16, n * g)
    dt = _out_code(out_dtype, "uintx_gemm")
    dev = x2.device
    _arg(packed, "packed", torch.uint8, max(uintx_packed_bytes(n * k, nbits), 0))
    _arg(zp, "zp", torch.uint8, n * g)
    out = _out(out, "out", out_dtype, (m, n), dev)
    _on_device(dev, x=x2, packed=packed, scale=scale, zp=zp, out=out)
    _check(lib().uintx_gemm(_ptr(x2), m, _ptr(packed), _ptr(scale), _ptr(zp), n, k, nbits, group, dt,
                            _ptr(out), _stream(dev)), "uintx_gemm")
    return out


def mxfp4_linear(x, packed, e8m0, out_dtype=torch.float32, *, out=None):
    """y = x deq(W)^T for a decode batch (x bf16 [m, k], 1 <= m <= 8) straight from
    the MXFP4 codes [n, k/2] and E8M0 bytes [n, k/32]; y binary32 or bf16 [m, n]."""
    x2, m = _acts(x)
    k = x2.shape[1]
    dt = _out_code(out_dtype, "mxfp4_linear")
    dev = x2.device
    _matrix(packed, "packed", torch.uint8)
    n = packed.shape[0]
    _arg(packed, "packed", torch.uint8, n * (k // 2))
    _arg(e8m0, "e8m0", torch.uint8, n * (k // 32))
    out = _out(out, "out", out_dtype, (m, n), dev)
    _on_device(dev, x=x2, packed=packed, e8m0=e8m0, out=out)
    _check(lib().mxfp4_linear(_ptr(x2), m, _ptr(packed), _ptr(e8m0), n, k, dt, _ptr(out),
                              _stream(dev)), "mxfp4_linear")
    return out


def awq_fold(w, s, axis: int = 0, op: int = 0, *, out=None):
    """quantize_dflash_mxfp4.py main()'s fold on the GPU: (w.float() * s or / s)
    rounded to bf16, s per column (axis 0, [K]) or per row (axis 1, [N]); op 0
    multiplies, op 1 divides.  out may be w (in place).  w: bf16 [N, K] or [K]."""
    _arg(w, "w", torch.bfloat16)
    w2 = w.view(1, -1) if w.dim() == 1 else w
    if w2.dim() != 2:
        raise ValueError(f"w must be [n, k] or [k], got shape {tuple(w.shape)}")
    n, k = w2.shape
    if axis not in (0, 1):
        raise ValueError(f"axis must be 0 (columns) or 1 (rows), got {axis}")
    _arg(s, "s", torch.float32, k if axis == 0 else n)
    out = _out(out, "out", torch.bfloat16, tuple(w.shape), w.device)
    _on_device(w.device, w=w, s=s, out=out)
    _check(lib().awq_fold(_ptr(w), n, k, _ptr(s), axis, op, _ptr(out), _stream(w.device)), "awq_fold")
    return out


# ------------------------------------------------------------------ SNR
def quant_snr(w, deq, layout="nk", *, snr_db=None, rel_err=None, ws=None):
    """Reconstruction SNR (dB) and relative error of deq against w -> two 0-dim f64 tensors.
    w: bf16 [N, K]; deq: float32 or bfloat16, [N, K] (layout 'nk') or [K, N] ('kn')."""
    _matrix(w, "w", torch.bfloat16)
    n, k = w.shape
    dev = w.device
    lay = _layout(layout)
    _arg(deq, "deq", tuple(_OUT_DTYPES), n * k)
    dt = _OUT_DTYPES[deq.dtype]
    snr_db = _out(snr_db, "snr_db", torch.float64, (), dev)
    rel_err = _out(rel_err, "rel_err", torch.float64, (), dev)
    ws = _ws(ws, workspace_bytes(WQ_OP_QUANT_SNR, n, k, 0), dev)
    _on_device(dev, w=w, deq=deq, snr_db=snr_db, rel_err=rel_err, ws=ws)
    st = lib().quant_snr(_ptr(w), _ptr(deq), dt, lay, n, k, _ptr(snr_db), _ptr(rel_err), _ptr(ws),
                         ws.numel(), _stream(dev))
    _check(st, "quant_snr")
    return snr_db, rel_err
