"""Python binding of libwqgb300.so (group-wise low-bit weight quantization on GB300).

Argument marshalling only: every step of every operation runs in the CUDA
kernels behind the C ABI declared in ``include/wqgb300.h``.  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: if the
library is not built, importing works but the first call raises.

Functions mirror the C entry points and take/return torch tensors on the GPU:

    gptq_quantize_sym / gptq_quantize_asym(w, group=128, snr=True)
    gptq_dequantize(qweight, qzeros, scales, n, k, group, sym, out_dtype, layout)
    mxfp4_quantize(w, tie_mode) / mxfp4_dequantize(packed, e8m0, out_dtype)
    awq_search(w, a, alphas, max_rows=2048, tie_mode)
    uintx_quantize(w, nbits, group=64) / uintx_dequantize(...)
    quant_snr(w, deq, layout)

Every function accepts preallocated outputs (``out=``-style keyword arguments)
so timed loops allocate nothing.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from ._build import LIB as _LIB_PATH

WQ_OK = 0
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
                "mxfp4_dequantize": (I, [P, P, I64, I64, I, P, P]),
                "awq_search": (I, [P, I64, I64, P, P, I, I, I, P, P, P, P, P, SZ, P]),
                "uintx_packed_bytes": (I64, [I64, I]),
                "uintx_quantize": (I, [P, I64, I64, I, I, P, P, P, P]),
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


def _u16(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype in (torch.bfloat16, torch.float16, torch.int16, torch.uint16), t.dtype
    assert t.is_contiguous(), "tensor must be contiguous"
    return t


def _bf16(t: torch.Tensor, what: str) -> torch.Tensor:
    """A bf16 operand (activations, bf16 scales): other 16-bit types would be read as
    bf16 bit patterns, so they are refused here."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{what} must be bfloat16, got {t.dtype}")
    assert t.is_contiguous(), f"{what} must be contiguous"
    return t


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


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
_WIDE = {torch.float32: WQ_DTYPE_F32, torch.float16: WQ_DTYPE_F16}


def _gptq_quantize(name, w, group, snr, qweight, qzeros, scales, g_idx, snr_db, ws):
    wide = w.dtype in _WIDE and w.dtype != torch.bfloat16
    if not wide:
        _u16(w)
    assert w.is_contiguous(), "tensor must be contiguous"
    n, k = w.shape
    g = k // group
    qweight = _empty((k // 8, n), torch.int32, w) if qweight is None else qweight
    qzeros = _empty((g, n // 8), torch.int32, w) if qzeros is None else qzeros
    scales = _empty((g, n), torch.float16, w) if scales is None else scales
    g_idx = _empty((k,), torch.int32, w) if g_idx is None else g_idx
    if snr:
        snr_db = _empty((), torch.float64, w) if snr_db is None else snr_db
        ws = workspace(WQ_OP_GPTQ_QUANTIZE, n, k, group, w.device) if ws is None else ws
    else:
        snr_db = None
    if wide:  # fp16 / fp32 weights: the binary32 path of gptq_quantize_ex
        st = lib().gptq_quantize_ex(_ptr(w), _WIDE[w.dtype], n, k, group, int(name == "gptq_quantize_sym"),
                                    _ptr(qweight), _ptr(qzeros), _ptr(scales), _ptr(g_idx), _ptr(snr_db),
                                    _ptr(ws), 0 if ws is None else ws.numel(), _stream(w.device))
    else:
        st = getattr(lib(), name)(_ptr(w), n, k, group, _ptr(qweight), _ptr(qzeros), _ptr(scales),
                                  _ptr(g_idx), _ptr(snr_db), _ptr(ws), 0 if ws is None else ws.numel(),
                                  _stream(w.device))
    _check(st, name)
    return {"qweight": qweight, "qzeros": qzeros, "scales": scales, "g_idx": g_idx,
            "snr_db": snr_db}


def gptq_quantize_sym(w, group=128, snr=True, *, qweight=None, qzeros=None, scales=None,
                      g_idx=None, snr_db=None, ws=None):
    """export_gptq_cpu.py quantize_sym on the GPU. w: bf16 [N, K] CUDA tensor."""
    return _gptq_quantize("gptq_quantize_sym", w, group, snr, qweight, qzeros, scales, g_idx,
                          snr_db, ws)


def gptq_quantize_asym(w, group=128, snr=True, *, qweight=None, qzeros=None, scales=None,
                       g_idx=None, snr_db=None, ws=None):
    """export_gptq_cpu.py quantize_asym on the GPU. w: bf16 [N, K] CUDA tensor."""
    return _gptq_quantize("gptq_quantize_asym", w, group, snr, qweight, qzeros, scales, g_idx,
                          snr_db, ws)


def gptq_dequantize(qweight, qzeros, scales, n, k, group=128, sym=True,
                    out_dtype=torch.bfloat16, layout="nk", *, out=None):
    lay = WQ_LAYOUT_NK if layout == "nk" else WQ_LAYOUT_KN
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    if out is None:
        out = _empty((n, k) if lay == WQ_LAYOUT_NK else (k, n), out_dtype, qweight)
    st = lib().gptq_dequantize(_ptr(qweight), _ptr(qzeros), _ptr(scales), n, k, group, int(sym),
                               dt, lay, _ptr(out), _stream(qweight.device))
    _check(st, "gptq_dequantize")
    return out


# ------------------------------------------------------------------ MXFP4
def mxfp4_quantize(w, tie_mode=WQ_TIE_HALF_EVEN, *, packed=None, e8m0=None):
    """quantize_dflash_mxfp4.py quantize_mxfp4 on the GPU -> (packed u8 [N,K/2], e8m0 u8 [N,K/32]).
    w: bf16, fp16 or fp32 [N, K]."""
    wide = w.dtype in (torch.float32, torch.float16)
    if not wide:
        _u16(w)
    assert w.is_contiguous(), "tensor must be contiguous"
    n, k = w.shape
    packed = _empty((n, k // 2), torch.uint8, w) if packed is None else packed
    e8m0 = _empty((n, k // 32), torch.uint8, w) if e8m0 is None else e8m0
    if wide:
        st = lib().mxfp4_quantize_ex(_ptr(w), _WIDE[w.dtype], n, k, tie_mode, _ptr(packed), _ptr(e8m0),
                                     _stream(w.device))
    else:
        st = lib().mxfp4_quantize(_ptr(w), n, k, tie_mode, _ptr(packed), _ptr(e8m0), _stream(w.device))
    _check(st, "mxfp4_quantize")
    return packed, e8m0


def mxfp4_dequantize(packed, e8m0, out_dtype=torch.float32, *, out=None):
    n, k = packed.shape[0], packed.shape[1] * 2
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    out = _empty((n, k), out_dtype, packed) if out is None else out
    st = lib().mxfp4_dequantize(_ptr(packed), _ptr(e8m0), n, k, dt, _ptr(out), _stream(packed.device))
    _check(st, "mxfp4_dequantize")
    return out


def awq_search(w, a, alphas, max_rows=2048, tie_mode=WQ_TIE_HALF_EVEN, *, best_s=None,
               best_idx=None, best_alpha=None, errs=None, ws=None):
    """quantize_dflash_mxfp4.py search_scale -> (best_s f32 [K], best_idx, best_alpha, errs f64)."""
    _u16(w)
    n, k = w.shape
    al = (ctypes.c_float * len(alphas))(*[float(x) for x in alphas])
    best_s = _empty((k,), torch.float32, w) if best_s is None else best_s
    best_idx = _empty((), torch.int32, w) if best_idx is None else best_idx
    best_alpha = _empty((), torch.float32, w) if best_alpha is None else best_alpha
    errs = _empty((len(alphas),), torch.float64, w) if errs is None else errs
    ws = workspace(WQ_OP_AWQ_SEARCH, n, k, len(alphas), w.device) if ws is None else ws
    st = lib().awq_search(_ptr(w), n, k, _ptr(a), al, len(alphas), max_rows, tie_mode,
                          _ptr(best_s), _ptr(best_idx), _ptr(best_alpha), _ptr(errs), _ptr(ws),
                          ws.numel(), _stream(w.device))
    _check(st, "awq_search")
    return best_s, best_idx, best_alpha, errs


# ------------------------------------------------------------------ uintx
def uintx_packed_bytes(numel: int, nbits: int) -> int:
    return int(lib().uintx_packed_bytes(numel, nbits))


def uintx_quantize(w, nbits, group=64, *, packed=None, scale=None, zp=None):
    """uintx_quant.py _quantize_impl + pack_uintx -> (packed u8, scale [N,K/g] in the weight's
    dtype, zp u8).  w: bf16, fp16 or fp32 [N, K]; the arithmetic runs in that dtype."""
    wide = w.dtype in (torch.float32, torch.float16)
    if not wide:
        _u16(w)
    assert w.is_contiguous(), "tensor must be contiguous"
    n, k = w.shape
    packed = _empty((uintx_packed_bytes(n * k, nbits),), torch.uint8, w) if packed is None else packed
    scale = _empty((n, k // group), w.dtype if wide else torch.bfloat16, w) if scale is None else scale
    zp = _empty((n, k // group), torch.uint8, w) if zp is None else zp
    if wide:
        st = lib().uintx_quantize_ex(_ptr(w), _WIDE[w.dtype], n, k, nbits, group, _ptr(packed), _ptr(scale),
                                     _ptr(zp), _stream(w.device))
    else:
        st = lib().uintx_quantize(_ptr(w), n, k, nbits, group, _ptr(packed), _ptr(scale), _ptr(zp),
                                  _stream(w.device))
    _check(st, "uintx_quantize")
    return packed, scale, zp


def uintx_dequantize(packed, scale, zp, n, k, nbits, group=64, out_dtype=torch.bfloat16, *,
                     out=None):
    """_dequantize_native.  A bf16 scale gives bf16 (or its exact binary32 widening,
    out_dtype); an fp16 / fp32 scale computes and returns in that dtype."""
    if scale.dtype in (torch.float32, torch.float16):
        out = torch.empty((n, k), dtype=scale.dtype, device=packed.device) if out is None else out
        _check(lib().uintx_dequantize_ex(_ptr(packed), _ptr(scale), _WIDE[scale.dtype], _ptr(zp), n, k, nbits,
                                         group, _ptr(out), _stream(packed.device)), "uintx_dequantize_ex")
        return out
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    out = _empty((n, k), out_dtype, packed) if out is None else out
    st = lib().uintx_dequantize(_ptr(packed), _ptr(scale), _ptr(zp), n, k, nbits, group, dt,
                                _ptr(out), _stream(packed.device))
    _check(st, "uintx_dequantize")
    return out


# ------------------------------------------------------------------ SNR
def gptq_linear(x, qweight, qzeros, scales, n, k, group=128, sym=True, out_dtype=torch.float32,
                *, out=None, ws=None):
    """y = x deq(W)^T for a decode batch (x bf16 [m, k], 1 <= m <= 8) straight from
    the GPTQ tensors; y binary32 or bf16 [m, n]."""
    _bf16(x, "x")
    x2 = x.view(1, -1) if x.dim() == 1 else x
    m = x2.shape[0]
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=x.device)
    nbytes = int(lib().gptq_linear_workspace_bytes(m, n))
    if ws is None:  # zeroed once, as the ABI requires; reusable afterwards
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=x.device)
    _check(lib().gptq_linear(_ptr(x2), m, _ptr(qweight), _ptr(qzeros), _ptr(scales), n, k, group,
                             int(sym), dt, _ptr(out), _ptr(ws), ws.numel(), _stream(x.device)),
           "gptq_linear")
    return out


def gptq_gemm(x, qweight, qzeros, scales, n, k, group=128, sym=True, out_dtype=torch.float32,
              *, out=None):
    """y = x deq(W)^T on the tensor cores for prefill batches (x bf16 [m, k], any
    m >= 1) straight from the GPTQ tensors; y binary32 or bf16 [m, n]."""
    _bf16(x, "x")
    x2 = x.view(1, -1) if x.dim() == 1 else x
    m = x2.shape[0]
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=x.device)
    _check(lib().gptq_gemm(_ptr(x2), m, _ptr(qweight), _ptr(qzeros), _ptr(scales), n, k, group,
                           int(sym), dt, _ptr(out), _stream(x.device)), "gptq_gemm")
    return out


def uintx_gemm(x, packed, scale, zp, n, k, nbits, group=64, out_dtype=torch.float32, *, out=None):
    """uintx_quant.py forward on the tensor cores: y = x deq(W)^T with deq the
    page's bf16 values (x bf16 [m, k], any m >= 1); y binary32 or bf16 [m, n]."""
    _bf16(x, "x")
    _bf16(scale, "scale (uintx_gemm takes the bf16 weights' scales)")
    x2 = x.view(1, -1) if x.dim() == 1 else x
    m = x2.shape[0]
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=x.device)
    _check(lib().uintx_gemm(_ptr(x2), m, _ptr(packed), _ptr(scale), _ptr(zp), n, k, nbits, group, dt,
                            _ptr(out), _stream(x.device)), "uintx_gemm")
    return out


def mxfp4_linear(x, packed, e8m0, out_dtype=torch.float32, *, out=None):
    """y = x deq(W)^T for a decode batch (x bf16 [m, k], 1 <= m <= 8) straight from
    the MXFP4 codes [n, k/2] and E8M0 bytes [n, k/32]; y binary32 or bf16 [m, n]."""
    _bf16(x, "x")
    x2 = x.view(1, -1) if x.dim() == 1 else x
    m, k = x2.shape
    n = packed.shape[0]
    dt = WQ_DTYPE_BF16 if out_dtype == torch.bfloat16 else WQ_DTYPE_F32
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=x.device)
    _check(lib().mxfp4_linear(_ptr(x2), m, _ptr(packed), _ptr(e8m0), n, k, dt, _ptr(out),
                              _stream(x.device)), "mxfp4_linear")
    return out


def awq_fold(w, s, axis: int = 0, op: int = 0, *, out=None):
    """quantize_dflash_mxfp4.py main()'s fold on the GPU: (w.float() * s or / s)
    rounded to bf16, s per column (axis 0, [K]) or per row (axis 1, [N]); op 0
    multiplies, op 1 divides.  out may be w (in place).  w: bf16 [N, K] or [K]."""
    _u16(w)
    w2 = w.view(1, -1) if w.dim() == 1 else w
    n, k = w2.shape
    assert s.dtype == torch.float32 and s.is_contiguous()
    if out is None:
        out = torch.empty_like(w)
    _check(lib().awq_fold(_ptr(w), n, k, _ptr(s), axis, op, _ptr(out), _stream(w.device)), "awq_fold")
    return out


def quant_snr(w, deq, layout="nk", *, snr_db=None, rel_err=None, ws=None):
    """Reconstruction SNR (dB) and relative error of deq against w -> two 0-dim f64 tensors."""
    _u16(w)
    n, k = w.shape
    lay = WQ_LAYOUT_NK if layout == "nk" else WQ_LAYOUT_KN
    dt = WQ_DTYPE_BF16 if deq.dtype == torch.bfloat16 else WQ_DTYPE_F32
    snr_db = _empty((), torch.float64, w) if snr_db is None else snr_db
    rel_err = _empty((), torch.float64, w) if rel_err is None else rel_err
    ws = workspace(WQ_OP_QUANT_SNR, n, k, 0, w.device) if ws is None else ws
    st = lib().quant_snr(_ptr(w), _ptr(deq), dt, lay, n, k, _ptr(snr_db), _ptr(rel_err), _ptr(ws),
                         ws.numel(), _stream(w.device))
    _check(st, "quant_snr")
    return snr_db, rel_err
