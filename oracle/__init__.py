"""CPU oracle for group-wise low-bit weight quantization -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding in ``weight_only_bit_group_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``oracle.c`` (plain C, one IEEE op per statement, no
fusion).  This module only compiles that file with gcc and marshals numpy arrays
in and out through ctypes.  Every function returns fresh numpy arrays; bf16 and
fp16 values are carried as their uint16 bit patterns.

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` against
hand-worked values, closed forms, brute force or independent library conversions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

TIE_HALF_EVEN = 0
TIE_PAGE_LITERAL = 1

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, strict IEEE flags)."""
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            sig = {
                "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_floor_log2": (I, [ctypes.c_float]),
                "orc_e2m1_code": (I, [ctypes.c_float, I]),
                "orc_pack_int32": (None, [P, I64, I64, I, P]),
                "orc_gptq_quantize": (None, [P, I64, I64, I, I, P, P, P, P, P]),
                "orc_gptq_quantize_f32": (None, [P, I64, I64, I, I, P, P, P, P, P]),
                "orc_gptq_dequantize": (None, [P, P, P, I64, I64, I, I, I, P]),
                "orc_mxfp4_quantize_f32": (None, [P, I64, I64, I, P, P]),
                "orc_mxfp4_quantize": (None, [P, I64, I64, I, P, P]),
                "orc_mxfp4_dequantize": (None, [P, P, I64, I64, P]),
                "orc_awq_prepare_scales": (None, [P, I64, P, I, P, P]),
                "orc_awq_search": (None, [P, I64, I64, P, P, I, I, I, P, P, P, P]),
                "orc_quant_snr": (None, [P, P, I, I, I64, I64, P, P]),
                "orc_awq_fold": (None, [P, I64, I64, P, I, I, P]),
                "orc_uintx_packed_bytes": (I64, [I64, I]),
                "orc_uintx_pack": (None, [P, I64, I, P]),
                "orc_uintx_unpack": (None, [P, I64, I, P]),
                "orc_uintx_quantize": (None, [P, I64, I64, I, I, P, P, P, P]),
                "orc_uintx_quantize_dt": (None, [P, I, I64, I64, I, I, P, P, P, P]),
                "orc_uintx_dequantize_dt": (None, [P, P, I, P, I64, I64, I, I, P]),
                "orc_uintx_dequantize": (None, [P, P, P, I64, I64, I, I, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _is_torch(a) -> bool:
    return type(a).__module__.startswith("torch")


def _u16(a) -> np.ndarray:
    """Accept a numpy uint16 array or a torch bf16/fp16 tensor (bit view)."""
    if _is_torch(a):
        import torch  # only for the bit view of a caller's tensor

        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


# --------------------------------------------------------------------------- scalars
def bf16_to_f32(h: int) -> float:
    return _load().orc_bf16_to_f32(h)


def f32_to_bf16(x: float) -> int:
    return _load().orc_f32_to_bf16(x)


def f16_to_f32(h: int) -> float:
    return _load().orc_f16_to_f32(h)


def f32_to_f16(x: float) -> int:
    return _load().orc_f32_to_f16(x)


def floor_log2(x: float) -> int:
    return _load().orc_floor_log2(x)


def e2m1_code(v: float, tie_mode: int = TIE_HALF_EVEN) -> int:
    return _load().orc_e2m1_code(v, tie_mode)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift, no rounding)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------- GPTQ
def pack_int32(codes: np.ndarray, dim: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int32)
    k, n = codes.shape
    out = np.zeros((k // 8, n) if dim == 0 else (k, n // 8), dtype=np.int32)
    _load().orc_pack_int32(_p(codes), k, n, dim, _p(out))
    return out


def gptq_quantize(w, group: int = 128, sym: bool = True):
    """-> (qweight i32 [K/8,N], qzeros i32 [K/g,N/8], scales f16-bits [K/g,N], g_idx, snr_db)."""
    w = _u16(w)
    n, k = w.shape
    g = k // group
    qw = np.zeros((k // 8, n), np.int32)
    qz = np.zeros((g, n // 8), np.int32)
    sc = np.zeros((g, n), np.uint16)
    gi = np.zeros((k,), np.int32)
    snr = ctypes.c_double()
    _load().orc_gptq_quantize(_p(w), n, k, group, int(sym), _p(qw), _p(qz), _p(sc), _p(gi),
                              ctypes.byref(snr))
    return qw, qz, sc, gi, snr.value


def gptq_quantize_f32(w: np.ndarray, group: int = 128, sym: bool = True):
    """The same from a binary32 weight (an fp16 or fp32 input after the page's
    w.float()).  -> as gptq_quantize."""
    w = np.ascontiguousarray(w, np.float32)
    n, k = w.shape
    g = k // group
    qw = np.zeros((k // 8, n), np.int32)
    qz = np.zeros((g, n // 8), np.int32)
    sc = np.zeros((g, n), np.uint16)
    gi = np.zeros((k,), np.int32)
    snr = ctypes.c_double()
    _load().orc_gptq_quantize_f32(_p(w), n, k, group, int(sym), _p(qw), _p(qz), _p(sc), _p(gi),
                                  ctypes.byref(snr))
    return qw, qz, sc, gi, snr.value


def gptq_dequantize(qweight, qzeros, scales, n: int, k: int, group: int, sym: bool,
                    out_kn: bool = False) -> np.ndarray:
    qweight = np.ascontiguousarray(qweight, np.int32)
    qzeros = np.ascontiguousarray(qzeros, np.int32)
    scales = _u16(scales)
    out = np.zeros((k, n) if out_kn else (n, k), np.float32)
    _load().orc_gptq_dequantize(_p(qweight), _p(qzeros), _p(scales), n, k, group, int(sym),
                                int(out_kn), _p(out))
    return out


def gptq_linear(x, qweight, qzeros, scales, n: int, k: int, group: int, sym: bool):
    """The consumer of an exported GPTQ checkpoint (export_gptq_cpu.py module
    docstring: vLLM's W4A16 uint4b8 layer): y = x @ deq(W)^T with deq the
    dequantized weight [n, k] of the docstring's rule and x bf16 [m, k].  Every
    product x * deq is exact in binary64 and the sums are binary64 (matmul), so
    this is the exact result up to binary64 rounding.  Also returns
    sum_k |x * deq| per output, the scale of the rounding error bound of any
    binary32 evaluation.  -> (y f64 [m, n], mag f64 [m, n])."""
    deq = gptq_dequantize(qweight, qzeros, scales, n, k, group, sym).astype(np.float64)
    xf = bf16_bits_to_f32(_u16(x)).astype(np.float64)
    if xf.ndim == 1:
        xf = xf.reshape(1, -1)
    return xf @ deq.T, np.abs(xf) @ np.abs(deq).T


# --------------------------------------------------------------------------- MXFP4
def mxfp4_quantize(w, tie_mode: int = TIE_HALF_EVEN):
    """bf16 [N,K] -> (packed u8 [N,K/2], e8m0 u8 [N,K/32])."""
    w = _u16(w)
    n, k = w.shape
    packed = np.zeros((n, k // 2), np.uint8)
    e8 = np.zeros((n, k // 32), np.uint8)
    _load().orc_mxfp4_quantize(_p(w), n, k, tie_mode, _p(packed), _p(e8))
    return packed, e8


def mxfp4_quantize_f32(w: np.ndarray, tie_mode: int = TIE_HALF_EVEN):
    w = np.ascontiguousarray(w, np.float32)
    n, k = w.shape
    packed = np.zeros((n, k // 2), np.uint8)
    e8 = np.zeros((n, k // 32), np.uint8)
    _load().orc_mxfp4_quantize_f32(_p(w), n, k, tie_mode, _p(packed), _p(e8))
    return packed, e8


def mxfp4_dequantize(packed, e8m0) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    e8m0 = np.ascontiguousarray(e8m0, np.uint8)
    n = packed.shape[0]
    k = packed.shape[1] * 2
    out = np.zeros((n, k), np.float32)
    _load().orc_mxfp4_dequantize(_p(packed), _p(e8m0), n, k, _p(out))
    return out


def mxfp4_linear(x, packed, e8m0):
    """The consumer of MXFP4 weights (the drafter served quantized: y = x @ deq(W)^T)
    with deq from dequantize_mxfp4 and x bf16 [m, k]; every product is exact in
    binary64 and the sums are binary64.  -> (y f64 [m, n], sum_k |x deq| f64 [m, n])."""
    deq = mxfp4_dequantize(packed, e8m0).astype(np.float64)
    xf = bf16_bits_to_f32(_u16(x)).astype(np.float64)
    if xf.ndim == 1:
        xf = xf.reshape(1, -1)
    return xf @ deq.T, np.abs(xf) @ np.abs(deq).T


# --------------------------------------------------------------------------- AWQ
def awq_prepare_scales(a: np.ndarray, alphas):
    a = np.ascontiguousarray(a, np.float32)
    al = np.ascontiguousarray(alphas, np.float32)
    k = a.shape[0]
    s = np.zeros((al.shape[0], k), np.float32)
    ac = np.zeros((k,), np.float32)
    _load().orc_awq_prepare_scales(_p(a), k, _p(al), al.shape[0], _p(s), _p(ac))
    return s, ac


def awq_search(w, a: np.ndarray, alphas, max_rows: int = 2048,
               tie_mode: int = TIE_HALF_EVEN):
    """-> (best_s f32 [K], best_idx, best_alpha, errs f64 [n_alpha])."""
    w = _u16(w)
    n, k = w.shape
    a = np.ascontiguousarray(a, np.float32)
    al = np.ascontiguousarray(alphas, np.float32)
    best_s = np.zeros((k,), np.float32)
    bi = ctypes.c_int32()
    ba = ctypes.c_float()
    errs = np.zeros((al.shape[0],), np.float64)
    _load().orc_awq_search(_p(w), n, k, _p(a), _p(al), al.shape[0], max_rows, tie_mode,
                           _p(best_s), ctypes.byref(bi), ctypes.byref(ba), _p(errs))
    return best_s, bi.value, ba.value, errs


# --------------------------------------------------------------------------- SNR
def quant_snr(w, deq, deq_kn: bool = False):
    """-> (snr_db, rel_err).  deq: float32 array or bf16 bit patterns (uint16)."""
    w = _u16(w)
    n, k = w.shape
    if _is_torch(deq):
        import torch

        deq = _u16(deq) if deq.dtype == torch.bfloat16 else deq.detach().cpu().numpy()
    deq = np.ascontiguousarray(deq)
    is_bf16 = deq.dtype == np.uint16
    if not is_bf16:
        deq = np.ascontiguousarray(deq, np.float32)
    snr = ctypes.c_double()
    rel = ctypes.c_double()
    _load().orc_quant_snr(_p(w), _p(deq), int(is_bf16), int(deq_kn), n, k, ctypes.byref(snr),
                          ctypes.byref(rel))
    return snr.value, rel.value


# --------------------------------------------------------------------------- AWQ fold
def awq_fold(w, s, axis: int, op: int) -> np.ndarray:
    """(W.float() * s or / s) rounded to bf16, per column (axis 0, s [k]) or per
    row (axis 1, s [n]); op 0 multiplies, op 1 divides.  -> uint16 bf16 bits."""
    w = _u16(w)
    if w.ndim == 1:
        w = w.reshape(1, -1)
    n, k = w.shape
    s = np.ascontiguousarray(s, np.float32).reshape(-1)
    assert s.size == (k if axis == 0 else n)
    out = np.empty_like(w)
    _load().orc_awq_fold(_p(w), n, k, _p(s), axis, op, _p(out))
    return out


# --------------------------------------------------------------------------- uintx
def uintx_packed_bytes(numel: int, nbits: int) -> int:
    return _load().orc_uintx_packed_bytes(numel, nbits)


def uintx_pack(codes: np.ndarray, nbits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8).reshape(-1)
    out = np.zeros((uintx_packed_bytes(codes.size, nbits),), np.uint8)
    _load().orc_uintx_pack(_p(codes), codes.size, nbits, _p(out))
    return out


def uintx_unpack(packed: np.ndarray, nbits: int, numel: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, np.uint8)
    out = np.zeros((numel,), np.uint8)
    _load().orc_uintx_unpack(_p(packed), numel, nbits, _p(out))
    return out


def uintx_quantize(w, nbits: int, group: int = 64):
    """-> (packed u8, scale bf16-bits [N,K/g], zp u8 [N,K/g], codes u8 [N,K])."""
    w = _u16(w)
    n, k = w.shape
    packed = np.zeros((uintx_packed_bytes(n * k, nbits),), np.uint8)
    sc = np.zeros((n, k // group), np.uint16)
    zp = np.zeros((n, k // group), np.uint8)
    codes = np.zeros((n, k), np.uint8)
    _load().orc_uintx_quantize(_p(w), n, k, nbits, group, _p(packed), _p(sc), _p(zp), _p(codes))
    return packed, sc, zp, codes


def uintx_dequantize(packed, scale, zp, n: int, k: int, nbits: int, group: int = 64):
    """-> bf16 bit patterns [N,K]."""
    packed = np.ascontiguousarray(packed, np.uint8)
    scale = _u16(scale)
    zp = np.ascontiguousarray(zp, np.uint8)
    out = np.zeros((n, k), np.uint16)
    _load().orc_uintx_dequantize(_p(packed), _p(scale), _p(zp), n, k, nbits, group, _p(out))
    return out


# uintx in the weight's own dtype: dt 0 = binary32 (float32 arrays), 1 = bf16,
# 2 = binary16 (uint16 bit patterns for the 16-bit types)
def _dt_array(w, dt: int) -> np.ndarray:
    if _is_torch(w):
        import torch

        w = w.detach().cpu().contiguous()
        w = w.numpy() if w.dtype == torch.float32 else w.view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(w, np.float32 if dt == 0 else np.uint16)


def uintx_quantize_dt(w, dt: int, nbits: int, group: int = 64):
    """-> (packed u8, scale [N,K/g] in dt (float32 or uint16 bits), zp u8, codes u8)."""
    w = _dt_array(w, dt)
    n, k = w.shape
    packed = np.zeros((uintx_packed_bytes(n * k, nbits),), np.uint8)
    sc = np.zeros((n, k // group), np.float32 if dt == 0 else np.uint16)
    zp = np.zeros((n, k // group), np.uint8)
    codes = np.zeros((n, k), np.uint8)
    _load().orc_uintx_quantize_dt(_p(w), dt, n, k, nbits, group, _p(packed), _p(sc), _p(zp), _p(codes))
    return packed, sc, zp, codes


def uintx_dequantize_dt(packed, scale, dt: int, zp, n: int, k: int, nbits: int, group: int = 64):
    """-> [N,K] in dt (float32, or uint16 bit patterns)."""
    packed = np.ascontiguousarray(packed, np.uint8)
    scale = _dt_array(scale, dt)
    zp = np.ascontiguousarray(zp, np.uint8)
    out = np.zeros((n, k), np.float32 if dt == 0 else np.uint16)
    _load().orc_uintx_dequantize_dt(_p(packed), _p(scale), dt, _p(zp), n, k, nbits, group, _p(out))
    return out
