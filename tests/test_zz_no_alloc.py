"""awq_search_static_scratch: the AWQ search for callers that cannot allocate
device memory (code running inside another component's memory pool, framework
plug-ins that must not allocate on their threads, paths that must not risk the
synchronisation an allocation can cause).  It keeps its scratch in an array
built into the library instead of a caller workspace.

Checked here through the C ABI against the ordinary awq_search (which takes a
caller-allocated workspace), on two calls in a row, since every call reuses the
same built-in array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
REL = 1e-4  # the tolerance the AWQ parity tests use for the errors


def _fn():
    L = wq.lib()
    f = L.awq_search_static_scratch
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.restype = I
    f.argtypes = [P, I64, I64, P, P, I, I, I, P, P, P, P, P]
    return f


def _call(f, w, a, alphas, max_rows):
    n, k = w.shape
    al = (ctypes.c_float * len(alphas))(*[float(x) for x in alphas])
    best_s = torch.empty(k, dtype=torch.float32, device=w.device)
    best_idx = torch.empty((), dtype=torch.int32, device=w.device)
    best_alpha = torch.empty((), dtype=torch.float32, device=w.device)
    errs = torch.empty(len(alphas), dtype=torch.float64, device=w.device)
    st = f(ctypes.c_void_p(w.data_ptr()), n, k, ctypes.c_void_p(a.data_ptr()), al, len(alphas),
           max_rows, 0, ctypes.c_void_p(best_s.data_ptr()), ctypes.c_void_p(best_idx.data_ptr()),
           ctypes.c_void_p(best_alpha.data_ptr()), ctypes.c_void_p(errs.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, wq.lib().wq_status_string(st)
    torch.cuda.synchronize()
    return best_s.cpu(), int(best_idx), float(best_alpha), errs.cpu().numpy()


def test_static_scratch_matches_workspace_version_twice():
    f = _fn()
    dev = torch.device("cuda")
    cases = [(synth.normal_bf16((6144, 4096), 0.02, 31, device=dev), synth.awq_activation(4096, 32, dev), 1024),
             (synth.mxfp4_gate_up(device=dev)[:8192].contiguous(), synth.awq_activation(5120, 4, dev), 2048)]
    for w, a, max_rows in cases:
        ref_s, ref_i, ref_a, ref_e = wq.awq_search(w, a, synth.ALPHAS, max_rows)
        ref_s, ref_i, ref_a, ref_e = ref_s.cpu(), int(ref_i), float(ref_a), ref_e.cpu().numpy()
        for _ in range(2):  # the second call runs on the first call's leftover scratch
            s, i, al, e = _call(f, w, a, synth.ALPHAS, max_rows)
            np.testing.assert_allclose(e, ref_e, rtol=REL, atol=0)
            assert i == ref_i and al == ref_a
            np.testing.assert_allclose(s.numpy(), ref_s.numpy(), rtol=REL, atol=0)


def test_static_scratch_rejects_k_beyond_its_maximum():
    f = _fn()
    w = torch.zeros(32, 16416, dtype=torch.bfloat16, device="cuda")
    a = torch.ones(16416, dtype=torch.float32, device="cuda")
    al = (ctypes.c_float * 2)(0.0, 1.0)
    out = torch.empty(16416, dtype=torch.float32, device="cuda")
    st = f(ctypes.c_void_p(w.data_ptr()), 32, 16416, ctypes.c_void_p(a.data_ptr()), al, 2, 16, 0,
           ctypes.c_void_p(out.data_ptr()), None, None, None, None)
    assert st == 2  # WQ_ERR_BAD_SHAPE: 16416 > 16384 columns, nothing launched
