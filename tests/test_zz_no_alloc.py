"""awq_search_static_scratch: the AWQ search for callers that cannot allocate
device memory (code running inside another component's memory pool, framework
plug-ins that must not allocate on their threads, paths that must not risk the
synchronisation an allocation can cause).  It keeps its scratch in an array
built into the library instead of a caller workspace.

Checked here through the C ABI on two calls in a row (every call reuses the same
built-in array): bit-identical to the ordinary awq_search, which takes a
caller-allocated workspace and runs the same kernels in the same order, and
within the AWQ parity tolerance of the CPU oracle.  Around a call neither
torch's allocator nor the device's free memory changes, and out-of-range sizes
are refused before any launch.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle

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


def _outputs(k, n_alpha, dev):
    return (torch.empty(k, dtype=torch.float32, device=dev), torch.empty((), dtype=torch.int32, device=dev),
            torch.empty((), dtype=torch.float32, device=dev),
            torch.empty(n_alpha, dtype=torch.float64, device=dev))


def _call(f, w, a, alphas, max_rows, outs):
    n, k = w.shape
    al = (ctypes.c_float * len(alphas))(*[float(x) for x in alphas])
    best_s, best_idx, best_alpha, errs = outs
    return f(ctypes.c_void_p(w.data_ptr()), n, k, ctypes.c_void_p(a.data_ptr()), al, len(alphas),
             max_rows, 0, ctypes.c_void_p(best_s.data_ptr()), ctypes.c_void_p(best_idx.data_ptr()),
             ctypes.c_void_p(best_alpha.data_ptr()), ctypes.c_void_p(errs.data_ptr()),
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _host(outs):
    s, i, al, e = outs
    return s.cpu().numpy(), int(i), float(al), e.cpu().numpy()


CASES = [((6144, 4096), 31, 32, 1024), ((8192, 5120), 3, 4, 2048)]


def _case(shape, wseed, aseed, dev):
    if shape[1] == 5120:  # rows of the gate_up workload [34816, 5120]
        w = synth.outlier_blocks_bf16(shape[0], shape[1], 0.015, 0.01, 50.0, wseed, device=dev)
    else:
        w = synth.normal_bf16(shape, 0.02, wseed, device=dev)
    return w, synth.awq_activation(shape[1], aseed, dev)


@pytest.mark.parametrize("shape,wseed,aseed,max_rows", CASES)
def test_static_scratch_matches_workspace_version_and_oracle_twice(shape, wseed, aseed, max_rows):
    f = _fn()
    dev = torch.device("cuda")
    w, a = _case(shape, wseed, aseed, dev)
    ref = _host(wq.awq_search(w, a, synth.ALPHAS, max_rows))
    s_or, i_or, a_or, e_or = oracle.awq_search(w.cpu(), a.cpu().numpy(), synth.ALPHAS, max_rows)
    order = np.sort(e_or)
    margin = (order[1] - order[0]) / order[0]
    for _ in range(2):  # the second call runs on the first call's leftover scratch
        outs = _outputs(shape[1], len(synth.ALPHAS), dev)
        assert _call(f, w, a, synth.ALPHAS, max_rows, outs) == 0
        torch.cuda.synchronize()
        s, i, al, e = _host(outs)
        # the same kernels over the same data in the same order: the same bits
        assert np.array_equal(e.view(np.uint64), ref[3].view(np.uint64))
        assert np.array_equal(s.view(np.uint32), ref[0].view(np.uint32))
        assert i == ref[1] and al == ref[2]
        # and the CPU oracle's search (binary64 sums) within the parity tolerance
        np.testing.assert_allclose(e, e_or, rtol=REL, atol=0)
        if margin > 1e-9:
            assert i == i_or and al == a_or
            np.testing.assert_allclose(s, s_or, rtol=2e-7, atol=0)


def test_static_scratch_allocates_no_device_memory():
    f = _fn()
    dev = torch.device("cuda")
    w, a = _case((4096, 4096), 41, 42, dev)
    outs = _outputs(4096, len(synth.ALPHAS), dev)
    assert _call(f, w, a, synth.ALPHAS, 2048, outs) == 0  # first call: lookups, lazy module loads
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated(dev)
    free_before, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        assert _call(f, w, a, synth.ALPHAS, 2048, outs) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated(dev) == torch_before
    free_after, _ = torch.cuda.mem_get_info(dev)
    assert free_after == free_before


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    f = _fn()
    k = 16416
    w = torch.zeros(32, k, dtype=torch.bfloat16, device="cuda")
    a = torch.ones(k, dtype=torch.float32, device="cuda")
    al = (ctypes.c_float * 2)(0.0, 1.0)
    out = torch.empty(k, dtype=torch.float32, device="cuda")
    st = f(ctypes.c_void_p(w.data_ptr()), 32, k, ctypes.c_void_p(a.data_ptr()), al, 2, 16, 0,
           ctypes.c_void_p(out.data_ptr()), None, None, None, None)
    assert st == 2  # WQ_ERR_BAD_SHAPE: 16416 > 16384 columns, nothing launched
    # 17 alphas: refused with the code awq_search gives for the same input
    w2 = torch.zeros(32, 64, dtype=torch.bfloat16, device="cuda")
    a2 = torch.ones(64, dtype=torch.float32, device="cuda")
    al17 = (ctypes.c_float * 17)(*[i / 16 for i in range(17)])
    st = f(ctypes.c_void_p(w2.data_ptr()), 32, 64, ctypes.c_void_p(a2.data_ptr()), al17, 17, 16, 0,
           None, None, None, None, None)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    st_ws = wq.lib().awq_search(ctypes.c_void_p(w2.data_ptr()), 32, 64, ctypes.c_void_p(a2.data_ptr()), al17,
                                17, 16, 0, None, None, None, None, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                None)
    assert st == st_ws == 5  # WQ_ERR_UNSUPPORTED
