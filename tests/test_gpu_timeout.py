"""The bounded-wait timeout paths of the kernels that wait on hardware events,
made to run without any fault or hang.

wq_set_wait_budget(site, 0) makes every wait of one class give up at its first
poll.  The kernel then stops its work, lets the copies and MMAs it already issued
complete (those drains keep their own budgets), frees what it holds and records
WQ_ERR_DEVICE_TIMEOUT, which wq_device_status() reports once and clears.  The
next call with the default budget must give the oracle's result and leave the
status at WQ_OK: the context stays usable.

  WQ_WAIT_GPTQ_STAGE  gptq_quant_kernel's waits on the mbarriers of its TMA loads
  WQ_WAIT_GEMM_MMA    the MMA-issuing thread of gptq_gemm / uintx_gemm: it gives up
                      before its first MMA and raises the CTA's abort flag; the
                      TMA thread drains the loads it issued, the dequant and
                      epilogue warps leave at their next wait, and TMEM is freed
                      after every tensor-core store has completed
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
WQ_WAIT_GPTQ_STAGE = 0
WQ_WAIT_GEMM_MMA = 1


def _budget(site: int, value: int) -> int:
    f = wq.lib().wq_set_wait_budget
    f.restype = ctypes.c_uint
    f.argtypes = [ctypes.c_int, ctypes.c_uint]
    return int(f(site, value))


class zero_budget:
    """Budget 0 for one wait site inside the block, the previous one restored after."""

    def __init__(self, site):
        self.site = site

    def __enter__(self):
        self.prev = _budget(self.site, 0)
        return self

    def __exit__(self, *exc):
        torch.cuda.synchronize()
        assert _budget(self.site, self.prev) == 0


def test_wait_budget_defaults_and_unknown_site():
    assert _budget(WQ_WAIT_GPTQ_STAGE, 1 << 22) == 1 << 22
    assert _budget(WQ_WAIT_GEMM_MMA, 512) == 512
    assert _budget(7, 5) == 0xFFFFFFFF


@pytest.mark.parametrize("sym,group", [(False, 128), (True, 256), (False, 32)])
def test_gptq_quantize_timeout_is_reported_and_recovered(sym, group):
    w = synth.outlier_columns_bf16(2048, 4096, 0.02, 0.005, 20.0, 90 + group, device="cpu")
    wd = w.to("cuda")
    fn = wq.gptq_quantize_sym if sym else wq.gptq_quantize_asym
    torch.cuda.synchronize()
    assert wq.device_status() == wq.WQ_OK  # nothing pending from earlier tests
    with zero_budget(WQ_WAIT_GPTQ_STAGE):
        fn(wd, group, True)  # every stage wait gives up at once
    assert wq.device_status() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.device_status() == wq.WQ_OK  # reported once, then cleared
    # the context is intact: a normal call gives the oracle's tensors bit for bit
    r = fn(wd, group, True)
    qw, qz, sc, gi, snr = oracle.gptq_quantize(w, group, sym)
    assert np.array_equal(r["qweight"].cpu().numpy(), qw)
    assert np.array_equal(r["qzeros"].cpu().numpy(), qz)
    assert np.array_equal(r["scales"].cpu().view(torch.int16).numpy().view(np.uint16), sc)
    assert abs(float(r["snr_db"]) - snr) <= 1e-4 * abs(snr)
    torch.cuda.synchronize()
    assert wq.device_status() == wq.WQ_OK


def _gemm_bound_ok(y, ref, mag, k):
    # the GEMM's derived bound: (k + 2) 2^-23 sum |x deq| of the binary64 product
    return np.all(np.abs(y.double().cpu().numpy() - ref) <= (k + 2) * 2.0 ** -23 * mag + 1e-30)


def test_gptq_gemm_mma_timeout_is_reported_and_recovered():
    n, k, m = 1024, 4096, 256  # 16 CTAs, 64 K blocks: the loads fill all 8 stages first
    w = synth.outlier_columns_bf16(n, k, 0.02, 0.005, 20.0, 97, device="cpu")
    qw, qz, sc, gi, _ = oracle.gptq_quantize(w, 128, False)
    qw_d, qz_d = torch.from_numpy(qw).cuda(), torch.from_numpy(qz).cuda()
    sc_d = torch.from_numpy(sc.view(np.int16)).view(torch.float16).cuda()
    x = synth.normal_bf16((m, k), 1.0, 98, device="cpu")
    xd = x.cuda()
    torch.cuda.synchronize()
    assert wq.device_status() == wq.WQ_OK
    with zero_budget(WQ_WAIT_GEMM_MMA):
        wq.gptq_gemm(xd, qw_d, qz_d, sc_d, n, k, 128, False)
    assert wq.device_status() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.device_status() == wq.WQ_OK
    y = wq.gptq_gemm(xd, qw_d, qz_d, sc_d, n, k, 128, False)
    ref, mag = oracle.gptq_linear(x, qw, qz, sc, n, k, 128, False)
    assert _gemm_bound_ok(y, ref, mag, k)
    torch.cuda.synchronize()
    assert wq.device_status() == wq.WQ_OK


def test_uintx_gemm_mma_timeout_is_reported_and_recovered():
    n, k, m, nbits = 512, 2048, 130, 5
    w = synth.normal_bf16((n, k), 0.02, 99, device="cpu")
    packed, scale, zp, _ = oracle.uintx_quantize(w, nbits, 64)
    deq = oracle.bf16_bits_to_f32(oracle.uintx_dequantize(packed, scale, zp, n, k, nbits, 64)).astype(np.float64)
    p_d = torch.from_numpy(packed).cuda()
    s_d = torch.from_numpy(np.asarray(scale).view(np.int16)).view(torch.bfloat16).reshape(n, k // 64).cuda()
    z_d = torch.from_numpy(np.asarray(zp)).reshape(n, k // 64).cuda()
    x = synth.normal_bf16((m, k), 1.0, 100, device="cpu")
    xd = x.cuda()
    torch.cuda.synchronize()
    assert wq.device_status() == wq.WQ_OK
    with zero_budget(WQ_WAIT_GEMM_MMA):
        wq.uintx_gemm(xd, p_d, s_d, z_d, n, k, nbits, 64)
    assert wq.device_status() == wq.WQ_ERR_DEVICE_TIMEOUT
    assert wq.device_status() == wq.WQ_OK
    y = wq.uintx_gemm(xd, p_d, s_d, z_d, n, k, nbits, 64)
    xf = oracle.bf16_bits_to_f32(x.view(torch.int16).numpy().view(np.uint16)).astype(np.float64)
    ref, mag = xf @ deq.T, np.abs(xf) @ np.abs(deq).T
    assert _gemm_bound_ok(y, ref, mag, k)
    torch.cuda.synchronize()
    assert wq.device_status() == wq.WQ_OK
