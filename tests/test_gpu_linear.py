"""GPU parity of the GPTQ W4A16 consumer (gptq_linear: y = x deq(W)^T for decode
batches) against the oracle's binary64 product of the dequantized weight.

Tolerance, from the arithmetic: every product x * (code - zp) is exact in
binary32; the kernel adds at most k of them, one group scaling and one addition
per group and per K-slice in binary32, so by the standard bound for recursive
summation |y - y_exact| <= (k + 2) * 2^-24 * sum_k |x_k * deq_k| (mag below).
A bf16 output may differ by half a bf16 ulp more (2^-8 relative)."""
import numpy as np
import pytest
import torch

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


def quantized(n, k, group, sym, seed):
    w = synth.outlier_columns_bf16(n, k, 0.02, 0.005, 20.0, seed, device=DEV)
    fn = wq.gptq_quantize_sym if sym else wq.gptq_quantize_asym
    r = fn(w, group, False)
    return r["qweight"], r["qzeros"], r["scales"]


def acts(m, k, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(m, k, generator=g) * torch.exp(torch.randn(k, generator=g))).to(torch.bfloat16)


def check(x, qw, qz, sc, n, k, group, sym, out_dtype=torch.float32):
    y = wq.gptq_linear(x.to(DEV), qw, qz, sc, n, k, group, sym, out_dtype)
    ref, mag = oracle.gptq_linear(x, qw.cpu().numpy(), qz.cpu().numpy(), sc.cpu(), n, k, group, sym)
    got = y.float().cpu().numpy().astype(np.float64)
    bound = (k + 2) * U * mag
    if out_dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(ref) + bound)  # half an ulp of an 8-bit significand
    err = np.abs(got - ref)
    assert np.all(err <= bound + 1e-30), (float((err / (bound + 1e-30)).max()))
    return y


@pytest.mark.parametrize("group", [32, 64, 128, 256])
@pytest.mark.parametrize("sym", [True, False])
def test_gptq_linear_groups(group, sym):
    n, k = 264, 1024  # a ragged column block
    qw, qz, sc = quantized(n, k, group, sym, 60 + group)
    for m in (1, 3, 8):
        check(acts(m, k, 61 + m), qw, qz, sc, n, k, group, sym)
    check(acts(2, k, 62), qw, qz, sc, n, k, group, sym, torch.bfloat16)


@pytest.mark.parametrize("shape", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_gptq_linear_layer_shapes(shape):
    n, k = shape
    qw, qz, sc = quantized(n, k, 128, False, 63)
    for m in (1, 4):
        y1 = check(acts(m, k, 64 + m), qw, qz, sc, n, k, 128, False)
        # one workspace, zeroed once, reused: the kernel leaves its counters at zero
        ws = torch.zeros(wq.lib().gptq_linear_workspace_bytes(m, n), dtype=torch.uint8, device=DEV)
        for _ in range(3):
            y2 = wq.gptq_linear(acts(m, k, 64 + m).to(DEV), qw, qz, sc, n, k, 128, False, ws=ws)
            assert torch.equal(y1, y2)  # the same bits from run to run
        assert torch.count_nonzero(ws[:256]) == 0


def test_gptq_linear_empty_k_writes_zeros():
    y = torch.full((2, 64), 7.0, device=DEV)
    x = torch.empty(2, 0, dtype=torch.bfloat16, device=DEV)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    wq.gptq_linear(x, e, e, torch.empty(0, dtype=torch.float16, device=DEV), 64, 0, 128, True, out=y)
    assert torch.count_nonzero(y) == 0


# ------------------------------------------------------------------ MXFP4 consumer
def check_mx(x, p, e, out_dtype=torch.float32):
    y = wq.mxfp4_linear(x.to(DEV), p, e, out_dtype)
    ref, mag = oracle.mxfp4_linear(x, p.cpu().numpy(), e.cpu().numpy())
    k = x.shape[-1]
    got = y.float().cpu().numpy().astype(np.float64)
    bound = (k + 2) * U * mag
    if out_dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(ref) + bound)
    err = np.abs(got - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
    return y


@pytest.mark.parametrize("shape", [(10, 96), (257, 1056), (4096, 4096), (14336, 4096), (4096, 14336)])
def test_mxfp4_linear(shape):
    n, k = shape
    w = synth.outlier_columns_bf16(n, k, 0.02, 0.005, 20.0, 80 + n, device=DEV)
    p, e = wq.mxfp4_quantize(w)
    for m in (1, 3, 8):
        y1 = check_mx(acts(m, k, 81 + m), p, e)
        y2 = wq.mxfp4_linear(acts(m, k, 81 + m).to(DEV), p, e)
        assert torch.equal(y1, y2)
    check_mx(acts(2, k, 82), p, e, torch.bfloat16)
