"""GPU parity of the tensor-core GPTQ W4A16 GEMM (gptq_gemm: y = x deq(W)^T for
prefill batches) against the oracle's binary64 product of the dequantized weight.

Tolerance, from the arithmetic: every product x * (code - zp) is exact; the
tensor cores add them in binary32 with internal additions whose rounding is not
documented as round-to-nearest (so one binary32 ulp, 2^-23, is allowed for each),
and one FMA per group folds the scaled group sums, so
|y - y_exact| <= (k + 2) * 2^-23 * sum_k |x * deq|.  A bf16 output may differ by
half a bf16 ulp more."""
import numpy as np
import pytest
import torch

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -23


def quantized(n, k, group, sym, seed):
    w = synth.outlier_columns_bf16(n, k, 0.02, 0.005, 20.0, seed, device=DEV)
    fn = wq.gptq_quantize_sym if sym else wq.gptq_quantize_asym
    r = fn(w, group, False)
    return r["qweight"], r["qzeros"], r["scales"]


def acts(m, k, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(m, k, generator=g) * torch.exp(torch.randn(k, generator=g))).to(torch.bfloat16)


def check(x, qw, qz, sc, n, k, group, sym, out_dtype=torch.float32, rows=None):
    y = wq.gptq_gemm(x.to(DEV), qw, qz, sc, n, k, group, sym, out_dtype)
    xs = x if rows is None else x[rows]
    ref, mag = oracle.gptq_linear(xs, qw.cpu().numpy(), qz.cpu().numpy(), sc.cpu(), n, k, group, sym)
    got = y.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    bound = (k + 2) * U * mag
    if out_dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(ref) + bound)
    err = np.abs(got - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
    assert wq.device_status() == 0
    return y


@pytest.mark.parametrize("group", [32, 64, 128, 256])
@pytest.mark.parametrize("sym", [True, False])
def test_gptq_gemm_groups_ragged(group, sym):
    n, k = 264, 1024  # a ragged feature tile (264 = 2 * 128 + 8)
    qw, qz, sc = quantized(n, k, group, sym, 90 + group)
    for m in (1, 17, 128, 200):  # one token, ragged token tiles, exactly one tile
        check(acts(m, k, 91 + m), qw, qz, sc, n, k, group, sym)
    check(acts(33, k, 92), qw, qz, sc, n, k, group, sym, torch.bfloat16)


def test_gptq_gemm_partial_last_k_block():
    n, k = 136, 1056  # k = 33 groups of 32: the last 64-wide K block is half full
    for sym in (True, False):
        qw, qz, sc = quantized(n, k, 32, sym, 93)
        check(acts(40, k, 94), qw, qz, sc, n, k, 32, sym)


def test_gptq_gemm_odd_number_of_k_blocks():
    # k = 17 blocks of 64 with group 64: the MMA thread's last pair holds one block
    n, k = 136, 1088
    for sym in (True, False):
        qw, qz, sc = quantized(n, k, 64, sym, 97)
        check(acts(70, k, 98), qw, qz, sc, n, k, 64, sym)


@pytest.mark.parametrize("shape", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_gptq_gemm_layer_shapes_prefill(shape):
    n, k = shape
    m = 512
    qw, qz, sc = quantized(n, k, 128, False, 95)
    x = acts(m, k, 96)
    rows = np.r_[0:8, 120:136, 505:512]  # first, a tile boundary, last
    y1 = check(x, qw, qz, sc, n, k, 128, False, rows=rows)
    y2 = wq.gptq_gemm(x.to(DEV), qw, qz, sc, n, k, 128, False)
    assert torch.equal(y1, y2)  # the same bits from run to run


def test_gptq_gemm_sym_layer_full():
    n, k, m = 4096, 4096, 256
    qw, qz, sc = quantized(n, k, 128, True, 97)
    check(acts(m, k, 98), qw, qz, sc, n, k, 128, True)


def test_gptq_gemm_agrees_with_decode_consumer_bound():
    # both consumers stay within their bounds of the same exact product
    n, k = 1024, 2048
    qw, qz, sc = quantized(n, k, 128, False, 99)
    x = acts(4, k, 100)
    a = wq.gptq_gemm(x.to(DEV), qw, qz, sc, n, k, 128, False).double().cpu().numpy()
    b = wq.gptq_linear(x.to(DEV), qw, qz, sc, n, k, 128, False).double().cpu().numpy()
    ref, mag = oracle.gptq_linear(x, qw.cpu().numpy(), qz.cpu().numpy(), sc.cpu(), n, k, 128, False)
    assert np.all(np.abs(a - b) <= (k + 2) * (U + 2.0 ** -24) * mag + 1e-30)


def test_gptq_gemm_empty_k_writes_zeros():
    y = torch.full((3, 64), 7.0, device=DEV)
    x = torch.empty(3, 0, dtype=torch.bfloat16, device=DEV)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    wq.gptq_gemm(x, e, e, torch.empty(0, dtype=torch.float16, device=DEV), 64, 0, 128, True, out=y)
    assert torch.count_nonzero(y) == 0


# ------------------------------------------------------------------ uintx consumer
def uintx_inputs(n, k, nbits, group, seed):
    w = synth.normal_bf16((n, k), 0.02, seed)
    packed, sc, zp, _ = oracle.uintx_quantize(w, nbits, group)  # the oracle's own codes
    deq = oracle.bf16_bits_to_f32(oracle.uintx_dequantize(packed, sc, zp, n, k, nbits, group))
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(DEV)
    return t(packed, torch.uint8), t(sc.view(np.int16), torch.bfloat16), t(zp, torch.uint8), deq


def check_ux(x, packed, sc, zp, deq, n, k, nbits, group, out_dtype=torch.float32):
    y = wq.uintx_gemm(x.to(DEV), packed, sc, zp, n, k, nbits, group, out_dtype)
    xf = oracle.bf16_bits_to_f32(u16x(x)).astype(np.float64)
    d = deq.astype(np.float64)
    ref, mag = xf @ d.T, np.abs(xf) @ np.abs(d).T
    got = y.float().cpu().numpy().astype(np.float64)
    bound = (k + 2) * U * mag
    if out_dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * (np.abs(ref) + bound)
    err = np.abs(got - ref)
    assert np.all(err <= bound + 1e-30), float((err / (bound + 1e-30)).max())
    assert wq.device_status() == 0
    return y


def u16x(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("nbits", [2, 3, 4, 5, 6, 7])
def test_uintx_gemm_bits(nbits):
    n, k = 264, 1024  # ragged feature tile
    packed, sc, zp, deq = uintx_inputs(n, k, nbits, 64, 110 + nbits)
    for m in (1, 40, 128, 200):
        check_ux(acts(m, k, 111 + m), packed, sc, zp, deq, n, k, nbits, 64)
    check_ux(acts(33, k, 112), packed, sc, zp, deq, n, k, nbits, 64, torch.bfloat16)


@pytest.mark.parametrize("group", [32, 128, 256])
def test_uintx_gemm_groups(group):
    n, k = 136, 512
    for nbits in (3, 7):
        packed, sc, zp, deq = uintx_inputs(n, k, nbits, group, 113 + group)
        check_ux(acts(70, k, 114), packed, sc, zp, deq, n, k, nbits, group)


@pytest.mark.parametrize("n", [1, 3, 7, 9])
def test_uintx_gemm_tiny_n_shard_wraps(n):
    # with n < 8 the shard chunks are shorter than a row: runs wrap inside rows
    k = 128
    for nbits in (3, 5, 6, 7):
        packed, sc, zp, deq = uintx_inputs(n, k, nbits, 64, 115 + n)
        check_ux(acts(5, k, 116), packed, sc, zp, deq, n, k, nbits, 64)


def test_uintx_gemm_layer_shape():
    n, k, m = 4096, 4096, 256
    packed, sc, zp, deq = uintx_inputs(n, k, 4, 64, 117)
    x = acts(m, k, 118)
    y1 = check_ux(x, packed, sc, zp, deq, n, k, 4, 64)
    y2 = wq.uintx_gemm(x.to(DEV), packed, sc, zp, n, k, 4, 64)
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("nbits", [3, 5])
def test_uintx_gemm_odd_number_of_k_blocks(nbits):
    # k = 15 blocks of 64: the last pair of K blocks holds one block
    n, k = 136, 960
    packed, sc, zp, deq = uintx_inputs(n, k, nbits, 64, 119 + nbits)
    check_ux(acts(70, k, 120), packed, sc, zp, deq, n, k, nbits, 64)
