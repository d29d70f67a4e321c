"""GPU parity of GPTQ and MXFP4 quantization of fp16 and fp32 weights (the pages
quantize w.float(): export_gptq_cpu.py quantize_sym / quantize_asym,
quantize_dflash_mxfp4.py quantize_mxfp4) against the oracle's binary32 path:
codes, scales, zero points and E8M0 bytes bit for bit, the SNR within 1e-4
relative."""
import numpy as np
import pytest
import torch

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL = 1e-4


def f32_weight(n, k, seed, dtype):
    w = synth.normal_f32((n, k), 0.02, seed)
    g = torch.Generator().manual_seed(seed + 1)
    cols = torch.randperm(k, generator=g)[: max(1, k // 200)]
    w[:, cols] *= 20.0
    return w.to(dtype)


def check_gptq(w, group, sym):
    n, k = w.shape
    fn = wq.gptq_quantize_sym if sym else wq.gptq_quantize_asym
    r = fn(w.to(DEV), group, True)
    qw, qz, sc, gi, snr = oracle.gptq_quantize_f32(w.float().numpy(), group, sym)
    assert np.array_equal(r["qweight"].cpu().numpy(), qw), "qweight"
    assert np.array_equal(r["scales"].cpu().view(torch.int16).numpy().view(np.uint16), sc), "scales"
    assert np.array_equal(r["qzeros"].cpu().numpy(), qz), "qzeros"
    assert np.array_equal(r["g_idx"].cpu().numpy(), gi), "g_idx"
    got = float(r["snr_db"])
    assert abs(got - snr) <= REL * abs(snr), (got, snr)
    assert wq.device_status() == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("group", [32, 128, 256])
@pytest.mark.parametrize("sym", [True, False])
def test_gptq_wide_inputs(dtype, group, sym):
    check_gptq(f32_weight(264, 1024, 40 + group, dtype), group, sym)


def test_gptq_wide_layer_shape():
    check_gptq(f32_weight(4096, 4096, 47, torch.float32), 128, False)
    check_gptq(f32_weight(1024, 4096, 48, torch.float16), 128, True)


def test_gptq_wide_hand_groups_tiled():
    # the oracle pins' binary32 groups tiled to a 32-wide group: the group's
    # max / min / amax are unchanged, so every code is the hand-worked one
    e = 2.0 ** -26
    sym_vals = [1.0, -0.5, 0.1875 - e, 0.1875 + e, 0.3125, -0.0625, 2.0 ** -30, -1.0]
    asym_vals = [-0.46875, 0.46875, 0.03125 + 2.0 ** -28, 0.03125, -0.09375, 0.15625 - 2.0 ** -26, 0.0, -0.25]
    for vals, sym, codes in ((sym_vals, True, [15, 4, 9, 10, 10, 8, 8, 0]),
                             (asym_vals, False, [0, 15, 9, 8, 6, 10, 8, 4])):
        w = torch.tensor(vals, dtype=torch.float32).repeat(8, 4)  # [8, 32]
        r = (wq.gptq_quantize_sym if sym else wq.gptq_quantize_asym)(w.to(DEV), 32, False)
        word = int(np.int32(np.uint32(sum(c << (4 * i) for i, c in enumerate(codes)))))
        assert np.all(r["qweight"].cpu().numpy() == word)


def degenerate_weight(dtype, group, seed):
    """Rows of groups that take every special path of the fp16 / fp32 kernel:
    constant groups (range 0, scale from the 1e-9 floor), narrow all-positive and
    all-negative groups (zero point clamped to 0 / 15, so codes leave [0, 15]
    before the clamp), values far beyond 2^16 x the range (the IEEE-division
    path), a single outlier, exact zeros and (fp32) subnormals, next to ordinary
    groups in the same warp tile."""
    g = torch.Generator().manual_seed(seed)
    n, k = 64, 4 * max(group, 128)
    w = torch.randn(n, k, generator=g) * 0.02
    big = 1e12 if dtype == torch.float32 else 3.0e4  # squares and their sums stay finite
    tiny = 1e-40 if dtype == torch.float32 else 1e-7
    for r in range(n):
        kind = r % 8
        for g0 in range(0, k, group):
            seg = slice(g0, g0 + group)
            u = torch.rand(group, generator=g)
            if kind == 0:
                w[r, seg] = 0.3 if (g0 // group) % 2 == 0 else -2.0   # constant groups
            elif kind == 1:
                w[r, seg] = 1.0 + 1e-3 * u                            # narrow, all positive
            elif kind == 2:
                w[r, seg] = -1.0 - 1e-3 * u                           # narrow, all negative
            elif kind == 3:
                w[r, seg] = big * (1.0 + 1e-6 * u)                    # |w| far beyond 2^16 range
            elif kind == 4:
                w[r, seg] = 0.0
                w[r, g0 + 3] = 5.0                                    # one outlier among zeros
            elif kind == 5:
                w[r, seg] = tiny * (u - 0.5)                          # tiny / subnormal values
    return w.to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("group", [32, 128])
@pytest.mark.parametrize("sym", [True, False])
def test_gptq_wide_degenerate_groups(dtype, group, sym):
    w = degenerate_weight(dtype, group, 60 + group)
    fn = wq.gptq_quantize_sym if sym else wq.gptq_quantize_asym
    r = fn(w.to(DEV), group, True)
    qw, qz, sc, gi, snr = oracle.gptq_quantize_f32(w.float().numpy(), group, sym)
    assert np.array_equal(r["qweight"].cpu().numpy(), qw), "qweight"
    assert np.array_equal(r["scales"].cpu().view(torch.int16).numpy().view(np.uint16), sc), "scales"
    assert np.array_equal(r["qzeros"].cpu().numpy(), qz), "qzeros"
    # the large groups' errors dominate both norms here, so the SNR can sit near
    # 0 dB: 1e-4 relative to it, or 1e-4 dB
    got = float(r["snr_db"])
    assert np.isfinite(snr) and abs(got - snr) <= REL * max(abs(snr), 1.0), (got, snr)
    assert wq.device_status() == 0


def check_mx(w, tie):
    p, e = wq.mxfp4_quantize(w.to(DEV), tie)
    rp, re = oracle.mxfp4_quantize_f32(w.float().numpy(), tie)
    assert np.array_equal(p.cpu().numpy(), rp) and np.array_equal(e.cpu().numpy(), re)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("tie", [0, 1])
def test_mxfp4_wide_inputs(dtype, tie):
    check_mx(f32_weight(257, 1056, 50 + tie, dtype), tie)


@pytest.mark.parametrize("tie", [0, 1])
def test_mxfp4_wide_edge_blocks(tie):
    rows = []
    for ex in (-140, -126, -100, -3, 0, 5, 100, 125):
        s = 2.0 ** ex
        # a block topped by 6 * 2^e with every e2m1 midpoint and neighbours of it
        mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
        vals = [6.0] + [m for m in mids] + [-m for m in mids] + [m * (1 + 2.0 ** -20) for m in mids] \
            + [m * (1 - 2.0 ** -20) for m in mids] + [0.0, -0.0, 1e-30, 4.0]
        rows.append(np.asarray(vals[:32], np.float64) * s)
    rows.append(np.zeros(32))                         # an all-zero block
    rows.append(np.full(32, 2.0 ** -149))             # subnormal amax
    w = torch.from_numpy(np.stack(rows).astype(np.float32)).repeat(1, 2)  # [10, 64]
    check_mx(w, tie)
    check_mx(w.clamp(-60000, 60000).to(torch.float16), tie)


def test_mxfp4_wide_dequant_round_trip_and_consumer():
    w = f32_weight(512, 1024, 55, torch.float32)
    p, e = wq.mxfp4_quantize(w.to(DEV))
    d = wq.mxfp4_dequantize(p, e).cpu().numpy()
    assert np.array_equal(d, oracle.mxfp4_dequantize(*oracle.mxfp4_quantize_f32(w.numpy())))


# ------------------------------------------------------------------ uintx in the weight dtype
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
@pytest.mark.parametrize("nbits", [2, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("shape,group", [((37, 192), 64), ((37, 192), 24), ((256, 1024), 32)])
def test_uintx_wide(dtype, nbits, shape, group):
    n, k = shape
    w = f32_weight(n, k, 60 + nbits, dtype)
    packed, sc, zp = wq.uintx_quantize(w.to(DEV), nbits, group)
    dt = 0 if dtype == torch.float32 else 2
    rp, rs, rz, _ = oracle.uintx_quantize_dt(w, dt, nbits, group)
    bits = (lambda t: t.cpu().numpy()) if dt == 0 else (lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(packed.cpu().numpy(), rp), "packed"
    assert np.array_equal(bits(sc), rs), "scale"
    assert np.array_equal(zp.cpu().numpy(), rz), "zp"
    d = wq.uintx_dequantize(packed, sc, zp, n, k, nbits, group)
    assert d.dtype == dtype
    assert np.array_equal(bits(d), oracle.uintx_dequantize_dt(rp, rs, dt, rz, n, k, nbits, group)), "deq"
    assert wq.device_status() == 0
