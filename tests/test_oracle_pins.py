"""Pins for the CPU oracle: checks against what the pages and the mathematics fix,
never against the oracle itself.

Sources: export_gptq_cpu.py (pack_int32, quantize_sym, quantize_asym, the uint4b8
dequant rule in the module docstring), quantize_dflash_mxfp4.py (E2M1,
quantize_mxfp4, dequantize_mxfp4, search_scale), uintx_quant.py (module docstring,
_pack_shard, pack_uintx, unpack_uintx, _quantize_impl, _dequantize_native).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a skipped rounding) fails it:
hand-worked golden groups (tests/golden/*.json), closed forms, brute force over
small domains, metamorphic relations and independent library conversions.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from conftest import GOLDEN

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits(values) -> np.ndarray:
    """Exact bf16 bit patterns of values that are bf16-representable (asserted)."""
    f = np.asarray(values, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)


def round_bf16(values) -> np.ndarray:
    """bf16 bit patterns of arbitrary values (torch's CPU cast, round to nearest even)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


# --------------------------------------------------------------------------- P0: formats
def test_bf16_rounding_matches_torch():
    """orc_f32_to_bf16 (hand-written RNE) against torch's CPU float->bfloat16 cast."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, size=40000, dtype=np.uint64).astype(np.uint32)
    # exact ties, max-finite neighbours, subnormals, zeros and infinities
    special = np.array([0x3F808000, 0x3F818000, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF,
                        0x00008000, 0x00018000, 0x00000001, 0x80000000, 0x7F800000,
                        0xFF800000, 0x3F800001, 0xBF808000], dtype=np.uint32)
    f = np.concatenate([bits, special]).view(np.float32)
    f = f[~np.isnan(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(x)) for x in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_bf16_op_rule_matches_torch_arithmetic():
    """P8: a bf16 tensor op equals the binary32 op on the bf16 operands rounded
    once to bf16 (the reading the uintx oracle uses), for mul, div, sub, add."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    a = torch.from_numpy(rng.normal(0, 1, 20000).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy(rng.lognormal(0, 2, 20000).astype(np.float32)).to(torch.bfloat16)
    af = a.float().numpy()
    bf_ = b.float().numpy()
    for op, ref in ((torch.mul, np.multiply), (torch.div, np.divide),
                    (torch.sub, np.subtract), (torch.add, np.add)):
        want = op(a, b).view(torch.int16).numpy().view(np.uint16)
        f32 = ref(af, bf_).astype(np.float32)  # one IEEE binary32 op
        got = np.array([oracle.f32_to_bf16(float(x)) for x in f32], dtype=np.uint16)
        assert np.array_equal(got, want), op


def test_f16_rounding_matches_numpy():
    """orc_f32_to_f16 against numpy's IEEE binary32->binary16 conversion,
    including subnormals, the overflow threshold and exact ties."""
    rng = np.random.default_rng(13)
    mags = np.concatenate([
        rng.uniform(0, 7e4, 20000),
        np.exp(rng.uniform(np.log(1e-9), np.log(1e-3), 20000)),
        [65504.0, 65519.99, 65520.0, 65536.0, 2.0**-24, 2.0**-25, 1.5 * 2.0**-25,
         2.0**-14, 2.0**-14 - 2.0**-25, 1e-9, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11]])
    vals = np.concatenate([mags, -mags]).astype(np.float32)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(x)) for x in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_f16_decode_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = h.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(x)) for x in h], dtype=np.float32)
    ok = (got == want) | (np.isnan(got) & np.isnan(want))
    assert ok.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(want[~np.isnan(want)]))


# --------------------------------------------------------------------------- P1: packing
def test_pack_int32_golden():
    """pack_int32: 8 nibbles per int32, low-order nibble first (hand values)."""
    col = np.arange(1, 9, dtype=np.int32).reshape(8, 1)  # K=8, N=1
    assert oracle.pack_int32(col, 0).view(np.uint32)[0, 0] == 0x87654321
    top = np.zeros((8, 1), np.int32)
    top[7, 0] = 15
    assert oracle.pack_int32(top, 0).view(np.uint32)[0, 0] == 0xF0000000  # bit 31: negative int32
    row = np.arange(1, 9, dtype=np.int32).reshape(1, 8)  # along N
    assert oracle.pack_int32(row, 1).view(np.uint32)[0, 0] == 0x87654321


def test_pack_int32_positions_brute_force():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 16, size=(32, 24), dtype=np.int32)
    p0 = oracle.pack_int32(codes, 0).view(np.uint32)
    p1 = oracle.pack_int32(codes, 1).view(np.uint32)
    for kk in range(32):
        for n in range(24):
            assert (int(p0[kk // 8, n]) >> (4 * (kk % 8))) & 15 == codes[kk, n]
            assert (int(p1[kk, n // 8]) >> (4 * (n % 8))) & 15 == codes[kk, n]


def test_uintx_pack_golden():
    g = load("uintx_hand.json")
    for case in g["pack_cases"]:
        got = oracle.uintx_pack(np.array(case["codes"], np.uint8), case["nbits"])
        assert got.tolist() == case["packed"], case
    for case in g["packed_sizes"]:
        assert oracle.uintx_packed_bytes(case["numel"], case["nbits"]) == case["bytes"]


@pytest.mark.parametrize("nbits", [2, 3, 4, 5, 6, 7, 8])
def test_uintx_pack_roundtrip_exhaustive_small(nbits):
    """unpack(pack(c)) == c for every numel 1..64 (padding included)."""
    rng = np.random.default_rng(nbits)
    for numel in range(1, 65):
        codes = rng.integers(0, 2**nbits, size=numel, dtype=np.int64).astype(np.uint8)
        packed = oracle.uintx_pack(codes, nbits)
        assert packed.size == oracle.uintx_packed_bytes(numel, nbits)
        assert np.array_equal(oracle.uintx_unpack(packed, nbits, numel), codes)


def test_uintx_pack_single_bit_positions():
    """A lone 1 bit in code e, bit b, must appear in exactly one packed byte at
    the place the shard/chunk rule puts it: shard of the power-of-two piece
    containing b, chunk j = e // L, byte i = e % L, bit j*k + (b - offset)."""
    numel, nbits = 37, 7
    shards = [(4, 0), (2, 4), (1, 6)]  # (k, offset) for 7 = 4 + 2 + 1
    for e in range(numel):
        for b in range(nbits):
            codes = np.zeros(numel, np.uint8)
            codes[e] = 1 << b
            packed = oracle.uintx_pack(codes, nbits)
            base = 0
            expect = np.zeros_like(packed)
            for k, off in shards:
                vpb = 8 // k
                length = -(-numel // vpb)
                if off <= b < off + k:
                    expect[base + e % length] = 1 << ((e // length) * k + (b - off))
                base += length
            assert np.array_equal(packed, expect), (e, b)


# --------------------------------------------------------------------------- P2/P3: GPTQ
def _gptq_from_column(col, group, sym, ncols=8):
    """A weight [N=ncols, K=len(col)] whose every row is `col` (the group runs along K)."""
    w = np.tile(bf16_bits(col), (ncols, 1))
    return oracle.gptq_quantize(w, group=group, sym=sym)


def test_gptq_hand_groups():
    for case in load("gptq_hand_groups.json")["cases"]:
        qw, qz, sc, gi, snr = _gptq_from_column(case["column"], case["group"], case["sym"])
        assert np.all(qw.view(np.uint32) == int(case["qweight_word"], 16)), case["name"]
        assert np.all(sc == int(case["scale_f16"], 16)), case["name"]
        assert np.all(qz.view(np.uint32) == int(case["qzeros_word"], 16)), case["name"]
        assert gi.tolist() == [k // case["group"] for k in range(len(case["column"]))]
        if "snr_db" in case:
            assert snr == float(case["snr_db"])


def test_gptq_dequant_golden_words():
    """Module docstring: uint4b8 dequant w = (code - 8) * scale; asym (code - zp) * scale."""
    n, k = 8, 8
    qw = np.full((1, n), 0x87654321, np.uint32).view(np.int32)
    sc = np.full((1, n), 0x3C00, np.uint16)  # fp16 1.0
    deq = oracle.gptq_dequantize(qw, np.zeros((1, 1), np.int32), sc, n, k, 8, True, out_kn=True)
    assert np.array_equal(deq[:, 0], np.arange(1, 9) - 8.0)
    qz = np.array([[0x76543210]], np.uint32).view(np.int32)  # zp of column c = c
    deq = oracle.gptq_dequantize(qw, qz, sc, n, k, 8, False, out_kn=False)  # [N, K]
    for c in range(n):
        assert np.array_equal(deq[c], np.arange(1, 9) - float(c))


@pytest.mark.parametrize("sym", [True, False])
def test_gptq_grid_reconstruction(sym):
    """P3: a group lying on the quantizer's own grid reconstructs exactly, through
    both the binary32 scale (SNR) and the stored fp16 scale (dequant)."""
    rng = np.random.default_rng(3)
    n, k, group = 16, 256, 128
    s = 2.0 ** -7  # fp16-exact, and (j * s) is bf16-exact for |j| <= 15
    if sym:
        j = rng.integers(-8, 8, size=(n, k))
        j[:, 0] = -8  # amax = 8s so scale = s
        j[:, 128] = -8
    else:
        zp = 5
        j = rng.integers(-zp, 16 - zp, size=(n, k))
        j[:, 0] = -zp  # wmin = -5s, wmax = 10s: range 15s -> scale s
        j[:, 1] = 15 - zp
        j[:, 128] = -zp
        j[:, 129] = 15 - zp
    w = (j * s).astype(np.float32)
    qw, qz, sc, gi, snr = oracle.gptq_quantize(bf16_bits(w), group=group, sym=sym)
    deq = oracle.gptq_dequantize(qw, qz, sc, n, k, group, sym, out_kn=False)
    assert np.array_equal(deq, w)
    assert np.all(sc == np.float16(s).view(np.uint16))
    norm = math.sqrt(float(np.sum(w.astype(np.float64) ** 2)))
    assert snr == pytest.approx(20 * math.log10(norm / 1e-12), rel=1e-12)


def test_gptq_sym_snr_closed_form():
    """P9: ramp w_i = s(-8 + i/8), i < 128, in one group of 128 (s = 2^-6).
    amax = 8s so scale = s; residues of i/8 give sum(e^2)/s^2 = 15*(44/64) + 140/64
    = 12.5 (the top half-bin clamps to code 15); sum(w^2)/s^2 = 2731.
    SNR = 10 log10(2731 / 12.5)."""
    s = 2.0 ** -6
    col = [s * (-8 + i / 8) for i in range(128)]
    qw, qz, sc, gi, snr = _gptq_from_column(col, 128, True)
    assert snr == pytest.approx(10 * math.log10(2731 / 12.5), rel=1e-9)


def test_gptq_asym_snr_closed_form():
    """Asym analogue: w_i = s * min(i, 120)/8, i < 128: wmin = 0, wmax = 15s, so
    scale = s and zp = 0; sum(e^2)/s^2 = 15 * 44/64 = 10.3125 and
    sum(w^2)/s^2 = (1/64) * 120*121*241/6 + 7*225 = 10687.8125."""
    s = 2.0 ** -6
    col = [s * min(i, 120) / 8 for i in range(128)]
    qw, qz, sc, gi, snr = _gptq_from_column(col, 128, False)
    assert snr == pytest.approx(10 * math.log10(10687.8125 / 10.3125), rel=1e-9)
    assert np.all(qz.view(np.uint32) == 0)


def test_gptq_layout_is_transposed():
    """qweight is [K/8, N]: column n of qweight packs row n of w along K; scales are
    [K/group, N]; swapping two rows of w swaps two columns of every output."""
    rng = np.random.default_rng(5)
    w = round_bf16(rng.normal(0, 0.02, (16, 256)))
    for sym in (True, False):
        a = oracle.gptq_quantize(w, group=128, sym=sym)
        w2 = w.copy()
        w2[[3, 9]] = w2[[9, 3]]
        b = oracle.gptq_quantize(w2, group=128, sym=sym)
        qa = a[0].copy()
        qa[:, [3, 9]] = qa[:, [9, 3]]
        assert np.array_equal(qa, b[0])
        sa = a[2].copy()
        sa[:, [3, 9]] = sa[:, [9, 3]]
        assert np.array_equal(sa, b[2])


# --------------------------------------------------------------------------- P4-P6, P11: MXFP4
@pytest.mark.parametrize("tie_mode,key", [(0, "index_half_even"), (1, "index_page_literal")])
def test_mxfp4_tie_tables(tie_mode, key):
    """P4: blocks with one 6*2^e element and the rest +-k*0.25*2^e."""
    g = load("mxfp4_hand.json")
    table = g[key]
    ks = g["quarter_steps_k"]
    for e in g["tie_exponents"]:
        for sign in (1.0, -1.0):
            row = np.zeros(32, np.float64)
            row[0] = 6.0 * 2.0 ** e
            row[1:1 + len(ks)] = [sign * k * 0.25 * 2.0 ** e for k in ks]
            if sign < 0:
                row[1] = -0.0
            packed, e8 = oracle.mxfp4_quantize(bf16_bits([row.astype(np.float32)]), tie_mode)
            assert e8[0, 0] == e + 127
            codes = np.empty(32, np.int64)
            codes[0::2] = packed[0] & 15
            codes[1::2] = packed[0] >> 4
            assert codes[0] == 7
            for i, k in enumerate(ks):
                want = table[i] | (8 if sign < 0 else 0)
                assert codes[1 + i] == want, (e, sign, k)


def test_mxfp4_clamped_and_zero_blocks():
    g = load("mxfp4_hand.json")
    bits = np.zeros(64, np.uint16)
    bits[0] = 0x0008  # 2^-130 = 8 * 2^-133, a bf16 subnormal
    bits[1] = 0x8008
    bits[2] = 0x8000
    assert oracle.bf16_to_f32(0x0008) == 2.0 ** -130
    packed, e8 = oracle.mxfp4_quantize(bits.reshape(1, 64))
    assert e8[0, 0] == g["clamped_block"]["e8m0"]
    assert packed[0, :2].tolist() == g["clamped_block"]["packed_first_two"]
    assert np.all(packed[0, 2:16] == 0)
    assert e8[0, 1] == g["zero_block"]["e8m0"]
    assert np.all(packed[0, 16:] == 0)


def test_mxfp4_dequant_golden():
    for case in load("mxfp4_hand.json")["dequant_cases"]:
        packed = np.full((1, 16), int(case["byte"], 16), np.uint8)
        e8 = np.array([[case["e8m0"]]], np.uint8)
        out = oracle.mxfp4_dequantize(packed, e8)
        assert out[0, 0] == np.float32(case["values"][0])
        assert out[0, 1] == np.float32(case["values"][1])
        assert np.signbit(out[0, 1]) == (math.copysign(1, case["values"][1]) < 0)


def test_mxfp4_grid_reconstruction():
    """P5: every +-E2M1[i]*2^e in a block whose amax is 6*2^e or 4*2^e is coded
    exactly; -0.0 gives code 8."""
    rng = np.random.default_rng(7)
    for e in (-100, -3, 0, 5, 100):
        for top in (6.0, 4.0):
            vals = rng.choice(E2M1, size=(8, 32)) * rng.choice([-1.0, 1.0], size=(8, 32))
            vals = np.minimum(vals, top) if top == 4.0 else vals
            vals = np.clip(vals, -top, top)
            vals[:, 5] = top
            vals = (vals * 2.0 ** e).astype(np.float32)
            packed, e8 = oracle.mxfp4_quantize(bf16_bits(vals))
            assert np.all(e8 == e + 127)
            out = oracle.mxfp4_dequantize(packed, e8)
            assert np.array_equal(out, vals)
    packed, _ = oracle.mxfp4_quantize(np.array([[0x8000] * 32], np.uint16))
    assert np.all(packed == 0x88)


def test_floor_log2_brute_force_bf16():
    """P6: for every positive finite bf16, the exact exponent equals floor(log2 x)."""
    h = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    x = oracle.bf16_bits_to_f32(h)
    want = np.floor(np.log2(x.astype(np.float64))).astype(np.int64)
    got = np.array([oracle.floor_log2(float(v)) for v in x])
    assert np.array_equal(got, want)
    # binary32 just below a power of two: the exponent is one less
    for e in (-140, -126, -1, 0, 1, 10, 100, 127):
        below = np.nextafter(np.float32(2.0 ** e), np.float32(0))
        assert oracle.floor_log2(float(below)) == e - 1
        assert oracle.floor_log2(float(np.float32(2.0 ** e))) == e


@pytest.mark.parametrize("tie_mode", [0, 1])
def test_e2m1_nearest_brute_force(tie_mode):
    """P11: for every bf16 m in [0, 8) the chosen magnitude is a nearest grid value
    (binary64 distances); exact midpoints follow the mode's rule."""
    h = np.arange(0, 0x4100, dtype=np.uint32).astype(np.uint16)  # 0 .. 8 (exclusive)
    mags = oracle.bf16_bits_to_f32(h)
    grid = np.array(E2M1)
    page_ties = {0.25: 0, 0.75: 0, 1.25: 2, 1.75: 2, 2.5: 4, 3.5: 4, 5.0: 6}
    for m in mags:
        code = oracle.e2m1_code(float(m), tie_mode)
        assert code < 8
        d = np.abs(min(float(m), 6.0) - grid)
        tied = np.flatnonzero(d == d.min())
        if len(tied) == 1:
            assert code == tied[0]
        elif tie_mode == 0:
            assert code in tied and code % 2 == 0
        else:
            assert code == page_ties[float(m)]
    assert oracle.e2m1_code(-0.0, tie_mode) == 8
    assert oracle.e2m1_code(-1e-30, tie_mode) == 8


def test_mxfp4_idempotent_and_ranges():
    """P12: quant(dequant(quant(w))) == quant(w) away from the exponent clamp;
    e8m0 <= 254 always."""
    rng = np.random.default_rng(8)
    w = (rng.normal(0, 0.02, (64, 256)) * np.exp(rng.normal(0, 2, (64, 1))))
    wb = round_bf16(w)
    p1, e1 = oracle.mxfp4_quantize(wb)
    d1 = oracle.mxfp4_dequantize(p1, e1)
    p2, e2 = oracle.mxfp4_quantize_f32(d1)
    assert np.all(e1 > 0)
    assert np.array_equal(e1, e2)
    assert np.array_equal(p1, p2)
    assert e1.max() <= 254


def test_mxfp4_bf16_entry_equals_f32_entry():
    rng = np.random.default_rng(9)
    w = round_bf16(rng.normal(0, 1, (8, 128)))
    a = oracle.mxfp4_quantize(w)
    b = oracle.mxfp4_quantize_f32(oracle.bf16_bits_to_f32(w))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------------------- P7: uintx
def test_uintx_hand_group():
    g = load("uintx_hand.json")["quant_case"]
    vals = g["values_first"] + [g["rest_of_group"]] * (g["group"] - len(g["values_first"]))
    w = np.tile(bf16_bits(vals), (2, 2))  # [2, 128]: 4 identical groups
    packed, sc, zp, codes = oracle.uintx_quantize(w, g["nbits"], g["group"])
    assert np.all(sc == int(g["scale_bits"], 16))
    assert np.all(zp == g["zp"])
    want = g["codes_first"] + [g["code_rest"]] * (g["group"] - len(g["codes_first"]))
    assert np.array_equal(codes, np.tile(np.array(want, np.uint8), (2, 2)))
    deq = oracle.uintx_dequantize(packed, sc, zp, 2, 128, g["nbits"], g["group"])
    table = g["dequant_by_code"]
    want_deq = np.array([table[c] for c in codes.reshape(-1)], np.float32).reshape(2, 128)
    assert np.array_equal(oracle.bf16_bits_to_f32(deq), want_deq)


def test_uintx_bf16_rounding_points():
    """Two hand-worked groups where skipping one bf16 rounding (of 1/scale, or of
    mn'/scale) would change a code or the zero point."""
    for g in load("uintx_hand.json")["rounding_point_cases"]:
        vals = g["values_first"] + [g["rest_of_group"]] * (g["group"] - len(g["values_first"]))
        packed, sc, zp, codes = oracle.uintx_quantize(bf16_bits([vals]), g["nbits"], g["group"])
        assert sc[0, 0] == int(g["scale_bits"], 16), g["name"]
        assert zp[0, 0] == g["zp"], g["name"]
        want = g["codes_first"] + [g["code_rest"]] * (g["group"] - len(g["codes_first"]))
        assert codes[0].tolist() == want, g["name"]


@pytest.mark.parametrize("nbits", [2, 3, 4, 5, 6, 7])
def test_uintx_power_of_two_grid(nbits):
    """When mx' - mn' = (2^nbits - 1) * 2^e the scale is exactly 2^e, the
    reciprocal is exact, and every grid point (q - zp) * 2^e reconstructs exactly
    with q = value / 2^e + zp."""
    rng = np.random.default_rng(100 + nbits)
    qmax = 2**nbits - 1
    e = -9
    n, k = 4, 256
    zp = rng.integers(0, qmax + 1, size=(n, k // 64))
    zp[:, 0] = 0  # all non-negative group: mn' = 0
    zp[:, 1] = qmax  # all non-positive group: mx' = 0
    q = rng.integers(0, qmax + 1, size=(n, k))
    for gi in range(k // 64):
        q[:, gi * 64] = 0
        q[:, gi * 64 + 1] = qmax
    zfull = np.repeat(zp, 64, axis=1)
    vals = ((q - zfull) * 2.0 ** e).astype(np.float32)
    packed, sc, zpo, codes = oracle.uintx_quantize(bf16_bits(vals), nbits)
    assert np.all(oracle.bf16_bits_to_f32(sc) == np.float32(2.0 ** e))
    assert np.array_equal(zpo, zp.astype(np.uint8))
    assert np.array_equal(codes, q.astype(np.uint8))
    deq = oracle.uintx_dequantize(packed, sc, zpo, n, k, nbits)
    assert np.array_equal(oracle.bf16_bits_to_f32(deq), vals)


def test_uintx_degenerate_groups():
    """All-zero group: scale clamps to fp32 eps = 2^-23, zp = 0, codes 0.
    All-positive group: zp = 0.  All-negative group: zp = qmax."""
    w = np.zeros((3, 64), np.float32)
    w[1] = np.linspace(0.01, 0.5, 64)
    w[2] = -np.linspace(0.01, 0.5, 64)
    wb = round_bf16(w)
    for nbits in (2, 5, 7):
        packed, sc, zp, codes = oracle.uintx_quantize(wb, nbits)
        assert oracle.bf16_to_f32(int(sc[0, 0])) == 2.0 ** -23
        assert zp[0, 0] == 0 and np.all(codes[0] == 0)
        assert zp[1, 0] == 0 and codes[1].max() == 2**nbits - 1
        assert zp[2, 0] == 2**nbits - 1 and codes[2].min() == 0


# --------------------------------------------------------------------------- P9: SNR
def test_quant_snr_closed_form_and_layouts():
    """quant_snr on the sym ramp with the oracle's own deq in both layouts and
    both deq dtypes; rel_err = sqrt(12.5 / 2731)."""
    s = 2.0 ** -6
    col = np.array([s * (-8 + i / 8) for i in range(128)], np.float32)
    w = np.tile(bf16_bits(col), (8, 1))
    qw, qz, sc, gi, _ = oracle.gptq_quantize(w, 128, True)
    deq_kn = oracle.gptq_dequantize(qw, qz, sc, 8, 128, 128, True, out_kn=True)
    deq_nk = oracle.gptq_dequantize(qw, qz, sc, 8, 128, 128, True, out_kn=False)
    want_snr = 10 * math.log10(2731 / 12.5)
    want_rel = math.sqrt(12.5 / 2731)
    for deq, kn in ((deq_kn, True), (deq_nk, False)):
        snr, rel = oracle.quant_snr(w, deq, deq_kn=kn)
        assert snr == pytest.approx(want_snr, rel=1e-9)
        assert rel == pytest.approx(want_rel, rel=1e-9)
    snr, rel = oracle.quant_snr(w, bf16_bits(deq_nk), deq_kn=False)  # exact: (c-8) * 2^-6
    assert snr == pytest.approx(want_snr, rel=1e-9)


def test_quant_snr_zero_weight_is_minus_inf():
    w = np.zeros((2, 64), np.uint16)
    snr, _ = oracle.quant_snr(w, np.zeros((2, 64), np.float32))
    assert snr == -math.inf


# --------------------------------------------------------------------------- P10: AWQ
ALPHAS = np.array([i / 10 for i in range(11)], np.float32)


def test_awq_scales_closed_form():
    """Without clamping, s = an^alpha / gm(an^alpha) = (a / gm(a))^alpha: the mean
    cancels.  alpha = 0 gives exactly 1."""
    rng = np.random.default_rng(20)
    a = np.exp(rng.normal(0, 0.5, 512)).astype(np.float32)
    s, ac = oracle.awq_prepare_scales(a, ALPHAS)
    assert np.all(s[0] == 1.0)
    gm = math.exp(np.mean(np.log(a.astype(np.float64))))
    for i, al in enumerate(ALPHAS):
        want = (a.astype(np.float64) / gm) ** float(al)
        np.testing.assert_allclose(s[i], want, rtol=2e-6)
    assert np.array_equal(ac, a)


def test_awq_scales_clamp_and_floor():
    """an^alpha is clamped to [1e-2, 1e2] before the geometric-mean normalisation,
    and a is floored at 1e-8 BEFORE the mean: with 99 channels at 1e-12 and one
    at 1e-4 the floored mean is (99e-8 + 1e-4)/100, which puts the small
    channels just under the 1e-2 clamp and the large one at 99.02 (not 100)."""
    a = np.array([1e-12] * 99 + [1e-4], np.float32)
    s, ac = oracle.awq_prepare_scales(a, np.array([1.0], np.float32))
    assert ac[0] == np.float32(1e-8) and ac[-1] == np.float32(1e-4)
    a_c = np.array([1e-8] * 99 + [1e-4])
    t = np.clip(a_c / a_c.mean(), 1e-2, 1e2)
    want = t / math.exp(np.mean(np.log(t)))
    np.testing.assert_allclose(s[0], want, rtol=1e-5)
    assert want[-1] / want[0] == pytest.approx(9902.0, rel=1e-3)


def test_awq_constant_activation_picks_first():
    """a = const -> an = 1 -> s = 1 for every alpha -> all errors equal -> the
    strict '<' keeps alpha 0."""
    rng = np.random.default_rng(21)
    w = round_bf16(rng.normal(0, 0.02, (64, 128)))
    best_s, bi, ba, errs = oracle.awq_search(w, np.full(128, 0.7, np.float32), ALPHAS)
    assert bi == 0 and ba == 0.0
    assert np.all(errs == errs[0])
    assert np.all(best_s == 1.0)


def test_awq_row_subsample_rule():
    """Rows 0, stride, 2*stride, ... (stride = N // max_rows), first max_rows of
    them: every other row can be garbage without changing anything."""
    rng = np.random.default_rng(22)
    n, k, max_rows = 40, 64, 16  # stride 2 -> rows 0, 2, ..., 30
    w = oracle.bf16_bits_to_f32(round_bf16(rng.normal(0, 0.02, (n, k))))
    a = np.exp(rng.normal(0, 1, k)).astype(np.float32)
    sub = w[0:32:2][:max_rows]
    poisoned = w.copy()
    mask = np.ones(n, bool)
    mask[0:32:2] = False
    poisoned[mask] = 1000.0
    r1 = oracle.awq_search(bf16_bits(poisoned), a, ALPHAS, max_rows=max_rows)
    r2 = oracle.awq_search(bf16_bits(sub), a, ALPHAS, max_rows=max_rows)
    assert np.array_equal(r1[3], r2[3]) and r1[1] == r2[1]
    # N not a multiple: N = 37 -> stride 2 -> rows 0..36 step 2 (19 rows) -> first 16
    w37 = w[:37]
    r3 = oracle.awq_search(bf16_bits(w37), a, ALPHAS, max_rows=16)
    r4 = oracle.awq_search(bf16_bits(w37[0:37:2][:16]), a, ALPHAS, max_rows=16)
    assert np.array_equal(r3[3], r4[3])


def test_awq_error_scales_with_activation():
    """Multiplying a by 2^j leaves s unchanged and multiplies every error by 4^j
    exactly (all roundings commute with a power-of-two scale)."""
    rng = np.random.default_rng(23)
    w = round_bf16(rng.normal(0, 0.02, (32, 128)))
    a = np.exp(rng.normal(0, 1, 128)).astype(np.float32)
    r1 = oracle.awq_search(w, a, ALPHAS)
    r2 = oracle.awq_search(w, (a * 8).astype(np.float32), ALPHAS)
    assert np.array_equal(r1[0], r2[0]) and r1[1] == r2[1]
    np.testing.assert_array_equal(r2[3], r1[3] * 64.0)


def test_awq_error_definition_small():
    """Brute force on a tiny W: err(alpha) = sum(((deq(quant(W*s))/s) - W) * a)^2
    composed in numpy from the separately pinned MXFP4 pieces."""
    rng = np.random.default_rng(24)
    wb = round_bf16(rng.normal(0, 0.02, (4, 64)))
    a = np.exp(rng.normal(0, 1, 64)).astype(np.float32)
    a[7] = 50.0  # one dominant channel
    best_s, bi, ba, errs = oracle.awq_search(wb, a, ALPHAS)
    s_all, ac = oracle.awq_prepare_scales(a, ALPHAS)
    wf = oracle.bf16_bits_to_f32(wb)
    want = []
    for i in range(len(ALPHAS)):
        ws = (wf * s_all[i]).astype(np.float32)
        d = oracle.mxfp4_dequantize(*oracle.mxfp4_quantize_f32(ws))
        e = ((d / s_all[i]).astype(np.float32) - wf).astype(np.float32) * ac
        want.append(float(np.sum((e.astype(np.float32) ** 2).astype(np.float64))))
    np.testing.assert_allclose(errs, want, rtol=1e-12)
    assert bi == int(np.argmin(want)) and ba == ALPHAS[bi]
    assert np.array_equal(best_s, s_all[bi])


# --------------------------------------------------------------------------- AWQ fold
# quantize_dflash_mxfp4.py, main(): (W.float() * s).to(bfloat16) on columns,
# (norm.float() / s).to(bfloat16), (up.float() / s.unsqueeze(1)).to(bfloat16) on rows.

def _fold_inputs(seed, n, k):
    rng = np.random.default_rng(seed)
    w = round_bf16(rng.normal(0, 0.02, (n, k)) * np.exp2(rng.integers(-30, 30, (n, k))))
    s_k = (np.exp(rng.normal(0, 1, k)) * np.exp2(rng.integers(-20, 20, k))).astype(np.float32)
    s_n = (np.exp(rng.normal(0, 1, n)) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
    return w, s_k, s_n


@pytest.mark.parametrize("op", [0, 1])
def test_awq_fold_matches_torch_expression(op):
    """P-F1: the page's own expression run by CPU torch, per column and per row."""
    torch = pytest.importorskip("torch")
    w, s_k, s_n = _fold_inputs(31 + op, 24, 64)
    wt = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)
    for axis, s in ((0, s_k), (1, s_n)):
        st = torch.from_numpy(s)
        st = st if axis == 0 else st.unsqueeze(1)
        ref = (wt.float() * st) if op == 0 else (wt.float() / st)
        ref = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(oracle.awq_fold(w, s, axis, op), ref)


def test_awq_fold_rounds_twice():
    """P-F2: binary32 product first, then bf16 (the page's .float() * s then
    .to(bfloat16)).  With w = W/128 (W odd) and s = m/2^23 the exact product is
    W*m*2^-30.  When it lies less than half a binary32 ulp (64 units) below a bf16
    midpoint whose upper neighbour is the even one, binary32 rounds it up onto
    the midpoint and bf16 then rounds the tie up, while a single rounding to bf16
    would go down.  Such (W, m) are built here; the values are checked with exact
    rational arithmetic."""
    from fractions import Fraction as F

    def rn(x: F, bits: int) -> F:  # nearest even with `bits` significant bits, x in [1, 2)
        scaled = x * 2 ** (bits - 1)
        fl = scaled.numerator // scaled.denominator
        rem = scaled - fl
        if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
            fl += 1
        return F(fl, 2 ** (bits - 1))

    cases = 0
    for W in range(129, 160, 2):                 # bf16 w = W/128 in (1, 1.25)
        for j in range(1, 127, 2):               # midpoint 1 + (2j+1) 2^-8, upper neighbour even
            M = 2 ** 30 + (2 * j + 1) * 2 ** 22
            r = M % W
            m = (M - r) // W
            if not (0 < r < 64 and 2 ** 23 <= m < 2 ** 24):
                continue
            w, sv = F(W, 128), F(m, 2 ** 23)
            once, twice = rn(w * sv, 8), rn(rn(w * sv, 24), 8)
            assert once != twice
            got = oracle.awq_fold(np.array([[0x3F80 + (W - 128)]], np.uint16),
                                  np.array([float(sv)], np.float32), 0, 0)
            assert F(float(oracle.bf16_bits_to_f32(got)[0, 0])) == twice
            cases += 1
    assert cases >= 3


def test_awq_fold_power_of_two_scales_are_exact():
    """P-F3: s = 2^j scales every finite bf16 exactly (no overflow/underflow here)."""
    rng = np.random.default_rng(33)
    w = round_bf16(rng.normal(0, 1, (8, 32)))
    j = rng.integers(-8, 9, 32)
    s = np.exp2(j).astype(np.float32)
    want = round_bf16(oracle.bf16_bits_to_f32(w) * s)
    assert np.array_equal(oracle.awq_fold(w, s, 0, 0), want)
    assert np.array_equal(oracle.awq_fold(w, (1.0 / s).astype(np.float32), 0, 1), want)


def test_awq_fold_rows_are_transposed_columns():
    """P-F4: folding rows of W equals folding columns of W^T, transposed back."""
    w, _, s_n = _fold_inputs(34, 16, 40)
    for op in (0, 1):
        a = oracle.awq_fold(w, s_n, 1, op)
        b = oracle.awq_fold(np.ascontiguousarray(w.T), s_n, 0, op).T
        assert np.array_equal(a, b)


# --------------------------------------------------------------------------- GPTQ consumer
def test_gptq_linear_one_hot_rows_pick_dequantized_columns():
    """P-L1: x = e_j (one-hot bf16 1.0) gives y[:, n] = deq[n, j] for every n:
    pins the orientation of the product (deq is [n, k], y = x deq^T), checked
    against the module-docstring dequant words of the hand-packed golden."""
    rng = np.random.default_rng(51)
    w = round_bf16(rng.normal(0, 0.02, (16, 256)))
    for sym in (True, False):
        qw, qz, sc, _, _ = oracle.gptq_quantize(w, 128, sym)
        codes = np.array([[(int(qw[kk // 8, nn]) >> (4 * (kk % 8))) & 15 for kk in range(256)]
                          for nn in range(16)])
        sc16 = sc.view(np.float16).astype(np.float64)  # [k/g, n]
        if sym:
            zp = np.full((2, 16), 8)
        else:
            zp = np.array([[(int(qz[g, nn // 8]) >> (4 * (nn % 8))) & 15 for nn in range(16)] for g in range(2)])
        for j in (0, 5, 127, 128, 255):
            x = np.zeros((1, 256), np.uint16)
            x[0, j] = 0x3F80
            y, _ = oracle.gptq_linear(x, qw, qz, sc, 16, 256, 128, sym)
            g = j // 128
            want = (codes[:, j] - zp[g]) * sc16[g]
            np.testing.assert_array_equal(y[0], want)


def test_gptq_linear_rows_are_independent_and_scale_exactly():
    """P-L2: each row of x gives its own output row (stacking rows stacks
    outputs), and a power-of-two factor on x scales y exactly."""
    rng = np.random.default_rng(52)
    w = round_bf16(rng.normal(0, 0.02, (24, 256)))
    qw, qz, sc, _, _ = oracle.gptq_quantize(w, 128, False)
    x = round_bf16(rng.normal(0, 1, (3, 256)))
    y, mag = oracle.gptq_linear(x, qw, qz, sc, 24, 256, 128, False)
    assert y.shape == mag.shape == (3, 24) and np.all(mag >= np.abs(y))
    for r in range(3):
        yr, _ = oracle.gptq_linear(x[r:r + 1], qw, qz, sc, 24, 256, 128, False)
        np.testing.assert_array_equal(yr[0], y[r])
    y4, _ = oracle.gptq_linear(round_bf16(oracle.bf16_bits_to_f32(x) * 4.0), qw, qz, sc, 24, 256, 128, False)
    np.testing.assert_array_equal(y4, 4.0 * y)


def test_mxfp4_linear_one_hot_rows_pick_dequantized_columns():
    """P-L3: x = e_j gives y[:, n] = +-E2M1[code] * 2^(e8m0 - 127) of weight
    (n, j), decoded here by hand from the packed nibble (even k low nibble) and
    the block's E8M0 byte: pins the orientation of the consumer's product."""
    rng = np.random.default_rng(53)
    w = round_bf16(rng.normal(0, 0.02, (12, 96)))
    p, e = oracle.mxfp4_quantize(w)
    for j in (0, 1, 31, 32, 95):
        x = np.zeros((1, 96), np.uint16)
        x[0, j] = 0x3F80
        y, _ = oracle.mxfp4_linear(x, p, e)
        byte = p[:, j // 2].astype(int)
        code = (byte >> 4) if j % 2 else (byte & 15)
        mag = np.array([E2M1[c & 7] for c in code]) * np.where(code & 8, -1.0, 1.0)
        want = mag * np.exp2(e[:, j // 32].astype(float) - 127)
        np.testing.assert_array_equal(y[0], want)


# ---------------------------------------------------------------- binary32 GPTQ input
# export_gptq_cpu.py quantizes w.float(): an fp16 or fp32 weight reaches the same
# binary32 arithmetic with more significant bits than bf16 holds.  Two hand-worked
# groups (k = group = 8, eight identical columns) use values that only binary32
# represents, placed so that rounding the input to bf16 first changes a code.
def _col8(vals):
    return np.tile(np.asarray(vals, np.float32).reshape(1, 8), (8, 1))


def _word(codes):
    return int(np.int32(np.uint32(sum(int(c) << (4 * i) for i, c in enumerate(codes)))))


def test_gptq_f32_sym_hand_group():
    e = 2.0 ** -26
    # amax 1.0 -> scale 1/8 exactly; x/scale = 8, -4, 1.5-2^-23, 1.5+2^-23, 2.5, -0.5, 2^-27, -8
    w = _col8([1.0, -0.5, 0.1875 - e, 0.1875 + e, 0.3125, -0.0625, 2.0 ** -30, -1.0])
    qw, qz, sc, gi, snr = oracle.gptq_quantize_f32(w, 8, True)
    codes = [15, 4, 9, 10, 10, 8, 8, 0]  # round half even, +8, clamp (16 -> 15)
    assert np.all(qw == _word(codes)) and np.all(sc == 0x3000) and np.all(qz == 0x77777777)
    deq = (np.asarray(codes, np.float64) - 8) * 0.125
    x = w[0].astype(np.float64)
    ref = 20 * np.log10(np.sqrt((x * x).sum()) / np.sqrt(((x - deq) ** 2).sum()))
    assert abs(snr - ref) <= 1e-6 * abs(ref)
    # the same values rounded to bf16 first give a different code (0.1875 - 2^-26 -> 0.1875 -> 1.5 -> 2)
    import torch

    wb = oracle.bf16_bits_to_f32(oracle._u16(torch.from_numpy(w).to(torch.bfloat16)))
    assert not np.array_equal(oracle.gptq_quantize_f32(wb, 8, True)[0], qw)


def test_gptq_f32_asym_hand_group():
    # wmin -0.46875, wmax 0.46875: scale = 0.9375 / 15 = 1/16 exactly; zp = rne(7.5) = 8
    w = _col8([-0.46875, 0.46875, 0.03125 + 2.0 ** -28, 0.03125, -0.09375, 0.15625 - 2.0 ** -26, 0.0, -0.25])
    qw, qz, sc, gi, snr = oracle.gptq_quantize_f32(w, 8, False)
    # x/scale = -7.5, 7.5, 0.5+2^-24, 0.5, -1.5, 2.5-2^-22, 0, -4 -> rne -8, 8, 1, 0, -2, 2, 0, -4; + 8
    codes = [0, 15, 9, 8, 6, 10, 8, 4]
    assert np.all(qw == _word(codes)) and np.all(sc == 0x2C00) and np.all(qz == _word([8] * 8))
    assert np.array_equal(gi, np.zeros(8, np.int32))


def test_gptq_f32_path_equals_bf16_path_on_bf16_values():
    from weight_only_bit_group_gb300 import synth

    w = synth.outlier_columns_bf16(64, 256, 0.02, 0.01, 20.0, 31)
    for sym in (True, False):
        a = oracle.gptq_quantize(w, 64, sym)
        b = oracle.gptq_quantize_f32(oracle.bf16_bits_to_f32(oracle._u16(w)), 64, sym)
        assert all(np.array_equal(x, y) for x, y in zip(a[:4], b[:4])) and a[4] == b[4]


# ---------------------------------------------------------------- uintx in the weight dtype
# uintx_quant.py works in the weight's own dtype.  Pins for binary16 and binary32:
# a hand-worked group whose every step is exact in all three types, and a
# cross-check of the oracle's C rounding against numpy's own float16 / float32
# arithmetic (each numpy op on those dtypes is the binary32 op rounded once to
# the dtype, the reading the oracle follows).
def test_uintx_dt_hand_group():
    vals = [-1.25, 2.5, 0.5, 0.375, -0.625, 1.0, 0.0, 0.125]
    # min_neg -1.25, max_pos 2.5: scale 3.75/15 = 0.25, 1/scale = 4, zp = 0 - round(-5) = 5
    # w * 4 = -5, 10, 2, 1.5, -2.5, 4, 0, 0.5 -> round half even -5, 10, 2, 2, -2, 4, 0, 0 -> + 5
    codes = [0, 15, 7, 7, 3, 9, 5, 5]
    for dt, npt in ((0, np.float32), (2, np.float16)):
        w = np.asarray([vals] * 2, npt)
        arr = w if dt == 0 else w.view(np.uint16)
        packed, sc, zp, c = oracle.uintx_quantize_dt(arr, dt, 4, 8)
        assert c.tolist() == [codes] * 2 and zp.tolist() == [[5], [5]]
        assert (sc.view(npt) if dt else sc).tolist() == [[0.25], [0.25]]
        d = oracle.uintx_dequantize_dt(packed, sc, dt, zp, 2, 8, 4, 8)
        d = d if dt == 0 else d.view(np.float16).astype(np.float32)
        assert d[0].tolist() == [-1.25, 2.5, 0.5, 0.5, -0.5, 1.0, 0.0, 0.0]


def _numpy_uintx(w, nbits, group):
    T = w.dtype.type
    n, k = w.shape
    qmax = (1 << nbits) - 1
    wg = w.reshape(n, k // group, group)
    mn = np.minimum(wg.min(axis=2), T(0))
    mx = np.maximum(wg.max(axis=2), T(0))
    sc = np.maximum((mx - mn) / T(qmax), T(np.finfo(np.float32).eps))
    zp = np.clip(T(0) - np.round(mn / sc), 0, qmax)
    inv = T(1) / sc
    q = np.clip(np.round(wg * inv[..., None]) + zp[..., None], 0, qmax)
    deq = (q - zp[..., None]) * sc[..., None]
    return q.reshape(n, k).astype(np.uint8), sc, zp.astype(np.uint8), deq.reshape(n, k)


@pytest.mark.parametrize("nbits", [2, 3, 5, 7])
def test_uintx_dt_matches_numpy_dtype_arithmetic(nbits):
    rng = np.random.default_rng(70 + nbits)
    base = rng.standard_normal((24, 256)) * np.exp(rng.standard_normal((24, 1)))
    for dt, npt in ((0, np.float32), (2, np.float16)):
        w = (base * 0.05).astype(npt)
        arr = w if dt == 0 else w.view(np.uint16)
        packed, sc, zp, codes = oracle.uintx_quantize_dt(arr, dt, nbits, 64)
        q_ref, sc_ref, zp_ref, deq_ref = _numpy_uintx(w, nbits, 64)
        assert np.array_equal(codes, q_ref) and np.array_equal(zp, zp_ref)
        assert np.array_equal(sc.view(npt) if dt else sc, sc_ref)
        d = oracle.uintx_dequantize_dt(packed, sc, dt, zp, 24, 256, nbits, 64)
        assert np.array_equal(d.view(npt) if dt else d, deq_ref.astype(npt))
