"""GPU parity of the AWQ fold (quantize_dflash_mxfp4.py, main(): the rewrite of
the weights after search_scale, then quantize_mxfp4 of every target and its
relative error) against the CPU oracle.  Bit-exact on every folded bf16 weight,
packed code and E8M0 byte; relative errors within 1e-4."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL = 1e-4


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def wide_weights(seed, n, k):
    """bf16 weights over a wide exponent range, with values near the bf16 maximum
    (products overflow to inf) and subnormal bf16 values (quotients underflow)."""
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(n, k, generator=g) * torch.exp2(torch.randint(-40, 40, (n, k), generator=g).float())
    w = w.to(torch.bfloat16)
    w.view(-1)[::97] = torch.tensor(3.0e38, dtype=torch.bfloat16)
    w.view(-1)[5::101] = torch.tensor(-2.0e-39, dtype=torch.bfloat16)
    w.view(-1)[7::103] = torch.tensor(-0.0, dtype=torch.bfloat16)
    return w


def scales(seed, m):
    g = torch.Generator().manual_seed(seed)
    s = torch.exp(torch.randn(m, generator=g)) * torch.exp2(torch.randint(-24, 24, (m,), generator=g).float())
    return s.float().contiguous()


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("op", [0, 1])
@pytest.mark.parametrize("shape", [(300, 1024), (7, 4104), (1, 4096)])
def test_awq_fold_bit_exact(axis, op, shape):
    n, k = shape
    w = wide_weights(40 + n, n, k)
    s = scales(41 + k, k if axis == 0 else n)
    got = wq.awq_fold(w.to(DEV), s.to(DEV), axis, op)
    want = oracle.awq_fold(w, s.numpy(), axis, op)
    assert np.array_equal(u16(got), want)


def test_awq_fold_in_place_norm_vector():
    """The norm weight [K] divided by s in place, as the page rewrites it."""
    k = 4096
    norm = (1.0 + 0.1 * torch.randn(k, generator=torch.Generator().manual_seed(42))).to(torch.bfloat16)
    s = scales(43, k)
    d = norm.to(DEV).clone()
    out = wq.awq_fold(d, s.to(DEV), 0, 1, out=d)
    assert out.data_ptr() == d.data_ptr()
    assert np.array_equal(u16(d), oracle.awq_fold(norm.view(1, -1), s.numpy(), 0, 1).reshape(-1))


def _pool(fn, items):
    with cf.ThreadPoolExecutor(max_workers=min(len(items), os.cpu_count() or 4)) as ex:
        return list(ex.map(fn, items))


def test_fold_then_mxfp4_layer_full_size():
    """The page's per-layer sequence on the seven projections: search on
    q||k||v and gate||up, fold s into those columns, search on down, divide up's
    rows and multiply down's columns by it, then quantize_mxfp4 every projection
    and take its relative error.  The searches run on the GPU; the oracle folds
    with the same s (the search itself is checked in test_gpu_parity.py)."""
    layer = dict(synth.gptq_layer(device="cpu"))
    q, k_, v = layer["q_proj"], layer["k_proj"], layer["v_proj"]
    g, u, d = layer["gate_proj"], layer["up_proj"], layer["down_proj"]
    dev = {name: t.to(DEV) for name, t in layer.items()}
    a_qkv = synth.awq_activation(q.shape[1], seed=4)
    a_gu = synth.awq_activation(g.shape[1], seed=5)
    a_d = synth.awq_activation(d.shape[1], seed=6)

    def search(ws, a):
        best_s, *_ = wq.awq_search(torch.cat(ws, 0), a.to(DEV), synth.ALPHAS, 2048)
        return best_s

    s_qkv = search([dev["q_proj"], dev["k_proj"], dev["v_proj"]], a_qkv)
    s_gu = search([dev["gate_proj"], dev["up_proj"]], a_gu)
    folded, want = {}, {}
    for name, s in (("q_proj", s_qkv), ("k_proj", s_qkv), ("v_proj", s_qkv),
                    ("gate_proj", s_gu), ("up_proj", s_gu)):
        folded[name] = wq.awq_fold(dev[name], s, 0, 0)
        want[name] = oracle.awq_fold(layer[name], s.cpu().numpy(), 0, 0)
    s_d = search([dev["down_proj"]], a_d)
    folded["up_proj"] = wq.awq_fold(folded["up_proj"], s_d, 1, 1, out=folded["up_proj"])
    want["up_proj"] = oracle.awq_fold(want["up_proj"], s_d.cpu().numpy(), 1, 1)
    folded["down_proj"] = wq.awq_fold(dev["down_proj"], s_d, 0, 0)
    want["down_proj"] = oracle.awq_fold(layer["down_proj"], s_d.cpu().numpy(), 0, 0)
    folded["o_proj"] = dev["o_proj"]
    want["o_proj"] = u16(layer["o_proj"])
    names = list(folded)
    for name in names:
        assert np.array_equal(u16(folded[name]), want[name]), name

    def ref(name):
        p, e = oracle.mxfp4_quantize(want[name])
        deq = oracle.mxfp4_dequantize(p, e)
        return p, e, oracle.quant_snr(want[name], deq)[1]

    refs = _pool(ref, names)
    for name, (p, e, rel) in zip(names, refs):
        gp, ge = wq.mxfp4_quantize(folded[name])
        assert np.array_equal(gp.cpu().numpy(), p), name
        assert np.array_equal(ge.cpu().numpy(), e), name
        deq = wq.mxfp4_dequantize(gp, ge, torch.float32)
        _, grel = wq.quant_snr(folded[name], deq, "nk")
        assert abs(float(grel) - rel) <= REL * rel, (name, float(grel), rel)
