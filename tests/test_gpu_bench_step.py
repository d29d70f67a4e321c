"""The benchmark's own step (bench.Workload: seven projections per phase on
concurrent streams, AWQ on a side stream, all captured in one CUDA graph) gives
the same products as the oracle: every output of the small projections and of
one large projection is compared, so a race between the concurrent calls would
show here."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REL = 1e-4


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.fixture(scope="module")
def step_outputs():
    sys.path.insert(0, ROOT)
    import bench

    dev = torch.device("cuda", 0)
    wl = bench.Workload(dev)
    phases = wl.phases()
    side = torch.cuda.Stream(dev)

    def body():
        main = torch.cuda.current_stream(dev)
        fork = torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        for name, fn, *rest in phases:
            if rest[-1] is None:
                with torch.cuda.stream(side):
                    fn()
            else:
                fn()
        join = torch.cuda.Event()
        join.record(side)
        main.wait_event(join)

    body()  # eager once (builds caches), then the captured step
    torch.cuda.synchronize(dev)
    for o in wl.out:  # poison the outputs so that the replay must rewrite them
        for tag in ("asym", "sym"):
            o[tag]["qweight"].fill_(0x5A5A5A5A)
            o[tag]["snr_db"].fill_(float("nan"))
        o["mx"]["packed"].fill_(0xA5)
        o["snr"]["rel_err"].fill_(float("nan"))
        o["ux"]["packed"].fill_(0xA5)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    g.replay()
    torch.cuda.synchronize(dev)
    return wl


@pytest.mark.parametrize("name", ["k_proj", "v_proj", "gate_proj"])
def test_step_products_match_oracle(step_outputs, name):
    wl = step_outputs
    idx = [n for n, _ in wl.layer].index(name)
    w = wl.layer[idx][1].cpu()
    o = wl.out[idx]
    for tag, sym in (("asym", False), ("sym", True)):
        qw, qz, sc, gi, snr = oracle.gptq_quantize(w, 128, sym)
        assert np.array_equal(o[tag]["qweight"].cpu().numpy(), qw), (name, tag)
        assert np.array_equal(o[tag]["qzeros"].cpu().numpy(), qz), (name, tag)
        assert np.array_equal(u16(o[tag]["scales"]), sc), (name, tag)
        got = float(o[tag]["snr_db"])
        assert abs(got - snr) <= REL * abs(snr), (name, tag, got, snr)
    p, e = oracle.mxfp4_quantize(w)
    assert np.array_equal(o["mx"]["packed"].cpu().numpy(), p), name
    assert np.array_equal(o["mx"]["e8m0"].cpu().numpy(), e), name
    _, rel = oracle.quant_snr(w, oracle.mxfp4_dequantize(p, e))
    assert abs(float(o["snr"]["rel_err"]) - rel) <= REL * rel, name
    packed, scale, zp, _ = oracle.uintx_quantize(w, 4, 64)
    assert np.array_equal(o["ux"]["packed"].cpu().numpy(), packed), name
    assert np.array_equal(u16(o["ux"]["scale"]).reshape(-1), np.asarray(scale).reshape(-1)), name
    assert np.array_equal(o["ux"]["zp"].cpu().numpy().reshape(-1), np.asarray(zp).reshape(-1)), name


def test_step_awq_alpha_matches_oracle(step_outputs):
    wl = step_outputs
    gu = wl.gate_up.cpu()
    best_s, bi, ba, errs = oracle.awq_search(gu, wl.act.cpu().numpy(), wl.alphas, 2048)
    got = wl.awq_out
    np.testing.assert_allclose(got["errs"].cpu().numpy(), errs, rtol=REL)
    order = np.argsort(errs)
    if errs[order[1]] - errs[order[0]] > 1e-9 * errs[order[0]]:  # not a near-tie
        assert int(got["best_idx"]) == bi
        np.testing.assert_allclose(got["best_s"].cpu().numpy(), best_s, rtol=2e-7)
