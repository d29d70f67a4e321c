"""Host side of checkpoint export (no GPU): the safetensors writer checked against
the file layout parsed independently here, the fused q_k_v split, and the
quantization_config schemas the serving side reads (export_gptq_cpu.py main();
quantize_dflash_mxfp4.py main())."""
import json
import struct

import numpy as np
import pytest
import torch

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import export, synth  # noqa: E402


def tensors():
    g = torch.Generator().manual_seed(3)
    return {
        "b.bf16": torch.randn(3, 5, generator=g).to(torch.bfloat16),
        "a.f16": torch.randn(7, generator=g).to(torch.float16),
        "c.i32": torch.randint(-2**31, 2**31 - 1, (4, 2), generator=g, dtype=torch.int64).to(torch.int32),
        "d.u8": torch.randint(0, 256, (9,), generator=g, dtype=torch.int64).to(torch.uint8),
        "e.f32": torch.randn(2, 2, 2, generator=g),
        "f.empty": torch.empty(0, 4, dtype=torch.bfloat16),
        "g.scalar": torch.tensor(2.5, dtype=torch.float64),
    }


def test_safetensors_layout(tmp_path):
    t = tensors()
    p = str(tmp_path / "m.safetensors")
    export.save_safetensors(p, t, metadata={"format": "pt"})
    raw = open(p, "rb").read()
    hl = int.from_bytes(raw[:8], "little")
    assert hl % 8 == 0 and 8 + hl <= len(raw)
    header = json.loads(raw[8:8 + hl].decode().rstrip(" "))
    assert header.pop("__metadata__") == {"format": "pt"}
    names = {"BF16": 2, "F16": 2, "I32": 4, "U8": 1, "F32": 4, "F64": 8}
    spans = []
    for name, e in header.items():
        ref = t[name]
        assert e["shape"] == list(ref.shape)
        b, en = e["data_offsets"]
        assert en - b == ref.numel() * names[e["dtype"]]
        blob = raw[8 + hl + b:8 + hl + en]
        # little-endian element bytes, row-major
        if e["dtype"] in ("BF16", "F16"):
            want = ref.contiguous().view(torch.int16).numpy().astype("<i2").tobytes()
        else:
            want = ref.numpy().astype(ref.numpy().dtype.newbyteorder("<")).tobytes()
        assert blob == want, name
        spans.append((b, en))
    spans.sort()
    assert spans[0][0] == 0 and all(x[1] == y[0] for x, y in zip(spans, spans[1:]))
    assert 8 + hl + spans[-1][1] == len(raw)


def test_safetensors_round_trip(tmp_path):
    t = tensors()
    p = str(tmp_path / "m.safetensors")
    export.save_safetensors(p, t)
    back, meta = export.load_safetensors(p)
    assert meta == {} and set(back) == set(t)
    for n in t:
        assert back[n].dtype == t[n].dtype and back[n].shape == t[n].shape
        assert torch.equal(back[n], t[n]), n


def test_split_fused_qkv():
    state, cfg = synth.tiny_decoder_state(n_layers=1)
    hd = cfg["head_dim"]
    qd, kvd = cfg["num_attention_heads"] * hd, cfg["num_key_value_heads"] * hd
    fused = state["model.layers.0.self_attn.q_k_v_proj.weight"]
    s = export.split_fused_qkv(state, qd, kvd)
    assert "model.layers.0.self_attn.q_k_v_proj.weight" not in s
    assert "model.layers.0.self_attn.q_k_v_proj.weight" in state  # caller's dict untouched
    for part, lo, hi in (("q_proj", 0, qd), ("k_proj", qd, qd + kvd), ("v_proj", qd + kvd, qd + 2 * kvd)):
        assert torch.equal(s[f"model.layers.0.self_attn.{part}.weight"], fused[lo:hi])
    assert hi == fused.shape[0]
    rest = {n for n in state if "q_k_v_proj" not in n}
    assert all(s[n] is state[n] for n in rest)
    # every quantized projection is one the page names; norms and the table pass through
    targets = [n for n in s if n.endswith(export.GPTQ_TARGET_SUFFIXES)]
    assert len(targets) == 7


def test_gptq_config_schema():
    c = export.gptq_quantization_config(64, True, True)
    assert c == {"quant_method": "gptq", "bits": 4, "group_size": 64, "desc_act": False, "sym": False,
                 "true_sequential": True, "checkpoint_format": "gptq", "lm_head": True}
    assert export.gptq_quantization_config(128, False, False)["sym"] is True


def test_quark_config_schema():
    c = export.quark_mxfp4_quantization_config()
    assert c["quant_method"] == "quark" and c["export"]["weight_format"] == "real_quantized"
    w, x = c["global_quant_config"]["weight"], c["global_quant_config"]["input_tensors"]
    for spec in (w, x):
        assert (spec["dtype"], spec["group_size"], spec["scale_format"], spec["round_method"],
                spec["qscheme"]) == ("fp4", 32, "e8m0", "half_even", "per_group")
    assert w["is_dynamic"] is False and x["is_dynamic"] is True
    json.dumps(c)  # serialisable as written


def test_mxfp4_targets():
    t = export.mxfp4_targets(2)
    assert len(t) == 15 and t[-1] == "fc.weight"
    st, act, cfg = synth.tiny_drafter_state(n_layers=2)
    assert set(t) <= set(st)
    assert len(act) == 6


def test_cli_requires_arguments():
    with pytest.raises(SystemExit):
        export.main(["gptq"])
    with pytest.raises(SystemExit):
        export.main([])


# ------------------------------------------------------------------ exporter logic on the CPU
# The exporters' host logic (q_k_v split, suffix selection, lm_head untie, report,
# config, the AWQ fold order) run with the kernel calls replaced by oracle-backed
# stand-ins: what is written must then equal the oracle composition exactly.
import oracle  # noqa: E402


@pytest.fixture
def oracle_kernels(monkeypatch):
    def bits(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dt)

    def gq(sym):
        def f(w, group=128, snr=True, **_):
            if w.dtype == torch.bfloat16:
                qw, qz, sc, gi, s = oracle.gptq_quantize(w, group, sym)
            else:  # fp16 / fp32 weights: the binary32 entry (the page's w.float())
                qw, qz, sc, gi, s = oracle.gptq_quantize_f32(w.float().numpy(), group, sym)
            return {"qweight": torch.from_numpy(qw), "qzeros": torch.from_numpy(qz),
                    "scales": bits(sc, torch.float16), "g_idx": torch.from_numpy(gi),
                    "snr_db": torch.tensor(s, dtype=torch.float64)}
        return f

    def gdq(qw, qz, sc, n, k, group, sym, out_dtype=torch.float32, **_):
        return torch.from_numpy(oracle.gptq_dequantize(qw.numpy(), qz.numpy(), sc, n, k, group, sym))

    def qsnr(w, deq, **_):
        s, r = oracle.quant_snr(w, deq)
        return torch.tensor(s), torch.tensor(r)

    def aws(w, a, alphas, max_rows=2048, **_):
        s, i, al, e = oracle.awq_search(w, a.numpy(), alphas, max_rows)
        return torch.from_numpy(s), torch.tensor(i), torch.tensor(al), torch.from_numpy(e)

    def fold(w, s, axis=0, op=0, *, out=None):
        r = bits(oracle.awq_fold(w, s.numpy(), axis, op).reshape(w.shape), torch.bfloat16)
        return out.copy_(r) if out is not None else r

    def mq(w, *a, **_):
        p, e = oracle.mxfp4_quantize(w)
        return torch.from_numpy(p), torch.from_numpy(e)

    def mdq(p, e, dt=torch.float32, **_):
        return torch.from_numpy(oracle.mxfp4_dequantize(p.numpy(), e.numpy()))

    monkeypatch.setattr(export, "gptq_quantize_sym", gq(True))
    monkeypatch.setattr(export, "gptq_quantize_asym", gq(False))
    for name, fn in (("gptq_dequantize", gdq), ("quant_snr", qsnr), ("awq_search", aws), ("awq_fold", fold),
                     ("mxfp4_quantize", mq), ("mxfp4_dequantize", mdq)):
        monkeypatch.setattr(wq, name, fn)


def test_gptq_export_logic(tmp_path, oracle_kernels):
    state, cfg = synth.tiny_decoder_state(n_layers=1)
    hd = cfg["head_dim"]
    state = export.split_fused_qkv(state, cfg["num_attention_heads"] * hd, cfg["num_key_value_heads"] * hd)
    out, report, summary = export.export_gptq(state, 64, True, quantize_embedding=False,
                                              quantize_lm_head=True, device="cpu")
    names = {r["name"] for r in report}
    assert names == {n for n in state if n.endswith(export.GPTQ_TARGET_SUFFIXES)} | {"lm_head"}
    assert export.EMBED_NAME in out and "lm_head.qweight" in out  # table kept, head untied
    qw, qz, sc, gi, snr = oracle.gptq_quantize(state[export.EMBED_NAME], 64, False)
    assert np.array_equal(out["lm_head.qweight"].numpy(), qw)
    assert summary["tensors"] == len(report) and summary["bits_per_weight"] == 4 + 20 / 64
    export.write_gptq_checkpoint(str(tmp_path), out, cfg, report, summary, 64, True, True)
    c = json.load(open(tmp_path / "config.json"))
    assert c["quantization_config"]["sym"] is False and c["tie_word_embeddings"] is False
    back, meta = export.load_safetensors(str(tmp_path / "model.safetensors"))
    assert set(back) == set(out) and all(torch.equal(back[k], out[k]) for k in out)
    res = export.verify_gptq_checkpoint(str(tmp_path), state, report, 64, True, device="cpu")
    assert [r["name"] for r in res] == [r["name"] for r in report]


def test_mxfp4_export_logic_fold_order(oracle_kernels):
    state, act, cfg = synth.tiny_drafter_state(n_layers=1)
    before = {k: v.clone() for k, v in state.items()}
    out, alphas, errs = export.export_mxfp4_awq(state, 1, act, device="cpu")
    assert [a for a, _ in alphas] == ["layers.0.qkv", "layers.0.gate_up", "layers.0.down"]
    # the norm is divided by the attention scale: redo that one fold by hand
    w = state["layers.0.self_attn.q_proj.weight"]
    cat = torch.cat([w, state["layers.0.self_attn.k_proj.weight"], state["layers.0.self_attn.v_proj.weight"]])
    s, _, _, _ = oracle.awq_search(cat, act["layers.0.self_attn.qkv_proj"].numpy(), synth.ALPHAS, 2048)
    ln = oracle.awq_fold(state["layers.0.input_layernorm.weight"], s, 0, 1).reshape(-1)
    assert np.array_equal(out["layers.0.input_layernorm.weight"].view(torch.int16).numpy().view(np.uint16), ln)
    assert "fc.weight_scale" in out and out["fc.weight"].dtype == torch.uint8
    assert len(errs) == len(export.mxfp4_targets(1))
    # the folds run in place on the exporter's own copies, never on the caller's tensors
    assert all(torch.equal(state[k], before[k]) for k in state)


def test_gptq_export_keeps_fp16_weights(oracle_kernels):
    """An fp16 checkpoint is quantized from its own values (export_gptq_cpu.py
    quantize_* start from w.float()), not from a bf16 rounding of them."""
    state, cfg = synth.tiny_decoder_state(n_layers=1)
    hd = cfg["head_dim"]
    state = export.split_fused_qkv(state, cfg["num_attention_heads"] * hd, cfg["num_key_value_heads"] * hd)
    g = torch.Generator().manual_seed(5)
    state = {k: (v.float() + torch.randn(v.shape, generator=g) * 1e-4).half() for k, v in state.items()}
    out, report, _ = export.export_gptq(state, 64, True, device="cpu")
    name = "model.layers.0.mlp.down_proj.weight"
    w = state[name]
    qw, qz, sc, gi, snr = oracle.gptq_quantize_f32(w.float().numpy(), 64, False)
    base = name[: -len(".weight")]
    assert np.array_equal(out[f"{base}.qweight"].numpy(), qw)
    assert np.array_equal(out[f"{base}.scales"].view(torch.int16).numpy().view(np.uint16), sc)
    # and differs from what a bf16 rounding of the weights would give
    qw_bf, *_ = oracle.gptq_quantize(w.to(torch.bfloat16), 64, False)
    assert not np.array_equal(qw_bf, qw)
