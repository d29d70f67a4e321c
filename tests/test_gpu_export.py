"""Checkpoint export on the GPU (export_gptq_cpu.py main(); quantize_dflash_mxfp4.py
main()) against the same steps composed from the oracle on the CPU: every tensor
written must match bit for bit, the reported SNR / relative errors within the
reductions' tolerance, and the files must read back as written."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

wq = pytest.importorskip("weight_only_bit_group_gb300")
from weight_only_bit_group_gb300 import export, synth  # noqa: E402

pytestmark = pytest.mark.gpu
REL = 1e-4


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def write_src(d, state, cfg, shards=2):
    os.makedirs(d, exist_ok=True)
    names = sorted(state)
    for i in range(shards):
        export.save_safetensors(os.path.join(d, f"model-{i:05d}.safetensors"),
                                {n: state[n] for n in names[i::shards]})
    with open(os.path.join(d, "config.json"), "w") as fh:
        json.dump(cfg, fh)
    with open(os.path.join(d, "tokenizer.json"), "w") as fh:
        fh.write('{"model": "synthetic"}')


# ------------------------------------------------------------------ GPTQ
@pytest.mark.parametrize("group,asym", [(128, False), (128, True), (64, True)])
def test_gptq_export_cli_matches_oracle(tmp_path, group, asym):
    state, cfg = synth.tiny_decoder_state()
    src, dst = str(tmp_path / "src"), str(tmp_path / "dst")
    write_src(src, state, cfg)
    argv = ["gptq", "--src", src, "--dst", dst, "--group", str(group), "--quantize-embedding",
            "--quantize-lm-head", "--verify"] + (["--asym"] if asym else [])
    export.main(argv)

    out, meta = export.load_safetensors(os.path.join(dst, "model.safetensors"))
    assert meta == {"format": "pt"}
    rep = json.load(open(os.path.join(dst, "quantization_report.json")))
    snr_of = {r["name"]: r["snr_db"] for r in rep["per_tensor"]}
    hd = cfg["head_dim"]
    split = export.split_fused_qkv(state, cfg["num_attention_heads"] * hd, cfg["num_key_value_heads"] * hd)
    expect_q = {n for n in split if n.endswith(export.GPTQ_TARGET_SUFFIXES)} | {export.EMBED_NAME}
    assert set(snr_of) == expect_q | {"lm_head"}
    for name in expect_q | {"lm_head"}:
        w = split[export.EMBED_NAME if name == "lm_head" else name]
        base = "lm_head" if name == "lm_head" else name[: -len(".weight")]
        qw, qz, sc, gi, snr = oracle.gptq_quantize(w, group, not asym)
        assert np.array_equal(out[f"{base}.qweight"].numpy(), qw), name
        assert np.array_equal(out[f"{base}.qzeros"].numpy(), qz), name
        assert np.array_equal(u16(out[f"{base}.scales"]), sc), name
        assert np.array_equal(out[f"{base}.g_idx"].numpy(), gi), name
        # the report rounds to 0.01 dB
        assert abs(snr_of[name] - snr) <= 0.005 + REL * abs(snr) + 1e-9, (name, snr_of[name], snr)
    passthrough = set(split) - expect_q
    assert passthrough and all(torch.equal(out[n], split[n]) for n in passthrough)
    assert len(out) == len(passthrough) + 4 * len(snr_of)

    c = json.load(open(os.path.join(dst, "config.json")))
    assert c["quantization_config"] == {"quant_method": "gptq", "bits": 4, "group_size": group,
                                        "desc_act": False, "sym": not asym, "true_sequential": True,
                                        "checkpoint_format": "gptq", "lm_head": True}
    assert c["tie_word_embeddings"] is False and c["hidden_size"] == cfg["hidden_size"]
    assert rep["tensors"] == len(snr_of) and rep["bits_per_weight"] == 4 + 20 / group
    assert rep["snr_db_min"] == min(snr_of.values())
    assert os.path.exists(os.path.join(dst, "tokenizer.json"))


def test_gptq_verify_reads_back_stored_scales(tmp_path):
    state, cfg = synth.tiny_decoder_state(seed=8, n_layers=1)
    state = export.split_fused_qkv(state, 256, 128)
    out, report, summary = export.export_gptq(state, 128, True)
    export.write_gptq_checkpoint(str(tmp_path), out, cfg, report, summary, 128, True, False)
    res = export.verify_gptq_checkpoint(str(tmp_path), state, report, 128, True)
    for r in res:
        w = state[r["name"]]
        n, k = w.shape
        b = r["name"][: -len(".weight")]
        deq = oracle.gptq_dequantize(out[f"{b}.qweight"].numpy(), out[f"{b}.qzeros"].numpy(),
                                     out[f"{b}.scales"], n, k, 128, False)
        snr, _ = oracle.quant_snr(w, deq)
        assert abs(r["snr_db"] - snr) <= REL * abs(snr), (r, snr)


# ------------------------------------------------------------------ MXFP4 + AWQ
def oracle_mxfp4_export(state, act, n_layers):
    """quantize_dflash_mxfp4.py main()'s steps composed from the oracle (bf16 bits)."""
    T = {k: u16(v) for k, v in state.items()}
    alphas = []

    def search(w, a):
        s, _, al, errs = oracle.awq_search(w, a.numpy(), synth.ALPHAS, 2048)
        e = np.sort(errs)
        assert e[1] - e[0] > 1e-3 * e[0], "two alphas too close to call"  # seed precondition
        return s, al

    def fold(n, s, axis, op):
        T[n] = oracle.awq_fold(T[n], s, axis, op).reshape(T[n].shape)

    for l in range(n_layers):
        P = f"layers.{l}"
        for norm, conv, projs, key, tag in (
                ("input_layernorm", "attention_conv", ["self_attn.q_proj", "self_attn.k_proj",
                                                       "self_attn.v_proj"], "self_attn.qkv_proj", "qkv"),
                ("post_attention_layernorm", "mlp_conv", ["mlp.gate_proj", "mlp.up_proj"],
                 "mlp.gate_up_proj", "gate_up")):
            names = [f"{P}.{p}.weight" for p in projs]
            s, al = search(np.concatenate([T[n] for n in names], 0), act[f"{P}.{key}"])
            fold(f"{P}.{norm}.weight", s, 0, 1)
            fold(f"{P}.{conv}.kernel_projection.weight", s, 0, 0)
            for n in names:
                fold(n, s, 0, 0)
            alphas.append((f"{P}.{tag}", al))
        s, al = search(T[f"{P}.mlp.down_proj.weight"], act[f"{P}.mlp.down_proj"])
        fold(f"{P}.mlp.up_proj.weight", s, 1, 1)
        fold(f"{P}.mlp.down_proj.weight", s, 0, 0)
        alphas.append((f"{P}.down", al))
    out, errs = {}, {}
    for n in export.mxfp4_targets(n_layers):
        p, e = oracle.mxfp4_quantize(T[n])
        out[n], out[n[: -len(".weight")] + ".weight_scale"] = p, e
        errs[n] = oracle.quant_snr(T[n], oracle.mxfp4_dequantize(p, e))[1]
    for n in T:
        out.setdefault(n, T[n])
    return out, alphas, errs


def check_mx_out(out, ref):
    assert set(out) == set(ref)
    for n, t in out.items():
        got = u16(t) if t.dtype == torch.bfloat16 else t.numpy()
        assert np.array_equal(got, ref[n]), n


def test_mxfp4_awq_export_matches_oracle():
    state, act, cfg = synth.tiny_drafter_state()
    nl = cfg["num_hidden_layers"]
    dev = {k: v.cuda() for k, v in state.items()}  # already resident: the folds must not reach them
    out, alphas, errs = export.export_mxfp4_awq(dev, nl, act)
    assert all(torch.equal(dev[k].cpu(), state[k]) for k in state)
    ref, ref_alphas, ref_errs = oracle_mxfp4_export(state, act, nl)
    assert [a for a, _ in alphas] == [a for a, _ in ref_alphas]
    assert np.allclose([v for _, v in alphas], [v for _, v in ref_alphas], rtol=0, atol=1e-6)
    check_mx_out(out, ref)
    for n, e in errs:
        assert abs(e - ref_errs[n]) <= REL * ref_errs[n], (n, e, ref_errs[n])


def test_mxfp4_export_cli_round_trip(tmp_path):
    state, act, cfg = synth.tiny_drafter_state(seed=10, n_layers=1)
    src, out_dir = str(tmp_path / "src"), str(tmp_path / "out")
    os.makedirs(src)
    export.save_safetensors(os.path.join(src, "model.safetensors"), state)
    json.dump(cfg, open(os.path.join(src, "config.json"), "w"))
    prefix = str(tmp_path / "calib")
    half = act["layers.0.mlp.down_proj"].numel() // 2  # down_proj's inputs, split over two ranks
    for r in range(2):
        d = {}
        for name, a in act.items():
            d[name] = {"absmean": a[r * half:(r + 1) * half] if name.endswith("down_proj") else a}
        torch.save(d, f"{prefix}.tp{r}.pt")
    export.main(["mxfp4", src, prefix, out_dir])
    got, meta = export.load_safetensors(os.path.join(out_dir, "model.safetensors"))
    assert meta == {"format": "pt"}
    ref, _, _ = oracle_mxfp4_export(state, act, 1)
    check_mx_out(got, ref)
    qc = json.load(open(os.path.join(out_dir, "config.json")))["quantization_config"]
    assert qc["quant_method"] == "quark" and qc["global_quant_config"]["weight"]["scale_format"] == "e8m0"
