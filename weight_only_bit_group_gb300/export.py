"""Checkpoint export around the quantize kernels.

GPTQ (export_gptq_cpu.py, main()): load a model's safetensors shards, split the
fused q_k_v projection along its output rows, quantize every linear weight whose
name ends with one of the page's suffixes (optionally the embedding, and an
untied copy of it as the lm_head), store four tensors per quantized weight --
<base>.qweight, .qzeros, .scales, .g_idx -- and write model.safetensors, a
config.json carrying the GPTQ quantization_config, and quantization_report.json
with the per-tensor SNR.  `--verify` re-reads the written tensors and measures
the SNR a consumer sees.

MXFP4 (quantize_dflash_mxfp4.py, main()): per decoder layer, search and fold the
AWQ scales (attention, MLP, down_proj), then store every served linear as packed
e2m1 codes under the weight's name and its E8M0 bytes under <base>.weight_scale,
with a quark quantization_config.

The same steps run on in-memory tensors, with every quantize, dequantize, scale
search, fold and SNR done by the library's kernels.  The file formats
(safetensors; the config fields) are the ones serving engines read, so they are
kept as they are.  Host-side plumbing only: no arithmetic of the method lives
here.
"""
from __future__ import annotations

import json
import os
import struct

import numpy as np
import torch

from . import gptq_quantize_asym, gptq_quantize_sym

# linear weights the page quantizes (by name suffix), and its embedding name
GPTQ_TARGET_SUFFIXES = (
    "self_attn.q_proj.weight", "self_attn.k_proj.weight", "self_attn.v_proj.weight",
    "self_attn.out_proj.weight", "mlp.gate_proj.weight", "mlp.up_proj.weight",
    "mlp.down_proj.weight",
)
EMBED_NAME = "model.embedding.weight"

# ------------------------------------------------------------------ safetensors
# File layout: u64 little-endian header length, a JSON header {name: {dtype,
# shape, data_offsets: [begin, end)}, "__metadata__": {...}} padded with spaces
# to a multiple of 8 bytes, then the tensors' bytes back to back.
_DTYPES = {torch.bfloat16: "BF16", torch.float16: "F16", torch.float32: "F32", torch.float64: "F64",
           torch.int32: "I32", torch.int64: "I64", torch.uint8: "U8", torch.int8: "I8",
           torch.int16: "I16", torch.bool: "BOOL"}
_BACK = {v: k for k, v in _DTYPES.items()}


def save_safetensors(path: str, tensors: dict, metadata: dict | None = None) -> None:
    header, blobs, off = {}, [], 0
    for name in sorted(tensors):
        t = tensors[name].detach().to("cpu").contiguous()
        raw = t.reshape(-1).view(torch.uint8).numpy().tobytes() if t.numel() else b""
        header[name] = {"dtype": _DTYPES[t.dtype], "shape": list(t.shape), "data_offsets": [off, off + len(raw)]}
        blobs.append(raw)
        off += len(raw)
    if metadata:
        header["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    h = json.dumps(header, separators=(",", ":")).encode()
    h += b" " * (-len(h) % 8)
    with open(path, "wb") as fh:
        fh.write(struct.pack("<Q", len(h)))
        fh.write(h)
        for raw in blobs:
            fh.write(raw)


def load_safetensors(path: str) -> tuple[dict, dict]:
    """-> (tensors on the CPU, metadata)."""
    with open(path, "rb") as fh:
        (hl,) = struct.unpack("<Q", fh.read(8))
        header = json.loads(fh.read(hl))
        data = fh.read()
    meta = header.pop("__metadata__", {})
    out = {}
    for name, e in header.items():
        b, en = e["data_offsets"]
        dt = _BACK[e["dtype"]]
        if en == b:
            out[name] = torch.empty(e["shape"], dtype=dt)
            continue
        buf = np.frombuffer(data[b:en], dtype=np.uint8).copy()
        out[name] = torch.from_numpy(buf).view(dt).reshape(e["shape"])
    return out, meta


# ------------------------------------------------------------------ GPTQ export
def split_fused_qkv(state: dict, q_dim: int, kv_dim: int) -> dict:
    """Replace every *.self_attn.q_k_v_proj.* tensor by its q/k/v parts along
    dim 0 (output rows); the grouping runs along K, so the split commutes with
    quantization and the parts are quantized as the ordinary projections."""
    state = dict(state)
    for name in [k for k in state if ".self_attn.q_k_v_proj." in k]:
        q, k, v = state.pop(name).split([q_dim, kv_dim, kv_dim], dim=0)
        for part, t in (("q_proj", q), ("k_proj", k), ("v_proj", v)):
            state[name.replace("q_k_v_proj", part)] = t.contiguous()
    return state


def gptq_quantization_config(group: int, asym: bool, lm_head: bool) -> dict:
    """The GPTQ quantization_config fields the serving side reads."""
    return {"quant_method": "gptq", "bits": 4, "group_size": group, "desc_act": False,
            "sym": not asym, "true_sequential": True, "checkpoint_format": "gptq", "lm_head": lm_head}


def export_gptq(state: dict, group: int = 128, asym: bool = False, quantize_embedding: bool = False,
                quantize_lm_head: bool = False, device="cuda"):
    """Quantize the page's target tensors of `state` ({name: bf16 CPU tensor})
    with the GPU kernels.  -> (out tensors on the CPU, per-tensor report, summary)."""
    quantize = gptq_quantize_asym if asym else gptq_quantize_sym
    out, report = {}, []

    def q(name, t, base):
        # bf16, fp16 and fp32 weights are quantized as they are (the page starts
        # from w.float(); fp16 / fp32 take the library's binary32 path); any other
        # floating type is widened to binary32 first
        if t.dtype not in (torch.bfloat16, torch.float16, torch.float32):
            t = t.float()
        r = quantize(t.to(device=device).contiguous(), group, True)
        for key in ("qweight", "qzeros", "scales", "g_idx"):
            out[f"{base}.{key}"] = r[key].cpu()
        report.append({"name": name, "snr_db": round(float(r["snr_db"]), 2)})

    for name, t in sorted(state.items()):
        if name.endswith(GPTQ_TARGET_SUFFIXES) or (name == EMBED_NAME and quantize_embedding):
            q(name, t, name[: -len(".weight")])
        else:
            out[name] = t
    if quantize_lm_head:
        # the head is untied from the embedding table and gets its own 4-bit copy
        q("lm_head", state[EMBED_NAME], "lm_head")
    snrs = [r["snr_db"] for r in report]
    summary = {"group": group, "tensors": len(report),
               "snr_db_mean": round(sum(snrs) / len(snrs), 2) if snrs else None,
               "snr_db_min": round(min(snrs), 2) if snrs else None,
               "bits_per_weight": 4 + (16 + 4) / group,  # codes + fp16 scale + 4-bit zero per group
               "quantized_embedding": quantize_embedding, "quantized_lm_head": quantize_lm_head}
    return out, report, summary


def write_gptq_checkpoint(dst: str, out: dict, config: dict, report: list, summary: dict,
                          group: int, asym: bool, quantize_lm_head: bool) -> None:
    """model.safetensors, config.json (+ quantization_config) and
    quantization_report.json in `dst`."""
    os.makedirs(dst, exist_ok=True)
    save_safetensors(os.path.join(dst, "model.safetensors"), out, metadata={"format": "pt"})
    cfg = dict(config)
    cfg["quantization_config"] = gptq_quantization_config(group, asym, quantize_lm_head)
    if quantize_lm_head:
        cfg["tie_word_embeddings"] = False
    with open(os.path.join(dst, "config.json"), "w") as fh:
        json.dump(cfg, fh, indent=2)
    with open(os.path.join(dst, "quantization_report.json"), "w") as fh:
        json.dump({**summary, "per_tensor": report}, fh, indent=2)


def verify_gptq_checkpoint(dst: str, state: dict, report: list, group: int, asym: bool,
                           device="cuda") -> list:
    """Re-read model.safetensors from `dst` and measure each quantized tensor's
    reconstruction SNR as a consumer sees it: dequantized from the stored fp16
    scales (the quantize step's own SNR uses the unrounded binary32 scale).
    -> [{"name", "snr_db"}] in report order."""
    from . import gptq_dequantize, quant_snr

    t, _ = load_safetensors(os.path.join(dst, "model.safetensors"))
    res = []
    for r in report:
        name = r["name"]
        base = "lm_head" if name == "lm_head" else name[: -len(".weight")]
        w = (state[EMBED_NAME] if name == "lm_head" else state[name]).to(device=device, dtype=torch.bfloat16)
        n, k = w.shape
        deq = gptq_dequantize(*(t[f"{base}.{x}"].to(device) for x in ("qweight", "qzeros", "scales")),
                              n, k, group, not asym, torch.float32)
        snr, _ = quant_snr(w.contiguous(), deq)
        res.append({"name": name, "snr_db": float(snr)})
    return res


# ------------------------------------------------------------------ MXFP4 + AWQ export
# quantize_dflash_mxfp4.py main(): per decoder layer, three AWQ scale searches
# and folds, then every served linear goes to packed e2m1 [N, K/2] (stored under
# the weight's own name) plus its E8M0 bytes [N, K/32] under "<base>.weight_scale".
def mxfp4_targets(n_layers: int) -> list:
    t = []
    for l in range(n_layers):
        t += [f"layers.{l}.self_attn.{x}_proj.weight" for x in ("q", "k", "v", "o")]
        t += [f"layers.{l}.mlp.{x}_proj.weight" for x in ("gate", "up", "down")]
    return t + ["fc.weight"]


def awq_fold_layers(T: dict, n_layers: int, act: dict, alphas=None, max_rows: int = 2048) -> list:
    """Search and fold the AWQ scales of every layer in place on the device tensors
    T (bf16).  act["layers.{l}.self_attn.qkv_proj" | ".mlp.gate_up_proj" |
    ".mlp.down_proj"] = per-input-channel mean |x| (f32 [K], tensor-parallel
    shards already concatenated).  -> [(group name, alpha)].

    attention: s from [q; k; v]; input_layernorm /= s; the conv's
      kernel_projection columns *= s (its coefficients then see the unscaled
      input); q, k, v columns *= s.
    mlp: the same with post_attention_layernorm, mlp_conv and [gate; up].
    down_proj: s from down alone; up's output rows /= s, down's columns *= s.
    Every fold rounds to bf16, in this order."""
    from . import awq_fold, awq_search
    from .synth import ALPHAS

    alphas = ALPHAS if alphas is None else alphas
    MUL, DIV, COLS, ROWS = 0, 1, 0, 1
    chosen = []

    def search(w, name):
        s, _, alpha, _ = awq_search(w.contiguous(), act[name].to(w.device, torch.float32).contiguous(),
                                    alphas, max_rows)
        return s, round(float(alpha), 6)

    def fold(name, s, axis, op):
        awq_fold(T[name], s, axis, op, out=T[name])

    for l in range(n_layers):
        P = f"layers.{l}"
        for norm, conv, projs, key in (
                ("input_layernorm", "attention_conv", [f"self_attn.{x}_proj" for x in "qkv"],
                 "self_attn.qkv_proj"),
                ("post_attention_layernorm", "mlp_conv", ["mlp.gate_proj", "mlp.up_proj"],
                 "mlp.gate_up_proj")):
            names = [f"{P}.{p}.weight" for p in projs]
            s, alpha = search(torch.cat([T[n] for n in names], 0), f"{P}.{key}")
            fold(f"{P}.{norm}.weight", s, COLS, DIV)
            fold(f"{P}.{conv}.kernel_projection.weight", s, COLS, MUL)
            for n in names:
                fold(n, s, COLS, MUL)
            chosen.append((f"{P}.{'qkv' if key.startswith('self_attn') else 'gate_up'}", alpha))
        dn, un = f"{P}.mlp.down_proj.weight", f"{P}.mlp.up_proj.weight"
        s, alpha = search(T[dn], f"{P}.mlp.down_proj")
        fold(un, s, ROWS, DIV)
        fold(dn, s, COLS, MUL)
        chosen.append((f"{P}.down", alpha))
    return chosen


def export_mxfp4_awq(state: dict, n_layers: int, act: dict, alphas=None, max_rows: int = 2048,
                     device="cuda"):
    """AWQ fold + MXFP4 quantization of a bf16 state dict (all on the GPU).
    -> (out tensors on the CPU, [(group, alpha)], [(target, relative error)])."""
    from . import mxfp4_dequantize, mxfp4_quantize, quant_snr

    # a copy: the folds run in place and must not reach the caller's tensors
    T = {k: v.to(device=device, dtype=torch.bfloat16, copy=True).contiguous() for k, v in state.items()}
    alphas_chosen = awq_fold_layers(T, n_layers, act, alphas, max_rows)
    targets = set(mxfp4_targets(n_layers))
    out, errs = {}, []
    for name, w in T.items():
        if name in targets:
            packed, e8m0 = mxfp4_quantize(w)
            _, rel = quant_snr(w, mxfp4_dequantize(packed, e8m0, torch.float32))
            out[name] = packed.cpu()
            out[name[: -len(".weight")] + ".weight_scale"] = e8m0.cpu()
            errs.append((name, float(rel)))
        else:
            out[name] = w.cpu()
    return out, alphas_chosen, errs


def quark_mxfp4_quantization_config(version: str = "0.12+wq-gb300-awq-mxfp4") -> dict:
    """The quark quantization_config a serving engine reads for OCP MXFP4
    weights: fp4 per-group-32 with E8M0 scales and half-even rounding for the
    (static) weights and the (dynamic) activations, real_quantized export."""
    def spec(dynamic: bool) -> dict:
        return {"dtype": "fp4", "qscheme": "per_group", "group_size": 32, "ch_axis": -1,
                "scale_format": "e8m0", "scale_type": "float", "scale_calculation_mode": "even",
                "round_method": "half_even", "observer_cls": "PerBlockMXObserver",
                "is_dynamic": dynamic, "is_scale_quant": False, "symmetric": None, "block_size": None,
                "mx_element_dtype": None, "enable_buffer_reuse": False, "max_input_numel": 4194304}
    return {"quant_method": "quark", "quant_mode": "eager_mode", "version": version,
            "global_quant_config": {"weight": spec(False), "input_tensors": spec(True),
                                    "output_tensors": None, "bias": None, "target_device": None},
            "export": {"weight_format": "real_quantized", "pack_method": "reorder",
                       "kv_cache_group": [], "min_kv_scale": 0.0, "weight_merge_groups": None},
            "exclude": [], "algo_config": None, "layer_quant_config": {}, "layer_type_quant_config": {},
            "kv_cache_quant_config": {}, "kv_cache_post_rope": False, "softmax_quant_spec": None}


# ------------------------------------------------------------------ command line
_SIDE_FILES = ("tokenizer.json", "tokenizer_config.json", "special_tokens_map.json", "vocab.json",
               "merges.txt", "generation_config.json", "chat_template.jinja")


def _gptq_main(a) -> None:
    import shutil

    state = {}
    for shard in sorted(f for f in os.listdir(a.src) if f.endswith(".safetensors")):
        state.update(load_safetensors(os.path.join(a.src, shard))[0])
    with open(os.path.join(a.src, "config.json")) as fh:
        cfg = json.load(fh)
    head_dim = cfg.get("head_dim") or cfg["hidden_size"] // cfg["num_attention_heads"]
    state = split_fused_qkv(state, cfg["num_attention_heads"] * head_dim,
                            cfg["num_key_value_heads"] * head_dim)
    out, report, summary = export_gptq(state, a.group, a.asym, a.quantize_embedding, a.quantize_lm_head)
    write_gptq_checkpoint(a.dst, out, cfg, report, summary, a.group, a.asym, a.quantize_lm_head)
    for f in _SIDE_FILES:
        if os.path.exists(os.path.join(a.src, f)):
            shutil.copy(os.path.join(a.src, f), os.path.join(a.dst, f))
    print(json.dumps(summary, indent=2))
    if a.verify:
        for r in verify_gptq_checkpoint(a.dst, state, report, a.group, a.asym):
            print(f"  {r['name']:<48} {r['snr_db']:.2f} dB (re-read)")


def _mxfp4_main(a) -> None:
    state, _ = load_safetensors(os.path.join(a.src, "model.safetensors"))
    with open(os.path.join(a.src, "config.json")) as fh:
        cfg = json.load(fh)
    nl = cfg["num_hidden_layers"]
    c0 = torch.load(f"{a.calib_prefix}.tp0.pt", map_location="cpu", weights_only=True)
    c1 = torch.load(f"{a.calib_prefix}.tp1.pt", map_location="cpu", weights_only=True)
    act = {}
    for l in range(nl):
        P = f"layers.{l}"
        for key in ("self_attn.qkv_proj", "mlp.gate_up_proj"):  # replicated input: rank 0's
            act[f"{P}.{key}"] = c0[f"{P}.{key}"]["absmean"]
        # row-parallel: each rank saw half of down_proj's input channels
        act[f"{P}.mlp.down_proj"] = torch.cat([c0[f"{P}.mlp.down_proj"]["absmean"],
                                               c1[f"{P}.mlp.down_proj"]["absmean"]])
    out, alphas, errs = export_mxfp4_awq(state, nl, act, max_rows=a.max_rows)
    os.makedirs(a.out, exist_ok=True)
    save_safetensors(os.path.join(a.out, "model.safetensors"), out, metadata={"format": "pt"})
    cfg["quantization_config"] = quark_mxfp4_quantization_config()
    with open(os.path.join(a.out, "config.json"), "w") as fh:
        json.dump(cfg, fh, indent=2)
    print(f"quantized {len(errs)} linears -> {a.out}")
    for name, al in alphas:
        print(f"  {name:<28} alpha={al:.2f}")
    errs.sort(key=lambda e: -e[1])
    for name, e in errs[:6]:
        print(f"  {name:<44} {e:.4f}")
    if errs:
        print(f"  mean {sum(e for _, e in errs) / len(errs):.4f} over {len(errs)} tensors")


def main(argv=None) -> None:
    import argparse

    ap = argparse.ArgumentParser(prog="python -m weight_only_bit_group_gb300.export")
    sub = ap.add_subparsers(dest="cmd", required=True)
    g = sub.add_parser("gptq", help="4-bit GPTQ checkpoint (sym or asym, group-wise along K)")
    g.add_argument("--src", required=True)
    g.add_argument("--dst", required=True)
    g.add_argument("--group", type=int, default=128)
    g.add_argument("--asym", action="store_true")
    g.add_argument("--quantize-embedding", action="store_true")
    g.add_argument("--quantize-lm-head", action="store_true")
    g.add_argument("--verify", action="store_true", help="re-read the written tensors, report SNR")
    m = sub.add_parser("mxfp4", help="AWQ-folded OCP MXFP4 checkpoint (quark format)")
    m.add_argument("src")
    m.add_argument("calib_prefix")
    m.add_argument("out")
    m.add_argument("--max-rows", type=int, default=2048)
    a = ap.parse_args(argv)
    (_gptq_main if a.cmd == "gptq" else _mxfp4_main)(a)


if __name__ == "__main__":
    main()
