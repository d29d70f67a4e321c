"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no quantization arithmetic: it only draws random tensors
(torch generators, seeded) and hands back bf16 weights / fp32 activation
statistics.  Tests feed the same tensors to the CUDA library and to the CPU
oracle; the benchmark uses them as its workload.  The pages' real inputs are
model checkpoints and calibration statistics that are not available, so these
stand in for their shapes and value ranges:

  * GPTQ layer (export_gptq_cpu.py targets q/k/v/o/gate/up/down): hidden 4096,
    intermediate 14336, 8 KV heads of 128 -> k/v [1024, 4096]; N(0, 0.02) with
    0.5% of input columns scaled x20 (activation-outlier channels).
  * MXFP4 gate_up (quantize_dflash_mxfp4.py docstring, [34816, 5120]): N(0,
    0.015) with 1% of the 32-value blocks scaled x50.
  * AWQ activation statistics: per-channel mean |x| ~ LogNormal(0, 1).
  * uintx: 8 layers of the GPTQ layer shapes, N(0, 0.02).
"""
from __future__ import annotations

import math

import torch

LAYER_SHAPES = [
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 14336, 4096),
    ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
]
GATE_UP_SHAPE = (34816, 5120)
ALPHAS = [i / 10 for i in range(11)]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_f32(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(std)


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    return normal_f32(shape, std, seed, device).to(torch.bfloat16)


def outlier_columns_bf16(n: int, k: int, std: float, frac: float, factor: float, seed: int,
                         device="cpu") -> torch.Tensor:
    """N(0, std) with ceil(frac * k) randomly chosen input columns multiplied by factor."""
    w = normal_f32((n, k), std, seed, device)
    g = _gen(seed + 1000, device)
    cols = torch.randperm(k, generator=g, device=device)[: math.ceil(frac * k)]
    w[:, cols] *= factor
    return w.to(torch.bfloat16)


def outlier_blocks_bf16(n: int, k: int, std: float, frac: float, factor: float, seed: int,
                        block: int = 32, device="cpu") -> torch.Tensor:
    """N(0, std) with a random fraction of the contiguous `block`-value blocks scaled."""
    w = normal_f32((n, k), std, seed, device)
    nb = n * k // block
    g = _gen(seed + 1000, device)
    sel = torch.randperm(nb, generator=g, device=device)[: int(frac * nb)]
    w.view(nb, block)[sel] *= factor
    return w.to(torch.bfloat16)


def gptq_layer(seed: int = 2, device="cpu", shapes=LAYER_SHAPES):
    """One transformer layer's seven projections: [(name, bf16 [N, K])]."""
    return [(name, outlier_columns_bf16(n, k, 0.02, 0.005, 20.0, seed + i, device))
            for i, (name, n, k) in enumerate(shapes)]


def small_gptq(seed: int = 1, device="cpu") -> torch.Tensor:
    return normal_bf16((256, 512), 0.02, seed, device)


def gptq_packed(n: int, k: int, group: int, seed: int, device="cpu"):
    """Random stored GPTQ tensors of an [n, k] weight, as a checkpoint would hold
    them: qweight int32 [k/8, n] and qzeros int32 [k/group, n/8] with uniformly
    random nibbles (every code and zero point), scales fp16 [k/group, n] drawn
    LogNormal around 0.0025 (the scale of N(0, 0.02) weights at 4 bits).
    -> (qweight, qzeros, scales)."""
    g = _gen(seed, "cpu")
    qw = torch.randint(-2 ** 31, 2 ** 31, (k // 8, n), generator=g, dtype=torch.int64).to(torch.int32)
    qz = torch.randint(-2 ** 31, 2 ** 31, (k // group, n // 8), generator=g, dtype=torch.int64).to(torch.int32)
    sc = (torch.randn((k // group, n), generator=g) + math.log(0.0025)).exp_().to(torch.float16)
    return qw.to(device), qz.to(device), sc.to(device)


def mxfp4_gate_up(seed: int = 3, device="cpu", shape=GATE_UP_SHAPE) -> torch.Tensor:
    n, k = shape
    return outlier_blocks_bf16(n, k, 0.015, 0.01, 50.0, seed, 32, device)


def mxfp4_tie_rows(n_rows: int = 64, k: int = 5120, seed: int = 6, device="cpu") -> torch.Tensor:
    """Blocks built to land on exact e2m1 midpoints: each 32-block has one
    element 6 * 2^e (fixing the block exponent at e) and the rest k * 0.25 * 2^e
    with k in 0..24, random signs, e drawn from [-120, 120]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    nb = n_rows * k // 32
    e = torch.randint(-120, 121, (nb, 1), generator=g).to(torch.float64)
    steps = torch.randint(0, 25, (nb, 32), generator=g).to(torch.float64) * 0.25
    signs = torch.where(torch.rand((nb, 32), generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    vals = steps * signs
    pos = torch.randint(0, 32, (nb,), generator=g)
    vals[torch.arange(nb), pos] = 6.0
    w = (vals * torch.exp2(e)).to(torch.float32).view(n_rows, k)
    return w.to(torch.bfloat16).to(device)


def awq_activation(k: int = 5120, seed: int = 4, device="cpu") -> torch.Tensor:
    return normal_f32((k,), 1.0, seed, device).exp_()


def uintx_layers(n_layers: int = 8, seed: int = 5, device="cpu", shapes=LAYER_SHAPES):
    """n_layers x seven projections: [(name, bf16 [N, K])]."""
    out = []
    for layer in range(n_layers):
        for i, (name, n, k) in enumerate(shapes):
            out.append((f"layers.{layer}.{name}",
                        normal_bf16((n, k), 0.02, seed + 100 * layer + i, device)))
    return out


def tiny_decoder_state(seed: int = 7, n_layers: int = 2, hidden: int = 256, heads: int = 4,
                       kv_heads: int = 2, head_dim: int = 64, inter: int = 512, vocab: int = 1024):
    """A small decoder's bf16 state dict under the GPTQ exporter's tensor names,
    with the fused q_k_v projection [(heads + 2 kv_heads) * head_dim, hidden],
    plus the config fields the exporter reads.  -> (state, config)."""
    st, i = {}, 0

    def w(shape, std=0.02):
        nonlocal i
        i += 1
        if len(shape) == 2:
            return outlier_columns_bf16(shape[0], shape[1], std, 0.005, 20.0, seed * 100 + i)
        return (1.0 + normal_f32(shape, 0.1, seed * 100 + i)).to(torch.bfloat16)

    qkv = (heads + 2 * kv_heads) * head_dim
    st["model.embedding.weight"] = w((vocab, hidden))
    st["model.norm.weight"] = w((hidden,))
    for l in range(n_layers):
        P = f"model.layers.{l}"
        st[f"{P}.input_layernorm.weight"] = w((hidden,))
        st[f"{P}.post_attention_layernorm.weight"] = w((hidden,))
        st[f"{P}.self_attn.q_k_v_proj.weight"] = w((qkv, hidden))
        st[f"{P}.self_attn.out_proj.weight"] = w((hidden, heads * head_dim))
        st[f"{P}.mlp.gate_proj.weight"] = w((inter, hidden))
        st[f"{P}.mlp.up_proj.weight"] = w((inter, hidden))
        st[f"{P}.mlp.down_proj.weight"] = w((hidden, inter))
    cfg = {"hidden_size": hidden, "num_attention_heads": heads, "num_key_value_heads": kv_heads,
           "head_dim": head_dim, "intermediate_size": inter, "num_hidden_layers": n_layers,
           "vocab_size": vocab, "tie_word_embeddings": True}
    return st, cfg


def tiny_drafter_state(seed: int = 9, n_layers: int = 2, hidden: int = 256, q_dim: int = 256,
                       kv_dim: int = 64, inter: int = 512, taps: int = 8, target_hidden: int = 512):
    """A small drafter's bf16 state dict under the MXFP4 exporter's tensor names
    (separate q/k/v, dynamic-conv kernel projections, fc over the target's
    hidden states) and its per-channel activation statistics mean |x| ~
    LogNormal(0, 1).  -> (state, act, config)."""
    st, act, i = {}, {}, 0

    def w(shape, std=0.02):
        nonlocal i
        i += 1
        if len(shape) == 2:
            return outlier_columns_bf16(shape[0], shape[1], std, 0.005, 20.0, seed * 100 + i)
        return (1.0 + normal_f32(shape, 0.1, seed * 100 + i)).to(torch.bfloat16)

    def a(k):
        nonlocal i
        i += 1
        return normal_f32((k,), 1.0, seed * 100 + i).exp_()

    st["fc.weight"] = w((hidden, target_hidden))
    for l in range(n_layers):
        P = f"layers.{l}"
        st[f"{P}.input_layernorm.weight"] = w((hidden,))
        st[f"{P}.post_attention_layernorm.weight"] = w((hidden,))
        st[f"{P}.attention_conv.kernel_projection.weight"] = w((taps, hidden))
        st[f"{P}.mlp_conv.kernel_projection.weight"] = w((taps, hidden))
        st[f"{P}.self_attn.q_proj.weight"] = w((q_dim, hidden))
        st[f"{P}.self_attn.k_proj.weight"] = w((kv_dim, hidden))
        st[f"{P}.self_attn.v_proj.weight"] = w((kv_dim, hidden))
        st[f"{P}.self_attn.o_proj.weight"] = w((hidden, q_dim))
        st[f"{P}.mlp.gate_proj.weight"] = w((inter, hidden))
        st[f"{P}.mlp.up_proj.weight"] = w((inter, hidden))
        st[f"{P}.mlp.down_proj.weight"] = w((hidden, inter))
        act[f"{P}.self_attn.qkv_proj"] = a(hidden)
        act[f"{P}.mlp.gate_up_proj"] = a(hidden)
        act[f"{P}.mlp.down_proj"] = a(inter)
    return st, act, {"num_hidden_layers": n_layers, "hidden_size": hidden}
