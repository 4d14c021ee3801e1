"""Seeded synthetic workloads for the K-FAC preconditioning step.

This module only draws random inputs and shapes them like the workloads of
"Accelerating Distributed K-FAC with Smart Parallelism of Computing and
Communication Tasks" (§V: ResNet-style CNNs) and of BERT-large linear layers.
It holds none of the K-FAC arithmetic (no factor, average, damping, inverse or
preconditioning): the oracle and the CUDA path each implement that on their own
and both receive the arrays produced here.

Readings used for the draws (the pages give no values for them):
  * ``N(0, s)`` means a normal with standard deviation ``s``.
  * A bias column of ones is appended to every layer input ``a``.
  * bf16 inputs are rounded once on the host, round-to-nearest-even.
  * The weight gradient of a layer is ``grad = g^T a / B`` (the mean over the
    B samples), computed in float64 from the rounded ``a``, ``g`` and rounded
    once to float32; it is an input of the step, not part of it.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np

__all__ = [
    "Layer", "Config", "CONFIGS", "config", "rng_for",
    "to_bf16_bits", "bf16_bits_to_f32", "round_bf16",
    "layer_inputs", "padded_ld", "conv_shape", "conv_activations", "device_conv_activations",
]


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    d_in: int          # dimension of factor A (layer input width incl. bias column)
    d_out: int         # dimension of factor G (layer output width)
    kind: str = "linear"   # "linear" | "conv3x3"
    hw: int = 1        # spatial positions per sample (conv layers)


@dataclasses.dataclass(frozen=True)
class Config:
    key: str
    title: str
    layers: tuple
    batch: int               # samples B per step
    P: int                   # emulated data-parallel workers (equal row shards)
    steps: int               # K-FAC steps (running average length)
    gamma: float             # Tikhonov damping
    decay: Optional[float]   # running-average weight on the previous value
    in_dtype: str            # "fp32" | "bf16" (dtype of a and g)
    a_dist: str              # "normal" | "relu_normal" | "mlp"
    a_sigma: float
    g_sigma: float

    def rows(self, layer: Layer) -> int:
        return self.batch * layer.hw


def _bert_layers(prefix: str = ""):
    return (
        Layer(prefix + "qkv", 1025, 3072),
        Layer(prefix + "attn_out", 1025, 1024),
        Layer(prefix + "ffn_in", 1025, 4096),
        Layer(prefix + "ffn_out", 4097, 1024),
    )


CONFIGS = {
    "single_linear": Config(
        key="single_linear",
        title="single linear layer 64(+1)->32, B=128, fp32 inputs",
        layers=(Layer("fc", 65, 32),),
        batch=128, P=1, steps=1, gamma=0.03, decay=None, in_dtype="fp32",
        a_dist="normal", a_sigma=1.0, g_sigma=0.01),
    "mlp": Config(
        key="mlp",
        title="3-layer MLP 784-1024-1024-10, B=256 in 4 shards, 10 steps",
        layers=(Layer("fc1", 785, 1024), Layer("fc2", 1025, 1024), Layer("fc3", 1025, 10)),
        batch=256, P=4, steps=10, gamma=1e-3, decay=0.95, in_dtype="bf16",
        a_dist="mlp", a_sigma=1.0, g_sigma=1e-3),
    "resnet_conv": Config(
        key="resnet_conv",
        title="ResNet-50 3x3 convs C=64/128/256/512 at 56/28/14/7, B=32 in 8 shards",
        layers=(Layer("conv3x3_c64", 577, 64, "conv3x3", 56 * 56),
                Layer("conv3x3_c128", 1153, 128, "conv3x3", 28 * 28),
                Layer("conv3x3_c256", 2305, 256, "conv3x3", 14 * 14),
                Layer("conv3x3_c512", 4609, 512, "conv3x3", 7 * 7)),
        batch=32, P=8, steps=1, gamma=1e-3, decay=None, in_dtype="bf16",
        a_dist="relu_normal", a_sigma=1.0, g_sigma=1e-3),
    "bert_layer": Config(
        key="bert_layer",
        title="one BERT-large encoder layer (QKV, attn-out, FFN-in, FFN-out), 4096 rows in 4 shards",
        layers=_bert_layers(),
        batch=4096, P=4, steps=20, gamma=1e-3, decay=0.95, in_dtype="bf16",
        a_dist="normal", a_sigma=1.0, g_sigma=1e-4),
    "bert_large": Config(
        key="bert_large",
        title="24-layer BERT-large stack (96 linears, 192 factors), 4096 rows in 8 shards",
        layers=tuple(l for i in range(24) for l in _bert_layers(f"l{i:02d}.")),
        batch=4096, P=8, steps=20, gamma=1e-3, decay=0.95, in_dtype="bf16",
        a_dist="normal", a_sigma=1.0, g_sigma=1e-4),
}


def config(key: str) -> Config:
    return CONFIGS[key]


def padded_ld(d: int, elem_bytes: int) -> int:
    """Leading dimension padded to a 16-byte multiple (TMA stride rule)."""
    per = 16 // elem_bytes
    return (d + per - 1) // per * per


def rng_for(*keys) -> np.random.Generator:
    """Independent PCG64 stream per (config, step, layer, tensor) key tuple."""
    h = hashlib.sha256(repr(keys).encode()).digest()
    words = [int.from_bytes(h[i:i + 4], "little") for i in range(0, 16, 4)]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(to_bf16_bits(x))


def _draw(rng, shape, dist, sigma):
    z = rng.standard_normal(shape, dtype=np.float64) * sigma
    if dist == "relu_normal":
        z = np.maximum(z, 0.0)
    return z


def _mlp_weights(cfg: Config):
    """He-initialised weights N(0, 2/fan_in) with zero bias, fixed across steps."""
    ws = []
    for li, layer in enumerate(cfg.layers[:-1]):
        fan_in = layer.d_in - 1
        rng = rng_for(cfg.key, "weights", li)
        ws.append(rng.standard_normal((layer.d_out, fan_in)) * np.sqrt(2.0 / fan_in))
    return ws


def _round(cfg: Config, x: np.ndarray) -> np.ndarray:
    x32 = x.astype(np.float32)
    return round_bf16(x32) if cfg.in_dtype == "bf16" else x32


def conv_shape(cfg: Config, layer: Layer):
    """(B, H, W, C) of the NHWC input of a 3 x 3 conv layer: C = (d_in - 1) / 9
    channels, square H = W images of `hw` positions, B = cfg.batch images."""
    assert layer.kind == "conv3x3" and (layer.d_in - 1) % 9 == 0
    side = int(round(layer.hw ** 0.5))
    assert side * side == layer.hw
    return cfg.batch, side, side, (layer.d_in - 1) // 9


def conv_activations(shape, seed_keys, dist: str = "relu_normal", sigma: float = 1.0) -> np.ndarray:
    """NHWC activations x[b, h, w, c] of `shape`, drawn from `dist` (ReLU of
    N(0, sigma) for the conv workloads) and rounded to bf16; float32."""
    return round_bf16(_draw(rng_for("conv", *seed_keys), tuple(shape), dist, sigma).astype(np.float32))


def device_conv_activations(shape, seed_keys, dist: str = "relu_normal", sigma: float = 1.0, device="cuda"):
    """The same distribution as ``conv_activations``, drawn on the device from a
    seeded torch generator (bf16 tensor, NHWC contiguous)."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(torch_seed("conv", *seed_keys))
    z = torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32) * sigma
    if dist == "relu_normal":
        z.clamp_(min=0.0)
    return z.to(torch.bfloat16)


def torch_seed(*keys) -> int:
    h = hashlib.sha256(repr(("torch",) + keys).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def device_layer_inputs(cfg: Config, step: int, layer_index: int, device="cuda"):
    """Same shapes and distributions as ``layer_inputs``, drawn on the device
    from seeded torch generators (for sizes where host generation is slow).
    Supports the "normal" and "relu_normal" workloads.  The weight gradient
    is g^T a / B in float32 (an input of the step, made outside it)."""
    import torch

    if cfg.a_dist == "mlp":
        raise ValueError("the MLP workload is generated on the host (layer_inputs)")
    layer = cfg.layers[layer_index]
    rows = cfg.rows(layer)
    dt = torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32
    gen = torch.Generator(device=device)
    gen.manual_seed(torch_seed(cfg.key, step, layer_index, "a"))
    body = torch.randn((rows, layer.d_in - 1), generator=gen, device=device, dtype=torch.float32) * cfg.a_sigma
    if cfg.a_dist == "relu_normal":
        body.clamp_(min=0.0)
    a = torch.empty((rows, layer.d_in), dtype=dt, device=device)
    a[:, :-1] = body.to(dt)
    a[:, -1] = 1.0
    del body
    gen.manual_seed(torch_seed(cfg.key, step, layer_index, "g"))
    g = (torch.randn((rows, layer.d_out), generator=gen, device=device, dtype=torch.float32) * cfg.g_sigma).to(dt)
    grad = (g.float().t() @ a.float()) / cfg.batch
    return {"a": a, "g": g, "grad": grad}


def layer_inputs(cfg: Config, step: int, layer_index: int, with_grad: bool = True):
    """Inputs of one layer at one step, as float32 arrays holding the exact
    values given to the GPU (bf16-representable when ``cfg.in_dtype`` is bf16).

    Returns a dict with
      ``a``    (rows, d_in): layer input with the ones column last,
      ``g``    (rows, d_out): gradient w.r.t. the layer output,
      ``grad`` (d_out, d_in) float32: weight gradient g^T a / B (if with_grad).
    """
    layer = cfg.layers[layer_index]
    rows = cfg.rows(layer)
    if cfg.a_dist == "mlp":
        rng = rng_for(cfg.key, step, "x")
        h = rng.standard_normal((cfg.batch, cfg.layers[0].d_in - 1))
        ws = _mlp_weights(cfg)
        for li in range(layer_index):
            h = np.maximum(_round(cfg, h).astype(np.float64) @ ws[li].T, 0.0)
        body = h
    else:
        body = _draw(rng_for(cfg.key, step, layer_index, "a"),
                     (rows, layer.d_in - 1), cfg.a_dist, cfg.a_sigma)
    a = np.empty((rows, layer.d_in), dtype=np.float32)
    a[:, :-1] = _round(cfg, body)
    a[:, -1] = 1.0
    g = _round(cfg, _draw(rng_for(cfg.key, step, layer_index, "g"),
                          (rows, layer.d_out), "normal", cfg.g_sigma))
    out = {"a": a, "g": g}
    if with_grad:
        grad = (g.astype(np.float64).T @ a.astype(np.float64)) / cfg.batch
        out["grad"] = grad.astype(np.float32)
    return out
