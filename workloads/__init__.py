"""Seeded synthetic inputs for the routed-expert MoE layer.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no routing, no SwiGLU, no combine).  Both the CUDA path and
the CPU oracle are fed from here, and neither imports the other.

Workloads (geometry from AFN-019 "Hide SSD misses before the router knows they
exist", section "Why overlap alone cannot defeat the byte roofline": 512 routed
experts, top-10, hidden 2,560, routed intermediate 640):

  tiny      T=16, H=256,  E=64,  k=4,  I=64;  no router bias; seed 0
  decode    T=16, H=2560, E=512, k=10, I=640; Zipf(s=1) router bias; seed 1
  prefill   T=4096, same geometry; uniform router (no bias); seed 2
  stack48   48 layers x 32 blocks of T=16, int4 g64 expert weights; seed 3
  sweep     route predictor 2560->512 per layer over the stack48 routes; seed 4

x ~ N(0,1) and every weight ~ N(0, 0.02), all rounded to bf16.  Random
sub-streams are drawn from independent generators in a fixed order:
x, router, bias permutation, gate/up, down, predictor.

The int4 codes of ``stack48`` are made here once, at generation time: signed
symmetric int4 in [-8, 7] with one bf16 scale per 64 consecutive input
elements of a weight row (scale = bf16(max|w|/7)); the codes and scales *are*
the input data that both sides dequantise.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

STD_W = 0.02

# sub-stream indices (fixed draw order)
_S_X, _S_ROUTER, _S_BIAS, _S_GATEUP, _S_DOWN, _S_PRED = range(6)


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    bias: Optional[str]  # None or "zipf"
    seed: int
    zipf_s: float = 1.0

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def params_per_expert(self) -> int:
        # gate [I,H] + up [I,H] + down [H,I]
        return 3 * self.H * self.I


TINY = LayerConfig("tiny", T=16, H=256, E=64, k=4, I=64, bias=None, seed=0)
DECODE = LayerConfig("decode", T=16, H=2560, E=512, k=10, I=640, bias="zipf", seed=1)
PREFILL = LayerConfig("prefill", T=4096, H=2560, E=512, k=10, I=640, bias=None, seed=2)
STACK48 = LayerConfig("stack48", T=16, H=2560, E=512, k=10, I=640, bias=None, seed=3)
SWEEP_SEED = 4
STACK_LAYERS = 48
STACK_BLOCKS = 32
SWEEP_BLOCKS = (1, 4, 16, 64)

CONFIGS = {c.name: c for c in (TINY, DECODE, PREFILL, STACK48)}


def with_tokens(cfg: LayerConfig, T: int) -> LayerConfig:
    return replace(cfg, T=T)


def _gen(device, seed: int, stream: int, layer: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + layer * 101 + stream)
    return g


def _normal_bf16(shape, std, g, device, chunk_rows: int = 0) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 then rounded to bf16; chunked along dim 0."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    step = chunk_rows if chunk_rows > 0 else n0
    for a in range(0, n0, step):
        b = min(n0, a + step)
        tmp = torch.randn((b - a,) + tuple(shape[1:]), generator=g, device=device,
                          dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        out[a:b].copy_(tmp)
        del tmp
    return out


def zipf_bias(E: int, seed: int, s: float = 1.0, layer: int = 0) -> torch.Tensor:
    """Router bias carrying a Zipf(s) popularity prior over experts.

    b[e] = -s * ln(rank(e)), rank = 1 + pi(e), pi a seeded permutation of the
    experts: the log of an unnormalised Zipf prior.  Drawn on the CPU so that
    it is identical on every machine.
    """
    g = _gen("cpu", seed, _S_BIAS, layer)
    pi = torch.randperm(E, generator=g)
    rank = (pi + 1).to(torch.float64)
    return (-s * torch.log(rank)).to(torch.float32)


def layer_inputs(cfg: LayerConfig, device="cpu", layer: int = 0, x_seed_offset: int = 0,
                 with_x: bool = True) -> dict:
    """All tensors of one MoE layer for ``cfg``.

    Returns x [T,H] bf16, w_router [E,H] bf16, bias [E] f32 or None,
    w_gateup [E, 2I, H] bf16 (gate rows 0..I-1 then up rows I..2I-1 of each
    expert, one contiguous record per expert), w_down [E, H, I] bf16.
    """
    dev = torch.device(device)
    out = {}
    if with_x:
        gx = _gen(dev, cfg.seed + x_seed_offset * 7919, _S_X, layer)
        out["x"] = _normal_bf16((cfg.T, cfg.H), 1.0, gx, dev)
    out["w_router"] = _normal_bf16((cfg.E, cfg.H), STD_W, _gen(dev, cfg.seed, _S_ROUTER, layer), dev)
    if cfg.bias == "zipf":
        out["bias"] = zipf_bias(cfg.E, cfg.seed, cfg.zipf_s, layer).to(dev)
    else:
        out["bias"] = None
    per_chunk = max(1, (1 << 26) // (2 * cfg.I * cfg.H))
    out["w_gateup"] = _normal_bf16((cfg.E, 2 * cfg.I, cfg.H), STD_W,
                                   _gen(dev, cfg.seed, _S_GATEUP, layer), dev, per_chunk)
    out["w_down"] = _normal_bf16((cfg.E, cfg.H, cfg.I), STD_W,
                                 _gen(dev, cfg.seed, _S_DOWN, layer), dev, per_chunk)
    return out


def router_inputs(cfg: LayerConfig, device="cpu", layer: int = 0):
    """(w_router, bias) of layer_inputs(cfg, device, layer) without the experts."""
    dev = torch.device(device)
    wr = _normal_bf16((cfg.E, cfg.H), STD_W, _gen(dev, cfg.seed, _S_ROUTER, layer), dev)
    bias = zipf_bias(cfg.E, cfg.seed, cfg.zipf_s, layer).to(dev) if cfg.bias == "zipf" else None
    return wr, bias


SIDECAR_SEED = 5


def sidecar_weights(F: int, r: int, E: int, L: int, device="cpu", seed: int = SIDECAR_SEED) -> dict:
    """Random route-sidecar weights (bf16): trunk [r,F] ~ N(0, 1/F), layer
    embeddings [L,r] ~ N(0, 1), expert heads [E,r] ~ N(0, 1/r); the trunk
    output and the layer embeddings are then of one scale, so the layer
    changes the ranking."""
    dev = torch.device(device)
    return {"w_trunk": _normal_bf16((r, F), F ** -0.5, _gen(dev, seed, _S_PRED, 1), dev),
            "layer_emb": _normal_bf16((L, r), 1.0, _gen(dev, seed, _S_PRED, 2), dev),
            "w_head": _normal_bf16((E, r), r ** -0.5, _gen(dev, seed, _S_PRED, 3), dev)}


def token_batch(cfg: LayerConfig, device="cpu", index: int = 0, T: Optional[int] = None) -> torch.Tensor:
    """An independent x ~ N(0,1) bf16 batch [T,H] (index selects the draw)."""
    dev = torch.device(device)
    g = _gen(dev, cfg.seed + 7919 * (index + 1), _S_X, 0)
    return _normal_bf16((T or cfg.T, cfg.H), 1.0, g, dev)


def predictor_weights(H: int, E: int, layer: int, device="cpu") -> torch.Tensor:
    """Pre-attention linear route predictor weights [E,H] ~ N(0,0.02) bf16."""
    dev = torch.device(device)
    return _normal_bf16((E, H), STD_W, _gen(dev, SWEEP_SEED, _S_PRED, layer), dev)


# ---------------------------------------------------------------------------
# int4 g64 codes: the stored form of the stack48 expert weights.
# ---------------------------------------------------------------------------
INT4_GROUP = 64


def quantize_int4_g64(w: torch.Tensor):
    """Quantise rows of w [..., K] (bf16/f32) to signed int4 codes, group 64.

    Returns (packed uint8 [..., K/2] with the even-k code in the low nibble,
    scales bf16 [..., K/64]).  q = clamp(round_half_even(w/s), -8, 7),
    s = bf16(max|w_group| / 7) (s = 1 for an all-zero group).
    """
    K = w.shape[-1]
    assert K % INT4_GROUP == 0
    wf = w.to(torch.float32).reshape(*w.shape[:-1], K // INT4_GROUP, INT4_GROUP)
    amax = wf.abs().amax(dim=-1, keepdim=True)
    s = (amax / 7.0).to(torch.bfloat16)
    s = torch.where(s == 0, torch.ones_like(s), s)
    q = torch.round(wf / s.to(torch.float32)).clamp_(-8, 7).to(torch.int8)
    q = q.reshape(*w.shape[:-1], K)
    lo = (q[..., 0::2].to(torch.int16) & 0xF)
    hi = (q[..., 1::2].to(torch.int16) & 0xF)
    packed = (lo | (hi << 4)).to(torch.uint8)
    return packed, s.squeeze(-1)


def stack_layer_weights(layer: int, device="cpu", cfg: LayerConfig = STACK48) -> dict:
    """One layer of the 48-layer int4 stack: bf16 router, int4 g64 experts."""
    dev = torch.device(device)
    wr = _normal_bf16((cfg.E, cfg.H), STD_W, _gen(dev, cfg.seed, _S_ROUTER, layer), dev)
    per_chunk = max(1, (1 << 26) // (2 * cfg.I * cfg.H))
    gu_q, gu_s, d_q, d_s = [], [], [], []
    ggu = _gen(dev, cfg.seed, _S_GATEUP, layer)
    gd = _gen(dev, cfg.seed, _S_DOWN, layer)
    for a in range(0, cfg.E, per_chunk):
        b = min(cfg.E, a + per_chunk)
        wgu = _normal_bf16((b - a, 2 * cfg.I, cfg.H), STD_W, ggu, dev)
        q, s = quantize_int4_g64(wgu)
        gu_q.append(q); gu_s.append(s)
        wd = _normal_bf16((b - a, cfg.H, cfg.I), STD_W, gd, dev)
        q, s = quantize_int4_g64(wd)
        d_q.append(q); d_s.append(s)
    return {
        "w_router": wr,
        "w_gateup_q": torch.cat(gu_q), "s_gateup": torch.cat(gu_s),
        "w_down_q": torch.cat(d_q), "s_down": torch.cat(d_s),
    }


__all__ = [
    "LayerConfig", "TINY", "DECODE", "PREFILL", "STACK48", "CONFIGS", "STD_W", "router_inputs", "sidecar_weights",
    "STACK_LAYERS", "STACK_BLOCKS", "SWEEP_BLOCKS", "SWEEP_SEED", "with_tokens",
    "layer_inputs", "token_batch", "zipf_bias", "predictor_weights",
    "quantize_int4_g64", "stack_layer_weights", "INT4_GROUP"
]
