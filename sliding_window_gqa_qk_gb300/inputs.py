"""Seeded synthetic inputs for the attention block (shared by the tests, the
benchmark and the oracle checks).

This module holds no arithmetic of the method: it only draws random tensors
with a fixed seed recipe and rounds them to the dtypes the library consumes,
so that the CUDA path and the float64 oracle see identical bits.

Recipe:
  * base seed 42 (the training script's fixed seed, autoresearch Administrator
    & Developer Guide §3.4), plus ``100 * layer``; one ``torch.Generator`` per
    tensor, seeded base + i in the order q, k, v, gq, gk, dO, VE, tok.
  * q, k, v, dO ~ N(0, 1), rounded to bf16 (or kept fp32 for the fp32 build).
  * gains gq, gk ~ 1 + gain_std * N(0, 1) in fp32 (None when gain_std is None).
  * VE table [vocab, Hkv*d] ~ N(0, 0.02^2) in bf16; token ids ~ U[0, vocab) int32.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch

BASE_SEED = 42
VOCAB = 8192


@dataclasses.dataclass(frozen=True)
class Problem:
    """Shapes and per-layer options of one attention call."""

    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    window: int = -1          # -1: no window (full causal)
    causal: bool = True
    gain_std: Optional[float] = None   # None: unit gains (NULL at the ABI)
    ve: bool = False          # value-embedding mix on this layer
    ve_scale: float = 0.5
    vocab: int = VOCAB
    eps: float = 1e-6

    def replace(self, **kw) -> "Problem":
        return dataclasses.replace(self, **kw)


# The workloads of the benchmark configurations.
TINY = Problem(B=1, T=256, Hq=2, Hkv=1, d=64, window=128)
S_LAYER = Problem(B=16, T=2048, Hq=6, Hkv=3, d=128, window=1024, gain_std=0.1)
L_LAYER = Problem(B=16, T=2048, Hq=6, Hkv=3, d=128, window=-1, gain_std=0.1)
LONG_S = Problem(B=2, T=16384, Hq=16, Hkv=4, d=128, window=8192, gain_std=0.1)
LONG_L = Problem(B=2, T=16384, Hq=16, Hkv=4, d=128, window=-1, gain_std=0.1)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_inputs(p: Problem, layer: int = 0, dtype: torch.dtype = torch.bfloat16,
                seed: int = BASE_SEED, device="cpu") -> dict:
    """Draw the inputs of one layer.

    Returns a dict with q, k, v, dO (``dtype``), gq, gk (fp32 [d] or None),
    ve ([vocab, Hkv*d] in ``dtype`` or None) and tok (int32 [B, T] or None).
    With ``device`` a CUDA device the same recipe draws from that device's
    generator (another stream of numbers than the CPU's, same distributions),
    for sizes whose CPU draw would take minutes.
    """
    s = seed + 100 * layer
    B, T, Hq, Hkv, d = p.B, p.T, p.Hq, p.Hkv, p.d
    kw = dict(device=device)
    out = {}
    out["q"] = torch.randn(B, T, Hq, d, generator=_gen(s + 0, device), **kw).to(dtype)
    out["k"] = torch.randn(B, T, Hkv, d, generator=_gen(s + 1, device), **kw).to(dtype)
    out["v"] = torch.randn(B, T, Hkv, d, generator=_gen(s + 2, device), **kw).to(dtype)
    if p.gain_std is None:
        out["gq"] = None
        out["gk"] = None
    else:
        out["gq"] = 1.0 + p.gain_std * torch.randn(d, generator=_gen(s + 3, device), **kw)
        out["gk"] = 1.0 + p.gain_std * torch.randn(d, generator=_gen(s + 4, device), **kw)
    out["dO"] = torch.randn(B, T, Hq, d, generator=_gen(s + 5, device), **kw).to(dtype)
    if p.ve:
        out["ve"] = (0.02 * torch.randn(p.vocab, Hkv * d, generator=_gen(s + 6, device),
                                        **kw)).to(dtype)
        out["tok"] = torch.randint(0, p.vocab, (B, T), generator=_gen(s + 7, device),
                                   dtype=torch.int64, **kw).to(torch.int32)
    else:
        out["ve"] = None
        out["tok"] = None
    return out


def make_block_inputs(p: Problem, C: int, layer: int = 0, dtype: torch.dtype = torch.bfloat16,
                      gate_ch: Optional[int] = None, seed: int = BASE_SEED, device="cpu") -> dict:
    """Draw the inputs of one whole attention block (pre-norm, projections,
    residual around the attention) of model width C.

    Recipe: seeds base + 100 * layer + 10.. in the order x, wq, wk, wv, wo,
    dout, gate_w; x, dout ~ N(0, 1) [B, T, C]; the projection weights in the
    torch.nn.Linear layout, uniform with variance 1 / fan_in (wq, wk, wv:
    [H*d, C], fan_in C; wo: [C, Hq*d], fan_in Hq*d; the pages' initialisation
    zeroes c_proj, which would hide the attention from the output, so wo is
    drawn like the others); gate_w ~ 0.25 N(0, 1) fp32 [Hkv, gate_ch] when
    gate_ch is given. Gains, VE table and token ids come from make_inputs
    (same seeds). All elem tensors are rounded to ``dtype``."""
    s = seed + 100 * layer + 10
    B, T, Hq, Hkv, d = p.B, p.T, p.Hq, p.Hkv, p.d
    kw = dict(device=device)

    def uniform(shape, fan_in, i):
        a = (3.0 / fan_in) ** 0.5
        return ((2.0 * torch.rand(*shape, generator=_gen(s + i, device), **kw) - 1.0) * a).to(dtype)

    base = make_inputs(p, layer=layer, dtype=dtype, seed=seed, device=device)
    out = {k: base[k] for k in ("gq", "gk", "ve", "tok")}
    out["x"] = torch.randn(B, T, C, generator=_gen(s + 0, device), **kw).to(dtype)
    out["wq"] = uniform((Hq * d, C), C, 1)
    out["wk"] = uniform((Hkv * d, C), C, 2)
    out["wv"] = uniform((Hkv * d, C), C, 3)
    out["wo"] = uniform((C, Hq * d), Hq * d, 4)
    out["dout"] = torch.randn(B, T, C, generator=_gen(s + 5, device), **kw).to(dtype)
    out["gate_w"] = (None if gate_ch is None else
                     0.25 * torch.randn(Hkv, gate_ch, generator=_gen(s + 6, device), **kw))
    return out


def as_f64(t):
    """The exact float64 value of a tensor (or None), as a NumPy array."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
