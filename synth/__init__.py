"""Seeded synthetic inputs shared by the oracle and the CUDA library.

This module only draws numbers: model shapes, random-init weights, prompt
token ids and forced exit schedules.  It holds none of the method's
arithmetic (no normalisation, attention, quantisation or exit rule), so both
sides of every parity test can take their inputs from here without sharing
any computation.

Recipe (one fixed order, so a seed names one model):

* weights: ``N(0, 0.02)`` per tensor, drawn in the order embed, then for each
  layer wq, wk, wv, wo, wg, wu, wd, then lm_head; rounded to bf16.  Both sides
  receive the bf16 values (the oracle computes on ``float32(bf16)``).
  The tiny shape is drawn on the CPU generator; the Llama-1B/8B shapes are
  drawn with the CUDA generator when a GPU is present (the CPU generator
  manages only ~30 M normals/s) and on the CPU otherwise.
* RMSNorm gains: 1.0 (``gains="ones"``) or ``1 + N(0, 0.1)`` (``gains="random"``,
  used by parity tests so that a dropped gain cannot go unnoticed).
* prompt ids: uniform over ``[0, vocab)`` from ``numpy.random.default_rng(1)``.
* forced exit schedules: ``numpy.random.default_rng(2)``; each step is the full
  depth ``L`` with probability ``full_share`` (0.05), otherwise
  ``min(G, L-1)`` with ``G ~ Geometric(p)`` on {1, 2, ...}; ``p`` is solved so
  that the mean exit layer equals the target (3.8 of 16 for the 1B shape,
  8 of 32 for the 8B shape).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LINEARS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 1e4
    group_size: int = 128

    def linear_shapes(self):
        """(out, in) of each decoder-layer linear, in draw order."""
        d, hq, hkv, hd, f = self.d_model, self.n_q_heads, self.n_kv_heads, self.head_dim, self.ffn_dim
        return {
            "wq": (hq * hd, d), "wk": (hkv * hd, d), "wv": (hkv * hd, d),
            "wo": (d, hq * hd), "wg": (f, d), "wu": (f, d), "wd": (d, f),
        }


# Shapes of the workloads.  rope_theta 5e5 for the Llama-3 shapes is the
# family default (no rope scaling: random weights make scaling moot).
TINY = Shape("tiny", 4, 256, 4, 2, 64, 688, 1024, 1e-5, 1e4)
LLAMA_1B = Shape("llama-3.2-1b", 16, 2048, 32, 8, 64, 8192, 128256, 1e-5, 5e5)
LLAMA_8B = Shape("llama-3.1-8b", 32, 4096, 32, 8, 128, 14336, 128256, 1e-5, 5e5)
SHAPES = {s.name: s for s in (TINY, LLAMA_1B, LLAMA_8B)}


def scaled(shape: Shape, **kw) -> Shape:
    """A copy of ``shape`` with some fields replaced (small test variants)."""
    return dataclasses.replace(shape, **kw)


def _torch():
    import torch
    return torch


def gen_weights(shape: Shape, seed: int = 0, device: str | None = None, gains: str = "ones"):
    """Draw the model's weights; returns a dict of bf16 torch tensors.

    Keys: ``embed [V][d]``, ``lm_head [V][d]``, ``g_final [d]`` and
    ``layers``: a list of dicts with ``wq wk wv wo wg wu wd g_attn g_ffn``.
    Linear weights are row-major ``[out][in]``.
    """
    torch = _torch()
    if device is None:
        device = "cuda" if (shape.name != "tiny" and torch.cuda.is_available()) else "cpu"
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def normal(rows, cols, std=0.02):
        t = torch.empty((rows, cols), dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=g)
        return t.to(torch.bfloat16)

    d, V = shape.d_model, shape.vocab
    out = {"embed": normal(V, d)}
    layers = []
    for _ in range(shape.n_layers):
        lw = {}
        for name, (o, i) in shape.linear_shapes().items():
            lw[name] = normal(o, i)
        layers.append(lw)
    out["lm_head"] = normal(V, d)
    # Gains are drawn after everything else so that the linear weights do not
    # depend on the gain mode.
    for lw in layers:
        lw["g_attn"] = _gain(shape, gains, g, device)
        lw["g_ffn"] = _gain(shape, gains, g, device)
    out["g_final"] = _gain(shape, gains, g, device)
    out["layers"] = layers
    return out


def _gain(shape, mode, g, device):
    torch = _torch()
    if mode == "ones":
        return torch.ones(shape.d_model, dtype=torch.bfloat16, device=device)
    if mode == "random":
        t = torch.empty(shape.d_model, dtype=torch.float32, device=device)
        t.normal_(1.0, 0.1, generator=g)
        return t.to(torch.bfloat16)
    raise ValueError(mode)


def weights_to_numpy(w):
    """float32 numpy copies of a weight dict (exact: bf16 -> fp32 is exact)."""
    torch = _torch()

    def cv(t):
        return t.detach().to("cpu", torch.float32).numpy()

    return {
        "embed": cv(w["embed"]), "lm_head": cv(w["lm_head"]), "g_final": cv(w["g_final"]),
        "layers": [{k: cv(v) for k, v in lw.items()} for lw in w["layers"]],
    }


def gen_tokens(vocab: int, shape, seed: int = 1) -> np.ndarray:
    """Uniform token ids in [0, vocab) as int32, of the given shape."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=shape, dtype=np.int64).astype(np.int32)


def schedule_mean(n_layers: int, p: float, full_share: float) -> float:
    """Mean of the schedule distribution: full_share*L + (1-full_share)*E[min(G, L-1)]."""
    n = n_layers - 1
    e_min = (1.0 - (1.0 - p) ** n) / p  # sum_{k=0}^{n-1} P(G > k)
    return full_share * n_layers + (1.0 - full_share) * e_min


def solve_geometric_p(n_layers: int, target_mean: float, full_share: float = 0.05) -> float:
    """Bisection for p such that schedule_mean(L, p) == target_mean."""
    lo, hi = 1e-9, 1.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if schedule_mean(n_layers, mid, full_share) > target_mean:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def gen_schedule(n_layers: int, n_steps: int, target_mean: float, full_share: float = 0.05,
                 seed: int = 2) -> np.ndarray:
    """Forced per-step exit layers (int32 in [1, L]); see the module docstring."""
    p = solve_geometric_p(n_layers, target_mean, full_share)
    rng = np.random.default_rng(seed)
    full = rng.random(n_steps) < full_share
    geo = rng.geometric(p, size=n_steps)
    e = np.minimum(geo, n_layers - 1)
    e = np.where(full, n_layers, e)
    return e.astype(np.int32)


def random_kv_fill(n: int, seed: int = 3, device="cpu"):
    """N(0, 1) bf16 values used to fill a KV cache for timing-only runs."""
    torch = _torch()
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.empty(n, dtype=torch.float32, device=device)
    t.normal_(0.0, 1.0, generator=g)
    return t.to(torch.bfloat16)


__all__ = [
    "Shape", "TINY", "LLAMA_1B", "LLAMA_8B", "SHAPES", "LINEARS", "scaled",
    "gen_weights", "weights_to_numpy", "gen_tokens", "gen_schedule",
    "solve_geometric_p", "schedule_mean", "random_kv_fill",
]
