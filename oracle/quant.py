"""W4A16 exit-layer quantizer of the oracle (test infrastructure only).

River-LLM explainer, section 三: each exit layer is a copy of the backbone
layer's parameters, shrunk with 4-bit weight / 16-bit activation (W4A16)
quantization, training-free; section 六 names HQQ as the quantizer and AWQ
as a drop-in.  The format (asymmetric, groups of 128 consecutive inputs,
fp16 scale and zero, eight nibbles per uint32) is the library's contract.

Reading taken where the page is silent: plain min-max round-to-nearest
(HQQ's starting point, without its half-quadratic refinement), float zero
point stored in fp16, round half to even, clamp to [0, 15]; a degenerate
group (max == min, or a scale that rounds to 0 in fp16) gets scale 1.0; a
ragged last group (K not a multiple of 128) covers the remaining inputs.

Every step is IEEE fp32 with a single rounding, then fp16 rounding where the
value is stored:
    s = fp16( (mx - mn) / 15 )
    z = fp16( -mn / s )
    q = clamp( rint( (w / s) + z ), 0, 15 )      (division and add separately)
    qweight[n][k // 8] |= q << (4 * (k % 8))
    w_hat = (q - z) * s
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def _group_bounds(K: int, group: int):
    return [(g0, min(g0 + group, K)) for g0 in range(0, K, group)]


def quantize_linear(w: np.ndarray, group: int = 128):
    """Quantize ``w [N][K]`` (float32 holding bf16 values).

    Returns ``(qweight uint32 [N][K/8], scales fp16 [N][G], zeros fp16 [N][G])``
    with ``G = ceil(K / group)``.
    """
    w = np.asarray(w, dtype=F32)
    N, K = w.shape
    if K % 8:
        raise ValueError("K must be a multiple of 8 (eight nibbles per uint32)")
    bounds = _group_bounds(K, group)
    G = len(bounds)
    scales = np.empty((N, G), dtype=np.float16)
    zeros = np.empty((N, G), dtype=np.float16)
    q = np.empty((N, K), dtype=np.uint32)
    for j, (k0, k1) in enumerate(bounds):
        blk = w[:, k0:k1]
        mn = blk.min(axis=1)
        mx = blk.max(axis=1)
        rng = (mx - mn).astype(F32)                       # fp32 subtract
        s16 = (rng / F32(15.0)).astype(F32).astype(np.float16)
        degenerate = (mx == mn) | (s16 == np.float16(0.0))
        s16 = np.where(degenerate, np.float16(1.0), s16)
        s32 = s16.astype(F32)
        z16 = ((-mn).astype(F32) / s32).astype(F32).astype(np.float16)
        z32 = z16.astype(F32)
        v = (blk / s32[:, None]).astype(F32)              # fp32 divide
        v = (v + z32[:, None]).astype(F32)                # separate fp32 add
        qq = np.clip(np.rint(v), F32(0.0), F32(15.0))
        q[:, k0:k1] = qq.astype(np.uint32)
        scales[:, j] = s16
        zeros[:, j] = z16
    qw = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        qw |= q[:, i::8] << np.uint32(4 * i)
    return qw, scales, zeros


def unpack_nibbles(qweight: np.ndarray, K: int) -> np.ndarray:
    """Inverse of the packing: ``q [N][K]`` uint8 with q[n][k] at bits 4*(k%8)."""
    qweight = np.asarray(qweight, dtype=np.uint32)
    N = qweight.shape[0]
    shifts = (np.arange(8, dtype=np.uint32) * np.uint32(4))[None, None, :]
    q = (qweight[:, :, None] >> shifts) & np.uint32(0xF)          # [N][K/8][8]
    return q.reshape(N, K).astype(np.uint8)


def dequantize_linear(qweight, scales, zeros, K: int, group: int = 128) -> np.ndarray:
    """``w_hat[n][k] = (q - z) * s`` in fp32, group of k = k // group."""
    q = unpack_nibbles(qweight, K).astype(F32)
    N = q.shape[0]
    s = np.asarray(scales).astype(F32)
    z = np.asarray(zeros).astype(F32)
    G = s.shape[1]
    qg = np.zeros((N, G * group), F32)
    qg[:, :K] = q
    qg = qg.reshape(N, G, group)
    w = ((qg - z[:, :, None]).astype(F32) * s[:, :, None]).astype(F32)
    return w.reshape(N, G * group)[:, :K].copy()
