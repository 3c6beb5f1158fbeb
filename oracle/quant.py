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


# ---------------------------------------------------------------------------
# HQQ refinement of the zero point (River-LLM explainer, section 六: HQQ is
# the exit layers' default quantizer; it needs no calibration data).
#
# Half-quadratic quantization (Badri and Shaji, 2023) keeps the min-max scale
# and moves the zero point z of each group to lower an lp norm (p < 1) of the
# reconstruction error w - s (q - z), by splitting that error into an
# auxiliary variable e and alternating two closed-form steps while the
# penalty weight beta grows by kappa per iteration:
#   e <- shrink_p(w - s (q(z) - z), beta)         (proximal step of |.|^p)
#   z <- mean over the group of  q(z) - (w - e) / s   (least-squares step)
# with q(z) = clamp(rint(w / s + z), 0, 15).
#
# Readings taken where the page (and the method) leave a choice open:
#   * the iteration runs per group, in float64, for a fixed number of
#     iterations (20, p = 0.7, beta = 10, kappa = 1.01: the method's usual
#     settings); the zero point kept is the fp16 value, among the min-max one
#     and those of the iterations, whose stored codes give the lowest
#     sum |w - s (q - z)|^p in that group (ties keep the earlier), so the
#     stored result is never worse than min-max rounding by that measure;
#   * the scale and the code rule are min-max's (fp16 s, codes from the fp32
#     divide and add with the stored fp16 zero), so the packed format is
#     unchanged.
# ---------------------------------------------------------------------------

HQQ_ITERS, HQQ_P, HQQ_BETA, HQQ_KAPPA = 20, 0.7, 10.0, 1.01
F64 = np.float64


def hqq_shrink(x: np.ndarray, beta: float, p: float) -> np.ndarray:
    """Generalised soft threshold of |.|^p at weight beta:
    sign(x) max(|x| - |x|^(p-1) / beta, 0), and 0 where x == 0."""
    x = np.asarray(x, F64)
    ax = np.abs(x)
    with np.errstate(divide="ignore"):
        t = np.where(ax > 0, np.power(np.where(ax > 0, ax, 1.0), p - 1.0) / beta, 0.0)
    return np.where(ax > 0, np.sign(x) * np.maximum(ax - t, 0.0), 0.0)


def hqq_zero_step(w, q, e, s, mask) -> np.ndarray:
    """Least-squares zero point: mean over each group's valid entries of
    q - (w - e) / s.  Arrays [..][n]; s [..]; mask marks valid entries."""
    v = np.where(mask, q - (w - e) / s[..., None], 0.0)
    return v.sum(axis=-1) / mask.sum(axis=-1)


def _codes(w32, s32, z16):
    """Stored codes of min-max rounding for a given fp16 zero (fp32 steps)."""
    v = (w32 / s32[..., None]).astype(F32)
    v = (v + z16.astype(F32)[..., None]).astype(F32)
    return np.clip(np.rint(v), F32(0.0), F32(15.0))


def _lp_error(w32, s32, z16, mask, p):
    """sum |w - s (q - z)|^p over each group's valid entries, float64."""
    q = _codes(w32, s32, z16).astype(F64)
    r = w32.astype(F64) - s32.astype(F64)[..., None] * (q - z16.astype(F64)[..., None])
    return np.where(mask, np.power(np.abs(r), p), 0.0).sum(axis=-1)


def _groups(w, group, G):
    """``w [N][K]`` as [N][G][group] (zero padded) and the mask of valid entries."""
    N, K = w.shape
    wg = np.zeros((N, G * group), F32)
    wg[:, :K] = w
    mask = np.zeros(G * group, bool)
    mask[:K] = True
    return wg.reshape(N, G, group), np.broadcast_to(mask.reshape(G, group), (N, G, group))


def hqq_iterates(wg, s16, z16, mask, iters: int = HQQ_ITERS, p: float = HQQ_P,
                 beta: float = HQQ_BETA, kappa: float = HQQ_KAPPA):
    """The fp16 zero points of the refinement's iterations, in order, starting
    from min-max's scale ``s16`` and zero ``z16`` ([N][G]) on groups ``wg``."""
    s64 = s16.astype(F32).astype(F64)
    w64 = wg.astype(F64)
    z = z16.astype(F64)
    b = float(beta)
    out = []
    for _ in range(iters):
        q = np.clip(np.rint(w64 / s64[..., None] + z[..., None]), 0.0, 15.0)
        r = w64 - s64[..., None] * (q - z[..., None])
        e = hqq_shrink(r, b, p)
        z = hqq_zero_step(w64, q, e, s64, mask)
        b *= kappa
        out.append(z.astype(np.float16))
    return out


def quantize_linear_hqq(w: np.ndarray, group: int = 128, iters: int = HQQ_ITERS, p: float = HQQ_P,
                        beta: float = HQQ_BETA, kappa: float = HQQ_KAPPA):
    """Min-max quantization of ``w [N][K]`` followed by the HQQ zero-point
    refinement of every group.  Same return format as ``quantize_linear``."""
    w = np.asarray(w, dtype=F32)
    N, K = w.shape
    _, s16, z16 = quantize_linear(w, group)
    wg, mask = _groups(w, group, s16.shape[1])
    s32 = s16.astype(F32)
    best_z = z16.copy()
    best_err = _lp_error(wg, s32, z16, mask, p)
    for zc in hqq_iterates(wg, s16, z16, mask, iters, p, beta, kappa):
        err = _lp_error(wg, s32, zc, mask, p)
        better = err < best_err
        best_z = np.where(better, zc, best_z)
        best_err = np.where(better, err, best_err)
    # repack with the refined zeros
    q = _codes(wg, s32, best_z).astype(np.uint32).reshape(N, -1)[:, :K]
    qw = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        qw |= q[:, i::8] << np.uint32(4 * i)
    return qw, s16, best_z
