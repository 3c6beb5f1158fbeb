"""Pins of the oracle's W4A16 quantizer against things other than itself.

River-LLM explainer, section 三: exit layers are training-free 4-bit copies
of the backbone layers' parameters.  Format: asymmetric, groups of 128
consecutive inputs, fp16 scale and zero, eight nibbles per uint32.
"""
import json
import os

import numpy as np
import pytest

from oracle.quant import quantize_linear, dequantize_linear, unpack_nibbles

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_example_by_hand():
    ex = json.load(open(os.path.join(GOLDEN, "quant_worked_example.json")))
    w = np.array([ex["w"]], dtype=np.float32)
    qw, s, z = quantize_linear(w, group=ex["group_size"])
    assert int(s.view(np.uint16)[0, 0]) == ex["scale_fp16_bits"]
    assert float(z[0, 0]) == ex["zero"]
    assert unpack_nibbles(qw, 8)[0].tolist() == ex["q"]
    assert int(qw[0, 0]) == ex["qweight"]
    wh = dequantize_linear(qw, s, z, 8, group=ex["group_size"])
    expect = (np.array(ex["q"], np.float32) - np.float32(ex["zero"])) * np.float32(s[0, 0])
    assert np.array_equal(wh[0], expect)


def test_packing_closed_form():
    # q[k] = k mod 16 on a row: the word for k = 8j..8j+7 has nibble i = (8j+i) % 16.
    K = 256
    q = (np.arange(K) % 16).astype(np.uint8)
    # Grid-aligned weights that reproduce exactly these q (see below): s=1, z=0
    # needs a group holding both 0 and 15, which every 16-run does.
    w = q.astype(np.float32)[None, :]
    qw, s, z = quantize_linear(w, group=128)
    assert np.all(s == 1.0) and np.all(z == 0.0)
    assert qw[0, 0] == 0x76543210 and qw[0, 1] == 0xFEDCBA98
    assert np.array_equal(unpack_nibbles(qw, K)[0], q)


@pytest.mark.parametrize("j", [2, 5, 9])
def test_grid_aligned_round_trip_is_exact(j):
    """Weights on a power-of-two grid with an integer zero, each group holding
    nibbles 0 and 15, quantize and dequantize back to themselves."""
    rng = np.random.default_rng(7 + j)
    N, K, G = 6, 384, 128
    s = np.float32(2.0 ** -j)
    zint = rng.integers(0, 16, size=(N, K // G))
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::G] = 0
    q[:, 1::G] = 15
    zfull = np.repeat(zint, G, axis=1)
    w = ((q - zfull).astype(np.float32) * s).astype(np.float32)
    qw, sc, zz = quantize_linear(w, group=G)
    assert np.all(sc.astype(np.float32) == s)
    assert np.array_equal(zz.astype(np.float32), zint.astype(np.float32))
    assert np.array_equal(unpack_nibbles(qw, K), q.astype(np.uint8))
    assert np.array_equal(dequantize_linear(qw, sc, zz, K, G), w)


def _random_bf16(rng, N, K, std=0.02):
    import torch
    w = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32) * std)
    return w.to(torch.bfloat16).float().numpy()


def test_error_bound_and_grid_membership():
    rng = np.random.default_rng(0)
    N, K, G = 64, 1024, 128
    w = _random_bf16(rng, N, K)
    qw, s, z = quantize_linear(w, G)
    wh = dequantize_linear(qw, s, z, K, G)
    sf = np.repeat(s.astype(np.float32), G, axis=1)
    zf = np.repeat(z.astype(np.float32), G, axis=1)
    # |w - w_hat| <= s/2 plus the rounding slack of the fp16 scale/zero.
    assert np.all(np.abs(w - wh) <= sf * 0.5 * (1 + 1e-2) + 1e-7)
    # w_hat / s + z is an integer code in [0, 15].
    codes = wh / sf + zf
    assert np.allclose(codes, np.round(codes), atol=1e-3)
    assert codes.min() > -1e-3 and codes.max() < 15 + 1e-3


def test_nearest_grid_point_brute_force():
    """Each code is the grid point nearest to w (brute force over all 16)."""
    rng = np.random.default_rng(1)
    N, K, G = 8, 256, 128
    w = _random_bf16(rng, N, K)
    qw, s, z = quantize_linear(w, G)
    q = unpack_nibbles(qw, K).astype(np.int64)
    sf = np.repeat(s.astype(np.float64), G, axis=1)
    zf = np.repeat(z.astype(np.float64), G, axis=1)
    grid = (np.arange(16)[None, None, :] - zf[:, :, None]) * sf[:, :, None]   # [N][K][16]
    dist = np.abs(grid - w.astype(np.float64)[:, :, None])
    best = dist.min(axis=2)
    chosen = np.take_along_axis(dist, q[:, :, None], axis=2)[:, :, 0]
    # Equal up to the fp32 rounding of w/s + z (a tie may go either way).
    assert np.all(chosen <= best + 1e-6 * sf)


def test_min_and_max_map_to_the_ends():
    rng = np.random.default_rng(2)
    N, K, G = 16, 512, 128
    w = _random_bf16(rng, N, K)
    qw, s, z = quantize_linear(w, G)
    q = unpack_nibbles(qw, K)
    for g in range(K // G):
        blk = w[:, g * G:(g + 1) * G]
        qb = q[:, g * G:(g + 1) * G]
        assert np.all(qb[np.arange(N), blk.argmin(axis=1)] == 0)
        assert np.all(qb[np.arange(N), blk.argmax(axis=1)] == 15)


def test_degenerate_group_gets_unit_scale():
    w = np.full((2, 128), 0.375, np.float32)
    w[1] = -0.125
    qw, s, z = quantize_linear(w, 128)
    assert np.all(s == 1.0)
    assert z[0, 0] == np.float16(-0.375) and z[1, 0] == np.float16(0.125)
    assert np.all(unpack_nibbles(qw, 128) == 0)
    assert np.array_equal(dequantize_linear(qw, s, z, 128), w)


def test_ragged_last_group():
    """K = 688 (the tiny shape's FFN width): five full groups and one of 48."""
    rng = np.random.default_rng(3)
    K = 688
    w = _random_bf16(rng, 3, K)
    w[:, 640:] = np.linspace(-1.0, 2.0, 48, dtype=np.float32)[None, :]
    qw, s, z = quantize_linear(w, 128)
    assert s.shape == (3, 6) and qw.shape == (3, 86)
    # The last group's range is that of its 48 members only.
    assert np.all(s[:, 5] == np.float16(np.float32(3.0) / np.float32(15.0)))
    q = unpack_nibbles(qw, K)
    assert np.all(q[:, 640] == 0) and np.all(q[:, 687] == 15)


def test_fp16_rounding_matches_torch():
    """numpy's float32 -> float16 conversion is round-to-nearest-even, as
    torch's (library cross-check, ties and subnormals included)."""
    import torch
    rng = np.random.default_rng(4)
    base = rng.standard_normal(20000).astype(np.float32) * np.float32(0.01)
    h = base.astype(np.float16).astype(np.float32)
    ties = (h + np.float32(2.0 ** -12) * np.abs(h)).astype(np.float32)  # near-midpoints
    sub = (rng.random(2000).astype(np.float32) * np.float32(6e-5))      # fp16 subnormal range
    x = np.concatenate([base, ties, sub])
    a = x.astype(np.float16).view(np.uint16)
    b = torch.from_numpy(x).to(torch.float16).numpy().view(np.uint16)
    assert np.array_equal(a, b)
