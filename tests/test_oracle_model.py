"""Pins of the oracle's decoder and exit river against things other than itself.

River-LLM explainer: section 三 (exit layers share the backbone's KV slots),
section 四 (batch-min state-transition similarity vs tau, one-shot), section
五 (sequence-level exit in prefill, per-step exit in generation).
"""
import numpy as np
import pytest
import scipy.spatial.distance as ssd
import torch
import torch.nn.functional as F

import synth
from oracle import model as om
from oracle.model import OracleModel, Policy, KVState

SMALL = synth.scaled(synth.TINY, name="tiny", n_layers=3, vocab=256)


@pytest.fixture(scope="module")
def tiny_weights():
    return synth.weights_to_numpy(synth.gen_weights(SMALL, seed=0, device="cpu", gains="random"))


@pytest.fixture(scope="module")
def tiny_weights_full():
    return synth.weights_to_numpy(synth.gen_weights(synth.TINY, seed=0, device="cpu", gains="random"))


# ---------------------------------------------------------------- building blocks

def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 256)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(256)).astype(np.float32)
    ref = F.rms_norm(torch.from_numpy(x).double(), (256,), torch.from_numpy(g).double(), eps=1e-5)
    assert np.allclose(om.rmsnorm(x, g, 1e-5), ref.numpy(), rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("hd,theta", [(64, 1e4), (128, 5e5)])
def test_rope_is_complex_rotation(hd, theta):
    """Rotate-half RoPE equals multiplying (x_i + i x_{i+hd/2}) by e^{i p w_i}."""
    rng = np.random.default_rng(1)
    n, H = 7, 3
    x = rng.standard_normal((n, H, hd)).astype(np.float32)
    pos = np.array([0, 1, 5, 100, 511, 2047, 4351])
    half = hd // 2
    w = theta ** (-np.arange(half) * 2.0 / hd)
    z = x[..., :half].astype(np.float64) + 1j * x[..., half:].astype(np.float64)
    r = z * np.exp(1j * pos[:, None, None] * w[None, None, :])
    ref = np.concatenate([r.real, r.imag], axis=-1)
    # fp32 angle: error grows with the position (2^-24 * p relative).
    assert np.allclose(om.rope(x, pos, theta), ref, atol=2e-3, rtol=1e-4)
    assert np.allclose(om.rope(x[:3], pos[:3], theta), ref[:3], atol=1e-5)


def test_silu_matches_torch():
    a = np.linspace(-30, 30, 1001).astype(np.float32)
    assert np.allclose(om.silu(a), F.silu(torch.from_numpy(a).double()).numpy(), rtol=1e-6, atol=1e-6)


def test_cosine_matches_scipy():
    rng = np.random.default_rng(2)
    a = rng.standard_normal((4, 300)).astype(np.float32)
    b = (a + 0.7 * rng.standard_normal((4, 300))).astype(np.float32)
    ref = [1.0 - ssd.cosine(a[i].astype(np.float64), b[i].astype(np.float64)) for i in range(4)]
    assert np.allclose(om.cosine(a, b), ref, atol=1e-6)
    assert om.cosine(np.zeros((1, 8), np.float32), np.ones((1, 8), np.float32))[0] == 0.0


@pytest.mark.parametrize("Hq,Hkv,hd", [(4, 2, 64), (8, 2, 16), (3, 3, 8)])
def test_attention_matches_sdpa(Hq, Hkv, hd):
    """Causal GQA attention vs torch's scaled_dot_product_attention."""
    rng = np.random.default_rng(3)
    T, n = 9, 4
    q = rng.standard_normal((n, Hq, hd)).astype(np.float32)
    k = rng.standard_normal((Hkv, T, hd)).astype(np.float32)
    v = rng.standard_normal((Hkv, T, hd)).astype(np.float32)
    qpos = np.arange(T - n, T)
    out = om.attention(q, k, v, qpos)
    rep = Hq // Hkv
    kt = torch.from_numpy(k).double().repeat_interleave(rep, 0)
    vt = torch.from_numpy(v).double().repeat_interleave(rep, 0)
    qt = torch.from_numpy(q).double().transpose(0, 1)            # [Hq][n][hd]
    mask = torch.from_numpy(np.arange(T)[None, :] <= qpos[:, None])
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    assert np.allclose(out, ref.transpose(0, 1).numpy(), atol=1e-5)


def test_attention_three_tokens_by_hand():
    """Explicit softmax matrix on a 3-token, 1-head case."""
    q = np.array([[[1.0, 0.0]], [[0.0, 2.0]], [[1.0, 1.0]]], np.float32)   # [3][1][2]
    k = np.array([[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]], np.float32)         # [1][3][2]
    v = np.array([[[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]]], np.float32)
    out = om.attention(q, k, v, np.array([0, 1, 2]))
    sc = 1 / np.sqrt(2.0)
    expect = []
    for i, qi in enumerate(q[:, 0]):
        s = np.array([qi @ k[0, j] * sc for j in range(i + 1)])
        p = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
        expect.append(p @ v[0, :i + 1])
    assert np.allclose(out[:, 0], np.array(expect), atol=1e-6)


# ------------------------------------------------ whole decoder vs an independent one

def _torch_llama(shape, w, tokens):
    """Standard Llama forward in float64 from torch library routines
    (rms_norm, linear, complex RoPE, scaled_dot_product_attention, silu)."""
    S = shape
    t = lambda a: torch.from_numpy(np.asarray(a)).double()
    B, T = tokens.shape
    Hq, Hkv, hd = S.n_q_heads, S.n_kv_heads, S.head_dim
    h = t(w["embed"])[torch.from_numpy(tokens).long()]
    pos = torch.arange(T, dtype=torch.float64)
    freqs = S.rope_theta ** (-torch.arange(hd // 2, dtype=torch.float64) * 2 / hd)
    rot = torch.polar(torch.ones(T, hd // 2, dtype=torch.float64), pos[:, None] * freqs[None])

    def rope(x):                       # [B][T][H][hd]
        z = torch.complex(x[..., :hd // 2], x[..., hd // 2:]) * rot[None, :, None, :]
        return torch.cat([z.real, z.imag], -1)

    for lw in w["layers"]:
        x = F.rms_norm(h, (S.d_model,), t(lw["g_attn"]), eps=S.rms_eps)
        q = rope(F.linear(x, t(lw["wq"])).view(B, T, Hq, hd))
        k = rope(F.linear(x, t(lw["wk"])).view(B, T, Hkv, hd))
        v = F.linear(x, t(lw["wv"])).view(B, T, Hkv, hd)
        rep = Hq // Hkv
        o = F.scaled_dot_product_attention(
            q.transpose(1, 2), k.transpose(1, 2).repeat_interleave(rep, 1),
            v.transpose(1, 2).repeat_interleave(rep, 1), is_causal=True)
        h = h + F.linear(o.transpose(1, 2).reshape(B, T, Hq * hd), t(lw["wo"]))
        x2 = F.rms_norm(h, (S.d_model,), t(lw["g_ffn"]), eps=S.rms_eps)
        h = h + F.linear(F.silu(F.linear(x2, t(lw["wg"]))) * F.linear(x2, t(lw["wu"])), t(lw["wd"]))
    hf = F.rms_norm(h, (S.d_model,), t(w["g_final"]), eps=S.rms_eps)
    return F.linear(hf, t(w["lm_head"])).numpy()


def test_full_depth_matches_independent_llama(tiny_weights_full):
    S = synth.TINY
    toks = synth.gen_tokens(S.vocab, (2, 12), seed=1)
    ref = _torch_llama(S, tiny_weights_full, toks)
    m = OracleModel(S, tiny_weights_full)
    st = KVState(S, 2, 32)
    r = m.prefill(toks[:, :8], st, Policy.tau_(1.01))
    assert r.exit_layer == S.n_layers
    assert np.allclose(r.logits, ref[:, 7], atol=2e-4, rtol=1e-4)
    for i in range(8, 12):
        r = m.decode_step(toks[:, i], st, Policy.tau_(1.01))
        assert np.allclose(r.logits, ref[:, i], atol=2e-4, rtol=1e-4)


# ------------------------------------------------------------- exit-river invariants

def _decode_run(m, S, toks, policies, B=1, prompt=6):
    st = KVState(S, B, 64)
    res = [m.prefill(toks[:, :prompt], st, policies[0])]
    for i, pol in enumerate(policies[1:]):
        res.append(m.decode_step(toks[:, prompt + i], st, pol))
    return res, st


def test_tau_above_one_is_full_model(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (2, 12), seed=5)
    a, _ = _decode_run(m, S, toks, [Policy.tau_(1.01)] * 7, B=2)
    b, _ = _decode_run(m, S, toks, [Policy.forced(S.n_layers)] * 7, B=2)
    for x, y in zip(a, b):
        assert x.exit_layer == S.n_layers
        assert np.array_equal(x.logits, y.logits)


def test_tau_below_minus_one_exits_at_layer_one(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (1, 12), seed=6)
    a, _ = _decode_run(m, S, toks, [Policy.tau_(-1.01)] * 7)
    b, _ = _decode_run(m, S, toks, [Policy.forced(1)] * 7)
    for x, y in zip(a, b):
        assert x.exit_layer == 1
        assert np.array_equal(x.logits, y.logits)


def test_first_layer_above_tau_decides(tiny_weights):
    """One-shot rule: e is the first l < L whose batch-min cosine exceeds tau."""
    S = synth.scaled(SMALL, n_layers=4)
    w = synth.weights_to_numpy(synth.gen_weights(S, seed=11, device="cpu", gains="random"))
    m = OracleModel(S, w)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (2, 10), seed=7)
    ref, _ = _decode_run(m, S, toks, [Policy.tau_(1.01)] * 4, B=2)
    for tau in sorted(set(float(c) for r in ref for c in r.min_cos[:-1])):
        for pick in (np.nextafter(np.float32(tau), np.float32(-2)), np.float32(tau)):
            res, _ = _decode_run(m, S, toks, [Policy.tau_(float(pick))] * 1, B=2)
            r = res[0]
            # Layers up to the decision are backbone layers, so their cosines
            # equal the full-depth run's; the decision is the first strict excess.
            above = [l + 1 for l in range(S.n_layers - 1) if ref[0].min_cos[l] > pick]
            assert r.exit_layer == (above[0] if above else S.n_layers)
            e = r.exit_layer
            assert np.array_equal(r.min_cos[:e], ref[0].min_cos[:e])


def test_batch_min_is_the_minimum_over_tokens(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    toks = synth.gen_tokens(S.vocab, (3, 5), seed=8)
    st = KVState(S, 3, 16)
    r = m.prefill(toks, st, Policy.tau_(1.01))
    # Recompute the per-token cosines from the hidden trace of single-sequence runs.
    for l in range(S.n_layers):
        per = []
        for b in range(3):
            st1 = KVState(S, 1, 16)
            m2 = OracleModel(S, tiny_weights)
            rb = m2.prefill(toks[b:b + 1], st1, Policy.tau_(1.01))
            per.append(rb.min_cos[l])
        assert r.min_cos[l] == np.float32(min(per)) or np.isclose(r.min_cos[l], min(per), atol=1e-7)


def test_unquantized_exit_river_equals_backbone(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.copy_exit_layers_unquantized()
    toks = synth.gen_tokens(S.vocab, (2, 12), seed=9)
    ref, _ = _decode_run(m, S, toks, [Policy.forced(S.n_layers)] * 7, B=2)
    for sched in ([0, 1, 2, 3, 1, 0, 2], [1, 1, 1, 1, 1, 1, 1], [2, 0, 3, 1, 2, 3, 0]):
        res, _ = _decode_run(m, S, toks, [Policy.forced(e) for e in sched], B=2)
        for x, y in zip(res, ref):
            assert np.allclose(x.logits, y.logits, atol=1e-6)


def test_quantized_exit_river_differs_but_stays_close(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (1, 8), seed=10)
    a, _ = _decode_run(m, S, toks, [Policy.forced(S.n_layers)] * 3)
    b, _ = _decode_run(m, S, toks, [Policy.forced(0)] * 3)
    d = np.abs(a[-1].logits - b[-1].logits).max()
    assert 0 < d < 0.5


def test_cached_decode_equals_recompute(tiny_weights):
    """Incremental decode with per-step exits == full-prefix recompute in which
    every position uses its own step's exit layer (the KV slots it wrote)."""
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (2, 14), seed=12)
    prompt = 6
    sched = [2, 0, 3, 1, 1, 2, 0, 3]
    res, _ = _decode_run(m, S, toks, [Policy.forced(e) for e in sched], B=2, prompt=prompt)
    per_pos = np.array([sched[0]] * prompt + sched[1:])
    full = m.recompute(toks[:, :prompt + len(sched) - 1], per_pos)
    assert np.allclose(res[0].logits, full[:, prompt - 1], atol=1e-5)
    for i, r in enumerate(res[1:]):
        assert np.allclose(r.logits, full[:, prompt + i], atol=1e-5)


def test_exit_writes_exactly_slot_p_of_every_layer(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (2, 10), seed=13)
    st = KVState(S, 2, 32)
    m.prefill(toks[:, :6], st, Policy.tau_(1.01))
    for e in (0, 1, S.n_layers):
        before = [(k.copy(), v.copy()) for k, v in zip(st.K, st.V)]
        p = st.pos
        r = m.decode_step(toks[:, p], st, Policy.forced(e))
        assert r.exit_layer == e
        for l in range(S.n_layers):
            for new, old in ((st.K[l], before[l][0]), (st.V[l], before[l][1])):
                changed = np.any(new != old, axis=(0, 1, 3))
                assert changed[p] and changed.sum() == 1


def test_prefill_takes_one_decision_for_all_tokens(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (2, 8), seed=14)
    st = KVState(S, 2, 16)
    ref = m.prefill(toks, st, Policy.tau_(1.01))
    tau = float(ref.min_cos[0]) - 1e-3
    st2 = KVState(S, 2, 16)
    r = m.prefill(toks, st2, Policy.tau_(tau))
    assert r.exit_layer == 1
    st3 = KVState(S, 2, 16)
    f = m.prefill(toks, st3, Policy.forced(1))
    assert np.array_equal(r.logits, f.logits)
    for l in range(S.n_layers):
        assert np.array_equal(st2.K[l], st3.K[l]) and np.array_equal(st2.V[l], st3.V[l])


def test_capacity_and_policy_errors(tiny_weights):
    S = SMALL
    m = OracleModel(S, tiny_weights)
    st = KVState(S, 1, 4)
    with pytest.raises(ValueError):
        m.prefill(np.zeros((1, 5), np.int32), st, Policy.tau_(1.01))
    with pytest.raises(ValueError):
        m.prefill(np.zeros((1, 2), np.int32), st, Policy.forced(1))   # exit river not built
    with pytest.raises(ValueError):
        m.prefill(np.zeros((1, 2), np.int32), st, Policy.forced(S.n_layers + 1))


def test_schedule_generator_mean():
    assert abs(synth.solve_geometric_p(16, 3.8) - 0.31559) < 1e-4
    assert abs(synth.solve_geometric_p(32, 8.0) - 0.14738) < 1e-4
    s = synth.gen_schedule(16, 200000, 3.8)
    assert abs(s.mean() - 3.8) < 0.05 and s.min() >= 1 and s.max() == 16
    assert abs(np.mean(s == 16) - 0.05) < 0.005
