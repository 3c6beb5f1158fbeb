"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin
catches each one.  This shows the pins are sensitive, not just green."""
import numpy as np
import pytest

import synth
from oracle import model as om
from oracle import quant as oq
from oracle.model import OracleModel, Policy, KVState
from tests.test_oracle_model import _torch_llama

S = synth.scaled(synth.TINY, n_layers=2, vocab=128)


@pytest.fixture(scope="module")
def w():
    return synth.weights_to_numpy(synth.gen_weights(S, seed=0, device="cpu", gains="random"))


def _matches_independent(w):
    toks = synth.gen_tokens(S.vocab, (1, 6), seed=1)
    ref = _torch_llama(S, w, toks)
    m = OracleModel(S, w)
    st = KVState(S, 1, 8)
    r = m.prefill(toks, st, Policy.tau_(1.01))
    return np.allclose(r.logits, ref[:, -1], atol=2e-4, rtol=1e-4)


def _rmsnorm_no_gain(x, g, eps):
    x = x.astype(np.float32)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rope_wrong_sign(x, positions, theta):
    hd = x.shape[-1]
    return _ORIG["rope"](x, -np.asarray(positions), theta)


def _rope_adjacent_pairs(x, positions, theta):
    # Interleaved-pair RoPE instead of rotate-half.
    y = np.concatenate([x[..., 0::2], x[..., 1::2]], axis=-1)
    r = _ORIG["rope"](y, positions, theta)
    out = np.empty_like(r)
    half = x.shape[-1] // 2
    out[..., 0::2] = r[..., :half]
    out[..., 1::2] = r[..., half:]
    return out


def _attention_no_scale(q, k, v, q_pos):
    return _ORIG["attention"](q * np.float32(np.sqrt(q.shape[-1])), k, v, q_pos)


def _attention_wrong_group(q, k, v, q_pos):
    # Query head h reads KV head h % Hkv instead of h // (Hq/Hkv).
    Hq, Hkv = q.shape[1], k.shape[0]
    return np.stack([_ORIG["attention"](q[:, h:h + 1], k[h % Hkv][None], v[h % Hkv][None], q_pos)[:, 0]
                     for h in range(Hq)], axis=1)


def _attention_not_causal(q, k, v, q_pos):
    return _ORIG["attention"](q, k, v, np.full_like(np.asarray(q_pos), k.shape[1] - 1))


def _silu_is_sigmoid(a):
    return (1.0 / (1.0 + np.exp(-a))).astype(np.float32)


_ORIG = {"rope": om.rope, "attention": om.attention}

MODEL_MUTATIONS = {
    "rmsnorm drops the gain": ("rmsnorm", _rmsnorm_no_gain),
    "RoPE angle sign flipped": ("rope", _rope_wrong_sign),
    "RoPE on adjacent pairs": ("rope", _rope_adjacent_pairs),
    "attention without 1/sqrt(hd)": ("attention", _attention_no_scale),
    "GQA head-to-group map wrong": ("attention", _attention_wrong_group),
    "attention not causal": ("attention", _attention_not_causal),
    "silu replaced by sigmoid": ("silu", _silu_is_sigmoid),
}


@pytest.mark.parametrize("name", sorted(MODEL_MUTATIONS))
def test_model_mutation_is_caught(name, w, monkeypatch):
    attr, fn = MODEL_MUTATIONS[name]
    assert _matches_independent(w)
    monkeypatch.setattr(om, attr, fn)
    assert not _matches_independent(w), f"pin missed mutation: {name}"


def test_transposed_operand_is_caught(w):
    w2 = dict(w)
    w2["layers"] = [dict(lw) for lw in w["layers"]]
    w2["layers"][0]["wo"] = np.ascontiguousarray(w["layers"][0]["wo"].T)   # square: still runs
    toks = synth.gen_tokens(S.vocab, (1, 6), seed=1)
    ref = _torch_llama(S, w, toks)
    r = OracleModel(S, w2).prefill(toks, KVState(S, 1, 8), Policy.tau_(1.01))
    assert not np.allclose(r.logits, ref[:, -1], atol=2e-4)


def test_exit_rule_mutations_are_caught(w, monkeypatch):
    """Non-strict compare, or deciding again after an exit, breaks the
    first-excess pin."""
    m = OracleModel(S, w)
    m.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (1, 6), seed=2)
    ref = m.prefill(toks, KVState(S, 1, 8), Policy.tau_(1.01))
    tau = float(ref.min_cos[0])
    # Strict compare: tau equal to the first layer's cosine must not exit there.
    r = m.prefill(toks, KVState(S, 1, 8), Policy.tau_(tau))
    assert r.exit_layer != 1
    # A '>=' mutation would exit at layer 1: show the pin would see it.
    orig_run = OracleModel.run

    def run_ge(self, tokens, st, policy):
        return orig_run(self, tokens, st, Policy.tau_(float(np.nextafter(np.float32(policy.tau), np.float32(-2)))))

    monkeypatch.setattr(OracleModel, "run", run_ge)
    assert m.prefill(toks, KVState(S, 1, 8), Policy.tau_(tau)).exit_layer == 1


def test_quant_mutations_are_caught(monkeypatch):
    """A reversed nibble order fails the closed-form packing pin; truncation
    instead of rounding fails the nearest-grid-point pin."""
    from tests import test_oracle_quant as tq
    orig_q = oq.quantize_linear

    def reversed_nibbles(w, group=128):
        qw, s, z = orig_q(w, group)
        q = oq.unpack_nibbles(qw, w.shape[1])
        q = q.reshape(q.shape[0], -1, 8)[:, :, ::-1].reshape(q.shape[0], -1).astype(np.uint32)
        out = np.zeros_like(qw)
        for i in range(8):
            out |= q[:, i::8] << np.uint32(4 * i)
        return out, s, z

    monkeypatch.setattr(tq, "quantize_linear", reversed_nibbles)
    with pytest.raises(AssertionError):
        tq.test_packing_closed_form()

    orig_rint = np.rint
    monkeypatch.setattr(tq, "quantize_linear", orig_q)
    monkeypatch.setattr(oq.np, "rint", np.trunc)
    try:
        with pytest.raises(AssertionError):
            tq.test_nearest_grid_point_brute_force()
    finally:
        monkeypatch.setattr(oq.np, "rint", orig_rint)
