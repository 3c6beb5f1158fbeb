"""Pins of the oracle's exit-vs-backbone K/V similarity (River-LLM explainer,
section 三: an exit layer's K/V lands in the backbone's own slot and stays
close to what the backbone layer would have written there).

* it is the cosine between the cache entries the two weight sets actually
  write: run the layer once on each weight set at the same position and
  compare the K/V slots head by head;
* an exit river built from the unquantized weights gives cosine 1;
* RoPE rotates both keys alike, so the result does not depend on the position.
"""
import numpy as np

import synth
from oracle.model import KVState, OracleModel

S = synth.TINY


def _model():
    w = synth.weights_to_numpy(synth.gen_weights(S, seed=0, device="cpu", gains="random"))
    om = OracleModel(S, w)
    om.quantize_exit_layers()
    return om


def _head_cos(a, b):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    return (a * b).sum(-1) / (np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1))


def test_equals_the_cosine_of_the_slots_each_weight_set_writes():
    om = _model()
    rng = np.random.default_rng(0)
    B, pos = 3, 5
    h = rng.standard_normal((B, S.d_model)).astype(np.float32)
    for l in (0, S.n_layers - 1):
        got = om.exit_kv_cosine(l, h, pos)
        sb, se = KVState(S, B, pos + 1), KVState(S, B, pos + 1)
        om.layer(l, om.backbone[l], h[:, None, :], sb, pos)
        om.layer(l, om.exit[l], h[:, None, :], se, pos)
        for j, (cb, ce) in enumerate(((sb.K, se.K), (sb.V, se.V))):
            ref = _head_cos(cb[l][:, :, pos], ce[l][:, :, pos])   # [B][Hkv]
            assert np.allclose(got[:, j], ref, atol=2e-6), (l, j, got[:, j], ref)
        assert np.all(got < 1.0 - 1e-6), "W4 copies differ from the backbone"


def test_unquantized_exit_river_gives_one():
    om = _model()
    om.copy_exit_layers_unquantized()
    h = np.random.default_rng(1).standard_normal((2, S.d_model)).astype(np.float32)
    assert np.allclose(om.exit_kv_cosine(1, h, 3), 1.0, atol=1e-6)


def test_does_not_depend_on_the_position():
    om = _model()
    h = np.random.default_rng(2).standard_normal((2, S.d_model)).astype(np.float32)
    a, b = om.exit_kv_cosine(2, h, 0), om.exit_kv_cosine(2, h, 977)
    assert np.allclose(a, b, atol=2e-6)
