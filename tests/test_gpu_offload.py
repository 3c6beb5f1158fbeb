"""Backbone offloading (River-LLM explainer, section 五): the backbone weights
of the deep layers live in pinned host memory and are read only by steps that
run those layers on the backbone.

* the model's device footprint shrinks by the offloaded layers' two bf16
  copies (less one layer's staging buffer), and the host holds them;
* prefill and decode steps on every path (persistent step kernel, fused,
  generic) give bit-identical logits, tokens and exit layers to the same
  model fully resident, under a forced schedule that runs offloaded layers
  on the backbone (full depth, exit after layer 3) and on the exit river,
  and under tau; and they match the oracle;
* offloading needs the exit river and happens once.
"""
import numpy as np
import pytest

import synth
from oracle.model import KVState, Policy as OPolicy
from tests.harness import build_pair, check_step, to_cuda

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TINY = synth.TINY
FIRST = 2  # layers 3 and 4 (1-based) offloaded


@pytest.fixture(scope="module")
def river():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_gb300 as r
    return r


@pytest.fixture(scope="module")
def stream(river):
    return torch.cuda.Stream()


@pytest.fixture(scope="module")
def pair(river, stream):
    """(resident model, offloaded model, oracle) from the same weights."""
    with torch.cuda.stream(stream):
        res, om, w = build_pair(TINY, seed=0, gains="random", stream=stream)
        off = river.Model(TINY, to_cuda(w), stream)
        off.quantize_exit_layers(stream)
    stream.synchronize()
    d0, h0 = off.memory()
    off.offload_backbone(FIRST, stream)
    d1, h1 = off.memory()
    return res, off, om, (d0, h0, d1, h1)


def test_footprint_moves_to_host(pair):
    _, _, _, (d0, h0, d1, h1) = pair
    S = TINY
    Kd = (S.d_model + 127) // 128 * 128
    Ko = (S.n_q_heads * S.head_dim + 127) // 128 * 128
    Kf = (S.ffn_dim + 127) // 128 * 128
    layer = 2 * ((S.n_q_heads + 2 * S.n_kv_heads) * S.head_dim * Kd + S.d_model * Ko +
                 2 * S.ffn_dim * Kd + S.d_model * Kf)  # bf16 bytes of one layer's four matrices
    n_off = S.n_layers - FIRST
    assert h0 == 0 and h1 == 2 * n_off * layer
    assert d0 - d1 == 2 * n_off * layer - layer


def _sequence(river, m, stream, B, path, policies, toks, steps):
    kv = m.kv_cache_alloc(B, 64)
    kv.set_decode_path(path)
    assert kv.decode_path(B) == path
    outs = []
    with torch.cuda.stream(stream):
        o = river.prefill(m, kv, torch.from_numpy(toks[:, :-steps]).cuda(), policies[0], stream=stream)
        kv.sync(stream)
        outs.append({k: v.clone() for k, v in o.items()})
        for i in range(steps):
            o = river.decode_step(m, kv, torch.from_numpy(toks[:, -steps + i].copy()).cuda(),
                                  policies[1 + i], stream=stream)
            kv.sync(stream)
            outs.append({k: v.clone() for k, v in o.items()})
    return outs


@pytest.mark.parametrize("B,path", [(1, 1), (2, 2), (3, 3)])
def test_offloaded_steps_are_bit_identical_and_match_the_oracle(river, pair, stream, B, path):
    res, off, om, _ = pair
    S = TINY
    L = S.n_layers
    sched = [L, 3, 2, 0, L, 1, 3, L]
    d_sched = torch.tensor(sched, dtype=torch.int32, device="cuda")
    steps = len(sched)
    toks = synth.gen_tokens(S.vocab, (B, 16 + steps), seed=1)
    pols = [river.Policy.tau_(1.01)] + [river.Policy.forced(d_sched)] * steps
    a = _sequence(river, res, stream, B, path, pols, toks, steps)
    b = _sequence(river, off, stream, B, path, pols, toks, steps)
    for i, (x, y) in enumerate(zip(a, b)):
        for k in ("logits", "next_token", "exit_layer"):
            assert torch.equal(x[k], y[k]), f"step {i}: {k} differs after offloading"
    # and the oracle, teacher-forced on the same tokens
    st = KVState(S, B, 64)
    ref = om.prefill(toks[:, :16], st, OPolicy.tau_(1.01))
    check_step(b[0], ref, None, B, "prefill")
    for i, e in enumerate(sched):
        ref = om.decode_step(toks[:, 16 + i], st, OPolicy.forced(e))
        assert int(b[1 + i]["exit_layer"].item()) == e
        check_step(b[1 + i], ref, None, B, f"decode step {i} (exit layer {e})")


def test_offloaded_tau_steps_are_bit_identical(river, pair, stream):
    res, off, _, _ = pair
    toks = synth.gen_tokens(TINY.vocab, (1, 24), seed=2)
    pols = [river.Policy.tau_(0.5)] * 9
    for path in (1, 3):
        a = _sequence(river, res, stream, 1, path, pols, toks, 8)
        b = _sequence(river, off, stream, 1, path, pols, toks, 8)
        for x, y in zip(a, b):
            assert torch.equal(x["logits"], y["logits"]) and torch.equal(x["exit_layer"], y["exit_layer"])


def test_offloading_needs_the_exit_river_and_happens_once(river, pair, stream):
    _, off, _, _ = pair
    with pytest.raises(river.RiverError) as ei:
        off.offload_backbone(1, stream)
    assert ei.value.status == river.RL_ERR_STATE
    w = synth.gen_weights(TINY, seed=0, device="cpu", gains="ones")
    with torch.cuda.stream(stream):
        m = river.Model(TINY, to_cuda(w), stream)
    with pytest.raises(river.RiverError) as ei:
        m.offload_backbone(1, stream)
    assert ei.value.status == river.RL_ERR_STATE
    with pytest.raises(river.RiverError):
        river.rl_model_offload_backbone(m.handle, TINY.n_layers + 1, stream)
