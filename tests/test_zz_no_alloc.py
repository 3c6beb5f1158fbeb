"""rl_lm_head_static, the allocation-free LM-head entry point: on the final
residual rows of a decode step it must give the logits and greedy tokens that
rl_decode_step's own LM head gave, on two calls in a row (the second call
finds the static scratch as the first one left it)."""
import numpy as np
import pytest

import synth
from tests.harness import LOGIT_TOL, build_pair

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

S = synth.TINY
GAP = 0.1  # greedy tokens compared where the top-1 / top-2 logit gap exceeds this


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
def model(river, stream):
    with torch.cuda.stream(stream):
        m, _, _ = build_pair(S, seed=0, gains="random", stream=stream)
    stream.synchronize()
    return m


def _decode_step_outputs(river, m, stream, B, exit_layer):
    """One decode step through rl_decode_step; returns its outputs and the
    residual rows that entered its final RMSNorm (from the layer trace)."""
    kv = m.kv_cache_alloc(B, 64)
    tr = torch.zeros((S.n_layers + 1, B, S.d_model), dtype=torch.float32, device="cuda")
    kv.set_trace(tr)
    prompt = torch.from_numpy(synth.gen_tokens(S.vocab, (B, 16), seed=1)).cuda()
    tok = torch.from_numpy(synth.gen_tokens(S.vocab, (1, B), seed=4)[0].copy()).cuda()
    sched = torch.tensor([exit_layer], dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        river.prefill(m, kv, prompt, river.Policy.tau_(1.01), stream=stream)
        out = river.decode_step(m, kv, tok, river.Policy.forced(sched), stream=stream)
        kv.sync(stream)
    h = tr[S.n_layers].clone()
    kv.set_trace(None)
    return out, h, kv


@pytest.mark.parametrize("B,exit_layer", [(1, S.n_layers), (3, 2), (8, 0)])
def test_static_lm_head_matches_decode_step(river, model, stream, B, exit_layer):
    out, h, kv = _decode_step_outputs(river, model, stream, B, exit_layer)
    ref_logits = out["logits"].cpu().numpy()
    ref_tok = out["next_token"].cpu().numpy()
    top2 = np.sort(ref_logits, axis=-1)[:, -2:]
    decided = (top2[:, 1] - top2[:, 0]) > GAP
    for call in range(2):
        logits = torch.full((B, S.vocab), float("nan"), dtype=torch.float32, device="cuda")
        tok = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            river.rl_lm_head_static(model.handle, h, B, logits, tok, err, stream)
        stream.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error bits {int(err.item())}"
        got = logits.cpu().numpy()
        d = np.abs(got - ref_logits).max()
        assert d <= LOGIT_TOL, f"call {call}: max |dlogit| {d:.4g} > {LOGIT_TOL}"
        t = tok.cpu().numpy()
        assert np.array_equal(t[decided], ref_tok[decided]), f"call {call}: {t} vs {ref_tok}"
        assert np.all(t == got.argmax(-1)), f"call {call}: token is not the argmax of its logits"
    del kv


def test_static_lm_head_rejects_sizes_beyond_its_limit(river, model, stream):
    h = torch.zeros((9, S.d_model), dtype=torch.float32, device="cuda")
    logits = torch.full((9, S.vocab), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(river.RiverError) as ei:
        river.rl_lm_head_static(model.handle, h, 9, logits, None, None, stream)
    assert ei.value.status == river.RL_ERR_UNSUPPORTED
    assert "batch" in str(ei.value)
    stream.synchronize()
    assert bool((logits == 7.0).all()), "a rejected call must enqueue nothing"
