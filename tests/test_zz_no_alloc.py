"""rl_lm_head_static, the allocation-free LM-head entry point: on the final
residual rows of a decode step it must give the logits and greedy tokens that
rl_decode_step's own LM head gave and that the oracle's final RMSNorm + LM
head computes from the same rows, on two calls in a row (the second call
finds the static scratch as the first one left it).  Sizes beyond its limits
(batch above 8, or rows that do not fit in shared memory beside the weight
ring, as batch 7 at d_model 8192) are rejected before anything is enqueued."""
import dataclasses

import numpy as np
import pytest

import synth
from oracle.model import rmsnorm
from tests.harness import LOGIT_TOL, build_pair, to_cuda

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
    # the oracle's final RMSNorm + LM head on the same rows (fp32 CPU)
    w = synth.gen_weights(S, seed=0, device="cpu", gains="random")
    wn = synth.weights_to_numpy(w)
    ora = rmsnorm(h.cpu().numpy(), wn["g_final"], S.rms_eps) @ wn["lm_head"].T
    srt = np.sort(ora, axis=-1)
    ora_decided = (srt[:, -1] - srt[:, -2]) > GAP
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
        d_or = np.abs(got - ora).max()
        assert d_or <= LOGIT_TOL, f"call {call}: max |dlogit| vs the oracle {d_or:.4g} > {LOGIT_TOL}"
        assert np.array_equal(t[ora_decided], ora.argmax(-1)[ora_decided]), \
            f"call {call}: tokens {t} vs the oracle's {ora.argmax(-1)}"
    del kv


# A one-layer model whose d_model is the entry point's maximum (8192): only its
# LM head, final gain and embedding matter here.
WIDE = dataclasses.replace(synth.TINY, name="wide-lm-head", n_layers=1, d_model=8192, n_q_heads=1,
                           n_kv_heads=1, head_dim=64, ffn_dim=128, vocab=512)


@pytest.fixture(scope="module")
def wide(river, stream):
    w = synth.gen_weights(WIDE, seed=0, device="cpu", gains="random")
    with torch.cuda.stream(stream):
        m = river.Model(WIDE, to_cuda(w), stream)
    stream.synchronize()
    return m, synth.weights_to_numpy(w)


def test_static_lm_head_at_d_model_8192_matches_the_oracle(river, wide, stream):
    m, wn = wide
    B = 6  # the largest batch whose rows fit beside the weight ring at d_model 8192
    rng = np.random.default_rng(5)
    h_np = rng.standard_normal((B, WIDE.d_model)).astype(np.float32)
    h = torch.from_numpy(h_np).cuda()
    ora = rmsnorm(h_np, wn["g_final"], WIDE.rms_eps) @ wn["lm_head"].T
    srt = np.sort(ora, axis=-1)
    decided = (srt[:, -1] - srt[:, -2]) > GAP
    for call in range(2):
        logits = torch.full((B, WIDE.vocab), float("nan"), dtype=torch.float32, device="cuda")
        tok = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            river.rl_lm_head_static(m.handle, h, B, logits, tok, err, stream)
        stream.synchronize()
        assert int(err.item()) == 0
        got = logits.cpu().numpy()
        d = np.abs(got - ora).max()
        assert d <= LOGIT_TOL, f"call {call}: max |dlogit| {d:.4g}"
        t = tok.cpu().numpy()
        assert np.array_equal(t[decided], ora.argmax(-1)[decided]), f"call {call}: {t}"


def test_static_lm_head_rejects_rows_beyond_shared_memory(river, wide, stream):
    m, _ = wide
    B = 7  # batch 7 at d_model 8192: 7 * (2*8192 + 64 + 256) bytes > 115,712
    h = torch.zeros((B, WIDE.d_model), dtype=torch.float32, device="cuda")
    logits = torch.full((B, WIDE.vocab), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(river.RiverError) as ei:
        river.rl_lm_head_static(m.handle, h, B, logits, None, None, stream)
    assert ei.value.status == river.RL_ERR_UNSUPPORTED
    assert "shared memory" in str(ei.value)
    stream.synchronize()
    assert bool((logits == 7.0).all()), "a rejected call must enqueue nothing"


def test_static_lm_head_rejects_sizes_beyond_its_limit(river, model, stream):
    h = torch.zeros((9, S.d_model), dtype=torch.float32, device="cuda")
    logits = torch.full((9, S.vocab), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(river.RiverError) as ei:
        river.rl_lm_head_static(model.handle, h, 9, logits, None, None, stream)
    assert ei.value.status == river.RL_ERR_UNSUPPORTED
    assert "batch" in str(ei.value)
    stream.synchronize()
    assert bool((logits == 7.0).all()), "a rejected call must enqueue nothing"
