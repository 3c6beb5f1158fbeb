"""HQQ exit river on the GPU against the oracle (River-LLM explainer, section
六: HQQ, which needs no calibration data, is the exit layers' quantizer).

* every stored byte (packed codes, fp16 scales and zeros) of the tiny
  model's exit river equals the oracle's HQQ result, including the ragged
  last group of the 688-input down projection;
* at the Llama-3.2-1B shape, sampled rows of layer 1's query and down
  projections equal the oracle's (rows are independent groups);
* with no shrinkage (beta = infinity) the refinement leaves min-max's
  result bit-identical;
* a teacher-forced decode sequence on the HQQ exit river matches the oracle
  built with the same quantizer;
* bad settings are rejected before anything is enqueued.
"""
import numpy as np
import pytest

import synth
from oracle.model import OracleModel, Policy as OPolicy
from oracle.quant import quantize_linear_hqq
from tests.harness import check_step, to_cuda

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TINY = synth.TINY


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


def _views(river, m, l, i):
    qt, st, zt = m.exit_layer_view(l, i)
    return (qt.cpu().numpy().view(np.uint32), st.cpu().numpy().view(np.uint16),
            zt.cpu().numpy().view(np.uint16))


@pytest.fixture(scope="module")
def tiny_hqq(river, stream):
    w = synth.gen_weights(TINY, seed=0, device="cpu", gains="random")
    with torch.cuda.stream(stream):
        m = river.Model(TINY, to_cuda(w), stream)
        m.quantize_exit_layers(stream, method="hqq")
    stream.synchronize()
    om = OracleModel(TINY, synth.weights_to_numpy(w))
    om.quantize_exit_layers(method="hqq")
    return m, om


def test_hqq_quantizer_is_bit_exact(river, tiny_hqq):
    m, om = tiny_hqq
    changed = 0
    for l in range(TINY.n_layers):
        for i, name in enumerate(river.LINEAR_NAMES):
            q, s, z = _views(river, m, l, i)
            q_ref, s_ref, z_ref = om.quant[l][name]
            assert np.array_equal(q, q_ref), (l, name)
            assert np.array_equal(s, s_ref.view(np.uint16)), (l, name)
            assert np.array_equal(z, z_ref.view(np.uint16)), (l, name)
            changed += 1
    assert changed == 7 * TINY.n_layers


def test_hqq_rows_at_the_1b_shape(river, stream):
    S = synth.LLAMA_1B
    S1 = synth.scaled(S, n_layers=1, name="llama-3.2-1b, one layer")
    w = synth.gen_weights(S1, seed=0, device="cuda", gains="ones")
    with torch.cuda.stream(stream):
        m = river.Model(S1, w, stream)
        m.quantize_exit_layers(stream, method="hqq")
    stream.synchronize()
    for i, name in ((river.RL_WQ, "wq"), (river.RL_WD, "wd")):
        q, s, z = _views(river, m, 0, i)
        rows = slice(0, 96)   # independent rows: a sample the oracle finishes in seconds
        wn = w["layers"][0][name][rows].float().cpu().numpy()
        q_ref, s_ref, z_ref = quantize_linear_hqq(wn, S.group_size)
        assert np.array_equal(q[rows], q_ref), name
        assert np.array_equal(s[rows], s_ref.view(np.uint16)), name
        assert np.array_equal(z[rows], z_ref.view(np.uint16)), name
    del m, w
    torch.cuda.empty_cache()


def test_no_shrinkage_leaves_min_max_unchanged(river, stream):
    w = synth.gen_weights(TINY, seed=0, device="cpu", gains="random")
    wd = to_cuda(w)
    with torch.cuda.stream(stream):
        a = river.Model(TINY, wd, stream)
        a.quantize_exit_layers(stream)
        b = river.Model(TINY, wd, stream)
        river.rl_quantize_exit_layers_hqq(b.handle, 20, 0.7, float("inf"), 1.01, stream)
    stream.synchronize()
    for l in range(TINY.n_layers):
        for i in range(7):
            for x, y in zip(_views(river, a, l, i), _views(river, b, l, i)):
                assert np.array_equal(x, y)


def test_decode_on_the_hqq_exit_river_matches_oracle(river, tiny_hqq, stream):
    from oracle.model import KVState
    m, om = tiny_hqq
    S = TINY
    sched = [2, 0, 1, 3, 4, 2, 1, 0]
    kv = m.kv_cache_alloc(1, 64)
    st = KVState(S, 1, 64)
    toks = synth.gen_tokens(S.vocab, (1, 24), seed=1)
    d_sched = torch.tensor(sched, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        out = river.prefill(m, kv, torch.from_numpy(toks).cuda(), river.Policy.tau_(1.01),
                            stream=stream)
        kv.sync(stream)
        ref = om.prefill(toks, st, OPolicy.tau_(1.01))
        check_step(out, ref, None, 1, "prefill")
        nxt = ref.logits.argmax(-1).astype(np.int32)
        for i, e in enumerate(sched):
            out = river.decode_step(m, kv, torch.from_numpy(nxt.copy()).cuda(),
                                    river.Policy.forced(d_sched), stream=stream)
            kv.sync(stream)
            ref = om.decode_step(nxt, st, OPolicy.forced(e))
            assert int(out["exit_layer"].item()) == e
            check_step(out, ref, None, 1, f"decode step {i} (exit layer {e})")
            nxt = ref.logits.argmax(-1).astype(np.int32)


def test_bad_settings_are_rejected(river, stream):
    w = synth.gen_weights(TINY, seed=0, device="cpu", gains="ones")
    with torch.cuda.stream(stream):
        m = river.Model(TINY, to_cuda(w), stream)
    for args in ((-1, 0.7, 10.0, 1.01), (20, 0.0, 10.0, 1.01), (20, 0.7, 0.0, 1.01),
                 (20, 0.7, 10.0, 0.5), (20, float("nan"), 10.0, 1.01)):
        with pytest.raises(river.RiverError) as ei:
            river.rl_quantize_exit_layers_hqq(m.handle, *args, stream)
        assert ei.value.status == river.RL_ERR_INVALID_ARG
    river.rl_quantize_exit_layers_hqq(m.handle, 20, 0.7, 10.0, 1.01, stream)
    with pytest.raises(river.RiverError) as ei:
        river.rl_quantize_exit_layers_hqq(m.handle, 20, 0.7, 10.0, 1.01, stream)
    assert ei.value.status == river.RL_ERR_STATE
