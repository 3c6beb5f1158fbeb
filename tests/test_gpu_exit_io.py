"""rl_save_exit_layers / rl_load_exit_layers: an exit river written in the
published packing and read back into a fresh model of the same weights is
bit-identical (every qweight / scale / zero word), decodes exactly like the
model that quantized it, and matches the oracle's exit river (River-LLM
explainer, section 三: the exit layers are a fixed W4 copy of each layer).
Bad files are refused without touching the model."""
import numpy as np
import pytest

import synth
from oracle.model import Policy as OPolicy
from tests.harness import build_pair, to_cuda
from tests.test_gpu_parity import _run_sequence

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


def _fresh(river, S, seed, stream):
    w = synth.gen_weights(S, seed=seed, device="cpu", gains="random")
    with torch.cuda.stream(stream):
        return river.Model(S, to_cuda(w), stream)


def _forced(river, sched):
    d_pre = torch.tensor([sched[0]], dtype=torch.int32, device="cuda")
    d_sched = torch.tensor(sched[1:], dtype=torch.int32, device="cuda")
    pol = [(river.Policy.forced(d_pre), OPolicy.forced(sched[0]))]
    pol += [(river.Policy.forced(d_sched), OPolicy.forced(e)) for e in sched[1:]]
    return pol


def test_saved_exit_river_loads_bit_identical(river, stream, tmp_path):
    with torch.cuda.stream(stream):
        ma, om, _ = build_pair(TINY, seed=0, gains="random", stream=stream)
    path = tmp_path / "exit.rlw4"
    ma.save_exit_layers(path)
    mb = _fresh(river, TINY, 0, stream)
    with pytest.raises(river.RiverError) as e:  # nothing to save before the river is built
        mb.save_exit_layers(tmp_path / "none.rlw4")
    assert e.value.status == river.RL_ERR_STATE
    mb.load_exit_layers(path, stream)
    for l in range(TINY.n_layers):
        for i in range(7):
            for ta, tb in zip(ma.exit_layer_view(l, i), mb.exit_layer_view(l, i)):
                assert torch.equal(ta.view(torch.int16) if ta.dtype == torch.float16 else ta,
                                   tb.view(torch.int16) if tb.dtype == torch.float16 else tb), (l, i)
    # the loaded river decodes like the quantized one (all layers on W4, then mixed)
    sched = [0, 0, 2, 1]
    ra, _ = _run_sequence(river, ma, om, stream, _forced(river, sched), B=2, prompt=10, steps=3, seed=91)
    rb, _ = _run_sequence(river, mb, om, stream, _forced(river, sched), B=2, prompt=10, steps=3, seed=91)
    for (oa, _), (ob, _) in zip(ra, rb):
        assert torch.equal(oa["logits"], ob["logits"])
        assert torch.equal(oa["next_token"], ob["next_token"])
    with pytest.raises(river.RiverError) as e:  # built once
        mb.load_exit_layers(path, stream)
    assert e.value.status == river.RL_ERR_STATE


def test_bad_files_are_refused_and_leave_the_model_usable(river, stream, tmp_path):
    S3 = synth.scaled(TINY, n_layers=3)
    with torch.cuda.stream(stream):
        m3, _, _ = build_pair(S3, seed=2, gains="random", stream=stream)
    other = tmp_path / "three_layers.rlw4"
    m3.save_exit_layers(other)
    m = _fresh(river, TINY, 0, stream)
    with pytest.raises(river.RiverError) as e:  # another shape
        m.load_exit_layers(other, stream)
    assert e.value.status == river.RL_ERR_INVALID_ARG
    with torch.cuda.stream(stream):
        ma, _, _ = build_pair(TINY, seed=0, gains="random", stream=stream)
    good = tmp_path / "exit.rlw4"
    ma.save_exit_layers(good)
    data = good.read_bytes()
    for bad_bytes in (data[:-2], data + b"\0", b"XXXXXXXX" + data[8:]):
        bad = tmp_path / "bad.rlw4"
        bad.write_bytes(bad_bytes)
        with pytest.raises(river.RiverError) as e:
            m.load_exit_layers(bad, stream)
        assert e.value.status == river.RL_ERR_INVALID_ARG
    with pytest.raises(river.RiverError) as e:
        m.load_exit_layers(tmp_path / "missing.rlw4", stream)
    assert e.value.status == river.RL_ERR_INVALID_ARG
    m.load_exit_layers(good, stream)  # still loads after the refusals
    q0, _, _ = m.exit_layer_view(0, 0)
    q1, _, _ = ma.exit_layer_view(0, 0)
    assert torch.equal(q0, q1)
    assert np.array_equal(q0.cpu().numpy(), q1.cpu().numpy())
