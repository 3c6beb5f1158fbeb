"""The streaming decode attention (the decode path for batches beyond the
persistent step kernel) against the oracle over long contexts: chunks of up
to 128 positions staged by 64-row and 16-row TMA boxes, a ragged last chunk,
empty trailing chunks, and every query-heads-per-KV-head ratio it serves (1,
2 and 4) at head dims 64 and 128 (River-LLM explainer, section 三: every
layer reads the backbone's own K/V slots, which the exit layers also write).
"""
import numpy as np
import pytest

import synth
from tests.harness import build_pair
from tests.test_gpu_parity import _run_sequence
from tests.test_gpu_tc_gemm import _forced

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


# (d_model, q heads, KV heads, batch, prompt): with 152 SMs the chunk lengths
# come out at 128 (two 64-row boxes; last chunk 61-63 rows = four 16-row
# boxes), 80 (one 64-row + one 16-row box; last chunk 41-43 rows) and 32 (two
# 16-row boxes; the last of three chunks empty).
CASES = [
    pytest.param(256, 4, 2, 40, 700, id="hd64-rep2-chunk128"),
    pytest.param(512, 4, 1, 24, 1000, id="hd128-rep4-chunk80"),
    pytest.param(256, 4, 4, 12, 60, id="hd64-rep1-chunk32"),
]


@pytest.mark.parametrize("d_model,hq,hkv,B,T", CASES)
def test_streaming_attention_long_contexts(river, stream, d_model, hq, hkv, B, T):
    S = synth.scaled(TINY, d_model=d_model, n_q_heads=hq, n_kv_heads=hkv, n_layers=3, vocab=512)
    assert S.d_model // S.n_q_heads in (64, 128)
    with torch.cuda.stream(stream):
        m, om, _ = build_pair(S, seed=11, gains="random", stream=stream)
    sched = [3, 3, 1, 0]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=B, prompt=T,
                           steps=len(sched) - 1, seed=70 + B, path="generic", max_seq=T + 20)
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched
    # the greedy token is the first maximum of the GPU's own logits, every row
    for o, _ in res[1:]:
        lg = o["logits"].float().cpu().numpy()
        assert np.array_equal(o["next_token"].cpu().numpy(), lg.argmax(-1))
