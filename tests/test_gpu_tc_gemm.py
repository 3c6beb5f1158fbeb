"""The tensor-core GEMM path (tcgen05 + TMA; used from 16 tokens up) against
the oracle: prompts and decode batches whose token counts span several token
tiles with a ragged tail, every token-tile width (32, 64, 128, 256), weight
matrices whose row count is not a multiple of the 128-row tile (the tiny
shape's gate/up: 1376 rows), and prefills whose sequence-level exit puts the
later layers on the W4 exit river (River-LLM explainer, section 五: one exit
decision for the whole prompt; section 三: the exit layers write the
backbone's KV slots).
"""
import numpy as np
import pytest

import synth
from oracle.model import Policy as OPolicy
from tests.harness import build_pair
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


@pytest.fixture(scope="module")
def tiny(river, stream):
    with torch.cuda.stream(stream):
        m, om, w = build_pair(TINY, seed=0, gains="random", stream=stream)
    return m, om, w


def _forced(river, sched):
    """Prefill forced at sched[0] (a one-entry schedule), then one decode
    step per remaining entry."""
    d_pre = torch.tensor([sched[0]], dtype=torch.int32, device="cuda")
    d_sched = torch.tensor(sched[1:], dtype=torch.int32, device="cuda")
    pol = [(river.Policy.forced(d_pre), OPolicy.forced(sched[0]))]
    pol += [(river.Policy.forced(d_sched), OPolicy.forced(e)) for e in sched[1:]]
    return pol


@pytest.mark.parametrize("B", [16, 21, 40])
def test_decode_batches_on_tensor_cores(river, tiny, stream, B):
    """Decode batches of 16 / 21 / 40 sequences run the GEMM with 32- and
    64-token tiles (ragged); exit layers mix in (W4 weights dequantised in
    shared memory for the tensor cores)."""
    m, om, _ = tiny
    L = TINY.n_layers
    sched = [L, L, 0, 2, 1, L]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=B, prompt=9,
                           steps=len(sched) - 1, seed=20 + B, path="generic")
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched


@pytest.mark.parametrize("B", [16, 40])
def test_decode_batches_split_k_and_w4_on_tensor_cores(river, stream, B):
    """A wider model (d_model 1024, FFN 2816: 16 to 44 k-blocks of 64 inputs)
    whose projections at batch 16 / 40 have fewer 128-row tiles than SMs: the
    GEMM splits K across CTAs (partial tiles summed by the tile's last CTA) on
    the bf16 backbone; at batch 40 (one 64-column token tile) every W4
    projection runs on the tensor cores too, dequantised in shared memory and
    split, while at batch 16 the W4 projections (at most 44 tiles) stay on the
    dequantising GEMV."""
    S = synth.scaled(TINY, d_model=1024, n_q_heads=8, n_kv_heads=2, ffn_dim=2816, n_layers=3,
                     vocab=512)
    with torch.cuda.stream(stream):
        m, om, _ = build_pair(S, seed=7, gains="random", stream=stream)
    sched = [3, 3, 0, 1, 2]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=B, prompt=6,
                           steps=len(sched) - 1, seed=60 + B, path="generic")
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched


@pytest.mark.parametrize("tau", [0.3, 0.7])
def test_decode_batch40_tau_decided_on_device(river, tiny, stream, tau):
    """Batch 40 under tau (section 四, batch minimum): the GEMM reads the exit
    layer the previous layer end decided on the device and runs the bf16 or
    the W4 weights accordingly (above 32 tokens every W4 projection is on the
    tensor cores and no group sums are launched)."""
    m, om, _ = tiny
    pol = [(river.Policy.tau_(tau), OPolicy.tau_(tau))] * 4
    _run_sequence(river, m, om, stream, pol, B=40, prompt=9, steps=3, seed=80 + int(10 * tau),
                  path="generic")


@pytest.mark.parametrize("e_pre", [0, 1, 3])
def test_prefill_exit_runs_later_layers_on_w4(river, tiny, stream, e_pre):
    """A forced prefill exit at e: layers <= e on the tensor cores, layers > e
    on the W4 GEMV over all 2 x 40 prompt tokens (two 64-token blocks)."""
    m, om, _ = tiny
    sched = [e_pre, 2, TINY.n_layers]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=2, prompt=40,
                           steps=2, seed=31 + e_pre)
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched


def test_prefill_tau_sequence_level(river, tiny, stream):
    """tau = 0.5 over a 3 x 50 prompt: the batch-and-sequence minimum decides."""
    m, om, _ = tiny
    pol = [(river.Policy.tau_(0.5), OPolicy.tau_(0.5))] * 3
    _run_sequence(river, m, om, stream, pol, B=3, prompt=50, steps=2, seed=41)


@pytest.mark.parametrize("B,T", [(1, 1100), (2, 2048)])
def test_long_prompts_every_tile_width(river, tiny, stream, B, T):
    """1100 tokens (128-token tiles, ragged tail of 76) and 2 x 2048 tokens
    (256-token tiles on gate/up, 64 on QKV, 32 on O and down)."""
    m, om, _ = tiny
    L = TINY.n_layers
    sched = [L, 1, L]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=B, prompt=T,
                           steps=2, seed=50 + T, max_seq=T + 4)
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched


@pytest.mark.parametrize("e_pre", [0, 2])
def test_prompt_long_reduction_split_k(river, stream, e_pre):
    """A prompt projection with a long reduction (FFN 8192: the down
    projection has 128 k-blocks of 64 inputs) and few 128-token tiles splits
    K in two per tile (partial tiles summed by the tile's last CTA): 300
    tokens (a ragged 44-token tail), on the bf16 backbone (e = 2, full depth)
    and on the W4 exit river (e = 0, every layer's down projection W4 on the
    tensor cores)."""
    S = synth.scaled(TINY, d_model=512, n_q_heads=8, n_kv_heads=2, ffn_dim=8192, n_layers=2,
                     vocab=512)
    with torch.cuda.stream(stream):
        m, om, _ = build_pair(S, seed=9, gains="random", stream=stream)
    sched = [e_pre, 1, 2]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=1, prompt=300,
                           steps=2, seed=90 + e_pre, max_seq=320)
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched

