"""Tensor-core causal prompt attention against the oracle (River-LLM
explainer, section 五: one pass over the prompt writes every layer's cache).

Small decoders with each supported grouping (1, 4 and 8 query heads per KV
head) and head dims 64 / 128 run a prefill of prompts whose lengths leave
ragged query and key blocks; the oracle runs the same prefill.  Compared:
the logits and every layer's residual of the last position, and the whole
K/V cache of the second layer (its inputs are the first layer's attention
output at every prompt position, so a wrong attention row anywhere shows).
"""
import numpy as np
import pytest

import synth
from oracle.model import KVState, Policy as OPolicy
from tests.harness import build_pair, check_step, cos_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def river():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_gb300 as r
    return r


SHAPES = [
    synth.scaled(synth.TINY, name="pf-rep4-hd128", n_layers=2, d_model=512, n_q_heads=8, n_kv_heads=2,
                 head_dim=128, ffn_dim=256, vocab=512),
    synth.scaled(synth.TINY, name="pf-rep1-hd64", n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=4,
                 head_dim=64, ffn_dim=256, vocab=512),
    synth.scaled(synth.TINY, name="pf-rep8-hd64", n_layers=2, d_model=512, n_q_heads=8, n_kv_heads=1,
                 head_dim=64, ffn_dim=256, vocab=512),
]


@pytest.mark.parametrize("S", SHAPES, ids=[s.name for s in SHAPES])
@pytest.mark.parametrize("B,T", [(1, 77), (2, 300)])
def test_prefill_attention_matches_oracle(river, S, B, T):
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        m, om, _ = build_pair(S, seed=0, gains="random", stream=stream)
    stream.synchronize()
    kv = m.kv_cache_alloc(B, T + 4)
    tr = torch.zeros((S.n_layers + 1, B, S.d_model), dtype=torch.float32, device="cuda")
    kv.set_trace(tr)
    toks = synth.gen_tokens(S.vocab, (B, T), seed=7)
    with torch.cuda.stream(stream):
        out = river.prefill(m, kv, torch.from_numpy(toks).cuda(), river.Policy.tau_(1.01), stream=stream)
        kv.sync(stream)
    st = KVState(S, B, T + 4)
    ref = om.prefill(toks, st, OPolicy.tau_(1.01))
    check_step(out, ref, tr, B, f"{S.name} prefill B={B} T={T}")
    k1, v1 = kv.view(1)
    for name, gpu, ora in (("K", k1, st.K[1]), ("V", v1, st.V[1])):
        g = gpu[:B, :, :T].float().cpu().numpy().reshape(-1, S.head_dim)
        o = ora[:, :, :T].reshape(-1, S.head_dim)
        c = cos_rows(g, o)
        assert c.min() > 0.999, f"{name} cache of layer 2: min row cosine {c.min():.5f}"
        err = np.abs(g - o).max()
        assert err <= 2e-2 * max(1.0, float(np.abs(o).max())), f"{name} cache of layer 2: {err:.4g}"
