"""rl_exit_kv_cosine (exit-vs-backbone K/V similarity, River-LLM explainer
section 三) against the oracle's, on the tiny model (every layer, three
sequences) and on one layer of the Llama-3.2-1B shape."""
import numpy as np
import pytest

import synth
from oracle.model import OracleModel
from tests.harness import to_cuda

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


@pytest.mark.parametrize("shape,B", [(synth.TINY, 3),
                                     (synth.scaled(synth.LLAMA_1B, n_layers=1, name="1b-one-layer"), 2)])
def test_exit_kv_cosine_matches_oracle(river, shape, B):
    stream = torch.cuda.Stream()
    w = synth.gen_weights(shape, seed=0, device="cpu", gains="random")
    with torch.cuda.stream(stream):
        m = river.Model(shape, to_cuda(w), stream)
        m.quantize_exit_layers(stream)
    stream.synchronize()
    om = OracleModel(shape, synth.weights_to_numpy(w))
    om.quantize_exit_layers()
    rng = np.random.default_rng(9)
    h = rng.standard_normal((B, shape.d_model)).astype(np.float32)
    for l in range(shape.n_layers):
        with torch.cuda.stream(stream):
            got = m.exit_kv_cosine(l, torch.from_numpy(h).cuda(), stream)
        stream.synchronize()
        ref = om.exit_kv_cosine(l, h, pos=0)
        g = got.cpu().numpy()
        assert g.shape == (B, 2, shape.n_kv_heads)
        assert np.abs(g - ref).max() < 1e-4, (l, g, ref)
        assert np.all(g < 1.0) and np.all(g > 0.9)
    with pytest.raises(river.RiverError):
        river.rl_exit_kv_cosine(m.handle, shape.n_layers, torch.zeros((1, shape.d_model), device="cuda"),
                                1, torch.zeros((1, 2, shape.n_kv_heads), device="cuda"), stream)
