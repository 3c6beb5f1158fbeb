"""Parity at the full Llama-3.2-1B and Llama-3.1-8B shapes, batch 1, in the
launch configuration bench.py times (the persistent decode-step kernel).

The oracle cannot run these models end to end in seconds, so it recomputes
sampled outputs one by one from the GPU's own inputs (River-LLM explainer,
sections 三 and 四): for a decode step under a forced exit layer e, the
layers 1, e (last backbone layer), e + 1 (first exit layer, W4 weights
quantized by the oracle's own quantizer) and L get, from the GPU, the
residual entering the layer and the K/V history of earlier positions; the
oracle's layer output is compared with the GPU's residual leaving it, and
the oracle's K/V for this position with the slot the GPU wrote.  The final
RMSNorm + LM head is recomputed from the GPU's last residual and compared
with the GPU's logits and greedy token.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle.model import KVState, OracleModel, rmsnorm
from oracle.quant import dequantize_linear, quantize_linear
from tests.harness import LOGIT_TOL, cos_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GAP = 0.1          # greedy tokens compared where the oracle's top-1/top-2 gap exceeds this
HIDDEN_COS = 0.999
LAYERS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


@pytest.fixture(scope="module")
def river():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    import early_exit_decoding_gb300 as r
    return r


def _f32(t):
    return t.detach().to("cpu", torch.float32).numpy()


def _layer_oracle(S, lw_gpu, exit_layer: bool):
    """A one-layer oracle holding layer weights copied from the GPU model's
    inputs (bf16 -> fp32, exact); W4 copies made by the oracle's quantizer."""
    lw = {k: _f32(v) for k, v in lw_gpu.items()}
    S1 = dataclasses.replace(S, n_layers=1)
    w = {"embed": np.zeros((1, S.d_model), np.float32), "lm_head": np.zeros((1, S.d_model), np.float32),
         "g_final": np.ones(S.d_model, np.float32), "layers": [lw]}
    om = OracleModel(S1, w)
    W = om.backbone[0]
    if exit_layer:
        W = {}
        for name in LAYERS:
            qw, s, z = quantize_linear(lw[name], S.group_size)
            W[name] = dequantize_linear(qw, s, z, lw[name].shape[1], S.group_size)
    return om, W


@pytest.mark.parametrize("name,prompt", [("llama-3.2-1b", 512), ("llama-3.1-8b", 2048)])
def test_full_size_sampled_layers_and_logits(river, name, prompt):
    S = synth.SHAPES[name]
    L = S.n_layers
    e = L // 2
    stream = torch.cuda.Stream()
    w = synth.gen_weights(S, seed=0, device="cuda", gains="random")
    with torch.cuda.stream(stream):
        m = river.Model(S, w, stream)
        m.quantize_exit_layers(stream)
    stream.synchronize()
    kv = m.kv_cache_alloc(1, prompt + 8)
    assert kv.decode_path(1) == 1, "batch 1 must run the persistent step kernel"
    tr = torch.zeros((L + 1, 1, S.d_model), dtype=torch.float32, device="cuda")
    toks = torch.from_numpy(synth.gen_tokens(S.vocab, (1, prompt), seed=1)).cuda()
    sched = torch.tensor([e], dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        river.prefill(m, kv, toks, river.Policy.tau_(1.01), stream=stream)
        nxt = torch.from_numpy(synth.gen_tokens(S.vocab, (1,), seed=4)).cuda()
        river.decode_step(m, kv, nxt, river.Policy.forced(sched), stream=stream)   # graph capture
        kv.set_trace(tr)
        out = river.decode_step(m, kv, nxt, river.Policy.forced(sched), stream=stream)
        kv.sync(stream)
    kv.set_trace(None)
    pos = prompt + 1                      # this step's slot
    assert int(out["exit_layer"].item()) == e
    hid = _f32(tr)[:, 0]                  # [L+1][d]

    for l in sorted({1, e, e + 1, L}):    # 1-based layer index
        om, W = _layer_oracle(S, w["layers"][l - 1], exit_layer=l > e)
        st = KVState(om.shape, 1, pos + 1)
        kc, vc = kv.view(l - 1)
        st.K[0][0, :, :pos] = _f32(kc[0, :, :pos])
        st.V[0][0, :, :pos] = _f32(vc[0, :, :pos])
        h_out = om.layer(0, W, hid[l - 1][None, None, :], st, pos)[0, 0]
        c = float(cos_rows(h_out[None], hid[l][None])[0])
        d = float(np.abs(h_out - hid[l]).max())
        scale = float(np.abs(h_out).max())
        assert c >= HIDDEN_COS, f"{name} layer {l}: cos {c:.6f}"
        assert d <= 2e-2 * max(1.0, scale), f"{name} layer {l}: max |dh| {d:.4g} (|h| {scale:.3g})"
        # the K/V slot written by this step (bf16 on the GPU)
        k_gpu = _f32(kc[0, :, pos])
        v_gpu = _f32(vc[0, :, pos])
        for ref, got, what in ((st.K[0][0, :, pos], k_gpu, "K"), (st.V[0][0, :, pos], v_gpu, "V")):
            err = np.abs(ref - got).max()
            assert err <= 2e-2 * max(1.0, float(np.abs(ref).max())), f"{name} layer {l} {what} slot: {err:.4g}"

    # final RMSNorm + LM head on the GPU's last residual
    lm = _f32(w["lm_head"])
    g = _f32(w["g_final"])
    logits = (rmsnorm(hid[L][None], g, S.rms_eps) @ lm.T)[0]
    got = _f32(out["logits"])[0]
    assert np.abs(logits - got).max() <= LOGIT_TOL, f"{name}: max |dlogit| {np.abs(logits - got).max():.4g}"
    top = np.sort(logits)[-2:]
    if top[1] - top[0] > GAP:
        assert int(out["next_token"][0].item()) == int(np.argmax(logits))
    del m, kv, w
    torch.cuda.empty_cache()
