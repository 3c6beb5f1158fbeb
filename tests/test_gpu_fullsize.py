"""Parity at the full Llama-3.2-1B and Llama-3.1-8B shapes, in the launch
configurations bench.py times: batch 1 on the persistent decode-step kernel,
and the batch workloads (1B at batch 32, 8B at batch 64) on the generic path
(tensor-core GEMMs with split K and W4 dequantised in shared memory, the
streaming decode attention), under a forced exit layer and under tau.

The oracle cannot run these models end to end in seconds, so it recomputes
sampled outputs one by one from the GPU's own inputs (River-LLM explainer,
sections 三 and 四): for a decode step with exit layer e, the layers 1, e
(last backbone layer), e + 1 (first exit layer, W4 weights quantized by the
oracle's own quantizer) and L get, from the GPU, the residual entering the
layer and the K/V history of earlier positions; the oracle's layer output is
compared with the GPU's residual leaving it, and the oracle's K/V for this
position with the slot the GPU wrote.  The final RMSNorm + LM head is
recomputed from the GPU's last residual of every sequence and compared with
the GPU's logits and greedy tokens.  Under tau, the exit layer must be the
first layer whose batch-minimum cosine between the GPU's own residuals
entering and leaving it exceeds tau, unless a deciding cosine lies within
1e-3 of tau.

The batch workloads fill the K/V cache of the prompt positions with N(0, 1)
values (as bench.py does for the 8B batch-64 timing); the sampled layers then
read that history from the GPU.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle.model import KVState, OracleModel, rmsnorm
from oracle.quant import dequantize_linear, quantize_linear
from tests.harness import LOGIT_TOL, TAU_BAND, cos_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GAP = 0.1          # greedy tokens compared where the oracle's top-1/top-2 gap exceeds this
HIDDEN_COS = 0.999
LAYERS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
PATH_STEP, PATH_GENERIC = 1, 3


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


class Built:
    """A model on the GPU and the seeded weights it was made from."""

    def __init__(self, river, name):
        self.S = synth.SHAPES[name]
        self.stream = torch.cuda.Stream()
        self.w = synth.gen_weights(self.S, seed=0, device="cuda", gains="random")
        with torch.cuda.stream(self.stream):
            self.m = river.Model(self.S, self.w, self.stream)
            self.m.quantize_exit_layers(self.stream)
        self.stream.synchronize()
        self._layer_cache = {}

    def layer_oracle(self, l, exit_layer):
        """A one-layer oracle holding layer l's weights (bf16 -> fp32, exact);
        W4 copies made by the oracle's own quantizer."""
        key = (l, exit_layer)
        if key not in self._layer_cache:
            S = self.S
            lw = {k: _f32(v) for k, v in self.w["layers"][l - 1].items()}
            S1 = dataclasses.replace(S, n_layers=1)
            w = {"embed": np.zeros((1, S.d_model), np.float32),
                 "lm_head": np.zeros((1, S.d_model), np.float32),
                 "g_final": np.ones(S.d_model, np.float32), "layers": [lw]}
            om = OracleModel(S1, w)
            W = om.backbone[0]
            if exit_layer:
                W = {}
                for name in LAYERS:
                    qw, s, z = quantize_linear(lw[name], S.group_size)
                    W[name] = dequantize_linear(qw, s, z, lw[name].shape[1], S.group_size)
            self._layer_cache = {key: (om, W)}  # one layer's fp32 copy at a time
        return self._layer_cache[key]


@pytest.fixture(scope="module")
def llama1b(river):
    b = Built(river, "llama-3.2-1b")
    yield b
    del b
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def llama8b(river):
    b = Built(river, "llama-3.1-8b")
    yield b
    del b
    torch.cuda.empty_cache()


def _decode(river, bm, B, T, policy, fill, path):
    """One decode step at position T after a prompt of T tokens (a real
    prefill, or N(0, 1) K/V history); returns (outputs, trace [L+1][B][d],
    kv)."""
    S, stream = bm.S, bm.stream
    kv = bm.m.kv_cache_alloc(B, T + 8)
    assert kv.decode_path(B) == path
    tr = torch.zeros((S.n_layers + 1, B, S.d_model), dtype=torch.float32, device="cuda")
    nxt = torch.from_numpy(synth.gen_tokens(S.vocab, (B,), seed=4)).cuda()
    with torch.cuda.stream(stream):
        if fill == "prefill":
            toks = torch.from_numpy(synth.gen_tokens(S.vocab, (B, T), seed=1)).cuda()
            river.prefill(bm.m, kv, toks, river.Policy.tau_(1.01), stream=stream)
            river.decode_step(bm.m, kv, nxt, policy, stream=stream)   # graph capture
            pos = T + 1
        else:
            g = torch.Generator(device="cuda")
            g.manual_seed(3)
            for l in range(S.n_layers):
                k, v = kv.view(l)
                k[:B, :, :T].normal_(generator=g)
                v[:B, :, :T].normal_(generator=g)
            kv.set_position(T, 0, stream)
            pos = T
        kv.set_trace(tr)
        out = river.decode_step(bm.m, kv, nxt, policy, stream=stream)
        kv.sync(stream)
    kv.set_trace(None)
    return out, _f32(tr), kv, pos


def _check_layers(bm, kv, hid, pos, e, sel):
    """Sampled layers 1, e, e + 1, L of sequences `sel` against the oracle."""
    S = bm.S
    L = S.n_layers
    for l in sorted({1, max(e, 1), min(e + 1, L), L}):
        om, W = bm.layer_oracle(l, exit_layer=l > e)
        st = KVState(om.shape, len(sel), pos + 1)
        kc, vc = kv.view(l - 1)
        for i, b in enumerate(sel):
            st.K[0][i, :, :pos] = _f32(kc[b, :, :pos])
            st.V[0][i, :, :pos] = _f32(vc[b, :, :pos])
        h_out = om.layer(0, W, hid[l - 1][sel][:, None, :], st, pos)[:, 0]
        c = cos_rows(h_out, hid[l][sel])
        assert c.min() >= HIDDEN_COS, f"{S.name} layer {l}: cos {c.min():.6f} (seqs {sel})"
        d = np.abs(h_out - hid[l][sel]).max()
        scale = float(np.abs(h_out).max())
        assert d <= 2e-2 * max(1.0, scale), f"{S.name} layer {l}: max |dh| {d:.4g} (|h| {scale:.3g})"
        for i, b in enumerate(sel):   # the K/V slot written by this step (bf16 on the GPU)
            k_gpu = _f32(kc[b, :, pos])
            v_gpu = _f32(vc[b, :, pos])
            for ref, got, what in ((st.K[0][i, :, pos], k_gpu, "K"), (st.V[0][i, :, pos], v_gpu, "V")):
                err = np.abs(ref - got).max()
                assert err <= 2e-2 * max(1.0, float(np.abs(ref).max())), \
                    f"{S.name} layer {l} seq {b} {what} slot: {err:.4g}"


def _check_logits(bm, out, hid, B):
    """Final RMSNorm + LM head of every sequence's last residual."""
    S = bm.S
    lm = _f32(bm.w["lm_head"])
    g = _f32(bm.w["g_final"])
    logits = rmsnorm(hid[S.n_layers][:B], g, S.rms_eps) @ lm.T
    got = _f32(out["logits"])[:B]
    d = np.abs(logits - got).max()
    assert d <= LOGIT_TOL, f"{S.name}: max |dlogit| {d:.4g}"
    srt = np.sort(logits, axis=-1)
    clear = (srt[:, -1] - srt[:, -2]) > GAP
    nt = out["next_token"][:B].cpu().numpy()
    assert np.array_equal(nt[clear], logits.argmax(-1)[clear]), f"{S.name}: greedy tokens"


def _tau_decision(hid, B, L, tau):
    """Exit layer by the rule on the GPU's own residuals: the first l < L whose
    batch-minimum cosine (fp64 here) between the residual entering and leaving
    layer l exceeds tau; L if none.  Also returns the per-layer minima."""
    m = np.array([cos_rows(hid[l - 1][:B], hid[l][:B]).min() for l in range(1, L + 1)])
    e = L
    for l in range(1, L):
        if m[l - 1] > tau:
            e = l
            break
    return e, m


CASES_FORCED = [
    # (model, batch, prompt, K/V history, decode path)
    ("llama1b", 1, 512, "prefill", PATH_STEP),
    ("llama8b", 1, 2048, "prefill", PATH_STEP),
    ("llama1b", 32, 1030, "random", PATH_GENERIC),
    ("llama8b", 64, 4100, "random", PATH_GENERIC),
    # 8 KV heads x 21 chunks of 128 exceed the 152 CTAs: two chunks per CTA
    ("llama8b", 1, 2600, "prefill", PATH_STEP),
]


@pytest.mark.parametrize("which,B,T,fill,path", CASES_FORCED)
def test_full_size_forced_sampled_layers_and_logits(river, request, which, B, T, fill, path):
    bm = request.getfixturevalue(which)
    L = bm.S.n_layers
    e = L // 2
    sched = torch.tensor([e], dtype=torch.int32, device="cuda")
    out, hid, kv, pos = _decode(river, bm, B, T, river.Policy.forced(sched), fill, path)
    assert int(out["exit_layer"].item()) == e
    sel = sorted({0, B // 2, B - 1})
    _check_layers(bm, kv, hid, pos, e, sel)
    _check_logits(bm, out, hid, B)
    del kv
    torch.cuda.empty_cache()


CASES_TAU = [
    ("llama1b", 1, 512, "prefill", PATH_STEP, 0.5),
    ("llama8b", 1, 2048, "prefill", PATH_STEP, 0.5),
    ("llama1b", 32, 1030, "random", PATH_GENERIC, 0.5),
]


@pytest.mark.parametrize("which,B,T,fill,path,tau", CASES_TAU)
def test_full_size_tau_decision_layers_and_logits(river, request, which, B, T, fill, path, tau):
    bm = request.getfixturevalue(which)
    L = bm.S.n_layers
    out, hid, kv, pos = _decode(river, bm, B, T, river.Policy.tau_(tau), fill, path)
    e_gpu = int(out["exit_layer"].item())
    e_ref, m = _tau_decision(hid, B, L, tau)
    # the GPU's reported per-layer batch minima are the cosines of its residuals
    mc = out["min_cos"].cpu().numpy()
    hi = min(e_gpu, L - 1)
    assert np.abs(mc[:hi] - m[:hi]).max() < 1e-4, f"min_cos {mc[:hi]} vs {m[:hi]}"
    if e_gpu != e_ref:
        hi = min(max(e_gpu, e_ref), L - 1)
        assert np.any(np.abs(m[:hi] - tau) <= TAU_BAND), \
            f"{bm.S.name} B={B}: exit layer {e_gpu}, rule on the GPU's residuals gives {e_ref}"
    assert 1 <= e_gpu <= L
    sel = sorted({0, B // 2, B - 1})
    _check_layers(bm, kv, hid, pos, e_gpu, sel)
    _check_logits(bm, out, hid, B)
    del kv
    torch.cuda.empty_cache()
