"""GPU parity: the CUDA path (through the C ABI) against the oracle.

River-LLM explainer: section 三 (W4A16 exit layers that share the backbone's
KV slots), 四 (batch-min state-transition similarity vs tau), 五 (one exit
decision for the prompt in prefill, one per generation step).
"""
import numpy as np
import pytest

import synth
from oracle.model import Policy as OPolicy, KVState
from oracle.quant import quantize_linear
from tests.harness import build_pair, check_step, tau_band_ok

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


PATHS = {"step": 1, "fused": 2, "generic": 3}


def _run_sequence(river, m, om, stream, policies, B=1, prompt=32, steps=16, seed=1, trace=True,
                  max_seq=128, path=None):
    """Prefill + decode with teacher forcing on the oracle's greedy tokens.
    ``policies``: (gpu Policy, oracle Policy) for prefill, then per decode step.
    ``path``: force the decode kernels (step / fused / generic)."""
    S = m.shape
    toks = synth.gen_tokens(S.vocab, (B, prompt), seed=seed)
    kv = m.kv_cache_alloc(B, max_seq)
    if path is not None:
        kv.set_decode_path(PATHS[path])
        assert kv.decode_path(B) == PATHS[path], f"path {path} does not fit batch {B}"
    st = KVState(S, B, max_seq)
    tr = None
    if trace:
        tr = torch.zeros((S.n_layers + 1, B, S.d_model), dtype=torch.float32, device="cuda")
        kv.set_trace(tr)
    results = []
    with torch.cuda.stream(stream):
        gp, op = policies[0]
        out = river.prefill(m, kv, torch.from_numpy(toks).cuda(), gp, stream=stream)
        kv.sync(stream)
        ref = om.prefill(toks, st, op)
        assert int(out["exit_layer"].item()) == ref.exit_layer or \
            (op.mode == "tau" and tau_band_ok(ref, op.tau, int(out["exit_layer"].item())))
        if int(out["exit_layer"].item()) == ref.exit_layer:
            check_step(out, ref, tr, B, "prefill")
        results.append((out, ref))
        nxt = ref.logits.argmax(-1).astype(np.int32)
        for i in range(steps):
            gp, op = policies[1 + i]
            p, s_idx = kv.position()
            tin = torch.from_numpy(nxt.copy()).cuda()
            out = river.decode_step(m, kv, tin, gp, stream=stream)
            kv.sync(stream)
            ref = om.decode_step(nxt, st, op)
            e = int(out["exit_layer"].item())
            if e != ref.exit_layer:
                assert op.mode == "tau" and tau_band_ok(ref, op.tau, e), \
                    f"step {i}: exit layer {e} vs oracle {ref.exit_layer}, min_cos {ref.min_cos}"
                # teacher-force the oracle's decision: the step rewrites the same slots
                kv.set_position(p, 0, stream)
                sched = torch.tensor([ref.exit_layer], dtype=torch.int32, device="cuda")
                out = river.decode_step(m, kv, tin, river.Policy.forced(sched), stream=stream)
                kv.sync(stream)
                kv.set_position(p + 1, s_idx + 1, stream)
            check_step(out, ref, tr, B, f"decode step {i}")
            results.append((out, ref))
            nxt = ref.logits.argmax(-1).astype(np.int32)
    kv.set_trace(None)
    return results, kv


def _forced(river, sched):
    """(gpu, oracle) policies for prefill + decode steps: prefill at sched[0],
    decode step i at sched[1 + i]."""
    d = torch.tensor(sched[1:], dtype=torch.int32, device="cuda")
    return [(river.Policy.forced(torch.tensor(sched[:1], dtype=torch.int32, device="cuda")),
             OPolicy.forced(sched[0]))] + \
        [(river.Policy.forced(d), OPolicy.forced(e)) for e in sched[1:]]


def test_quantizer_is_bit_exact(river, tiny):
    m, om, w = tiny
    for l in range(TINY.n_layers):
        for i, name in enumerate(river.LINEAR_NAMES):
            qt, st, zt = m.exit_layer_view(l, i)
            q_ref, s_ref, z_ref = om.quant[l][name]
            assert np.array_equal(qt.cpu().numpy().view(np.uint32), q_ref), (l, name)
            assert np.array_equal(st.cpu().numpy().view(np.uint16), s_ref.view(np.uint16)), (l, name)
            assert np.array_equal(zt.cpu().numpy().view(np.uint16), z_ref.view(np.uint16)), (l, name)


@pytest.mark.parametrize("path", ["step", "fused", "generic"])
def test_full_depth_matches_oracle(river, tiny, stream, path):
    """tau = 1.01 > 1 >= cos: never exits; prompt 32, 16 greedy steps."""
    m, om, _ = tiny
    pol = [(river.Policy.tau_(1.01), OPolicy.tau_(1.01))] * 17
    res, _ = _run_sequence(river, m, om, stream, pol, path=path)
    assert all(int(o["exit_layer"].item()) == TINY.n_layers for o, _ in res)


@pytest.mark.parametrize("path", ["step", "fused", "generic"])
def test_tau_half_matches_oracle(river, tiny, stream, path):
    m, om, _ = tiny
    pol = [(river.Policy.tau_(0.5), OPolicy.tau_(0.5))] * 17
    _run_sequence(river, m, om, stream, pol, path=path)


@pytest.mark.parametrize("path", ["step", "fused", "generic"])
def test_forced_schedule_exit_layers_bit_exact(river, tiny, stream, path):
    m, om, _ = tiny
    L = TINY.n_layers
    sched = [L, 1, 0, 2, 3, 4, 1, 1, 2, 0, 4, 3, 2, 1, 0, 1, 2]
    d_sched = torch.tensor(sched[1:], dtype=torch.int32, device="cuda")
    d_pre = torch.tensor([sched[0]], dtype=torch.int32, device="cuda")
    pol = [(river.Policy.forced(d_pre), OPolicy.forced(sched[0]))]
    pol += [(river.Policy.forced(d_sched), OPolicy.forced(e)) for e in sched[1:]]
    res, _ = _run_sequence(river, m, om, stream, pol, path=path)
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched


@pytest.mark.parametrize("path", ["step", "fused", "generic"])
def test_batch_min_rule_batch3(river, tiny, stream, path):
    """Batch of 3: the minimum over the batch decides (section 四)."""
    m, om, _ = tiny
    for tau in (0.3, 0.5, 0.7):
        pol = [(river.Policy.tau_(tau), OPolicy.tau_(tau))] * 7
        _run_sequence(river, m, om, stream, pol, B=3, prompt=12, steps=6, seed=4, path=path)


def test_batch_forced_and_ragged_shapes(river, stream):
    """B = 5 and 13 (several n-tiles, ragged), forced exits, prompt 7."""
    S = synth.scaled(TINY, n_layers=3)
    with torch.cuda.stream(stream):
        m, om, _ = build_pair(S, seed=3, stream=stream)
    for B in (5, 13):
        sched = [3, 0, 1, 2, 3]
        d_pre = torch.tensor([sched[0]], dtype=torch.int32, device="cuda")
        d_sched = torch.tensor(sched[1:], dtype=torch.int32, device="cuda")
        pol = [(river.Policy.forced(d_pre), OPolicy.forced(sched[0]))]
        pol += [(river.Policy.forced(d_sched), OPolicy.forced(e)) for e in sched[1:]]
        _run_sequence(river, m, om, stream, pol, B=B, prompt=7, steps=4, seed=5 + B)


@pytest.mark.parametrize("B,prompt", [(8, 1300), (4, 2500)])
def test_step_attention_two_chunks_per_cta(river, tiny, stream, B, prompt):
    """More chunks of 128 positions than CTAs (8 x 2 KV heads x 11 at context
    ~1300; 4 x 2 x 20 at ~2500), so the step kernel's CTAs take two
    consecutive attention chunks each: at batch 8 an odd chunk count per head
    group (every chunk's partial merged by the last CTA of its group), at
    batch 4 an even one (a CTA's two chunks of one group folded into one
    partial in shared memory first)."""
    m, om, _ = tiny
    L = TINY.n_layers
    sched = [L, 2, 0, L]
    _run_sequence(river, m, om, stream, _forced(river, sched), B=B, prompt=prompt, steps=3,
                  seed=61, max_seq=prompt + 10, path="step")


# (d_model, q heads, KV heads, batch, prompt, cache positions) for the step
# kernel's attention phase, one 128-position chunk or fewer per CTA.
STEP_ATTN_CASES = [
    # 8 chunks of 113-114 positions per head group (more chunks than ring
    # slots in one CTA's ring over the step), the step's own row in the last
    pytest.param(256, 4, 2, 1, 900, 1000, id="hd64-rep2-8chunks"),
    # 16 head groups of a single ragged chunk
    pytest.param(256, 4, 2, 8, 40, 128, id="hd64-rep2-b8"),
    # head_dim 128 (K and V in separate slots), four query heads per KV head
    pytest.param(512, 4, 1, 2, 400, 500, id="hd128-rep4"),
    pytest.param(512, 4, 2, 1, 300, 700, id="hd128-rep2"),
]


@pytest.mark.parametrize("d_model,hq,hkv,B,T,cap", STEP_ATTN_CASES)
def test_step_attention_shapes(river, stream, d_model, hq, hkv, B, T, cap):
    """The step kernel's attention at more head dims, GQA ratios, batches and
    chunk counts (section 三: every layer reads the backbone's K/V slots),
    forced exits so that both weight paths write and read them."""
    S = synth.scaled(TINY, d_model=d_model, n_q_heads=hq, n_kv_heads=hkv, n_layers=3, vocab=512)
    with torch.cuda.stream(stream):
        m, om, _ = build_pair(S, seed=13, gains="random", stream=stream)
    sched = [3, 1, 3, 0]
    res, _ = _run_sequence(river, m, om, stream, _forced(river, sched), B=B, prompt=T, steps=3,
                           seed=80 + B, max_seq=cap, path="step")
    assert [int(o["exit_layer"].item()) for o, _ in res] == sched


def test_exit_writes_slot_p_of_every_layer(river, tiny, stream):
    """Exit layers write their K/V into the backbone's own slot p (section 三);
    nothing else in any layer's cache changes."""
    m, om, _ = tiny
    S = TINY
    kv = m.kv_cache_alloc(2, 64)
    toks = torch.from_numpy(synth.gen_tokens(S.vocab, (2, 10), seed=6)).cuda()
    with torch.cuda.stream(stream):
        river.prefill(m, kv, toks[:, :6].contiguous(), river.Policy.tau_(1.01), stream=stream)
        for e in (0, 1, S.n_layers):
            stream.synchronize()
            before = [tuple(t.clone() for t in kv.view(l)) for l in range(S.n_layers)]
            p, _ = kv.position()
            sched = torch.tensor([e], dtype=torch.int32, device="cuda")
            kv.set_position(p, 0, stream)
            out = river.decode_step(m, kv, toks[:, p].contiguous(), river.Policy.forced(sched),
                                    stream=stream)
            kv.sync(stream)
            assert int(out["exit_layer"].item()) == e
            for l in range(S.n_layers):
                for new, old in zip(kv.view(l), before[l]):
                    changed = (new[:2] != old[:2]).any(dim=3).any(dim=1).any(dim=0)
                    idx = torch.nonzero(changed).flatten().tolist()
                    assert idx == [p], (e, l, idx)
                    assert not (new[2:] != old[2:]).any() if new.shape[0] > 2 else True


def test_grid_aligned_exit_river_equals_backbone(river, stream):
    """Weights on the W4 grid (each group holds nibbles 0 and 15, power-of-two
    scale, integer zero) quantize exactly, so the exit river must reproduce the
    backbone: the W4 kernels are then checked against the bf16 ones."""
    S = synth.scaled(TINY, n_layers=2, vocab=512)
    w = synth.gen_weights(S, seed=9, device="cpu", gains="random")
    rng = np.random.default_rng(0)
    for lw in w["layers"]:
        for name in synth.LINEARS:
            N, K = lw[name].shape
            Gn = (K + 127) // 128
            q = rng.integers(0, 16, size=(N, K))
            for g in range(Gn):
                q[:, g * 128] = 0
                q[:, min(g * 128 + 1, K - 1)] = 15
            z = np.repeat(rng.integers(0, 16, size=(N, Gn)), 128, axis=1)[:, :K]
            lw[name] = torch.from_numpy(((q - z) * 2.0 ** -7).astype(np.float32)).to(torch.bfloat16)
    import early_exit_decoding_gb300 as r
    from tests.harness import to_cuda
    m = r.Model(S, to_cuda(w), stream)
    m.quantize_exit_layers(stream)
    toks = torch.from_numpy(synth.gen_tokens(S.vocab, (2, 9), seed=7)).cuda()
    outs, hid = [], []
    for e in (S.n_layers, 0):
        kv = m.kv_cache_alloc(2, 32)
        tr = torch.zeros((S.n_layers + 1, 2, S.d_model), dtype=torch.float32, device="cuda")
        kv.set_trace(tr)
        sched = torch.tensor([e], dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            r.prefill(m, kv, toks[:, :8].contiguous(), r.Policy.forced(sched), stream=stream)
            o = r.decode_step(m, kv, toks[:, 8].contiguous(), r.Policy.forced(sched), stream=stream)
            kv.sync(stream)
        outs.append(o["logits"].cpu().numpy())
        hid.append(tr.cpu().numpy())
    # Same weight values on both paths: only fp32 summation order differs,
    # which can flip a bf16 activation rounding by one ulp (2^-8 relative).
    scale = np.abs(outs[0]).max()
    assert np.abs(outs[0] - outs[1]).max() <= 1e-2 * max(1.0, scale)
    from tests.harness import cos_rows
    assert cos_rows(hid[0], hid[1]).min() >= 0.99999


def test_graph_replay_is_deterministic_and_matches_eager(river, tiny, stream):
    m, om, _ = tiny
    S = TINY
    toks = torch.from_numpy(synth.gen_tokens(S.vocab, (1, 20), seed=8)).cuda()
    sched = torch.tensor([2, 0, 4, 1], dtype=torch.int32, device="cuda")

    def run(use_stream):
        kv = m.kv_cache_alloc(1, 64)
        outs = []
        ctx = torch.cuda.stream(use_stream) if use_stream is not None else torch.cuda.stream(
            torch.cuda.default_stream())
        with ctx:
            river.prefill(m, kv, toks[:, :12].contiguous(), river.Policy.tau_(1.01), stream=use_stream)
            for i in range(8):
                o = river.decode_step(m, kv, toks[:, 12 + i].contiguous(),
                                      river.Policy.forced(sched), stream=use_stream)
                outs.append(o["logits"].clone())
            kv.sync(use_stream)
        return torch.stack(outs)

    a = run(stream)
    b = run(stream)
    c = run(torch.cuda.default_stream())
    assert torch.equal(a, b)
    assert torch.equal(a, c)


def test_error_paths(river, tiny, stream):
    m, om, _ = tiny
    S = TINY
    kv = m.kv_cache_alloc(2, 8)
    toks = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        river.prefill(m, kv, toks, river.Policy.tau_(1.01), stream=stream)
        with pytest.raises(river.RiverError) as e:
            river.decode_step(m, kv, toks[:, 0].contiguous(), river.Policy.tau_(1.01), stream=stream)
        assert e.value.status == river.RL_ERR_CAPACITY
        with pytest.raises(river.RiverError) as e:
            river.prefill(m, kv, torch.zeros((3, 4), dtype=torch.int32, device="cuda"),
                          river.Policy.tau_(1.01), stream=stream)
        assert e.value.status == river.RL_ERR_CAPACITY
        bad = torch.full((2, 4), S.vocab + 5, dtype=torch.int32, device="cuda")
        river.prefill(m, kv, bad, river.Policy.tau_(1.01), stream=stream)
        with pytest.raises(river.RiverError) as e:
            kv.sync(stream)
        assert e.value.status == river.RL_ERR_DEVICE
        sched = torch.tensor([S.n_layers + 3], dtype=torch.int32, device="cuda")
        river.decode_step(m, kv, toks[:, 0].contiguous(), river.Policy.forced(sched), stream=stream)
        with pytest.raises(river.RiverError) as e:
            kv.sync(stream)
        assert e.value.status == river.RL_ERR_DEVICE
        kv.sync(stream)  # cleared
    import early_exit_decoding_gb300 as r
    m2 = r.Model(S, __import__("tests.harness", fromlist=["to_cuda"]).to_cuda(
        synth.gen_weights(S, seed=1, device="cpu")), stream)
    kv2 = m2.kv_cache_alloc(1, 16)
    with pytest.raises(river.RiverError) as e:
        river.prefill(m2, kv2, toks[:1, :4].contiguous(),
                      river.Policy.forced(torch.tensor([1], dtype=torch.int32, device="cuda")),
                      stream=stream)
    assert e.value.status == river.RL_ERR_STATE


def test_host_buffer_entry_point(river, tiny, stream):
    """rl_decode_step_host (host buffers, copies inside) equals rl_decode_step."""
    m, om, _ = tiny
    S = TINY
    toks = synth.gen_tokens(S.vocab, (2, 10), seed=11)
    sched = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    res = []
    for host in (False, True):
        kv = m.kv_cache_alloc(2, 32)
        with torch.cuda.stream(stream):
            river.prefill(m, kv, torch.from_numpy(toks[:, :8]).cuda(), river.Policy.tau_(1.01),
                          stream=stream)
            for i in range(2):
                if host:
                    ht = torch.from_numpy(toks[:, 8 + i].copy()).pin_memory()
                    lg = torch.empty((2, S.vocab), dtype=torch.float32).pin_memory()
                    nt = torch.empty((2,), dtype=torch.int32).pin_memory()
                    ex = torch.empty((1,), dtype=torch.int32).pin_memory()
                    river.rl_decode_step_host(m.handle, kv.handle, ht, 2,
                                              river.Policy.forced(sched).c(), lg, nt, ex, None,
                                              stream)
                    res.append((lg.clone(), nt.clone(), int(ex.item())))
                else:
                    o = river.decode_step(m, kv, torch.from_numpy(toks[:, 8 + i].copy()).cuda(),
                                          river.Policy.forced(sched), stream=stream)
                    kv.sync(stream)
                    res.append((o["logits"].cpu(), o["next_token"].cpu(), int(o["exit_layer"].item())))
    for a, b in zip(res[:2], res[2:]):
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and a[2] == b[2]


@pytest.mark.parametrize("emb_scale", [2.0 ** 22, 2.0 ** -20])
def test_w4_path_activations_outside_fp16_range(river, stream, emb_scale):
    """The exit river's MMAs read the bf16 activations as fp16 after scaling
    each row by a power of two: residual streams far above the fp16 range
    (embedding x 2^22) or deep in its subnormals (x 2^-20) must give the
    oracle's logits and each layer's contribution to the residual."""
    from oracle.model import OracleModel
    from tests.harness import to_cuda, cos_rows
    S = synth.scaled(TINY, n_layers=2)
    w = synth.gen_weights(S, seed=11, device="cpu", gains="random")
    w["embed"] = (w["embed"].float() * emb_scale).to(torch.bfloat16)  # exact: power of two
    m = river.Model(S, to_cuda(w), stream)
    m.quantize_exit_layers(stream)
    om = OracleModel(S, synth.weights_to_numpy(w))
    om.quantize_exit_layers()
    toks = synth.gen_tokens(S.vocab, (1, 10), seed=12)
    kv = m.kv_cache_alloc(1, 32)
    kv.set_decode_path(PATHS["step"])
    st = KVState(S, 1, 32)
    tr = torch.zeros((S.n_layers + 1, 1, S.d_model), dtype=torch.float32, device="cuda")
    kv.set_trace(tr)
    sched = torch.tensor([0], dtype=torch.int32, device="cuda")  # every layer on the exit river
    with torch.cuda.stream(stream):
        river.prefill(m, kv, torch.from_numpy(toks[:, :9]).cuda(), river.Policy.forced(sched),
                      stream=stream)
        om.prefill(toks[:, :9], st, OPolicy.forced(0))
        out = river.decode_step(m, kv, torch.from_numpy(toks[:, 9].copy()).cuda(),
                                river.Policy.forced(sched), stream=stream)
        kv.sync(stream)
    ref = om.decode_step(toks[:, 9], st, OPolicy.forced(0))
    kv.set_trace(None)
    logits = out["logits"].cpu().numpy()
    assert np.isfinite(logits).all()
    assert np.abs(logits - ref.logits).max() <= 5e-2
    h = tr.cpu().numpy().astype(np.float64)
    for l in range(S.n_layers):
        c = cos_rows(h[l + 1] - h[l], ref.hidden[l + 1] - ref.hidden[l])
        assert c.min() >= 0.99, (l, c)


def test_step_timeline_orders_every_phase(river, tiny, stream):
    """Per-CTA timeline of the persistent step kernel (profiling level 2): no
    CTA starts phase p + 1 before every CTA has arrived at the end of phase p
    (the grid barrier), and each CTA's stamps of a phase are in order."""
    m, om, _ = tiny
    S = TINY
    kv = m.kv_cache_alloc(1, 64)
    kv.set_decode_path(PATHS["step"])
    toks = torch.from_numpy(synth.gen_tokens(S.vocab, (1, 10), seed=13)).cuda()
    with torch.cuda.stream(stream):
        river.prefill(m, kv, toks[:, :8].contiguous(), river.Policy.tau_(1.01), stream=stream)
        river.rl_kv_set_profiling(kv.handle, 2)
        river.decode_step(m, kv, toks[:, 8].contiguous(), river.Policy.tau_(0.5), stream=stream)
        river.rl_kv_profile(kv.handle, stream)
        tl = river.rl_kv_timeline(kv.handle, stream).astype(np.int64)
        river.rl_kv_set_profiling(kv.handle, 0)
        kv.sync(stream)
    nph, grid, nst = tl.shape
    assert nph == 5 * S.n_layers + 1 and nst == 8
    BAR, ARRIVE = 0, 4
    assert (tl[:, :, BAR] > 0).all() and (tl[:, :, ARRIVE] > 0).all()
    assert (tl[:, :, ARRIVE] >= tl[:, :, BAR]).all()
    for p in range(nph - 1):
        assert tl[p + 1, :, BAR].min() >= tl[p, :, ARRIVE].max(), p
