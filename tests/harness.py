"""Shared helpers of the GPU parity tests: build the same model on both
sides from the seeded generators and compare step by step.

Tolerances (fixed by the specification of the method's parity bar):
logits max |diff| <= 5e-2; per-layer hidden-state cosine >= 0.999; integer
results (packed nibbles, scales/zeros bits, KV slot indices, exit layer under
a forced schedule) bit-exact; greedy tokens equal wherever the oracle's
top-1/top-2 gap exceeds 0.1.  Under tau, an exit layer may differ only when
the oracle's batch-minimum cosine of a layer up to the decision lies within
1e-3 of tau; the step is then re-run forced at the oracle's exit layer.
"""
from __future__ import annotations

import numpy as np

import synth
from oracle.model import OracleModel, Policy as OPolicy, KVState

LOGIT_TOL = 5e-2
HIDDEN_COS = 0.999
TAU_BAND = 1e-3
GAP = 0.1


def to_cuda(w):
    return {"embed": w["embed"].cuda(), "lm_head": w["lm_head"].cuda(),
            "g_final": w["g_final"].cuda(),
            "layers": [{k: v.cuda() for k, v in lw.items()} for lw in w["layers"]]}


def build_pair(shape, seed=0, gains="random", device=None, quantize=True, stream=None):
    import early_exit_decoding_gb300 as river
    w = synth.gen_weights(shape, seed=seed, device=device or "cpu", gains=gains)
    wd = to_cuda(w)
    m = river.Model(shape, wd, stream)
    if quantize:
        m.quantize_exit_layers(stream)
    om = OracleModel(shape, synth.weights_to_numpy(w))
    if quantize:
        om.quantize_exit_layers()
    del wd
    return m, om, w


def cos_rows(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.sum(a * b, -1) / np.maximum(np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1), 1e-30)


def check_step(gpu_out, ref, trace=None, B=None, label=""):
    """Compare one GPU call's outputs with the oracle's StepResult."""
    logits = gpu_out["logits"].float().cpu().numpy()
    d = np.abs(logits - ref.logits).max()
    assert d <= LOGIT_TOL, f"{label}: max |dlogit| {d:.4g} > {LOGIT_TOL}"
    if trace is not None:
        tr = trace.cpu().numpy()[:, :B]
        c = cos_rows(tr, ref.hidden)
        assert c.min() >= HIDDEN_COS, f"{label}: hidden-state cosine {c.min():.6f} < {HIDDEN_COS}"
    mc = gpu_out["min_cos"].cpu().numpy()
    assert np.abs(mc - ref.min_cos).max() < 5e-3, f"{label}: min_cos {mc} vs {ref.min_cos}"
    # greedy token where the oracle's decision is clear
    nt = gpu_out["next_token"].cpu().numpy()
    srt = np.sort(ref.logits, axis=-1)
    clear = (srt[:, -1] - srt[:, -2]) > GAP
    top = ref.logits.argmax(-1)
    assert np.all(nt[clear] == top[clear]), f"{label}: greedy tokens {nt} vs {top}"
    return d


def tau_band_ok(ref, tau, e_gpu):
    """The exit layers may differ only if a deciding cosine is within the band."""
    hi = min(max(ref.exit_layer, e_gpu), len(ref.min_cos) - 1)
    return bool(np.any(np.abs(ref.min_cos[:hi] - tau) <= TAU_BAND))
