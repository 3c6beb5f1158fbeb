"""fp32 Llama-style decoder with the River-LLM exit river (test infrastructure only).

Method (River-LLM explainer page):

* section 三: beside every backbone layer l sits an exit layer l, a W4A16
  copy of its parameters; the exit layer writes its K/V into backbone layer
  l's cache slot, so later tokens find every slot filled.
* section 四: at layer l the state-transition similarity is the cosine
  between the hidden state entering and leaving the layer; the minimum over
  all tokens processed together is compared with tau, and when it exceeds tau
  the remaining layers l+1..L run on the exit river.  Similarity rises with
  depth, so once the rule fires no later layer is checked.
* section 五: prefill takes one sequence-level decision (all prompt tokens
  exit at the same layer); generation decides per decode step.

Readings where the page is silent (each restated in the design notes):
"exit layer e" is the number of backbone layers run (1..L, e = L means no
exit); the cosine uses the fp32 residual stream before the pre-attention norm
and after the down projection, with denominator max(|a||b|, 1e-12); the
compare is strict (m > tau); no decision follows layer L; the embedding,
final norm and LM head are shared and unquantized; RoPE is rotate-half with
inv_freq[i] = theta^(-2i/hd) and angle = position * inv_freq in fp32.

Layer arithmetic (standard Llama):  x = RMSNorm(h)*g_attn; q,k,v = x W^T;
RoPE(q,k) at the token's position; append k,v to the layer's cache;
o = softmax(q K^T / sqrt(hd)) V over positions 0..p with H_q/H_kv query heads
per KV head; h1 = h + o W_o^T; x2 = RMSNorm(h1)*g_ffn;
u = silu(x2 W_g^T) * (x2 W_u^T); h2 = h1 + u W_d^T.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .quant import dequantize_linear, quantize_linear, quantize_linear_hqq

F32 = np.float32
LINEARS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


# ----------------------------------------------------------------------------
# Building blocks (each pinned by a library routine or an independent form)
# ----------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis, fp32."""
    x = x.astype(F32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=F32)
    return (x / np.sqrt(ms + F32(eps))).astype(F32) * g.astype(F32)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """inv_freq[i] = theta^(-2i/hd), i < hd/2, rounded once to fp32."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return (float(theta) ** (-2.0 * i / head_dim)).astype(F32)


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half RoPE.  ``x [..., n, H, hd]``, ``positions [n]`` (int).

    angle = fp32(position) * inv_freq (fp32 product); cos/sin of that fp32
    angle; out[:hd/2] = a cos - b sin, out[hd/2:] = b cos + a sin with
    a = x[:hd/2], b = x[hd/2:].
    """
    hd = x.shape[-1]
    half = hd // 2
    inv = rope_inv_freq(hd, theta)
    ang = (np.asarray(positions).astype(F32)[:, None] * inv[None, :]).astype(F32)  # [n][half]
    c = np.cos(ang.astype(np.float64)).astype(F32)[:, None, :]
    s = np.sin(ang.astype(np.float64)).astype(F32)[:, None, :]
    a = x[..., :half]
    b = x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1).astype(F32)


def silu(a: np.ndarray) -> np.ndarray:
    """a * sigmoid(a)."""
    a = a.astype(F32)
    return (a / (F32(1.0) + np.exp(-a))).astype(F32)


def cosine(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Row-wise <a,b> / max(|a||b|, 1e-12) over the last axis, fp32."""
    a = a.astype(F32)
    b = b.astype(F32)
    dot = np.sum(a * b, axis=-1, dtype=F32)
    na = np.sqrt(np.sum(a * a, axis=-1, dtype=F32))
    nb = np.sqrt(np.sum(b * b, axis=-1, dtype=F32))
    return (dot / np.maximum(na * nb, F32(1e-12))).astype(F32)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention for one sequence.

    q [n][Hq][hd] at positions q_pos [n]; k, v [Hkv][T][hd] for positions
    0..T-1.  Query head h reads KV head h // (Hq / Hkv).  A query at position
    p attends to keys 0..p.  Softmax in fp32 with max subtraction.
    Returns o [n][Hq][hd].
    """
    n, Hq, hd = q.shape
    Hkv, T, _ = k.shape
    rep = Hq // Hkv
    scale = F32(1.0 / np.sqrt(hd))
    out = np.empty((n, Hq, hd), dtype=F32)
    mask = np.arange(T)[None, :] <= np.asarray(q_pos)[:, None]  # [n][T]
    for h in range(Hq):
        g = h // rep
        s = (q[:, h, :] @ k[g].T).astype(F32) * scale            # [n][T]
        s = np.where(mask, s, -np.inf).astype(F32)
        m = np.max(s, axis=1, keepdims=True)
        p = np.exp(s - m).astype(F32)
        p = (p / np.sum(p, axis=1, keepdims=True, dtype=F32)).astype(F32)
        out[:, h, :] = (p @ v[g]).astype(F32)
    return out


# ----------------------------------------------------------------------------
# Policy and model
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Policy:
    """Exit policy: ``mode='tau'`` with threshold ``tau``, or ``mode='forced'``
    with exit layer ``e`` (0..L; layers l > e run on the exit river)."""
    mode: str = "tau"
    tau: float = 1.01
    e: int = 0

    @staticmethod
    def tau_(t):
        return Policy("tau", float(t), 0)

    @staticmethod
    def forced(e):
        return Policy("forced", 0.0, int(e))


@dataclasses.dataclass
class StepResult:
    logits: np.ndarray        # [B][V] fp32, last position of each sequence
    exit_layer: int           # e for this call
    min_cos: np.ndarray       # [L] batch-min cosine of every layer
    hidden: np.ndarray        # [L+1][B][d] residual stream at the last position (0 = embedding)


class KVState:
    """Per-layer K/V cache, fp32 ``[B][Hkv][max_seq][hd]``, plus the write position."""

    def __init__(self, shape, B: int, max_seq: int):
        hkv, hd = shape.n_kv_heads, shape.head_dim
        self.K = [np.zeros((B, hkv, max_seq, hd), F32) for _ in range(shape.n_layers)]
        self.V = [np.zeros((B, hkv, max_seq, hd), F32) for _ in range(shape.n_layers)]
        self.pos = 0
        self.B = B
        self.max_seq = max_seq


class OracleModel:
    """The oracle.  ``weights`` is the dict of float32 arrays from
    ``synth.weights_to_numpy`` (values already rounded to bf16)."""

    def __init__(self, shape, weights):
        self.shape = shape
        self.w = weights
        self.L = shape.n_layers
        self.backbone = [{k: lw[k] for k in LINEARS} for lw in weights["layers"]]
        self.exit = None
        self.quant = None

    # -- exit river ---------------------------------------------------------
    def quantize_exit_layers(self, method: str = "rtn"):
        """Build the exit river: a W4 copy of every linear of every layer, by
        min-max rounding (``"rtn"``) or with HQQ's zero-point refinement
        (``"hqq"``, section 六)."""
        quant = {"rtn": quantize_linear, "hqq": quantize_linear_hqq}[method]
        self.quant = []
        self.exit = []
        for lw in self.backbone:
            qd, ed = {}, {}
            for name in LINEARS:
                qw, s, z = quant(lw[name], self.shape.group_size)
                qd[name] = (qw, s, z)
                ed[name] = dequantize_linear(qw, s, z, lw[name].shape[1], self.shape.group_size)
            self.quant.append(qd)
            self.exit.append(ed)
        return self.quant

    def copy_exit_layers_unquantized(self):
        """Exit river built from the unquantized weights (invariant tests)."""
        self.exit = [{k: v.copy() for k, v in lw.items()} for lw in self.backbone]

    # -- exit-vs-backbone K/V similarity (diagnostic) -------------------------
    def exit_kv_cosine(self, l: int, h: np.ndarray, pos: int = 0) -> np.ndarray:
        """Section 三: the K/V an exit layer writes into the backbone's slot
        stays close to what the backbone layer would have written.  For
        residual rows ``h [B][d]`` entering layer ``l`` (0-based) at position
        ``pos``, the cosine per sequence and KV head between the exit layer's
        and the backbone layer's cache entries: ``[B][2][Hkv]`` (K, then V),
        each side RMSNorm'd, projected and (K) rotated as the layer does."""
        S = self.shape
        Hkv, hd = S.n_kv_heads, S.head_dim
        h = np.asarray(h, F32)
        B = h.shape[0]
        x = rmsnorm(h, self.w["layers"][l]["g_attn"], S.rms_eps)
        posa = np.array([pos])
        out = np.empty((B, 2, Hkv), F32)
        for j, name in enumerate(("wk", "wv")):
            yb = (x @ self.backbone[l][name].T).astype(F32).reshape(B, 1, Hkv, hd)
            ye = (x @ self.exit[l][name].T).astype(F32).reshape(B, 1, Hkv, hd)
            if name == "wk":
                yb = rope(yb, posa, S.rope_theta)
                ye = rope(ye, posa, S.rope_theta)
            out[:, j, :] = cosine(yb[:, 0], ye[:, 0])
        return out

    # -- one decoder layer -------------------------------------------------
    def layer(self, l: int, W: dict, h: np.ndarray, st: KVState, pos0: int) -> np.ndarray:
        """Layer ``l`` (0-based) on tokens at positions pos0..pos0+n-1.

        ``h [B][n][d]``; writes K/V slots pos0..pos0+n-1 of layer l.
        """
        S = self.shape
        B, n, d = h.shape
        Hq, Hkv, hd = S.n_q_heads, S.n_kv_heads, S.head_dim
        lw = self.w["layers"][l]
        x = rmsnorm(h, lw["g_attn"], S.rms_eps)
        q = (x @ W["wq"].T).astype(F32).reshape(B, n, Hq, hd)
        k = (x @ W["wk"].T).astype(F32).reshape(B, n, Hkv, hd)
        v = (x @ W["wv"].T).astype(F32).reshape(B, n, Hkv, hd)
        pos = np.arange(pos0, pos0 + n)
        q = rope(q, pos, S.rope_theta)
        k = rope(k, pos, S.rope_theta)
        st.K[l][:, :, pos0:pos0 + n, :] = k.transpose(0, 2, 1, 3)
        st.V[l][:, :, pos0:pos0 + n, :] = v.transpose(0, 2, 1, 3)
        T = pos0 + n
        o = np.empty((B, n, Hq, hd), F32)
        for b in range(B):
            o[b] = attention(q[b], st.K[l][b, :, :T], st.V[l][b, :, :T], pos)
        h1 = (h + (o.reshape(B, n, Hq * hd) @ W["wo"].T)).astype(F32)
        x2 = rmsnorm(h1, lw["g_ffn"], S.rms_eps)
        u = (silu((x2 @ W["wg"].T).astype(F32)) * (x2 @ W["wu"].T)).astype(F32)
        h2 = (h1 + (u @ W["wd"].T)).astype(F32)
        return h2

    # -- the exit river over all layers ---------------------------------------
    def run(self, tokens: np.ndarray, st: KVState, policy: Policy) -> StepResult:
        """Process ``tokens [B][n]`` at positions st.pos.. and advance st.pos.

        Prefill (n > 1) and decode (n == 1) share the rule: the minimum is
        taken over every token processed together.
        """
        S = self.shape
        L = self.L
        tokens = np.asarray(tokens)
        B, n = tokens.shape
        if st.pos + n > st.max_seq:
            raise ValueError("KV cache capacity exceeded")
        if policy.mode == "forced":
            if not (0 <= policy.e <= L):
                raise ValueError("forced exit layer outside [0, L]")
            exit_layer = policy.e
        else:
            exit_layer = L
        if exit_layer < L and self.exit is None:
            raise ValueError("exit river not built")
        h = self.w["embed"][tokens].astype(F32)                  # [B][n][d]
        min_cos = np.zeros(L, F32)
        hidden = [h[:, -1].copy()]
        for l in range(1, L + 1):
            W = self.backbone[l - 1] if l <= exit_layer else self.exit[l - 1]
            h_new = self.layer(l - 1, W, h, st, st.pos)
            c = cosine(h.reshape(B * n, -1), h_new.reshape(B * n, -1))
            m = F32(np.min(c))
            min_cos[l - 1] = m
            if policy.mode == "tau" and exit_layer == L and l < L and m > F32(policy.tau):
                exit_layer = l
                if self.exit is None:
                    raise ValueError("exit river not built")
            h = h_new
            hidden.append(h[:, -1].copy())
        st.pos += n
        hf = rmsnorm(h[:, -1], self.w["g_final"], S.rms_eps)
        logits = (hf @ self.w["lm_head"].T).astype(F32)
        return StepResult(logits, int(exit_layer), min_cos, np.stack(hidden))

    def prefill(self, tokens, st, policy):
        return self.run(tokens, st, policy)

    def decode_step(self, tokens, st, policy):
        return self.run(np.asarray(tokens).reshape(-1, 1), st, policy)

    # -- full-prefix recompute with a per-position exit layer -----------------
    def recompute(self, tokens: np.ndarray, exit_layers: np.ndarray) -> np.ndarray:
        """Recompute logits at every position from scratch, no cache reuse.

        ``tokens [B][T]``; ``exit_layers [T]``: position t ran layers 1..e_t on
        the backbone and the rest on the exit river.  All positions are
        processed together; attention reads K/V made by each key position's
        own weight choice.  Returns logits [B][T][V].
        """
        S = self.shape
        B, T = tokens.shape
        Hq, Hkv, hd = S.n_q_heads, S.n_kv_heads, S.head_dim
        e = np.asarray(exit_layers)
        h = self.w["embed"][tokens].astype(F32)
        pos = np.arange(T)
        for l in range(1, self.L + 1):
            lw = self.w["layers"][l - 1]
            use_exit = (l > e)[None, :, None]                     # [1][T][1]

            def lin(name, xx):
                yb = (xx @ self.backbone[l - 1][name].T).astype(F32)
                if self.exit is None:
                    return yb
                ye = (xx @ self.exit[l - 1][name].T).astype(F32)
                return np.where(use_exit, ye, yb)

            x = rmsnorm(h, lw["g_attn"], S.rms_eps)
            q = rope(lin("wq", x).reshape(B, T, Hq, hd), pos, S.rope_theta)
            k = rope(lin("wk", x).reshape(B, T, Hkv, hd), pos, S.rope_theta)
            v = lin("wv", x).reshape(B, T, Hkv, hd)
            o = np.empty((B, T, Hq, hd), F32)
            for b in range(B):
                o[b] = attention(q[b], k[b].transpose(1, 0, 2), v[b].transpose(1, 0, 2), pos)
            h1 = (h + lin("wo", o.reshape(B, T, Hq * hd))).astype(F32)
            x2 = rmsnorm(h1, lw["g_ffn"], S.rms_eps)
            u = (silu(lin("wg", x2)) * lin("wu", x2)).astype(F32)
            h = (h1 + lin("wd", u)).astype(F32)
        hf = rmsnorm(h, self.w["g_final"], S.rms_eps)
        return (hf @ self.w["lm_head"].T).astype(F32)
