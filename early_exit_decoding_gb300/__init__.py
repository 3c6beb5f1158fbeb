"""Python binding of libriver.so (River-LLM KV-shared exit river on GB300).

Argument marshalling only: every step of the decode/prefill path runs in the
library's CUDA kernels.  PyTorch supplies device memory (tensors) and
streams.  The binding fails loudly when libriver.so is missing: there is no
CPU fallback.

The ``rl_*`` functions mirror the C ABI in ``include/river.h`` one to one;
``Model``, ``KVCache`` and ``Policy`` are small conveniences on top of them.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libriver.so")

RL_OK, RL_ERR_INVALID_ARG, RL_ERR_OOM, RL_ERR_CUDA, RL_ERR_CAPACITY, RL_ERR_STATE, \
    RL_ERR_DEVICE, RL_ERR_UNSUPPORTED = range(8)
RL_DEVERR_TOKEN, RL_DEVERR_CAPACITY, RL_DEVERR_SCHEDULE, RL_DEVERR_TIMEOUT = 1, 2, 4, 8
RL_EXIT_TAU, RL_EXIT_FORCED = 0, 1
RL_WQ, RL_WK, RL_WV, RL_WO, RL_WG, RL_WU, RL_WD = range(7)
LINEAR_NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")

EXPORTS = (
    "rl_version", "rl_last_error", "rl_model_create", "rl_model_destroy",
    "rl_quantize_exit_layers", "rl_quantize_exit_layers_hqq", "rl_exit_layer_view", "rl_kv_cache_alloc", "rl_kv_cache_free",
    "rl_kv_view", "rl_kv_position", "rl_kv_set_position", "rl_kv_set_trace", "rl_prefill",
    "rl_decode_step", "rl_decode_step_host", "rl_sync", "rl_decode_kernel_count",
    "rl_kv_set_profiling", "rl_kv_profile", "rl_kv_timeline", "rl_lm_head_static", "rl_kv_set_decode_path",
    "rl_kv_decode_path", "rl_save_exit_layers", "rl_load_exit_layers", "rl_exit_kv_cosine",
    "rl_kv_set_wait_limit", "rl_debug_fail_allocations", "rl_model_offload_backbone",
    "rl_model_memory",
)
RL_PATH_AUTO, RL_PATH_STEP, RL_PATH_FUSED, RL_PATH_GENERIC = range(4)
KERNEL_KINDS = ("embed", "qkv", "attention", "group_sums", "o_proj", "norm", "gate_up", "down",
                "layer_end", "lm_head", "argmax", "decode_step")


class rl_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_dim", "vocab",
        "group_size")] + [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


class rl_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "wq", "wk", "wv", "wo", "wg", "wu", "wd", "g_attn", "g_ffn")]


class rl_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("g_final", ctypes.c_void_p), ("layers", ctypes.POINTER(rl_layer_weights))]


class rl_exit_policy(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("tau", ctypes.c_float),
                ("d_schedule", ctypes.c_void_p), ("schedule_len", ctypes.c_int32)]


class RiverError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"libriver status {status}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                          "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, V = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, None
    PP = ctypes.POINTER(ctypes.c_void_p)
    PI = ctypes.POINTER(ctypes.c_int32)
    sig = {
        "rl_version": (ctypes.c_char_p, []),
        "rl_last_error": (ctypes.c_char_p, []),
        "rl_model_create": (I, [ctypes.POINTER(rl_config), ctypes.POINTER(rl_weights), P, PP]),
        "rl_model_destroy": (V, [P]),
        "rl_quantize_exit_layers": (I, [P, P]),
        "rl_quantize_exit_layers_hqq": (I, [P, I, ctypes.c_double, ctypes.c_double, ctypes.c_double, P]),
        "rl_exit_layer_view": (I, [P, I, I, PP, PP, PP, PI, PI]),
        "rl_kv_cache_alloc": (I, [P, I, I, PP]),
        "rl_kv_cache_free": (I, [P]),
        "rl_kv_view": (I, [P, I, PP, PP]),
        "rl_kv_position": (I, [P, PI, PI]),
        "rl_kv_set_position": (I, [P, I, I, P]),
        "rl_kv_set_trace": (I, [P, P]),
        "rl_prefill": (I, [P, P, P, I, I, ctypes.POINTER(rl_exit_policy), P, P, P, P, P]),
        "rl_decode_step": (I, [P, P, P, I, ctypes.POINTER(rl_exit_policy), P, P, P, P, P]),
        "rl_decode_step_host": (I, [P, P, P, I, ctypes.POINTER(rl_exit_policy), P, P, P, P, P]),
        "rl_sync": (I, [P, P, P]),
        "rl_decode_kernel_count": (I, [P, I]),
        "rl_kv_set_profiling": (I, [P, I]),
        "rl_kv_profile": (I, [P, P, I, PI, PI, PI, ctypes.POINTER(ctypes.c_float),
                              ctypes.POINTER(ctypes.c_double), PI]),
        "rl_kv_timeline": (I, [P, P, ctypes.c_int64, P, PI, PI, PI]),
        "rl_lm_head_static": (I, [P, P, I, P, P, P, P]),
        "rl_kv_set_decode_path": (I, [P, I]),
        "rl_kv_decode_path": (I, [P, I]),
        "rl_save_exit_layers": (I, [P, ctypes.c_char_p]),
        "rl_exit_kv_cosine": (I, [P, I, P, I, P, P]),
        "rl_kv_set_wait_limit": (I, [P, ctypes.c_int64]),
        "rl_model_offload_backbone": (I, [P, I, P]),
        "rl_model_memory": (I, [P, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
        "rl_debug_fail_allocations": (I, [ctypes.c_int64]),
        "rl_load_exit_layers": (I, [P, ctypes.c_char_p, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def _check(status):
    if status != RL_OK:
        raise RiverError(status, _lib.rl_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ----------------------------------------------------------------- C ABI, 1:1

def rl_version():
    return _lib.rl_version().decode()


def rl_last_error():
    return _lib.rl_last_error().decode()


def rl_model_create(cfg: rl_config, weights: rl_weights, stream=None):
    out = ctypes.c_void_p()
    _check(_lib.rl_model_create(ctypes.byref(cfg), ctypes.byref(weights), _stream(stream),
                                ctypes.byref(out)))
    return out


def rl_model_destroy(model):
    _lib.rl_model_destroy(model)


def rl_quantize_exit_layers(model, stream=None):
    _check(_lib.rl_quantize_exit_layers(model, _stream(stream)))


def rl_quantize_exit_layers_hqq(model, iters=20, lp_norm=0.7, beta=10.0, kappa=1.01, stream=None):
    _check(_lib.rl_quantize_exit_layers_hqq(model, int(iters), float(lp_norm), float(beta),
                                            float(kappa), _stream(stream)))


def rl_exit_kv_cosine(model, layer, d_h, B, d_cos, stream=None):
    _check(_lib.rl_exit_kv_cosine(model, int(layer), _ptr(d_h), int(B), _ptr(d_cos), _stream(stream)))


def rl_save_exit_layers(model, path):
    _check(_lib.rl_save_exit_layers(model, os.fsencode(path)))


def rl_load_exit_layers(model, path, stream=None):
    _check(_lib.rl_load_exit_layers(model, os.fsencode(path), _stream(stream)))


def rl_exit_layer_view(model, layer, which):
    q, s, z = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    n, k = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.rl_exit_layer_view(model, layer, which, ctypes.byref(q), ctypes.byref(s),
                                   ctypes.byref(z), ctypes.byref(n), ctypes.byref(k)))
    return q.value, s.value, z.value, n.value, k.value


def rl_kv_cache_alloc(model, max_batch, max_seq):
    out = ctypes.c_void_p()
    _check(_lib.rl_kv_cache_alloc(model, max_batch, max_seq, ctypes.byref(out)))
    return out


def rl_kv_cache_free(kv):
    _check(_lib.rl_kv_cache_free(kv))


def rl_kv_view(kv, layer):
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(_lib.rl_kv_view(kv, layer, ctypes.byref(k), ctypes.byref(v)))
    return k.value, v.value


def rl_kv_position(kv):
    p, s = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.rl_kv_position(kv, ctypes.byref(p), ctypes.byref(s)))
    return p.value, s.value


def rl_kv_set_position(kv, pos, decode_step, stream=None):
    _check(_lib.rl_kv_set_position(kv, pos, decode_step, _stream(stream)))


def rl_kv_set_trace(kv, d_hidden):
    _check(_lib.rl_kv_set_trace(kv, _ptr(d_hidden)))


def rl_prefill(model, kv, d_tokens, B, T, policy, d_logits, d_next_token, d_exit_layer,
               d_min_cos, stream=None):
    _check(_lib.rl_prefill(model, kv, _ptr(d_tokens), B, T, ctypes.byref(policy), _ptr(d_logits),
                           _ptr(d_next_token), _ptr(d_exit_layer), _ptr(d_min_cos),
                           _stream(stream)))


def rl_decode_step(model, kv, d_tokens, B, policy, d_logits, d_next_token, d_exit_layer,
                   d_min_cos, stream=None):
    _check(_lib.rl_decode_step(model, kv, _ptr(d_tokens), B, ctypes.byref(policy),
                               _ptr(d_logits), _ptr(d_next_token), _ptr(d_exit_layer),
                               _ptr(d_min_cos), _stream(stream)))


def rl_decode_step_host(model, kv, h_tokens, B, policy, h_logits, h_next_token, h_exit_layer,
                        h_min_cos, stream=None):
    _check(_lib.rl_decode_step_host(model, kv, _ptr(h_tokens), B, ctypes.byref(policy),
                                    _ptr(h_logits), _ptr(h_next_token), _ptr(h_exit_layer),
                                    _ptr(h_min_cos), _stream(stream)))


def rl_sync(model, kv, stream=None):
    _check(_lib.rl_sync(model, kv, _stream(stream)))


def rl_decode_kernel_count(model, B):
    return int(_lib.rl_decode_kernel_count(model, B))


def rl_lm_head_static(model, d_h, B, d_logits, d_next_token=None, d_err=None, stream=None):
    """Final RMSNorm + LM head + greedy argmax of ``d_h [B][d]`` using only the
    library's static scratch (allocates nothing)."""
    _check(_lib.rl_lm_head_static(model, _ptr(d_h), B, _ptr(d_logits), _ptr(d_next_token),
                                  _ptr(d_err), _stream(stream)))


def rl_model_offload_backbone(model, first_layer, stream=None):
    _check(_lib.rl_model_offload_backbone(model, int(first_layer), _stream(stream)))


def rl_model_memory(model):
    """(device bytes, pinned host bytes) the model holds."""
    d, h = ctypes.c_uint64(), ctypes.c_uint64()
    _check(_lib.rl_model_memory(model, ctypes.byref(d), ctypes.byref(h)))
    return d.value, h.value


def rl_kv_set_wait_limit(kv, polls):
    """Test hook: grid-barrier / first GEMM-epilogue waits give up after
    ``polls`` polls (0 = the kernels' own limits)."""
    _check(_lib.rl_kv_set_wait_limit(kv, int(polls)))


def rl_debug_fail_allocations(after):
    """Test hook: the next ``after`` library allocations succeed, later ones
    fail (RL_ERR_OOM); negative switches it off."""
    _check(_lib.rl_debug_fail_allocations(int(after)))


def rl_kv_set_decode_path(kv, path):
    _check(_lib.rl_kv_set_decode_path(kv, int(path)))


def rl_kv_decode_path(kv, B):
    return int(_lib.rl_kv_decode_path(kv, B))


def rl_kv_set_profiling(kv, enable):
    """0 off; 1 (or True) event records and the per-phase timeline; 2 also the
    per-CTA timeline of the step kernel (rl_kv_timeline)."""
    _check(_lib.rl_kv_set_profiling(kv, int(enable)))


def rl_kv_timeline(kv, stream=None):
    """Per-CTA timeline of the last profiled step: numpy uint64 array
    [phase][CTA][stamp] of globaltimer nanoseconds (0 = no such event)."""
    import numpy as np
    n_ph, n_cta, n_st = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    cap = 1 << 22
    buf = np.zeros(cap, dtype=np.uint64)
    _check(_lib.rl_kv_timeline(kv, _stream(stream), cap, buf.ctypes.data_as(ctypes.c_void_p),
                               ctypes.byref(n_ph), ctypes.byref(n_cta), ctypes.byref(n_st)))
    return buf[: n_ph.value * n_cta.value * n_st.value].reshape(n_ph.value, n_cta.value, n_st.value)


def rl_kv_profile(kv, stream=None, cap=1024):
    """List of (kind name, layer, path, ms, algorithmic bytes) of the last
    profiled decode step."""
    k = (ctypes.c_int32 * cap)()
    ly = (ctypes.c_int32 * cap)()
    pa = (ctypes.c_int32 * cap)()
    ms = (ctypes.c_float * cap)()
    by = (ctypes.c_double * cap)()
    n = ctypes.c_int32()
    _check(_lib.rl_kv_profile(kv, _stream(stream), cap, k, ly, pa, ms, by, ctypes.byref(n)))
    return [(KERNEL_KINDS[k[i]], ly[i], pa[i], ms[i], by[i]) for i in range(n.value)]


# --------------------------------------------------------------- conveniences

class _DevArray:
    """Wraps a library-owned device buffer for torch.as_tensor (no copy)."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {
            "shape": tuple(shape), "typestr": typestr, "data": (ptr, False), "version": 3,
            "strides": None,
        }


class Policy:
    """Exit policy: ``Policy.tau(t)`` or ``Policy.forced(schedule_tensor)``
    (device int32, decode step i uses schedule[i % len], prefill schedule[0])."""

    def __init__(self, mode, tau=1.01, schedule=None):
        self.mode, self.tau, self.schedule = mode, float(tau), schedule

    @staticmethod
    def tau_(t):
        return Policy(RL_EXIT_TAU, t)

    @staticmethod
    def forced(schedule):
        return Policy(RL_EXIT_FORCED, 0.0, schedule)

    def c(self):
        s = self.schedule
        return rl_exit_policy(self.mode, self.tau, None if s is None else s.data_ptr(),
                              0 if s is None else int(s.numel()))


class Model:
    """A model on the current CUDA device built from a weight dict
    (``embed, lm_head, g_final, layers[{wq..wd, g_attn, g_ffn}]``, bf16 CUDA
    tensors, linear weights row-major [out][in])."""

    def __init__(self, shape, weights, stream=None):
        import torch
        self.shape = shape
        cfg = rl_config(shape.n_layers, shape.d_model, shape.n_q_heads, shape.n_kv_heads,
                        shape.head_dim, shape.ffn_dim, shape.vocab, shape.group_size,
                        shape.rms_eps, shape.rope_theta)
        layers = (rl_layer_weights * shape.n_layers)()
        keep = []
        for i, lw in enumerate(weights["layers"]):
            vals = []
            for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd", "g_attn", "g_ffn"):
                t = lw[n]
                assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous(), n
                keep.append(t)
                vals.append(t.data_ptr())
            layers[i] = rl_layer_weights(*vals)
        for n in ("embed", "lm_head", "g_final"):
            t = weights[n]
            assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous(), n
        w = rl_weights(weights["embed"].data_ptr(), weights["lm_head"].data_ptr(),
                       weights["g_final"].data_ptr(), layers)
        self.handle = rl_model_create(cfg, w, stream)

    def close(self):
        if getattr(self, "handle", None):
            rl_model_destroy(self.handle)
            self.handle = None

    __del__ = close

    def quantize_exit_layers(self, stream=None, method="rtn", **hqq):
        """Build the exit river: min-max rounding (``method="rtn"``) or with
        HQQ's zero-point refinement (``method="hqq"``; keyword settings
        iters, lp_norm, beta, kappa)."""
        if method == "hqq":
            rl_quantize_exit_layers_hqq(self.handle, stream=stream, **hqq)
        elif method == "rtn":
            rl_quantize_exit_layers(self.handle, stream)
        else:
            raise ValueError(f"unknown quantizer {method!r}")

    def save_exit_layers(self, path):
        """Write the exit river (published packing) to ``path``."""
        rl_save_exit_layers(self.handle, path)

    def load_exit_layers(self, path, stream=None):
        """Build the exit river from a file written by save_exit_layers."""
        rl_load_exit_layers(self.handle, path, stream)

    def offload_backbone(self, first_layer, stream=None):
        """Backbone weights of layers first_layer.. (0-based) to pinned host memory."""
        rl_model_offload_backbone(self.handle, first_layer, stream)

    def memory(self):
        """(device bytes, pinned host bytes) the model holds."""
        return rl_model_memory(self.handle)

    def exit_kv_cosine(self, layer, h, stream=None):
        """Cosine between the exit layer's and the backbone layer's K and V of
        residual rows ``h [B][d]`` (fp32 CUDA) entering ``layer`` (0-based):
        a tensor [B][2][n_kv_heads] (K, then V)."""
        import torch
        B = h.shape[0]
        out = torch.empty((B, 2, self.shape.n_kv_heads), dtype=torch.float32, device="cuda")
        rl_exit_kv_cosine(self.handle, layer, h.contiguous(), B, out, stream)
        return out

    def exit_layer_view(self, layer, which):
        """(qweight int32 [N][K/8], scales fp16 [N][G], zeros fp16 [N][G]) torch views."""
        import torch
        q, s, z, n, k = rl_exit_layer_view(self.handle, layer, which)
        g = (k + 127) // 128
        qt = torch.as_tensor(_DevArray(q, (n, k // 8), "<i4"), device="cuda")
        st = torch.as_tensor(_DevArray(s, (n, g), "<f2"), device="cuda")
        zt = torch.as_tensor(_DevArray(z, (n, g), "<f2"), device="cuda")
        return qt, st, zt

    def kv_cache_alloc(self, max_batch, max_seq):
        return KVCache(self, max_batch, max_seq)

    def kernel_count(self, B):
        return rl_decode_kernel_count(self.handle, B)


class KVCache:
    def __init__(self, model: Model, max_batch, max_seq):
        self.model = model
        self.max_batch, self.max_seq = max_batch, max_seq
        self.handle = rl_kv_cache_alloc(model.handle, max_batch, max_seq)
        self._trace = None

    def close(self):
        if getattr(self, "handle", None):
            rl_kv_cache_free(self.handle)
            self.handle = None

    __del__ = close

    def view(self, layer):
        """(K, V) torch views, bf16 [max_batch][Hkv][max_seq][hd]."""
        import torch
        S = self.model.shape
        k, v = rl_kv_view(self.handle, layer)
        shp = (self.max_batch, S.n_kv_heads, self.max_seq, S.head_dim)
        kt = torch.as_tensor(_DevArray(k, shp, "<i2"), device="cuda").view(torch.bfloat16)
        vt = torch.as_tensor(_DevArray(v, shp, "<i2"), device="cuda").view(torch.bfloat16)
        return kt, vt

    def position(self):
        return rl_kv_position(self.handle)

    def set_position(self, pos, decode_step=0, stream=None):
        rl_kv_set_position(self.handle, pos, decode_step, stream)

    def set_trace(self, t):
        self._trace = t
        rl_kv_set_trace(self.handle, t)

    def set_decode_path(self, path):
        rl_kv_set_decode_path(self.handle, path)

    def decode_path(self, B):
        return rl_kv_decode_path(self.handle, B)

    def sync(self, stream=None):
        rl_sync(self.model.handle, self.handle, stream)


def _outputs(model, B, out):
    import torch
    S = model.shape
    if out is None:
        out = {}
    o = dict(out)
    o.setdefault("logits", torch.empty((B, S.vocab), dtype=torch.float32, device="cuda"))
    o.setdefault("next_token", torch.empty((B,), dtype=torch.int32, device="cuda"))
    o.setdefault("exit_layer", torch.empty((1,), dtype=torch.int32, device="cuda"))
    o.setdefault("min_cos", torch.empty((S.n_layers,), dtype=torch.float32, device="cuda"))
    return o


def prefill(model: Model, kv: KVCache, tokens, policy: Policy, out=None, stream=None):
    """tokens: CUDA int32 [B][T].  Returns a dict of output tensors."""
    B, T = tokens.shape
    o = _outputs(model, B, out)
    rl_prefill(model.handle, kv.handle, tokens, B, T, policy.c(), o["logits"], o["next_token"],
               o["exit_layer"], o["min_cos"], stream)
    return o


def decode_step(model: Model, kv: KVCache, tokens, policy: Policy, out=None, stream=None):
    """tokens: CUDA int32 [B].  Returns a dict of output tensors."""
    B = tokens.shape[0]
    o = _outputs(model, B, out)
    rl_decode_step(model.handle, kv.handle, tokens, B, policy.c(), o["logits"], o["next_token"],
                   o["exit_layer"], o["min_cos"], stream)
    return o


def quantize_exit_layers(model: Model, stream=None):
    model.quantize_exit_layers(stream)


def kv_cache_alloc(model: Model, max_batch, max_seq):
    return model.kv_cache_alloc(max_batch, max_seq)


__all__ = [*EXPORTS, "Model", "KVCache", "Policy", "RiverError", "prefill", "decode_step",
           "quantize_exit_layers", "kv_cache_alloc", "LIB_PATH"]
