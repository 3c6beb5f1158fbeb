"""Decode benchmark of the River-LLM KV-shared exit river on GB300.

One bench step = one decode step of the whole hot path (embedding, every
layer on the backbone or the exit river with its KV append and attention,
layer-end similarity / exit decision, LM head, argmax) for one batch.

Default workload: Llama-3.2-1B shape (random init N(0, 0.02), seed 0), batch 1,
prompt of 512 uniform-random ids (seed 1), a 256-step generation under the
seeded forced exit schedule (mean exit layer 3.8 of 16, 5% full-depth steps,
seed 2); the timed steps cycle through that generation (positions 512..767).
Also timed: the same library with no exit (tau = 1.01) and with tau = 0.5.

  python bench.py [--gpus N --steps K --warmup W] [--impl river|reference]
                  [--config 1b-b1|tiny|1b-b32|8b-b1|8b-b64] [--no-cpu-baseline]

Under torchrun (N > 1) every rank runs an independent replica (the batch-min
rule couples the sequences of a batch, so a batch does not shard; see the
design notes): value = all ranks' tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s at Llama-1B/8B shapes; achieved HBM GB/s vs GB300 peak"

CONFIGS = {
    # name: (shape, batch, prompt, generation steps, forced-schedule mean, taus, kv fill)
    "tiny": ("tiny", 1, 32, 16, 2.0, (0.5, 1.01), "prefill"),
    "1b-b1": ("llama-3.2-1b", 1, 512, 256, 3.8, (0.5,), "prefill"),
    "1b-b32": ("llama-3.2-1b", 32, 1024, 512, 3.8, (0.3, 0.5, 0.7), "prefill"),
    "8b-b1": ("llama-3.1-8b", 1, 2048, 512, 8.0, (0.5,), "prefill"),
    "8b-b64": ("llama-3.1-8b", 64, 4096, 256, 8.0, (0.3, 0.5, 0.7), "random"),
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], "measured"
    return 6800.0, "fallback"


def shape_of(shape_name, args):
    import dataclasses
    import synth
    S = synth.SHAPES[shape_name]
    if getattr(args, "layers", 0):
        S = dataclasses.replace(S, n_layers=args.layers, name=f"{S.name} cut to {args.layers} layers")
    return S


def workload_desc(name, shape, B, T, G, mean):
    return (f"{shape.name} shape, random init N(0,0.02) seed 0, batch {B}, prompt {T} uniform ids "
            f"(seed 1), {G}-step generation under a forced exit schedule (geometric, target mean "
            f"exit layer {mean} of {shape.n_layers}, 5% full-depth steps, seed 2)")


# ------------------------------------------------------------------- algorithmic bytes

def layer_bytes(S, w4):
    d, hq, hkv, hd, f = S.d_model, S.n_q_heads, S.n_kv_heads, S.head_dim, S.ffn_dim
    shapes = [(hq * hd, d), (hkv * hd, d), (hkv * hd, d), (d, hq * hd), (f, d), (f, d), (d, f)]
    tot = 0.0
    for n, k in shapes:
        tot += n * k / 2 + n * ((k + 127) // 128) * 4 if w4 else n * k * 2
    return tot


def step_bytes(S, B, e, pos):
    """Weights of layers <= e in bf16, layers > e in W4 (+ fp16 scale/zero),
    the LM head, K/V rows 0..pos of every layer (read) and slot pos (write)."""
    w = e * layer_bytes(S, False) + (S.n_layers - e) * layer_bytes(S, True)
    w += S.vocab * S.d_model * 2
    kv = S.n_layers * B * S.n_kv_heads * S.head_dim * 2 * 2 * (pos + 1 + 1)
    return w + kv


# ---------------------------------------------------------------------- clocks

class Clocks:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_id):
        self.proc = None
        try:
            fd, self.out = tempfile.mkstemp(prefix="river_clocks_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", dev_id, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.out) as f:
            lines = f.read().splitlines()
        os.unlink(self.out)
        for line in lines:
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 8:
                try:
                    rows.append((float(p[0]), float(p[1]), p[4], p[5], p[6], p[7]))
                except ValueError:
                    pass
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                "sw_power_cap"), r[2:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def max_over_ranks(x, device):
    """The slowest rank's time: replicas are timed together and the job's
    throughput divides every rank's units by it (NCCL on GPUs, gloo on CPU)."""
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds):
    """Whole-job units per second: every rank processed units_per_rank."""
    return world * units_per_rank / seconds


# ---------------------------------------------------------------------- the library arm

def timed_indices(sched, K):
    """Generation indices of K timed steps.  K >= G: a cycle through the
    G-step generation.  K < G: a stratified sample of it, the K quantiles
    of its steps ordered by exit layer (index order among equal layers), so
    that any K sees the schedule's mix of exit layers and full-depth steps,
    run in generation order.  Each step runs at its own position (prompt +
    index)."""
    G = len(sched)
    if K >= G:
        return [i % G for i in range(K)]
    order = sorted(range(G), key=lambda j: (int(sched[j]), j))
    return sorted(order[int((i + 0.5) * G / K)] for i in range(K))  # in generation order


def schedule_stats(sched, idx, L):
    """Mean exit layer and full-depth share of the schedule entries ``idx``."""
    e = [int(sched[j]) for j in idx]
    return {"mean_exit_layer": sum(e) / len(e), "full_depth_share": sum(x == L for x in e) / len(e),
            "steps": len(e)}


class Arm:
    """One model + KV cache of a configuration, with the step driver the
    timed passes share."""

    def __init__(self, args, cfg, rank, world):
        import torch
        import synth
        import early_exit_decoding_gb300 as river
        self.torch, self.river = torch, river
        shape_name, B, T, G, mean, taus, kvfill = CONFIGS[cfg]
        S = shape_of(shape_name, args)
        self.S, self.B, self.T, self.G, self.mean, self.taus = S, B, T, G, mean, taus
        self.world = world
        self.stream = stream = torch.cuda.Stream()
        t0 = time.time()
        w = synth.gen_weights(S, seed=0, device="cuda", gains="ones")
        with torch.cuda.stream(stream):
            self.model = river.Model(S, w, stream)
            self.model.quantize_exit_layers(stream)
        stream.synchronize()
        del w
        torch.cuda.empty_cache()
        self.kv = kv = self.model.kv_cache_alloc(B, T + G + 1)
        self.sched_np = synth.gen_schedule(S.n_layers, G, mean, seed=2)
        self.sched = torch.from_numpy(self.sched_np).cuda()
        self.prompt = prompt = torch.from_numpy(synth.gen_tokens(S.vocab, (B, T), seed=1)).cuda()
        self.dec_np = synth.gen_tokens(S.vocab, (G, B), seed=4)
        dec = torch.from_numpy(self.dec_np).cuda()
        self.out = {"logits": torch.empty((B, S.vocab), dtype=torch.float32, device="cuda"),
                    "next_token": torch.empty((B,), dtype=torch.int32, device="cuda"),
                    "exit_layer": torch.empty((1,), dtype=torch.int32, device="cuda"),
                    "min_cos": torch.empty((S.n_layers,), dtype=torch.float32, device="cuda")}
        with torch.cuda.stream(stream):
            if kvfill == "prefill":
                river.prefill(self.model, kv, prompt, river.Policy.tau_(1.01), out=self.out,
                              stream=stream)
            else:  # timing-only fill of the cache at the target context
                for l in range(S.n_layers):
                    k, v = kv.view(l)
                    k[:B, :, :T].normal_()
                    v[:B, :, :T].normal_()
                kv.set_position(T, 0, stream)
            kv.sync(stream)
        self.tok = [dec[i].contiguous() for i in range(G)]
        self.cur = None  # generation index the cache position stands at
        self.repositions = 0
        self.forced = river.Policy.forced(self.sched)
        log(f"[rank {rank}] setup {time.time() - t0:.1f}s ({S.name}, B={B}, prompt {T})")

    def close(self):
        self.kv.close()
        self.model.close()
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()

    def goto(self, j):
        """Put the cache at generation index j (position T + j, decode step j),
        unless the previous step left it there."""
        if self.cur != j:
            self.kv.set_position(self.T + j, j, self.stream)
            self.repositions += 1
        self.cur = j

    def step(self, j, policy):
        self.goto(j)
        self.river.decode_step(self.model, self.kv, self.tok[j], policy, out=self.out,
                               stream=self.stream)
        self.cur = j + 1

    def timed(self, policy, K, W, clocks_dev=None):
        """W untimed warm-up steps, then K steps at the generation indices
        timed_indices(schedule, K), each at position T + index.  Every step is bracketed by
        its own pair of CUDA events on the launching stream; a reposition of
        the cache between two steps falls outside them.  Returns (ms summed
        over the K steps, clocks sampled during them, repositions)."""
        torch = self.torch
        idx = timed_indices(self.sched_np, K)
        clocks = Clocks(clocks_dev) if clocks_dev else None
        with torch.cuda.stream(self.stream):
            t_w, n_w = time.time(), 0
            # the clock sampler starts before the warm-up, which runs at least
            # W steps and half a second, so that neither the sampler's start-up
            # nor a GPU leaving idle clocks falls in the timed region
            while n_w < W or time.time() - t_w < 0.5:
                self.step(idx[n_w % K], policy)
                n_w += 1
                if n_w % 32 == 0:
                    self.stream.synchronize()
            self.kv.sync(self.stream)
            if self.world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            self.repositions = 0
            for i in range(K):
                j = idx[i]
                self.goto(j)
                ev[i][0].record(self.stream)
                self.river.decode_step(self.model, self.kv, self.tok[j], policy, out=self.out,
                                       stream=self.stream)
                ev[i][1].record(self.stream)
                self.cur = j + 1
            ev[-1][1].synchronize()
            torch.cuda.synchronize()
            if self.world > 1:
                torch.distributed.barrier()
            ck = clocks.stop() if clocks else None
            self.kv.sync(self.stream)
        ms = sum(a.elapsed_time(b) for a, b in ev)
        if self.world > 1:
            ms = max_over_ranks(ms, "cuda")
        return ms, ck, self.repositions

    def timed_bytes(self, K, forced):
        """Algorithmic bytes of the K timed steps (schedule exit layers or full depth)."""
        S = self.S
        tot = 0.0
        for j in timed_indices(self.sched_np, K):
            e = int(self.sched_np[j]) if forced else S.n_layers
            tot += step_bytes(S, self.B, e, self.T + j)
        return tot

    def time_prefill(self, n):
        """Mean device time (ms) of n prefills of the prompt, after one warm-up."""
        torch, river = self.torch, self.river
        ms = []
        with torch.cuda.stream(self.stream):
            for i in range(n + 1):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                river.prefill(self.model, self.kv, self.prompt, river.Policy.tau_(1.01), out=self.out,
                              stream=self.stream)
                e1.record(self.stream)
                e1.synchronize()
                if i:
                    ms.append(e0.elapsed_time(e1))
            self.kv.sync(self.stream)
        self.cur = None
        return sum(ms) / len(ms)

    def exit_kv_cosine(self):
        """Per layer, the cosine between the K (and V) the exit layer would
        write and the backbone layer's, for the residual entering the layer in
        one full-depth decode step: minimum and mean over sequences and KV heads."""
        torch, river, S = self.torch, self.river, self.S
        tr = torch.zeros((S.n_layers + 1, self.B, S.d_model), dtype=torch.float32, device="cuda")
        self.kv.set_trace(tr)
        with torch.cuda.stream(self.stream):
            self.step(0, river.Policy.tau_(1.01))
            self.kv.sync(self.stream)
        self.kv.set_trace(None)
        out = {"k_min": [], "k_mean": [], "v_min": [], "v_mean": []}
        with torch.cuda.stream(self.stream):
            for l in range(S.n_layers):
                c = self.model.exit_kv_cosine(l, tr[l], self.stream)
                self.stream.synchronize()
                k, v = c[:, 0].float().cpu(), c[:, 1].float().cpu()
                out["k_min"].append(round(float(k.min()), 5))
                out["k_mean"].append(round(float(k.mean()), 5))
                out["v_min"].append(round(float(v.min()), 5))
                out["v_mean"].append(round(float(v.mean()), 5))
        return out

    def profile(self, policy, n):
        """Live per-kernel records of n decode steps (a separate pass)."""
        river = self.river
        rows = []
        river.rl_kv_set_profiling(self.kv.handle, True)
        with self.torch.cuda.stream(self.stream):
            for i in range(n + 2):
                self.step(i % self.G, policy)
                r = river.rl_kv_profile(self.kv.handle, self.stream)
                if i >= 2:
                    rows.extend(r)
        river.rl_kv_set_profiling(self.kv.handle, False)
        return rows


def run_river(args, rank, world, dev):
    import torch
    torch.cuda.set_device(dev)
    arm = Arm(args, args.config, rank, world)
    S, B, G = arm.S, arm.B, arm.G
    river = arm.river
    K, W = args.steps, args.warmup
    res = {"arm": arm}
    res["ms_forced"], res["clocks"], res["repos"] = arm.timed(arm.forced, K, W, args.smi_id)
    res["ms_full"], _, _ = arm.timed(river.Policy.tau_(1.01), K, W)
    # every layer on its W4 exit copy (exit layer 0): the pages' full-quantisation comparison point
    sched0 = torch.zeros((1,), dtype=torch.int32, device="cuda")
    Kw = min(K, 4 * G)
    res["ms_w4"] = arm.timed(river.Policy.forced(sched0), Kw, W)[0] / Kw
    res["tau"] = {}
    for tau in arm.taus:
        ms_t, _, _ = arm.timed(river.Policy.tau_(tau), Kw, W)
        exits = []
        with torch.cuda.stream(arm.stream):
            for j in range(min(G, 64)):
                arm.step(j, river.Policy.tau_(tau))
                exits.append(int(arm.out["exit_layer"].item()))
        res["tau"][tau] = (ms_t / Kw, sum(exits) / len(exits))
    res["prof"] = arm.profile(arm.forced, min(G, 64))
    res["prefill_ms"] = arm.time_prefill(3)
    res["kv_cos"] = arm.exit_kv_cosine()

    # end to end: host buffers through rl_decode_step_host (pinned host tokens
    # in; next tokens, exit layer and logits out), copies inside each call
    ht = torch.zeros((B,), dtype=torch.int32).pin_memory()
    hn = torch.zeros((B,), dtype=torch.int32).pin_memory()
    he = torch.zeros((1,), dtype=torch.int32).pin_memory()
    hl = torch.zeros((B, S.vocab), dtype=torch.float32).pin_memory()
    Ke = min(K, G)
    idx_e = timed_indices(arm.sched_np, Ke)
    with torch.cuda.stream(arm.stream):
        for i in range(W):
            j = idx_e[i % Ke]
            arm.goto(j)
            ht.numpy()[:] = arm.dec_np[j]
            river.rl_decode_step_host(arm.model.handle, arm.kv.handle, ht, B, arm.forced.c(), hl,
                                      hn, he, None, arm.stream)
            arm.cur = j + 1
        arm.stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e2e_s = 0.0
        for i in range(Ke):
            j = idx_e[i]
            arm.goto(j)
            arm.stream.synchronize()
            t1 = time.perf_counter()
            ht.numpy()[:] = arm.dec_np[j]
            river.rl_decode_step_host(arm.model.handle, arm.kv.handle, ht, B, arm.forced.c(), hl,
                                      hn, he, None, arm.stream)
            e2e_s += time.perf_counter() - t1
            arm.cur = j + 1
    if world > 1:
        e2e_s = max_over_ranks(e2e_s, "cuda")
    res["e2e"] = (Ke, e2e_s)
    res["kernels_per_step"] = arm.model.kernel_count(B)
    res["timed_sched"] = schedule_stats(arm.sched_np, timed_indices(arm.sched_np, K), S.n_layers)
    res["gen_sched"] = schedule_stats(arm.sched_np, range(G), S.n_layers)
    return res


def dominant_kernel(prof, B):
    """(name, launches, phase records, traffic ratio) of the kernel with the
    most time in a live profile.  B <= 8: the persistent step kernel (one
    launch per step, every byte of the step; its phase records give the
    shares).  B > 8: one launch per kernel kind and layer; the kind with the
    most time."""
    steps = [r for r in prof if r[0] == "decode_step"]
    if steps:
        return ("k_decode_step (persistent decode step: every layer's projections, attention, "
                "LM head)", steps, [r for r in prof if r[0] != "decode_step"],
                traffic_note("step_dram_traffic.txt", "decode_step.cu", "attn_tc.cuh"))
    by_kind = {}
    for r in prof:
        by_kind[r[0]] = by_kind.get(r[0], 0.0) + r[3]
    top = max(by_kind, key=by_kind.get)
    launches = [r for r in prof if r[0] == top]
    if top == "attention":
        return ("k_attn_stream + k_attn_combine (streaming decode attention: K/V chunks by TMA, "
                "tensor cores; bytes = K and V rows 0..p of every sequence)", launches, prof,
                traffic_note("attn_stream_dram_traffic.txt", "attn_stream.cu", "attn_tc.cuh"))
    if B >= 16:
        return (f"k_gemm_tc ({top}: tcgen05 GEMM; W4 layers dequantised in shared memory or on "
                "k_gemv_fused)", launches, prof, None)
    return (f"k_gemv_fused ({top}: bf16 / W4 GEMV)", launches, prof,
            traffic_note("gemv_dram_traffic.txt", "gemv_fused.cu"))


def roofline_of(prof, B, peak, peak_src):
    kname, launches, phases, ratio = dominant_kernel(prof, B)
    g_ms = sum(r[3] for r in launches)
    g_bytes = sum(r[4] for r in launches)
    per_launch_bytes = g_bytes / max(1, len(launches))
    per_launch_ms = g_ms / max(1, len(launches))
    achieved = per_launch_bytes / (per_launch_ms / 1e3) / 1e9 if launches else 0.0
    all_ms = sum(r[3] for r in phases)
    shares = {}
    for r in phases:
        shares[r[0]] = shares.get(r[0], 0.0) + r[3]
    shares = {k: round(v / all_ms, 4) for k, v in sorted(shares.items(), key=lambda kv: -kv[1])}
    roof = {"kernel": kname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": ratio * per_launch_bytes if ratio is not None else None,
            "bytes_per_launch": per_launch_bytes, "ms_per_launch": per_launch_ms,
            "launches_profiled": len(launches), "peak_source": f"{peak_src} (copy test)"}
    return roof, shares


def run_8b_b1(args, world, hbm_peak, peak_src):
    """The Llama-3.1-8B batch-1 workload next to the default one: forced
    schedule (mean exit 8 of 32) and full depth (the >= 70 % roofline target),
    plus the step kernel's live roofline at full depth."""
    import torch
    arm = Arm(args, "8b-b1", 0, world)
    try:
        S, B, G = arm.S, arm.B, arm.G
        K, W = args.steps, args.warmup
        ms_f, ck, _ = arm.timed(arm.forced, K, W, args.smi_id)
        ms_n, _, _ = arm.timed(arm.river.Policy.tau_(1.01), K, W)
        roof, shares = roofline_of(arm.profile(arm.river.Policy.tau_(1.01), min(G, 32)), B,
                                   hbm_peak, peak_src)
        bf, bn = arm.timed_bytes(K, True), arm.timed_bytes(K, False)
        out = {
            "workload": workload_desc("8b-b1", S, B, arm.T, G, arm.mean),
            "steps": K,
            "forced": {"tokens_per_s": world * B * K / (ms_f / 1e3), "ms_per_step": ms_f / K,
                       "hbm_frac": bf / (ms_f / 1e3) / 1e9 / hbm_peak,
                       "timed_schedule": schedule_stats(arm.sched_np, timed_indices(arm.sched_np, K),
                                                        S.n_layers),
                       "generation_schedule": schedule_stats(arm.sched_np, range(G), S.n_layers),
                       "target_mean_exit_layer": arm.mean},
            "no_exit": {"tokens_per_s": world * B * K / (ms_n / 1e3), "ms_per_step": ms_n / K,
                        "hbm_frac": bn / (ms_n / 1e3) / 1e9 / hbm_peak,
                        "target_hbm_frac": 0.70},
            "forced_over_no_exit": ms_n / ms_f,
            "roofline_no_exit": roof,
            "kernel_time_shares_no_exit": shares,
            "clocks": ck,
        }
        # backbone offloading: layers L/2+1..L in pinned host memory, read over
        # NVLink-C2C only by steps that run them on the backbone
        first = S.n_layers // 2
        dev0, _ = arm.model.memory()
        arm.model.offload_backbone(first, arm.stream)
        dev1, host1 = arm.model.memory()
        ms_fo, _, _ = arm.timed(arm.forced, K, W)
        Kn = min(K, 8)
        ms_no, _, _ = arm.timed(arm.river.Policy.tau_(1.01), Kn, W)
        idx = timed_indices(arm.sched_np, K)
        touch = sum(int(arm.sched_np[j]) > first for j in idx)
        out["offload"] = {
            "offloaded_layers": f"{first + 1}..{S.n_layers} (backbone bf16 weights in pinned host memory)",
            "device_bytes_resident": dev0, "device_bytes_offloaded": dev1, "host_bytes": host1,
            "forced": {"tokens_per_s": world * B * K / (ms_fo / 1e3), "ms_per_step": ms_fo / K,
                       "timed_steps_running_offloaded_layers_on_the_backbone": touch},
            "full_depth_ms_per_step": ms_no / Kn,
            "full_depth_stall_ms_per_step": ms_no / Kn - ms_n / K,
        }
    finally:
        arm.close()
    return out


def source_hash(*sources):
    """sha256 prefix of the kernel's source files (csrc/), concatenated in order."""
    h = hashlib.sha256()
    for src in sources:
        h.update(open(os.path.join(ROOT, "early_exit_decoding_gb300", "csrc", src), "rb").read())
    return h.hexdigest()[:16]


def traffic_note(summary, *sources):
    """DRAM bytes over algorithmic bytes of a kernel from a committed ncu
    summary, if it was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    h = source_hash(*sources)
    if kv.get("source_sha256_16") != h:
        return None
    try:
        return float(kv["read_over_algorithmic"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------- the oracle (CPU)

def oracle_setup(args, need_exit=True):
    import numpy as np
    import torch
    import synth
    from oracle.model import OracleModel, Policy as OPolicy, KVState

    shape_name, B, T, G, mean, taus, kvfill = CONFIGS[args.config]
    S = synth.SHAPES[shape_name]
    t0 = time.time()
    dev = "cuda" if (S.name != "tiny" and torch.cuda.is_available()) else "cpu"
    w = synth.gen_weights(S, seed=0, device=dev, gains="ones")
    wn = synth.weights_to_numpy(w)
    del w
    om = OracleModel(S, wn)
    if need_exit:
        om.quantize_exit_layers()
    st = KVState(S, B, T + G + 1)
    prompt = synth.gen_tokens(S.vocab, (B, T), seed=1)
    if kvfill == "prefill":
        om.prefill(prompt, st, OPolicy.tau_(1.01))
    else:
        rng = np.random.default_rng(3)
        for l in range(S.n_layers):
            st.K[l][:, :, :T] = rng.standard_normal(st.K[l][:, :, :T].shape, dtype=np.float32)
            st.V[l][:, :, :T] = rng.standard_normal(st.V[l][:, :, :T].shape, dtype=np.float32)
        st.pos = T
    sched = synth.gen_schedule(S.n_layers, G, mean, seed=2)
    dec = synth.gen_tokens(S.vocab, (G, B), seed=4)
    log(f"oracle setup {time.time() - t0:.1f}s")
    return om, st, sched, dec, OPolicy, (S, B, T, G)


def run_oracle_steps(om, st, sched, dec, OPolicy, dims, n, budget_s):
    """Up to n oracle decode steps (stopping once budget_s seconds of them
    have run) at the generation indices timed_indices(schedule, n), each at
    position T + index, as the library arm's timed steps run."""
    S, B, T, G = dims
    done, t = 0, 0.0
    for j in timed_indices(sched, n):
        st.pos = T + j
        t1 = time.perf_counter()
        om.decode_step(dec[j], st, OPolicy.forced(int(sched[j])))
        t += time.perf_counter() - t1
        done += 1
        if t > budget_s:
            break
    return done, t


def threads_used():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


def oracle_sample(args):
    """Oracle decode tokens/s over a bounded sample (15 s) of the workload."""
    om, st, sched, dec, OPolicy, dims = oracle_setup(args)
    S, B, T, G = dims
    n, t = run_oracle_steps(om, st, sched, dec, OPolicy, dims, 64, 15.0)
    return n, B, T, t


def cpu_baseline(args):
    n, B, T, t = oracle_sample(args)
    out = {"value": n * B / t, "unit": "tokens/s", "cores": threads_used(), "kind": "oracle",
           "sample": f"{n} decode steps of the same workload (after the full {T}-token prefill, "
                     f"untimed), NumPy fp32 oracle on the host CPU"}
    # the same sample on one core, in a fresh process whose BLAS uses one thread
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--config", args.config,
                            "--oracle-sample-only"], env=env, capture_output=True, text=True,
                           timeout=600)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        out["one_core"] = {"value": one["value"], "unit": "tokens/s", "cores": 1,
                           "sample": f"{one['steps']} decode steps, the same sample on one core"}
    except Exception as ex:  # reported, never required
        out["one_core"] = {"value": None, "unit": "tokens/s", "cores": 1, "sample": f"failed: {ex!r}"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="river", choices=("river", "reference"))
    ap.add_argument("--config", default="1b-b1", choices=sorted(CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-8b", action="store_true",
                    help="skip the Llama-3.1-8B batch-1 block that the default workload adds")
    ap.add_argument("--oracle-sample-only", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: the config's shape cut to this many layers (a small "
                         "case for detailed ncu captures); the bench line names it")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    shape_name, B, T, G, mean, taus, kvfill = CONFIGS[args.config]
    import synth
    S = shape_of(shape_name, args)
    hbm_peak, peak_src = load_peaks()

    if args.oracle_sample_only:  # cpu_baseline's one-core leg (a child process, no GPU)
        n, B, T, t = oracle_sample(args)
        print(json.dumps({"value": n * B / t, "steps": n, "seconds": t, "cores": threads_used()}))
        return

    if args.impl == "reference":
        # The reference arm is the oracle, timed as it stands on the host cores.
        if rank != 0:
            return
        om, st, sched, dec, OPolicy, dims = oracle_setup(args)
        run_oracle_steps(om, st, sched, dec, OPolicy, dims, args.warmup, 60.0)
        n, t = run_oracle_steps(om, st, sched, dec, OPolicy, dims, args.steps, 120.0)
        v = n * B / t
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1,
                "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * t / n,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": {"workload": workload_desc(args.config, S, B, T, G, mean), "batch": B,
                           "prompt": T, "decode_steps": G},
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads_used(),
                                 "kind": "oracle",
                                 "sample": f"{n} decode steps (bounded to ~120 s) of the workload"},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    dev = local
    props = torch.cuda.get_device_properties(dev)
    args.smi_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(dev)
    res = run_river(args, rank, world, dev)
    arm = res["arm"]
    S, B, T, G = arm.S, arm.B, arm.T, arm.G
    K = args.steps
    ms_step = res["ms_forced"] / K
    tok_s = job_throughput(B * K, world, res["ms_forced"] / 1e3)
    full_ms_step = res["ms_full"] / K

    # algorithmic bytes of the timed steps: the schedule's exit layers at their positions
    tot_bytes = arm.timed_bytes(K, True)
    gbs = tot_bytes / (res["ms_forced"] / 1e3) / 1e9
    full_gbs = arm.timed_bytes(K, False) / (res["ms_full"] / 1e3) / 1e9
    roof, shares = roofline_of(res["prof"], B, hbm_peak, peak_src)
    Ke, e2e_s = res["e2e"]
    line_variants = {
        "no_exit": {"tokens_per_s": world * B / (full_ms_step / 1e3), "ms_per_step": full_ms_step,
                    "hbm_frac": full_gbs / hbm_peak},
        "forced_over_no_exit": full_ms_step / ms_step,
        "all_w4": {"tokens_per_s": world * B / (res["ms_w4"] / 1e3), "ms_per_step": res["ms_w4"],
                   "over_no_exit": full_ms_step / res["ms_w4"]},
        **{f"tau_{t}": {"tokens_per_s": world * B / (v[0] / 1e3), "ms_per_step": v[0],
                        "mean_exit_layer": v[1]} for t, v in res["tau"].items()},
        "prefill": {"ms": res["prefill_ms"], "tokens_per_s": B * T / (res["prefill_ms"] / 1e3),
                    "note": f"{B} x {T}-token prompt, full depth (tau 1.01), CUDA events"},
        "exit_kv_cosine_per_layer": {**res["kv_cos"],
                                     "note": "cosine of the exit layer's K / V against the backbone "
                                             "layer's for one decode step's residual entering each layer "
                                             "(rl_exit_kv_cosine); min and mean over KV heads"},
    }
    arm.close()
    del arm, res["arm"]
    if args.config == "1b-b1" and not args.no_8b and not args.layers:
        try:
            line_variants["llama8b_b1"] = run_8b_b1(args, world, hbm_peak, peak_src)
        except Exception as ex:  # reported, never required
            line_variants["llama8b_b1"] = {"failed": repr(ex)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(args)
        except Exception as ex:  # the baseline is reported, never required
            cpu = {"value": None, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"failed: {ex!r}"}

    ts, gs = res["timed_sched"], res["gen_sched"]
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (random-init weights, uniform token ids)",
        "config": {"workload": workload_desc(args.config, S, B, T, G, CONFIGS[args.config][4]),
                   "batch": B, "prompt": T, "decode_steps": G, "policy": "forced exit schedule",
                   "timed_steps": ("K < G: the K quantiles of the generation's steps ordered by "
                                   "exit layer, K >= G: a cycle through it; each step at its own "
                                   "position (prompt + generation index); time = the sum of "
                                   "per-step CUDA-event intervals on the launching stream"),
                   "schedule_mean_exit_layer": ts["mean_exit_layer"],
                   "schedule_full_depth_share": ts["full_depth_share"],
                   "generation_mean_exit_layer": gs["mean_exit_layer"],
                   "generation_full_depth_share": gs["full_depth_share"],
                   "target_mean_exit_layer": CONFIGS[args.config][4],
                   "l2": "inputs larger than L2: every step streams >= 1.4 GB of weights (L2 129 MB)",
                   "parallelism": f"replicas x{world}"},
        "hbm": {"algorithmic_bytes_per_step": tot_bytes / K, "achieved_gbs": gbs,
                "peak_gbs": hbm_peak, "frac": gbs / hbm_peak, "peak_source": peak_src},
        "roofline": roof,
        "kernel_time_shares": shares,
        "variants": line_variants,
        "e2e": {"value": world * B * Ke / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * B,
                "d2h_bytes_per_step": 4 * B + 4 + 4 * B * S.vocab,
                "note": ("rl_decode_step_host: pinned host tokens in; next tokens, exit layer and "
                         "fp32 logits out; each call timed from the token write to its return")},
        "gpu_launches": K * res["kernels_per_step"] + res["repos"],
        "clocks": res["clocks"],
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
