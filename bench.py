#!/usr/bin/env python3
"""Benchmark of the ds4 layer step on one GB300 (or N independent replicas).

Headline: batch-1 decode tok/s of one full-width layer (hidden 4096, 64 x 128 MQA over a
128-token window, 256 experts top-6 + shared expert, BF16 weights and KV, KV pre-filled
with 4096 seeded positions): each step is one token through the whole layer step.  The
same JSON line carries layer-major prefill tok/s (8 layers, 4096 tokens), stack decode
tok/s with lm_head + top-p sampling (8 layers), and the common-prefix resync latency
(16994 live -> 16846 common -> 91-token suffix), each with its roofline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

HBM_FALLBACK_GBS = 6800.0
BF16_FALLBACK_TFLOPS = 1900.0


# --------------------------------------------------------------------------- workload facts

def layer_bytes(m: synth.ModelShape) -> dict:
    """Algorithmic bytes per decode-step launch of each kernel (weights streamed once,
    the K/V window and activations counted)."""
    H, QD, RQ, RKV, HD = m.hidden, m.n_heads * m.head_dim, m.q_rank, m.kv_rank, m.head_dim
    E, K, I, W = m.n_experts, m.top_k, m.expert_inter, m.window
    w = 2  # bf16
    return {
        "qkv_a": (RQ + RKV) * H * w + H * 4 + (RQ + RKV) * 4,
        "qkv_b": (QD * RQ + 2 * HD * RKV) * w + (RQ + RKV) * 4 + QD * 4 + 2 * HD * w,
        "attn": 2 * W * HD * w + 2 * QD * 4,
        "wo": H * QD * w + QD * 4 + 2 * H * 4,
        "router": E * H * w + 2 * H * 4 + E * 4,
        "expert_gu": (K + 1) * 2 * I * H * w + H * 4 + (K + 1) * I * 4,
        "expert_down": (K + 1) * H * I * w + (K + 1) * I * 4 + 2 * H * 4,
    }


def lm_head_bytes(m):
    return m.vocab * m.hidden * 2 + m.hidden * 4 + m.vocab * 4


def prefill_flops_per_token_layer(m) -> float:
    H, QD, RQ, RKV, HD = m.hidden, m.n_heads * m.head_dim, m.q_rank, m.kv_rank, m.head_dim
    E, K, I, W = m.n_experts, m.top_k, m.expert_inter, m.window
    mac = (H * (RQ + RKV) + RQ * QD + RKV * 2 * HD + QD * H + H * E
           + (K + 1) * (2 * H * I + I * H)) + 2 * m.n_heads * W * HD
    return 2.0 * mac


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), \
            "measured"
    except Exception:
        return HBM_FALLBACK_GBS, BF16_FALLBACK_TFLOPS, 1700.0, "fallback"


def ncu_traffic(kernel: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, if it was
    taken on the current kernel source (same digest of decode_persistent.cu,
    common.cuh and sm100.cuh), else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    csrc = os.path.join(ROOT, "prefill_decode_layer_gb300", "csrc")
    try:
        h = hashlib.sha1()
        for name in ("decode_persistent.cu", "common.cuh", "sm100.cuh"):
            h.update(open(os.path.join(csrc, name), "rb").read())
        digest = h.hexdigest()[:12]
        for line in open(path):
            parts = line.split()
            if len(parts) >= 3 and parts[0] == kernel and parts[1] == digest:
                return int(float(parts[2]))
    except OSError:
        pass
    return None


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()   # nvidia-smi takes a moment to start: wait for its first sample
            while not self.lines and time.time() - t0 < 5.0 and self.proc.poll() is None:
                time.sleep(0.01)
            self.lines.clear()   # keep only samples taken from here on (the timed region)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- helpers

def replica_rate(local_ms: float, units: int, dist=None, device: str = "cuda"):
    """Whole-job rate of N independent replicas (no data-path collective): every rank
    processed `units` in its own `local_ms`; the slowest rank bounds the job, so the
    value is N * units over the maximum time.  Returns (max ms, units per second)."""
    world, total = 1, float(local_ms)
    if dist is not None:
        import torch
        t = torch.tensor([total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total = float(t.item())
        world = dist.get_world_size()
    return total, world * units / (total / 1000.0)


def nproc():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_decode_rate(m: synth.ModelShape, n_pre: int, seconds: float, seed: int = 0,
                       steps: int = 256, warmup: int = 0):
    """Oracle decode steps/s on the single-layer workload (one thread): `warmup`
    untimed steps, then up to `steps` timed steps, stopping early once `seconds` have
    passed.  Returns (rate, timed steps, seconds)."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from helpers import LazyOracleModel, OracleKV, oracle_embed, oracle_layer
    om = LazyOracleModel(m.with_(n_layers=1), seed)
    om.layer(0)                                   # generate weights outside the timing
    total = warmup + steps
    kv = OracleKV(m.with_(n_layers=1), n_pre + total + 1)
    hk, hv = synth.host_kv(m, 0, n_pre, seed)
    kv.k[0][:n_pre] = hk
    kv.v[0][:n_pre] = hv
    toks = synth.host_tokens(total, m.vocab, seed, stream=5)
    for i in range(warmup):
        oracle_layer(om, kv, 0, n_pre + i, oracle_embed(om, toks[i]))
    t0 = time.perf_counter()
    n = 0
    while n < steps:
        x = oracle_embed(om, toks[warmup + n])
        oracle_layer(om, kv, 0, n_pre + warmup + n, x)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    del oracle
    return n / dt, n, dt


# --------------------------------------------------------------------------- reference arm

def run_reference(args) -> dict:
    """The oracle (single-threaded C, double precision) on the headline workload:
    `warmup` untimed decode steps, then `steps` timed ones, the timed part cut short
    after DS4G_REF_SECONDS (default 120 s); `steps` reports the steps it timed."""
    secs = float(os.environ.get("DS4G_REF_SECONDS", "120"))
    m = synth.LAYER
    warm = min(args.warmup, 3)   # oracle warm-up: weights are generated outside the timing
    rate, n, dt = oracle_decode_rate(m, 4096, secs, steps=args.steps, warmup=warm)
    value = rate
    bounded = n < args.steps
    return {
        "metric": "decode tok/s (batch 1)", "value": value, "unit": "tok/s", "n_gpus": 0,
        "steps": n, "warmup": warm, "ms_per_step": 1000.0 / value, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": workload_config(m),
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} timed oracle decode steps after {warm} untimed ones "
                                   f"(positions 4096.., {dt:.1f} s, single thread, "
                                   f"{cpu_model()}, {nproc()} cores present)"
                                   + (f"; time-bounded at {secs:.0f} s, {args.steps} requested"
                                      if bounded else "")},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def workload_config(m):
    return {"workload": "decode_layer: 1 layer, hidden 4096, 64x128 MQA (1 KV head), q/kv "
                        "rank 1024/512, window 128, 256 experts top-6 + shared (inter 1024), "
                        "BF16 weights ~N(0,0.02), BF16 KV pre-filled with 4096 seeded N(0,1) "
                        "positions, batch 1, random token ids",
            "global_batch": 1, "kv_prefill": 4096, "lm_head": "none (layer step only)",
            "l2": "inputs larger than L2: each step streams ~275 MB of weights (L2 129 MB), "
                  "steps back to back; a flushed-L2 run is reported in l2_flushed_each_step",
            "parallelism": "replicas"}


# --------------------------------------------------------------------------- profiling cases

# decode-full: the headline workload (one full-width layer, 4096 positions of KV);
# decode-small: the same layer with 32 routed experts and a 8192-token vocabulary,
#   so that a multi-pass ncu capture holds about 1 GB on the device while every step
#   still streams more weight bytes (about 265 MB) than the 129 MB L2.
# prefill-full: the layer-major prefill workload (8 full-width layers, 4096 tokens),
#   each step truncates the session to 0 and prefills the same prompt again.
# prefill-small: one full-width layer with 128 routed experts and 2048 tokens (about
#   3 GB on the device; still 96 tokens per expert, as in prefill-full).
# prefill-layer: one full-width layer with 128 routed experts and 4096 tokens (about
#   5 GB on the device): the dense GEMMs and the attention at prefill-full's shapes.
CASES = {"decode-full": dict(), "decode-small": dict(n_experts=32, vocab=8192),
         "prefill-full": dict(n_layers=8), "prefill-small": dict(n_layers=1, n_experts=128),
         "prefill-layer": dict(n_layers=1, n_experts=128)}
PREFILL_TOKENS = {"prefill-full": 4096, "prefill-small": 2048, "prefill-layer": 4096}


def run_case(args):
    import torch
    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw
    shape = synth.LAYER.with_(**CASES[args.case])
    if args.case.startswith("prefill"):
        emb, lm, layers = tw.dev_model(shape)
        m = pdl.Model(shape, emb, lm, layers)
        nt = PREFILL_TOKENS[args.case]
        s = pdl.Session(m, nt + 8)
        toks = synth.host_tokens(nt, shape.vocab, stream=41)
        stream = torch.cuda.current_stream()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(args.warmup + args.steps):
            if i == args.warmup:
                torch.cuda.synchronize()
                ev0.record(stream)
            assert s.truncate(0) == 0 and s.prefill(toks) == 0
        ev1.record(stream)
        torch.cuda.synchronize()
        assert s.status() == 0
        ms = ev0.elapsed_time(ev1) / max(1, args.steps)
        line = {"case": args.case, "steps": args.steps, "warmup": args.warmup,
                "launches": int(s.launches), "ms_per_prefill": ms, "tok_per_s": nt / ms * 1e3}
        if args.timeline:
            # per-launch times: an event after every launch (no overlap between launches)
            s.set_timing(True)
            s.timing()
            for i in range(args.steps):
                assert s.truncate(0) == 0 and s.prefill(toks) == 0
            torch.cuda.synchronize()
            t = {k: v for k, v in s.timing().items() if k.startswith("p_") and v[1] > 0}
            s.set_timing(False)
            tot = sum(v[0] for v in t.values())
            line["timeline"] = {"note": "CUDA event after every launch; us per launch, share of "
                                        "the evented prefill", "ms_per_prefill_with_events": tot / args.steps,
                                "per_kind": {k[2:]: {"launches_per_prefill": v[1] / args.steps,
                                                     "us_per_launch": round(1e3 * v[0] / v[1], 1),
                                                     "share": round(v[0] / tot, 4)}
                                             for k, v in sorted(t.items(), key=lambda kv: -kv[1][0])}}
        print(json.dumps(line), flush=True)
        return
    emb, lm, layers = tw.dev_model(shape)
    m = pdl.Model(shape, emb, lm, layers)
    n_pre = 4096
    s = pdl.Session(m, n_pre + args.warmup + args.steps + 16)
    k, v = s.kv(0)
    tw.fill_kv(shape, 0, k, v, n_pre)
    assert s.restore(synth.host_tokens(n_pre, shape.vocab, stream=11)) == 0
    toks = synth.host_tokens(args.warmup + args.steps, shape.vocab, stream=5)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            torch.cuda.synchronize()
            ev0.record(stream)
        assert s.decode_layers(int(toks[i])) == 0
    ev1.record(stream)
    torch.cuda.synchronize()
    assert s.status() == 0
    us = ev0.elapsed_time(ev1) * 1e3 / max(1, args.steps)
    out = {"case": args.case, "steps": args.steps, "warmup": args.warmup,
           "launches": int(s.launches), "us_per_step": us}
    if args.timeline:
        out["timeline_us"] = decode_timeline(torch, s, shape, synth.host_tokens(6, shape.vocab, stream=6))
    print(json.dumps(out), flush=True)


# Stage starts of the persistent decode kernel (globaltimer stamps of every CTA,
# the session's trace buffer): per event, the earliest, median and latest CTA, in
# us after the first CTA started, averaged over a few steps run back to back.
# Events per layer l: 7 l + 0 stage 1, + 1 stages 2-3, + 2 stages 2-3 after the
# query/K/V items, + 3 stage 4, + 4 stage 5, + 5 stage 6, + 6 stage 7; then the
# lm_head and the end.
TIMELINE_NAMES = ["stage 1 (norm, W_qa/W_kva)", "stages 2-3 (queries, K/V, attention)",
                  "stages 2-3 after the query/K/V rows", "stage 4 (W_o)", "stage 5 (norm, router)",
                  "stage 6 (gate/up, after the top-k)", "stage 7 (down, combine)"]


def decode_timeline(torch, sess, shape, toks):
    ev = 7 * shape.n_layers + 2
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(ev * nsm, dtype=torch.int64, device="cuda")
    acc = np.zeros((ev, 3))
    for t in toks:
        buf.zero_()
        sess.set_trace(buf)
        assert sess.decode_layers(int(t)) == 0
        sess.set_trace(None)
        torch.cuda.synchronize()
        st = buf.cpu().numpy().reshape(ev, nsm).astype(np.float64)
        t0 = st[0].min()
        for e in range(ev):
            row = (st[e] - t0) / 1e3
            acc[e] += [row.min(), np.median(row), row.max()]
    acc /= len(toks)
    names = [f"layer {l}: {n}" for l in range(shape.n_layers) for n in TIMELINE_NAMES]
    names += ["lm_head", "end"]
    return {n: [round(v, 2) for v in acc[e]] for e, n in enumerate(names)}


# --------------------------------------------------------------------------- our arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the prefill / stack / resync measurements")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--min-seconds", type=float, default=1.25,
                    help="the headline's K timed steps are repeated until the timed region "
                         "lasts about this long")
    ap.add_argument("--timeline", action="store_true",
                    help="with --case decode-*: also print the kernel's stage start times; with "
                         "--case prefill-*: per-launch times from events after every launch")
    ap.add_argument("--case", default=None, choices=list(CASES),
                    help="run only warmup + steps of one workload (the profiling commands "
                         "recorded in profiles/ use this) and print a one-line summary")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.case:
        run_case(args)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    def barrier():
        if dist is not None:
            dist.barrier()

    import prefill_decode_layer_gb300 as pdl
    from synth import torch_weights as tw

    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()
    stack = synth.STACK
    layer = synth.LAYER
    extra = not args.no_extra and rank == 0
    n_layers_alloc = stack.n_layers if extra else 1
    emb = tw.dev_embedding(stack)
    lm = tw.dev_lm_head(stack)
    layers = [tw.dev_layer(stack, l) for l in range(n_layers_alloc)]
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    # ---------------- headline: single full-width decode layer at batch 1
    m1 = pdl.Model(layer, emb, lm, layers[:1])
    n_pre = 4096
    n_flushed = min(args.steps, 200)
    # positions: warm-up and each repeat of the timed steps restart at n_pre; then the
    # flushed steps, the per-kernel timing pass (48) and the end-to-end steps (64)
    n_ctx = n_pre + max(args.warmup, args.steps) + n_flushed + 48 + 64 + 16
    sess = pdl.Session(m1, n_ctx)
    k, v = sess.kv(0)
    tw.fill_kv(layer, 0, k, v, n_pre)
    assert sess.restore(synth.host_tokens(n_pre, layer.vocab, stream=11)) == 0
    toks = synth.host_tokens(args.warmup + args.steps + n_flushed + 64, layer.vocab, stream=5)

    def timed_steps(first, n, flush_l2):
        # CUDA events on the session's (current) stream; returns total ms.  Steps run back
        # to back between one pair of events; with an L2 flush before every step, each
        # step has its own pair so that the flushes stay outside the timed time.
        if not flush_l2:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n):
                rc = sess.decode_layers(int(toks[first + i]))
                if rc != 0:
                    raise RuntimeError(f"decode failed: {rc}")
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i in range(n):
            if flush_l2:
                flush.zero_()
            ev[i][0].record(stream)
            rc = sess.decode_layers(int(toks[first + i]))
            ev[i][1].record(stream)
            if rc != 0:
                raise RuntimeError(f"decode failed: {rc}")
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev)

    # Headline: steps back to back.  Every step streams ~275 MB of weights, more than
    # the 129 MB L2, so no weight is still cached when the next step reads it.  The K
    # steps are repeated R times, the session truncated back to its 4096 pre-filled
    # positions between repeats (host bookkeeping only: nothing is launched, so the
    # stream stays back to back), so that the timed region lasts at least about a
    # second whatever K is and the clock samples cover it.
    est = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    est[0].record(stream)
    for i in range(args.warmup):
        assert sess.decode_layers(int(toks[i])) == 0
    est[1].record(stream)
    torch.cuda.synchronize()
    assert sess.truncate(n_pre) == 0
    est_ms = est[0].elapsed_time(est[1]) / args.warmup
    repeats = max(1, int(np.ceil(args.min_seconds * 1000.0 / (args.steps * est_ms))))

    def timed_batches(n, reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for r in range(reps):
            if r:
                assert sess.truncate(n_pre) == 0
            for i in range(n):
                rc = sess.decode_layers(int(toks[args.warmup + i]))
                if rc != 0:
                    raise RuntimeError(f"decode failed: {rc}")
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    launches0 = sess.launches
    total_ms = timed_batches(args.steps, repeats)
    barrier()
    clk = clocks.stop()
    gpu_launches = sess.launches - launches0
    assert sess.status() == 0
    total_ms, value = replica_rate(total_ms, args.steps * repeats, dist)
    ms_per_step = total_ms / (args.steps * repeats)
    # Secondary: the same with a 512 MB L2 flush before every step (cold code and data).
    fl_ms = timed_steps(args.warmup + args.steps, n_flushed, True) / n_flushed
    flushed = {"ms_per_step": round(fl_ms, 5), "value": round(world * 1000.0 / fl_ms, 1),
               "steps": n_flushed, "how": "512 MB write before every step (L2 cold: code, "
                                          "KV and weights), per-step CUDA events"}

    # per-kernel timing pass (events between kernels) for the dominant kernel's roofline
    sess.set_timing(True)
    sess.timing()
    base = args.warmup + args.steps
    for i in range(48):
        flush.zero_()
        assert sess.decode_layers(int(toks[(base + i) % len(toks)])) == 0
    kt = sess.timing()
    sess.set_timing(False)
    lb = layer_bytes(layer)
    per_kernel = {}
    for kname, (ms, cnt) in kt.items():
        if cnt and kname in lb:
            avg = ms / cnt
            per_kernel[kname] = {"avg_us": round(avg * 1000, 2),
                                 "gbs": round(lb[kname] / (avg / 1000) / 1e9, 1)}
    # The timed step is one launch of the persistent kernel: its roofline is the step's.
    step_bytes = sum(lb.values())
    achieved = step_bytes / (ms_per_step / 1000) / 1e9
    roofline = {"kernel": "k_decode_persistent (one launch = one layer step)", "bound": "hbm",
                "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "peak_source": f"{peak_src} hbm_gbs (copy, read+write; burst)",
                "traffic": ncu_traffic("k_decode_persistent"), "algorithmic_bytes": step_bytes,
                "timing": "CUDA events around the timed region (R repeats of K back-to-back "
                          "steps), average per launch"}
    staged = {"note": "one kernel per stage (decode_kernel=1), per-kernel CUDA events, "
                      "L2 flushed between steps", "per_kernel": per_kernel}

    # ---------------- end to end through the C ABI with host buffers
    # Per step, one call (ds4g_decode_layers_host): the token from pinned host memory
    # in, the layer step, the 16 KB hidden state copied to pinned host memory, the
    # stream synchronised; timed on the host clock.
    hidden_host = torch.empty(layer.hidden, dtype=torch.float32, pin_memory=True)
    tok_host = [int(t) for t in toks[:64]]   # host-side token ids
    e2e_ms = []
    for i in range(64):
        t0 = time.perf_counter()
        rc = sess.decode_layers_host(tok_host[i], hidden_host)
        t1 = time.perf_counter()
        assert rc == 0
        if i >= 8:
            e2e_ms.append((t1 - t0) * 1000)
    e2e = {"value": round(1000.0 / statistics.mean(e2e_ms) * world, 1), "unit": "tok/s",
           "h2d_bytes_per_step": 4, "d2h_bytes_per_step": layer.hidden * 4,
           "us_per_step": round(statistics.mean(e2e_ms) * 1000, 2),
           "device_us_per_step_back_to_back": round(ms_per_step * 1000, 2),
           "how": "host wall clock per step over 56 steps of ds4g_decode_layers_host from "
                  "Python: the token id from host memory (a launch argument), the layer "
                  "step, the hidden state copied back to pinned host memory and the stream "
                  "synchronised, in one call"}
    del sess, m1

    line = {
        "metric": "decode tok/s (batch 1)", "value": round(value, 1), "unit": "tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "repeats": repeats,
        "timed_steps": args.steps * repeats, "timed_ms": round(total_ms, 2),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based generator)",
        "config": workload_config(layer), "roofline": roofline, "staged_kernels": staged,
        "e2e": e2e, "gpu_launches": int(gpu_launches), "clocks": clk,
        "l2_flushed_each_step": flushed,
    }

    if extra:
        line.update(extra_measurements(pdl, tw, torch, stack, emb, lm, layers, flush, hbm_peak,
                                       bf16_peak, bf16_sus, local))

    if rank == 0:
        rate, n, dt = oracle_decode_rate(layer, n_pre, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(rate, 4), "unit": "tok/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{n} oracle decode steps of the same layer at positions "
                                          f"4096.. ({dt:.1f} s, single thread, {cpu_model()}, "
                                          f"{nproc()} cores present)"}
        print(json.dumps(line), flush=True)
    barrier()
    if dist is not None:
        dist.destroy_process_group()


def extra_measurements(pdl, tw, torch, stack, emb, lm, layers, flush, hbm_peak, bf16_peak,
                       bf16_sus, local=0):
    """Secondary lines, each timed with CUDA events on the session stream and with
    its own clock samples: layer-major prefill, the 8-layer stack with lm_head and
    sampler, the common-prefix resync, and the same decode at depth 43."""
    out = {}
    model = pdl.Model(stack, emb, lm, layers)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()

    # layer-major prefill: 8 layers x 4096 tokens; 3 untimed, then 20 timed back to back
    toks = synth.host_tokens(4096, stack.vocab, stream=31)
    sess = pdl.Session(model, 4200)
    for _ in range(3):
        assert sess.truncate(0) == 0 and sess.prefill(toks) == 0
    torch.cuda.synchronize()
    reps = 20
    clk = ClockSampler(local)
    clk.start()
    ev0.record(stream)
    for _ in range(reps):
        assert sess.truncate(0) == 0 and sess.prefill(toks) == 0
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    assert sess.status() == 0
    t = ev0.elapsed_time(ev1) / 1000.0 / reps
    flops = prefill_flops_per_token_layer(stack) * 4096 * stack.n_layers
    wbytes = sum(np.prod(s) for _, k, s, sg in synth.layer_tensors(stack) if sg) * 2 * stack.n_layers
    out["prefill"] = {
        "metric": "prefill tok/s", "value": round(4096 / t, 1), "unit": "tok/s",
        "workload": "8 layers of the full-width shapes, 4096 prompt tokens, layer-major",
        "ms": round(t * 1000, 3), "reps": reps,
        "roofline": {"bound": "tensor", "achieved": round(flops / t / 1e12, 2),
                     "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(flops / t / 1e12 / bf16_peak, 4),
                     "frac_of_sustained": round(flops / t / 1e12 / bf16_sus, 4),
                     "algorithmic_flops": flops,
                     "memory_floor_ms": round(wbytes / (hbm_peak * 1e9) * 1000, 2),
                     "compute_floor_ms": round(flops / (bf16_peak * 1e12) * 1000, 2),
                     "frac_of_binding_floor": round(max(wbytes / (hbm_peak * 1e9),
                                                        flops / (bf16_peak * 1e12)) / t, 4)},
        "clocks": clocks,
    }
    del sess

    # decode stack + lm_head + top-p sampler: prompt 512, 256 generated tokens
    out["stack"] = sampled_decode_line(pdl, torch, model, stack, 256, local, hbm_peak)
    out["stack"]["metric"] = "decode tok/s (8 layers + lm_head + top-p 0.95, T 0.7)"

    # common-prefix resync: live 16994 -> common 16846 -> canonical 16937
    P = synth.host_tokens(16846, stack.vocab, stream=51)
    live_tail = synth.host_tokens(148, stack.vocab, stream=52)
    new_tail = synth.host_tokens(91, stack.vocab, stream=53)
    new_tail[0] = (live_tail[0] + 1) % stack.vocab
    prompt = np.concatenate([P, new_tail])
    live = pdl.Session(model, 17100)
    assert live.prefill(np.concatenate([P, live_tail])) == 0
    torch.cuda.synchronize()
    cp = live.common_prefix(prompt)
    # the resync itself, then 20 more times (truncating back to the common prefix
    # redoes exactly the same work), timed as one region with its clock samples
    reps = 20
    times = []
    clk = ClockSampler(local)
    clk.start()
    for rep in range(1 + reps):
        ev0.record(stream)
        assert live.truncate(cp) == 0
        assert live.prefill(prompt[cp:]) == 0
        ev1.record(stream)
        torch.cuda.synchronize()
        times.append(ev0.elapsed_time(ev1))
    clocks = clk.stop()
    resync_ms = statistics.mean(times[1:])
    ws2 = torch.empty(pdl.sample_workspace_bytes(stack.vocab), dtype=torch.uint8, device="cuda")
    ids_live = []
    t0 = time.perf_counter()
    for i in range(64):
        tk, _ = pdl.sample(live.logits(), 0.0, 1.0, None, ws2)
        ids_live.append(tk)
        assert live.decode(tk) == 0
    torch.cuda.synchronize()
    dec_s = time.perf_counter() - t0
    logits_live = live.logits().clone()
    del live
    scratch = pdl.Session(model, 17100)
    assert scratch.prefill(prompt) == 0
    ids_scratch = []
    for i in range(64):
        tk, _ = pdl.sample(scratch.logits(), 0.0, 1.0, None, ws2)
        ids_scratch.append(tk)
        assert scratch.decode(tk) == 0
    torch.cuda.synchronize()
    same = ids_live == ids_scratch and torch.equal(logits_live, scratch.logits())
    del scratch
    sfl = prefill_flops_per_token_layer(stack) * 91 * stack.n_layers
    out["resync"] = {
        "metric": "resync latency (truncate + 91-token prefill, 8 layers)",
        "value": round(resync_ms, 3), "unit": "ms", "common_prefix": cp,
        "first_ms": round(times[0], 3), "reps": reps,
        "greedy_decode_tok_s": round(64 / dec_s, 1),
        "matches_scratch_prefill": bool(same),
        "algorithmic_flops": sfl, "clocks": clocks,
    }

    # depth 43 (the pages' decode loop): the 8 generated layers used in turn, each of
    # the 43 layers with its own K/V cache; same sampled workload as the stack line
    deep_shape = stack.with_(name="depth43", n_layers=43)
    deep = pdl.Model(deep_shape, emb, lm, [layers[l % stack.n_layers] for l in range(43)])
    out["depth43"] = sampled_decode_line(pdl, torch, deep, deep_shape, 64, local, hbm_peak)
    out["depth43"]["metric"] = "decode tok/s (43 layers + lm_head + top-p 0.95, T 0.7)"
    out["depth43"]["note"] = ("layer l uses the weights of generated layer l mod 8; each layer "
                              "streams 275 MB per token, more than L2 holds, so the aliasing "
                              "gives no cache advantage")
    return out


def sampled_decode_line(pdl, torch, model, shape, n_gen, local, hbm_peak):
    """Decode with lm_head and top-p sampling after a 512-token prompt: n_gen tokens
    at T 0.7 / top-p 0.95 from a seeded xorshift64* state, timed with CUDA events."""
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sess = pdl.Session(model, 512 + n_gen + 16)
    prompt = synth.host_tokens(512, shape.vocab, stream=41)
    assert sess.prefill(prompt) == 0
    ws = torch.empty(pdl.sample_workspace_bytes(shape.vocab), dtype=torch.uint8, device="cuda")
    state = 0x9E3779B97F4A7C15
    tok, state = pdl.sample(sess.logits(), 0.7, 0.95, state, ws)
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    ev0.record(stream)
    for i in range(n_gen):
        tok, state = sess.decode_sample(tok, 0.7, 0.95, state, ws)   # one call per token
        assert tok >= 0
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = clk.stop()
    assert sess.status() == 0
    t = ev0.elapsed_time(ev1) / 1000.0
    tok_bytes = shape.n_layers * sum(layer_bytes(shape).values()) + lm_head_bytes(shape)
    return {
        "value": round(n_gen / t, 1), "unit": "tok/s", "tokens": n_gen,
        "roofline": {"bound": "hbm", "bytes_per_token": int(tok_bytes),
                     "achieved": round(tok_bytes * n_gen / t / 1e9, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(tok_bytes * n_gen / t / 1e9 / hbm_peak, 4)},
        "note": "one ds4g_decode_sample call per token (layers, lm_head, top-p draw); each "
                "synchronises to return the sampled id to the host",
        "clocks": clocks,
    }


if __name__ == "__main__":
    main()
