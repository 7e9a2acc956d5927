#!/usr/bin/env python
"""Paged-MoE decode benchmark on one GB300 (one JSON line on stdout).

A step is one decode token through the whole 48-layer paged MoE stack: per
layer, routing + device LRU planning, page-in of the missing experts from the
pinned host store, the SiLU-gated expert MLP of the token's top-8 entries and
the top-k sum.  The default workload is the 48-layer bf16 stack (H=2048,
I=768, E=128, top-8) with K=32 resident experts per layer at batch 1; router
logits follow the drifting-bias recipe, so consecutive tokens reuse experts.

Timed passes (each starts from empty slots and replays the same W+K tokens):
  value  graph-replayed decode with inputs already in HBM (CUDA events);
  e2e    the same through host buffers: the token's hidden states and logits
         are copied in from pinned memory and the 48 outputs copied back,
         inside the timed region;
  trace  eager decode with per-kernel CUDA events (libpe's profiler) and
         per-layer counters, used for the roofline figures.
The oracle leg times the CPU reference on the host cores on a bounded sample.

``--impl reference`` times the CPU reference as the reference arm.
Multi-GPU: replicas only (one independent stack per GPU, no collective on
the data path); launch with torchrun, value = sum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from host_paged_expert_gb300 import replicas, synth  # noqa: E402

METRIC = "paged-MoE decode tok/s (48 layers, K resident)"
_T0 = time.time()


def log(msg: str) -> None:
    print(f"[bench {time.time() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)
HBM_NOMINAL_GBS = 7900.0


RESIDENT = "_resident"


def workload(name: str):
    """(shape, batch or chunk tokens, description) of a named workload.  A
    prefill workload with the suffix "_resident" runs with K = E after a
    warm-up that leaves every expert resident: no page-in, the expert GEMMs
    alone."""
    if name.endswith(RESIDENT) and "prefill48_T" in name:
        shape, t, desc = workload(name[: -len(RESIDENT)])
        return (shape.with_slots(shape.num_experts), t,
                desc.split(", K=")[0] + f", K=E={shape.num_experts} (every expert resident after warm-up), "
                + desc.split(", K=")[1].split(", ", 1)[1])
    base = synth.STACK48
    if name == "decode48":
        return base.with_slots(32), 1, "48 layers, H=2048, I=768, E=128, top-8, K=32, bf16 experts, batch 1"
    if name.startswith("graphed48_b"):
        b = int(name[len("graphed48_b"):])
        return base.with_slots(64), b, f"48 layers, H=2048, I=768, E=128, top-8, K=64, bf16, batch {b}"
    if name.startswith("prefill48_T"):
        t = int(name[len("prefill48_T"):])
        return base.with_slots(32), t, f"48 layers, H=2048, I=768, E=128, top-8, K=32, bf16, prefill chunks of {t} tokens"
    if name.startswith("fp8prefill48_T"):
        t = int(name[len("fp8prefill48_T"):])
        return synth.STACK48_FP8, t, f"48 layers, H=2048, I=768, E=128, top-8, K=40, block-FP8, prefill chunks of {t} tokens"
    if name.startswith("int4_48_b"):
        b = int(name[len("int4_48_b"):])
        return synth.STACK48_INT4, b, f"48 layers, H=2048, I=768, E=128, top-8, K=92, GPTQ int4 (group 128), batch {b}"
    if name.startswith("int4prefill48_T"):
        t = int(name[len("int4prefill48_T"):])
        return synth.STACK48_INT4, t, f"48 layers, H=2048, I=768, E=128, top-8, K=92, GPTQ int4 (group 128), prefill chunks of {t} tokens"
    for fmt, shape4, label in (("mxfp4", synth.STACK48_MXFP4, "MXFP4 (E8M0 per 32)"),
                               ("nvfp4", synth.STACK48_NVFP4, "NVFP4 (E4M3 per 16, fp32 per tensor)")):
        if name.startswith(f"{fmt}prefill48_T"):
            t = int(name[len(f"{fmt}prefill48_T"):])
            return shape4, t, f"48 layers, H=2048, I=768, E=128, top-8, K=92, {label}, prefill chunks of {t} tokens"
        if name.startswith(f"{fmt}_48_b"):
            b = int(name[len(f"{fmt}_48_b"):])
            return shape4, b, f"48 layers, H=2048, I=768, E=128, top-8, K=92, {label}, batch {b}"
    if name.startswith("fp8_48_b"):
        b = int(name[len("fp8_48_b"):])
        return synth.STACK48_FP8, b, f"48 layers, H=2048, I=768, E=128, top-8, K=40, block-FP8, batch {b}"
    raise SystemExit(f"unknown workload {name}")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=256)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode48")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-trace", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--probe-bytes", type=int, default=2 << 30)
    p.add_argument("--layers", type=int, default=0,
                   help="profiling only: run a shorter stack of the same layer shape")
    p.add_argument("--repeats", type=int, default=5,
                   help="timed passes of the value and e2e measurements (median reported)")
    p.add_argument("--oracle-leg", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args()


# ------------------------------------------------------------------ inputs


def make_inputs(shape, batch, n_tokens, seed=0):
    zipf = 1.1 if shape.dtype == "fp8" else None
    lg = synth.decode_logits(shape.num_layers, shape.num_experts, n_tokens, batch=batch, seed=seed, zipf_s=zipf)
    lg = np.ascontiguousarray(lg.transpose(1, 0, 2, 3))  # [S, L, B, E]
    hs = synth.hidden_states((n_tokens, shape.num_layers, batch), shape.hidden, seed=seed)  # [S, L, B, H]
    return lg, hs


def touch_host_store(model, nbytes, stream):
    """Read every host-store row once from the GPU before anything is timed.
    The first device access to a page of the mapped store is slow (its
    translation is set up on first use); a long-running server pays that
    once, and without this the first timed pass would pay it for every
    expert it pages in first.  Uses the link probe's copy over the whole
    store; its figures are discarded."""
    model.probe_host_link(nbytes, 1, stream)


def load_weights(model, weights):
    s = weights.shape
    for l in range(s.num_layers):
        for e in range(s.num_experts):
            model.load_expert(l, e, weights.row(l, e))


# ------------------------------------------------------------------ clocks


class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"pe_clocks_dev{device}_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        try:
            return self._summary()
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass

    def _summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ peaks / traffic


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# The sources each timed kernel is compiled from: a DRAM-traffic record is
# reported only while these still hash to the value it was captured on.
KERNEL_SOURCES = {
    "decode_step": ("k_decode.cu", "plan_block.cuh", "pe_device.cuh", "fp8_device.cuh", "int4_device.cuh",
                    "fp4_device.cuh", "pe_internal.h"),
    "prefill_step": ("k_prefill.cu", "tc_sm100.cuh", "pe_device.cuh", "fp8_device.cuh", "int4_device.cuh",
                     "fp4_device.cuh", "pe_internal.h"),
}


def max_miss_rate_for_rate(link_gbs: float, tok_s: float, layers: int, top_k: int, expert_bytes: int) -> float:
    """The largest per-entry miss rate a token rate allows over a link of
    link_gbs if every missed entry moved a whole expert row: the link's bytes
    per token over the bytes of a token whose every routed expert missed
    ("¿Por qué es rápido…?": the pages' bound on the unmeasured miss rate)."""
    return link_gbs * 1e9 / tok_s / (layers * top_k * expert_bytes)


def _code_only(text: str) -> str:
    """Source text without its // and /* */ comments or blank lines, so that
    a comment-only edit keeps a kernel's hash (no string literal in these
    sources holds a comment marker)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(kernel: str):
    files = KERNEL_SOURCES.get(kernel)
    if not files:
        return None
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "host_paged_expert_gb300", "csrc")
    for n in files:
        h.update(_code_only(open(os.path.join(csrc, n)).read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload_name, {}).get(kernel)
        if e and e.get("source_hash") == kernel_source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


# ------------------------------------------------------------------ our arm


def run_ours(args, rep):
    import torch

    from host_paged_expert_gb300 import _lib

    dev, world = rep.local_rank, rep.world
    torch.cuda.set_device(dev)
    shape, B, desc = workload(args.workload)
    if args.layers:
        import dataclasses

        shape = dataclasses.replace(shape, num_layers=args.layers)
        desc = desc.replace("48 layers", f"{args.layers} layers (profiling subset)")
    L, E, H, k = shape.num_layers, shape.num_experts, shape.hidden, shape.top_k
    W, K = args.warmup, args.steps
    S = W + K

    t0 = time.time()
    weights = synth.ExpertWeights(shape, seed=0)
    log("weights pool ready")
    store = None
    if world > 1:
        # one host store for all replicas on the host: replica 0 fills a
        # shared mapping, every replica registers the same pages
        from host_paged_expert_gb300 import shared_store

        made = {}

        def fill(st):
            made["model"] = _lib.PagedMoE(shape, max_tokens=B, device=dev, host_store=st, filled=False)
            load_weights(made["model"], weights)

        path = shared_store.default_path(f"{os.environ.get('MASTER_PORT', '0')}_{args.workload}")
        store = shared_store.open_for_replicas(rep, path, _lib.host_store_bytes(shape), fill)
        model = made.get("model") or _lib.PagedMoE(shape, max_tokens=B, device=dev, host_store=store, filled=True)
        log(f"handle created on the shared host store {path} ({store.nbytes / 1e9:.2f} GB, one copy per host)")
    else:
        model = _lib.PagedMoE(shape, max_tokens=B, device=dev)
        log(f"handle created: arena {model.arena.numel() / 1e9:.2f} GB, host store "
            f"{shape.num_layers * shape.num_experts * model.layout['row_stride'] / 1e9:.2f} GB pinned")
        load_weights(model, weights)
    t_load = time.time() - t0
    log("experts loaded into the host store")
    payload = model.layout["payload_bytes"]

    lg_h, hs_h = make_inputs(shape, B, S, seed=replicas.input_seed(0, rep))
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    with torch.cuda.stream(stream):
        lg_d = torch.from_numpy(lg_h).to(dev)
        hs_d = torch.from_numpy(hs_h.view(np.int16)).view(torch.bfloat16).to(dev)
        x_st = torch.zeros((L, B, H), dtype=torch.bfloat16, device=dev)
        l_st = torch.zeros((L, B, E), dtype=torch.float32, device=dev)
        y_st = torch.zeros((L, B, H), dtype=torch.bfloat16, device=dev)
    stream.synchronize()

    store_bytes = L * E * model.layout["row_stride"]
    touch_host_store(model, store_bytes, stream)
    log("host store touched by the GPU once")
    # host-link probe: pinned host store -> HBM, copy engine and device-side loads
    ce_gbs, kn_gbs = model.probe_host_link(min(args.probe_bytes, store_bytes), 3, stream)
    link_gbs = max(ce_gbs, kn_gbs)
    log(f"host link probe: copy engine {ce_gbs:.1f} GB/s, device loads {kn_gbs:.1f} GB/s")

    xp, lp, yp = x_st.data_ptr(), l_st.data_ptr(), y_st.data_ptr()
    xs, ls, ys = B * H * 2, B * E * 4, B * H * 2

    def launch_token():
        for l in range(L):
            model.forward_ptr(l, xp + l * xs, lp + l * ls, yp + l * ys, B, sp)

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            launch_token()

    def step(t):
        x_st.copy_(hs_d[t], non_blocking=True)
        l_st.copy_(lg_d[t], non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            launch_token()

    def barrier():
        replicas.barrier(rep)

    # ---- value pass: `repeats` timed passes of K tokens, each from empty slots
    def value_pass():
        with torch.cuda.stream(stream):
            model.reset_residency(stream)
            for t in range(W):
                step(t)
            s0 = model.stats(-1)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            barrier()
            torch.cuda.synchronize()
            ev0.record(stream)
            for t in range(W, S):
                step(t)
            ev1.record(stream)
            stream.synchronize()
            torch.cuda.synchronize()
            barrier()
            s1 = model.stats(-1)
        return ev0.elapsed_time(ev1), s0, s1

    runs = []
    with ClockSampler(dev) as clk:
        for _ in range(max(1, args.repeats)):
            runs.append(value_pass())
    clocks = clk.summary()
    run_ms = [replicas.max_over_replicas(rep, r_[0], device=dev) for r_ in runs]
    ms = statistics.median(run_ms)
    s0, s1 = runs[0][1], runs[0][2]
    tok_s = replicas.job_rate(K * B, world, ms)
    spread = {"runs_tok_s": [round(replicas.job_rate(K * B, world, m), 2) for m in run_ms],
              "min": round(replicas.job_rate(K * B, world, max(run_ms)), 2),
              "max": round(replicas.job_rate(K * B, world, min(run_ms)), 2)}
    log(f"value pass: median {ms:.1f} ms for {K} steps -> {tok_s:.1f} tok/s (runs {spread['runs_tok_s']})")
    d = {n: s1[n] - s0[n] for n in ("steps", "waves", "entries", "distinct", "hits", "page_ins")}

    # ---- e2e pass: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        hs_pin = torch.from_numpy(hs_h.view(np.int16)).view(torch.bfloat16).pin_memory()
        lg_pin = torch.from_numpy(lg_h).pin_memory()
        y_pin = torch.empty((S, L, B, H), dtype=torch.bfloat16).pin_memory()

        def step_host(t):
            x_st.copy_(hs_pin[t], non_blocking=True)
            l_st.copy_(lg_pin[t], non_blocking=True)
            if graph is not None:
                graph.replay()
            else:
                launch_token()
            y_pin[t].copy_(y_st, non_blocking=True)

        e_runs = []
        for _ in range(max(1, args.repeats)):
            with torch.cuda.stream(stream):
                model.reset_residency(stream)
                for t in range(W):
                    step_host(t)
                stream.synchronize()
                barrier()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for t in range(W, S):
                    step_host(t)
                b.record(stream)
                stream.synchronize()
                e_runs.append(replicas.max_over_replicas(rep, a.elapsed_time(b), device=dev))
        e_ms = statistics.median(e_runs)
        e2e = {"value": round(replicas.job_rate(K * B, world, e_ms), 2), "unit": "tok/s",
               "h2d_bytes_per_step": L * B * (H * 2 + E * 4), "d2h_bytes_per_step": L * B * H * 2,
               "runs_tok_s": [round(replicas.job_rate(K * B, world, m), 2) for m in e_runs],
               "timed": f"median of {len(e_runs)} passes of {K} steps"}
        log(f"e2e pass: {e2e['value']} tok/s (runs {e2e['runs_tok_s']})")

    # ---- trace pass: per-kernel events, per-layer counters, layer-step latency
    trace = None
    if not args.no_trace:
        peaks = measured_peaks()
        with torch.cuda.stream(stream):
            model.reset_residency(stream)
            for t in range(W):
                step(t)
            stream.synchronize()
            model.profile_enable(True)
            prev = [model.stats(l) for l in range(L)]
            roof_s = 0.0
            lat = []
            for t in range(W, S):
                x_st.copy_(hs_d[t], non_blocking=True)
                l_st.copy_(lg_d[t], non_blocking=True)
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(L + 1)]
                evs[0].record(stream)
                for l in range(L):
                    model.forward_ptr(l, xp + l * xs, lp + l * ls, yp + l * ys, B, sp)
                    evs[l + 1].record(stream)
                stream.synchronize()
                lat += [evs[l].elapsed_time(evs[l + 1]) * 1e3 for l in range(L)]
                cur = [model.stats(l) for l in range(L)]
                for l in range(L):
                    dist = cur[l]["distinct"] - prev[l]["distinct"]
                    pin = cur[l]["page_ins"] - prev[l]["page_ins"]
                    roof_s += max(dist * payload / (peaks["hbm_gbs"] * 1e9), pin * payload / (link_gbs * 1e9))
                prev = cur
            prof = model.profile_read()
            model.profile_enable(False)
        trace = {"prof": prof, "roof_s": roof_s, "lat_us": lat, "peaks": peaks}

    out = {"tok_s": tok_s, "ms": ms, "spread": spread, "clocks": clocks, "d": d, "e2e": e2e, "trace": trace,
           "link": {"copy_engine_gbs": round(ce_gbs, 1), "kernel_gbs": round(kn_gbs, 1)},
           "t_load": t_load, "shape": shape, "B": B, "desc": desc, "payload": payload,
           "layout": model.layout, "lg_h": lg_h, "hs_h": hs_h, "weights": weights,
           "host_store": "shared by all replicas on the host" if store is not None else "pinned by this process"}
    model.close()
    if store is not None:
        replicas.barrier(rep)  # every replica is done with the mapping
        store.close()
    return out


def launches_per_layer_step(shape, B):
    """Kernel launches pe_forward makes for one decode layer-step of B tokens
    (the path choice the library makes from shapes and B)."""
    from host_paged_expert_gb300 import _lib

    ent = B * shape.top_k
    if (ent <= min(64, shape.num_slots) and shape.num_experts <= 256 and shape.num_slots <= 256
            and shape.hidden <= 2048 and shape.intermediate <= 1024):
        return 1  # the whole decode step is one kernel (every format)
    Wm = _lib.max_waves(shape, B)
    route = 1 if B > 32 else 0
    if ent > 64:  # the pipelined prefill step: route, plan, align, gather, step, top-k sum
        return 5 + route
    return route + 1 + 2 * Wm + (1 if Wm > 1 else 0)  # plan, per wave gate/up+page-in and down, sum


# ------------------------------------------------------------------ prefill workload


def run_prefill(args):
    """Prefill chunks through the 48-layer stack (one chunk per step, a few
    distinct chunks cycled).  Eager launches; per-kernel events in a second
    pass give the pipelined step's host-link and tensor-core throughput."""
    import torch

    from host_paged_expert_gb300 import _lib

    shape, T, desc = workload(args.workload)
    if args.layers:
        import dataclasses

        shape = dataclasses.replace(shape, num_layers=args.layers)
        desc = desc.replace("48 layers", f"{args.layers} layers (profiling subset)")
    L, E, H, I, k = shape.num_layers, shape.num_experts, shape.hidden, shape.intermediate, shape.top_k
    W, K = args.warmup, args.steps
    weights = synth.ExpertWeights(shape, seed=0)
    model = _lib.PagedMoE(shape, max_tokens=T)
    load_weights(model, weights)
    log("experts loaded")
    payload = model.layout["payload_bytes"]
    nchunk = 2
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    lgs, hss = [], []
    for c in range(nchunk):
        lgs.append(torch.from_numpy(synth.prefill_logits(L, E, T, seed=c)).cuda())
        hss.append(torch.from_numpy(synth.hidden_states((L, T), H, seed=c, tag=5).view(np.int16)).view(torch.bfloat16).cuda())
    out = torch.empty((L, T, H), dtype=torch.bfloat16, device="cuda")
    touch_host_store(model, L * E * model.layout["row_stride"], stream)
    ce_gbs, kn_gbs = model.probe_host_link(min(args.probe_bytes, L * E * model.layout["row_stride"]), 3, stream)
    link = max(ce_gbs, kn_gbs)
    log(f"link {ce_gbs:.1f} / {kn_gbs:.1f} GB/s")
    torch.cuda.synchronize()

    def step(t):
        lg, hs = lgs[t % nchunk], hss[t % nchunk]
        for l in range(L):
            model.forward_ptr(l, hs[l].data_ptr(), lg[l].data_ptr(), out[l].data_ptr(), T, sp)

    with torch.cuda.stream(stream):
        model.reset_residency(stream)
        for t in range(W):
            step(t)
        s0 = model.stats(-1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        with ClockSampler(0) as clk:
            a.record(stream)
            for t in range(W, W + K):
                step(t)
            b.record(stream)
            stream.synchronize()
        ms = a.elapsed_time(b)
        s1 = model.stats(-1)
        # trace pass: per-kernel events and per-layer counters
        model.reset_residency(stream)
        for t in range(W):
            step(t)
        stream.synchronize()
        model.profile_enable(True)
        prev = [model.stats(l) for l in range(L)]
        roof_s = 0.0
        peaks = measured_peaks()
        for t in range(W, W + K):
            step(t)
            stream.synchronize()
            cur = [model.stats(l) for l in range(L)]
            for l in range(L):
                dist = cur[l]["distinct"] - prev[l]["distinct"]
                pin = cur[l]["page_ins"] - prev[l]["page_ins"]
                roof_s += max(dist * payload / (peaks["hbm_gbs"] * 1e9), pin * payload / (link * 1e9))
            prev = cur
        prof = model.profile_read()
        model.profile_enable(False)
    d = {n: s1[n] - s0[n] for n in ("steps", "waves", "entries", "distinct", "hits", "page_ins")}
    tok_s = K * T / (ms * 1e-3)
    log(f"prefill value pass: {ms:.1f} ms for {K} chunks -> {tok_s:.0f} tok/s")
    ent = d["entries"]
    flops = 2.0 * ent * H * 2 * I + 2.0 * ent * I * H  # both expert GEMMs over every routed entry
    kernels = {}
    for name, v in prof.items():
        if not v["launches"]:
            continue
        e = {"launches": v["launches"], "total_ms": round(v["total_ms"], 3),
             "avg_us": round(v["total_ms"] / v["launches"] * 1e3, 2)}
        if name == "prefill_step":  # page-in and both GEMMs of every wave, pipelined
            gbs = d["page_ins"] * payload / (v["total_ms"] * 1e-3) / 1e9
            tf = flops / (v["total_ms"] * 1e-3) / 1e12
            e.update({"bound": "host_link", "achieved_gbs": round(gbs, 1), "peak_gbs": round(link, 1),
                      "frac": round(gbs / link, 4), "gemm_tflops_over_step": round(tf, 1),
                      "gemm_frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4)})
        if name == "pagein":
            gbs = d["page_ins"] * payload / (v["total_ms"] * 1e-3) / 1e9
            e.update({"bound": "host_link", "achieved_gbs": round(gbs, 1), "peak_gbs": round(link, 1),
                      "frac": round(gbs / link, 4)})
        kernels[name] = e
    line = {"metric": "paged-MoE prefill tok/s (48 layers, K resident)", "value": round(tok_s, 1), "unit": "tok/s",
            "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": round(ms / K, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype, "data": "synthetic",
            "config": {"workload": f"{args.workload}: {desc}", "chunks_cycled": nchunk,
                       "l2": f"inputs larger than L2: each chunk reads ~{d['distinct'] / K * payload / 1e9:.1f} GB "
                             "of expert weights"},
            "clocks": clk.summary(),
            "page_in": {"per_layer_step": round(d["page_ins"] / (K * L), 2), "link_probe_gbs": [round(ce_gbs, 1), round(kn_gbs, 1)],
                        "waves_per_layer_step": round(d["waves"] / (K * L), 2),
                        "distinct_per_layer_step": round(d["distinct"] / (K * L), 2)},
            "layer_roofline": {"frac": round(roof_s * 1e3 / (sum(v["total_ms"] for v in prof.values())), 4),
                               "definition": "sum over layer-steps of max(distinct*expert_bytes/HBM, page_ins*expert_bytes/link) "
                                             "divided by the summed kernel time of the trace pass"},
            "kernels": kernels}
    resident = args.workload.endswith(RESIDENT)
    if resident and "prefill_step" in kernels:
        # every expert resident: the step is the expert GEMMs alone, bound by
        # the tensor pipe or, below the ridge, by streaming the weights once
        kd = kernels["prefill_step"]
        if d["page_ins"]:
            log(f"warning: {d['page_ins']} page-ins in the timed region of a resident workload")
        sec = prof["prefill_step"]["total_ms"] * 1e-3
        wbytes = d["distinct"] * payload  # each routed expert's weights read once per layer-step
        tf = flops / sec / 1e12
        hbm = wbytes / sec / 1e9
        ai = flops / wbytes
        ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        ceiling = min(1.0, ai / ridge)
        tensor = {"achieved": round(tf, 1), "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                  "frac": round(tf / peaks["bf16_tflops_sustained"], 4),
                  "peak_src": f"MEASURED_PEAKS.json bf16_tflops_sustained ({peaks['src']})",
                  "flops_per_launch": round(flops / kd["launches"])}
        hbm_o = {"achieved": round(hbm, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": round(hbm / peaks["hbm_gbs"], 4), "bytes_per_launch": round(wbytes / kd["launches"])}
        bound = "tensor" if ceiling >= 1.0 else "hbm"
        main = tensor if bound == "tensor" else hbm_o
        line["roofline"] = {"kernel": "prefill_step", "bound": bound, "achieved": main["achieved"],
                            "peak": main["peak"], "unit": main["unit"], "frac": main["frac"],
                            "traffic": ncu_traffic("prefill_step", args.workload),
                            "tensor": tensor, "hbm": hbm_o,
                            "arithmetic_intensity_flop_per_byte": round(ai, 1),
                            "ridge_flop_per_byte": round(ridge, 1),
                            "tensor_ceiling_from_ai": round(ceiling, 4),
                            "tensor_frac_of_ceiling": round(tensor["frac"] / ceiling, 4),
                            "definition": "FLOP = 2*entries*H*2I + 2*entries*I*H over the prefill_step kernel's "
                                          "CUDA-event time; bytes = distinct experts x expert bytes"}
        line["metric"] = "paged-MoE prefill tok/s (48 layers, every expert resident)"
        kd.update({"bound": bound, "gemm_tflops": round(tf, 1),
                   "gemm_frac_of_bf16_sustained": tensor["frac"], "weight_gbs": round(hbm, 1)})
        for k_ in ("achieved_gbs", "peak_gbs", "frac"):
            kd.pop(k_, None)
    elif "prefill_step" in kernels:  # the dominant kernel: page-ins over the link with the GEMMs underneath
        kd = kernels["prefill_step"]
        line["roofline"] = {"kernel": "prefill_step", "bound": "host_link", "achieved": kd["achieved_gbs"],
                            "peak": kd["peak_gbs"], "unit": "GB/s", "frac": kd["frac"],
                            "traffic": ncu_traffic("prefill_step", args.workload),
                            "peak_src": "same-run host-link probe (best of copy engine and device loads)",
                            "bytes_per_launch": round(d["page_ins"] * payload / kd["launches"]),
                            "tensor": {"achieved": kd["gemm_tflops_over_step"], "peak": peaks["bf16_tflops"],
                                       "unit": "TFLOP/s", "frac": kd["gemm_frac_of_bf16_peak"]}}
    line["gpu_launches"] = sum(v["launches"] for v in prof.values())  # the trace pass runs the same K chunks
    print(json.dumps(line), flush=True)
    model.close()


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)


def oracle_layer_steps(shape, weights, lg_h, hs_h, budget_s=None, n_steps=None, warm=0):
    """Run the CPU oracle over layer-steps in token order (token t, layer l),
    converting each routed expert's weights from storage every time, until
    ``budget_s`` seconds or ``n_steps`` layer-steps.  Returns (steps, seconds)."""
    from oracle import mlp as omlp

    L = shape.num_layers
    layers = [omlp.PagedLayer(shape.num_experts, shape.num_slots, shape.top_k,
                              (lambda l: (lambda e: omlp.expert_weights(weights.row(l, e), shape.dtype)))(l))
              for l in range(L)]
    done, t0 = 0, None
    total = lg_h.shape[0] * L
    i = 0
    while i < total:
        if i == warm:
            t0 = time.perf_counter()
        t, l = divmod(i, L)
        layers[l].step(hs_h[t, l], lg_h[t, l])
        i += 1
        if i > warm:
            done += 1
            el = time.perf_counter() - t0
            if (budget_s is not None and el >= budget_s) or (n_steps is not None and done >= n_steps):
                return done, el
    return done, time.perf_counter() - t0 if t0 else 0.0


def blas_threads():
    """Threads the BLAS under numpy actually uses: threadpoolctl where it is
    installed, else the OpenBLAS library numpy loaded, asked directly."""
    try:
        import threadpoolctl

        n = sum(i["num_threads"] for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas")
        if n:
            return int(n)
    except Exception:
        pass
    try:
        import ctypes

        libs = sorted({ln.split()[-1] for ln in open("/proc/self/maps") if "openblas" in ln.lower()
                       and ln.split()[-1].startswith("/")})
        for path in libs:
            lib = ctypes.CDLL(path)
            for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                        "openblas_get_num_threads"):
                fn = getattr(lib, sym, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    return int(fn())
    except Exception:
        pass
    return None


ONE_CORE_ENV = {"OPENBLAS_NUM_THREADS": "1", "OMP_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def oracle_leg(args):
    """The oracle on this process's cores over the workload's steady state
    (after one whole token of warm-up); prints one JSON object.  Run by
    oracle_one_core() in a fresh process pinned to one core."""
    shape, B, _ = workload(args.workload)
    weights = synth.ExpertWeights(shape, seed=0)
    L = shape.num_layers
    warm = max(1, args.warmup)
    lg_h, hs_h = make_inputs(shape, B, warm + int(args.cpu_seconds * 4 / L) + 8)
    steps, sec = oracle_layer_steps(shape, weights, lg_h, hs_h, budget_s=args.cpu_seconds, warm=warm * L)
    print(json.dumps({"steps": steps, "seconds": sec, "tok_s": steps / L * B / sec,
                      "blas_threads": blas_threads(), "cores": len(os.sched_getaffinity(0))}), flush=True)


def oracle_one_core(workload_name: str, seconds: float, warm_tokens: int = 1):
    """The same oracle leg in a fresh interpreter confined to one core, with
    one BLAS thread (a new process, never a fork of this CUDA process)."""
    env = dict(os.environ, **ONE_CORE_ENV)
    cpu = sorted(os.sched_getaffinity(0))[0]
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-leg", "--workload", workload_name,
           "--cpu-seconds", str(seconds), "--warmup", str(warm_tokens)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=seconds * 6 + 120,
                           preexec_fn=lambda: os.sched_setaffinity(0, {cpu}))
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as exc:  # reported, not fatal: the GPU line stands on its own
        return {"error": f"{type(exc).__name__}: {exc}"}


def cpu_baseline_entry(shape, B, weights, lg_h, hs_h, seconds, workload_name, warm_tokens):
    """cpu_baseline: the oracle at all cores and at one core, steady state:
    from the token the GPU arm's timed passes start at (after its warm-up)."""
    L = shape.num_layers
    warm_tokens = max(1, warm_tokens)
    steps, sec = oracle_layer_steps(shape, weights, lg_h, hs_h, budget_s=seconds, warm=warm_tokens * L)
    one = oracle_one_core(workload_name, seconds, warm_tokens)
    out = {"value": round(steps / L * B / sec, 4), "unit": "tok/s", "cores": len(os.sched_getaffinity(0)),
           "blas_threads": blas_threads(), "kind": "oracle",
           "sample": f"{steps} layer-steps (token-major) from token {warm_tokens} on, after {warm_tokens} "
                     f"warm-up tokens, {sec:.1f} s, fp64 numpy"}
    if "tok_s" in one:
        out["one_core"] = {"value": round(one["tok_s"], 4), "unit": "tok/s", "cores": one["cores"],
                           "blas_threads": one["blas_threads"],
                           "sample": f"{one['steps']} layer-steps after one token of warm-up, "
                                     f"{one['seconds']:.1f} s, one core"}
    else:
        out["one_core"] = one
    return out


def run_reference(args, rep):
    if not rep.is_root:  # the oracle arm runs once, on rank 0
        return
    shape, B, desc = workload(args.workload)
    weights = synth.ExpertWeights(shape, seed=0)
    L = shape.num_layers
    # a step is what a step of our arm is: one token (all L layer-steps) of
    # the same workload, after W tokens of warm-up (steady state)
    lg_h, hs_h = make_inputs(shape, B, args.warmup + args.steps)
    steps, sec = oracle_layer_steps(shape, weights, lg_h, hs_h, n_steps=args.steps * L, warm=args.warmup * L)
    tok_s = steps / L * B / sec
    line = {"impl": "reference", "metric": METRIC, "value": round(tok_s, 4), "unit": "tok/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / (steps / L) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{args.workload}: {desc}",
                                            "step": f"one token through the {L} layers of the CPU oracle"},
            "cpu_baseline": {"value": round(tok_s, 4), "unit": "tok/s", "cores": len(os.sched_getaffinity(0)),
                             "blas_threads": blas_threads(), "kind": "oracle",
                             "sample": f"tokens {args.warmup}..{args.warmup + args.steps - 1} of the workload "
                                       f"({steps} layer-steps) after {args.warmup} warm-up tokens"},
            "e2e": {"value": round(tok_s, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main


def main():
    args = parse()
    if args.oracle_leg:
        oracle_leg(args)
        return
    rep = replicas.from_env()
    rank, world, local_rank = rep.rank, rep.world, rep.local_rank
    if args.impl == "reference":
        run_reference(args, rep)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    import torch

    if world > 1:
        torch.cuda.set_device(local_rank)
        replicas.init(rep, "nccl", device=torch.device("cuda", local_rank))
    if "prefill48_T" in args.workload:
        if world > 1:
            raise SystemExit("prefill workloads time one replica; run them with --gpus 1")
        run_prefill(args)
        return
    r = run_ours(args, rep)
    if rank != 0:
        replicas.finish(rep)
        return
    shape, B = r["shape"], r["B"]
    L = shape.num_layers
    lay = r["layout"]
    d = r["d"]
    line = {
        "metric": METRIC, "value": round(r["tok_s"], 2), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["ms"] / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype,
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {r['desc']}", "global_batch": B * world,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "host_store": r["host_store"],
                   "graph": not args.no_graph,
                   "host_store_touched": "every row read once by the GPU before timing (first-touch cost excluded)",
                   "l2": "inputs larger than L2: each step streams ~%.1f GB of expert weights"
                         % (d["distinct"] / args.steps * r["payload"] / 1e9)},
        "clocks": r["clocks"],
        "value_spread": dict(r["spread"], timed=f"value = median of {len(r['spread']['runs_tok_s'])} passes, "
                                                 f"each {args.warmup} warm-up and {args.steps} timed steps "
                                                 "from empty slots"),
        "gpu_launches": args.steps * L * launches_per_layer_step(shape, B),  # per timed pass of K steps
        "page_in": {"per_token": round(d["page_ins"] / args.steps, 3),
                    "miss_rate_per_entry": round(d["page_ins"] / max(1, d["entries"]), 4),
                    "miss_rate_per_distinct": round(d["page_ins"] / max(1, d["distinct"]), 4),
                    "bytes_per_token": int(d["page_ins"] / args.steps * r["payload"]),
                    "random_routing_miss_rate": round(1.0 - shape.num_slots / shape.num_experts, 4),
                    "max_miss_rate_for_rate": round(max_miss_rate_for_rate(
                        max(r["link"]["copy_engine_gbs"], r["link"]["kernel_gbs"]), r["tok_s"] / world, L,
                        shape.top_k, r["payload"]), 4),
                    "link_probe_gbs": r["link"]},
        "setup_s": round(r["t_load"], 1),
    }
    if r["e2e"]:
        line["e2e"] = r["e2e"]
    tr = r["trace"]
    if tr:
        peaks = tr["peaks"]
        prof = tr["prof"]
        link = max(r["link"]["copy_engine_gbs"], r["link"]["kernel_gbs"])
        alg = {"pagein": d["page_ins"] * r["payload"],
               "gateup_pagein": d["page_ins"] * r["payload"],
               "decode_step": d["page_ins"] * r["payload"],
               "gateup": d["distinct"] * (lay["w13_bytes"] + lay["s13_bytes"]),
               "down": d["distinct"] * (lay["w2_bytes"] + lay["s2_bytes"])}
        kernels = {}
        for name, v in prof.items():
            if not v["launches"]:
                continue
            ent = {"launches": v["launches"], "total_ms": round(v["total_ms"], 3),
                   "avg_us": round(v["total_ms"] / v["launches"] * 1e3, 2)}
            if name in alg:
                on_link = name in ("pagein", "gateup_pagein", "decode_step")
                bound = "host_link" if on_link else "hbm"
                peak = link if on_link else peaks["hbm_gbs"]
                ach = alg[name] / (v["total_ms"] * 1e-3) / 1e9 if v["total_ms"] > 0 else 0.0
                ent.update({"bound": bound, "achieved_gbs": round(ach, 1), "peak_gbs": round(peak, 1),
                            "frac": round(ach / peak, 4),
                            "bytes_per_launch": round(alg[name] / v["launches"])})
            kernels[name] = ent
        dom = max((n for n in kernels if n in alg), key=lambda n: kernels[n]["total_ms"])
        kd = kernels[dom]
        line["roofline"] = {"kernel": dom, "bound": kd["bound"], "achieved": kd["achieved_gbs"],
                            "peak": kd["peak_gbs"], "unit": "GB/s", "frac": kd["frac"],
                            "traffic": ncu_traffic(dom, args.workload),
                            "peak_src": ("same-run host-link probe (best of copy engine and device loads)"
                                         if kd["bound"] == "host_link"
                                         else f"MEASURED_PEAKS.json hbm_gbs ({peaks['src']})"),
                            "bytes_per_launch": kd["bytes_per_launch"],
                            "source": "eager trace pass (per-kernel CUDA events)"}
        if dom == "decode_step" and not args.no_graph and launches_per_layer_step(shape, B) == 1:
            # one kernel per layer-step: in the graph-timed value pass its
            # average duration is at most the pass time / (K*L), gaps included
            avg_us = r["ms"] * 1e3 / (args.steps * L)
            ach = d["page_ins"] * r["payload"] / (r["ms"] * 1e-3) / 1e9
            line["roofline"].update({"achieved": round(ach, 1), "frac": round(ach / kd["peak_gbs"], 4),
                                     "bytes_per_launch": round(d["page_ins"] * r["payload"] / (args.steps * L)),
                                     "avg_launch_us": round(avg_us, 2),
                                     "source": "graph-replayed value pass (median pass): one decode_step launch "
                                               "per layer-step, average duration = pass time / (steps x layers), "
                                               "launch gaps included",
                                     "eager_trace": {"achieved": kd["achieved_gbs"], "frac": kd["frac"],
                                                     "avg_launch_us": kd["avg_us"]}})
        line["kernels"] = kernels
        lat = sorted(tr["lat_us"])
        line["layer_step_us"] = {"p50": round(lat[len(lat) // 2], 1), "p99": round(lat[int(len(lat) * 0.99)], 1),
                                 "mean": round(sum(lat) / len(lat), 1), "source": "eager trace pass"}
        line["layer_roofline"] = {
            "frac": round(tr["roof_s"] * 1e3 / r["ms"], 4),
            "roofline_ms_per_step": round(tr["roof_s"] * 1e3 / args.steps, 4),
            "definition": "sum over layer-steps of max(distinct*expert_bytes/HBM, page_ins*expert_bytes/link) "
                          "divided by the graph-timed value pass",
            "hbm_gbs": peaks["hbm_gbs"], "link_gbs": link}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_entry(shape, B, r["weights"], r["lg_h"], r["hs_h"], args.cpu_seconds,
                                                  args.workload, args.warmup)
    print(json.dumps(line), flush=True)
    replicas.finish(rep)


if __name__ == "__main__":
    main()
