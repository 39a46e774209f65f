"""Decode throughput with eviction on one GB300 (or N replicas under torchrun).

A step is one token for the whole batch through every layer: n_layers calls
of kvevict_decode_step (attention + score + evict + in-place insert), each one
kernel launch (Random adds a cut launch every r steps). Inputs for the timed
steps are generated on the device beforehand; the per-layer KV working set
(>1 GB for the default workload) is far larger than the 129 MB L2, so no L2
flush is needed between steps.

Default workload: StreamingLLM sink + window (4 + 1020 slots), bf16, B=64,
32 layers x 32 heads, head_dim 128, steady state (cache full).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import configs, synth, traffic  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "kv_cache_eviction_decode_gb300", "csrc")


# The decode kernel's device sources; a committed traffic figure counts only
# for the kernel built from these.
DECODE_SOURCES = ("decode_bf16.cu", "decode_dispatch.h", "decode_f32.cu", "decode_kernel.cuh", "device_common.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(workload: str):
    """DRAM bytes per decode launch from a committed ncu capture, or None if
    absent or taken on other kernel sources."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed helpers (one process per GPU; replicas, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host cores, on a sample
# ---------------------------------------------------------------------------

def oracle_sampler(w, n_units: int, target_s: float, max_steps: int = 4096):
    """Builds n_units units of one layer in the oracle, already in steady state
    (prompt or fill built by the oracle's own prefill), and sizes one sample to
    as many decode steps as fit ~target_s. Returns (sample, unit_steps, threads,
    description): sample() runs one sample and returns its seconds."""
    import numpy as np
    import oracle
    P = w.prompt_len if w.prompt_len else w.capacity  # stream-from-empty workloads: fill the cache first
    ids = []
    for i in range(n_units):
        seq, h = divmod(i, w.n_kv_heads)
        ids.append((seq % w.batch, h))
    units = []
    for seq, h in ids:
        x = synth.UnitInputs(w, seq, 0, h, 1, P)
        u = oracle.Unit.for_workload(w, seq, 0, h)
        u.prefill(x.prompt_k, x.prompt_v)
        if w.policy == configs.POLICY_RANDOM:  # reach the post-cut steady state with staged tokens
            z = np.zeros(w.head_dim, np.float32)
            for _ in range(w.budget + w.r):
                u.stage(z, z)
                u.commit(u.choose())
        units.append(u)
    threads = min(oracle.online_cores(), n_units)

    def stacked(xs, a, b):
        return (np.stack([x.q[a:b] for x in xs]), np.stack([x.k_new[a:b] for x in xs]),
                np.stack([x.v_new[a:b] for x in xs]))

    def timed(qkv):
        t0 = time.perf_counter()
        oracle.run(units, *qkv, n_threads=threads)
        return time.perf_counter() - t0

    one = timed(stacked([synth.UnitInputs(w, seq, 0, h, 1, P) for seq, h in ids], 0, 1))
    M = int(max(1, min(max_steps, target_s / max(one, 1e-6))))
    # the same M inputs for every sample: a unit's work per step does not depend on them
    qkv = stacked([synth.UnitInputs(w, seq, 0, h, 1 + M, P) for seq, h in ids], 1, 1 + M)
    start = "the cache after the prompt" if w.policy == configs.POLICY_H2O_POOLS else "a full cache"
    desc = (f"{n_units} units of one layer (of {w.batch * w.n_kv_heads} per layer, {w.n_layers} layers) "
            f"x {M} decode steps from {start}")
    return (lambda: timed(qkv)), n_units * M, threads, desc


def oracle_sample_rate(w, n_units: int, target_s: float, max_steps: int = 4096):
    """One timed sample of the oracle (see oracle_sampler). Returns
    (unit_steps_per_s, threads, description, seconds)."""
    sample, work, threads, desc = oracle_sampler(w, n_units, target_s, max_steps)
    dt = sample()
    return work / dt, threads, f"{desc}, {dt:.1f} s", dt


def cpu_tokens_per_s(w, unit_steps_per_s: float) -> float:
    units_per_token_step = w.batch * w.n_kv_heads * w.n_layers
    return unit_steps_per_s / units_per_token_step * w.batch


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def steady_state(cache, w, device):
    """Brings every layer to the workload's steady state before timing."""
    import torch
    if w.policy == configs.POLICY_SINK_WINDOW and w.prompt_len == 0:
        # The sink-window state depends on positions only: a full cache from
        # the prefill of the first C tokens equals C streamed decode steps.
        P = w.capacity
    else:
        P = w.prompt_len
    for layer in range(w.n_layers):
        if P:
            K, V = synth.device_prompt(w, layer, device, P)
            cache.prefill(layer, K, V)
            del K, V
    torch.cuda.synchronize(device)
    return P


def run_ours(args, w, rank, world, device, steps=None, warmup=None, extras=True):
    """Times `steps` token-steps (after `warmup` untimed) of the workload at
    steady state. extras: also the isolated launch times, the end-to-end
    host-buffer run and (two-pool H2O) the held fraction."""
    import torch
    from kv_cache_eviction_decode_gb300 import KVEvictCache, lib

    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        cache = KVEvictCache.from_workload(w, device=device, stream=stream)
        if args.tail_split >= 0:
            cache.set_tail_split(bool(args.tail_split))
        if args.alias != -1:
            cache.set_partials_alias(args.alias)
        if args.split:
            cache.set_split(args.split)
        if args.clusters:
            cache.set_clusters(args.clusters)
        if args.path:
            cache.set_path(args.path)
        if args.ring:
            cache.set_ring(args.ring)
        P = steady_state(cache, w, device)
        L, B, Hq, Hkv, D = w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
        n_pre = 0
        if args.no_preroll:
            pass
        elif w.policy == configs.POLICY_RANDOM:  # pass the first cut
            n_pre = w.budget + w.r
        elif w.policy in (configs.POLICY_H2O, configs.POLICY_H2O_BLOCK) and P < w.capacity:
            # fill the cache: every timed step evicts (H2O_BLOCK: releases a block every r steps)
            n_pre = w.capacity - P
        elif w.policy == configs.POLICY_H2O_POOLS and (w.hh_threshold >= 0 or P < w.capacity):
            # the prompt leaves the recent pool only; the heavy-hitter pool fills with
            # the promotions of the next steps (held counts are read after timing)
            n_pre = 2 * w.capacity
        n_win = warmup + steps
        q, kn, vn = synth.device_window(w, P + n_pre, n_win, device)
        out = torch.empty((2, L, B, Hq, D), dtype=q.dtype, device=device)
        Lb = lib()
        h = cache.h
        dec = Lb.kvevict_decode_step

        def token_step(s):
            for layer in range(L):
                rc = dec(h, layer, q[s, layer].data_ptr(), kn[s, layer].data_ptr(), vn[s, layer].data_ptr(),
                         out[s & 1, layer].data_ptr())
                if rc:
                    raise RuntimeError(f"kvevict_decode_step failed: {rc}")

        for i in range(n_pre):  # Random: generated tokens up to the first cut
            token_step(i % n_win)
        for s in range(warmup):
            token_step(s)
        stream.synchronize()
        launches_before = cache.stats()
        barrier(device)
        torch.cuda.synchronize(device)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        graph = None
        if args.graph:
            # the timed token-steps captured once on the handle's stream (each
            # launch with its own step's arguments) and replayed once
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for s in range(warmup, n_win):
                    token_step(s)
            stream.synchronize()
        with ClockSampler(device.index) as clk:
            # the device sleeps ~1 ms before the start event, so the host has
            # queued the first steps when it is recorded: the timed region
            # holds the steps' own work, not the first launch's host latency
            torch.cuda._sleep(2_000_000)
            ev0.record(stream)
            if graph is not None:
                with torch.cuda.stream(stream):
                    graph.replay()
            else:
                for s in range(warmup, n_win):
                    token_step(s)
            ev1.record(stream)
            ev1.synchronize()
        del graph
        torch.cuda.synchronize(device)
        barrier(device)
        err = cache.check()
        if err:
            raise RuntimeError(f"device error word {err:#x}")
        st = cache.stats()
        dt_ms = ev0.elapsed_time(ev1)
        dt_ms = reduce_max(dt_ms, device)
        decode_launches = st["decode_steps"] - launches_before["decode_steps"]
        cut_launches = st["cuts"] - launches_before["cuts"]

        # validation mode, after the timed region: the H2O decisions whose runner-up
        # candidate was within 1e-5 relative of the evicted token (kvevict_set_tie_audit)
        near = None
        if w.policy == configs.POLICY_H2O and args.tie_steps > 0:
            n_dec = 0
            cache.set_tie_audit(True)
            for i in range(args.tie_steps):
                token_step((warmup + i) % n_win)
            stream.synchronize()
            cache.set_tie_audit(False)
            n_dec = args.tie_steps * L * B * Hkv  # at steady state every step evicts in every unit
            cnt = cache.stats()["near_ties"]
            near = {"count": cnt, "decisions": n_dec, "rate": cnt / n_dec, "steps": args.tie_steps,
                    "rule": "runner-up candidate within 1e-5 relative of the evicted token's stored score"}

        # isolated kernel time of single launches (events around each), for context
        iso = []
        for s in range(min(8, n_win) if extras else 0):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dec(h, s % L, q[s, s % L].data_ptr(), kn[s, s % L].data_ptr(), vn[s, s % L].data_ptr(),
                out[0, 0].data_ptr())
            e1.record(stream)
            e1.synchronize()
            iso.append(e0.elapsed_time(e1))

        # end to end through the host-buffer C-ABI call
        e2e = None
        if extras and not args.no_e2e:
            qh = q[:2].cpu().pin_memory()
            kh = kn[:2].cpu().pin_memory()
            vh = vn[:2].cpu().pin_memory()
            oh = torch.empty((L, B, Hq, D), dtype=q.dtype).pin_memory()
            # every layer-step through the host-buffer call that does not wait (inputs
            # in on the copy stream while the previous step runs, output back), one
            # kvevict_sync per token-step: its outputs are on the host when it returns
            dech = Lb.kvevict_decode_step_host_async
            n_e2e = max(2, min(steps, 10))
            barrier(device)
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            for s in range(n_e2e):
                for layer in range(L):
                    rc = dech(h, layer, qh[s & 1, layer].data_ptr(), kh[s & 1, layer].data_ptr(),
                              vh[s & 1, layer].data_ptr(), oh[layer].data_ptr())
                    if rc:
                        raise RuntimeError(f"kvevict_decode_step_host_async failed: {rc}")
                rc = Lb.kvevict_sync(h)
                if rc:
                    raise RuntimeError(f"kvevict_sync failed: {rc}")
            e2e_s = reduce_max(time.perf_counter() - t0, device)
            h2d = L * (q[0, 0].numel() + kn[0, 0].numel() + vn[0, 0].numel()) * q.element_size()
            d2h = L * out[0, 0].numel() * q.element_size()
            in_place = all(Lb.kvevict_host_buffer_mapped(t.data_ptr()) for t in (qh, kh, vh, oh))
            e2e = {"value": world * B * n_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "steps": n_e2e,
                   "path": ("pinned host buffers read and written in place by the kernels over the CPU-GPU link"
                            if in_place else "staging copies on copy-in/copy-out streams")}
        held = None
        if w.policy == configs.POLICY_H2O_POOLS:  # data-dependent occupancy: the mean held fraction
            held = float(np.mean([(cache.slot_positions(layer) >= 0).float().mean().item() for layer in range(L)]))
        cache.close()
    return dict(dt_ms=dt_ms, clocks=clk.summary(), decode_launches=decode_launches, cut_launches=cut_launches,
                iso_ms=iso, e2e=e2e, split=st["split"], clusters=st["clusters"], tensor_cores=st["tensor_cores"],
                ring_stages=st["ring_stages"], held=held, tail_split=st["tail_split"],
                partials_alias=st["partials_alias"], near_ties=near)


# ---------------------------------------------------------------------------
# The score-keeping and Random workloads, measured beside the headline
# ---------------------------------------------------------------------------

# (alias, steps per repeat, repeats): the GQA layer is one ~0.1 ms launch per
# step, so it is timed as several repeats, each on a fresh one-layer handle
# (its own prompt; every repeat within the workload's 512 decode steps)
EXTRA_WORKLOADS = (("h2o_mha", None, 1), ("h2o_gqa", 200, 5), ("random", None, 1), ("h2o_reasoning", None, 1))


def workload_summary(w, r, steps):
    """One workload's figures from a run_ours result."""
    dt_s = r["dt_ms"] / 1e3
    launches = max(1, r["decode_launches"])
    avg = dt_s / launches
    layer_bytes = traffic.steady_layer_step_bytes(w)
    achieved = layer_bytes / avg / 1e9
    peak, peak_kind = measured_hbm_peak()
    tr = profiled_traffic(w.name)
    return {"tokens_per_s": w.batch * steps / dt_s, "layer_step_us": 1e6 * avg,
            "algorithmic_bytes_per_launch": layer_bytes, "achieved_gbs": achieved, "peak_gbs": peak,
            "peak_kind": peak_kind, "frac": achieved / peak, "frac_of_8TBs": achieved / 8000.0,
            "dram_traffic_over_algorithmic": (tr / layer_bytes) if tr else None,
            "steps": steps, "gpu_launches": r["decode_launches"] + r["cut_launches"],
            "split": r["split"], "tail_split": bool(r["tail_split"]), "partials_alias": bool(r["partials_alias"]),
            "clusters": r["clusters"], "ring_stages": r["ring_stages"], "clocks": r["clocks"],
            "near_ties": r["near_ties"]}


def extra_workloads(args, rank, world, device):
    """Every score-keeping configuration and Random at full shape, each with
    its own clock record: per layer-step time, algorithmic bytes per launch,
    fractions of the measured copy peak and of 8 TB/s, and the ncu DRAM bytes
    over the algorithmic bytes where a capture of the current kernel exists."""
    res = {}
    for name, rep_steps, reps in EXTRA_WORKLOADS:
        w = configs.get(name)
        if reps == 1:
            r = run_ours(args, w, rank, world, device, extras=False)
            res[w.name] = workload_summary(w, r, args.steps)
            continue
        one = w.with_(n_layers=1)  # GQA: one layer; a fresh handle and prompt per repeat
        runs = [run_ours(args, one, rank, world, device, steps=rep_steps, extras=False) for _ in range(reps)]
        per = [workload_summary(one, r, rep_steps) for r in runs]
        us = sorted(p["layer_step_us"] for p in per)
        best = min(per, key=lambda p: p["layer_step_us"])
        mid = sorted(per, key=lambda p: p["layer_step_us"])[len(per) // 2]
        mhz = [p["clocks"]["sm_mhz"] for p in per if p["clocks"]["sm_mhz"] is not None]
        e = dict(mid)
        e.update({"repeats": reps, "steps_per_repeat": rep_steps, "layer_step_us_median": mid["layer_step_us"],
                  "layer_step_us_min": best["layer_step_us"], "layer_step_us_all": us,
                  "frac_min_time": best["frac"], "sm_mhz_median": statistics.median(mhz) if mhz else None,
                  "clocks": {"sm_mhz": statistics.median(mhz) if mhz else None,
                             "sm_max_mhz": max((p["clocks"]["sm_max_mhz"] or 0) for p in per) or None,
                             "reasons": sorted({x for p in per for x in p["clocks"]["reasons"]}),
                             "samples": sum(p["clocks"]["samples"] for p in per)},
                  "note": "median repeat; each repeat a fresh one-layer handle, steps within the 512 decode steps"})
        res[w.name] = e
    return res


# ---------------------------------------------------------------------------
# Q-seeded prefill (H2O): prompt scoring on the tensor cores, then the cut
# ---------------------------------------------------------------------------

def prefill_flops(w, P: int) -> int:
    """Algorithmic FLOPs of one layer's scoring: two passes over the causal
    triangle of q.k (2 d flops per product) for every query head."""
    return w.batch * w.n_q_heads * 2 * P * (P + 1) * w.head_dim


def measured_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def oracle_prefill_sampler(w, P: int, target_s: float):
    """One sample = one oracle unit (one sequence's KV head) scored per host
    core, in parallel, timed as the oracle stands. A unit whose full prompt
    would take more than about target_s is sampled on a shorter prompt and
    scaled by the FLOP ratio (said in the description). Returns (sample,
    units per sample, threads, description, scale): sample() runs one sample
    and returns its seconds; call sample.close() when done."""
    import concurrent.futures as cf
    import oracle
    threads = oracle.online_cores()
    G, d = w.group, w.head_dim
    rng = np.random.default_rng(w.seed)
    # per-unit cost model from the oracle's own loop: G * P^2 / 2 rows-by-keys products of d
    Pt = P
    est = G * P * P / 2 * d / 4e8  # about 0.4 G multiply-adds per second per core
    if est > target_s:
        Pt = max(256, int(P * (target_s / est) ** 0.5))
    inputs = [(rng.standard_normal((G, Pt, d)).astype(np.float32), rng.standard_normal((Pt, d)).astype(np.float32),
               rng.standard_normal((Pt, d)).astype(np.float32)) for _ in range(threads)]

    def unit(i):
        u = oracle.Unit(oracle.H2O, w.n_sink, w.n_heavy, w.n_recent, w.budget, 0, 0, G, d)
        u.prefill_scored(*inputs[i])

    ex = cf.ThreadPoolExecutor(max_workers=threads)

    def sample():
        t0 = time.perf_counter()
        list(ex.map(unit, range(threads)))
        return time.perf_counter() - t0

    sample.close = ex.shutdown
    scale = (Pt * (Pt + 1)) / (P * (P + 1))
    desc = f"{threads} units (one sequence x KV head) of prompt {Pt} per round"
    if Pt != P:
        desc += f"; scaled to prompt {P} by the FLOP ratio {scale:.4g}"
    return sample, threads, threads, desc, scale


def oracle_prefill_rate(w, P: int, target_s: float):
    """Oracle units scored per second over about target_s (see oracle_prefill_sampler)."""
    sample, n, threads, desc, scale = oracle_prefill_sampler(w, P, target_s / 2)
    dt, done = 0.0, 0
    while dt < target_s or done == 0:
        dt += sample()
        done += n
    sample.close()
    return done / dt * scale, threads, f"{done // n} rounds of {desc}, {dt:.1f} s"


def run_reference_samples(args, one_round, n):
    """The reference arm's W untimed and K timed bench steps. A step repeats
    one_round (n units, returning its seconds) until it has run for
    reference_step_seconds; returns (units per second over the timed steps,
    their summed seconds)."""
    target = reference_step_seconds(args)

    def step():
        dt, units = 0.0, 0
        while dt < target or units == 0:
            dt += one_round()
            units += n
        return dt, units

    for _ in range(args.warmup):
        step()
    timed = [step() for _ in range(args.steps)]
    secs = sum(t for t, _ in timed)
    return sum(u for _, u in timed) / secs, secs


def reference_step_seconds(args) -> float:
    """Seconds per reference bench step: half of --cpu-seconds (at least 1 s),
    capped so that the whole run takes about 150 s."""
    return min(max(1.0, args.cpu_seconds / 2), max(0.2, 150.0 / (args.steps + args.warmup)))


def prefill_phase(args, w, rank, world, local):
    metric = "Q-seeded prefill prompt tokens/s (H2O scoring + cut); tensor TFLOP/s vs bf16 peak"
    P = w.prompt_len
    if w.policy != configs.POLICY_H2O or w.dtype != configs.DTYPE_BF16 or P < 1:
        raise SystemExit("--phase prefill needs an H2O bf16 workload with a prompt")
    cfg = {"workload": w.name, "phase": "prefill_scored", "policy": "h2o", "batch": w.batch, "q_heads": w.n_q_heads,
           "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "prompt_len": P, "budget": w.budget,
           "n_sink": w.n_sink, "n_heavy": w.n_heavy, "n_recent": w.n_recent}
    flops = prefill_flops(w, P)
    tokens = w.batch * P  # prompt tokens per call (one layer)
    if args.impl == "reference":
        if rank != 0:
            return
        sample, n, threads, desc, scale = oracle_prefill_sampler(w, P, reference_step_seconds(args))
        rate, tsum = run_reference_samples(args, sample, n)
        sample.close()
        v = rate * scale * P / w.n_kv_heads
        desc = (f"{desc}; rounds of them repeated for {reference_step_seconds(args):.1f} s per bench step, "
                f"{args.steps} timed steps after {args.warmup} untimed, {tsum:.1f} s")
        print(json.dumps({"impl": "reference", "metric": metric, "value": v, "unit": "tokens/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * tokens / v,
                          "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": cfg,
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                           "sample": desc},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    import torch
    from kv_cache_eviction_decode_gb300 import KVEvictCache
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    n_calls = args.warmup + args.steps
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        Q = synth.device_prompt_queries(w, 0, device, P)
        K, V = synth.device_prompt(w, 0, device, P)
        # one layer per call: the scored prefill fills an empty layer
        cache = KVEvictCache.from_workload(w.with_(n_layers=n_calls + (0 if args.no_e2e else 2)), device=device,
                                           stream=stream)
        ws = torch.empty(cache.prefill_scored_workspace_bytes(P), dtype=torch.uint8, device=device)
        for i in range(args.warmup):
            cache.prefill_scored(i, Q, K, V, workspace=ws)
        stream.synchronize()
        barrier(device)
        torch.cuda.synchronize(device)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(device.index) as clk:
            ev0.record(stream)
            for i in range(args.warmup, n_calls):
                cache.prefill_scored(i, Q, K, V, workspace=ws)
            ev1.record(stream)
            ev1.synchronize()
        torch.cuda.synchronize(device)
        barrier(device)
        err = cache.check()
        if err:
            raise RuntimeError(f"device error word {err:#x}")
        dt_ms = reduce_max(ev0.elapsed_time(ev1), device)
        e2e = None
        if not args.no_e2e:
            # through the binding from pinned host buffers: Q/K/V in, the slot table out
            Qh, Kh, Vh = Q.cpu().pin_memory(), K.cpu().pin_memory(), V.cpu().pin_memory()
            pos_h = torch.empty((w.batch, w.n_kv_heads, cache.capacity), dtype=torch.int32).pin_memory()
            Qd, Kd, Vd = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
            barrier(device)
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            for j, layer in enumerate((n_calls, n_calls + 1)):
                Qd.copy_(Qh, non_blocking=True)
                Kd.copy_(Kh, non_blocking=True)
                Vd.copy_(Vh, non_blocking=True)
                cache.prefill_scored(layer, Qd, Kd, Vd, workspace=ws)
                pos_h.copy_(cache.slot_positions(layer), non_blocking=True)
                stream.synchronize()
            e2e_s = reduce_max(time.perf_counter() - t0, device)
            e2e = {"value": world * tokens * 2 / e2e_s, "unit": "tokens/s",
                   "h2d_bytes_per_step": (Q.numel() + K.numel() + V.numel()) * Q.element_size(),
                   "d2h_bytes_per_step": pos_h.numel() * 4, "steps": 2}
        cache.close()
    per_call_s = dt_ms / 1e3 / args.steps
    value = world * tokens / per_call_s
    peak, peak_kind = measured_bf16_peak()
    achieved = flops / per_call_s / 1e12
    out = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) Q/K/V with hub and sink keys)",
        "config": dict(cfg, timing="CUDA events on the launching stream; a step = one layer's scored prefill "
                                   "(3 launches); Q/K/V of one layer exceed L2"),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind,
                     "algorithmic_flops_per_step": flops,
                     "exp2_per_step": w.batch * w.n_q_heads * P * (P + 1),
                     "note": "two tcgen05 passes over the causal triangle of q.k; the exp2 per product also bounds"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, desc = oracle_prefill_rate(w, P, args.cpu_seconds)
        out["cpu_baseline"] = {"value": rate * P / w.n_kv_heads, "unit": "tokens/s", "cores": threads,
                               "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def snapkv_phase(args, w, rank, world, local):
    """One layer's SnapKV prefill per step: the window's votes on the tensor
    cores, pooling, per-head top-k, union, copy. Bound by HBM: the prompt's K
    is read once, the votes go out and back, the kept rows are copied."""
    metric = "SnapKV prefill prompt tokens/s (window votes + selection); HBM GB/s vs measured copy"
    P, win = w.prompt_len, args.window
    if w.policy != configs.POLICY_H2O or w.dtype != configs.DTYPE_BF16 or P <= win:
        raise SystemExit("--phase snapkv needs an H2O bf16 workload with a prompt longer than the window")
    topk = args.topk or max(0, (w.capacity - win) // w.group)
    cfg = {"workload": w.name, "phase": "prefill_snapkv", "policy": "h2o", "batch": w.batch,
           "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "prompt_len": P,
           "window": win, "topk_per_head": topk, "capacity_slots": w.capacity}
    tokens = w.batch * P
    if args.impl == "reference":
        if rank != 0:
            return
        import concurrent.futures as cf
        import oracle
        threads = oracle.online_cores()
        G, d = w.group, w.head_dim
        rng = np.random.default_rng(w.seed)
        inputs = [(rng.standard_normal((G, win, d)).astype(np.float32), rng.standard_normal((P, d)).astype(np.float32))
                  for _ in range(threads)]

        def unit(i):
            q, k = inputs[i]
            u = oracle.Unit(oracle.H2O, w.n_sink, w.n_heavy, w.n_recent, w.budget, 0, 0, G, d)
            u.prefill_snapkv(q, k, k, topk)

        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            def sample():  # one unit per host core, in parallel
                t0 = time.perf_counter()
                list(ex.map(unit, range(threads)))
                return time.perf_counter() - t0
            rate, tsum = run_reference_samples(args, sample, threads)
        v = rate * P / w.n_kv_heads
        desc = (f"{threads} units (one sequence x KV head) of prompt {P} per round, rounds repeated for "
                f"{reference_step_seconds(args):.1f} s per bench step; {args.steps} timed steps after "
                f"{args.warmup} untimed, {tsum:.1f} s")
        print(json.dumps({"impl": "reference", "metric": metric, "value": v, "unit": "tokens/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * tokens / v,
                          "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": cfg,
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                           "sample": desc},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    import torch
    from kv_cache_eviction_decode_gb300 import KVEvictCache
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    n_calls = args.warmup + args.steps
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        Qo = synth.device_prompt_queries(w, 0, device, P)[:, :, P - win:].contiguous()
        K, V = synth.device_prompt(w, 0, device, P)
        cache = KVEvictCache.from_workload(w.with_(n_layers=n_calls + (0 if args.no_e2e else 2)), device=device,
                                           stream=stream)
        ws = torch.empty(cache.prefill_snapkv_workspace_bytes(P, win), dtype=torch.uint8, device=device)
        for i in range(args.warmup):
            cache.prefill_snapkv(i, Qo, K, V, topk, workspace=ws)
        stream.synchronize()
        barrier(device)
        torch.cuda.synchronize(device)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(device.index) as clk:
            ev0.record(stream)
            for i in range(args.warmup, n_calls):
                cache.prefill_snapkv(i, Qo, K, V, topk, workspace=ws)
            ev1.record(stream)
            ev1.synchronize()
        torch.cuda.synchronize(device)
        barrier(device)
        err = cache.check()
        if err:
            raise RuntimeError(f"device error word {err:#x}")
        dt_ms = reduce_max(ev0.elapsed_time(ev1), device)
        kept = int((cache.slot_positions(n_calls - 1) >= 0).sum().item())
        e2e = None
        if not args.no_e2e:
            Qh, Kh, Vh = Qo.cpu().pin_memory(), K.cpu().pin_memory(), V.cpu().pin_memory()
            pos_h = torch.empty((w.batch, w.n_kv_heads, cache.capacity), dtype=torch.int32).pin_memory()
            Qd, Kd, Vd = torch.empty_like(Qo), torch.empty_like(K), torch.empty_like(V)
            barrier(device)
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            for layer in (n_calls, n_calls + 1):
                Qd.copy_(Qh, non_blocking=True)
                Kd.copy_(Kh, non_blocking=True)
                Vd.copy_(Vh, non_blocking=True)
                cache.prefill_snapkv(layer, Qd, Kd, Vd, topk, workspace=ws)
                pos_h.copy_(cache.slot_positions(layer), non_blocking=True)
                stream.synchronize()
            e2e_s = reduce_max(time.perf_counter() - t0, device)
            e2e = {"value": world * tokens * 2 / e2e_s, "unit": "tokens/s",
                   "h2d_bytes_per_step": (Qo.numel() + K.numel() + V.numel()) * Qo.element_size(),
                   "d2h_bytes_per_step": pos_h.numel() * 4, "steps": 2}
        cache.close()
    e = 2
    row = w.head_dim * e
    algo = (w.batch * w.n_kv_heads * P * row            # the prompt's K, read once
            + w.batch * w.n_q_heads * win * row          # the window's queries
            + 2 * w.batch * w.n_q_heads * P * 4          # votes written, read back
            + 2 * 2 * kept * row)                        # kept K and V rows: read, write
    per_call_s = dt_ms / 1e3 / args.steps
    peak, peak_kind = measured_hbm_peak()
    achieved = algo / per_call_s / 1e9
    out = {
        "metric": metric, "value": world * tokens / per_call_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V with hub and sink keys)",
        "config": dict(cfg, timing="CUDA events on the launching stream; a step = one layer's SnapKV prefill "
                                   "(3 launches); the prompt's K exceeds L2", kept_tokens=kept),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_kind": peak_kind, "algorithmic_bytes_per_step": algo,
                     "frac_of_8TBs": achieved / 8000.0},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "e2e": e2e,
    }
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="sink_window")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--split", type=int, default=0)
    ap.add_argument("--clusters", type=int, default=0, help="persistent grid size in clusters (0 = automatic)")
    ap.add_argument("--alias", type=int, default=-1,
                    help="warp partial outputs over the logits: 1 where they fit, 0 never, -1 automatic")
    ap.add_argument("--tail-split", type=int, default=-1,
                    help="1: clusters split only their leftover units, 0: every unit split, -1: automatic")
    ap.add_argument("--path", type=int, default=0, help="0 automatic, 1 CUDA cores, 2 tensor cores")
    ap.add_argument("--ring", type=int, default=0, help="cap on ring stages per CTA (0 = fill shared memory)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time the decode steps as stream launches instead of one replay of a CUDA graph of them")
    ap.add_argument("--tie-steps", type=int, default=10,
                    help="H2O: token-steps run in validation mode after the timed region to count near-ties (0: none)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the score-keeping and Random workloads measured beside the default one")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling captures only; the line then names it)")
    ap.add_argument("--no-preroll", action="store_true",
                    help="time from the state right after prefill (small profiling captures only)")
    ap.add_argument("--phase", default="decode", choices=["decode", "prefill", "snapkv"],
                    help="decode (default): the decode step; prefill: the Q-seeded prefill of one layer (H2O); "
                         "snapkv: the SnapKV prefill selection of one layer (H2O)")
    ap.add_argument("--window", type=int, default=32, help="SnapKV observation window")
    ap.add_argument("--topk", type=int, default=0, help="SnapKV positions per query head (0: fill the budget)")
    ap.add_argument("--prompt", type=int, default=-1,
                    help="override the prompt length (small profiling captures only; decode launch shape unchanged "
                         "once the cache is full)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    w = configs.get(args.workload)
    if args.layers:
        w = w.with_(n_layers=args.layers, name=f"{w.name}_layers{args.layers}")
    if args.prompt >= 0:
        w = w.with_(prompt_len=args.prompt, max_prompt=max(w.max_prompt, args.prompt) if w.max_prompt else 0,
                    name=f"{w.name}_prompt{args.prompt}")
    rank, world, local = dist_env()
    metric = "decode tokens/s/GPU with eviction; attn+score+evict HBM GB/s vs 8 TB/s roofline"
    dtype = "bf16" if w.dtype == configs.DTYPE_BF16 else "f32"
    cfg = {"workload": w.name, "policy": configs.POLICY_NAMES[w.policy], "batch": w.batch, "layers": w.n_layers,
           "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "budget": w.budget,
           "n_sink": w.n_sink, "n_heavy": w.n_heavy, "n_recent": w.n_recent, "r": w.r,
           "prompt_len": w.prompt_len, "capacity_slots": w.capacity,
           "l2": "inputs larger than L2 (KV of one layer-step %.2f GB)" % (traffic.steady_layer_step_bytes(w) / 1e9)}

    if args.phase == "prefill":
        return prefill_phase(args, w, rank, world, local)
    if args.phase == "snapkv":
        return snapkv_phase(args, w, rank, world, local)

    if args.impl == "reference":
        # The reference arm is the CPU oracle, timed as it stands on the host
        # cores; rank 0 only.
        if rank != 0:
            return
        # W untimed and K timed samples of the same size, sized so that the whole
        # run takes about two and a half minutes of host time
        per_step = min(max(1.0, args.cpu_seconds / 2), max(0.2, 150.0 / (args.steps + args.warmup)))
        sample, work, threads, desc = oracle_sampler(w, n_units=min(256, w.batch * w.n_kv_heads),
                                                     target_s=per_step)
        for _ in range(args.warmup):
            sample()
        dts = [sample() for _ in range(args.steps)]
        v = cpu_tokens_per_s(w, work * args.steps / sum(dts))
        desc = f"{desc}, per bench step; {args.steps} timed steps after {args.warmup} untimed, {sum(dts):.1f} s"
        print(json.dumps({"impl": "reference", "metric": metric, "value": v, "unit": "tokens/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * w.batch / v,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": cfg,
                          "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                           "sample": desc},
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    device = torch.device(f"cuda:{local}")
    r = run_ours(args, w, rank, world, device)

    dt_s = r["dt_ms"] / 1e3
    tokens = world * w.batch * args.steps
    value = tokens / dt_s
    launches = r["decode_launches"]
    avg_launch_s = dt_s / max(1, launches)
    layer_bytes = traffic.steady_layer_step_bytes(w)
    if r["held"] is not None:  # two-pool H2O: the tokens actually held
        layer_bytes = w.batch * w.n_kv_heads * traffic.unit_step_bytes(w, int(round(r["held"] * w.capacity)))
        cfg["held_fraction"] = r["held"]
        cfg["hh_threshold"] = w.hh_threshold
    achieved = layer_bytes / avg_launch_s / 1e9
    peak, peak_kind = measured_hbm_peak()
    out = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["dt_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V with hub and sink keys, generated on the device)",
        "config": dict(cfg, split=r["split"], clusters=r["clusters"], tensor_cores=bool(r["tensor_cores"]),
                       ring_stages=r["ring_stages"], tail_split=bool(r["tail_split"]),
                       partials_alias=bool(r["partials_alias"]),
                       timing=("CUDA events on the launching stream around one replay of a CUDA graph of the "
                               "timed steps; no L2 flush needed") if args.graph else
                       "CUDA events on the launching stream; no L2 flush needed"),
        "layer_step_us": 1e6 * avg_launch_s,
        "kernel_us_isolated": 1e3 * statistics.median(r["iso_ms"]) if r["iso_ms"] else None,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(w.name), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": layer_bytes,
                     "frac_of_8TBs": achieved / 8000.0,
                     "note": "avg launch duration = timed region / decode launches (includes launch gaps)"},
        "gpu_launches": launches + r["cut_launches"],
        "clocks": r["clocks"],
        "e2e": r["e2e"],
    }
    if r["near_ties"] is not None:
        out["near_ties"] = r["near_ties"]
    headline = args.workload == "sink_window" and not args.layers and args.prompt < 0
    if world == 1 and headline and not args.no_workloads:
        out["workloads"] = extra_workloads(args, rank, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, desc, _ = oracle_sample_rate(w, n_units=min(256, w.batch * w.n_kv_heads),
                                                    target_s=args.cpu_seconds)
        out["cpu_baseline"] = {"value": cpu_tokens_per_s(w, rate), "unit": "tokens/s", "cores": threads,
                               "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
