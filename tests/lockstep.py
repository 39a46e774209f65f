"""Lockstep parity harness: the CUDA path runs a workload's full launch shape,
the CPU oracle replays the checked units step by step on the same inputs.

Inputs: every unit gets device-generated values; the checked units' slices
are overwritten with the host generator's values, which the oracle reads.
Units are independent, so the checked units see exactly the oracle's inputs.

Per step and checked unit the GPU trace gives the slot the new token took and
what it evicted. The oracle makes its own choice; StreamingLLM and Random
must agree bit-exactly. For H2O a different victim is accepted only as a
near-tie (the two candidates' oracle scores within 1e-5 relative), counted,
and the oracle then adopts the GPU's choice so both continue from the same
retained set. For two-pool H2O the trace also records the promotion; a
different decision is accepted only when one of the comparisons that made
the oracle's (the two lowest of a pool, a score against the threshold) was
within the same relative tolerance, and is then adopted whole.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from kv_cache_eviction_decode_gb300 import KVEvictCache
from workloads import synth
from workloads.configs import DTYPE_BF16, POLICY_H2O, POLICY_H2O_BLOCK, POLICY_H2O_POOLS, POLICY_RANDOM, Workload

NEAR_TIE_REL = 1e-5
BF16_REL_TOL = 2e-2
F32_ABS_TOL = 1e-4


def scored(w: Workload) -> bool:
    """Policies whose retained set depends on cumulative attention scores."""
    return w.policy in (POLICY_H2O, POLICY_H2O_BLOCK, POLICY_H2O_POOLS)


def torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == DTYPE_BF16 else torch.float32


@dataclass
class DeviceRun:
    trace: dict = field(default_factory=dict)       # layer -> int32 [T, B, Hkv, 4]
    out: dict = field(default_factory=dict)         # layer -> {seq: float32 [T, Hq, D]}
    pos_snap: dict = field(default_factory=dict)    # layer -> {t: int32 [B, Hkv, C]}; t = -1 after prefill
    score_snap: dict = field(default_factory=dict)  # layer -> {t: float32 [B, Hkv, C]}
    pool_snap: dict = field(default_factory=dict)   # layer -> {t: uint8 [B, Hkv, C]} (two-pool H2O)
    err: int = 0
    split: int = 0
    tensor_cores: int = 0


def host_inputs(w, units, n_steps, prompt_len):
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        res = list(ex.map(lambda u: synth.UnitInputs(w, u[0], u[1], u[2], n_steps, prompt_len), units))
    return dict(zip(units, res))


def run_gpu(w: Workload, layers, n_steps: int, inputs: dict, prompt_len: int, device, snap_steps=(),
            split: int | None = None, out_seqs=None, seed: int = 0, clusters: int | None = None,
            interleave: bool = True, path: int | None = None) -> DeviceRun:
    """Runs n_steps decode steps of the given layers at the workload's shape.

    interleave=True issues the steps token by token over the layers, as a
    model does (layer 0, 1, ... of token t, then token t + 1); otherwise all
    steps of one layer, then the next layer."""
    cache = KVEvictCache.from_workload(w, device=device)
    if split:
        cache.set_split(split)
    if clusters:
        cache.set_clusters(clusters)
    if path:
        cache.set_path(path)
    B, Hq, Hkv, D, G = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.group
    dt = torch_dtype(w)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000 + 17)
    st = cache.stats()
    run = DeviceRun(split=st["split"], tensor_cores=st["tensor_cores"])
    snap_steps = set(snap_steps)
    bufs = {}
    for layer in layers:
        mine = {u: x for u, x in inputs.items() if u[1] == layer}
        if prompt_len > 0:
            K, V = synth.device_prompt(w, layer, device, prompt_len, gen=gen)
            for (seq, _, h), x in mine.items():
                K[seq, h] = torch.from_numpy(x.prompt_k).to(device=device, dtype=dt)
                V[seq, h] = torch.from_numpy(x.prompt_v).to(device=device, dtype=dt)
            cache.prefill(layer, K, V)
            del K, V
        q = torch.randn((n_steps, B, Hq, D), generator=gen, device=device).to(dt)
        k = torch.randn((n_steps, B, Hkv, D), generator=gen, device=device).to(dt)
        v = torch.randn((n_steps, B, Hkv, D), generator=gen, device=device).to(dt)
        for (seq, _, h), x in mine.items():
            q[:, seq, h * G:(h + 1) * G] = torch.from_numpy(x.q).to(device=device, dtype=dt)
            k[:, seq, h] = torch.from_numpy(x.k_new).to(device=device, dtype=dt)
            v[:, seq, h] = torch.from_numpy(x.v_new).to(device=device, dtype=dt)
        out = torch.empty((n_steps, B, Hq, D), dtype=dt, device=device)
        trace = torch.full((n_steps, B, Hkv, 4), -7, dtype=torch.int32, device=device)
        cache.set_trace(layer, trace)
        run.pos_snap[layer] = {-1: cache.slot_positions(layer).cpu()}
        run.score_snap[layer] = {}
        run.pool_snap[layer] = {}
        if scored(w):
            run.score_snap[layer][-1] = cache.scores(layer).cpu()
        if w.policy == POLICY_H2O_POOLS:
            run.pool_snap[layer][-1] = cache.pools(layer).cpu()
        seqs = out_seqs if out_seqs is not None else sorted({u[0] for u in mine})
        bufs[layer] = (q, k, v, out, trace, seqs)

    def step(layer, t):
        q, k, v, out, _, _ = bufs[layer]
        cache.decode_step(layer, q[t], k[t], v[t], out[t])
        if t in snap_steps:
            run.pos_snap[layer][t] = cache.slot_positions(layer).cpu()
            if scored(w):
                run.score_snap[layer][t] = cache.scores(layer).cpu()
            if w.policy == POLICY_H2O_POOLS:
                run.pool_snap[layer][t] = cache.pools(layer).cpu()

    if interleave:
        for t in range(n_steps):
            for layer in layers:
                step(layer, t)
    else:
        for layer in layers:
            for t in range(n_steps):
                step(layer, t)
    run.err |= cache.check()
    for layer in layers:
        q, k, v, out, trace, seqs = bufs.pop(layer)
        run.trace[layer] = trace.cpu().numpy()
        run.out[layer] = {s: out[:, s].float().cpu().numpy() for s in seqs}
        del q, k, v, out
    cache.close()
    return run


@dataclass
class UnitReport:
    unit: tuple
    max_out_err: float = 0.0
    max_score_err: float = 0.0
    near_ties: int = 0
    steps: int = 0
    out_checks: int = 0


def out_error(w, got, ref):
    if w.dtype == DTYPE_BF16:
        return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-6))
    return float(np.max(np.abs(got - ref)))


def out_tol(w):
    return BF16_REL_TOL if w.dtype == DTYPE_BF16 else F32_ABS_TOL


def score_error(w, got, ref, qscale: float = 0.0):
    diff = np.abs(got - ref)
    if getattr(w, "score_int8", False):
        # INT8 storage: both quantise with their own unit maximum (fp32 vs fp64
        # sums before the same rounding); a midpoint may round one code apart
        # and the difference then persists: allow two codes of the oracle's scale
        diff = np.maximum(diff - 2.0 * qscale * (1 + 1e-3), 0.0)
    if getattr(w, "score_half", False):
        # binary16 storage: the GPU rounds its fp32 sum, the oracle its fp64 sum;
        # they may land one binary16 step apart (at most 2^-10 of the value)
        diff = np.maximum(diff - (2.0**-10 * np.abs(ref) + 2.0**-24), 0.0)
    if w.dtype == DTYPE_BF16:
        return float(np.max(diff) / max(np.max(np.abs(ref)), 1e-6))
    return float(np.max(diff))


def replay_unit(w: Workload, unit, x, run: DeviceRun, n_steps: int, out_steps=None,
                inputs_needed: bool = True) -> UnitReport:
    """Replays one unit on the oracle and checks it against the GPU run."""
    seq, layer, h = unit
    G = w.group
    rep = UnitReport(unit)
    u = oracle.Unit.for_workload(w, seq, layer, h)
    if x is not None and x.prompt_len:
        u.prefill(x.prompt_k, x.prompt_v)
    elif x is None and w.prompt_len:
        z = np.zeros((w.prompt_len, w.head_dim), np.float32)
        u.prefill(z, z)
    snaps = run.pos_snap[layer]
    ssnaps = run.score_snap.get(layer, {})
    psnaps = run.pool_snap.get(layer, {})
    np.testing.assert_array_equal(u.positions(), snaps[-1][seq, h].numpy(), err_msg=f"{unit} table after prefill")
    pools_policy = w.policy == POLICY_H2O_POOLS
    tie_rel = 2.0**-10 if getattr(w, "score_half", False) else NEAR_TIE_REL  # one binary16 step
    int8 = getattr(w, "score_int8", False)

    def check_pools(t):
        if t in psnaps:
            occ = u.positions() >= 0
            np.testing.assert_array_equal(u.pools()[occ], psnaps[t][seq, h].numpy()[occ].astype(np.int8),
                                          err_msg=f"{unit} pools, step {t}")

    check_pools(-1)
    tr = run.trace[layer][:, seq, h]
    zero = np.zeros(w.head_dim, np.float32)
    for t in range(n_steps):
        want_out = x is not None and (out_steps is None or t in out_steps)
        if scored(w) or want_out:
            ref = u.attend(x.q[t], x.k_new[t], x.v_new[t])
            if want_out:
                got = run.out[layer][seq][t, h * G:(h + 1) * G]
                e = out_error(w, got, ref)
                rep.max_out_err = max(rep.max_out_err, e)
                rep.out_checks += 1
                assert e <= out_tol(w), f"{unit} step {t}: output error {e:.3e}"
        else:
            u.stage(x.k_new[t] if x is not None else zero, x.v_new[t] if x is not None else zero)
        slot = u.choose()
        gslot, gold = int(tr[t, 0]), int(tr[t, 1])
        if pools_policy:
            mine = u.decision()
            grec = int(tr[t, 3])
            gdec = (u.cap if gslot < 0 else gslot, 1 if grec == -2 else 0, grec if grec >= 0 else -1)
            if gdec != mine:
                assert u.decision_margin < tie_rel, \
                    f"{unit} step {t}: GPU decision {gdec}, oracle {mine} (margin {u.decision_margin:.3e})"
                rep.near_ties += 1
            want_old = u.prompt_len + u.steps if gdec[0] == u.cap else u.pos_at(gdec[0])
            assert gold == want_old, f"{unit} step {t}: GPU evicted position {gold}, oracle {want_old}"
            u.commit_pools(*gdec)
        elif gslot != slot:
            assert w.policy == POLICY_H2O, f"{unit} step {t}: GPU slot {gslot}, oracle slot {slot}"
            sc = u.scores()
            a, b = sc[slot], sc[gslot]
            rel = abs(a - b) / max(a, b, 1e-300)
            tie_rel = 2.0**-10 if getattr(w, "score_half", False) else NEAR_TIE_REL  # one binary16 step
            if int8:  # within two and a half codes of the oracle's scale (see score_error)
                rel = abs(a - b) / max(2.5 * u.score_scale(), 1e-300)
                tie_rel = 1.0
            assert 0 <= gslot < u.cap and rel < tie_rel, \
                f"{unit} step {t}: GPU evicted slot {gslot} (pos {u.pos_at(gslot)}, score {b:.9g}), " \
                f"oracle slot {slot} (pos {u.pos_at(slot)}, score {a:.9g}), rel {rel:.3e}"
            rep.near_ties += 1
            slot = gslot
        if not pools_policy:
            assert gold == u.pos_at(slot), f"{unit} step {t}: GPU evicted position {gold}, oracle {u.pos_at(slot)}"
            u.commit(slot)
        if t in snaps:
            np.testing.assert_array_equal(u.positions(), snaps[t][seq, h].numpy(), err_msg=f"{unit} table, step {t}")
        check_pools(t)
        if t in ssnaps:
            pos = u.positions()
            occ = pos >= 0
            e = score_error(w, ssnaps[t][seq, h].numpy()[occ], u.scores()[occ], u.score_scale() if int8 else 0.0)
            rep.max_score_err = max(rep.max_score_err, e)
            assert e <= out_tol(w), f"{unit} step {t}: score error {e:.3e}"
        rep.steps += 1
    return rep


def replay_all(w, units, inputs, run, n_steps, out_steps=None, threads=None):
    threads = threads or min(16, os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(replay_unit, w, u, inputs.get(u), run, n_steps, out_steps) for u in units]
        return [f.result() for f in futs]


def check_selector(w: Workload, run: DeviceRun, layer: int, prompt_len: int):
    """Bit-exact check of the H2O selector on the GPU's own fp32 values: at
    every snapshot step the evicted token's (score, position) key is below
    the key of every other candidate left in the cache."""
    checked = 0
    for t, table in run.pos_snap[layer].items():
        if t < 0:
            continue
        scores = run.score_snap[layer][t].numpy()
        pos = table.numpy()
        tr = run.trace[layer][t]
        p = prompt_len + t
        slot, old_pos, old_bits = tr[..., 0], tr[..., 1], tr[..., 2].astype(np.uint32)
        if np.any(old_pos < 0):
            continue  # not a full-cache step
        keys = (scores.view(np.uint32).astype(np.uint64) << np.uint64(32)) | pos.astype(np.uint32).astype(np.uint64)
        elig = (pos >= w.n_sink) & (pos <= p - w.n_recent)
        B, H, C = pos.shape
        elig[np.arange(B)[:, None], np.arange(H)[None, :], slot] = False  # the new token's slot
        vkey = (old_bits.astype(np.uint64) << np.uint64(32)) | old_pos.astype(np.uint32).astype(np.uint64)
        others = np.where(elig, keys, np.uint64(np.iinfo(np.uint64).max)).min(axis=2)
        assert np.all(vkey < others), f"layer {layer} step {t}: a candidate has a smaller key than the victim"
        assert np.all((old_pos >= w.n_sink) & (old_pos <= p - w.n_recent)), "victim outside the candidate window"
        checked += 1
    return checked
