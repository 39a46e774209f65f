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

INT8 score storage is compared code by code at every step: the GPU's codes
(read after the step) must equal the oracle's, except one code apart where
the oracle's unrounded value s * 255 / M lay within MIDPOINT_TOL of a
rounding midpoint (the GPU sums and rounds in fp32, the oracle in fp64);
such a code is counted and adopted by the oracle. With equal codes both
sides order the candidates identically, so INT8 victims must then agree
exactly.
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
# INT8 codes: how far from a midpoint k + 1/2 (in codes) an fp32-vs-fp64
# difference may move the unrounded value. The scores agree to about 1e-6
# relative (fp32 accumulation over the steps), i.e. 2.6e-4 codes at code 255.
MIDPOINT_TOL = 1e-3


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
    code_snap: dict = field(default_factory=dict)   # layer -> {t: uint8 [B, Hkv, C]} INT8 codes after step t
    ledger: dict = field(default_factory=dict)      # layer -> float64 [B, Hkv] evicted mass after the last step
    scale_snap: dict = field(default_factory=dict)  # layer -> {t: float32 [B, Hkv]} INT8 scales after step t
    err: int = 0
    split: int = 0
    tensor_cores: int = 0
    tail_split: int = 0
    partials_alias: int = 0


def host_inputs(w, units, n_steps, prompt_len):
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        res = list(ex.map(lambda u: synth.UnitInputs(w, u[0], u[1], u[2], n_steps, prompt_len), units))
    return dict(zip(units, res))


def run_gpu(w: Workload, layers, n_steps: int, inputs: dict, prompt_len: int, device, snap_steps=(),
            split: int | None = None, out_seqs=None, seed: int = 0, clusters: int | None = None,
            interleave: bool = True, path: int | None = None, tail_split: bool | None = None,
            alias: int | None = None) -> DeviceRun:
    """Runs n_steps decode steps of the given layers at the workload's shape.

    interleave=True issues the steps token by token over the layers, as a
    model does (layer 0, 1, ... of token t, then token t + 1); otherwise all
    steps of one layer, then the next layer. INT8 score storage: the codes
    and scales are read after every step."""
    cache = KVEvictCache.from_workload(w, device=device)
    if tail_split is not None:
        cache.set_tail_split(tail_split)
    if alias is not None:
        cache.set_partials_alias(alias)
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
    run = DeviceRun(split=st["split"], tensor_cores=st["tensor_cores"], tail_split=st["tail_split"])
    first_step = [True]
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
        run.code_snap[layer] = {}
        run.scale_snap[layer] = {}
        if scored(w):
            run.score_snap[layer][-1] = cache.scores(layer).cpu()
        if w.policy == POLICY_H2O_POOLS:
            run.pool_snap[layer][-1] = cache.pools(layer).cpu()
        seqs = out_seqs if out_seqs is not None else sorted({u[0] for u in mine})
        bufs[layer] = (q, k, v, out, trace, seqs)

    int8 = getattr(w, "score_int8", False)

    def step(layer, t):
        q, k, v, out, _, _ = bufs[layer]
        cache.decode_step(layer, q[t], k[t], v[t], out[t])
        if first_step[0]:  # the launch configuration is known after the first step
            run.partials_alias = cache.stats()["partials_alias"]
            first_step[0] = False
        if int8:  # stored value = code * scale exactly: the code is the rounded ratio
            scl = cache.score_scales(layer)
            codes = torch.round(cache.scores(layer) / scl.clamp_min(1e-38)[..., None])
            assert bool(((codes >= 0) & (codes <= 255)).all()), f"layer {layer} step {t}: INT8 code out of range"
            run.code_snap[layer][t] = codes.to(torch.uint8).cpu()
            run.scale_snap[layer][t] = scl.cpu()
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
        if scored(w):
            run.ledger[layer] = cache.evicted_mass(layer).cpu().numpy()
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
    near_ties: int = 0       # victims (or two-pool decisions) that differed at a near-tie, adopted
    decisions: int = 0       # steps at which a victim was chosen among scored candidates
    midpoints: int = 0       # INT8 codes one apart at a rounding midpoint, adopted
    codes_compared: int = 0  # INT8 codes compared
    steps: int = 0
    out_checks: int = 0


def out_error(w, got, ref):
    if w.dtype == DTYPE_BF16:
        return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-6))
    return float(np.max(np.abs(got - ref)))


def out_tol(w):
    return BF16_REL_TOL if w.dtype == DTYPE_BF16 else F32_ABS_TOL


def score_error(w, got, ref):
    diff = np.abs(got - ref)
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
    csnaps = run.code_snap.get(layer, {})
    scsnaps = run.scale_snap.get(layer, {})

    def sync_int8_codes(t, gslot, gold):
        """INT8: compares the oracle's codes after its update at step t with
        the GPU's (read after the step: the destination slot then holds the
        new token, the evicted token's code is in the trace); a code one apart
        at a rounding midpoint is counted and adopted, any other difference
        fails."""
        assert t in csnaps, f"{unit} step {t}: INT8 codes not read"
        gcodes = csnaps[t][seq, h].numpy().astype(np.int64)
        gscale = float(scsnaps[t][seq, h])
        sc_err = abs(gscale - u.score_scale()) / max(u.score_scale(), 1e-300)
        assert sc_err <= out_tol(w), f"{unit} step {t}: INT8 scale {gscale:.9g}, oracle {u.score_scale():.9g}"
        xo, xnew = u.int8_unrounded()
        pos = u.positions()
        ocodes = u.score_codes().astype(np.int64)
        pairs = []  # (oracle slot or cap for the new token, GPU code)
        for s in np.nonzero(pos >= 0)[0]:
            if s != gslot:
                pairs.append((int(s), int(gcodes[s])))
        if gold >= 0 and 0 <= gslot < u.cap:  # the evicted token's code is in the trace
            ev = np.array([tr[t, 2]], dtype=np.int32).view(np.float32)[0]
            pairs.append((gslot, int(np.rint(ev / np.float32(gscale)))))
        gnew = np.array([tr[t, 3]], dtype=np.int32).view(np.float32)[0]
        pairs.append((u.cap, int(np.rint(gnew / np.float32(gscale)))))
        rep.codes_compared += len(pairs)
        for s, gc in pairs:
            oc = int(ocodes[s]) if s < u.cap else int(np.rint(u.new_score / u.score_scale()))
            if gc == oc:
                continue
            x = xo[s] if s < u.cap else xnew
            mid = abs(x - np.floor(x) - 0.5)
            assert abs(gc - oc) == 1 and mid < MIDPOINT_TOL, \
                f"{unit} step {t}: slot {s} GPU code {gc}, oracle {oc} (unrounded {x:.6f})"
            u.adopt_int8_code(s, gc)
            rep.midpoints += 1

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
        gslot, gold = int(tr[t, 0]), int(tr[t, 1])
        if int8:
            sync_int8_codes(t, gslot, gold)
        slot = u.choose()
        if scored(w) and not pools_policy and gold >= 0:
            rep.decisions += 1
        if pools_policy:
            mine = u.decision()
            if u.decision_margin != np.inf:  # the recent pool overflowed: a decision among scores
                rep.decisions += 1
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
            assert w.policy == POLICY_H2O and not int8, f"{unit} step {t}: GPU slot {gslot}, oracle slot {slot}"
            sc = u.scores()
            a, b = sc[slot], sc[gslot]
            rel = abs(a - b) / max(a, b, 1e-300)
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
            e = score_error(w, ssnaps[t][seq, h].numpy()[occ], u.scores()[occ])
            rep.max_score_err = max(rep.max_score_err, e)
            assert e <= out_tol(w), f"{unit} step {t}: score error {e:.3e}"
        rep.steps += 1
    if layer in run.ledger and rep.steps == n_steps:
        # the GPU's evicted-mass ledger against the oracle's, after the last step
        got, want = float(run.ledger[layer][seq, h]), u.evicted_mass
        err = abs(got - want) / max(abs(want), 1.0) if w.dtype == DTYPE_BF16 else abs(got - want)
        assert err <= out_tol(w), f"{unit}: evicted mass {got:.9g}, oracle {want:.9g}"
    return rep


def record_ties(record_property, reps, max_near_ties: int, max_midpoint_rate: float = 0.0,
                max_near_tie_rate: float = 0.0) -> dict:
    """Records a lockstep run's counts as test properties (a junit report
    carries them): victims that differed at a near-tie, eviction decisions,
    INT8 codes one apart at a midpoint and INT8 codes compared. Asserts the
    near-tie count (at most max_near_ties + max_near_tie_rate * decisions)
    and the midpoint rate against their bounds."""
    n = dict(near_ties=sum(r.near_ties for r in reps), decisions=sum(r.decisions for r in reps),
             midpoints=sum(r.midpoints for r in reps), codes_compared=sum(r.codes_compared for r in reps))
    for k, v in n.items():
        record_property(k, v)
    assert n["near_ties"] <= max_near_ties + max_near_tie_rate * n["decisions"], \
        f"{n['near_ties']} near-ties in {n['decisions']} decisions"
    assert n["midpoints"] <= max_midpoint_rate * n["codes_compared"], \
        f"{n['midpoints']} INT8 midpoint codes in {n['codes_compared']}"
    return n


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
