"""The H2O selector on the oracle's own scores, bit for bit.

The eviction decision of "h2o: heavy-hitter oracle" (summary, Algorithm 1:
remove the token whose removal leaves the highest cumulative score; with an
additive score, the lowest-score candidate; ties to the older position) is
run by kvevict_select_victims with the decode kernel's own selector code
(candidate rule, key, reductions) on scores the test uploads: the oracle's
fp64 scores rounded to fp32. The oracle decides on the same fp32 values (its
own greedy step, fed those values), and the two victims must be identical for
every checked unit at every step -- no tolerance, no near-tie allowance.

Between the selector calls the GPU runs its real decode steps (its own fp32
scores); the oracle follows them as in the lockstep tests (a different
victim accepted only at a near-tie, counted and adopted), so the handle's
slot table and the oracle's stay equal and the selector always sees the
oracle's retained set.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_decode_gb300 import KVEvictCache
from tests import lockstep as ls
from workloads import configs, synth

pytestmark = pytest.mark.gpu


def _selector_lockstep(w, layer, checked, T, device):
    """Runs T decode steps of one layer at the workload's shape; before every
    step, the selector on the checked units' fp32-rounded oracle scores.
    Returns counters."""
    B, Hq, Hkv, D, G, C = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.group, w.capacity
    dt = ls.torch_dtype(w)
    units = [(s, layer, h) for s, h in checked]
    inputs = ls.host_inputs(w, units, T, w.prompt_len)
    cache = KVEvictCache.from_workload(w, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(4321)
    K, V = synth.device_prompt(w, layer, device, w.prompt_len, gen=gen)
    for (s, _, h), x in inputs.items():
        K[s, h] = torch.from_numpy(x.prompt_k).to(device=device, dtype=dt)
        V[s, h] = torch.from_numpy(x.prompt_v).to(device=device, dtype=dt)
    cache.prefill(layer, K, V)
    del K, V
    q = torch.randn((T, B, Hq, D), generator=gen, device=device).to(dt)
    kn = torch.randn((T, B, Hkv, D), generator=gen, device=device).to(dt)
    vn = torch.randn((T, B, Hkv, D), generator=gen, device=device).to(dt)
    for (s, _, h), x in inputs.items():
        q[:, s, h * G:(h + 1) * G] = torch.from_numpy(x.q).to(device=device, dtype=dt)
        kn[:, s, h] = torch.from_numpy(x.k_new).to(device=device, dtype=dt)
        vn[:, s, h] = torch.from_numpy(x.v_new).to(device=device, dtype=dt)
    out = torch.empty((B, Hq, D), dtype=dt, device=device)
    trace = torch.full((T, B, Hkv, 4), -7, dtype=torch.int32, device=device)
    cache.set_trace(layer, trace)
    orc = {}
    for (s, _, h), x in inputs.items():
        u = oracle.Unit.for_workload(w, s, layer, h)
        u.prefill(x.prompt_k, x.prompt_v)
        orc[(s, h)] = u
    scores_dev = torch.zeros((B, Hkv, C), dtype=torch.float32, device=device)
    host = np.zeros((B, Hkv, C), dtype=np.float32)
    n = dict(selections=0, rounding_changed=0, near_ties=0, decisions=0)
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        for t in range(T):
            # the oracle's update of step t (attention, cumulative scores)
            list(ex.map(lambda k: orc[k].attend(inputs[(k[0], layer, k[1])].q[t],
                                                inputs[(k[0], layer, k[1])].k_new[t],
                                                inputs[(k[0], layer, k[1])].v_new[t]), list(orc)))
            want = {}
            for (s, h), u in orc.items():
                s64, n64 = u.scores(), u.new_score
                v64 = u.choose()
                s32 = s64.astype(np.float32)
                u.set_scores(s32.astype(np.float64), float(np.float32(n64)))
                v32 = u.choose()  # the oracle's greedy step on the fp32 values
                u.set_scores(s64, n64)  # the oracle itself goes on in fp64
                host[s, h] = s32
                want[(s, h)] = (v32, v64, u.count + 1 > w.budget)
            scores_dev.copy_(torch.from_numpy(host))
            victims = cache.select_victims(layer, scores_dev).cpu().numpy()
            for (s, h), (v32, v64, full) in want.items():
                if not full:
                    continue
                assert victims[s, h] == v32, \
                    f"step {t} unit ({s}, {h}): selector slot {victims[s, h]}, oracle slot {v32} on the same fp32 scores"
                n["selections"] += 1
                n["rounding_changed"] += int(v32 != v64)
            # the GPU's own decode step; the oracle follows its victim
            cache.decode_step(layer, q[t], kn[t], vn[t], out)
            tr = trace[t].cpu().numpy()
            for (s, h), u in orc.items():
                gslot, gold = int(tr[s, h, 0]), int(tr[s, h, 1])
                slot = u.choose()
                if gold >= 0:
                    n["decisions"] += 1
                if gslot != slot:
                    sc = u.scores()
                    a, b = sc[slot], sc[gslot]
                    assert abs(a - b) / max(a, b, 1e-300) < ls.NEAR_TIE_REL, f"step {t} unit ({s}, {h})"
                    n["near_ties"] += 1
                u.commit(gslot)
            if t % 32 == 31 or t == T - 1:
                pos = cache.slot_positions(layer).cpu().numpy()
                for (s, h), u in orc.items():
                    np.testing.assert_array_equal(pos[s, h], u.positions())
    assert cache.check() == 0
    cache.close()
    return n


def test_selector_on_oracle_scores_tiny(cuda_device, record_property):
    """The tiny H2O workload (fp32, 8 heads, K = 4 + 60 + 64, prompt 256):
    every unit, every one of the 256 steps."""
    w = configs.H2O_TINY
    n = _selector_lockstep(w, 0, [(0, h) for h in range(w.n_kv_heads)], w.decode_steps, cuda_device)
    for k, v in n.items():
        record_property(k, v)
    print("selector on oracle scores, tiny:", n)
    assert n["selections"] == w.n_kv_heads * w.decode_steps
    assert n["near_ties"] <= 1


def test_selector_on_oracle_scores_mha_slice(cuda_device, record_property):
    """One layer of the MHA H2O workload (bf16, B=16, 32 heads, K = 4 + 510 +
    510, prompt 2048): sequences {0, 15} x every head, 96 steps."""
    w = configs.H2O_MHA.with_(n_layers=1)
    checked = [(s, h) for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    T = 96
    n = _selector_lockstep(w, 0, checked, T, cuda_device)
    for k, v in n.items():
        record_property(k, v)
    print("selector on oracle scores, MHA slice:", n)
    assert n["selections"] == len(checked) * T
    assert n["near_ties"] <= 2


def test_selector_exact_ties_take_the_older_position(cuda_device):
    """Constructed scores on the tiny workload right after its prompt (sinks
    0-3, positions 132-255 held, candidates 132-192 for position 256): equal
    scores everywhere, equal minima at two candidates, the smallest values on
    protected tokens, and neighbouring fp32 values. The selector's victim
    equals the oracle's greedy step on the same values in every case."""
    w = configs.H2O_TINY
    B, Hkv, C = w.batch, w.n_kv_heads, w.capacity
    xs = [synth.UnitInputs(w, 0, 0, h, 1) for h in range(Hkv)]
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    K = torch.from_numpy(np.stack([x.prompt_k for x in xs])[None]).to(cuda_device)
    V = torch.from_numpy(np.stack([x.prompt_v for x in xs])[None]).to(cuda_device)
    cache.prefill(0, K, V)
    orc = []
    for h, x in enumerate(xs):
        u = oracle.Unit.for_workload(w, 0, 0, h)
        u.prefill(x.prompt_k, x.prompt_v)
        u.attend(x.q[0], x.k_new[0], x.v_new[0])  # a pending token, position 256
        orc.append(u)
    pos = orc[0].positions()
    p = w.prompt_len
    cand = np.nonzero((pos >= w.n_sink) & (pos <= p - w.n_recent))[0]
    prot = np.nonzero(~((pos >= w.n_sink) & (pos <= p - w.n_recent)))[0]
    assert len(cand) == w.n_heavy + 1
    rng = np.random.default_rng(7)
    cases = []
    cases.append(np.full(C, 0.25, np.float32))                      # all equal: the oldest candidate
    cases.append(np.zeros(C, np.float32))                           # all +0.0
    a = rng.uniform(0.1, 1.0, C).astype(np.float32)
    i, j = rng.choice(cand, 2, replace=False)
    a[i] = a[j] = np.float32(0.01)                                  # two equal minima: the older one
    cases.append(a)
    b = rng.uniform(0.1, 1.0, C).astype(np.float32)
    b[prot] = 0.0                                                   # smallest on sinks and the window
    cases.append(b)
    c = np.full(C, 0.5, np.float32)
    c[cand] = np.nextafter(np.float32(0.5), np.float32(1.0))
    c[cand[-1]] = np.float32(0.5)                                   # the newest candidate, one ulp lower
    cases.append(c)
    d = rng.integers(0, 4, C).astype(np.float32) / 8                # many exact ties at a few levels
    cases.append(d)
    for ci, case in enumerate(cases):
        host = np.zeros((B, Hkv, C), np.float32)
        want = []
        for h, u in enumerate(orc):
            sc = np.roll(case, h * 5) if ci >= 2 else case  # a different arrangement per unit
            host[0, h] = sc
            keep = u.scores(), u.new_score
            u.set_scores(sc.astype(np.float64), 1.0)
            want.append(u.choose())
            u.set_scores(*keep)
        got = cache.select_victims(0, torch.from_numpy(host).to(cuda_device)).cpu().numpy()
        assert list(got[0]) == want, f"case {ci}: selector {list(got[0])}, oracle {want}"
        if ci < 2:  # all equal: the oldest candidate leaves
            oldest = int(cand[np.argmin(pos[cand])])
            assert want == [oldest] * Hkv
    cache.close()


def test_selector_without_candidates(cuda_device):
    """A prompt shorter than the sinks: no slot holds a candidate, and the
    selector says so (-1) for every unit."""
    w = configs.H2O_TINY
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    K = torch.randn((1, w.n_kv_heads, 3, w.head_dim), device=cuda_device)
    cache.prefill(0, K, K)
    s = torch.rand((1, w.n_kv_heads, w.capacity), device=cuda_device)
    assert torch.all(cache.select_victims(0, s) == -1)
    cache.close()
