"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerances (from the method's statement of the target): attention outputs and
cumulative scores within 1e-4 max-abs for fp32 workloads and 2e-2 relative
(||gpu - oracle||_inf / ||oracle||_inf per unit and step) for bf16 workloads;
slot tables bit-exact for StreamingLLM and Random; H2O victims identical
except at near-ties (candidate scores within 1e-5 relative), which are
counted.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_decode_gb300 import DEV_NONFINITE, KVEvictCache
from tests import lockstep as ls
from workloads import configs, synth

pytestmark = pytest.mark.gpu


def _small(policy, dtype, G=2, d=64, B=3, L=2, **kw):
    base = dict(name="small", policy=policy, dtype=dtype, batch=B, n_layers=L, n_q_heads=4 * G, n_kv_heads=4,
                head_dim=d, n_sink=0, n_heavy=0, n_recent=0, budget=0, r=0, prompt_len=0, decode_steps=0,
                seed=77, max_prompt=0)
    base.update(kw)
    return configs.Workload(**base)


def _report(reps):
    return dict(units=len(reps), max_out_err=max(r.max_out_err for r in reps),
                max_score_err=max(r.max_score_err for r in reps), near_ties=sum(r.near_ties for r in reps))


def _all_units(w, layers):
    return [(s, l, h) for l in layers for s in range(w.batch) for h in range(w.n_kv_heads)]


# ----------------------------------------------------------------------------
# The tiny H2O workload, every unit, every step (fp32)
# ----------------------------------------------------------------------------

def test_h2o_tiny_lockstep(cuda_device, record_property):
    w = configs.H2O_TINY
    units = _all_units(w, [0])
    inputs = ls.host_inputs(w, units, w.decode_steps, w.prompt_len)
    snaps = range(w.decode_steps)
    run = ls.run_gpu(w, [0], w.decode_steps, inputs, w.prompt_len, cuda_device, snap_steps=snaps)
    assert run.err == 0
    reps = ls.replay_all(w, units, inputs, run, w.decode_steps)
    rep = _report(reps)
    print("h2o tiny:", rep)
    ls.record_ties(record_property, reps, max_near_ties=1)
    assert rep["max_out_err"] <= 1e-4 and rep["max_score_err"] <= 1e-4
    assert ls.check_selector(w, run, 0, w.prompt_len) == w.decode_steps


@pytest.mark.parametrize("split", [1, 2, 4])
def test_h2o_small_splits(cuda_device, split, record_property):
    """Ragged slot counts over several CTAs per unit; the cache fills during
    decode (prompt shorter than the budget) and then evicts."""
    w = _small(configs.POLICY_H2O, configs.DTYPE_F32, G=2, d=64, n_sink=3, n_heavy=40, n_recent=27, budget=70,
               prompt_len=37, decode_steps=90)
    units = _all_units(w, [0, 1])
    inputs = ls.host_inputs(w, units, w.decode_steps, w.prompt_len)
    run = ls.run_gpu(w, [0, 1], w.decode_steps, inputs, w.prompt_len, cuda_device,
                     snap_steps=range(0, w.decode_steps, 3), split=split, interleave=split != 2)
    assert run.split == split and run.err == 0
    reps = ls.replay_all(w, units, inputs, run, w.decode_steps)
    print(f"split {split}:", _report(reps))
    ls.record_ties(record_property, reps, max_near_ties=1)
    for layer in (0, 1):
        ls.check_selector(w, run, layer, w.prompt_len)


@pytest.mark.parametrize("policy,split,clusters", [
    (configs.POLICY_H2O, 1, 3), (configs.POLICY_H2O, 2, 5), (configs.POLICY_SINK_WINDOW, 1, 2),
    (configs.POLICY_SINK_WINDOW, 4, 3), (configs.POLICY_RANDOM, 2, 3)])
def test_persistent_loop_with_refills(cuda_device, policy, split, clusters, record_property):
    """Few clusters, many units each, and more K/V tiles per unit than ring
    stages: the ring keeps streaming across unit boundaries and every stage is
    refilled many times."""
    kw = {configs.POLICY_H2O: dict(n_sink=4, n_heavy=300, n_recent=100, budget=404, prompt_len=500),
          configs.POLICY_SINK_WINDOW: dict(n_sink=4, n_recent=700, budget=704, prompt_len=720),
          configs.POLICY_RANDOM: dict(budget=60, r=12, max_prompt=400, prompt_len=390)}[policy]
    T = 90
    w = _small(policy, configs.DTYPE_F32, G=2, d=64, B=5, L=1, decode_steps=T, **kw)
    units = _all_units(w, [0])
    inputs = ls.host_inputs(w, units, T, w.prompt_len)
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, cuda_device, snap_steps=range(0, T, 9), split=split,
                     clusters=clusters, alias=0)
    assert run.err == 0 and run.partials_alias == 0
    reps = ls.replay_all(w, units, inputs, run, T)
    print(f"persistent policy {policy} split {split} clusters {clusters}:", _report(reps))
    ls.record_ties(record_property, reps, max_near_ties=1)


@pytest.mark.parametrize("policy,G,dtype,B,split,clusters,budget,P,alias", [
    (configs.POLICY_H2O, 8, configs.DTYPE_BF16, 7, 2, 3, 96, 150, 0),     # tails of 0 and 1 unit
    (configs.POLICY_H2O, 4, configs.DTYPE_BF16, 9, 4, 2, 96, 150, 0),     # 4 whole + 2 split per cluster
    (configs.POLICY_H2O, 4, configs.DTYPE_F32, 5, 4, 3, 40, 20, 0),       # ranks with no tile; cache fills
    (configs.POLICY_SINK_WINDOW, 4, configs.DTYPE_BF16, 11, 2, 5, 70, 90, 0),
    (configs.POLICY_RANDOM, 4, configs.DTYPE_BF16, 7, 2, 3, 48, 60, 0),   # holes, free list, cuts
    (configs.POLICY_H2O_POOLS, 4, configs.DTYPE_BF16, 7, 2, 3, 64, 40, 0),
])
def test_tail_split_lockstep(cuda_device, policy, G, dtype, B, split, clusters, budget, P, alias, record_property):
    """Tail splitting: each CTA processes whole units alone and a cluster
    splits only its leftover units. Clusters with and without a tail, ranks
    with no tile of a split unit, the cache filling, Random's free list and
    the two-pool decision in split units."""
    kw = {configs.POLICY_H2O: dict(n_sink=2, n_heavy=budget - 2 - budget // 3, n_recent=budget // 3),
          configs.POLICY_SINK_WINDOW: dict(n_sink=4, n_recent=budget - 4),
          configs.POLICY_RANDOM: dict(budget=budget - 16, r=16, max_prompt=P),
          configs.POLICY_H2O_POOLS: dict(n_heavy=budget // 2, n_recent=budget - budget // 2,
                                         hh_threshold=0.012)}[policy]
    kw.setdefault("budget", budget)
    T = 90
    w = _small(policy, dtype, G=G, d=128 if dtype == configs.DTYPE_BF16 else 64, B=B, L=1, prompt_len=P,
               decode_steps=T, **kw)
    units = _all_units(w, [0])
    inputs = ls.host_inputs(w, units, T, P)
    run = ls.run_gpu(w, [0], T, inputs, P, cuda_device, snap_steps=range(0, T, 6), split=split, clusters=clusters,
                     tail_split=True, alias=alias)
    assert run.err == 0 and run.split == split and run.tail_split == 1 and run.partials_alias == alias
    reps = ls.replay_all(w, units, inputs, run, T)
    print(f"tail split policy {policy} G={G} S={split} clusters={clusters}:", _report(reps))
    ls.record_ties(record_property, reps, max_near_ties=1)
    if policy == configs.POLICY_H2O:
        ls.check_selector(w, run, 0, P)


@pytest.mark.parametrize("policy,split,tail,G,dtype", [
    (configs.POLICY_H2O, 1, False, 4, configs.DTYPE_F32),
    (configs.POLICY_H2O, 1, False, 8, configs.DTYPE_BF16),
    (configs.POLICY_H2O, 2, False, 4, configs.DTYPE_BF16),
    (configs.POLICY_H2O, 2, True, 8, configs.DTYPE_BF16),
    (configs.POLICY_SINK_WINDOW, 2, False, 4, configs.DTYPE_BF16),
    (configs.POLICY_SINK_WINDOW, 1, False, 4, configs.DTYPE_F32),
    (configs.POLICY_RANDOM, 2, False, 4, configs.DTYPE_BF16),
    (configs.POLICY_RANDOM, 2, True, 8, configs.DTYPE_BF16),
    (configs.POLICY_H2O_POOLS, 2, False, 4, configs.DTYPE_BF16),
    (configs.POLICY_H2O_POOLS, 1, False, 8, configs.DTYPE_BF16)])
def test_partials_over_logits_lockstep(cuda_device, policy, split, tail, G, dtype, record_property):
    """The warps' partial outputs written over the logits after the score
    pass (the layout that frees shared memory for ring stages), on units
    large enough for them to fit (>= 544 slots per CTA at head_dim 64): one
    CTA per unit, clusters, tail splitting; every policy's epilogue. (Built
    into the one-CTA-per-SM kernels, group sizes 4 and 8.)"""
    C = 1216
    kw = {configs.POLICY_H2O: dict(n_sink=4, n_heavy=C - 4 - 300, n_recent=300, budget=C, prompt_len=C + 30),
          configs.POLICY_SINK_WINDOW: dict(n_sink=4, n_recent=C - 4, budget=C, prompt_len=C + 10),
          configs.POLICY_RANDOM: dict(budget=64, r=16, max_prompt=C - 80, prompt_len=C - 80),
          configs.POLICY_H2O_POOLS: dict(n_heavy=C // 2, n_recent=C - C // 2, budget=C, prompt_len=C - 20,
                                         hh_threshold=0.0008)}[policy]
    T = 100
    w = _small(policy, dtype, G=G, d=64, B=3, L=1, decode_steps=T, **kw)
    units = _all_units(w, [0])
    inputs = ls.host_inputs(w, units, T, w.prompt_len)
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, cuda_device, snap_steps=range(0, T, 10), split=split,
                     clusters=5 if tail else None, tail_split=tail, alias=1)
    assert run.err == 0 and run.split == split and run.partials_alias == 1
    reps = ls.replay_all(w, units, inputs, run, T)
    print(f"partials over logits policy {policy} S={split} tail={tail} G={G}:", _report(reps))
    ls.record_ties(record_property, reps, max_near_ties=1)
    if policy == configs.POLICY_H2O:
        ls.check_selector(w, run, 0, w.prompt_len)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("G,d", [(1, 128), (2, 64), (4, 128), (8, 64), (8, 128)])
def test_h2o_small_bf16_gqa(cuda_device, G, d, path, record_property):
    """bf16 GQA on both decode paths: CUDA cores (1) and tensor cores (2)."""
    w = _small(configs.POLICY_H2O, configs.DTYPE_BF16, G=G, d=d, n_sink=2, n_heavy=50, n_recent=44, budget=96,
               prompt_len=150, decode_steps=70)
    units = _all_units(w, [0])
    inputs = ls.host_inputs(w, units, w.decode_steps, w.prompt_len)
    run = ls.run_gpu(w, [0], w.decode_steps, inputs, w.prompt_len, cuda_device, snap_steps=range(0, 70, 7),
                     path=path)
    assert run.err == 0 and run.tensor_cores == (path == 2)
    reps = ls.replay_all(w, units, inputs, run, w.decode_steps)
    print(f"G={G} d={d} path={path}:", _report(reps))
    ls.record_ties(record_property, reps, max_near_ties=1)
    ls.check_selector(w, run, 0, w.prompt_len)


@pytest.mark.parametrize("path", [1, 2])
def test_random_small_gqa_paths(cuda_device, path):
    """Random Attention with holes on both paths (G=4, bf16), several units
    per cluster."""
    w = _small(configs.POLICY_RANDOM, configs.DTYPE_BF16, G=4, d=128, B=4, L=2, budget=64, r=16,
               prompt_len=100, max_prompt=110, decode_steps=150)
    units = _all_units(w, [0, 1])
    inputs = ls.host_inputs(w, units, w.decode_steps, w.prompt_len)
    run = ls.run_gpu(w, [0, 1], w.decode_steps, inputs, w.prompt_len, cuda_device, snap_steps=range(0, 150, 5),
                     path=path, clusters=3)
    assert run.err == 0 and run.tensor_cores == (path == 2)
    reps = ls.replay_all(w, units, inputs, run, w.decode_steps)
    print(f"random G=4 path={path}:", _report(reps))


@pytest.mark.parametrize("P,T", [(0, 80), (45, 40)])
def test_sink_window_small(cuda_device, P, T):
    w = _small(configs.POLICY_SINK_WINDOW, configs.DTYPE_F32, G=1, d=64, n_sink=4, n_recent=33, budget=37,
               prompt_len=P, decode_steps=T)
    units = _all_units(w, [0, 1])
    inputs = ls.host_inputs(w, units, T, P)
    run = ls.run_gpu(w, [0, 1], T, inputs, P, cuda_device, snap_steps=range(T))
    assert run.err == 0
    reps = ls.replay_all(w, units, inputs, run, T)
    print("sink-window small:", _report(reps))


def test_random_small(cuda_device):
    w = _small(configs.POLICY_RANDOM, configs.DTYPE_BF16, G=2, d=128, budget=40, r=8, prompt_len=19,
               max_prompt=24, decode_steps=120)
    units = _all_units(w, [0, 1])
    inputs = ls.host_inputs(w, units, w.decode_steps, w.prompt_len)
    run = ls.run_gpu(w, [0, 1], w.decode_steps, inputs, w.prompt_len, cuda_device, snap_steps=range(120))
    assert run.err == 0
    reps = ls.replay_all(w, units, inputs, run, w.decode_steps)
    print("random small:", _report(reps))


@pytest.mark.parametrize("policy", [configs.POLICY_H2O, configs.POLICY_SINK_WINDOW, configs.POLICY_RANDOM])
def test_no_eviction_equals_full_attention(cuda_device, policy):
    """Budget >= sequence length: nothing is evicted and the output is full
    causal decode attention; compared with the oracle and with torch fp64
    scaled-dot-product attention."""
    P, T = 60, 50
    n = P + T
    kw = dict(h2o=dict(n_sink=4, n_heavy=n - 14, n_recent=10, budget=n),
              sw=dict(n_sink=4, n_recent=n, budget=n + 4),
              rnd=dict(budget=T, r=3, max_prompt=P))
    key = {configs.POLICY_H2O: "h2o", configs.POLICY_SINK_WINDOW: "sw", configs.POLICY_RANDOM: "rnd"}[policy]
    w = _small(policy, configs.DTYPE_F32, G=4, d=64, B=2, L=1, prompt_len=P, decode_steps=T, **kw[key])
    units = _all_units(w, [0])
    inputs = ls.host_inputs(w, units, T, P)
    run = ls.run_gpu(w, [0], T, inputs, P, cuda_device, snap_steps=[T - 1])
    ls.replay_all(w, units, inputs, run, T)
    import torch.nn.functional as F
    for (s, _, h), x in inputs.items():
        kk = np.concatenate([x.prompt_k, x.k_new]).astype(np.float64)
        vv = np.concatenate([x.prompt_v, x.v_new]).astype(np.float64)
        for t in (0, T // 2, T - 1):
            m = P + t + 1
            q = torch.from_numpy(x.q[t].astype(np.float64))[None, :, None, :]
            k = torch.from_numpy(kk[:m])[None, None].expand(1, w.group, m, w.head_dim)
            v = torch.from_numpy(vv[:m])[None, None].expand(1, w.group, m, w.head_dim)
            ref = F.scaled_dot_product_attention(q, k, v)[0, :, 0].numpy()
            got = run.out[0][s][t, h * w.group:(h + 1) * w.group]
            assert np.max(np.abs(got - ref)) <= 1e-4


@pytest.mark.parametrize("policy", [configs.POLICY_H2O, configs.POLICY_SINK_WINDOW, configs.POLICY_RANDOM])
def test_prefill_layout_chunked(cuda_device, policy):
    """Prompt appended in chunks: the slot table after prefill equals the
    oracle's token-by-token admission."""
    kw = {configs.POLICY_H2O: dict(n_sink=3, n_heavy=10, n_recent=8, budget=21),
          configs.POLICY_SINK_WINDOW: dict(n_sink=3, n_recent=18, budget=21),
          configs.POLICY_RANDOM: dict(budget=10, r=4, max_prompt=70)}[policy]
    w = _small(policy, configs.DTYPE_BF16, G=1, d=64, B=2, L=1, **kw)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    chunks = [2, 1, 30, 5, 0, 25]
    P = sum(chunks)
    prompts = {(s, h): synth.UnitInputs(w, s, 0, h, 1, P) for s in range(2) for h in range(4)}
    p0 = 0
    for c in chunks:
        K = torch.empty((2, 4, c, 64), dtype=torch.bfloat16, device=cuda_device)
        V = torch.empty_like(K)
        for (s, h), x in prompts.items():
            K[s, h] = torch.from_numpy(x.prompt_k[p0:p0 + c]).to(torch.bfloat16)
            V[s, h] = torch.from_numpy(x.prompt_v[p0:p0 + c]).to(torch.bfloat16)
        cache.prefill(0, K, V)
        p0 += c
    pos = cache.slot_positions(0).cpu().numpy()
    assert cache.layer_state(0)[0] == P
    for (s, h), x in prompts.items():
        u = oracle.Unit.for_workload(w, s, 0, h)
        u.prefill(x.prompt_k, x.prompt_v)
        np.testing.assert_array_equal(pos[s, h], u.positions())


def test_host_buffer_path_matches_device_path(cuda_device):
    w = _small(configs.POLICY_H2O, configs.DTYPE_BF16, G=4, d=128, B=2, L=1, n_sink=2, n_heavy=20,
               n_recent=10, budget=32, prompt_len=40, decode_steps=12)
    a = KVEvictCache.from_workload(w, device=cuda_device)
    b = KVEvictCache.from_workload(w, device=cuda_device)
    K, V = synth.device_prompt(w, 0, cuda_device, 40)
    a.prefill(0, K, V)
    b.prefill(0, K, V)
    g = torch.Generator(device=cuda_device)
    g.manual_seed(5)
    for t in range(w.decode_steps):
        q = torch.randn((2, 16, 128), generator=g, device=cuda_device).to(torch.bfloat16)
        k = torch.randn((2, 4, 128), generator=g, device=cuda_device).to(torch.bfloat16)
        v = torch.randn((2, 4, 128), generator=g, device=cuda_device).to(torch.bfloat16)
        o1 = a.decode_step(0, q, k, v)
        o2 = torch.empty((2, 16, 128), dtype=torch.bfloat16).pin_memory()
        b.decode_step_host(0, q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(), o2)
        assert torch.equal(o1.cpu(), o2)
    assert torch.equal(a.slot_positions(0), b.slot_positions(0))
    assert torch.equal(a.scores(0), b.scores(0))


@pytest.mark.parametrize("policy,pinned", [(configs.POLICY_H2O, True), (configs.POLICY_RANDOM, True),
                                           (configs.POLICY_H2O, False)])
def test_host_async_path_matches_device_path(cuda_device, policy, pinned):
    """The host-buffer calls that do not wait, three layers a token and one
    sync per token (Random's cut launches inside): outputs, slot tables and
    scores equal the device path's. Pinned buffers the GPU can address are read
    and written in place by the kernels; pageable ones go through the staging
    slots and the copy streams."""
    from kv_cache_eviction_decode_gb300 import lib
    mapped = lib().kvevict_host_buffer_mapped
    kw = dict(n_sink=2, n_heavy=20, n_recent=10, budget=32, prompt_len=40) if policy == configs.POLICY_H2O else \
        dict(budget=12, r=4, max_prompt=40, prompt_len=40)
    w = _small(policy, configs.DTYPE_BF16, G=4, d=128, B=2, L=3, decode_steps=14, **kw)
    a = KVEvictCache.from_workload(w, device=cuda_device)
    b = KVEvictCache.from_workload(w, device=cuda_device)
    for layer in range(w.n_layers):
        K, V = synth.device_prompt(w, layer, cuda_device, w.prompt_len)
        a.prefill(layer, K, V)
        b.prefill(layer, K, V)
    g = torch.Generator(device=cuda_device)
    g.manual_seed(6)
    for t in range(w.decode_steps):
        host = []
        for layer in range(w.n_layers):
            q = torch.randn((2, 16, 128), generator=g, device=cuda_device).to(torch.bfloat16)
            k = torch.randn((2, 4, 128), generator=g, device=cuda_device).to(torch.bfloat16)
            v = torch.randn((2, 4, 128), generator=g, device=cuda_device).to(torch.bfloat16)
            o1 = a.decode_step(layer, q, k, v)
            ins = tuple(x.cpu().pin_memory() if pinned else x.cpu() for x in (q, k, v))
            o2 = torch.empty((2, 16, 128), dtype=torch.bfloat16)
            if pinned:
                o2 = o2.pin_memory()
            if not pinned:
                assert not any(mapped(x.data_ptr()) for x in (*ins, o2))
            b.decode_step_host_async(layer, *ins, o2)
            host.append((o1, ins, o2))  # the host buffers stay alive until the sync
        b.sync()
        for o1, _, o2 in host:
            assert torch.equal(o1.cpu(), o2)
    for layer in range(w.n_layers):
        assert torch.equal(a.slot_positions(layer), b.slot_positions(layer))
        if policy == configs.POLICY_H2O:
            assert torch.equal(a.scores(layer), b.scores(layer))
    assert a.check() == 0 and b.check() == 0


def test_nonfinite_query_sets_error_bit_and_continues(cuda_device):
    """A NaN planted in q: the step completes, the device error word reports
    it, nothing traps, and the handle keeps working."""
    w = _small(configs.POLICY_H2O, configs.DTYPE_F32, G=1, d=64, B=1, L=1, n_sink=1, n_heavy=4, n_recent=3,
               budget=8, prompt_len=8, decode_steps=3)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    K, V = synth.device_prompt(w, 0, cuda_device, 8)
    cache.prefill(0, K, V)
    q = torch.randn((1, 4, 64), device=cuda_device)
    k = torch.randn((1, 4, 64), device=cuda_device)
    v = torch.randn((1, 4, 64), device=cuda_device)
    cache.decode_step(0, q, k, v)
    assert cache.check() == 0
    q[0, 2, 5] = float("nan")
    cache.decode_step(0, q, k, v)
    assert cache.check() & DEV_NONFINITE
    q[0, 2, 5] = 0.0
    cache.decode_step(0, q, k, v)
    torch.cuda.synchronize()
    assert cache.layer_state(0)[1] == 3


def test_wait_timeout_is_reported_and_the_handle_keeps_working(cuda_device):
    """A bounded wait on a barrier nothing completes (the decode pipeline's own
    wait) gives up after its limit: the device error word reports
    DEV_WAIT_TIMEOUT, nothing faults, and decode steps go on with a clean word."""
    from kv_cache_eviction_decode_gb300 import DEV_WAIT_TIMEOUT
    import time
    w = _small(configs.POLICY_H2O, configs.DTYPE_F32, G=1, d=64, B=1, L=1, n_sink=1, n_heavy=4, n_recent=3,
               budget=8, prompt_len=8, decode_steps=3)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    K, V = synth.device_prompt(w, 0, cuda_device, 8)
    cache.prefill(0, K, V)
    q = torch.randn((1, 4, 64), device=cuda_device)
    k = torch.randn((1, 4, 64), device=cuda_device)
    cache.decode_step(0, q, k, k)
    assert cache.check() == 0
    t0 = time.perf_counter()
    cache.probe_wait_timeout()
    assert cache.check() == DEV_WAIT_TIMEOUT
    assert time.perf_counter() - t0 >= 1.5  # the wait ran to its limit
    assert cache.check() == 0  # read and cleared
    out = cache.decode_step(0, q, k, k)
    assert cache.check() == 0 and torch.isfinite(out).all()
    assert cache.layer_state(0)[1] == 2
    cache.close()


def test_state_errors_on_device_handle(cuda_device):
    from kv_cache_eviction_decode_gb300 import KVEvictError
    w = _small(configs.POLICY_RANDOM, configs.DTYPE_F32, G=1, d=64, B=1, L=2, budget=8, r=2, max_prompt=10)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    K = torch.zeros((1, 4, 11, 64), device=cuda_device)
    with pytest.raises(KVEvictError):       # prompt beyond max_prompt
        cache.prefill(0, K, K)
    q = torch.zeros((1, 4, 64), device=cuda_device)
    with pytest.raises(KVEvictError):       # layer out of range
        cache.decode_step(2, q, q, q)
    cache.decode_step(1, q, q, q)
    with pytest.raises(KVEvictError):       # prefill after decode
        cache.prefill(1, K[:, :, :2].contiguous(), K[:, :, :2].contiguous())
    assert cache.check() == 0


# ----------------------------------------------------------------------------
# The benchmark workloads at full shape (sampled units, checked layers)
# ----------------------------------------------------------------------------

def test_sink_window_full_shape(cuda_device):
    """StreamingLLM 4 + 1020 at B=64, 32x32 heads, d=128: positions 0..1099
    streamed from an empty cache (fill, then ring)."""
    w = configs.SINK_WINDOW
    T = 1100
    layers = [0, w.n_layers - 1]
    checked = [(s, l, h) for l in layers for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, checked, T, 0)
    run = ls.run_gpu(w, layers, T, inputs, 0, cuda_device, snap_steps=[1022, 1023, 1024, T - 1])
    assert run.err == 0
    out_steps = set(range(0, T, 61)) | {1023, 1024, T - 1}
    reps = ls.replay_all(w, checked, inputs, run, T, out_steps=out_steps)
    print("sink-window full shape:", _report(reps), "split", run.split)
    # every unit of the checked layers: the ring slot, bit-exact
    for layer in layers:
        tr = run.trace[layer]
        for t in range(T):
            want = t if t < w.n_sink else w.n_sink + (t - w.n_sink) % w.n_recent
            assert np.all(tr[t, ..., 0] == want)


def test_h2o_mha_full_shape(cuda_device, record_property):
    """H2O 4 + 510 + 510 at B=16, 32x32 heads, d=128, prompt 2048."""
    w = configs.H2O_MHA
    T = 320
    layers = [0, w.n_layers - 1]
    checked = [(s, l, h) for l in layers for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, checked, T, w.prompt_len)
    snaps = [0, 1, 100, 200, T - 1]
    run = ls.run_gpu(w, layers, T, inputs, w.prompt_len, cuda_device, snap_steps=snaps)
    assert run.err == 0
    reps = ls.replay_all(w, checked, inputs, run, T)
    rep = _report(reps)
    print("h2o mha full shape:", rep, "split", run.split)
    ls.record_ties(record_property, reps, max_near_ties=5)
    for layer in layers:
        assert ls.check_selector(w, run, layer, w.prompt_len) == len(snaps)


def test_h2o_gqa_full_shape(cuda_device, record_property):
    """H2O GQA 64 query / 8 KV heads, K=2048, B=64, context 32768, 512 steps."""
    w = configs.H2O_GQA
    T = w.decode_steps
    checked = [(s, 0, h) for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, checked, T, w.prompt_len)
    snaps = [0, 255, T - 1]
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, cuda_device, snap_steps=snaps)
    assert run.err == 0
    reps = ls.replay_all(w, checked, inputs, run, T)
    print("h2o gqa full shape:", _report(reps), "split", run.split)
    ls.record_ties(record_property, reps, max_near_ties=5)
    assert ls.check_selector(w, run, 0, w.prompt_len) == len(snaps)


def test_tail_split_refused_by_two_cta_kernels(cuda_device):
    """Group sizes 1 and 2 run two CTAs per SM and do not build tail
    splitting; asking for it is an argument error and changes nothing."""
    from kv_cache_eviction_decode_gb300 import KVEvictError
    w = _small(configs.POLICY_H2O, configs.DTYPE_BF16, G=2, d=128, B=2, L=1, n_sink=2, n_heavy=60, n_recent=34,
               budget=96, prompt_len=10)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    with pytest.raises(KVEvictError):
        cache.set_tail_split(True)
    assert cache.stats()["tail_split"] == 0
    cache.set_partials_alias(1)  # accepted, and never applied: the partials keep their own area
    K, V = synth.device_prompt(w, 0, cuda_device, 10)
    cache.prefill(0, K, V)
    q = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device=cuda_device)
    k = torch.zeros((2, 4, 128), dtype=torch.bfloat16, device=cuda_device)
    cache.decode_step(0, q, k, k)
    assert cache.check() == 0 and cache.stats()["partials_alias"] == 0
    cache.close()


def test_h2o_gqa_full_shape_tail_split(cuda_device, record_property):
    """The GQA workload with tail splitting at clusters of two: every CTA of
    the GPU processes whole units and the clusters split their leftover unit."""
    w = configs.H2O_GQA
    T = 160
    checked = [(s, 0, h) for s in (0, 1, w.batch - 2, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, checked, T, w.prompt_len)
    snaps = [0, 80, T - 1]
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, cuda_device, snap_steps=snaps, split=2, tail_split=True)
    assert run.err == 0 and run.split == 2 and run.tail_split == 1
    reps = ls.replay_all(w, checked, inputs, run, T)
    print("h2o gqa full shape, tail split:", _report(reps))
    ls.record_ties(record_property, reps, max_near_ties=5)
    assert ls.check_selector(w, run, 0, w.prompt_len) == len(snaps)


def test_random_full_shape(cuda_device):
    """Random Attention, prompt 8192 kept, K=2048, r=128, B=32, 32 layers x
    8 KV heads (32 query heads): four cuts. Slot tables of every unit of the
    checked layers replayed bit-exactly; outputs of sampled units at sampled
    steps."""
    w = configs.RANDOM_REASONING
    first_cut = w.budget + w.r - 1
    T = first_cut + 3 * w.r + 2
    layers = [0, w.n_layers - 1]
    with_values = [(s, l, h) for l in layers for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, with_values, T, w.prompt_len)
    cuts = [first_cut + i * w.r for i in range(4)]
    snaps = sorted(set(cuts) | {c + 1 for c in cuts} | {0, T - 1})
    run = ls.run_gpu(w, layers, T, inputs, w.prompt_len, cuda_device, snap_steps=snaps)
    assert run.err == 0
    out_steps = {0, 1, 1000, first_cut, first_cut + 1, first_cut + 70, cuts[-1] + 1, T - 1}
    every_unit = _all_units(w, layers)
    reps = ls.replay_all(w, every_unit, inputs, run, T, out_steps=out_steps)
    print("random full shape:", _report(reps), "split", run.split)
    assert sum(r.out_checks for r in reps) == len(with_values) * len(out_steps)


def test_h2o_reasoning_full_shape(cuda_device, record_property):
    """H2O on the long-reasoning shape: the 8192-token prompt protected, 1024
    heavy + 1024 recent, K=10240; the cache fills for 2048 steps, then
    evicts."""
    w = configs.H2O_REASONING
    T = 2048 + 64
    checked = [(0, 0, h) for h in range(w.n_kv_heads)] + [(w.batch - 1, 0, h) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, checked, T, w.prompt_len)
    snaps = [2047, 2048, 2080, T - 1]
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, cuda_device, snap_steps=snaps)
    assert run.err == 0
    reps = ls.replay_all(w, checked, inputs, run, T)
    print("h2o reasoning full shape:", _report(reps), "split", run.split)
    ls.record_ties(record_property, reps, max_near_ties=5)
    assert ls.check_selector(w, run, 0, w.prompt_len) >= 3
