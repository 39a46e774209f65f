"""GPU parity of two-pool H2O (the H2OCache class of "KV Cache 驱逐策略：从 LRU 到
H2O", section "实现要点": recent pool, heavy-hitter pool, hh_threshold) through
the C ABI, in lockstep with the CPU oracle.

Outputs and scores as for H2O (2e-2 relative for bf16, 1e-4 max-abs for
fp32). Every step's decision (the slot the new token takes or its leaving,
the pool it joins, the promoted slot) equals the oracle's, except where one
of the comparisons that decided the oracle's was within 1e-5 relative (the
GPU sums in fp32, the oracle in fp64); the oracle then adopts the GPU's. The
decision is also checked bit-exact against the rule applied to the GPU's own
stored values, over runs of consecutive snapshots.
"""
import numpy as np
import pytest

from kv_cache_eviction_decode_gb300 import BF16, F32, H2O_POOLS, KVEvictCache, KVEvictError
from tests import lockstep as ls
from workloads import configs

pytestmark = pytest.mark.gpu


def _small(dtype, theta, forget=0.0, half=False, n_recent=24, n_heavy=40, prompt=30, G=2):
    return configs.Workload(name="pools", policy=H2O_POOLS, dtype=dtype, batch=3, n_layers=1, n_q_heads=4 * G,
                            n_kv_heads=4, head_dim=64, n_sink=0, n_heavy=n_heavy, n_recent=n_recent,
                            budget=n_heavy + n_recent, r=0, prompt_len=prompt, decode_steps=0, seed=93,
                            score_forget=forget, score_half=half, hh_threshold=theta)


def _key(score_f32, pos):
    """(score bits << 32 | position) of a non-negative fp32 score."""
    return (int(np.float32(score_f32).view(np.uint32)) << 32) | (int(pos) & 0xFFFFFFFF)


def _score_of(key):
    return np.array([key >> 32], np.uint32).view(np.float32)[0]


def check_decisions(w, run, layer, prompt_len):
    """Bit-exact: at every step t whose previous step t-1 is also a snapshot,
    the GPU's decision (trace: slot, position that left, promotion record) is
    the rule applied to its own fp32 values -- the pools before the step
    (snapshot t-1) and the scores after this step's update (snapshot t; a
    token that left carries its score in the trace). Returns the number of
    unit-steps checked."""
    checked = 0
    theta = np.float32(w.hh_threshold)
    for t, pos_t in run.pos_snap[layer].items():
        if t < 0 or t - 1 not in run.pos_snap[layer]:
            continue
        pos0, pool0 = run.pos_snap[layer][t - 1].numpy(), run.pool_snap[layer][t - 1].numpy()
        pos1, sc1 = pos_t.numpy(), run.score_snap[layer][t].numpy()
        tr = run.trace[layer][t]
        p = prompt_len + t
        B, Hkv, _ = pos0.shape
        for b in range(B):
            for h in range(Hkv):
                dest, old_pos, old_bits, rec = (int(x) for x in tr[b, h])
                old_score = np.array([old_bits], np.int32).view(np.float32)[0]
                held = pos0[b, h] >= 0
                sc = {}
                for s in np.flatnonzero(held):
                    if pos1[b, h, s] == pos0[b, h, s]:
                        sc[s] = sc1[b, h, s]
                    else:  # only the slot the new token took changes
                        assert s == dest and pos0[b, h, s] == old_pos, (t, b, h, s)
                        sc[s] = old_score
                new_score = sc1[b, h, dest] if dest >= 0 else old_score
                key = {s: _key(sc[s], pos0[b, h, s]) for s in sc}
                rec_keys = sorted((key[s], s) for s in sc if pool0[b, h, s] == 0)
                hh_keys = sorted((key[s], s) for s in sc if pool0[b, h, s] == 1)
                empty = np.flatnonzero(~held)
                em = int(empty[0]) if len(empty) else None
                kn = _key(new_score, p)
                if len(rec_keys) < w.n_recent:  # room in the recent pool
                    want = (em, -1, -1)
                else:
                    kv, sv = rec_keys[0]
                    v_new = kn < kv
                    k = kn if v_new else kv
                    kw, sw = hh_keys[0] if hh_keys else (2**64 - 1, -1)
                    if not (_score_of(k) > theta) or (em is None and k < kw):  # v leaves the cache
                        want = (-1 if v_new else sv, int(k & 0xFFFFFFFF), -1)
                    elif em is not None:  # promoted into a pool with room
                        want = (em, -1, -2 if v_new else sv)
                    else:  # promoted; the heavy-hitter pool's lowest leaves
                        want = (sw, int(pos0[b, h, sw]), -2 if v_new else sv)
                assert (dest, old_pos, rec) == want, (t, b, h, (dest, old_pos, rec), want)
                checked += 1
    return checked


@pytest.mark.parametrize("dtype,theta,forget,half,split", [
    (BF16, 0.012, 0.0, False, None), (BF16, 0.0, 0.0, False, 2), (F32, 0.02, 0.1, False, None),
    (BF16, 0.015, 0.0, True, 4), (F32, -1.0, 0.0, False, None), (BF16, 0.05, 0.2, False, 2)])
def test_pools_lockstep(cuda_device, dtype, theta, forget, half, split, record_property):
    w = _small(dtype, theta, forget, half)
    T = 160
    units = [(s, 0, h) for s in range(w.batch) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, units, T, w.prompt_len)
    snaps = sorted(set(range(0, T, 16)) | set(range(60, 90)))
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, cuda_device, snap_steps=snaps, split=split)
    assert run.err == 0
    if split:
        assert run.split == split
    reps = ls.replay_all(w, units, inputs, run, T)
    tr = run.trace[0]
    n_prom = int(np.sum(tr[..., 3] != -1))
    n_drop_new = int(np.sum(tr[..., 0] == -1))
    print(f"theta {theta} forget {forget} half {half} split {run.split}: promotions {n_prom}, new token left "
          f"{n_drop_new}, near ties {sum(r.near_ties for r in reps)}, "
          f"out {max(r.max_out_err for r in reps):.2e}")
    ls.record_ties(record_property, reps, max_near_ties=3, max_near_tie_rate=2e-3 if half else 0.0)
    assert check_decisions(w, run, 0, w.prompt_len) >= 30 * len(units)
    n_left = n_drop_new + int(np.sum((tr[..., 0] >= 0) & (tr[..., 1] >= 0)))  # a token left the cache
    assert n_prom > 0 and n_left > 0


def test_pools_prefill_layout(cuda_device):
    """The prompt layout (every score 0): a ring of n_recent slots for a
    threshold >= 0, of C slots with the older part in the heavy-hitter pool
    for a threshold < 0."""
    import torch
    for theta in (0.5, -0.5):
        w = _small(BF16, theta, prompt=150)
        c = KVEvictCache.from_workload(w, device=cuda_device)
        K = torch.randn((w.batch, w.n_kv_heads, w.prompt_len, w.head_dim), device=cuda_device).to(torch.bfloat16)
        c.prefill(0, K, K)
        pos = c.slot_positions(0).cpu().numpy()
        pools = c.pools(0).cpu().numpy()
        ring = w.n_recent if theta >= 0 else w.budget
        want = np.full(w.budget, -1)
        want_pool = np.zeros(w.budget, np.uint8)
        for q in range(w.prompt_len - ring, w.prompt_len):
            want[q % ring] = q
            want_pool[q % ring] = q < w.prompt_len - w.n_recent
        assert np.all(pos == want)
        held = want >= 0
        assert np.all(pools[..., held] == want_pool[held])
        assert c.layer_state(0)[2] == min(ring, w.prompt_len)
        with pytest.raises(KVEvictError):  # the whole prompt in one call
            c.prefill(0, K, K)
        c.close()


def test_pools_rejected_configs(cuda_device):
    base = dict(batch=1, n_layers=1, n_q_heads=2, n_kv_heads=2, head_dim=64, dtype=BF16, device=cuda_device)
    for bad in [dict(n_sink=2, n_heavy=30, n_recent=32, budget=64),   # no sinks
                dict(n_sink=0, n_heavy=30, n_recent=32, budget=64),   # pools do not add up
                dict(n_sink=0, n_heavy=64, n_recent=0, budget=64),    # empty recent pool
                dict(n_sink=0, n_heavy=32, n_recent=32, budget=64, hh_threshold=float("nan"))]:
        with pytest.raises(KVEvictError):
            KVEvictCache(policy=H2O_POOLS, **base, **bad)
    c = KVEvictCache(policy=configs.POLICY_H2O, budget=64, n_sink=2, n_heavy=30, n_recent=32, **base)
    with pytest.raises(KVEvictError):  # pool flags exist for the two-pool policy only
        c.pools(0)
    c.close()


def test_pools_full_shape(cuda_device, record_property):
    """Two-pool H2O 512 recent + 512 heavy hitters on the MHA shape (B=16,
    32x32 heads, d=128, prompt 2048), 300 steps; sequences {0, 15} x every
    head of layers {0, 31} in lockstep, decisions bit-exact over a run of
    snapshots."""
    w = configs.H2O_POOLS_MHA
    T = 300
    layers = [0, w.n_layers - 1]
    checked = [(s, l, h) for l in layers for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, checked, T, w.prompt_len)
    snaps = [0, 150, 151, 152, T - 1]
    run = ls.run_gpu(w, layers, T, inputs, w.prompt_len, cuda_device, snap_steps=snaps)
    assert run.err == 0
    reps = ls.replay_all(w, checked, inputs, run, T, out_steps=range(0, T, 7))
    n = ls.record_ties(record_property, reps, max_near_ties=8)
    print("pools full shape:", n, "max out err", max(r.max_out_err for r in reps))
    for layer in layers:
        assert check_decisions(w, run, layer, w.prompt_len) == 3 * w.batch * w.n_kv_heads
