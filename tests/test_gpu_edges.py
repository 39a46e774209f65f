"""GPU parity at the edges of the method, in lockstep with the CPU oracle
(same tolerances as the parity tests: 1e-4 max-abs for fp32, 2e-2 relative
for bf16; slot tables bit-exact, H2O victims equal up to counted near-ties):

  - decode from an empty cache (no prompt) for every policy: the cache fills
    during decode, then evicts;
  - the smallest caches: a budget of 1 (H2O keeps only the newest token, the
    ring holds one slot) and of 2;
  - degenerate H2O parts: no sinks, no heavy hitters (a pure recent window),
    a single recent slot;
  - Random with a buffer of r = 1 (a cut every step);
  - one unit in all (batch 1, one KV head), and the widest cluster split (16).
"""
import pytest

from tests import lockstep as ls
from workloads import configs

pytestmark = pytest.mark.gpu

F32, BF16 = configs.DTYPE_F32, configs.DTYPE_BF16


def _w(policy, dtype=F32, G=2, d=64, B=2, Hkv=3, **kw):
    base = dict(name="edge", policy=policy, dtype=dtype, batch=B, n_layers=1, n_q_heads=G * Hkv, n_kv_heads=Hkv,
                head_dim=d, n_sink=0, n_heavy=0, n_recent=0, budget=0, r=0, prompt_len=0, decode_steps=0,
                seed=505, max_prompt=0)
    base.update(kw)
    return configs.Workload(**base)


def _lockstep(w, T, split=None, snaps=None):
    units = [(s, 0, h) for s in range(w.batch) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, units, T, w.prompt_len)
    run = ls.run_gpu(w, [0], T, inputs, w.prompt_len, "cuda:0", snap_steps=snaps if snaps is not None else range(T),
                     split=split)
    assert run.err == 0
    if split:
        assert run.split == split
    reps = ls.replay_all(w, units, inputs, run, T)
    assert all(r.steps == T for r in reps)
    return run, reps


@pytest.mark.parametrize("w", [
    _w(configs.POLICY_H2O, n_sink=2, n_heavy=20, n_recent=10, budget=32),
    _w(configs.POLICY_H2O, BF16, G=4, d=128, n_sink=2, n_heavy=20, n_recent=10, budget=32),
    _w(configs.POLICY_SINK_WINDOW, n_sink=4, n_recent=28, budget=32),
    _w(configs.POLICY_RANDOM, budget=24, r=8, max_prompt=0),
    _w(configs.POLICY_H2O_BLOCK, n_sink=2, n_heavy=18, n_recent=12, budget=32, r=8),
    _w(configs.POLICY_H2O_POOLS, n_heavy=20, n_recent=12, budget=32, hh_threshold=0.01),
], ids=["h2o", "h2o_bf16_gqa", "sink_window", "random", "h2o_block", "h2o_pools"])
def test_decode_from_an_empty_cache(cuda_device, w):
    run, reps = _lockstep(w, 90)
    # the first step attends over the new token alone: no slot held before it
    assert (run.pos_snap[0][-1].numpy() == -1).all()


@pytest.mark.parametrize("w", [
    _w(configs.POLICY_H2O, n_recent=1, budget=1, prompt_len=5),          # only the newest token stays
    _w(configs.POLICY_H2O, n_sink=1, n_recent=1, budget=2, prompt_len=7),
    _w(configs.POLICY_H2O, n_heavy=1, n_recent=1, budget=2, prompt_len=3),
    _w(configs.POLICY_SINK_WINDOW, n_recent=1, budget=1, prompt_len=4),  # a one-slot ring
    _w(configs.POLICY_H2O_POOLS, n_recent=1, budget=1, prompt_len=4, hh_threshold=0.0),
], ids=["h2o_budget1", "h2o_sink1_recent1", "h2o_heavy1_recent1", "ring1", "pools_recent1"])
def test_smallest_caches(cuda_device, w):
    run, _ = _lockstep(w, 40)
    if w.budget == 1:
        # after every step the one slot holds the newest token
        for t, pos in run.pos_snap[0].items():
            if t >= 0 and w.policy != configs.POLICY_H2O_POOLS:
                assert (pos.numpy()[..., 0] == w.prompt_len + t).all()


def test_h2o_without_sinks_or_heavy_hitters_is_a_window(cuda_device):
    """n_sink = n_heavy = 0: H2O keeps exactly the last n_recent positions,
    the StreamingLLM ring without sinks; both run in lockstep with the oracle
    and hold the same position sets."""
    T = 60
    wh = _w(configs.POLICY_H2O, n_recent=16, budget=16, prompt_len=20)
    ws = _w(configs.POLICY_SINK_WINDOW, n_recent=16, budget=16, prompt_len=20)
    rh, _ = _lockstep(wh, T)
    rs, _ = _lockstep(ws, T)
    for t in range(T):
        a, b = rh.pos_snap[0][t].numpy(), rs.pos_snap[0][t].numpy()
        for s in range(wh.batch):
            for h in range(wh.n_kv_heads):
                assert sorted(a[s, h]) == sorted(b[s, h]) == list(range(20 + t - 15, 20 + t + 1))


def test_random_cut_every_step(cuda_device):
    w = _w(configs.POLICY_RANDOM, budget=12, r=1, max_prompt=10, prompt_len=10)
    run, _ = _lockstep(w, 50)
    assert all(int(x) == 10 + 12 for x in (run.pos_snap[0][49].numpy() >= 0).sum(axis=2).ravel())


@pytest.mark.parametrize("policy", [configs.POLICY_H2O, configs.POLICY_SINK_WINDOW, configs.POLICY_H2O_POOLS])
def test_one_unit(cuda_device, policy):
    kw = {configs.POLICY_H2O: dict(n_sink=2, n_heavy=30, n_recent=20, budget=52),
          configs.POLICY_SINK_WINDOW: dict(n_sink=2, n_recent=50, budget=52),
          configs.POLICY_H2O_POOLS: dict(n_heavy=30, n_recent=22, budget=52, hh_threshold=0.005)}[policy]
    w = _w(policy, B=1, Hkv=1, G=8, d=128, dtype=BF16, prompt_len=70, **kw)
    _lockstep(w, 60)


@pytest.mark.parametrize("policy", [configs.POLICY_H2O, configs.POLICY_H2O_POOLS])
def test_widest_split(cuda_device, policy):
    """16 CTAs per unit (a non-portable cluster), a few slots per CTA and some
    CTAs with none while the cache fills."""
    kw = {configs.POLICY_H2O: dict(n_sink=4, n_heavy=400, n_recent=200, budget=604),
          configs.POLICY_H2O_POOLS: dict(n_heavy=400, n_recent=204, budget=604, hh_threshold=0.002)}[policy]
    w = _w(policy, B=2, Hkv=2, prompt_len=300, **kw)
    _lockstep(w, 80, split=16, snaps=range(0, 80, 5))
