"""Checkpoint and resume through the C ABI: a handle restored from a
checkpoint continues exactly as the run that was saved (outputs, slot
tables, scores, counters and stats bit-identical) for H2O, whose scores
decide the victims, Random, whose cuts follow counter-based keys, and H2O
with INT8 scores; a record of another configuration is refused."""
import pytest
import torch

from kv_cache_eviction_decode_gb300 import KVEvictCache, KVEvictError
from workloads import configs, synth

pytestmark = pytest.mark.gpu


def _w(policy, **kw):
    base = dict(name="ckpt", policy=policy, dtype=configs.DTYPE_BF16, batch=2, n_layers=2, n_q_heads=8,
                n_kv_heads=4, head_dim=64, n_sink=2, n_heavy=20, n_recent=10, budget=32, r=0, prompt_len=24,
                decode_steps=0, seed=77, max_prompt=0)
    base.update(kw)
    return configs.Workload(**base)


CASES = {
    "h2o": _w(configs.POLICY_H2O),
    "random": _w(configs.POLICY_RANDOM, n_sink=0, n_heavy=0, n_recent=0, budget=16, r=8, max_prompt=24),
    "h2o_int8": _w(configs.POLICY_H2O, score_int8=True),
}


def _steps(cache, w, n, seed):
    g = torch.Generator(device=cache.device).manual_seed(seed)
    outs = []
    for _ in range(n):
        q = torch.randn((w.batch, w.n_q_heads, w.head_dim), generator=g, device=cache.device).to(cache.dtype)
        k = torch.randn((w.batch, w.n_kv_heads, w.head_dim), generator=g, device=cache.device).to(cache.dtype)
        v = torch.randn((w.batch, w.n_kv_heads, w.head_dim), generator=g, device=cache.device).to(cache.dtype)
        for layer in range(w.n_layers):
            outs.append(cache.decode_step(layer, q, k, v).clone())
    torch.cuda.synchronize()
    return outs


def _snapshot(cache, w):
    scored = w.policy != configs.POLICY_RANDOM
    st = cache.stats()
    return ([cache.slot_positions(l).cpu() for l in range(w.n_layers)],
            [cache.scores(l).cpu() for l in range(w.n_layers)] if scored else [],
            [cache.layer_state(l) for l in range(w.n_layers)],
            {k: st[k] for k in ("decode_steps", "prefill_tokens", "evictions", "cuts")})


@pytest.mark.parametrize("name", list(CASES))
def test_resume_is_bit_exact(cuda_device, name):
    w = CASES[name]
    a = KVEvictCache.from_workload(w, device=cuda_device)
    for layer in range(w.n_layers):
        K, V = synth.device_prompt(w, layer, cuda_device, w.prompt_len)
        a.prefill(layer, K, V)
    _steps(a, w, 20, 1)
    ck = a.checkpoint()
    out_a = _steps(a, w, 30, 2)
    snap_a = _snapshot(a, w)
    assert a.check() == 0
    a.close()

    b = KVEvictCache.from_workload(w, device=cuda_device)
    b.restore(ck)
    out_b = _steps(b, w, 30, 2)
    snap_b = _snapshot(b, w)
    assert b.check() == 0
    b.close()

    assert len(out_a) == len(out_b) == 30 * w.n_layers
    assert all(torch.equal(x, y) for x, y in zip(out_a, out_b))
    for x, y in zip(snap_a[0] + snap_a[1], snap_b[0] + snap_b[1]):
        assert torch.equal(x, y)
    assert snap_a[2] == snap_b[2] and snap_a[3] == snap_b[3]
    if w.policy == configs.POLICY_RANDOM:
        assert snap_a[3]["cuts"] > 0  # the resumed part crossed cuts


def test_restore_refuses_another_configuration(cuda_device):
    w = CASES["h2o"]
    a = KVEvictCache.from_workload(w, device=cuda_device)
    ck = a.checkpoint()
    b = KVEvictCache.from_workload(w.with_(seed=78), device=cuda_device)  # same layout, another seed
    with pytest.raises(KVEvictError):
        b.restore(ck)
    c = KVEvictCache.from_workload(w.with_(budget=64, n_heavy=52), device=cuda_device)
    with pytest.raises(ValueError):  # another state size
        c.restore(ck)
    for x in (a, b, c):
        x.close()
