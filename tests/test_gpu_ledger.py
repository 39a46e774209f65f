"""The evicted-mass ledger on the GPU ("KV Cache 驱逐策略：从 LRU 到 H2O" names
the evicted mass among the quantities to watch).

Every decode step hands each unit a mass of one: the mean over its G query
heads of a softmax over the retained tokens and the new token. With exact
cumulative scores (fp32 storage, no moving average) nothing else changes the
total, so after t steps, for every unit,

    sum of the retained scores + evicted mass = mass after the prompt + t,

where the prompt brings zero (scores start at 0) or, after a Q-seeded
prefill, the kept tokens' scores. Checked on every unit of the launch, for
H2O (MHA and GQA shapes), block-granular H2O and two-pool H2O, and after a
Q-seeded prefill; the scores are fp32 sums, so the balance holds to about
1e-6 relative per step. The lockstep tests also compare each checked unit's
ledger with the oracle's evicted mass.
"""
import numpy as np
import pytest
import torch

from kv_cache_eviction_decode_gb300 import KVEvictCache
from workloads import configs, synth

pytestmark = pytest.mark.gpu

REL = 2e-5


def _steps(cache, w, layer, T, device, seed=3):
    g = torch.Generator(device=device).manual_seed(seed)
    dt = torch.bfloat16 if w.dtype == configs.DTYPE_BF16 else torch.float32
    for _ in range(T):
        q = torch.randn((w.batch, w.n_q_heads, w.head_dim), generator=g, device=device).to(dt)
        k = torch.randn((w.batch, w.n_kv_heads, w.head_dim), generator=g, device=device).to(dt)
        v = torch.randn((w.batch, w.n_kv_heads, w.head_dim), generator=g, device=device).to(dt)
        cache.decode_step(layer, q, k, v)
    assert cache.check() == 0


def _balance(cache, layer):
    """Per unit: retained scores + evicted mass (fp64 on the host)."""
    pos = cache.slot_positions(layer).cpu().numpy()
    sc = cache.scores(layer).cpu().numpy().astype(np.float64)
    held = np.where(pos >= 0, sc, 0.0).sum(axis=2)
    return held + cache.evicted_mass(layer).cpu().numpy(), held


@pytest.mark.parametrize("w,T", [
    (configs.H2O_TINY, 256),
    (configs.H2O_MHA.with_(n_layers=1), 160),
    (configs.H2O_GQA.with_(prompt_len=4096), 96),
    (configs.H2O_BLOCK16.with_(n_layers=1), 96),
    (configs.H2O_POOLS_MHA.with_(n_layers=1, hh_threshold=2.0 ** -10), 128),
], ids=["tiny", "mha", "gqa", "block16", "pools"])
def test_retained_plus_evicted_equals_steps(cuda_device, w, T, record_property):
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    K, V = synth.device_prompt(w, 0, cuda_device, w.prompt_len)
    cache.prefill(0, K, V)
    del K, V
    _steps(cache, w, 0, T, cuda_device)
    total, held = _balance(cache, 0)
    err = np.abs(total - T) / T
    record_property("max_rel_balance_error", float(err.max()))
    assert err.max() <= REL, f"worst unit: retained + evicted = {total.flat[np.argmax(err)]:.9g}, steps {T}"
    led = cache.evicted_mass(0).cpu().numpy()
    if w.policy != configs.POLICY_H2O_POOLS or T > w.capacity:
        assert np.all(led > 0)  # something left every unit
    st = cache.stats()
    assert st["evicted_mass"] == pytest.approx(float(led.sum()), rel=1e-12)
    cache.close()


def test_ledger_after_scored_prefill(cuda_device):
    """After a Q-seeded prefill the balance starts from the kept tokens'
    scores (the tokens the prompt's own cut dropped are not in the ledger)."""
    w = configs.H2O_MHA.with_(n_layers=1, batch=4)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    Q = synth.device_prompt_queries(w, 0, cuda_device, w.prompt_len)
    K, V = synth.device_prompt(w, 0, cuda_device, w.prompt_len)
    cache.prefill_scored(0, Q, K, V)
    start, _ = _balance(cache, 0)
    assert np.all(cache.evicted_mass(0).cpu().numpy() == 0.0)
    T = 64
    _steps(cache, w, 0, T, cuda_device)
    total, _ = _balance(cache, 0)
    err = np.abs(total - (start + T)) / (start + T)
    assert err.max() <= REL
    cache.close()


def test_ledger_rejected_without_scores(cuda_device):
    from kv_cache_eviction_decode_gb300 import KVEvictError
    w = configs.SINK_WINDOW.with_(n_layers=1, batch=1)
    cache = KVEvictCache.from_workload(w, device=cuda_device)
    with pytest.raises(KVEvictError):
        cache.evicted_mass(0)
    assert cache.stats()["evicted_mass"] == 0.0
    cache.close()
