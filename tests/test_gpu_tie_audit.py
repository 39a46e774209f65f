"""The near-tie count of the validation mode (kvevict_set_tie_audit) on the GPU.

A decision is a near-tie when the runner-up candidate's stored score lies
within 1e-5 relative of the evicted token's (|a - b| < 1e-5 max(a, b), equal
scores included), the definition the parity harness applies between the
oracle's and the GPU's victims ("h2o: heavy-hitter oracle" summary, Algorithm 1:
the greedy removal of the lowest-score candidate). The count is checked
against the same rule applied on the host to the state the GPU left after
every step (slot positions, stored scores and the step's trace records), so
it must agree exactly: equal keys (every candidate ties), random keys (few
ties), binary16 and INT8 storage (coarser values, more ties), a cluster split
and a one-CTA-per-SM group size.
"""
import numpy as np
import pytest
import torch

from kv_cache_eviction_decode_gb300 import BF16, F32, H2O, SINK_WINDOW, KVEvictCache, KVEvictError

pytestmark = pytest.mark.gpu

REL = np.float32(1e-5)


def _host_count(pos_snaps, score_snaps, trace, P, n_sink, n_recent):
    """The rule on the host, in fp32 like the device: per step and unit that
    evicted, the smallest score among the candidates left."""
    T, B, H, _ = trace.shape
    n = 0
    for t in range(T):
        p = P + t
        pos, sc = pos_snaps[t], score_snaps[t]
        for b in range(B):
            for h in range(H):
                dest, old_pos = int(trace[t, b, h, 0]), int(trace[t, b, h, 1])
                if old_pos < 0:
                    continue
                s1 = trace[t, b, h, 2:3].view(np.float32)[0]
                ps = pos[b, h]
                cand = (ps >= n_sink) & (ps <= p - n_recent)
                cand[dest] = False
                if not cand.any():
                    continue
                mn = np.float32(sc[b, h][cand].min())
                if mn == s1 or np.float32(abs(mn - s1)) < REL * np.float32(max(mn, s1)):
                    n += 1
    return n


@pytest.mark.parametrize("keys,dtype,G,split,storage", [
    ("equal", F32, 2, 1, "fp32"),
    ("random", F32, 2, 1, "fp32"),
    ("random", BF16, 2, 2, "fp32"),       # a cluster of two per unit
    ("equal", BF16, 4, 1, "fp32"),        # one CTA per SM
    ("random", BF16, 1, 1, "half"),
    ("random", BF16, 1, 1, "int8"),
])
def test_near_tie_count_matches_host_rule(cuda_device, keys, dtype, G, split, storage):
    B, Hkv, d, T = 3, 4, 64 if dtype == F32 else 128, 60
    n_sink, n_heavy, n_recent = 4, 40, 20
    C = n_sink + n_heavy + n_recent
    P = C + 10  # the cache is full after the prompt: every step evicts
    cache = KVEvictCache(policy=H2O, budget=C, n_sink=n_sink, n_heavy=n_heavy, n_recent=n_recent, batch=B, n_layers=1,
                         n_q_heads=G * Hkv, n_kv_heads=Hkv, head_dim=d, dtype=dtype, score_half=storage == "half",
                         score_int8=storage == "int8", device=cuda_device)
    if split > 1:
        cache.set_split(split)
    dt = torch.float32 if dtype == F32 else torch.bfloat16
    g = torch.Generator(device=cuda_device).manual_seed(515)
    if keys == "equal":  # every key and value the same: equal probabilities, exact ties
        K = torch.ones((B, Hkv, P, d), device=cuda_device, dtype=dt)
    else:
        K = torch.randn((B, Hkv, P, d), generator=g, device=cuda_device).to(dt)
    V = torch.randn((B, Hkv, P, d), generator=g, device=cuda_device).to(dt)
    cache.prefill(0, K, V)
    trace = torch.full((T, B, Hkv, 4), -7, dtype=torch.int32, device=cuda_device)
    cache.set_trace(0, trace)
    cache.set_tie_audit(True)
    pos_snaps, score_snaps = [], []
    for t in range(T):
        q = torch.randn((B, G * Hkv, d), generator=g, device=cuda_device).to(dt)
        if keys == "equal":
            k = torch.ones((B, Hkv, d), device=cuda_device, dtype=dt)
        else:
            k = torch.randn((B, Hkv, d), generator=g, device=cuda_device).to(dt)
        v = torch.randn((B, Hkv, d), generator=g, device=cuda_device).to(dt)
        cache.decode_step(0, q, k, v)
        pos_snaps.append(cache.slot_positions(0).cpu().numpy())
        score_snaps.append(cache.scores(0).cpu().numpy().astype(np.float32))
    assert cache.check() == 0
    expect = _host_count(pos_snaps, score_snaps, trace.cpu().numpy(), P, n_sink, n_recent)
    got = cache.near_ties(0)
    st = cache.stats()
    print(f"{keys} {storage} G={G} split={split}: near-ties {got} of {T * B * Hkv} decisions")
    assert got == expect and st["near_ties"] == got
    if keys == "equal":
        assert got > 0
    cache.close()


def test_near_tie_count_off_and_on(cuda_device):
    """Off by default: nothing is counted; switched on, only the later steps
    count, without a trace set (the handle's own record buffer)."""
    B, Hkv, d, C = 2, 2, 64, 40
    cache = KVEvictCache(policy=H2O, budget=C, n_sink=2, n_heavy=20, n_recent=18, batch=B, n_layers=2, n_q_heads=Hkv,
                         n_kv_heads=Hkv, head_dim=d, dtype=F32, device=cuda_device)
    K = torch.ones((B, Hkv, C + 5, d), device=cuda_device)
    for layer in range(2):
        cache.prefill(layer, K, K)
    one = torch.ones((B, Hkv, d), device=cuda_device)
    for _ in range(5):
        cache.decode_step(0, one, one, one)
    assert cache.near_ties(0) == 0 and cache.stats()["near_ties"] == 0
    cache.set_tie_audit(True)
    for _ in range(5):
        cache.decode_step(0, one, one, one)
        cache.decode_step(1, one, one, one)
    assert cache.check() == 0
    n0, n1 = cache.near_ties(0), cache.near_ties(1)
    # equal keys and values: every candidate ties with the evicted one at every step
    assert n0 == 5 * B * Hkv and n1 == 5 * B * Hkv
    assert cache.stats()["near_ties"] == n0 + n1
    cache.set_tie_audit(False)
    cache.decode_step(0, one, one, one)
    assert cache.near_ties(0) == n0
    cache.close()


def test_tie_audit_refused_without_h2o(cuda_device):
    """The count is defined for the H2O decision only."""
    cache = KVEvictCache(policy=SINK_WINDOW, budget=64, n_sink=4, n_recent=60, batch=1, n_layers=1, n_q_heads=2,
                         n_kv_heads=2, head_dim=64, dtype=F32, device=cuda_device)
    with pytest.raises(KVEvictError):
        cache.set_tie_audit(True)
    cache.set_tie_audit(False)
    assert cache.stats()["near_ties"] == 0
    cache.close()
