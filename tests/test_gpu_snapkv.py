"""GPU parity of the SnapKV prefill ("Attention Sinks 与 KV Cache 淘汰策略" section
4.3) and of the decode steps that follow it, through the C ABI, against the
CPU oracle.

Votes within 2e-3 of the oracle's, relative to the unit's largest vote. The
selection (pooling, per-head top-k, union, window) is checked bit-exact on the
GPU's own fp32 votes, and against the oracle's selection up to near-ties. The
decode steps after the prefill fill each unit's empty slots, lowest first,
then evict by score: checked in lockstep with the oracle (outputs 2e-2
relative; a different victim only as a near-tie, which the oracle adopts).
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_decode_gb300 import BF16, H2O, KVEvictCache
from workloads import configs, synth

pytestmark = pytest.mark.gpu

VOTE_TOL = 2e-3
OUT_TOL = 2e-2
NEAR_TIE_REL = 1e-5


def _rand(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def host_select(votes: np.ndarray, P: int, w: int, k: int) -> np.ndarray:
    """Kept positions for one unit from fp32 votes [G][P], with the GPU's rule."""
    n_pre = P - w
    kept = set(range(n_pre, P))
    pos = np.arange(n_pre)
    for g in range(votes.shape[0]):
        v = votes[g, :n_pre].astype(np.float32)
        pad = np.concatenate([np.full(3, -np.inf, np.float32), v, np.full(3, -np.inf, np.float32)])
        pooled = np.max(np.stack([pad[o:o + n_pre] for o in range(7)]), axis=0)
        bits = pooled.view(np.uint32).astype(np.int64)
        order = np.lexsort((-pos, -bits))  # largest bit pattern first, then the newer position
        kept |= set(order[:min(k, n_pre)].tolist())
    return np.array(sorted(kept))


def _mean_votes(votes: np.ndarray, cols) -> np.ndarray:
    acc = np.zeros(len(cols), np.float32)
    for g in range(votes.shape[0]):
        acc = (acc + votes[g, cols].astype(np.float32)).astype(np.float32)
    return (acc * np.float32(1.0 / votes.shape[0])).astype(np.float32)


def _near_tie_equal(kept_gpu, kept_orc, votes_orc, P, w, tol):
    a, b = set(kept_gpu.tolist()), set(kept_orc.tolist())
    if a == b:
        return True
    n_pre = P - w
    pooled = np.stack([[votes_orc[g, max(0, j - 3):min(n_pre, j + 4)].max() for j in range(n_pre)]
                       for g in range(votes_orc.shape[0])]).max(axis=0)
    only_g, only_o = sorted(a - b, key=lambda j: pooled[j]), sorted(b - a, key=lambda j: pooled[j])
    if len(only_g) != len(only_o):
        return False
    top = max(float(pooled.max()), 1e-6)
    return all(abs(pooled[x] - pooled[y]) <= tol * top for x, y in zip(only_g, only_o))


def _check_prefill(cache, Qo, K, V, votes_t, k, units):
    B, Hq, w, d = Qo.shape
    Hkv, P = K.shape[1], K.shape[2]
    G = Hq // Hkv
    votes = votes_t.cpu().numpy()
    pos = cache.slot_positions(0).cpu().numpy()
    csc = cache.scores(0).cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            vg = votes[b, h * G:(h + 1) * G]
            kept = host_select(vg, P, w, k)
            n = len(kept)
            np.testing.assert_array_equal(pos[b, h, :n], kept)
            assert np.all(pos[b, h, n:] == -1)
            np.testing.assert_array_equal(csc[b, h, :n], _mean_votes(vg, kept))
    oracle_units = {}
    for b, h in units:
        u = oracle.Unit(oracle.H2O, cache.cfg.n_sink, cache.cfg.n_heavy, cache.cfg.n_recent, cache.cfg.budget, 0, 0,
                        G, d)
        v_orc = u.prefill_snapkv(Qo[b, h * G:(h + 1) * G].float().cpu().numpy(), K[b, h].float().cpu().numpy(),
                                 V[b, h].float().cpu().numpy(), k)
        vg = votes[b, h * G:(h + 1) * G]
        err = np.abs(vg - v_orc).max() / max(np.abs(v_orc).max(), 1e-6)
        assert err <= VOTE_TOL, (b, h, err)
        kept_gpu = pos[b, h, :u.count] if u.count <= cache.capacity else None
        assert _near_tie_equal(pos[b, h][pos[b, h] >= 0], u.positions()[:u.count], v_orc, P, w, 2 * VOTE_TOL), (b, h)
        oracle_units[(b, h)] = (u, np.array_equal(kept_gpu, u.positions()[:u.count]))
    return oracle_units


def _cache(device, B, Hq, Hkv, d, n_sink, n_heavy, n_recent):
    return KVEvictCache(policy=H2O, budget=n_sink + n_heavy + n_recent, n_sink=n_sink, n_heavy=n_heavy,
                        n_recent=n_recent, batch=B, n_layers=1, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d,
                        dtype=BF16, device=device)


@pytest.mark.parametrize("G,d,P,w,k", [(1, 64, 90, 8, 10), (4, 128, 300, 32, 20), (8, 128, 700, 32, 12),
                                       (2, 64, 257, 16, 100), (4, 64, 140, 20, 0), (4, 128, 500, 64, 30),
                                       (8, 64, 333, 96, 10), (2, 64, 400, 32, 40), (1, 128, 333, 32, 50),
                                       # prefixes past 2048 and 8192 positions: 16 and 64 pooled votes per
                                       # thread (pooling across the warps' spans, a wide cut with ties)
                                       (2, 64, 5000, 32, 300), (1, 64, 32800, 32, 16000),
                                       # past 32768: the selection with the pooled votes in shared memory
                                       (1, 64, 33000, 32, 100)])
def test_snapkv_prefill_small(cuda_device, G, d, P, w, k):
    gen = torch.Generator().manual_seed(7000 + G * P + k)
    B, Hkv = 2, 2
    Hq = G * Hkv
    Qo, K, V = _rand((B, Hq, w, d), gen), _rand((B, Hkv, P, d), gen), _rand((B, Hkv, P, d), gen)
    cap = G * k + w + 8
    cache = _cache(cuda_device, B, Hq, Hkv, d, 4, cap - 4 - 2, 2)
    votes = cache.prefill_snapkv(0, Qo.to(cuda_device), K.to(cuda_device), V.to(cuda_device), k)
    assert cache.check() == 0
    np.testing.assert_allclose(votes.float().sum(-1).cpu().numpy(), w, rtol=1e-4)  # each window row sums to 1
    _check_prefill(cache, Qo, K, V, votes, k, [(b, h) for b in range(B) for h in range(Hkv)])


@pytest.mark.parametrize("G,P,k", [(4, 1000, 20), (8, 5000, 40), (2, 9000, 300)])
def test_snapkv_select_many_units(cuda_device, G, P, k):
    """More units than SMs (B=40, 4 KV heads: 160 units, a second wave of
    selection CTAs). Every unit's slot table equals the selection rule applied
    to the GPU's votes; sampled units against the oracle. Prefixes of 1000,
    5000 and 9000 positions take the 4, 16 and 64 votes-per-thread kernels."""
    gen = torch.Generator().manual_seed(8300 + G * P + k)
    B, Hkv, d, w = 40, 4, 128, 32
    Hq = G * Hkv
    Qo, K, V = _rand((B, Hq, w, d), gen), _rand((B, Hkv, P, d), gen), _rand((B, Hkv, P, d), gen)
    cap = G * k + w + 8
    cache = _cache(cuda_device, B, Hq, Hkv, d, 4, cap - 4 - 2, 2)
    votes = cache.prefill_snapkv(0, Qo.to(cuda_device), K.to(cuda_device), V.to(cuda_device), k)
    assert cache.check() == 0
    np.testing.assert_allclose(votes.float().sum(-1).cpu().numpy(), w, rtol=1e-4)
    _check_prefill(cache, Qo, K, V, votes, k, [(0, 0), (17, 2), (39, 3)])


@pytest.mark.parametrize("G,w", [(4, 32), (8, 32), (2, 64)])
def test_snapkv_votes_many_units(cuda_device, G, w):
    """More (unit, key tile) items than SMs: the streamed votes kernel's CTAs
    cross unit boundaries (the window rows reloaded); sampled units against
    the oracle, every window row's votes summing to 1."""
    gen = torch.Generator().manual_seed(8100 + G * w)
    B, Hkv, d, P, k = 16, 4, 128, 1000, 20
    Hq = G * Hkv
    Qo, K, V = _rand((B, Hq, w, d), gen), _rand((B, Hkv, P, d), gen), _rand((B, Hkv, P, d), gen)
    cap = G * k + w + 8
    cache = _cache(cuda_device, B, Hq, Hkv, d, 4, cap - 4 - 2, 2)
    votes = cache.prefill_snapkv(0, Qo.to(cuda_device), K.to(cuda_device), V.to(cuda_device), k)
    assert cache.check() == 0
    np.testing.assert_allclose(votes.float().sum(-1).cpu().numpy(), w, rtol=1e-4)
    _check_prefill(cache, Qo, K, V, votes, k, [(0, 0), (5, 1), (10, 2), (15, 3)])


def test_snapkv_then_decode_lockstep(cuda_device):
    """After the SnapKV prefill every unit holds between k + w and G k + w tokens;
    100 decode steps fill each unit's empty slots, lowest first, then evict."""
    gen = torch.Generator().manual_seed(4242)
    B, Hkv, G, d, P, w, k, T = 2, 2, 4, 128, 300, 32, 20, 100
    Hq = G * Hkv
    n_sink, n_heavy, n_recent = 4, 100, 24  # 128 slots >= G k + w = 112
    Qo, K, V = _rand((B, Hq, w, d), gen), _rand((B, Hkv, P, d), gen), _rand((B, Hkv, P, d), gen)
    cache = _cache(cuda_device, B, Hq, Hkv, d, n_sink, n_heavy, n_recent)
    votes = cache.prefill_snapkv(0, Qo.to(cuda_device), K.to(cuda_device), V.to(cuda_device), k)
    units = [(b, h) for b in range(B) for h in range(Hkv)]
    orc = _check_prefill(cache, Qo, K, V, votes, k, units)
    assert all(same for _, same in orc.values()), "the prefill selections differ from the oracle's"
    q, kn, vn = _rand((T, B, Hq, d), gen), _rand((T, B, Hkv, d), gen), _rand((T, B, Hkv, d), gen)
    trace = torch.full((T, B, Hkv, 4), -7, dtype=torch.int32, device=cuda_device)
    cache.set_trace(0, trace)
    outs = []
    for t in range(T):
        outs.append(cache.decode_step(0, q[t].to(cuda_device), kn[t].to(cuda_device), vn[t].to(cuda_device))
                    .float().cpu().numpy())
    assert cache.check() == 0
    tr = trace.cpu().numpy()
    fills = near = 0
    for (b, h), (u, _) in orc.items():
        for t in range(T):
            ref = u.attend(q[t, b, h * G:(h + 1) * G].float().numpy(), kn[t, b, h].float().numpy(),
                           vn[t, b, h].float().numpy())
            got = outs[t][b, h * G:(h + 1) * G]
            assert np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-6) <= OUT_TOL, (b, h, t)
            slot = u.choose()
            gslot, gold = int(tr[t, b, h, 0]), int(tr[t, b, h, 1])
            if gslot != slot:
                sc = u.scores()
                rel = abs(sc[slot] - sc[gslot]) / max(sc[slot], sc[gslot], 1e-300)
                assert u.pos_at(slot) >= 0 and rel < NEAR_TIE_REL, (b, h, t, slot, gslot)
                near += 1
                slot = gslot
            assert gold == u.pos_at(slot), (b, h, t)
            fills += gold == -1
            u.commit(slot)
        np.testing.assert_array_equal(cache.slot_positions(0).cpu().numpy()[b, h], u.positions())
    print(f"fills {fills}, near ties {near}")
    assert fills > 0


def _full_shape(cuda_device, w: configs.Workload, P, window, k, sampled, steps, full_after):
    Q = synth.device_prompt_queries(w, 0, cuda_device, P)[:, :, P - window:].contiguous()
    K, V = synth.device_prompt(w, 0, cuda_device, P)
    cache = KVEvictCache.from_workload(w.with_(n_layers=1), device=cuda_device)
    votes = cache.prefill_snapkv(0, Q, K, V, k)
    assert cache.check() == 0
    np.testing.assert_allclose(votes.float().sum(-1).cpu().numpy(), window, rtol=2e-4)
    _check_prefill(cache, Q, K, V, votes, k, sampled)
    gen = torch.Generator(device=cuda_device).manual_seed(5)
    for _ in range(steps):  # decode continues from the selection (fill, then evict)
        qn = torch.randn((w.batch, w.n_q_heads, w.head_dim), generator=gen, device=cuda_device).to(torch.bfloat16)
        kn = torch.randn((w.batch, w.n_kv_heads, w.head_dim), generator=gen, device=cuda_device).to(torch.bfloat16)
        vn = torch.randn((w.batch, w.n_kv_heads, w.head_dim), generator=gen, device=cuda_device).to(torch.bfloat16)
        cache.decode_step(0, qn, kn, vn)
    assert cache.check() == 0
    pos = cache.slot_positions(0).cpu().numpy()
    assert bool(np.all(pos >= 0)) == full_after
    cache.close()


def test_snapkv_full_h2o_gqa(cuda_device):
    """GQA, B=64, 64 query / 8 KV heads, prompt 32768, window 32, 252 per head
    (the union fits the 2048 slots); the oracle on two sampled units."""
    _full_shape(cuda_device, configs.H2O_GQA, 32768, 32, 252, [(0, 0), (63, 7)], 8, full_after=False)


def test_snapkv_full_h2o_mha(cuda_device):
    """MHA, B=16, 32 heads, prompt 2048, window 32, 992 per head: every unit is
    full after the prefill, so decode evicts at once."""
    _full_shape(cuda_device, configs.H2O_MHA, 2048, 32, 992, [(0, 0), (15, 31), (8, 3)], 4, full_after=True)
