"""GPU parity of the Q-seeded prefill (H2O): the tcgen05 prompt-scoring passes
and the cut, through the C ABI, against the CPU oracle.

Tolerances: prompt scores within 2e-3 of the oracle's, relative to the unit's
largest score (bf16 inputs are identical on both sides; the GPU accumulates
the dot products and the column sums in fp32). The cut is checked bit-exact
on the GPU's own fp32 scores (the same rule evaluated on the host), and
against the oracle's cut up to near-ties (tokens whose oracle scores differ
by less than the score tolerance may trade places). Decode outputs after the
prefill: 2e-2 relative, as for every bf16 decode.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_decode_gb300 import BF16, H2O, SINK_WINDOW, KVEvictCache, KVEvictError, lib
from kv_cache_eviction_decode_gb300._lib import ERR_INVALID_ARG
from workloads import configs, synth

pytestmark = pytest.mark.gpu

SCORE_TOL = 2e-3
OUT_TOL = 2e-2


def _cache(device, B, Hq, Hkv, d, n_sink, n_heavy, n_recent, L=1):
    return KVEvictCache(policy=H2O, budget=n_sink + n_heavy + n_recent, n_sink=n_sink, n_heavy=n_heavy,
                        n_recent=n_recent, batch=B, n_layers=L, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d,
                        dtype=BF16, device=device)


def _rand(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def host_cut(s: np.ndarray, budget: int, n_sink: int, n_recent: int) -> np.ndarray:
    """Kept positions, ascending, for fp32 scores s: the P - budget smallest
    (bit pattern, position) among n_sink <= j < P - n_recent leave."""
    P = s.shape[0]
    if P <= budget:
        return np.arange(P)
    bits = s.astype(np.float32).view(np.uint32).astype(np.int64)
    elig = np.arange(n_sink, P - n_recent)
    order = elig[np.lexsort((elig, bits[elig]))]
    gone = np.zeros(P, dtype=bool)
    gone[order[:P - budget]] = True
    return np.nonzero(~gone)[0]


def _near_tie_equal(kept_gpu, kept_orc, s_orc, tol):
    a, b = set(kept_gpu.tolist()), set(kept_orc.tolist())
    only_g, only_o = sorted(a - b, key=lambda j: s_orc[j]), sorted(b - a, key=lambda j: s_orc[j])
    if len(only_g) != len(only_o):
        return False
    top = max(float(s_orc.max()), 1e-6)
    return all(abs(s_orc[x] - s_orc[y]) <= tol * top for x, y in zip(only_g, only_o))


def _check_units(cache, Q, K, V, scores, units, n_sink, n_heavy, n_recent, decode=True, gen=None):
    """Scores, the cut and one decode step of the sampled units against the oracle."""
    B, Hkv, P = scores.shape
    Hq, d = Q.shape[1], Q.shape[3]
    G = Hq // Hkv
    budget = n_sink + n_heavy + n_recent
    sc = scores.float().cpu().numpy()
    pos = cache.slot_positions(0).cpu().numpy()
    csc = cache.scores(0).cpu().numpy()
    kept_n = min(P, budget)
    # the cut, bit-exact on the GPU's own scores, for every unit
    for b in range(B):
        for h in range(Hkv):
            kept = host_cut(sc[b, h], budget, n_sink, n_recent)
            np.testing.assert_array_equal(pos[b, h, :kept_n], kept)
            assert np.all(pos[b, h, kept_n:] == -1)
            np.testing.assert_array_equal(csc[b, h, :kept_n].view(np.uint32), sc[b, h, kept].view(np.uint32))
    # scores and cut against the oracle, and one decode step
    if decode:
        qn = _rand((B, Hq, d), gen)
        kn = _rand((B, Hkv, d), gen)
        vn = _rand((B, Hkv, d), gen)
        out = cache.decode_step(0, qn.to(cache.device), kn.to(cache.device), vn.to(cache.device)).float().cpu().numpy()
    worst = 0.0
    for b, h in units:
        u = oracle.Unit(oracle.H2O, n_sink, n_heavy, n_recent, budget, 0, 0, G, d)
        s_orc = u.prefill_scored(Q[b, h * G:(h + 1) * G].float().numpy(), K[b, h].float().numpy(),
                                 V[b, h].float().numpy())
        err = np.abs(sc[b, h] - s_orc).max() / max(np.abs(s_orc).max(), 1e-6)
        worst = max(worst, err)
        assert err <= SCORE_TOL, (b, h, err)
        kept_orc = u.positions()[:kept_n]
        same = np.array_equal(pos[b, h, :kept_n], kept_orc)
        assert same or _near_tie_equal(pos[b, h, :kept_n], kept_orc, s_orc, 2 * SCORE_TOL), (b, h)
        if decode and same:
            o_orc, _ = u.step(qn[b, h * G:(h + 1) * G].float().numpy(), kn[b, h].float().numpy(),
                              vn[b, h].float().numpy())
            o_gpu = out[b, h * G:(h + 1) * G]
            rel = np.abs(o_gpu - o_orc).max() / max(np.abs(o_orc).max(), 1e-6)
            assert rel <= OUT_TOL, (b, h, rel)
    return worst


@pytest.mark.parametrize("G,d,P", [(1, 64, 77), (1, 128, 300), (4, 64, 700), (4, 128, 257), (8, 128, 520),
                                   (2, 128, 128), (1, 64, 50)])
def test_prefill_scored_small(cuda_device, G, d, P):
    gen = torch.Generator().manual_seed(1000 * G + P + d)
    B, Hkv = 2, 2
    Hq = G * Hkv
    n_sink, n_heavy, n_recent = 4, 36, 24  # budget 64: every prompt here is cut except within-budget ones
    Q, K, V = _rand((B, Hq, P, d), gen), _rand((B, Hkv, P, d), gen), _rand((B, Hkv, P, d), gen)
    cache = _cache(cuda_device, B, Hq, Hkv, d, n_sink, n_heavy, n_recent)
    scores = cache.prefill_scored(0, Q.to(cuda_device), K.to(cuda_device), V.to(cuda_device))
    assert cache.check() == 0
    assert cache.layer_state(0) == (P, 0, min(P, 64))
    units = [(b, h) for b in range(B) for h in range(Hkv)]
    worst = _check_units(cache, Q, K, V, scores, units, n_sink, n_heavy, n_recent, gen=gen)
    print(f"G={G} d={d} P={P}: max score err {worst:.2e}")


def test_prefill_scored_within_budget(cuda_device):
    gen = torch.Generator().manual_seed(5)
    B, Hq, Hkv, d, P = 1, 4, 2, 128, 100
    Q, K, V = _rand((B, Hq, P, d), gen), _rand((B, Hkv, P, d), gen), _rand((B, Hkv, P, d), gen)
    cache = _cache(cuda_device, B, Hq, Hkv, d, 4, 200, 16)
    scores = cache.prefill_scored(0, Q.to(cuda_device), K.to(cuda_device), V.to(cuda_device))
    assert cache.check() == 0
    pos = cache.slot_positions(0).cpu().numpy()
    assert np.all(pos[:, :, :P] == np.arange(P)) and np.all(pos[:, :, P:] == -1)
    # every query row's probabilities sum to 1: the scores of a unit sum to P
    np.testing.assert_allclose(scores.float().sum(-1).cpu().numpy(), P, rtol=1e-4)
    _check_units(cache, Q, K, V, scores, [(0, 0), (0, 1)], 4, 200, 16, gen=gen)


def test_prefill_scored_exact_tie(cuda_device):
    """Two keys that point against every query get probability exactly 0 in
    every row (fp32 exp2 underflows, as the oracle's fp64 exp does): their
    scores tie at 0.0 and the cut of one token removes the older."""
    gen = torch.Generator().manual_seed(17)
    B, Hq, Hkv, d, P = 1, 1, 1, 64, 200
    qd = torch.randn(d, generator=gen)
    qd /= qd.norm()
    Q = (qd * 4.0).expand(B, Hq, P, d).contiguous().to(torch.bfloat16)
    K = _rand((B, Hkv, P, d), gen, 0.1)
    K[0, 0, 50] = K[0, 0, 90] = (-1e4 * qd).to(torch.bfloat16)
    V = _rand((B, Hkv, P, d), gen)
    n_sink, n_recent = 4, 64
    n_heavy = P - 1 - n_sink - n_recent  # exactly one token leaves
    cache = _cache(cuda_device, B, Hq, Hkv, d, n_sink, n_heavy, n_recent)
    scores = cache.prefill_scored(0, Q.to(cuda_device), K.to(cuda_device), V.to(cuda_device)).cpu().numpy()
    assert scores[0, 0, 50] == 0.0 and scores[0, 0, 90] == 0.0
    assert np.all(np.delete(scores[0, 0], [50, 90]) > 0)
    pos = cache.slot_positions(0).cpu().numpy()[0, 0, :P - 1]
    np.testing.assert_array_equal(pos, np.delete(np.arange(P), 50))
    _check_units(cache, Q, K, V, torch.from_numpy(scores), [(0, 0)], n_sink, n_heavy, n_recent, gen=gen)


def test_prefill_scored_errors(cuda_device):
    gen = torch.Generator().manual_seed(3)
    B, Hq, Hkv, d, P = 1, 2, 2, 64, 64
    Q, K, V = (_rand((B, Hq, P, d), gen).to(cuda_device), _rand((B, Hkv, P, d), gen).to(cuda_device),
               _rand((B, Hkv, P, d), gen).to(cuda_device))
    cache = _cache(cuda_device, B, Hq, Hkv, d, 2, 20, 10, L=2)
    need = cache.prefill_scored_workspace_bytes(P)
    short = torch.empty(need - 256, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(ValueError):  # the binding checks the workspace size
        cache.prefill_scored(0, Q, K, V, workspace=short)
    # and so does the C ABI
    rc = lib().kvevict_prefill_scored(cache.h, 0, Q.data_ptr(), K.data_ptr(), V.data_ptr(), P, short.data_ptr(),
                                      short.numel())
    assert rc == ERR_INVALID_ARG
    cache.prefill(1, K, V)
    with pytest.raises(KVEvictError):  # layer not empty
        cache.prefill_scored(1, Q, K, V)
    cache.prefill_scored(0, Q, K, V)
    with pytest.raises(KVEvictError):  # twice
        cache.prefill_scored(0, Q, K, V)
    with pytest.raises(KVEvictError):  # prompt longer than the selection supports
        cache.prefill_scored_workspace_bytes(49153)
    sw = KVEvictCache(policy=SINK_WINDOW, budget=32, n_sink=2, n_recent=30, batch=B, n_layers=1, n_q_heads=Hq,
                      n_kv_heads=Hkv, head_dim=d, dtype=BF16, device=cuda_device)
    with pytest.raises(KVEvictError):  # H2O only
        sw.prefill_scored(0, Q, K, V)
    assert cache.check() == 0


def _full_shape_case(cuda_device, w, P, sampled_full, tail_units, tail_len):
    """The whole prompt of one layer at full shape on the GPU: every unit's cut
    bit-exact on its own scores and its score mass equal to P; the oracle's
    full scored prefill on `sampled_full` units, and its tail scores (keys
    j >= P - tail_len) on `tail_units`."""
    Q = synth.device_prompt_queries(w, 0, cuda_device, P)
    K, V = synth.device_prompt(w, 0, cuda_device, P)
    cache = KVEvictCache.from_workload(w.with_(n_layers=1), device=cuda_device)
    scores = cache.prefill_scored(0, Q, K, V)
    assert cache.check() == 0
    np.testing.assert_allclose(scores.float().sum(-1).cpu().numpy(), P, rtol=2e-4)
    sc = scores.float().cpu().numpy()
    pos = cache.slot_positions(0).cpu().numpy()
    kept_n = min(P, w.budget)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            np.testing.assert_array_equal(pos[b, h, :kept_n], host_cut(sc[b, h], w.budget, w.n_sink, w.n_recent))
    G = w.group
    for b, h in tail_units:
        qh = Q[b, h * G:(h + 1) * G].float().cpu().numpy()
        kh = K[b, h].float().cpu().numpy()
        t = oracle.prompt_tail_scores(qh, kh, P - tail_len)
        err = np.abs(sc[b, h, P - tail_len:] - t).max() / max(np.abs(t).max(), 1e-6)
        assert err <= SCORE_TOL, (b, h, err)
    if sampled_full:
        Qh, Kh, Vh = Q.cpu(), K.cpu(), V.cpu()
        _check_units(cache, Qh, Kh, Vh, scores.cpu(), sampled_full, w.n_sink, w.n_heavy, w.n_recent,
                     decode=False)
    cache.close()


def test_prefill_scored_full_h2o_mha(cuda_device):
    """H2O 4+510+510, B=16, 32 heads, d=128, prompt 2048: the oracle's whole
    scored prefill on four sampled units."""
    w = configs.H2O_MHA
    _full_shape_case(cuda_device, w, w.prompt_len, [(0, 0), (15, 31), (7, 13), (3, 30)], [(9, 5)], 48)


def test_prefill_scored_full_h2o_gqa(cuda_device):
    """H2O GQA, B=64, 64 query / 8 KV heads, prompt 32768: every unit's cut and
    mass; the oracle's tail scores (last 24 keys, each from its full rows) on
    three sampled units."""
    w = configs.H2O_GQA
    _full_shape_case(cuda_device, w, w.prompt_len, [], [(0, 0), (63, 7), (31, 4)], 24)
