"""Pins of the oracle's Q-seeded prefill (H2O) to things other than itself.

The prompt scores are the column sums of the prompt's causal attention,
averaged over the G query heads of the KV head; the budget is then enforced
by the greedy rule of Algorithm 1 ("h2o: heavy-hitter oracle" summary). The
pins: torch's fp64 scaled-dot-product attention with V = I (its output is
the attention matrix itself), the closed form for identical keys (harmonic
numbers), the mass invariant (every query row sums to 1), brute force over
retained sets on tiny prompts, and continuity with the decode step (a scored
prefill followed by decode steps that never evict equals the column sums of
the whole sequence's causal attention).
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import ESTATE, H2O, SINK_WINDOW, Unit


def _inputs(rng, G, P, d, scale=1.0):
    q = (rng.standard_normal((G, P, d)) * scale).astype(np.float32)
    k = (rng.standard_normal((P, d)) * scale).astype(np.float32)
    v = rng.standard_normal((P, d)).astype(np.float32)
    return q, k, v


def _sdpa_column_sums(q, k):
    """Column sums of softmax(q k^T / sqrt(d)) under the causal mask, per head,
    from torch's fp64 SDPA with V = I_P."""
    import torch
    import torch.nn.functional as F
    G, P, d = q.shape
    qt = torch.from_numpy(q.astype(np.float64))[None]
    kt = torch.from_numpy(k.astype(np.float64))[None, None].expand(1, G, P, d)
    eye = torch.eye(P, dtype=torch.float64)[None, None].expand(1, G, P, P)
    A = F.scaled_dot_product_attention(qt, kt, eye, is_causal=True)[0].numpy()  # [G][i][j]
    return A.sum(axis=1)  # [G][j]


@pytest.mark.parametrize("G,P,d", [(1, 23, 16), (4, 37, 8), (8, 64, 32)])
def test_scores_equal_sdpa_column_sums(G, P, d):
    rng = np.random.default_rng(1000 + G * P)
    q, k, v = _inputs(rng, G, P, d)
    u = Unit(H2O, 2, P, 3, P + 5, 0, 0, G, d)  # budget above P: nothing is cut
    s = u.prefill_scored(q, k, v)
    ref = _sdpa_column_sums(q, k).mean(axis=0)
    np.testing.assert_allclose(s, ref, rtol=0, atol=1e-12)
    # nothing cut: every prompt token in slot == position, with its score
    assert u.count == P
    np.testing.assert_array_equal(u.positions()[:P], np.arange(P))
    np.testing.assert_array_equal(u.scores()[:P], s)


def test_identical_keys_harmonic_closed_form():
    rng = np.random.default_rng(5)
    G, P, d = 3, 50, 8
    c = rng.standard_normal(d).astype(np.float32)
    q = rng.standard_normal((G, P, d)).astype(np.float32)
    k = np.tile(c, (P, 1))
    v = rng.standard_normal((P, d)).astype(np.float32)
    u = Unit(H2O, 1, P, 1, P + 2, 0, 0, G, d)
    s = u.prefill_scored(q, k, v)
    # query i attends i + 1 identical keys: p = 1 / (i + 1) for every j <= i,
    # so score_j = sum_{i=j}^{P-1} 1/(i+1) = H_P - H_j
    H = [Fraction(0)]
    for i in range(1, P + 1):
        H.append(H[-1] + Fraction(1, i))
    for j in range(P):
        assert s[j] == pytest.approx(float(H[P] - H[j]), rel=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_cut_layout_and_mass(seed):
    rng = np.random.default_rng(200 + seed)
    G, P, d = 2, 90, 16
    n_sink, n_heavy, n_recent = 4, 20, 10
    K = n_sink + n_heavy + n_recent
    q, k, v = _inputs(rng, G, P, d, scale=1.5)
    u = Unit(H2O, n_sink, n_heavy, n_recent, K, 0, 0, G, d)
    s = u.prefill_scored(q, k, v)
    assert math.fsum(s) == pytest.approx(P, rel=1e-13)
    assert u.count == K
    pos = u.positions()[:K]
    assert np.all(np.diff(pos) > 0)  # ascending position order in slots 0..K-1
    # sinks and the recent window stay; the heavy hitters are the n_heavy
    # largest (score, position) among the rest
    mid = np.arange(n_sink, P - n_recent)
    order = sorted(mid.tolist(), key=lambda j: (s[j], j), reverse=True)
    expect = set(range(n_sink)) | set(range(P - n_recent, P)) | set(order[:n_heavy])
    assert set(pos.tolist()) == expect
    np.testing.assert_array_equal(u.scores()[:K], s[pos])
    for slot in (0, K // 2, K - 1):
        kk, vv = u.slot_kv(slot)
        np.testing.assert_array_equal(kk, k[pos[slot]])
        np.testing.assert_array_equal(vv, v[pos[slot]])
    evicted = sorted(set(range(P)) - expect)
    assert u.evicted_mass == pytest.approx(math.fsum(s[evicted]), rel=1e-12)
    assert u.greedy_disagreements == 0


@pytest.mark.parametrize("seed", range(5))
def test_cut_equals_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    G, P, d = 2, 11, 4
    n_sink, n_heavy, n_recent = 1, 3, 2
    K = n_sink + n_heavy + n_recent
    q, k, v = _inputs(rng, G, P, d, scale=2.0)
    u = Unit(H2O, n_sink, n_heavy, n_recent, K, 0, 0, G, d)
    s = u.prefill_scored(q, k, v)
    protected = set(range(n_sink)) | set(range(P - n_recent, P))
    best, best_sets = -1.0, []
    for keep in itertools.combinations(range(P), K):
        if not protected <= set(keep):
            continue
        f = math.fsum(s[j] for j in keep)
        if f > best + 1e-15:
            best, best_sets = f, [set(keep)]
        elif abs(f - best) <= 1e-15:
            best_sets.append(set(keep))
    assert len(best_sets) == 1
    assert set(u.positions()[:K].tolist()) == best_sets[0]


def test_scored_prefill_then_decode_equals_whole_sequence_column_sums():
    rng = np.random.default_rng(9)
    G, P, T, d = 2, 30, 20, 16
    n = P + T
    qa = rng.standard_normal((G, n, d)).astype(np.float32)
    ka = rng.standard_normal((n, d)).astype(np.float32)
    va = rng.standard_normal((n, d)).astype(np.float32)
    u = Unit(H2O, 2, n, 3, n + 5, 0, 0, G, d)  # never evicts
    u.prefill_scored(qa[:, :P], ka[:P], va[:P])
    for t in range(T):
        u.step(qa[:, P + t], ka[P + t], va[P + t])
    ref = _sdpa_column_sums(qa, ka).mean(axis=0)
    pos, sc = u.positions(), u.scores()
    assert u.count == n
    for slot in range(n):
        assert sc[slot] == pytest.approx(ref[pos[slot]], abs=1e-12)


def test_scored_prefill_preconditions():
    rng = np.random.default_rng(2)
    G, P, d = 1, 8, 4
    q, k, v = _inputs(rng, G, P, d)
    u = Unit(H2O, 1, 4, 2, 7, 0, 0, G, d)
    u.prefill(k[:2], v[:2])
    with pytest.raises(RuntimeError, match=str(ESTATE)):
        u.prefill_scored(q, k, v)  # only on an empty unit
    w = Unit(SINK_WINDOW, 1, 0, 6, 7, 0, 0, G, d)
    with pytest.raises(RuntimeError, match=str(ESTATE)):
        w.prefill_scored(q, k, v)  # H2O only


def test_exact_tie_evicts_the_older():
    """Two keys that point against every query get weight exp(-huge) == 0 from
    every row (the first key always has a finite logit), so both scores are
    exactly 0.0; a cut of one token must remove the older of the two."""
    rng = np.random.default_rng(17)
    G, P, d = 1, 12, 8
    qd = rng.standard_normal(d)
    qd /= np.linalg.norm(qd)
    q = np.tile(qd * 4.0, (G, P, 1)).astype(np.float32)
    k = (rng.standard_normal((P, d)) * 0.1).astype(np.float32)
    k[4] = k[7] = (-1e4 * qd).astype(np.float32)
    v = rng.standard_normal((P, d)).astype(np.float32)
    n_sink, n_heavy, n_recent = 1, 8, 2  # K = 11: exactly one token goes
    u = Unit(H2O, n_sink, n_heavy, n_recent, 11, 0, 0, G, d)
    s = u.prefill_scored(q, k, v)
    assert s[4] == 0.0 and s[7] == 0.0 and np.all(np.delete(s, [4, 7]) > 0)
    kept = set(u.positions()[:11].tolist())
    assert kept == set(range(P)) - {4}


@pytest.mark.parametrize("j0", [0, 1, 57, 79])
def test_tail_scores_equal_sdpa_and_full(j0):
    import oracle
    rng = np.random.default_rng(40 + j0)
    G, P, d = 4, 80, 16
    q, k, v = _inputs(rng, G, P, d)
    tail = oracle.prompt_tail_scores(q, k, j0)
    ref = _sdpa_column_sums(q, k).mean(axis=0)[j0:]
    np.testing.assert_allclose(tail, ref, rtol=0, atol=1e-12)
    u = Unit(H2O, 2, P, 3, P + 5, 0, 0, G, d)
    full = u.prefill_scored(q, k, v)
    np.testing.assert_allclose(tail, full[j0:], rtol=0, atol=1e-13)
