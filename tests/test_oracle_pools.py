"""Pins of the oracle's two-pool H2O (the H2OCache class of "KV Cache 驱逐策略：
从 LRU 到 H2O", section "实现要点": a recent pool whose lowest-score member
leaves when it overflows, promoted to a heavy-hitter pool if its score is
above hh_threshold, the heavy-hitter pool dropping its own lowest member when
over capacity) to things other than itself:

  - the extreme thresholds reduce to subset problems solved by brute force:
    theta = -inf promotes every token, so the kept set is always the best
    budget-subset of (kept + new) by total score (the greedy of the
    "h2o: heavy-hitter oracle" summary, Algorithm 1, without a recent
    window); theta = +inf promotes none, so only n_recent tokens stay, the
    best n_recent-subset of (recent + new);
  - a restatement over Python lists and dicts (pools as lists in arrival
    order, scores keyed by position) driven by torch's fp64 SDPA weights of
    the kept tokens, compared slot-free: the kept positions, their pools,
    scores and K/V rows;
  - the prompt layout in closed form (every prompt score is 0);
  - invariants: pool sizes, promotions strictly above the threshold, the
    score mass conserved, occupancy contiguous and never shrinking.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import H2O, H2O_POOLS, Unit

G, D = 2, 8


def _sdpa_weights(q, keys):
    """Mean over the G query heads of softmax(q k / sqrt(d)) over `keys`
    (torch fp64 SDPA with V = I)."""
    import torch
    import torch.nn.functional as F
    n = keys.shape[0]
    qq = torch.from_numpy(q.astype(np.float64))[None, :, None, :]
    kk = torch.from_numpy(keys.astype(np.float64))[None, None].expand(1, q.shape[0], n, keys.shape[1])
    eye = torch.eye(n, dtype=torch.float64)[None, None].expand(1, q.shape[0], n, n)
    return F.scaled_dot_product_attention(qq, kk, eye)[0, :, 0, :].numpy().mean(axis=0)


def _state(u):
    """{position: (pool, score, slot)} of the kept tokens."""
    pos, pools, sc = u.positions(), u.pools(), u.scores()
    return {int(pos[s]): (int(pools[s]), float(sc[s]), s) for s in range(u.cap) if pos[s] >= 0}


def _inputs(rng, P, T, spread):
    K = rng.standard_normal((P + T, D)).astype(np.float32)
    V = rng.standard_normal((P + T, D)).astype(np.float32)
    Q = (rng.standard_normal((T, G, D)) * spread).astype(np.float32)
    return K, V, Q


class _ListModel:
    """The class's add step over lists; scores keyed by position."""

    def __init__(self, n_recent, n_heavy, theta):
        self.R, self.H, self.theta = n_recent, n_heavy, theta
        self.recent, self.hh, self.score = [], [], {}

    def add(self, p, weight):
        for q in self.recent + self.hh:
            self.score[q] += weight[q]
        self.score[p] = weight[p]
        self.recent.append(p)
        if len(self.recent) <= self.R:
            return
        v = min(self.recent, key=lambda q: (self.score[q], q))
        self.recent.remove(v)
        if self.score[v] > self.theta:
            self.hh.append(v)
            if len(self.hh) > self.H:
                self.hh.remove(min(self.hh, key=lambda q: (self.score[q], q)))

    def kept(self):
        return sorted(self.recent + self.hh)


@pytest.mark.parametrize("seed,n_recent,n_heavy,theta,spread,P", [
    (0, 3, 4, 0.08, 1.0, 5), (1, 4, 2, 0.2, 2.5, 0), (2, 2, 5, 0.0, 1.5, 9), (3, 5, 0, 0.1, 1.0, 3),
    (4, 1, 3, 0.3, 3.0, 6), (5, 6, 6, -1.0, 1.0, 20)])
def test_matches_list_restatement(seed, n_recent, n_heavy, theta, spread, P):
    rng = np.random.default_rng(300 + seed)
    T = 80
    K, V, Q = _inputs(rng, P, T, spread)
    u = Unit(H2O_POOLS, 0, n_heavy, n_recent, n_recent + n_heavy, 0, 0, G, D)
    u.set_hh_threshold(theta)
    u.prefill(K[:P], V[:P])
    m = _ListModel(n_recent, n_heavy, theta)
    for p in range(P):
        m.add(p, {q: 0.0 for q in m.recent + m.hh + [p]})
    for t in range(T):
        p = P + t
        keys = m.kept() + [p]
        w = _sdpa_weights(Q[t], K[keys])
        m.add(p, dict(zip(keys, w)))
        u.step(Q[t], K[p], V[p])
        st = _state(u)
        assert sorted(st) == m.kept(), t
        for q, (pool, sc, slot) in st.items():
            assert pool == (1 if q in m.hh else 0), (t, q)
            assert sc == pytest.approx(m.score[q], rel=1e-12, abs=1e-15)
            k, v = u.slot_kv(slot)
            np.testing.assert_array_equal(k, K[q])
            np.testing.assert_array_equal(v, V[q])


@pytest.mark.parametrize("seed,n_recent,n_heavy", [(0, 3, 3), (1, 2, 5), (2, 4, 1)])
def test_theta_minus_inf_is_the_best_subset(seed, n_recent, n_heavy):
    """Every token leaving the recent pool is promoted, so one token leaves the
    cache only when it is full: the lowest of (kept + new), which keeps the
    budget-subset with the highest total score."""
    rng = np.random.default_rng(40 + seed)
    C, P, T = n_recent + n_heavy, 2, 60
    K, V, Q = _inputs(rng, P, T, 2.0)
    u = Unit(H2O_POOLS, 0, n_heavy, n_recent, C, 0, 0, G, D)
    u.set_hh_threshold(-math.inf)
    u.prefill(K[:P], V[:P])
    for t in range(T):
        p = P + t
        before = set(_state(u))
        u.attend(Q[t], K[p], V[p])
        sc = {q: s for q, (_, s, _) in _state(u).items()}
        sc[p] = u.new_score
        u.commit(u.choose())
        after = set(_state(u))
        if len(before) < C:
            assert after == before | {p}  # nothing leaves before the cache is full
            continue
        best = max(itertools.combinations(sorted(sc), C), key=lambda ks: math.fsum(sc[q] for q in ks))
        assert after == set(best), t


@pytest.mark.parametrize("seed,n_recent,n_heavy", [(0, 3, 3), (1, 4, 0)])
def test_theta_plus_inf_keeps_only_the_recent_pool(seed, n_recent, n_heavy):
    rng = np.random.default_rng(70 + seed)
    P, T = 7, 50
    K, V, Q = _inputs(rng, P, T, 2.0)
    u = Unit(H2O_POOLS, 0, n_heavy, n_recent, n_recent + n_heavy, 0, 0, G, D)
    u.set_hh_threshold(math.inf)
    u.prefill(K[:P], V[:P])
    assert set(_state(u)) == set(range(P - n_recent, P))
    for t in range(T):
        p = P + t
        u.attend(Q[t], K[p], V[p])
        st = _state(u)
        sc = {q: s for q, (_, s, _) in st.items()}
        sc[p] = u.new_score
        u.commit(u.choose())
        after = _state(u)
        assert all(pool == 0 for pool, _, _ in after.values())
        best = max(itertools.combinations(sorted(sc), n_recent), key=lambda ks: math.fsum(sc[q] for q in ks))
        assert set(after) == set(best), t


@pytest.mark.parametrize("P,n_recent,n_heavy,theta", [(50, 8, 12, 0.0), (50, 8, 12, -0.5), (13, 8, 12, -0.5),
                                                      (5, 8, 12, 1.0), (64, 16, 0, -1.0)])
def test_prompt_layout_closed_form(P, n_recent, n_heavy, theta):
    """All prompt scores are 0, so the recent pool's oldest member leaves each
    time: theta >= 0 drops it (the last n_recent positions stay, position q in
    slot q mod n_recent), theta < 0 promotes it (the last C stay, q in slot
    q mod C, heavy-hitter pool = the positions before the last n_recent)."""
    C = n_recent + n_heavy
    u = Unit(H2O_POOLS, 0, n_heavy, n_recent, C, 0, 0, 1, 4)
    u.set_hh_threshold(theta)
    z = np.zeros((P, 4), np.float32)
    u.prefill(z, z)
    ring = n_recent if theta >= 0 else C
    want_pos = np.full(C, -1, np.int32)
    want_pool = np.zeros(C, np.int8)
    for q in range(max(0, P - ring), P):
        want_pos[q % ring] = q
        want_pool[q % ring] = 1 if q < P - n_recent else 0
    np.testing.assert_array_equal(u.positions(), want_pos)
    np.testing.assert_array_equal(np.where(want_pos >= 0, u.pools(), 0), want_pool)


def test_invariants_over_a_long_run():
    rng = np.random.default_rng(12)
    n_recent, n_heavy, theta = 6, 10, 0.05
    C, P, T = n_recent + n_heavy, 4, 400
    K, V, Q = _inputs(rng, P, T, 2.0)
    u = Unit(H2O_POOLS, 0, n_heavy, n_recent, C, 0, 0, G, D)
    u.set_hh_threshold(theta)
    u.prefill(K[:P], V[:P])
    count = u.count
    promotions = drops_new = 0
    for t in range(T):
        p = P + t
        u.attend(Q[t], K[p], V[p])
        sc_before = {q: s for q, (_, s, _) in _state(u).items()}
        sc_before[p] = u.new_score
        slot = u.choose()
        u.commit(slot)
        st = _state(u)
        pools = [pool for pool, _, _ in st.values()]
        assert pools.count(0) <= n_recent and pools.count(1) <= n_heavy
        pr = u.last_promote
        if pr != -1:
            promotions += 1
            q = p if pr == -2 else int(u.positions()[pr])
            assert sc_before[q] > theta  # promoted strictly above the threshold
        if slot == u.cap:
            drops_new += 1
            assert p not in st and u.last_victim_pos == p
        assert u.count >= count  # never shrinks
        count = u.count
        pos = u.positions()
        assert np.all(pos[:count] >= 0) and np.all(pos[count:] == -1)  # contiguous occupancy
    assert promotions > 10 and drops_new > 0
    occ = u.positions() >= 0
    assert math.fsum(u.scores()[occ]) + u.evicted_mass == pytest.approx(T, rel=1e-12)


def test_commit_pools_adopts_a_valid_decision_only():
    u = Unit(H2O_POOLS, 0, 2, 2, 4, 0, 0, 1, 4)
    u.set_hh_threshold(-1.0)
    z = np.ones((4, 4), np.float32)
    u.prefill(z, z)  # positions 0..3: slots 0, 1 heavy hitters, 2, 3 recent
    np.testing.assert_array_equal(u.pools(), [1, 1, 0, 0])
    u.attend(np.ones((1, 4), np.float32), z[0], z[0])
    for bad in [(0, 0, -1),   # three tokens in a recent pool of two
                (4, 1, -1),   # a dropped new token joins no pool
                (1, 1, 2),    # the new token and a held one both promoted
                (2, 0, 2)]:   # a slot both refilled and promoted
        with pytest.raises(RuntimeError):
            u.commit_pools(*bad)
    u.commit_pools(0, 0, 2)  # heavy hitter 0 leaves, recent 2 promoted, the new token recent
    np.testing.assert_array_equal(u.pools(), [0, 1, 1, 0])
    np.testing.assert_array_equal(u.positions(), [4, 1, 2, 3])
    assert u.last_promote == 2 and u.last_victim_pos == 0


def test_invalid_configs_rejected():
    with pytest.raises(ValueError):
        Unit(H2O_POOLS, 1, 3, 4, 8, 0, 0, 1, 4)  # no sinks in the two-pool class
    with pytest.raises(ValueError):
        Unit(H2O_POOLS, 0, 3, 0, 3, 0, 0, 1, 4)  # a recent pool of at least one
    with pytest.raises(ValueError):
        Unit(H2O_POOLS, 0, 3, 4, 8, 0, 0, 1, 4)  # pools must add up to the budget
    with pytest.raises(RuntimeError):
        Unit(H2O, 0, 3, 4, 7, 0, 0, 1, 4).set_hh_threshold(0.1)
    with pytest.raises(RuntimeError):
        Unit(H2O_POOLS, 0, 3, 4, 7, 0, 0, 1, 4).set_hh_threshold(math.nan)
