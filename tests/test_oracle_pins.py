"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against what the pages or the mathematics fix:
a library routine (numpy's Philox4x64-10, torch's fp64 scaled-dot-product
attention), a closed form (identical keys), brute force on tiny inputs, an
equivalence the pages state (StreamingLLM is H2O without heavy hitters),
figures the pages print (tests/golden/page_figures.txt) and invariants
(sinks, the recent window and the prompt are never evicted; the cache never
exceeds its budget; softmax mass is conserved).
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import H2O, RANDOM, SINK_WINDOW, Unit
from workloads import configs, synth, traffic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")


def golden():
    vals = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = float(v)
    return vals


# ----------------------------------------------------------------------------
# Philox4x64-10 against numpy's implementation of the same generator
# ----------------------------------------------------------------------------

def numpy_philox_block(ctr, key):
    """numpy advances the 256-bit counter before each block, so start one below."""
    val = sum(int(c) << (64 * i) for i, c in enumerate(ctr))
    val = (val - 1) % (1 << 256)
    cm1 = np.array([(val >> (64 * i)) & ((1 << 64) - 1) for i in range(4)], dtype=np.uint64)
    bg = np.random.Philox(key=np.array([int(k) for k in key], dtype=np.uint64), counter=cm1)
    return bg.random_raw(4)


def test_philox_matches_numpy():
    rng = np.random.default_rng(7)
    cases = [([0, 0, 0, 0], [0, 0]), ([2**64 - 1] * 4, [2**64 - 1] * 2), ([1, 0, 0, 0], [5, 6])]
    for _ in range(200):
        cases.append((rng.integers(0, 2**64, size=4, dtype=np.uint64).tolist(),
                      rng.integers(0, 2**64, size=2, dtype=np.uint64).tolist()))
    for ctr, key in cases:
        np.testing.assert_array_equal(oracle.philox4x64_10(ctr, key), numpy_philox_block(ctr, key))


def test_random_key_counter_layout():
    rng = np.random.default_rng(8)
    for _ in range(100):
        seed = int(rng.integers(0, 2**63))
        seq, layer, head, step, pos = (int(x) for x in rng.integers(0, 30000, size=5))
        layer %= 80
        head %= 64
        expect = numpy_philox_block([pos, step, (layer << 16) + head, seq], [seed, 0x5EED0001])[0]
        assert oracle.random_key(seed, seq, layer, head, step, pos) == int(expect)


# ----------------------------------------------------------------------------
# Attention: budget >= length means no eviction, so the output is plain
# causal decode attention (torch fp64 SDPA); identical keys give the mean of V
# ----------------------------------------------------------------------------

def _rand_inputs(rng, P, T, G, d):
    K = rng.standard_normal((P + T, d)).astype(np.float32)
    V = rng.standard_normal((P + T, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    return K, V, Q


@pytest.mark.parametrize("policy", [H2O, SINK_WINDOW, RANDOM])
def test_no_eviction_equals_full_attention(policy):
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(11 + policy)
    P, T, G, d = 12, 25, 4, 16
    n = P + T
    if policy == H2O:
        u = Unit(H2O, 2, n - 5, 3, n, 0, 0, G, d)
    elif policy == SINK_WINDOW:
        u = Unit(SINK_WINDOW, 2, 0, n, n + 2, 0, 0, G, d)
    else:
        u = Unit(RANDOM, 0, 0, 0, T, 1, P, G, d)  # budget T + r: never cuts
    K, V, Q = _rand_inputs(rng, P, T, G, d)
    u.prefill(K[:P], V[:P])
    for t in range(T):
        out, _ = u.step(Q[t], K[P + t], V[P + t])
        m = P + t + 1
        q = torch.from_numpy(Q[t].astype(np.float64))[None, :, None, :]
        k = torch.from_numpy(K[:m].astype(np.float64))[None, None].expand(1, G, m, d)
        v = torch.from_numpy(V[:m].astype(np.float64))[None, None].expand(1, G, m, d)
        ref = F.scaled_dot_product_attention(q, k, v)[0, :, 0, :].numpy()
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    assert u.count == n


def test_identical_keys_mean_of_values_and_harmonic_scores():
    rng = np.random.default_rng(3)
    P, T, G, d = 5, 30, 2, 8
    n = P + T
    u = Unit(H2O, 1, n - 2, 1, n, 0, 0, G, d)
    c = rng.standard_normal(d).astype(np.float32)
    K = np.tile(c, (n, 1))
    V = rng.standard_normal((n, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    u.prefill(K[:P], V[:P])
    for t in range(T):
        out, _ = u.step(Q[t], K[P + t], V[P + t])
        mean_v = V[:P + t + 1].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(out, np.broadcast_to(mean_v, out.shape), rtol=1e-12, atol=1e-13)
    # score(pos j) = sum over steps t >= max(0, j - P) of 1 / (P + t + 1)
    H = [Fraction(0)]
    for i in range(1, n + 1):
        H.append(H[-1] + Fraction(1, i))
    pos, sc = u.positions(), u.scores()
    for s in range(n):
        j = int(pos[s])
        expect = float(H[P + T] - H[max(P, j)])
        assert sc[s] == pytest.approx(expect, rel=1e-12)
    assert math.fsum(sc) == pytest.approx(T, rel=1e-13)


def test_identical_keys_eviction_trajectory():
    """Identical keys and P > K: every step attends K+1 tokens, each gets
    exactly 1/(K+1). For t <= n_recent all candidates tie and the older
    position leaves (FIFO over the prompt); afterwards the victim is always
    the token leaving the window, position p - n_recent."""
    rng = np.random.default_rng(5)
    n_sink, n_heavy, n_recent = 2, 3, 3
    K_ = n_sink + n_heavy + n_recent
    P, T, G, d = 20, 15, 1, 4
    u = Unit(H2O, n_sink, n_heavy, n_recent, K_, 0, 0, G, d)
    c = rng.standard_normal(d).astype(np.float32)
    Kk = np.tile(c, (P + T, 1))
    V = rng.standard_normal((P + T, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    u.prefill(Kk[:P], V[:P])
    # expected layout after prefill: sinks in slots 0..n_sink-1, the newest
    # K - n_sink prompt tokens in ring order
    slot_of = {p: p for p in range(n_sink)}
    for p in range(n_sink, P):
        slot_of[p] = n_sink + (p - n_sink) % (K_ - n_sink)
    retained = set(range(n_sink)) | set(range(P - (K_ - n_sink), P))
    expect = np.full(K_, -1, np.int32)
    for p in retained:
        expect[slot_of[p]] = p
    np.testing.assert_array_equal(u.positions(), expect)
    for t in range(T):
        p = P + t
        if t <= n_recent:
            victim = min(q for q in retained if q >= n_sink)
        else:
            victim = p - n_recent
        u.step(Q[t], Kk[p], V[p])
        slot = slot_of.pop(victim)
        retained.remove(victim)
        retained.add(p)
        slot_of[p] = slot
        expect[slot] = p
        np.testing.assert_array_equal(u.positions(), expect)
        assert u.last_victim_pos == victim
    # scores: (steps present) / (K+1), bit-identical for equal presence counts
    pos, sc = u.positions(), u.scores()
    by_count = {}
    for s in range(K_):
        q = int(pos[s])
        present = T if q < P else T - (q - P)
        by_count.setdefault(present, set()).add(sc[s])
        assert sc[s] == pytest.approx(present / (K_ + 1), rel=1e-13)
    for vals in by_count.values():
        assert len(vals) == 1


# ----------------------------------------------------------------------------
# H2O greedy (Algorithm 1) against brute-force enumeration of retained sets
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_h2o_greedy_equals_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n_sink, n_heavy, n_recent = 1, 3, 2
    K_ = n_sink + n_heavy + n_recent
    P, T, G, d = 3, 12, 2, 4
    u = Unit(H2O, n_sink, n_heavy, n_recent, K_, 0, 0, G, d)
    Kk, V, Q = _rand_inputs(rng, P, T, G, d)
    u.prefill(Kk[:P], V[:P])
    for t in range(T):
        p = P + t
        u.attend(Q[t], Kk[p], V[p])
        pos, sc = u.positions(), u.scores()
        cand = {int(pos[s]): sc[s] for s in range(K_) if pos[s] >= 0}
        cand[p] = u.new_score
        slot = u.choose()
        u.commit(slot)
        after = set(int(x) for x in u.positions() if x >= 0)
        if len(cand) <= K_:
            assert after == set(cand)
            continue
        protected = {q for q in cand if q < n_sink or q > p - n_recent}
        best, best_sets = -1.0, []
        for keep in itertools.combinations(sorted(cand), K_):
            if not protected <= set(keep):
                continue
            f = math.fsum(cand[q] for q in keep)
            if f > best + 1e-15:
                best, best_sets = f, [set(keep)]
            elif abs(f - best) <= 1e-15:
                best_sets.append(set(keep))
        assert len(best_sets) == 1
        assert after == best_sets[0]
    assert u.greedy_disagreements == 0


# ----------------------------------------------------------------------------
# StreamingLLM sink + window equals H2O with zero heavy hitters
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("P,T", [(0, 40), (9, 30)])
def test_sink_window_equals_h2o_without_heavy_hitters(P, T):
    rng = np.random.default_rng(21 + P)
    n_sink, n_recent, G, d = 2, 5, 2, 8
    a = Unit(SINK_WINDOW, n_sink, 0, n_recent, n_sink + n_recent, 0, 0, G, d)
    b = Unit(H2O, n_sink, 0, n_recent, n_sink + n_recent, 0, 0, G, d)
    Kk, V, Q = _rand_inputs(rng, P, T, G, d)
    a.prefill(Kk[:P], V[:P])
    b.prefill(Kk[:P], V[:P])
    np.testing.assert_array_equal(a.positions(), b.positions())
    for t in range(T):
        oa, sa = a.step(Q[t], Kk[P + t], V[P + t])
        ob, sb = b.step(Q[t], Kk[P + t], V[P + t])
        assert sa == sb
        np.testing.assert_array_equal(oa, ob)
        np.testing.assert_array_equal(a.positions(), b.positions())
        # closed-form ring slot of the newest token
        p = P + t
        expect_slot = p if p < n_sink else n_sink + (p - n_sink) % n_recent
        assert sa == expect_slot


# ----------------------------------------------------------------------------
# Invariants on the seeded H2O tiny workload (hub/sink structure)
# ----------------------------------------------------------------------------

def test_h2o_tiny_invariants():
    w = configs.H2O_TINY
    for head in range(w.n_kv_heads):
        x = synth.UnitInputs(w, 0, 0, head)
        u = Unit.for_workload(w, 0, 0, head)
        u.prefill(x.prompt_k, x.prompt_v)
        assert u.count == w.budget
        for t in range(w.decode_steps):
            p = w.prompt_len + t
            u.step(x.q[t], x.k_new[t], x.v_new[t])
            held = set(int(q) for q in u.positions() if q >= 0)
            assert len(held) == w.budget
            assert set(range(w.n_sink)) <= held
            assert set(range(p - w.n_recent + 1, p + 1)) <= held
            # softmax mass: every step adds exactly 1 to retained + evicted
            total = math.fsum(u.scores()) + u.evicted_mass
            assert total == pytest.approx(t + 1, rel=1e-12)
        assert u.greedy_disagreements == 0


def test_streaming_layout_from_the_pages():
    g = golden()
    n_sink, span, kept = int(g["streaming_n_sink"]), int(g["streaming_window_span"]), int(g["streaming_total_kept"])
    u = Unit(SINK_WINDOW, n_sink, 0, kept - n_sink, kept, 0, 0, 1, 2)
    rng = np.random.default_rng(9)
    N = 1500
    Kk = rng.standard_normal((N + 1, 2)).astype(np.float32)
    for p in range(N):
        u.step(Kk[p][None], Kk[p], Kk[p])
    u.attend(Kk[N][None], Kk[N], Kk[N])
    attended = set(int(q) for q in u.positions() if q >= 0) | {N}
    assert attended == set(range(n_sink)) | set(range(N - span, N + 1))
    u.commit(u.choose())
    held = set(int(q) for q in u.positions() if q >= 0)
    assert len(held) == kept
    assert held == set(range(n_sink)) | set(range(N - span + 1, N + 1))


def test_h2o_layout_from_the_pages():
    g = golden()
    s, h, r = int(g["h2o_n_sink"]), int(g["h2o_n_heavy"]), int(g["h2o_n_recent"])
    u = Unit(H2O, s, h, r, s + h + r, 0, 0, 1, 2)
    rng = np.random.default_rng(10)
    P, T = 1100, 60
    Kk = rng.standard_normal((P + T, 2)).astype(np.float32)
    u.prefill(Kk[:P], Kk[:P])
    for t in range(T):
        u.step(Kk[P + t][None], Kk[P + t], Kk[P + t])
        p = P + t
        held = set(int(q) for q in u.positions() if q >= 0)
        assert len(held) == s + h + r
        assert set(range(s)) <= held and set(range(p - r + 1, p + 1)) <= held


# ----------------------------------------------------------------------------
# Random Attention
# ----------------------------------------------------------------------------

def test_random_cut_invariants_and_selection():
    rng = np.random.default_rng(12)
    P, K_, r, G, d, T = 6, 10, 4, 2, 8, 60
    seed, seq, layer, head = 99, 3, 2, 1
    u = Unit(RANDOM, 0, 0, 0, K_, r, P, G, d, seed, seq, layer, head)
    Kk, V, Q = _rand_inputs(rng, P, T, G, d)
    u.prefill(Kk[:P], V[:P])
    before = set(range(P))
    n_gen, cuts = 0, 0
    for t in range(T):
        p = P + t
        u.step(Q[t], Kk[p], V[p])
        held = set(int(q) for q in u.positions() if q >= 0)
        assert set(range(P)) <= held  # the prompt is never evicted
        pre = before | {p}
        n_gen += 1
        if n_gen == K_ + r:
            cuts += 1
            assert t == K_ + r - 1 + (cuts - 1) * r
            gen = sorted(q for q in pre if q >= P)
            keys = {q: int(numpy_philox_block([q, t, (layer << 16) + head, seq], [seed, 0x5EED0001])[0])
                    for q in gen}
            evict = set(sorted(gen, key=lambda q: (keys[q], q))[:r])
            assert pre - held == evict
            n_gen = K_
        else:
            assert held == pre
        assert sum(1 for q in held if q >= P) == n_gen
        before = held
    assert u.cuts == cuts > 0


def test_random_prefill_capacity_error():
    u = Unit(RANDOM, 0, 0, 0, 4, 2, 3, 1, 2)
    with pytest.raises(RuntimeError):
        u.prefill(np.zeros((4, 2)), np.zeros((4, 2)))


def test_random_uniform_and_independent_per_head():
    """At the first cut all K+r generated tokens are candidates: every age rank
    must leave with probability r/(K+r) (chi-square), and two heads' evicted
    sets must overlap like independent draws (hypergeometric mean r^2/(K+r))."""
    from scipy import stats
    K_, r, d = 12, 4, 2
    n = K_ + r
    counts = np.zeros(n)
    overlaps = []
    z = np.zeros((n, d), np.float32)
    q = np.zeros((n, 1, d), np.float32)
    for seq in range(300):
        ev = []
        for head in range(2):
            u = Unit(RANDOM, 0, 0, 0, K_, r, 0, 1, d, 2024, seq, 0, head)
            for t in range(n):
                u.step(q[t], z[t], z[t])
            gone = set(range(n)) - set(int(x) for x in u.positions() if x >= 0)
            assert len(gone) == r
            ev.append(gone)
            for g in gone:
                counts[g] += 1
        overlaps.append(len(ev[0] & ev[1]))
    expect = counts.sum() / n
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert stats.chi2.sf(chi2, n - 1) > 1e-4
    hyper = stats.hypergeom(n, r, r)
    se = math.sqrt(hyper.var() / len(overlaps))
    assert abs(np.mean(overlaps) - hyper.mean()) < 5 * se


# ----------------------------------------------------------------------------
# Sizing formulas against the figures the pages print
# ----------------------------------------------------------------------------

def test_sizing_figures_from_the_pages():
    g = golden()
    kv70 = traffic.kv_cache_bytes(80, 8, 128, 2, 32768) / 1e9
    assert round(kv70, 1) == g["kv_llama2_70b_32k_gb"]
    kv30 = traffic.kv_cache_bytes(48, 56, 128, 2, 1024 * 128) / 1e9
    assert round(kv30) == g["kv_opt30b_b128_s1024_gb"]
    assert traffic.score_bytes(1_000_000) / 1e6 == g["score_fp32_1m_tokens_mb"]
    assert traffic.score_bytes(32 * 1_000_000) / 1e6 == g["score_fp32_1m_tokens_b32_mb"]


def test_invalid_unit_configs_rejected():
    with pytest.raises(ValueError):
        Unit(H2O, 4, 60, 0, 64, 0, 0, 1, 8)      # n_recent must be >= 1
    with pytest.raises(ValueError):
        Unit(H2O, 4, 60, 64, 100, 0, 0, 1, 8)    # budget != sink + heavy + recent
    with pytest.raises(ValueError):
        Unit(SINK_WINDOW, 4, 3, 10, 17, 0, 0, 1, 8)  # sink-window has no heavy hitters
    with pytest.raises(ValueError):
        Unit(RANDOM, 0, 0, 0, 10, 0, 5, 1, 8)    # r >= 1
