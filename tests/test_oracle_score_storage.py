"""Pins of the oracle's score-storage variants ("Attention Sinks 与 KV Cache 淘汰
策略" section 6.2: FP16 storage of the cumulative scores, or a moving average in
place of the exact accumulation) to things other than itself: the binary16
rounding against numpy's float16 conversion, the moving average against the
per-step attention weights of torch's fp64 SDPA weighted by powers of the
keep factor, FP16 storage against the same recursion rounded by numpy, the
exact accumulation as the forget = 0 case, and the selection on the stored
(rounded) scores against brute force (ties are common in FP16).
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle import H2O, H2O_BLOCK, SINK_WINDOW, Unit


def test_round_half_matches_numpy_float16():
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(0, 70000, 4000), np.exp(rng.uniform(-25, 11, 4000)),
                         [0.0, 2.0**-24, 2.0**-25, 3 * 2.0**-25, 2.0**-14, 65504.0, 65519.99, 65520.0, 1e5]])
    # the exact midpoints between neighbouring binary16 values: ties go to even
    h = np.arange(0, 0x7BFF, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    xs = np.concatenate([xs, (h[:-1] + h[1:]) / 2])
    for x in xs:
        with np.errstate(over="ignore"):
            ref = float(np.float16(x))
        assert oracle.round_half(float(x)) == ref, x


def _sdpa_weights(Q, K, t, P):
    """Attention of step t's query heads over positions 0..P+t (fp64 SDPA with
    V = I): [G][P + t + 1]."""
    import torch
    import torch.nn.functional as F
    n = P + t + 1
    G, d = Q.shape[1], Q.shape[2]
    q = torch.from_numpy(Q[t].astype(np.float64))[None, :, None, :]
    k = torch.from_numpy(K[:n].astype(np.float64))[None, None].expand(1, G, n, d)
    eye = torch.eye(n, dtype=torch.float64)[None, None].expand(1, G, n, n)
    return F.scaled_dot_product_attention(q, k, eye)[0, :, 0, :].numpy()


@pytest.mark.parametrize("forget,half", [(0.0, False), (0.1, False), (0.5, False), (0.0, True), (0.05, True)])
def test_storage_recursion_against_sdpa(forget, half):
    rng = np.random.default_rng(60 + int(forget * 100) + half)
    P, T, G, d = 6, 30, 2, 8
    n = P + T
    u = Unit(H2O, 2, n, 3, n + 5, 0, 0, G, d)  # never evicts
    u.set_score_storage(forget, half)
    K = rng.standard_normal((n, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    u.prefill(K[:P], K[:P])
    ref = np.zeros(n)
    rnd = (lambda x: np.float16(x).astype(np.float64)) if half else (lambda x: x)
    for t in range(T):
        u.step(Q[t], K[P + t], K[P + t])
        w = _sdpa_weights(Q, K, t, P).mean(axis=0)  # [P + t + 1]
        m = P + t + 1
        ref[:m - 1] = rnd((1.0 - forget) * ref[:m - 1] + w[:m - 1])
        ref[m - 1] = rnd(w[m - 1])
    pos, sc = u.positions(), u.scores()
    got = np.zeros(n)
    got[pos[pos >= 0]] = sc[pos >= 0]
    if half:  # the stored values are binary16 values, equal to the numpy-rounded recursion
        assert np.all(np.float16(got).astype(np.float64) == got)
        np.testing.assert_allclose(got, ref, rtol=2.0**-10, atol=2.0**-24)
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    if forget == 0.0 and not half:
        assert math.fsum(sc[pos >= 0]) == pytest.approx(T, rel=1e-12)


def test_forget_zero_is_the_exact_accumulation():
    rng = np.random.default_rng(8)
    P, T, G, d = 5, 40, 2, 8
    a, b = Unit(H2O, 1, 6, 3, 10, 0, 0, G, d), Unit(H2O, 1, 6, 3, 10, 0, 0, G, d)
    b.set_score_storage(0.0, False)
    K = rng.standard_normal((P + T, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    a.prefill(K[:P], K[:P])
    b.prefill(K[:P], K[:P])
    for t in range(T):
        a.step(Q[t], K[P + t], K[P + t])
        b.step(Q[t], K[P + t], K[P + t])
    np.testing.assert_array_equal(a.positions(), b.positions())
    np.testing.assert_array_equal(a.scores(), b.scores())


@pytest.mark.parametrize("forget", [0.0, 0.2])
def test_fp16_selection_equals_brute_force_on_stored_scores(forget):
    rng = np.random.default_rng(70 + int(forget * 10))
    n_sink, n_heavy, n_recent = 1, 3, 2
    K_ = n_sink + n_heavy + n_recent
    P, T, G, d = 3, 40, 2, 4
    u = Unit(H2O, n_sink, n_heavy, n_recent, K_, 0, 0, G, d)
    u.set_score_storage(forget, True)
    Kk = rng.standard_normal((P + T, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    u.prefill(Kk[:P], Kk[:P])
    ties = 0
    for t in range(T):
        p = P + t
        u.attend(Q[t], Kk[p], Kk[p])
        pos, sc = u.positions(), u.scores()
        cand = {int(pos[s]): sc[s] for s in range(K_) if pos[s] >= 0}
        cand[p] = u.new_score
        slot = u.choose()
        u.commit(slot)
        if len(cand) <= K_:
            continue
        after = set(int(x) for x in u.positions() if x >= 0)
        protected = {q for q in cand if q < n_sink or q > p - n_recent}
        elig = sorted(set(cand) - protected, key=lambda q: (cand[q], q))
        ties += len(elig) > 1 and cand[elig[0]] == cand[elig[1]]
        best = None
        for keep in itertools.combinations(sorted(cand), K_):
            if not protected <= set(keep):
                continue
            f = math.fsum(cand[q] for q in keep)
            gone = (set(cand) - set(keep)).pop()
            key = (-f, cand[gone], gone)
            if best is None or key < best[0]:
                best = (key, set(keep))
        assert after == best[1]
    assert u.greedy_disagreements == 0


def test_storage_modes_checked():
    with pytest.raises(RuntimeError):
        Unit(SINK_WINDOW, 1, 0, 4, 5, 0, 0, 1, 4).set_score_storage(0.1, False)
    with pytest.raises(RuntimeError):
        Unit(H2O_BLOCK, 1, 8, 3, 12, 3, 0, 1, 4).set_score_storage(0.0, True)  # FP16 for H2O only
    Unit(H2O_BLOCK, 1, 8, 3, 12, 3, 0, 1, 4).set_score_storage(0.3, False)
    with pytest.raises(RuntimeError):
        Unit(H2O, 1, 2, 1, 4, 0, 0, 1, 4).set_score_storage(1.0, False)
    u = Unit(H2O, 1, 2, 1, 4, 0, 0, 1, 4)
    u.prefill(np.zeros((2, 4), np.float32), np.zeros((2, 4), np.float32))
    with pytest.raises(RuntimeError):
        u.set_score_storage(0.1, False)  # only on an empty unit


# INT8 storage (section 6.2 names INT8 quantisation of the scores with no
# scale or zero point; the reading is absmax per unit: codes round(s * 255 / M),
# ties to even, M the unit's largest score after the update, the new token's
# included, stored as code * M / 255; fp64 like the rest of the oracle).


def _q8(x, M):
    """numpy fp64 absmax quantisation of values x with absmax M (np.rint
    rounds ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    c = np.clip(np.rint(x * 255.0 / M), 0.0, 255.0)
    return c * M / 255.0, c.astype(np.int64), M / 255.0


def _q8_fp32_rule(x, M):
    """The same codes taken in fp32, the order a GPU kernel takes them: s and
    M rounded to fp32, inv = 255 / M and the product in fp32, then rint."""
    M32 = np.float32(M)
    inv = np.float32(255.0) / M32
    c = np.minimum(np.rint(np.float32(x) * inv), np.float32(255.0))
    return c.astype(np.int64)


def test_int8_fp32_rule_differs_from_the_definition_only_at_midpoints():
    """The fp32 order of the codes (three roundings of at most 2^-24 relative
    each, plus those of s and M) moves s * 255 / M by at most 255 * 4 * 2^-24
    = 6.1e-5 codes: its code equals the fp64 definition's except where the
    unrounded value lies within 1e-4 of a midpoint k + 1/2, and then by one.
    Values placed exactly at midpoints show that such differences happen."""
    rng = np.random.default_rng(2026)
    M = rng.uniform(1e-3, 50.0, 4000)
    x = rng.uniform(0.0, 1.0, (4000, 64)) * M[:, None]
    # values right at midpoints of the code grid (k + 1/2) * M / 255
    k = rng.integers(0, 255, (4000, 16))
    mids = (k + 0.5) * M[:, None] / 255.0
    vals = np.concatenate([x, mids], axis=1)
    moved = 0
    for i in range(len(M)):
        _, c64, _ = _q8(vals[i], M[i])
        c32 = _q8_fp32_rule(vals[i], M[i])
        d = np.abs(c64 - c32)
        assert d.max() <= 1
        u = vals[i] * 255.0 / M[i]
        frac = np.abs(u - np.floor(u) - 0.5)
        assert np.all(frac[d == 1] < 1e-4)
        moved += int(d.sum())
    assert moved > 0  # midpoint values do round apart


@pytest.mark.parametrize("forget", [0.0, 0.1])
def test_int8_recursion_against_sdpa(forget):
    """Never evicting: the stored scores follow s <- q((1 - forget) s + a), a
    from torch's fp64 SDPA, q the numpy fp64 absmax quantisation over the
    unit (the new token included); codes, scale and values agree."""
    rng = np.random.default_rng(81 + int(forget * 10))
    P, T, G, d = 6, 30, 2, 8
    n = P + T
    u = Unit(H2O, 2, n, 3, n + 5, 0, 0, G, d)
    u.set_score_storage(forget, False)
    u.set_score_int8(True)
    K = rng.standard_normal((n, d)).astype(np.float32)
    Q = rng.standard_normal((T, G, d)).astype(np.float32)
    u.prefill(K[:P], K[:P])
    ref = np.zeros(n)
    moved = 0
    for t in range(T):
        u.step(Q[t], K[P + t], K[P + t])
        w = _sdpa_weights(Q, K, t, P).mean(axis=0)
        m = P + t + 1
        upd = np.concatenate([(1.0 - forget) * ref[:m - 1] + w[:m - 1], w[m - 1:m]])
        M = float(np.max(upd))
        q, codes, scale = _q8(upd, M)
        pos, sc = u.positions(), u.scores()
        got = np.zeros(n)
        got[pos[pos >= 0]] = sc[pos >= 0]
        gc = np.zeros(n, np.int64)
        gc[pos[pos >= 0]] = u.score_codes()[pos >= 0]
        assert u.score_scale() == pytest.approx(scale, rel=1e-12)
        assert gc[:m].max() == 255 and gc[:m].min() >= 0
        # the stored values are code * M / 255, within half a step of the update
        np.testing.assert_allclose(got[:m], gc[:m] * (255.0 * u.score_scale()) / 255.0, rtol=1e-15, atol=0)
        assert np.all(np.abs(got[:m] - upd) <= 0.5 * scale * (1 + 1e-12) + 1e-15)
        # codes equal numpy's: both fp64, from attention weights that agree to
        # rounding (SDPA and the oracle sum in different orders)
        diff = np.abs(gc[:m] - codes)
        assert diff.max() <= 1
        moved += int(diff.sum())
        ref[:m] = got[:m]  # the recursion continues from the stored values
    assert moved == 0


def test_int8_selection_equals_brute_force_on_stored_scores():
    rng = np.random.default_rng(90)
    n_sink, n_heavy, n_recent = 1, 3, 2
    K_ = n_sink + n_heavy + n_recent
    P, T, G, d = 10, 60, 2, 4
    u = Unit(H2O, n_sink, n_heavy, n_recent, K_, 0, 0, G, d)
    u.set_score_int8(True)
    Kk = rng.standard_normal((P + T, d)).astype(np.float32)
    # a sink that takes nearly all the weight: the prompt tokens held past the
    # window keep code 0 with the tokens leaving it, so equal codes meet
    Kk[0] = 10.0 * np.abs(Kk[0])
    Q = np.abs(rng.standard_normal((T, G, d))).astype(np.float32)
    u.prefill(Kk[:P], Kk[:P])
    ties = 0
    for t in range(T):
        p = P + t
        u.attend(Q[t], Kk[p], Kk[p])
        pos, sc, codes = u.positions(), u.scores(), u.score_codes()
        cand = {int(pos[s]): sc[s] for s in range(K_) if pos[s] >= 0}
        cand[p] = u.new_score
        assert max(codes.max(), round(u.new_score / u.score_scale())) == 255
        slot = u.choose()
        u.commit(slot)
        if len(cand) <= K_:
            continue
        after = set(int(x) for x in u.positions() if x >= 0)
        protected = {q for q in cand if q < n_sink or q > p - n_recent}
        elig = sorted(set(cand) - protected, key=lambda q: (cand[q], q))
        ties += len(elig) > 1 and cand[elig[0]] == cand[elig[1]]
        best = None
        for keep in itertools.combinations(sorted(cand), K_):
            if not protected <= set(keep):
                continue
            f = math.fsum(cand[q] for q in keep)
            gone = (set(cand) - set(keep)).pop()
            key = (-f, cand[gone], gone)
            if best is None or key < best[0]:
                best = (key, set(keep))
        assert after == best[1]
    assert u.greedy_disagreements == 0
    assert ties > 0  # 256 levels: equal codes happen, and the older token leaves


def test_int8_identical_keys_closed_form():
    """Identical keys, no eviction: every step spreads weight 1/n_t evenly, so
    tokens present for equal numbers of steps hold bit-identical codes, the
    prompt tokens (present longest) hold 255 and their stored value is the
    exact score, and each code stays within the rounding drift of the ratio
    of closed-form scores: half a code per step so far (the scale only grows,
    so an earlier step's half code is at most half a code now)."""
    P, T, G, d = 4, 25, 1, 4
    n = P + T
    u = Unit(H2O, 1, n, 1, n + 2, 0, 0, G, d)
    u.set_score_int8(True)
    k = np.ones((n, d), np.float32)
    u.prefill(k[:P], k[:P])
    q = np.ones((G, d), np.float32)
    for t in range(T):
        u.step(q, k[0], k[0])
        pos, codes = u.positions(), u.score_codes()
        by_pos = {int(pos[s]): int(codes[s]) for s in range(len(pos)) if pos[s] >= 0}
        assert all(by_pos[j] == 255 for j in range(P))
        # exact scores: a token first attended at step t0 holds sum_{t0 <= s <= t} 1/(P + s + 1)
        exact = {j: sum(1.0 / (P + s + 1) for s in range(max(0, j - P), t + 1)) for j in by_pos}
        top = exact[0]
        assert u.score_scale() * 255 == pytest.approx(top, rel=1e-6)
        for j, c in by_pos.items():
            assert abs(c - 255 * exact[j] / top) <= 0.5 * (t + 1) + 1e-3, (t, j, c)
        for j in range(P, P + t):  # monotone in age
            assert by_pos[j] >= by_pos[j + 1]


def test_int8_modes_checked():
    with pytest.raises(RuntimeError):
        Unit(SINK_WINDOW, 1, 0, 4, 5, 0, 0, 1, 4).set_score_int8(True)
    with pytest.raises(RuntimeError):
        Unit(H2O_BLOCK, 1, 8, 3, 12, 3, 0, 1, 4).set_score_int8(True)
    u = Unit(H2O, 1, 2, 1, 4, 0, 0, 1, 4)
    u.set_score_storage(0.0, True)
    with pytest.raises(RuntimeError):
        u.set_score_int8(True)  # not with binary16
    u = Unit(H2O, 1, 2, 1, 4, 0, 0, 1, 4)
    u.prefill(np.zeros((2, 4), np.float32), np.zeros((2, 4), np.float32))
    with pytest.raises(RuntimeError):
        u.set_score_int8(True)  # on an empty unit only


def test_int8_new_token_sets_the_scale():
    """Right after a prefill (scores 0) a new token whose key points along
    the query takes the largest weight: it alone sets the scale (code 255),
    and the prompt tokens' codes are their SDPA weights over its weight,
    rounded (fp64)."""
    rng = np.random.default_rng(12)
    P, G, d = 6, 1, 8
    u = Unit(H2O, 1, P, 2, P + 3, 0, 0, G, d)
    u.set_score_int8(True)
    K = rng.standard_normal((P + 1, d)).astype(np.float32)
    Q = rng.standard_normal((1, G, d)).astype(np.float32)
    K[P] = 2.0 * Q[0, 0]
    u.prefill(K[:P], K[:P])
    u.attend(Q[0], K[P], K[P])
    w = _sdpa_weights(Q, K, 0, P).mean(axis=0)
    assert np.argmax(w) == P
    q, codes, scale = _q8(w, float(w[P]))
    assert u.score_scale() == pytest.approx(scale, rel=1e-12)
    assert round(u.new_score / u.score_scale()) == 255
    pos = u.positions()
    got = u.score_codes()
    for s in range(len(pos)):
        if pos[s] >= 0:
            assert abs(int(got[s]) - int(codes[pos[s]])) <= 0  # no midpoint at these values
    assert int(codes[:P].max()) < 255
