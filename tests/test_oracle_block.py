"""Pins of the oracle's block-granular H2O ("Attention Sinks 与 KV Cache 淘汰策略"
section 5: a paged cache releases whole blocks) to things other than itself:
brute force over the blocks at every release (the released block maximises
the remaining cumulative score among the blocks wholly outside the sinks and
the recent window), the closed-form layout of a prompt longer than the cache
(all scores 0: the non-sink blocks are released round robin), and the
invariants (whole blocks leave, the freed slots refill lowest first, blocks
hold runs of consecutive positions, sinks and the recent window stay, the
score mass is conserved).
"""
import itertools
import math

import numpy as np
import pytest

from oracle import H2O_BLOCK, Unit


def _blocks(pos, bs):
    return [pos[b * bs:(b + 1) * bs] for b in range(len(pos) // bs)]


@pytest.mark.parametrize("seed,bs,n_sink,n_recent,C", [(0, 3, 1, 3, 12), (1, 4, 2, 5, 20), (2, 2, 0, 2, 10),
                                                       (3, 16, 4, 20, 96)])
def test_release_equals_brute_force(seed, bs, n_sink, n_recent, C):
    rng = np.random.default_rng(900 + seed)
    G, d, P, T = 2, 8, 6, 4 * C
    u = Unit(H2O_BLOCK, n_sink, C - n_sink - n_recent, n_recent, C, bs, 0, G, d)
    K = rng.standard_normal((P, d)).astype(np.float32)
    u.prefill(K, K)
    releases = 0
    for t in range(T):
        pos0, sc0 = u.positions().copy(), u.scores().copy()
        full = bool(np.all(pos0 >= 0))
        q = (rng.standard_normal((G, d)) * 1.5).astype(np.float32)
        kv = rng.standard_normal(d).astype(np.float32)
        _, slot = u.step(q, kv, kv)
        p = P + t
        if not full:
            assert u.last_block == -1
            assert slot == int(np.flatnonzero(pos0 < 0)[0])  # the lowest free slot
            continue
        releases += 1
        # brute force: every block wholly outside the sinks and the recent window
        best, best_key = None, None
        total = math.fsum(sc0)
        for b, (bp, bsc) in enumerate(zip(_blocks(pos0, bs), _blocks(sc0, bs))):
            if bp.min() < n_sink or bp.max() > p - n_recent:
                continue
            F = total - math.fsum(bsc)
            key = (-F, math.fsum(bsc), int(bp.min()))
            if best_key is None or key < best_key:
                best, best_key = b, key
        assert u.last_block == best, (t, u.last_block, best)
        assert slot == best * bs  # the incoming token takes the block's first slot
        pos = u.positions()
        assert pos[best * bs] == p and np.all(pos[best * bs + 1:(best + 1) * bs] == -1)
        assert u.greedy_disagreements == 0
    assert releases >= (T - C) // bs - 1


@pytest.mark.parametrize("P,bs,n_sink,n_recent,C", [(200, 16, 4, 20, 96), (77, 8, 10, 9, 64), (64, 8, 0, 8, 64)])
def test_long_prompt_layout_closed_form(P, bs, n_sink, n_recent, C):
    """With every prompt score 0 the released block is always the eligible one
    holding the oldest token: the non-sink blocks are recycled round robin."""
    G, d = 1, 4
    u = Unit(H2O_BLOCK, n_sink, C - n_sink - n_recent, n_recent, C, bs, 0, G, d)
    z = np.zeros((P, d), np.float32)
    u.prefill(z, z)
    nb, nsb = C // bs, -(-n_sink // bs)
    expect = np.full(C, -1, np.int32)
    for p in range(P):
        if p < C:
            slot = p
        else:
            k = p - C
            slot = (nsb + (k // bs) % (nb - nsb)) * bs + k % bs
        expect[slot] = p
    # the slots of the block released for the last round that are not refilled yet are empty
    if P > C and (P - C) % bs:
        blk = nsb + ((P - C) // bs) % (nb - nsb)
        expect[blk * bs + (P - C) % bs:(blk + 1) * bs] = -1
    np.testing.assert_array_equal(u.positions(), expect)


def test_invariants_over_a_long_run():
    rng = np.random.default_rng(11)
    G, d, bs, n_sink, n_recent, C = 4, 8, 4, 3, 9, 40
    u = Unit(H2O_BLOCK, n_sink, C - n_sink - n_recent, n_recent, C, bs, 0, G, d)
    P, T = 30, 400
    K = rng.standard_normal((P, d)).astype(np.float32)
    u.prefill(K, K)
    for t in range(T):
        q = rng.standard_normal((G, d)).astype(np.float32)
        kv = rng.standard_normal(d).astype(np.float32)
        u.step(q, kv, kv)
        pos = u.positions()
        p = P + t
        assert set(range(min(n_sink, p + 1))) <= set(pos.tolist())  # sinks stay
        assert set(range(max(0, p - n_recent + 1), p + 1)) <= set(pos.tolist())  # the recent window stays
        for blk in _blocks(pos, bs):  # a run of consecutive positions, then empty slots
            live = blk[blk >= 0]
            assert np.all(blk[:len(live)] >= 0) and np.all(np.diff(live) == 1)
    occ = u.positions() >= 0
    assert math.fsum(u.scores()[occ]) + u.evicted_mass == pytest.approx(T, rel=1e-12)


def test_invalid_block_configs_rejected():
    with pytest.raises(ValueError):
        Unit(H2O_BLOCK, 4, 50, 10, 64, 7, 0, 1, 8)   # budget not whole blocks
    with pytest.raises(ValueError):
        Unit(H2O_BLOCK, 4, 4, 40, 48, 16, 0, 1, 8)   # no block outside sinks and the recent window
    with pytest.raises(ValueError):
        Unit(H2O_BLOCK, 4, 50, 10, 65, 16, 0, 1, 8)  # parts do not add up to the budget
    with pytest.raises(ValueError):
        # 5 sinks occupy two blocks of 4, leaving one block (4 slots) outside them and
        # the recent window of 6: no block could ever be released
        Unit(H2O_BLOCK, 5, 5, 6, 16, 4, 0, 1, 8)
    Unit(H2O_BLOCK, 5, 7, 8, 20, 4, 0, 1, 8)  # blocks 2..4: two beyond the recent window of 8, accepted
