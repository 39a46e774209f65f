"""Pins of the oracle's SnapKV selection ("Attention Sinks 与 KV Cache 淘汰策略",
section 4.3) to things other than itself: the votes against torch's fp64
scaled-dot-product attention with V = I (the attention rows themselves), the
pooling against torch's max_pool1d, the per-head top-k and the GQA union
against a sort, the window's mass (every query row sums to 1), an exact tie on
a pooling plateau (the newer positions stay) and the capacity check.
"""
import numpy as np
import pytest

from oracle import ECAPACITY, H2O, Unit


def _inputs(rng, G, w, P, d, scale=1.0):
    q = (rng.standard_normal((G, w, d)) * scale).astype(np.float32)
    k = (rng.standard_normal((P, d)) * scale).astype(np.float32)
    v = rng.standard_normal((P, d)).astype(np.float32)
    return q, k, v


def _sdpa_votes(q, k):
    """votes[g][j]: sum over the window rows of softmax(q k^T / sqrt(d)) with
    row t of the window at position P - w + t, from fp64 SDPA with V = I_P."""
    import torch
    import torch.nn.functional as F
    G, w, d = q.shape
    P = k.shape[0]
    qt = torch.from_numpy(q.astype(np.float64))[None]
    kt = torch.from_numpy(k.astype(np.float64))[None, None].expand(1, G, P, d)
    eye = torch.eye(P, dtype=torch.float64)[None, None].expand(1, G, P, P)
    rows = torch.arange(P - w, P)[:, None]
    mask = torch.arange(P)[None, :] <= rows  # [w][P], True = attend
    A = F.scaled_dot_product_attention(qt, kt, eye, attn_mask=mask)[0].numpy()  # [G][w][P]
    return A.sum(axis=1)


def _expected_kept(votes, P, w, topk):
    import torch
    import torch.nn.functional as F
    G = votes.shape[0]
    n_pre = P - w
    pooled = F.max_pool1d(torch.from_numpy(votes[:, :n_pre])[None], 7, stride=1, padding=3)[0].numpy()
    kept = set(range(n_pre, P))
    pos = np.arange(n_pre)
    for g in range(G):
        order = np.lexsort((-pos, -pooled[g]))  # largest pooled vote first, then the newer position
        kept |= set(order[:min(topk, n_pre)].tolist())
    return sorted(kept)


@pytest.mark.parametrize("G,w,P,d,topk", [(1, 8, 50, 16, 10), (4, 8, 90, 8, 12), (8, 32, 200, 16, 20),
                                          (2, 5, 12, 8, 30)])
def test_votes_pooling_topk_union(G, w, P, d, topk):
    rng = np.random.default_rng(500 + G * P)
    q, k, v = _inputs(rng, G, w, P, d)
    u = Unit(H2O, 2, P, 3, P + 5, 0, 0, G, d)
    votes = u.prefill_snapkv(q, k, v, topk)
    np.testing.assert_allclose(votes, _sdpa_votes(q, k), rtol=0, atol=1e-12)
    np.testing.assert_allclose(votes.sum(axis=1), w, rtol=1e-13)
    kept = _expected_kept(votes, P, w, topk)
    assert u.count == len(kept)
    np.testing.assert_array_equal(u.positions()[:u.count], kept)
    np.testing.assert_allclose(u.scores()[:u.count], votes.mean(axis=0)[kept], rtol=1e-14)
    kk, vv = u.slot_kv(u.count - 1)
    np.testing.assert_array_equal(kk, k[kept[-1]])
    np.testing.assert_array_equal(vv, v[kept[-1]])


def test_plateau_tie_keeps_the_newer():
    """One key aligned with every window query dominates the votes; max pooling
    spreads its vote over positions 17..23 exactly, and a top-5 cut inside
    that plateau keeps the five newest of them."""
    rng = np.random.default_rng(21)
    G, w, P, d = 1, 4, 40, 8
    qd = rng.standard_normal(d)
    qd /= np.linalg.norm(qd)
    q = np.tile(qd * 3.0, (G, w, 1)).astype(np.float32)
    k = (rng.standard_normal((P, d)) * 0.05).astype(np.float32)
    k[20] = (qd * 6.0).astype(np.float32)
    v = rng.standard_normal((P, d)).astype(np.float32)
    u = Unit(H2O, 2, P, 3, P + 5, 0, 0, G, d)
    votes = u.prefill_snapkv(q, k, v, 5)
    assert np.argmax(votes[0, :P - w]) == 20
    assert u.positions()[:u.count].tolist() == [19, 20, 21, 22, 23] + list(range(P - w, P))


def test_capacity_checked():
    rng = np.random.default_rng(4)
    G, w, P, d = 4, 4, 60, 8
    q, k, v = _inputs(rng, G, w, P, d)
    u = Unit(H2O, 1, 10, 3, 14, 0, 0, G, d)  # 14 slots: the union of four top-10 lists cannot fit
    with pytest.raises(RuntimeError, match=str(ECAPACITY)):
        u.prefill_snapkv(q, k, v, 10)


def test_pooling_stays_inside_the_prefix():
    """The first window key draws most of every window query's attention; the
    pooling window of the last prefix positions must not reach it, so the
    top-2 stay on the strongest prefix key's plateau (positions 7..13, the
    two newest kept)."""
    rng = np.random.default_rng(33)
    G, w, P, d = 1, 4, 30, 8
    qd = rng.standard_normal(d)
    qd /= np.linalg.norm(qd)
    q = np.tile(qd * 3.0, (G, w, 1)).astype(np.float32)
    k = (rng.standard_normal((P, d)) * 0.05).astype(np.float32)
    k[10] = (qd * 3.0).astype(np.float32)
    k[P - w] = (qd * 8.0).astype(np.float32)
    v = rng.standard_normal((P, d)).astype(np.float32)
    u = Unit(H2O, 2, P, 3, P + 5, 0, 0, G, d)
    votes = u.prefill_snapkv(q, k, v, 2)
    assert votes[0, P - w] > votes[0, 10] > np.delete(votes[0, :P - w], 10).max()
    assert u.positions()[:u.count].tolist() == [12, 13] + list(range(P - w, P))
