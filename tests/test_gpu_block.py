"""GPU parity of block-granular H2O ("Attention Sinks 与 KV Cache 淘汰策略" section
5: whole blocks are released), through the C ABI, against the CPU oracle.

The slot tables must agree exactly at every step: which block is released
(and so where every new token goes) depends on block sums of fp32 scores
that the tests keep far from ties. Attention outputs and scores as for H2O:
1e-4 max-abs for fp32, 2e-2 relative for bf16.
"""
import numpy as np
import pytest
import torch

import oracle
from kv_cache_eviction_decode_gb300 import BF16, F32, H2O_BLOCK, KVEvictCache
from tests import lockstep as ls
from workloads import configs

pytestmark = pytest.mark.gpu


def _err(dtype, got, ref):
    if dtype == BF16:
        return np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-6)
    return np.abs(got - ref).max()


@pytest.mark.parametrize("dtype,G,d,bs,P", [(F32, 2, 64, 8, 100), (BF16, 4, 128, 16, 70), (BF16, 1, 64, 4, 40),
                                            (BF16, 2, 128, 8, 64)])
def test_block_lockstep_small(cuda_device, dtype, G, d, bs, P):
    gen = torch.Generator().manual_seed(300 + G * bs + P)
    B, Hkv, C, n_sink, n_recent, T = 2, 2, 64, 4, 12, 160
    Hq = G * Hkv
    tdt = torch.float32 if dtype == F32 else torch.bfloat16
    tol = 1e-4 if dtype == F32 else 2e-2
    cache = KVEvictCache(policy=H2O_BLOCK, budget=C, n_sink=n_sink, n_heavy=C - n_sink - n_recent, n_recent=n_recent,
                         r=bs, batch=B, n_layers=1, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, dtype=dtype,
                         device=cuda_device)
    K = torch.randn((B, Hkv, P, d), generator=gen).to(tdt)
    V = torch.randn((B, Hkv, P, d), generator=gen).to(tdt)
    cache.prefill(0, K.to(cuda_device), V.to(cuda_device))
    units = {}
    for b in range(B):
        for h in range(Hkv):
            u = oracle.Unit(oracle.H2O_BLOCK, n_sink, C - n_sink - n_recent, n_recent, C, bs, 0, G, d)
            u.prefill(K[b, h].float().numpy(), V[b, h].float().numpy())
            units[(b, h)] = u
    pos = cache.slot_positions(0).cpu().numpy()
    for (b, h), u in units.items():
        np.testing.assert_array_equal(pos[b, h], u.positions(), err_msg="after prefill")
    releases = 0
    for t in range(T):
        q = (torch.randn((B, Hq, d), generator=gen) * 1.5).to(tdt)
        kn = torch.randn((B, Hkv, d), generator=gen).to(tdt)
        vn = torch.randn((B, Hkv, d), generator=gen).to(tdt)
        out = cache.decode_step(0, q.to(cuda_device), kn.to(cuda_device), vn.to(cuda_device)).float().cpu().numpy()
        pos = cache.slot_positions(0).cpu().numpy()
        sc = cache.scores(0).cpu().numpy() if t % 20 == 19 else None
        for (b, h), u in units.items():
            ref, _ = u.step(q[b, h * G:(h + 1) * G].float().numpy(), kn[b, h].float().numpy(),
                            vn[b, h].float().numpy())
            e = _err(dtype, out[b, h * G:(h + 1) * G], ref)
            assert e <= tol, (b, h, t, e)
            releases += u.last_block >= 0
            np.testing.assert_array_equal(pos[b, h], u.positions(), err_msg=f"unit {(b, h)} step {t}")
            if sc is not None:
                occ = pos[b, h] >= 0
                assert _err(dtype, sc[b, h][occ], u.scores()[occ]) <= tol
    assert cache.check() == 0
    assert releases >= 4 * ((T - (C - min(P, C))) // bs - 1)
    print(f"{releases} releases over {len(units)} units")


@pytest.mark.parametrize("name,steps", [("h2o_block16", 48), ("h2o_block256", 300)])
def test_block_full_shape(cuda_device, name, steps):
    """The MHA shape (B=16, 32 heads, d=128, 1024 slots, prompt 2048) with
    blocks of 16 and of 256: every unit runs on the GPU; the oracle replays
    sequences {0, 15} x every head in lockstep."""
    w = configs.get(name).with_(n_layers=1)
    units = [(s, 0, h) for s in (0, w.batch - 1) for h in range(w.n_kv_heads)]
    inputs = ls.host_inputs(w, units, steps, w.prompt_len)
    run = ls.run_gpu(w, [0], steps, inputs, w.prompt_len, cuda_device, snap_steps=range(0, steps, 8))
    assert run.err == 0
    reps = ls.replay_all(w, units, inputs, run, steps, out_steps=range(0, steps, 4))
    worst = max(r.max_out_err for r in reps)
    assert sum(r.near_ties for r in reps) == 0
    print(f"{name}: {len(units)} units x {steps} steps, max out err {worst:.2e}")
