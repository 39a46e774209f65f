"""The allocation-free scored prefill, kvevict_prefill_scored_static, for
callers that cannot allocate device memory at prefill time.

It must leave the same cache as kvevict_prefill_scored with a caller
workspace. Two calls in a row go through the C ABI on different prompts, so
the second one runs on the scratch the first left behind; each is compared
with the workspace entry point on the same inputs: slot positions exactly,
scores and the next decode step's output within the tolerances of the other
GPU tests (2e-3 and 2e-2 relative). A prompt that needs more scratch than the
fixed area holds is refused with CAPACITY.

This file is collected last on purpose: it adds one entry point on the side,
so a run that stops at the first failure has run everything else first.
"""
import numpy as np
import pytest
import torch

from kv_cache_eviction_decode_gb300 import BF16, H2O, KVEvictCache, lib
from kv_cache_eviction_decode_gb300._lib import ERR_CAPACITY

pytestmark = pytest.mark.gpu

SCORE_TOL = 2e-3
OUT_TOL = 2e-2


def _cache(device, B=2, Hq=8, Hkv=2, d=128, layers=2):
    return KVEvictCache(policy=H2O, budget=128, n_sink=4, n_heavy=60, n_recent=64, batch=B, n_layers=layers,
                        n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, dtype=BF16, device=device)


def _rel(a, b):
    a, b = a.float().cpu().numpy(), b.float().cpu().numpy()
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-6)


def test_static_scratch_matches_workspace_entry_point(cuda_device):
    L = lib()
    gen = torch.Generator().manual_seed(2024)
    ref, sta = _cache(cuda_device), _cache(cuda_device)
    B, Hq, Hkv, d = 2, 8, 2, 128
    for layer, P in enumerate((700, 333)):  # two calls in a row, different prompts
        Q = torch.randn((B, Hq, P, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        K = torch.randn((B, Hkv, P, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        V = torch.randn((B, Hkv, P, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        ref.prefill_scored(layer, Q, K, V)
        rc = L.kvevict_prefill_scored_static(sta.h, layer, Q.data_ptr(), K.data_ptr(), V.data_ptr(), P)
        assert rc == 0
        assert sta.check() == 0 and ref.check() == 0
        assert sta.layer_state(layer) == ref.layer_state(layer)
        assert torch.equal(sta.slot_positions(layer), ref.slot_positions(layer))
        assert _rel(sta.scores(layer), ref.scores(layer)) <= SCORE_TOL
        qn = torch.randn((B, Hq, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        kn = torch.randn((B, Hkv, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        vn = torch.randn((B, Hkv, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        o_sta = sta.decode_step(layer, qn, kn, vn)
        o_ref = ref.decode_step(layer, qn, kn, vn)
        assert sta.check() == 0 and ref.check() == 0
        assert _rel(o_sta, o_ref) <= OUT_TOL
        assert torch.equal(sta.slot_positions(layer), ref.slot_positions(layer))
    sta.close()
    ref.close()


def test_static_scratch_refuses_oversized_prompt(cuda_device):
    # 16 sequences x 32 heads x 8192 prompt tokens need 32 MiB of scratch
    big = _cache(cuda_device, B=16, Hq=32, Hkv=32, layers=1)
    need = big.prefill_scored_workspace_bytes(8192)
    assert need > 16 << 20
    rc = lib().kvevict_prefill_scored_static(big.h, 0, None, None, None, 8192)
    assert rc == ERR_CAPACITY
    assert big.layer_state(0) == (0, 0, 0)  # nothing happened
    big.close()
