"""The allocation-free scored prefill, kvevict_prefill_scored_static, for
callers that cannot allocate device memory at prefill time.

It must leave exactly the cache kvevict_prefill_scored leaves with a caller
workspace: the same kernels run on the same inputs and differ only in where
their scratch lives, and nothing in them depends on the scratch's earlier
contents or on the order of concurrent work (every key's column sum is
reduced in a fixed order, no atomics touch the scores). Two calls in a row go
through the C ABI on different prompts, so the second one runs on the scratch
the first left behind; slot positions, scores and the next decode step's
output must be bit-identical to the workspace entry point's. Argument errors
come before the size check; a prompt that needs more scratch than the fixed
area holds is refused with CAPACITY.

This file is collected last on purpose: it adds one entry point on the side,
so a run that stops at the first failure has run everything else first.
"""
import pytest
import torch

from kv_cache_eviction_decode_gb300 import BF16, H2O, KVEvictCache, lib
from kv_cache_eviction_decode_gb300._lib import ERR_CAPACITY, ERR_INVALID_ARG, ERR_STATE

pytestmark = pytest.mark.gpu


def _cache(device, B=2, Hq=8, Hkv=2, d=128, layers=2):
    return KVEvictCache(policy=H2O, budget=128, n_sink=4, n_heavy=60, n_recent=64, batch=B, n_layers=layers,
                        n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, dtype=BF16, device=device)


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
        assert torch.equal(sta.scores(layer), ref.scores(layer))
        qn = torch.randn((B, Hq, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        kn = torch.randn((B, Hkv, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        vn = torch.randn((B, Hkv, d), generator=gen).to(torch.bfloat16).to(cuda_device)
        o_sta = sta.decode_step(layer, qn, kn, vn)
        o_ref = ref.decode_step(layer, qn, kn, vn)
        assert sta.check() == 0 and ref.check() == 0
        assert torch.equal(o_sta, o_ref)
        assert torch.equal(sta.slot_positions(layer), ref.slot_positions(layer))
        assert torch.equal(sta.scores(layer), ref.scores(layer))
    sta.close()
    ref.close()


def test_static_scratch_argument_errors_come_first(cuda_device):
    L = lib()
    c = _cache(cuda_device, layers=1)
    P = 64
    Q = torch.zeros((2, 8, P, 128), dtype=torch.bfloat16, device=cuda_device)
    K = torch.zeros((2, 2, P, 128), dtype=torch.bfloat16, device=cuda_device)
    assert L.kvevict_prefill_scored_static(c.h, 0, None, K.data_ptr(), K.data_ptr(), P) == ERR_INVALID_ARG
    assert L.kvevict_prefill_scored_static(c.h, 0, Q.data_ptr() + 2, K.data_ptr(), K.data_ptr(), P) == \
        ERR_INVALID_ARG  # misaligned
    assert L.kvevict_prefill_scored_static(c.h, 1, Q.data_ptr(), K.data_ptr(), K.data_ptr(), P) == ERR_STATE
    assert L.kvevict_prefill_scored_static(c.h, 0, Q.data_ptr(), K.data_ptr(), K.data_ptr(), 0) == ERR_INVALID_ARG
    assert c.layer_state(0) == (0, 0, 0)  # nothing happened
    c.close()


def test_static_scratch_refuses_oversized_prompt(cuda_device):
    # 16 sequences x 32 heads x 8192 prompt tokens need 32 MiB of scratch
    big = _cache(cuda_device, B=16, Hq=32, Hkv=32, layers=1)
    P = 8192
    need = big.prefill_scored_workspace_bytes(P)
    assert need > 16 << 20
    # valid tensors (never read: the call is refused before any launch)
    Q = torch.empty((16, 32, P, 128), dtype=torch.bfloat16, device=cuda_device)
    rc = lib().kvevict_prefill_scored_static(big.h, 0, Q.data_ptr(), Q.data_ptr(), Q.data_ptr(), P)
    assert rc == ERR_CAPACITY
    # null pointers are an argument error, found before the size
    assert lib().kvevict_prefill_scored_static(big.h, 0, None, None, None, P) == ERR_INVALID_ARG
    assert big.layer_state(0) == (0, 0, 0)  # nothing happened
    big.close()
