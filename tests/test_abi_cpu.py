"""The C ABI without a GPU: the library builds and loads, exports every
function include/kvevict.h declares, and validates configurations on the
host (kvevict_state_bytes launches nothing)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from kv_cache_eviction_decode_gb300 import build
    build.build()
    from kv_cache_eviction_decode_gb300 import _lib
    return _lib.lib()


def declared_functions():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            text = open(os.path.join(ROOT, "include", hdr)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(kvevict_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"kvevict_create", "kvevict_decode_step", "kvevict_prefill", "kvevict_slot_positions"} <= names
    for n in sorted(names):
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_internal_helpers_are_not_exported(L):
    """The helpers shared between the library's own translation units stay
    out of the C ABI."""
    for n in ("kvevict_handle_device", "kvevict_prefill_scored_check", "kvevict_static_scratch_address"):
        assert not hasattr(L, n), f"{n} is internal but exported"


def _cfg(**kw):
    from kv_cache_eviction_decode_gb300._lib import Config
    base = dict(policy=0, n_sink=4, n_heavy=60, n_recent=64, budget=128, r=0, seed=1, batch=2, n_layers=3,
                n_q_heads=8, n_kv_heads=8, head_dim=64, dtype=0, max_prompt=0)
    base.update(kw)
    return Config(**base)


def _bytes(L, c):
    n = ctypes.c_size_t(0)
    rc = L.kvevict_state_bytes(ctypes.byref(c), ctypes.byref(n))
    return rc, n.value


def test_state_bytes_counts_every_region(L):
    rc, n = _bytes(L, _cfg())
    assert rc == 0
    C, units, layers, d = 128, 2 * 8, 3, 64
    kv = 2 * layers * units * C * d * 4
    assert n >= kv + layers * units * C * 8  # + positions and scores
    rc, n_sw = _bytes(L, _cfg(policy=1, n_heavy=0, n_recent=124))
    assert rc == 0 and n_sw < n  # no score region
    rc, n_rnd = _bytes(L, _cfg(policy=2, n_sink=0, n_heavy=0, n_recent=0, budget=100, r=20, max_prompt=50))
    assert rc == 0 and n_rnd >= 2 * layers * units * (50 + 100 + 20) * d * 4


@pytest.mark.parametrize("bad", [
    dict(n_recent=0, budget=64),                       # H2O needs a recent window
    dict(budget=127),                                  # budget != sink + heavy + recent
    dict(policy=1, n_heavy=5, n_recent=119),           # sink-window has no heavy hitters
    dict(policy=2, n_sink=0, n_heavy=0, n_recent=0, r=0, max_prompt=10),   # Random needs r >= 1
    dict(policy=2, n_sink=0, n_heavy=0, n_recent=0, budget=8000, r=500),   # K + r beyond 8192
    dict(policy=7),
    dict(dtype=3),
    dict(head_dim=96),
    dict(n_q_heads=12),                                # G = 1.5
    dict(n_q_heads=8 * 16),                            # G = 16
    dict(batch=0),
    dict(n_layers=0),
])
def test_invalid_configs_rejected_on_host(L, bad):
    rc, _ = _bytes(L, _cfg(**bad))
    assert rc == -1


def test_null_handle_and_strerror(L):
    assert L.kvevict_decode_step(None, 0, None, None, None, None) == -1
    assert L.kvevict_prefill(None, 0, None, None, 0) == -1
    assert L.kvevict_check(None, None) == -1
    assert L.kvevict_state_bytes(None, None) == -1
    n = ctypes.c_size_t(0)
    assert L.kvevict_checkpoint_bytes(None, ctypes.byref(n)) == -1
    assert L.kvevict_checkpoint_save(None, None, 0) == -1
    assert L.kvevict_checkpoint_restore(None, None, 0) == -1
    assert L.kvevict_probe_wait_timeout(None) == -1
    assert L.kvevict_score_scales(None, 0, None, 0) == -1
    assert L.kvevict_select_victims(None, 0, None, None) == -1
    assert L.kvevict_set_tie_audit(None, 1) == -1
    assert L.kvevict_near_ties(None, 0, None) == -1
    assert L.kvevict_prefill_scored_static(None, 0, None, None, None, 1) == -1
    assert L.kvevict_strerror(0) == b"ok"
    assert L.kvevict_strerror(-2) == b"capacity exceeded"
    L.kvevict_destroy(None)


def test_create_rejects_bad_state_without_touching_the_gpu(L):
    c = _cfg()
    h = ctypes.c_void_p()
    assert L.kvevict_create(ctypes.byref(h), ctypes.byref(c), None, 0, None) == -1   # no state
    assert L.kvevict_create(ctypes.byref(h), ctypes.byref(c), ctypes.c_void_p(0x1001), 1 << 30, None) == -1  # misaligned
    assert L.kvevict_create(ctypes.byref(h), ctypes.byref(c), ctypes.c_void_p(0x1000), 16, None) == -2  # too small
    assert not h.value


@pytest.mark.parametrize("bad", [
    dict(policy=3, r=7),                                          # block H2O: budget not whole blocks
    dict(policy=3, r=0),                                          # block H2O: no block size
    dict(policy=3, n_sink=4, n_heavy=4, n_recent=120, r=16),      # no block outside sinks and the window
    dict(policy=4),                                               # two-pool H2O has no sinks
    dict(policy=4, n_sink=0, n_heavy=60, n_recent=64),            # pools do not add up to the budget
    dict(policy=4, n_sink=0, n_heavy=128, n_recent=0),            # an empty recent pool
    dict(policy=4, n_sink=0, n_heavy=64, n_recent=64, hh_threshold=float("nan")),
    dict(score_forget=1.0),                                       # the moving average needs forget < 1
    dict(score_forget=-0.1),
    dict(policy=1, n_heavy=0, n_recent=124, score_forget=0.1),    # StreamingLLM keeps no scores
    dict(policy=3, r=16, score_half=1),                           # binary16 scores: not block H2O
    dict(score_half=2),
    dict(score_int8=2),
    dict(score_int8=1, score_half=1),                             # INT8 or binary16, not both
    dict(policy=3, r=16, score_int8=1),                           # INT8 scores: plain H2O only
    dict(policy=4, n_sink=0, n_heavy=64, n_recent=64, score_int8=1),
    dict(policy=1, n_heavy=0, n_recent=124, score_int8=1),
])
def test_invalid_next_row_configs_rejected_on_host(L, bad):
    rc, _ = _bytes(L, _cfg(**bad))
    assert rc == -1


def test_state_bytes_of_the_next_rows(L):
    rc, n_h2o = _bytes(L, _cfg())
    assert rc == 0
    # binary16 scores: half the score region (within the 256-byte alignment of each region)
    rc, n_half = _bytes(L, _cfg(score_half=1))
    assert rc == 0 and n_h2o - n_half >= 3 * 16 * 128 * 2 - 2 * 256
    # two-pool H2O: a one-byte pool flag per slot on top of H2O's regions
    rc, n_pools = _bytes(L, _cfg(policy=4, n_sink=0, n_heavy=64, n_recent=64, hh_threshold=0.01))
    assert rc == 0 and n_pools - n_h2o >= 3 * 16 * 128
    # block H2O: a free list of r entries per unit
    rc, n_block = _bytes(L, _cfg(policy=3, r=16))
    assert rc == 0 and n_block - n_h2o >= 3 * 16 * 16 * 4
    # the moving average changes no layout
    rc, n_ema = _bytes(L, _cfg(score_forget=0.25))
    assert rc == 0 and n_ema == n_h2o
    # INT8 scores: a byte per slot instead of four, plus a 4-byte scale per unit
    rc, n_int8 = _bytes(L, _cfg(score_int8=1))
    assert rc == 0 and n_h2o - n_int8 >= 3 * 16 * 128 * 3 - 3 * 16 * 4 - 3 * 256
    rc, n_int8_ema = _bytes(L, _cfg(score_int8=1, score_forget=0.1))
    assert rc == 0 and n_int8_ema == n_int8
