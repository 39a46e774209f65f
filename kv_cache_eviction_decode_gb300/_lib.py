"""ctypes declarations of libkvevict.so (include/kvevict.h).

No fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvevict.so")

H2O, SINK_WINDOW, RANDOM, H2O_BLOCK, H2O_POOLS = 0, 1, 2, 3, 4
F32, BF16 = 0, 1

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_STATE, ERR_CUDA, ERR_DEVICE = 0, -1, -2, -3, -4, -5
DEV_NONFINITE, DEV_NO_CANDIDATE, DEV_WAIT_TIMEOUT, DEV_BAD_SLOT = 0x1, 0x2, 0x4, 0x8


class Config(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int), ("n_sink", ctypes.c_int), ("n_heavy", ctypes.c_int),
                ("n_recent", ctypes.c_int), ("budget", ctypes.c_int), ("r", ctypes.c_int),
                ("seed", ctypes.c_uint64), ("batch", ctypes.c_int), ("n_layers", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("max_prompt", ctypes.c_int), ("score_forget", ctypes.c_float),
                ("score_half", ctypes.c_int), ("hh_threshold", ctypes.c_float), ("score_int8", ctypes.c_int)]


class Stats(ctypes.Structure):
    _fields_ = [("decode_steps", ctypes.c_int64), ("prefill_tokens", ctypes.c_int64),
                ("evictions", ctypes.c_int64), ("cuts", ctypes.c_int64), ("split", ctypes.c_int),
                ("capacity", ctypes.c_int), ("clusters", ctypes.c_int), ("tensor_cores", ctypes.c_int),
                ("ring_stages", ctypes.c_int), ("tail_split", ctypes.c_int),
                ("partials_alias", ctypes.c_int), ("evicted_mass", ctypes.c_double),
                ("near_ties", ctypes.c_int64)]


class KVEvictError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            L.kvevict_state_bytes.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(SZ)]
            L.kvevict_create.argtypes = [ctypes.POINTER(P), ctypes.POINTER(Config), P, SZ, P]
            L.kvevict_prefill.argtypes = [P, I, P, P, I]
            L.kvevict_prefill_scored_workspace_bytes.argtypes = [P, I, ctypes.POINTER(SZ)]
            L.kvevict_prefill_scored.argtypes = [P, I, P, P, P, I, P, SZ]
            L.kvevict_prefill_scored_static.argtypes = [P, I, P, P, P, I]
            L.kvevict_prefill_snapkv_workspace_bytes.argtypes = [P, I, I, ctypes.POINTER(SZ)]
            L.kvevict_prefill_snapkv.argtypes = [P, I, P, P, P, I, I, I, P, SZ]
            L.kvevict_decode_step.argtypes = [P, I, P, P, P, P]
            L.kvevict_decode_step_host.argtypes = [P, I, P, P, P, P]
            L.kvevict_decode_step_host_async.argtypes = [P, I, P, P, P, P]
            L.kvevict_sync.argtypes = [P]
            L.kvevict_slot_positions.argtypes = [P, I, P, I]
            L.kvevict_scores.argtypes = [P, I, P, I]
            L.kvevict_slot_pools.argtypes = [P, I, P, I]
            L.kvevict_score_scales.argtypes = [P, I, P, I]
            L.kvevict_evicted_mass.argtypes = [P, I, P, I]
            L.kvevict_probe_wait_timeout.argtypes = [P]
            L.kvevict_select_victims.argtypes = [P, I, P, P]
            L.kvevict_checkpoint_bytes.argtypes = [P, ctypes.POINTER(SZ)]
            L.kvevict_checkpoint_save.argtypes = [P, P, SZ]
            L.kvevict_checkpoint_restore.argtypes = [P, P, SZ]
            L.kvevict_set_trace.argtypes = [P, I, P, I]
            L.kvevict_layer_state.argtypes = [P, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]
            L.kvevict_set_split.argtypes = [P, I]
            L.kvevict_set_clusters.argtypes = [P, I]
            L.kvevict_set_tail_split.argtypes = [P, I]
            L.kvevict_set_partials_alias.argtypes = [P, I]
            L.kvevict_set_tie_audit.argtypes = [P, I]
            L.kvevict_host_buffer_mapped.argtypes = [P]
            L.kvevict_near_ties.argtypes = [P, I, ctypes.POINTER(ctypes.c_uint64)]
            L.kvevict_set_path.argtypes = [P, I]
            L.kvevict_set_ring.argtypes = [P, I]
            L.kvevict_get_stats.argtypes = [P, ctypes.POINTER(Stats)]
            L.kvevict_check.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
            L.kvevict_strerror.argtypes = [I]
            L.kvevict_strerror.restype = ctypes.c_char_p
            L.kvevict_destroy.argtypes = [P]
            L.kvevict_destroy.restype = None
            for n in ("kvevict_state_bytes", "kvevict_create", "kvevict_prefill", "kvevict_prefill_scored_workspace_bytes",
                      "kvevict_prefill_scored", "kvevict_prefill_scored_static",
                      "kvevict_prefill_snapkv_workspace_bytes", "kvevict_prefill_snapkv", "kvevict_decode_step",
                      "kvevict_decode_step_host", "kvevict_decode_step_host_async", "kvevict_sync", "kvevict_slot_positions", "kvevict_scores", "kvevict_slot_pools",
                      "kvevict_score_scales", "kvevict_evicted_mass", "kvevict_probe_wait_timeout", "kvevict_select_victims", "kvevict_checkpoint_bytes",
                      "kvevict_checkpoint_save", "kvevict_checkpoint_restore",
                      "kvevict_set_trace",
                      "kvevict_layer_state", "kvevict_set_split", "kvevict_set_clusters", "kvevict_set_tail_split", "kvevict_set_partials_alias", "kvevict_set_tie_audit", "kvevict_near_ties", "kvevict_host_buffer_mapped", "kvevict_set_path", "kvevict_set_ring",
                      "kvevict_get_stats",
                      "kvevict_check"):
                getattr(L, n).restype = I
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().kvevict_strerror(code).decode()


def check(code: int, what: str) -> None:
    if code != OK:
        raise KVEvictError(code, what)
