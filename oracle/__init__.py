"""CPU oracle for decode over a budget-bounded KV cache with eviction.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The product path never
imports this package, and this package never imports the product package.

The arithmetic lives in ``kvevict_oracle.c`` (plain C, fp64, one unit at a
time, literal step order). This module compiles it with gcc on first use and
marshals arguments through ctypes; it adds no arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvevict_oracle.c")
_LIB = os.path.join(_HERE, "liborc_kvevict.so")

H2O, SINK_WINDOW, RANDOM, H2O_BLOCK, H2O_POOLS = 0, 1, 2, 3, 4
OK, EINVAL, ECAPACITY, ESTATE = 0, -1, -2, -3

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, U64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_double
            L.orc_new.restype = P
            L.orc_new.argtypes = [I, I, I, I, I, I, I, I, I, U64, I, I, I]
            L.orc_free.argtypes = [P]
            for name in ("orc_capacity", "orc_steps", "orc_prompt_len", "orc_cuts", "orc_count",
                         "orc_greedy_disagreements"):
                getattr(L, name).argtypes = [P]
                getattr(L, name).restype = I
            L.orc_last_victim_pos.argtypes = [P]
            L.orc_last_block.argtypes = [P]
            L.orc_last_block.restype = I
            L.orc_last_victim_pos.restype = ctypes.c_int32
            L.orc_evicted_mass.argtypes = [P]
            L.orc_evicted_mass.restype = D
            L.orc_new_score.argtypes = [P]
            L.orc_new_score.restype = D
            L.orc_pos_at.argtypes = [P, I]
            L.orc_pos_at.restype = ctypes.c_int32
            L.orc_positions.argtypes = [P, P]
            L.orc_scores.argtypes = [P, P]
            L.orc_slot_kv.argtypes = [P, I, P, P]
            L.orc_attend.argtypes = [P, P, P, P, P]
            L.orc_attend.restype = I
            L.orc_stage.argtypes = [P, P, P]
            L.orc_stage.restype = I
            L.orc_choose.argtypes = [P]
            L.orc_choose.restype = I
            L.orc_commit.argtypes = [P, I]
            L.orc_commit.restype = I
            L.orc_prefill.argtypes = [P, P, P, I]
            L.orc_prefill.restype = I
            L.orc_prefill_scored.argtypes = [P, P, P, P, I, P]
            L.orc_prefill_scored.restype = I
            L.orc_prefill_snapkv.argtypes = [P, P, P, P, I, I, I, P]
            L.orc_prefill_snapkv.restype = I
            L.orc_prompt_tail_scores.argtypes = [P, P, I, I, I, I, P]
            L.orc_prompt_tail_scores.restype = I
            L.orc_set_score_storage.argtypes = [P, ctypes.c_double, I]
            L.orc_set_score_storage.restype = I
            L.orc_set_score_int8.argtypes = [P, I]
            L.orc_set_score_int8.restype = I
            L.orc_score_scale.argtypes = [P]
            L.orc_score_scale.restype = ctypes.c_double
            L.orc_int8_unrounded.argtypes = [P, P, P]
            L.orc_adopt_int8_code.argtypes = [P, I, I]
            L.orc_adopt_int8_code.restype = I
            L.orc_set_scores.argtypes = [P, P, ctypes.c_double]
            L.orc_set_scores.restype = I
            L.orc_score_codes.argtypes = [P, P]
            L.orc_set_hh_threshold.argtypes = [P, ctypes.c_double]
            L.orc_set_hh_threshold.restype = I
            L.orc_pools.argtypes = [P, P]
            L.orc_last_promote.argtypes = [P]
            L.orc_last_promote.restype = I
            L.orc_decision_margin.argtypes = [P]
            L.orc_decision_margin.restype = D
            L.orc_decision.argtypes = [P, P]
            L.orc_commit_pools.argtypes = [P, I, I, I]
            L.orc_commit_pools.restype = I
            L.orc_round_half.argtypes = [ctypes.c_double]
            L.orc_round_half.restype = ctypes.c_double
            L.orc_step.argtypes = [P, P, P, P, P]
            L.orc_step.restype = I
            L.orc_run.argtypes = [P, I, I, P, P, P, P, I]
            L.orc_run.restype = I
            L.orc_online_cores.restype = I
            L.orc_philox4x64_10.argtypes = [P, P, P]
            L.orc_random_key.argtypes = [U64, I, I, I, I, I]
            L.orc_random_key.restype = U64
            _lib = L
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Unit:
    """One (sequence, layer, KV head) cache held by the oracle."""

    def __init__(self, policy: int, n_sink: int, n_heavy: int, n_recent: int, budget: int, r: int,
                 max_prompt: int, group: int, head_dim: int, seed: int = 0, seq: int = 0, layer: int = 0,
                 head: int = 0):
        self._L = lib()
        self.h = self._L.orc_new(policy, n_sink, n_heavy, n_recent, budget, r, max_prompt, group, head_dim,
                                 seed, seq, layer, head)
        if not self.h:
            raise ValueError("oracle: invalid unit configuration")
        self.policy, self.G, self.d = policy, group, head_dim
        self.cap = self._L.orc_capacity(self.h)

    @classmethod
    def for_workload(cls, w, seq: int, layer: int, kv_head: int) -> "Unit":
        u = cls(w.policy, w.n_sink, w.n_heavy, w.n_recent, w.budget, w.r, w.max_prompt, w.group,
                w.head_dim, w.seed, seq, layer, kv_head)
        forget, half = getattr(w, "score_forget", 0.0), getattr(w, "score_half", False)
        if forget or half:
            u.set_score_storage(forget, half)
        if getattr(w, "score_int8", False):
            u.set_score_int8(True)
        if w.policy == H2O_POOLS:
            u.set_hh_threshold(w.hh_threshold)
        return u

    def __del__(self):
        h, self.h = getattr(self, "h", None), None
        if h:
            self._L.orc_free(h)

    # -- steps ---------------------------------------------------------------
    def prefill(self, k, v) -> None:
        k, v = _f32(k), _f32(v)
        rc = self._L.orc_prefill(self.h, _ptr(k), _ptr(v), k.shape[0])
        if rc:
            raise RuntimeError(f"oracle prefill failed: {rc}")

    def set_score_storage(self, forget: float = 0.0, half: bool = False) -> None:
        rc = self._L.orc_set_score_storage(self.h, forget, 1 if half else 0)
        if rc:
            raise RuntimeError(f"oracle set_score_storage failed: {rc}")

    def set_score_int8(self, on: bool = True) -> None:
        """INT8 score storage: per unit, codes round(s * 255 / max) times max / 255."""
        rc = self._L.orc_set_score_int8(self.h, 1 if on else 0)
        if rc:
            raise RuntimeError(f"oracle set_score_int8 failed: {rc}")

    def score_scale(self) -> float:
        """INT8 storage: the unit's scale (its largest score / 255)."""
        return float(self._L.orc_score_scale(self.h))

    def int8_unrounded(self):
        """INT8 storage: every slot's s * 255 / max before the last rounding
        (0 for empty slots), and the pending new token's."""
        a = np.empty(self.cap, dtype=np.float64)
        x_new = ctypes.c_double(0.0)
        self._L.orc_int8_unrounded(self.h, _ptr(a), ctypes.byref(x_new))
        return a, x_new.value

    def adopt_int8_code(self, slot: int, code: int) -> None:
        """Test hook: the token in `slot` (slot == capacity: the pending new
        token) takes `code`, one code from its own (a midpoint rounded apart)."""
        rc = self._L.orc_adopt_int8_code(self.h, int(slot), int(code))
        if rc:
            raise RuntimeError(f"oracle adopt_int8_code failed: {rc}")

    def set_scores(self, scores, new_score: float) -> None:
        """Test hook: replaces the retained tokens' stored scores (per slot)
        and the pending new token's; the next choose() decides on them."""
        a = np.ascontiguousarray(scores, dtype=np.float64)
        if a.shape != (self.cap,):
            raise ValueError("oracle set_scores: one score per slot")
        rc = self._L.orc_set_scores(self.h, _ptr(a), float(new_score))
        if rc:
            raise RuntimeError(f"oracle set_scores failed: {rc}")

    def score_codes(self) -> np.ndarray:
        """INT8 storage: the code of every slot (0 for empty slots)."""
        a = np.empty(self.cap, dtype=np.uint8)
        self._L.orc_score_codes(self.h, _ptr(a))
        return a

    def set_hh_threshold(self, theta: float) -> None:
        """Two-pool H2O: promotion needs a score strictly above theta."""
        rc = self._L.orc_set_hh_threshold(self.h, float(theta))
        if rc:
            raise RuntimeError(f"oracle set_hh_threshold failed: {rc}")

    def prefill_scored(self, q, k, v) -> np.ndarray:
        """Q-seeded prefill of an empty H2O unit: q [G][P][d], k/v [P][d].
        Returns the P prompt scores (before the cut to the budget)."""
        q, k, v = _f32(q), _f32(k), _f32(v)
        P = k.shape[0]
        if q.shape != (self.G, P, self.d) or v.shape != k.shape:
            raise ValueError("oracle prefill_scored: q must be [G][P][d], k and v [P][d]")
        scores = np.empty(P, dtype=np.float64)
        rc = self._L.orc_prefill_scored(self.h, _ptr(q), _ptr(k), _ptr(v), P, _ptr(scores))
        if rc:
            raise RuntimeError(f"oracle prefill_scored failed: {rc}")
        return scores

    def prefill_snapkv(self, q_obs, k, v, topk: int) -> np.ndarray:
        """SnapKV selection on an empty H2O unit: q_obs [G][w][d] (the last w
        prompt tokens' queries), k/v [P][d]. Returns the votes [G][P]."""
        q_obs, k, v = _f32(q_obs), _f32(k), _f32(v)
        P, w = k.shape[0], q_obs.shape[1]
        if q_obs.shape != (self.G, w, self.d) or v.shape != k.shape:
            raise ValueError("oracle prefill_snapkv: q_obs must be [G][w][d], k and v [P][d]")
        votes = np.empty((self.G, P), dtype=np.float64)
        rc = self._L.orc_prefill_snapkv(self.h, _ptr(q_obs), _ptr(k), _ptr(v), P, w, topk, _ptr(votes))
        if rc:
            raise RuntimeError(f"oracle prefill_snapkv failed: {rc}")
        return votes

    def attend(self, q, k_new, v_new) -> np.ndarray:
        q, k, v = _f32(q), _f32(k_new), _f32(v_new)
        out = np.empty((self.G, self.d), dtype=np.float64)
        rc = self._L.orc_attend(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(out))
        if rc:
            raise RuntimeError(f"oracle attend failed: {rc}")
        return out

    def stage(self, k_new, v_new) -> None:
        """Stage a decode token without attention (sink-window and Random only)."""
        k, v = _f32(k_new), _f32(v_new)
        rc = self._L.orc_stage(self.h, _ptr(k), _ptr(v))
        if rc:
            raise RuntimeError(f"oracle stage failed: {rc}")

    def choose(self) -> int:
        s = self._L.orc_choose(self.h)
        if s < 0:
            raise RuntimeError(f"oracle choose failed: {s}")
        return s

    def commit(self, slot: int) -> None:
        rc = self._L.orc_commit(self.h, int(slot))
        if rc:
            raise RuntimeError(f"oracle commit failed: {rc}")

    def decision(self):
        """Two-pool H2O, after choose(): (slot or capacity, new token's pool,
        promoted slot or -1)."""
        a = (ctypes.c_int * 3)()
        self._L.orc_decision(self.h, a)
        return int(a[0]), int(a[1]), int(a[2])

    @property
    def decision_margin(self) -> float:
        """Smallest relative gap among the comparisons of the last choose()."""
        return self._L.orc_decision_margin(self.h)

    def commit_pools(self, slot: int, new_pool: int, promote: int) -> None:
        rc = self._L.orc_commit_pools(self.h, int(slot), int(new_pool), int(promote))
        if rc:
            raise RuntimeError(f"oracle commit_pools failed: {rc}")

    def step(self, q, k_new, v_new):
        out = self.attend(q, k_new, v_new)
        slot = self.choose()
        self.commit(slot)
        return out, slot

    # -- state ---------------------------------------------------------------
    def positions(self) -> np.ndarray:
        a = np.empty(self.cap, dtype=np.int32)
        self._L.orc_positions(self.h, _ptr(a))
        return a

    def pools(self) -> np.ndarray:
        """Two-pool H2O: 0 recent pool, 1 heavy-hitter pool (meaningful where a slot is held)."""
        a = np.empty(self.cap, dtype=np.int8)
        self._L.orc_pools(self.h, _ptr(a))
        return a

    @property
    def last_promote(self) -> int:
        """Promotion of the last commit: slot, -2 the new token itself, -1 none."""
        return self._L.orc_last_promote(self.h)

    def pos_at(self, slot: int) -> int:
        return int(self._L.orc_pos_at(self.h, int(slot)))

    def scores(self) -> np.ndarray:
        a = np.empty(self.cap, dtype=np.float64)
        self._L.orc_scores(self.h, _ptr(a))
        return a

    def slot_kv(self, slot: int):
        k = np.empty(self.d, dtype=np.float32)
        v = np.empty(self.d, dtype=np.float32)
        self._L.orc_slot_kv(self.h, int(slot), _ptr(k), _ptr(v))
        return k, v

    @property
    def steps(self) -> int:
        return self._L.orc_steps(self.h)

    @property
    def count(self) -> int:
        return self._L.orc_count(self.h)

    @property
    def cuts(self) -> int:
        return self._L.orc_cuts(self.h)

    @property
    def prompt_len(self) -> int:
        return self._L.orc_prompt_len(self.h)

    @property
    def evicted_mass(self) -> float:
        return self._L.orc_evicted_mass(self.h)

    @property
    def last_victim_pos(self) -> int:
        return self._L.orc_last_victim_pos(self.h)

    @property
    def new_score(self) -> float:
        return self._L.orc_new_score(self.h)

    @property
    def last_block(self) -> int:
        return self._L.orc_last_block(self.h)

    @property
    def greedy_disagreements(self) -> int:
        return self._L.orc_greedy_disagreements(self.h)


def run(units, q, k, v, n_threads: int = 0, keep_out: bool = False):
    """n_steps decode steps on each unit, units spread over threads.

    q: [n_units, n_steps, G, d]; k, v: [n_units, n_steps, d].
    """
    L = lib()
    q, k, v = _f32(q), _f32(k), _f32(v)
    n_units, n_steps = q.shape[0], q.shape[1]
    arr = (ctypes.c_void_p * n_units)(*[u.h for u in units])
    out = np.empty(q.shape, dtype=np.float64) if keep_out else None
    rc = L.orc_run(ctypes.cast(arr, ctypes.c_void_p), n_units, n_steps, _ptr(q), _ptr(k), _ptr(v),
                   _ptr(out) if keep_out else None, int(n_threads))
    if rc:
        raise RuntimeError(f"oracle run failed: {rc}")
    return out


def prompt_tail_scores(q, k, j0: int) -> np.ndarray:
    """Prompt scores of the keys j >= j0 (q [G][P][d], k [P][d]): the column
    sums over the rows i >= j of the causal softmax, mean over G."""
    q, k = _f32(q), _f32(k)
    G, P, d = q.shape
    if k.shape != (P, d):
        raise ValueError("prompt_tail_scores: k must be [P][d]")
    out = np.empty(P - j0, dtype=np.float64)
    rc = lib().orc_prompt_tail_scores(_ptr(q), _ptr(k), G, P, d, j0, _ptr(out))
    if rc:
        raise RuntimeError(f"oracle prompt_tail_scores failed: {rc}")
    return out


def round_half(x: float) -> float:
    """The oracle's binary16 rounding of a non-negative value."""
    return lib().orc_round_half(float(x))


def online_cores() -> int:
    return lib().orc_online_cores()


def philox4x64_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint64)
    kk = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.empty(4, dtype=np.uint64)
    lib().orc_philox4x64_10(_ptr(c), _ptr(kk), _ptr(out))
    return out


def random_key(seed: int, seq: int, layer: int, head: int, step: int, pos: int) -> int:
    return int(lib().orc_random_key(seed, seq, layer, head, step, pos))
