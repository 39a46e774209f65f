"""Python binding of libkvevict.so: argument marshalling only.

PyTorch supplies device memory (the handle's state buffer) and the CUDA
stream; every step of the decode path runs in the library's kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import BF16, F32, H2O, RANDOM, SINK_WINDOW, Config, Stats, check, lib

_DT = {F32: torch.float32, BF16: torch.bfloat16}


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


class KVEvictCache:
    """KV cache of n_layers x batch x n_kv_heads units with budget-bounded eviction."""

    def __init__(self, *, policy: int, budget: int, batch: int, n_layers: int, n_q_heads: int, n_kv_heads: int,
                 head_dim: int, dtype: int, n_sink: int = 0, n_heavy: int = 0, n_recent: int = 0, r: int = 0,
                 seed: int = 0, max_prompt: int = 0, score_forget: float = 0.0, score_half: bool = False,
                 hh_threshold: float = 0.0, score_int8: bool = False, device=None,
                 stream: torch.cuda.Stream | None = None):
        self._L = lib()
        self.cfg = Config(policy, n_sink, n_heavy, n_recent, budget, r, seed, batch, n_layers, n_q_heads,
                          n_kv_heads, head_dim, dtype, max_prompt, score_forget, 1 if score_half else 0,
                          hh_threshold, 1 if score_int8 else 0)
        nbytes = ctypes.c_size_t(0)
        check(self._L.kvevict_state_bytes(ctypes.byref(self.cfg), ctypes.byref(nbytes)), "kvevict_state_bytes")
        self.device = torch.device(device if device is not None else "cuda")
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.state = torch.empty(nbytes.value, dtype=torch.uint8, device=self.device)
        self.h = ctypes.c_void_p()
        check(self._L.kvevict_create(ctypes.byref(self.h), ctypes.byref(self.cfg), _ptr(self.state), nbytes.value,
                                     self.stream.cuda_stream), "kvevict_create")
        self.dtype = _DT[dtype]
        self.B, self.L, self.Hq, self.Hkv, self.D = batch, n_layers, n_q_heads, n_kv_heads, head_dim
        self.capacity = self.stats()["capacity"]
        self._trace = {}

    @classmethod
    def from_workload(cls, w, device=None, stream=None) -> "KVEvictCache":
        return cls(policy=w.policy, n_sink=w.n_sink, n_heavy=w.n_heavy, n_recent=w.n_recent, budget=w.budget,
                   r=w.r, seed=w.seed, batch=w.batch, n_layers=w.n_layers, n_q_heads=w.n_q_heads,
                   n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, dtype=w.dtype, max_prompt=w.max_prompt,
                   score_forget=getattr(w, "score_forget", 0.0), score_half=getattr(w, "score_half", False),
                   hh_threshold=getattr(w, "hh_threshold", 0.0), score_int8=getattr(w, "score_int8", False),
                   device=device, stream=stream)

    def close(self) -> None:
        if getattr(self, "h", None) and self.h.value:
            self._L.kvevict_destroy(self.h)
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- checks
    def _dev(self, t: torch.Tensor, shape, name: str, dtype=None) -> torch.Tensor:
        dtype = self.dtype if dtype is None else dtype
        if t.device != self.device or t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: need a contiguous {dtype} tensor of shape {tuple(shape)} on {self.device}, "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")
        return t

    def _host(self, t: torch.Tensor, shape, name: str) -> torch.Tensor:
        if t.device.type != "cpu" or t.dtype != self.dtype or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: need a contiguous CPU {self.dtype} tensor of shape {tuple(shape)}")
        return t

    # ----------------------------------------------------------------- steps
    def prefill(self, layer: int, K: torch.Tensor, V: torch.Tensor) -> None:
        n = K.shape[2]
        shp = (self.B, self.Hkv, n, self.D)
        self._dev(K, shp, "K")
        self._dev(V, shp, "V")
        check(self._L.kvevict_prefill(self.h, layer, _ptr(K), _ptr(V), n), "kvevict_prefill")

    def prefill_scored_workspace_bytes(self, prompt_len: int) -> int:
        n = ctypes.c_size_t()
        check(self._L.kvevict_prefill_scored_workspace_bytes(self.h, prompt_len, ctypes.byref(n)),
              "kvevict_prefill_scored_workspace_bytes")
        return n.value

    def prefill_scored(self, layer: int, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                       workspace: torch.Tensor | None = None) -> torch.Tensor:
        """Q-seeded prefill of an empty H2O layer: Q [B][Hq][P][d], K/V [B][Hkv][P][d].
        Returns the prompt scores before the cut, [B][Hkv][P] fp32: a view of
        the workspace, valid once the stream has passed the call."""
        n = K.shape[2]
        self._dev(Q, (self.B, self.Hq, n, self.D), "Q")
        self._dev(K, (self.B, self.Hkv, n, self.D), "K")
        self._dev(V, (self.B, self.Hkv, n, self.D), "V")
        need = self.prefill_scored_workspace_bytes(n)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        if workspace.device != self.device or workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace: need {need} bytes on {self.device}")
        check(self._L.kvevict_prefill_scored(self.h, layer, _ptr(Q), _ptr(K), _ptr(V), n, _ptr(workspace),
                                             workspace.numel() * workspace.element_size()),
              "kvevict_prefill_scored")
        ps = (n + 127) // 128 * 128
        off = (self.B * self.Hq * ps * 4 + 255) // 256 * 256
        raw = workspace.view(torch.uint8).reshape(-1)[off:off + self.B * self.Hkv * n * 4]
        return raw.view(torch.float32).view(self.B, self.Hkv, n)

    def prefill_snapkv_workspace_bytes(self, prompt_len: int, window: int) -> int:
        n = ctypes.c_size_t()
        check(self._L.kvevict_prefill_snapkv_workspace_bytes(self.h, prompt_len, window, ctypes.byref(n)),
              "kvevict_prefill_snapkv_workspace_bytes")
        return n.value

    def prefill_snapkv(self, layer: int, Q_obs: torch.Tensor, K: torch.Tensor, V: torch.Tensor, k_per_head: int,
                       workspace: torch.Tensor | None = None) -> torch.Tensor:
        """SnapKV prefill of an empty H2O layer: Q_obs [B][Hq][w][d] (the last w
        prompt tokens' queries), K/V [B][Hkv][P][d]. Returns the votes
        [B][Hq][P] fp32: a view of the workspace, valid once the stream has
        passed the call."""
        n, w = K.shape[2], Q_obs.shape[2]
        self._dev(Q_obs, (self.B, self.Hq, w, self.D), "Q_obs")
        self._dev(K, (self.B, self.Hkv, n, self.D), "K")
        self._dev(V, (self.B, self.Hkv, n, self.D), "V")
        need = self.prefill_snapkv_workspace_bytes(n, w)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        if workspace.device != self.device or workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace: need {need} bytes on {self.device}")
        check(self._L.kvevict_prefill_snapkv(self.h, layer, _ptr(Q_obs), _ptr(K), _ptr(V), n, w, k_per_head,
                                             _ptr(workspace), workspace.numel() * workspace.element_size()),
              "kvevict_prefill_snapkv")
        qs0 = (n - w) // 128 * 128
        ps = (n - qs0 + 127) // 128 * 128
        off = (self.B * self.Hq * ps * 4 + 255) // 256 * 256
        raw = workspace.view(torch.uint8).reshape(-1)[off:off + self.B * self.Hq * n * 4]
        return raw.view(torch.float32).view(self.B, self.Hq, n)

    def decode_step(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    out: torch.Tensor | None = None) -> torch.Tensor:
        self._dev(q, (self.B, self.Hq, self.D), "q")
        self._dev(k_new, (self.B, self.Hkv, self.D), "k_new")
        self._dev(v_new, (self.B, self.Hkv, self.D), "v_new")
        if out is None:
            out = torch.empty((self.B, self.Hq, self.D), dtype=self.dtype, device=self.device)
        self._dev(out, (self.B, self.Hq, self.D), "out")
        check(self._L.kvevict_decode_step(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)),
              "kvevict_decode_step")
        return out

    def decode_step_host(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                         out: torch.Tensor) -> torch.Tensor:
        self._host(q, (self.B, self.Hq, self.D), "q")
        self._host(k_new, (self.B, self.Hkv, self.D), "k_new")
        self._host(v_new, (self.B, self.Hkv, self.D), "v_new")
        self._host(out, (self.B, self.Hq, self.D), "out")
        check(self._L.kvevict_decode_step_host(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)),
              "kvevict_decode_step_host")
        return out

    def decode_step_host_async(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                               out: torch.Tensor) -> torch.Tensor:
        """decode_step_host without waiting: CPU tensors that must stay alive and
        unchanged until sync(); out holds the result after sync(). Pinned tensors
        the GPU can address are read and written in place by the kernels."""
        self._host(q, (self.B, self.Hq, self.D), "q")
        self._host(k_new, (self.B, self.Hkv, self.D), "k_new")
        self._host(v_new, (self.B, self.Hkv, self.D), "v_new")
        self._host(out, (self.B, self.Hq, self.D), "out")
        check(self._L.kvevict_decode_step_host_async(self.h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out)),
              "kvevict_decode_step_host_async")
        return out

    def sync(self) -> None:
        check(self._L.kvevict_sync(self.h), "kvevict_sync")

    # ----------------------------------------------------------------- state
    def slot_positions(self, layer: int, out: torch.Tensor | None = None) -> torch.Tensor:
        shp = (self.B, self.Hkv, self.capacity)
        if out is None:
            out = torch.empty(shp, dtype=torch.int32, device=self.device)
        on_dev = out.device.type == "cuda"
        if on_dev:
            self._dev(out, shp, "out", torch.int32)
        check(self._L.kvevict_slot_positions(self.h, layer, _ptr(out), 1 if on_dev else 0), "kvevict_slot_positions")
        return out

    def scores(self, layer: int, out: torch.Tensor | None = None) -> torch.Tensor:
        shp = (self.B, self.Hkv, self.capacity)
        if out is None:
            out = torch.empty(shp, dtype=torch.float32, device=self.device)
        on_dev = out.device.type == "cuda"
        if on_dev:
            self._dev(out, shp, "out", torch.float32)
        check(self._L.kvevict_scores(self.h, layer, _ptr(out), 1 if on_dev else 0), "kvevict_scores")
        return out

    def select_victims(self, layer: int, scores: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
        """H2O: the slot the layer's next decode step would evict per unit with
        these fp32 scores [batch][n_kv_heads][C] (-1: no candidate)."""
        self._dev(scores, (self.B, self.Hkv, self.capacity), "scores", torch.float32)
        if out is None:
            out = torch.empty((self.B, self.Hkv), dtype=torch.int32, device=self.device)
        self._dev(out, (self.B, self.Hkv), "out", torch.int32)
        check(self._L.kvevict_select_victims(self.h, layer, _ptr(scores), _ptr(out)), "kvevict_select_victims")
        return out

    def checkpoint(self) -> dict:
        """The handle's host record and a device copy of its state buffer,
        taken once every queued call has run."""
        n = ctypes.c_size_t(0)
        check(self._L.kvevict_checkpoint_bytes(self.h, ctypes.byref(n)), "kvevict_checkpoint_bytes")
        rec = (ctypes.c_uint8 * n.value)()
        check(self._L.kvevict_checkpoint_save(self.h, rec, n.value), "kvevict_checkpoint_save")
        self.stream.synchronize()
        with torch.cuda.stream(self.stream):
            state = self.state.clone()
        self.stream.synchronize()
        return {"record": bytes(rec), "state": state}

    def restore(self, ckpt: dict) -> None:
        """Resumes from checkpoint(): the saved state bytes into this handle's
        buffer, then its host record (same configuration required)."""
        if ckpt["state"].numel() != self.state.numel():
            raise ValueError("checkpoint state size differs from this handle's")
        self.stream.synchronize()
        with torch.cuda.stream(self.stream):
            self.state.copy_(ckpt["state"])
        self.stream.synchronize()
        rec = ckpt["record"]
        buf = (ctypes.c_uint8 * len(rec)).from_buffer_copy(rec)
        check(self._L.kvevict_checkpoint_restore(self.h, buf, len(rec)), "kvevict_checkpoint_restore")

    def probe_wait_timeout(self) -> None:
        """Queues the failure-detection probe: a bounded wait that runs out and
        sets DEV_WAIT_TIMEOUT in the error word (read by check())."""
        check(self._L.kvevict_probe_wait_timeout(self.h), "kvevict_probe_wait_timeout")

    def evicted_mass(self, layer: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """Every unit's evicted score mass (fp64, [batch][n_kv_heads])."""
        shp = (self.B, self.Hkv)
        if out is None:
            out = torch.empty(shp, dtype=torch.float64, device=self.device)
        on_dev = out.device.type == "cuda"
        if on_dev:
            self._dev(out, shp, "out", torch.float64)
        check(self._L.kvevict_evicted_mass(self.h, layer, _ptr(out), 1 if on_dev else 0), "kvevict_evicted_mass")
        return out

    def score_scales(self, layer: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """INT8 score storage: every unit's scale (its largest score / 255)."""
        shp = (self.B, self.Hkv)
        if out is None:
            out = torch.empty(shp, dtype=torch.float32, device=self.device)
        on_dev = out.device.type == "cuda"
        if on_dev:
            self._dev(out, shp, "out", torch.float32)
        check(self._L.kvevict_score_scales(self.h, layer, _ptr(out), 1 if on_dev else 0), "kvevict_score_scales")
        return out

    def pools(self, layer: int, out: torch.Tensor | None = None) -> torch.Tensor:
        """Two-pool H2O: 0 recent pool, 1 heavy-hitter pool per slot (where a token is held)."""
        shp = (self.B, self.Hkv, self.capacity)
        if out is None:
            out = torch.empty(shp, dtype=torch.uint8, device=self.device)
        on_dev = out.device.type == "cuda"
        if on_dev:
            self._dev(out, shp, "out", torch.uint8)
        check(self._L.kvevict_slot_pools(self.h, layer, _ptr(out), 1 if on_dev else 0), "kvevict_slot_pools")
        return out

    def set_trace(self, layer: int, buf: torch.Tensor | None) -> None:
        if buf is None:
            check(self._L.kvevict_set_trace(self.h, layer, None, 0), "kvevict_set_trace")
            self._trace.pop(layer, None)
            return
        if buf.dtype != torch.int32 or buf.device != self.device or not buf.is_contiguous() or \
                tuple(buf.shape[1:]) != (self.B, self.Hkv, 4):
            raise ValueError("trace buffer: contiguous int32 [n_steps, batch, n_kv_heads, 4] on the device")
        self._trace[layer] = buf  # keep it alive while the library writes it
        check(self._L.kvevict_set_trace(self.h, layer, _ptr(buf), buf.shape[0]), "kvevict_set_trace")

    def layer_state(self, layer: int):
        a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        check(self._L.kvevict_layer_state(self.h, layer, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)),
              "kvevict_layer_state")
        return a.value, b.value, c.value

    def set_split(self, split: int) -> None:
        check(self._L.kvevict_set_split(self.h, split), "kvevict_set_split")

    def set_tail_split(self, on) -> None:
        """Clusters split only their leftover units; each CTA's others are whole
        (True / False, or -1 for automatic)."""
        mode = on if isinstance(on, int) and not isinstance(on, bool) else (1 if on else 0)
        check(self._L.kvevict_set_tail_split(self.h, mode), "kvevict_set_tail_split")

    def set_tie_audit(self, on: bool) -> None:
        """Validation mode: count the H2O decisions whose runner-up was within 1e-5
        relative of the evicted token's score (kvevict_stats.near_ties)."""
        check(self._L.kvevict_set_tie_audit(self.h, 1 if on else 0), "kvevict_set_tie_audit")

    def near_ties(self, layer: int) -> int:
        """This layer's near-tie count (validation mode)."""
        v = ctypes.c_uint64(0)
        check(self._L.kvevict_near_ties(self.h, layer, ctypes.byref(v)), "kvevict_near_ties")
        return v.value

    def set_partials_alias(self, mode: int) -> None:
        """-1 automatic, 0 own area, 1 the warps' partial outputs over the logits."""
        check(self._L.kvevict_set_partials_alias(self.h, mode), "kvevict_set_partials_alias")

    def set_path(self, path: int) -> None:
        """0 automatic, 1 CUDA cores, 2 tensor cores (bf16 only)."""
        check(self._L.kvevict_set_path(self.h, path), "kvevict_set_path")

    def set_ring(self, stages: int) -> None:
        check(self._L.kvevict_set_ring(self.h, stages), "kvevict_set_ring")

    def set_clusters(self, clusters: int) -> None:
        check(self._L.kvevict_set_clusters(self.h, clusters), "kvevict_set_clusters")

    def stats(self) -> dict:
        s = Stats()
        check(self._L.kvevict_get_stats(self.h, ctypes.byref(s)), "kvevict_get_stats")
        return {f: getattr(s, f) for f, _ in Stats._fields_}

    def check(self) -> int:
        """Waits for the stream; returns the device error word (0 = clean) and clears it."""
        w = ctypes.c_uint32(0)
        rc = self._L.kvevict_check(self.h, ctypes.byref(w))
        if rc not in (_lib.OK, _lib.ERR_DEVICE):
            check(rc, "kvevict_check")
        return w.value
