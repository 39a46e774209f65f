"""Seeded synthetic Q/K/V for the decode workloads.

Both the CPU oracle and the CUDA path read the inputs this module makes; it
holds none of the method's arithmetic (no attention, no scores, no eviction,
no draw the method itself makes).

Recipe (one unit = one (sequence, layer, KV head)):
  * every value starts as a standard normal draw, from a numpy Philox stream
    keyed by (seed, kind, sequence, layer, head), one row of head_dim per
    position (K, V) or per decode step (Q);
  * hub positions: per (sequence, position), with probability 0.02, shared by
    all layers and heads; a hub key gets +4*u added, u one unit vector of
    head_dim drawn once from the seed, so heavy hitters emerge;
  * sink positions 0-3: the key is scaled by 3 (after the hub term);
  * bf16 workloads round the fp32 value to bf16 (round to nearest even); the
    arrays returned here hold those bf16 values exactly, as float32.

Host arrays are float32 and exact in the workload's dtype. The device window
generator (torch, for timing runs) follows the same recipe with torch's CUDA
generator; its values are not bit-identical to the host ones and are never
compared with the oracle.
"""
from __future__ import annotations

import numpy as np

from .configs import DTYPE_BF16, Workload

KIND_Q, KIND_K, KIND_V, KIND_HUB, KIND_U = 0, 1, 2, 3, 4
HUB_PROB = 0.02
HUB_GAIN = 4.0
SINK_GAIN = 3.0
N_SINK_POSITIONS = 4


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(np.random.SeedSequence([int(seed), *map(int, tags)])))


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest-even bf16, returned as float32 holding the bf16 value."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 holding bf16 values -> their uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def to_dtype(w: Workload, x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return round_to_bf16(x) if w.dtype == DTYPE_BF16 else x


def hub_vector(seed: int, d: int) -> np.ndarray:
    n = _rng(seed, KIND_U).standard_normal(d)
    return (n / np.linalg.norm(n)).astype(np.float32)


def hub_flags(seed: int, seq: int, n_pos: int) -> np.ndarray:
    return _rng(seed, KIND_HUB, seq).random(n_pos) < HUB_PROB


def _normal_rows(seed: int, kind: int, seq: int, layer: int, head: int, n: int, d: int) -> np.ndarray:
    return _rng(seed, kind, seq, layer, head).standard_normal((n, d), dtype=np.float32)


def keys(w: Workload, seq: int, layer: int, kv_head: int, n_pos: int) -> np.ndarray:
    """Keys for positions 0..n_pos-1 of one unit, [n_pos, d] float32."""
    k = _normal_rows(w.seed, KIND_K, seq, layer, kv_head, n_pos, w.head_dim)
    hub = hub_flags(w.seed, seq, n_pos)
    k = k + np.float32(HUB_GAIN) * hub_vector(w.seed, w.head_dim)[None, :] * hub[:, None].astype(np.float32)
    k[:N_SINK_POSITIONS] *= np.float32(SINK_GAIN)
    return to_dtype(w, k)


def values(w: Workload, seq: int, layer: int, kv_head: int, n_pos: int) -> np.ndarray:
    return to_dtype(w, _normal_rows(w.seed, KIND_V, seq, layer, kv_head, n_pos, w.head_dim))


def queries(w: Workload, seq: int, layer: int, kv_head: int, n_steps: int) -> np.ndarray:
    """Queries of the G query heads that share one KV head, [n_steps, G, d]."""
    G = w.group
    out = np.empty((n_steps, G, w.head_dim), dtype=np.float32)
    for g in range(G):
        out[:, g, :] = _normal_rows(w.seed, KIND_Q, seq, layer, kv_head * G + g, n_steps, w.head_dim)
    return to_dtype(w, out)


class UnitInputs:
    """All inputs of one (sequence, layer, KV head) unit.

    prompt_k, prompt_v: [P, d]; q: [T, G, d]; k_new, v_new: [T, d]. Decode
    step t is position prompt_len + t.
    """

    def __init__(self, w: Workload, seq: int, layer: int, kv_head: int, n_steps: int | None = None,
                 prompt_len: int | None = None):
        P = w.prompt_len if prompt_len is None else prompt_len
        T = w.decode_steps if n_steps is None else n_steps
        k = keys(w, seq, layer, kv_head, P + T)
        v = values(w, seq, layer, kv_head, P + T)
        self.prompt_k, self.prompt_v = k[:P], v[:P]
        self.k_new, self.v_new = k[P:], v[P:]
        self.q = queries(w, seq, layer, kv_head, T)
        self.seq, self.layer, self.kv_head = seq, layer, kv_head
        self.prompt_len, self.n_steps = P, T


# ----------------------------------------------------------------------------
# Device-side generation (timing runs only): same recipe, torch CUDA generator.
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def device_hub_vector(w: Workload, device):
    torch = _torch()
    return torch.from_numpy(hub_vector(w.seed, w.head_dim)).to(device)


def device_prompt(w: Workload, layer: int, device, prompt_len: int | None = None, gen=None):
    """Prompt K, V for one layer, [B, Hkv, P, d] in the workload dtype."""
    torch = _torch()
    P = w.prompt_len if prompt_len is None else prompt_len
    dt = torch.bfloat16 if w.dtype == DTYPE_BF16 else torch.float32
    if gen is None:
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 1000003 + layer)
    B, H, d = w.batch, w.n_kv_heads, w.head_dim
    u = device_hub_vector(w, device)
    K = torch.empty((B, H, P, d), dtype=dt, device=device)
    V = torch.empty((B, H, P, d), dtype=dt, device=device)
    for b in range(B):  # one sequence at a time keeps the fp32 temporaries small
        hub = (torch.rand((P,), generator=gen, device=device) < HUB_PROB).float()
        k = torch.randn((H, P, d), generator=gen, device=device)
        k += HUB_GAIN * hub[None, :, None] * u[None, None, :]
        k[:, :N_SINK_POSITIONS] *= SINK_GAIN
        K[b] = k.to(dt)
        V[b] = torch.randn((H, P, d), generator=gen, device=device).to(dt)
    return K, V


def device_prompt_queries(w: Workload, layer: int, device, prompt_len: int | None = None, gen=None):
    """Prompt queries for one layer, [B, Hq, P, d] in the workload dtype
    (seeded N(0, 1), like the decode queries)."""
    torch = _torch()
    P = w.prompt_len if prompt_len is None else prompt_len
    dt = torch.bfloat16 if w.dtype == DTYPE_BF16 else torch.float32
    if gen is None:
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 2000003 + layer)
    Q = torch.empty((w.batch, w.n_q_heads, P, w.head_dim), dtype=dt, device=device)
    for b in range(w.batch):
        Q[b] = torch.randn((w.n_q_heads, P, w.head_dim), generator=gen, device=device).to(dt)
    return Q


def device_window(w: Workload, start_pos: int, n_steps: int, device, gen=None):
    """Decode inputs for n_steps token-steps of all layers.

    Returns q [n_steps, L, B, Hq, d], k_new and v_new [n_steps, L, B, Hkv, d].
    """
    torch = _torch()
    dt = torch.bfloat16 if w.dtype == DTYPE_BF16 else torch.float32
    if gen is None:
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 7919 + start_pos)
    L, B, Hq, Hkv, d = w.n_layers, w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    u = device_hub_vector(w, device)
    q = torch.empty((n_steps, L, B, Hq, d), dtype=dt, device=device)
    kn = torch.empty((n_steps, L, B, Hkv, d), dtype=dt, device=device)
    vn = torch.empty((n_steps, L, B, Hkv, d), dtype=dt, device=device)
    pos = torch.arange(start_pos, start_pos + n_steps, device=device)
    for s in range(n_steps):
        hub = (torch.rand((B,), generator=gen, device=device) < HUB_PROB).float()
        q[s] = torch.randn((L, B, Hq, d), generator=gen, device=device).to(dt)
        k = torch.randn((L, B, Hkv, d), generator=gen, device=device)
        k += HUB_GAIN * hub[None, :, None, None] * u
        if int(pos[s]) < N_SINK_POSITIONS:
            k *= SINK_GAIN
        kn[s] = k.to(dt)
        vn[s] = torch.randn((L, B, Hkv, d), generator=gen, device=device).to(dt)
    return q, kn, vn
