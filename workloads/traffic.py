"""Algorithmic byte counts for one decode step (the roofline numerator).

These count what the method itself has to move through HBM per unit (one
(sequence, layer, KV head)) per decode step, independent of any kernel:

  * K/V of every retained token plus the new token's K/V:  (n_ret + 1) * 2 * d * e
  * the new token's K/V written into its slot:            2 * d * e
  * the G queries read and the G outputs written:          2 * G * d * e
  * H2O: the cumulative scores read and written (fp32), the new token's
    score and position written:                            8 * n_ret + 8
    (binary16 scores: 4 * n_ret + 6; INT8 codes: 2 * n_ret + 9, the
    unit's scale read and written)
  * two-pool H2O: as H2O, plus the pool flags read and the
    new token's and a promoted token's flags written:      n_ret + 2
  * Random: the slot-position table read to skip holes:   4 * n_slots
    and, on a cut step, the generated tokens' positions read and the freed
    slots written:                                         4 * (K + r) + 4 * r

KV cache size (the pages' sizing formula): 2 (K and V) * layers * KV heads *
head_dim * bytes per element * tokens.
"""
from __future__ import annotations

from .configs import POLICY_H2O, POLICY_H2O_BLOCK, POLICY_H2O_POOLS, POLICY_RANDOM, Workload


def kv_cache_bytes(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int, tokens: int) -> int:
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes * tokens


def score_bytes(tokens: int, score_elem_bytes: int = 4) -> int:
    return tokens * score_elem_bytes


def unit_step_bytes(w: Workload, n_retained: int, n_slots: int | None = None, cut: bool = False) -> int:
    d, e, G = w.head_dim, w.elem_bytes, w.group
    b = (n_retained + 1) * 2 * d * e + 2 * d * e + 2 * G * d * e
    if w.policy in (POLICY_H2O, POLICY_H2O_BLOCK, POLICY_H2O_POOLS):
        if w.score_int8:  # codes read and written, the new token's code, the unit's scale read and written
            b += 2 * n_retained + 9
        else:
            b += (4 if w.score_half else 8) * n_retained + (6 if w.score_half else 8)
    if w.policy == POLICY_H2O_POOLS:
        b += n_retained + 2
    if w.policy == POLICY_RANDOM:
        b += 4 * (n_slots if n_slots is not None else w.capacity)
        if cut:
            b += 4 * (w.budget + w.r) + 4 * w.r
    return b


def steady_layer_step_bytes(w: Workload) -> int:
    """Bytes of one layer-step over all B * Hkv units once the cache is full."""
    units = w.batch * w.n_kv_heads
    if w.policy == POLICY_RANDOM:
        # generated count cycles K .. K+r-1 before each step's insert; mean K + (r-1)/2
        n_ret = w.prompt_len + w.budget + (w.r - 1) / 2.0
        per = unit_step_bytes(w, int(round(n_ret)), w.prompt_len + w.budget + w.r)
        cut_extra = (4 * (w.budget + w.r) + 4 * w.r) / w.r
        return int(units * (per + cut_extra))
    if w.policy == POLICY_H2O_BLOCK:
        # a release every r steps empties a block of r slots that the next r
        # tokens refill: on average C - (r + 1) / 2 tokens are attended; the
        # release reads every slot's position and score and writes r slots
        # (position, score, zeroed K/V rows, free-list entry)
        bs, d, e = w.r, w.head_dim, w.elem_bytes
        n_ret = w.capacity - (bs + 1) / 2.0
        release = 8 * w.capacity + bs * (8 + 2 * d * e + 4)
        return int(units * (unit_step_bytes(w, int(round(n_ret))) + release / bs))
    return units * unit_step_bytes(w, w.capacity)
