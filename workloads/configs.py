"""Decode workloads for budget-bounded KV-cache eviction.

Each entry names one decode workload by what it is and its sizes. The
shapes follow the pages' own workloads: a Llama-2-7B-shaped MHA layer stack
(32 layers x 32 heads, head_dim 128), a Llama-2-70B-shaped GQA layer (64 query
heads over 8 KV heads), a long-reasoning trace with a kept prompt, and the
StreamingLLM sink + window cache ("Attention Sinks and KV-cache eviction",
section 4.1; "StreamingLLM and Heavy-Hitter", the layout diagram: 4 sink
tokens plus a rolling window, 1024 tokens in all).

This module holds sizes only: no arithmetic of the method lives here.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

POLICY_H2O = 0
POLICY_SINK_WINDOW = 1
POLICY_RANDOM = 2
POLICY_H2O_BLOCK = 3
POLICY_H2O_POOLS = 4

DTYPE_F32 = 0
DTYPE_BF16 = 1

POLICY_NAMES = {POLICY_H2O: "h2o", POLICY_SINK_WINDOW: "sink_window", POLICY_RANDOM: "random",
                POLICY_H2O_BLOCK: "h2o_block", POLICY_H2O_POOLS: "h2o_pools"}


@dataclass(frozen=True)
class Workload:
    name: str
    policy: int
    dtype: int
    batch: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_sink: int
    n_heavy: int
    n_recent: int
    budget: int
    r: int
    prompt_len: int
    decode_steps: int
    seed: int
    max_prompt: int = 0
    score_forget: float = 0.0  # H2O score storage: s <- (1 - score_forget) s + a
    score_half: bool = False   # H2O score storage: binary16
    score_int8: bool = False   # H2O score storage: 8-bit codes, one absmax scale per unit
    hh_threshold: float = 0.0  # two-pool H2O: promotion needs a score above this

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def capacity(self) -> int:
        """Slots per (sequence, layer, KV head)."""
        if self.policy == POLICY_RANDOM:
            return self.max_prompt + self.budget + self.r
        return self.budget

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == DTYPE_F32 else 2

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# H2O tiny, fp32: one layer, 8 MHA heads, head_dim 64, prompt 256 then 256
# decode steps; budget 128 = 4 sink + 60 heavy + 64 recent.
H2O_TINY = Workload(
    name="h2o_tiny_fp32_b1_h8_d64_k128", policy=POLICY_H2O, dtype=DTYPE_F32,
    batch=1, n_layers=1, n_q_heads=8, n_kv_heads=8, head_dim=64,
    n_sink=4, n_heavy=60, n_recent=64, budget=128, r=0,
    prompt_len=256, decode_steps=256, seed=1234)

# StreamingLLM sink + ring window, bf16: B=64, 32 layers x 32 heads, d=128;
# 16384 streamed tokens, cache 4 sink + 1020 window per head, no scores.
SINK_WINDOW = Workload(
    name="sink_window_bf16_b64_l32_h32_d128_k1024", policy=POLICY_SINK_WINDOW, dtype=DTYPE_BF16,
    batch=64, n_layers=32, n_q_heads=32, n_kv_heads=32, head_dim=128,
    n_sink=4, n_heavy=0, n_recent=1020, budget=1024, r=0,
    prompt_len=0, decode_steps=16384, seed=2026)

# H2O on a Llama-2-7B-shaped decode, bf16: B=16, 32 layers x 32 MHA heads,
# prompt 2048 then 2048 decode steps; budget 1024 = 4 + 510 + 510.
H2O_MHA = Workload(
    name="h2o_bf16_b16_l32_h32_d128_k1024", policy=POLICY_H2O, dtype=DTYPE_BF16,
    batch=16, n_layers=32, n_q_heads=32, n_kv_heads=32, head_dim=128,
    n_sink=4, n_heavy=510, n_recent=510, budget=1024, r=0,
    prompt_len=2048, decode_steps=2048, seed=2027)

# H2O on one Llama-2-70B-shaped GQA layer, bf16: 64 query heads over 8 KV
# heads, B=64, context 32768 then 512 decode steps; budget 2048 = 4 + 1020 + 1024;
# a KV head's score is the mean of its 8 query heads' probabilities.
H2O_GQA = Workload(
    name="h2o_gqa_bf16_b64_l1_hq64_hkv8_d128_k2048", policy=POLICY_H2O, dtype=DTYPE_BF16,
    batch=64, n_layers=1, n_q_heads=64, n_kv_heads=8, head_dim=128,
    n_sink=4, n_heavy=1020, n_recent=1024, budget=2048, r=0,
    prompt_len=32768, decode_steps=512, seed=2028)

# Random Attention on a long-reasoning trace, bf16: B=32, 32 layers x 8 KV
# heads (32 query heads); prompt 8192 always kept; every r=128 steps the
# reasoning tokens are cut per KV head back to K=2048 by uniform random choice.
RANDOM_REASONING = Workload(
    name="random_bf16_b32_l32_hq32_hkv8_d128_p8192_k2048_r128", policy=POLICY_RANDOM, dtype=DTYPE_BF16,
    batch=32, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
    n_sink=0, n_heavy=0, n_recent=0, budget=2048, r=128,
    prompt_len=8192, decode_steps=32768, seed=2029, max_prompt=8192)

# H2O scoring on the identical long-reasoning shape: the whole 8192-token
# prompt is protected (as Random protects it), plus 1024 heavy + 1024 recent.
H2O_REASONING = Workload(
    name="h2o_bf16_b32_l32_hq32_hkv8_d128_p8192_k10240", policy=POLICY_H2O, dtype=DTYPE_BF16,
    batch=32, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
    n_sink=8192, n_heavy=1024, n_recent=1024, budget=10240, r=0,
    prompt_len=8192, decode_steps=32768, seed=2029)

# Block-granular H2O on the MHA shape: blocks of 16 slots (a PagedAttention
# block) and of 256; r is the block size.
H2O_BLOCK16 = H2O_MHA.with_(name="h2o_block16_bf16_b16_l32_h32_d128_k1024", policy=POLICY_H2O_BLOCK, r=16)
H2O_BLOCK256 = H2O_MHA.with_(name="h2o_block256_bf16_b16_l32_h32_d128_k1024", policy=POLICY_H2O_BLOCK, r=256)

# H2O on the MHA shape with the scores stored in binary16 (half the score
# traffic), and with a moving average (forget 0.01 per step) in place of the sum.
H2O_MHA_FP16 = H2O_MHA.with_(name="h2o_fp16scores_bf16_b16_l32_h32_d128_k1024", score_half=True)
H2O_MHA_EMA = H2O_MHA.with_(name="h2o_ema0.01_bf16_b16_l32_h32_d128_k1024", score_forget=0.01)
# ... and as 8-bit codes with one absmax scale per (sequence, KV head): a quarter of the score traffic.
H2O_MHA_INT8 = H2O_MHA.with_(name="h2o_int8scores_bf16_b16_l32_h32_d128_k1024", score_int8=True)

# Two-pool H2O on the MHA shape: a recent pool of 512 and a heavy-hitter pool of
# 512 (no sinks); a token leaving the recent pool is promoted if its score is
# above 2^-10, the share of one step's attention spread evenly over 1024 tokens.
H2O_POOLS_MHA = H2O_MHA.with_(name="h2o_pools_bf16_b16_l32_h32_d128_r512_hh512", policy=POLICY_H2O_POOLS, n_sink=0,
                              n_heavy=512, n_recent=512, hh_threshold=2.0**-10)

ALL = {w.name: w for w in (H2O_TINY, SINK_WINDOW, H2O_MHA, H2O_GQA, RANDOM_REASONING, H2O_REASONING, H2O_BLOCK16,
                           H2O_BLOCK256, H2O_MHA_FP16, H2O_MHA_EMA, H2O_MHA_INT8, H2O_POOLS_MHA)}

# Short names used on command lines.
ALIASES = {
    "h2o_tiny": H2O_TINY.name,
    "sink_window": SINK_WINDOW.name,
    "h2o_mha": H2O_MHA.name,
    "h2o_gqa": H2O_GQA.name,
    "random": RANDOM_REASONING.name,
    "h2o_reasoning": H2O_REASONING.name,
    "h2o_block16": H2O_BLOCK16.name,
    "h2o_block256": H2O_BLOCK256.name,
    "h2o_fp16scores": H2O_MHA_FP16.name,
    "h2o_ema": H2O_MHA_EMA.name,
    "h2o_int8scores": H2O_MHA_INT8.name,
    "h2o_pools": H2O_POOLS_MHA.name,
}


def get(name: str) -> Workload:
    return ALL[ALIASES.get(name, name)]
