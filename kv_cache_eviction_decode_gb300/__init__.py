"""Decode step of attention over a budget-bounded KV cache with eviction (H2O,
StreamingLLM sink + window, Random Attention), hand-written CUDA for GB300
(sm_103a) behind a C ABI (include/kvevict.h, libkvevict.so)."""
from ._lib import (BF16, DEV_BAD_SLOT, DEV_NO_CANDIDATE, DEV_NONFINITE, DEV_WAIT_TIMEOUT, F32, H2O,  # noqa: F401
                   RANDOM, SINK_WINDOW, H2O_BLOCK, H2O_POOLS, KVEvictError, lib)
from .api import KVEvictCache  # noqa: F401
