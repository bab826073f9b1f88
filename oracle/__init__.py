"""Test infrastructure: the float64 CPU oracle.  Not part of the product path;
only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs use it."""
from .rkv_oracle import *  # noqa: F401,F403
from .rkv_oracle import (  # noqa: F401
    bf16_round, bookkeep, inv_freq, rope, softmax_attention, lse_merge,
    softmax_partial, RollingCacheOracle, StoredRotatedOracle, EpochRotatedOracle, rerotate,
    brute_force_window, brute_force_reprefill, SPLIT_HALF, INTERLEAVED)
