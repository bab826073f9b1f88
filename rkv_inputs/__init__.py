"""Seeded synthetic inputs for the rolling KV cache workloads.

This module is shared by the tests, the bench and the oracle's callers.  It
holds no arithmetic of the method itself: only the workload catalogue (shapes)
and seeded random draws.  Every value is drawn as float32 N(0, 1) from a CPU
``torch.Generator`` and, for bf16 workloads, rounded to bfloat16 (round to
nearest even, torch's conversion), so both the CUDA path and the oracle see the
same bf16-exact numbers.

Recipe:
* seed(config) = 20261202 + config index;
* inputs of step t come from Generator.manual_seed(seed * 1_000_003 + t),
  drawn in the order q, k, v;
* the 6-token chunk workload scales k by 2 on 1% of the (layer, stream, token,
  kv-head) rows, chosen by Bernoulli(0.01) draws from the same generator after
  v;
* the 64-stream workload draws per-stream fills uniform in [1, capacity] and
  origins uniform in [0, 1e6) from Generator(seed * 1_000_003 - 1), and the
  initial window contents of stream s from Generator(seed * 1_000_003 - 2 - s).
"""

from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    n_streams: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    capacity: int
    kv_dtype: str          # "bf16" or "f32"
    n_new: int             # tokens appended per step
    steps: int             # stream length of the workload
    rope_theta: float = 1e6
    k_outlier_p: float = 0.0
    k_outlier_scale: float = 1.0
    random_state: bool = False
    window: int | None = None   # pairs retained (None: the capacity)

    @property
    def retained(self) -> int:
        return self.capacity if self.window is None else self.window

    @property
    def seed(self) -> int:
        return 20261202 + self.index

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 4

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.kv_dtype == "bf16" else torch.float32

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads: a tiny correctness case, the Audio8-ASR-0.1B decoder shape,
# the Qwen2.5-3B-class decoder shape (single token and 6-token chunks), 64
# independent streams of the latter, and the causal audio encoder's sliding
# window (32 layers, 750 frames kept in 768 slots, 4 new frames per step,
# width 1280 split as 20 heads of 64, one KV head per query head).
WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 1, 2, 1, 64, 32, "f32", 1, 200),
    "audio8": Workload("audio8", 1, 1, 8, 8, 8, 64, 1024, "bf16", 1, 8192),
    "qwen3b": Workload("qwen3b", 2, 1, 36, 16, 2, 128, 4096, "bf16", 1, 20000),
    "qwen3b_chunk6": Workload("qwen3b_chunk6", 3, 1, 36, 16, 2, 128, 4096, "bf16", 6, 5000,
                              k_outlier_p=0.01, k_outlier_scale=2.0),
    "batch64": Workload("batch64", 4, 64, 36, 16, 2, 128, 8192, "bf16", 1, 2000,
                        random_state=True),
    "encoder750": Workload("encoder750", 5, 1, 32, 20, 20, 64, 768, "bf16", 4, 5000,
                           window=750),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def _round(x: torch.Tensor, wl: Workload) -> torch.Tensor:
    if wl.kv_dtype == "bf16":
        return x.to(torch.bfloat16).to(torch.float32)
    return x


def step_inputs(wl: Workload, t: int, n_new: int | None = None):
    """Inputs of step t: q [L][S][c][H_q][D], k and v [L][S][c][H_kv][D].

    float32 CPU tensors holding bf16-exact values for bf16 workloads."""
    c = wl.n_new if n_new is None else n_new
    g = torch.Generator("cpu").manual_seed(wl.seed * 1_000_003 + t)
    L, S, Hq, Hkv, D = wl.n_layers, wl.n_streams, wl.n_q_heads, wl.n_kv_heads, wl.head_dim
    q = torch.randn((L, S, c, Hq, D), generator=g, dtype=torch.float32)
    k = torch.randn((L, S, c, Hkv, D), generator=g, dtype=torch.float32)
    v = torch.randn((L, S, c, Hkv, D), generator=g, dtype=torch.float32)
    if wl.k_outlier_p > 0:
        hit = torch.rand((L, S, c, Hkv, 1), generator=g) < wl.k_outlier_p
        k = torch.where(hit, k * wl.k_outlier_scale, k)
    return _round(q, wl), _round(k, wl), _round(v, wl)


def initial_states(wl: Workload):
    """(origins, fills) per stream before the first step."""
    if not wl.random_state:
        return [0] * wl.n_streams, [0] * wl.n_streams
    g = torch.Generator("cpu").manual_seed(wl.seed * 1_000_003 - 1)
    fills = torch.randint(1, wl.capacity + 1, (wl.n_streams,), generator=g)
    origins = torch.randint(0, 1_000_000, (wl.n_streams,), generator=g)
    return [int(o) for o in origins], [int(f) for f in fills]


def initial_window(wl: Workload, stream: int, fill: int):
    """Initial window contents of one stream: k, v [L][H_kv][fill][D] in
    position order (the i-th row is absolute position origin + i)."""
    g = torch.Generator("cpu").manual_seed(wl.seed * 1_000_003 - 2 - stream)
    shape = (wl.n_layers, wl.n_kv_heads, fill, wl.head_dim)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    return _round(k, wl), _round(v, wl)


def random_rows(shape, seed: int, dtype=torch.float32):
    """Generic seeded N(0,1) tensor (float32 values, bf16-exact if dtype is bf16)."""
    g = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if dtype == torch.bfloat16:
        x = x.to(torch.bfloat16).to(torch.float32)
    return x
