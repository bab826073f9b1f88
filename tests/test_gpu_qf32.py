"""float32 queries on bf16 caches (rkv_config.q_dtype = f32), through the C ABI
(GPU).

The attention kernels rotate each query in f32 by R(r_j) ("Audio8 ASR
Infinite: What It Actually Takes to Listen Forever", "Inside the Rolling KV
Cache and Exact RoPE Re-Basing") whatever its storage type, and round the
rotated query to bf16 only as an operand of the bf16 tensor-core product.
Queries drawn in full float32 precision (not bf16-exact) exercise the f32
loads of every kernel family: the decode kernel (attend and the fused step),
the tcgen05 chunk kernel and the mma.sync chunk kernel.  Outputs must stay
within max-abs 2e-2 / mean-abs 2e-3 of the float64 oracle given the same
float32 queries.
"""
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, step_inputs
from tests.gpu_util import compare, dev

pytestmark = pytest.mark.gpu


def _q32(shape, t):
    g = torch.Generator("cpu").manual_seed(90_001 + t)
    return torch.randn(shape, generator=g, dtype=torch.float32)


@pytest.mark.parametrize("c,impl,fused", [(1, "auto", False), (1, "auto", True),
                                          (2, "auto", False), (6, "auto", False),
                                          (4, "mma", False)])
def test_f32_queries_on_bf16_cache(c, impl, fused):
    """From an empty 256-slot ring (2 layers, GQA 16/2 x 128) through fill and
    eviction; every few steps against the oracle."""
    from rolling_kv_cache_buffer_b300 import RollingKV
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=256, n_new=c)
    cache = RollingKV(1, 2, 16, 2, 128, 256, max_chunk=c, q_dtype="f32", attend_impl=impl)
    orc = O.RollingCacheOracle(1, 2, 16, 2, 128, 256)
    for t in range(1, 300 // c):
        _, k, v = step_inputs(wl, t)
        q = _q32((2, 1, c, 16, 128), t)
        kd, vd, qd = dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.float32)
        if fused:
            out = cache.step(kd, vd, qd)
        else:
            cache.append(kd, vd)
            out = cache.attend(qd)
        orc.append(k.double().numpy(), v.double().numpy())
        if t % 7 == 0 or t == 300 // c - 1:
            compare(out, orc.attend(q.double().numpy()))
