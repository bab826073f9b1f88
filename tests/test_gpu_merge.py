"""Split-unit merges with many partials, through the C ABI (GPU).

A (layer, KV head) window that many CTAs stream is finished by the last CTA
to take the unit's ticket, which combines the CTAs' partial softmax states
(m, l and the unnormalised O of each row):
  out = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k,   M = max_k m_k,
the split form of the attention over the window of "Audio8 ASR Infinite: What
It Actually Takes to Listen Forever" ("Inside the Rolling KV Cache and Exact
RoPE Re-Basing").  The kernels keep the per-partial weights in shared scratch
when they fit and recompute them per element when they do not; the windows
here are long enough (one unit cut into more than a hundred CTAs) to take the
second path, and the outputs must stay within max-abs 2e-2 / mean-abs 2e-3 of
the float64 oracle like every other GPU test.
"""
import pytest
import torch

from rkv_inputs import WORKLOADS, random_rows, step_inputs
from tests.gpu_util import compare, dev, make_cache, make_oracle, write_window

pytestmark = pytest.mark.gpu


def _full_window(wl, cache, orc, origin, seed):
    W = wl.capacity
    k = random_rows((wl.n_layers, wl.n_kv_heads, W, wl.head_dim), seed, torch.bfloat16)
    v = random_rows((wl.n_layers, wl.n_kv_heads, W, wl.head_dim), seed + 1, torch.bfloat16)
    write_window(cache, 0, origin, W, k, v)
    orc.set_state(0, origin, W, k.double().numpy(), v.double().numpy())


@pytest.mark.parametrize("path", ["calls", "fused"])
def test_decode_one_unit_over_many_ctas(path):
    """One layer, one KV head of 8 query heads, a full 65,536-slot window: the
    unit is cut into one share per SM and merged from all of them (more
    partials than the decode kernel's scratch holds)."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=1, n_q_heads=8, n_kv_heads=1, capacity=65536)
    cache = make_cache(wl)
    orc = make_oracle(wl)
    _full_window(wl, cache, orc, 9_876_543, 70)
    for t in range(1, 3):
        q, k, v = step_inputs(wl, t)
        kd, vd, qd = dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.bfloat16)
        if path == "fused":
            out = cache.step(kd, vd, qd)
        else:
            cache.append(kd, vd)
            out = cache.attend(qd)
        orc.append(k.double().numpy(), v.double().numpy())
        compare(out, orc.attend(q.double().numpy()))
    o, f, st = cache.get_stream_state()
    assert (int(o[0]), int(f[0]), int(st[0])) == (9_876_545, 65536, 0)


@pytest.mark.parametrize("impl,W", [("tc", 32768), ("mma", 65536)])
def test_chunk_one_unit_over_many_ctas(impl, W):
    """Six queries per step (48 rows) over one long window on each tensor-core
    chunk kernel: the unit is cut into a hundred or more shares."""
    wl = WORKLOADS["qwen3b_chunk6"].replace(n_layers=1, n_q_heads=8, n_kv_heads=1, capacity=W)
    cache = make_cache(wl, attend_impl=impl, max_chunk=6)
    orc = make_oracle(wl)
    _full_window(wl, cache, orc, 5_555, 80)
    q, k, v = step_inputs(wl, 1)
    cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
    out = cache.attend(dev(q, torch.bfloat16))
    orc.append(k.double().numpy(), v.double().numpy())
    compare(out, orc.attend(q.double().numpy()))
