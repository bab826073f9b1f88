"""Retained window smaller than the ring, on the GPU (through the C ABI).

The causal audio encoder of "audio8-asr-infinite-p150" ("At a glance") keeps a
sliding window of 750 frames; the cache keeps it in a ring of 768 slots (whole
32-slot blocks), four new frames per step.  Step logs must equal the oracle's
bookkeeping bit for bit at every step; attention outputs must stay within
max-abs 2e-2 / mean-abs 2e-3 of the float64 oracle on the same bf16 inputs.
"""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, initial_window, step_inputs
from tests.gpu_util import compare, dev, make_cache, make_oracle, poison_outside, write_window

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("impl", ["auto", "fma"])
def test_encoder_window_fill_evict_wrap(impl):
    """Encoder shape cut to 2 layers: 500 steps of 4 frames from an empty
    window, past the fill (step 188), the first eviction and several trips
    around the 768 slots; logs checked every step, outputs at sampled steps."""
    wl = WORKLOADS["encoder750"].replace(n_layers=2)
    cache = make_cache(wl, attend_impl=impl)
    orc = make_oracle(wl)
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    o, n = 0, 0
    check = {1, 2, 8, 187, 188, 189, 190, 192, 250, 383, 384, 385, 499, 500}
    for t in range(1, 501):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16), step_log=log)
        bk = O.bookkeep(o, n, 4, 750, 768)
        o, n = bk.origin, bk.fill
        assert tuple(log[0].tolist()) == bk.log(), f"step {t}"
        orc.append(k.double().numpy(), v.double().numpy())
        if t in check:
            out = cache.attend(dev(q, torch.bfloat16))
            compare(out, orc.attend(q.double().numpy()))
    og, fg, st = cache.get_stream_state()
    assert (int(og[0]), int(fg[0]), int(st[0])) == (2000 - 750, 750, 0)


def test_encoder_window_full_size_sampled_layers():
    """All 32 layers of the encoder shape in one attend launch (the benchmarked
    call), a full 750-frame window at origin 777777 whose ring start is not
    block aligned; layers 0, 13 and 31 checked over three evicting steps, with
    every slot outside the window poisoned with NaN (evicted frames and the
    18 slots the window never uses are never read)."""
    wl = WORKLOADS["encoder750"]
    layers = [0, 13, 31]
    cache = make_cache(wl)
    orc = make_oracle(wl, n_layers=len(layers))
    origin = 777_777
    k, v = initial_window(wl, 0, 750)
    write_window(cache, 0, origin, 750, k, v)
    orc.set_state(0, origin, 750, k[layers].double().numpy(), v[layers].double().numpy())
    for t in range(1, 4):
        q, kn, vn = step_inputs(wl, t)
        o, f, _ = cache.get_stream_state()
        poison_outside(cache, o, f)
        cache.append(dev(kn, torch.bfloat16), dev(vn, torch.bfloat16))
        out = cache.attend(dev(q, torch.bfloat16))
        orc.append(kn[layers].double().numpy(), vn[layers].double().numpy())
        compare(out[layers], orc.attend(q[layers].double().numpy()))
    og, fg, st = cache.get_stream_state()
    assert (int(og[0]), int(fg[0]), int(st[0])) == (origin + 12, 750, 0)


@pytest.mark.parametrize("layout", ["pre_rope", "stored_rotated"])
def test_decode_window_fused_step_and_layouts(layout):
    """One token per step with a window of 1000 in 1024 slots: the fused step
    (pre-RoPE) or append + re-base + attend (stored-rotated keys, re-rotated at
    every eviction) against the oracle through fill, eviction and a wrap."""
    wl = WORKLOADS["audio8"].replace(n_layers=2, window=1000)
    cache = make_cache(wl, layout=layout)
    orc = make_oracle(wl, cls=O.StoredRotatedOracle if layout == "stored_rotated" else
                      O.RollingCacheOracle)
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    o, n = 0, 0
    check = {1, 999, 1000, 1001, 1024, 1025, 1500, 2100}
    for t in range(1, 2101):
        q, k, v = step_inputs(wl, t)
        kd, vd, qd = dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.bfloat16)
        bk = O.bookkeep(o, n, 1, 1000, 1024)
        o, n = bk.origin, bk.fill
        orc.append(k.double().numpy(), v.double().numpy())
        if layout == "stored_rotated":
            orc.rebase()
            cache.append(kd, vd, step_log=log)
            cache.rebase()
            out = cache.attend(qd) if t in check else None
        else:
            out = cache.step(kd, vd, qd, step_log=log)
        assert tuple(log[0].tolist()) == bk.log(), f"step {t}"
        if t in check:
            compare(out, orc.attend(q.double().numpy()))


def test_window_rejects_fill_above_window():
    wl = WORKLOADS["encoder750"].replace(n_layers=1)
    cache = make_cache(wl)
    import rolling_kv_cache_buffer_b300 as R
    with pytest.raises(R.RkvError):
        cache.set_stream_state(0, 5, 751)
    cache.set_stream_state(0, 5, 750)
