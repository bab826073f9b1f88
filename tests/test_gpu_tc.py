"""Chunk attention on the tcgen05 tensor cores (attend_impl "tc") against the
float64 oracle, through the C ABI (GPU).

Steps that insert c >= 2 tokens per stream, causal among the chunk ("Audio8
ASR Infinite: What It Actually Takes to Listen Forever", "Inside the Rolling
KV Cache and Exact RoPE Re-Basing"; the 6-token workload is causal among its
tokens).  Outputs must stay within max-abs 2e-2 / mean-abs 2e-3 of the oracle
on the same bf16-rounded inputs.
"""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, initial_window, random_rows, step_inputs
from tests.gpu_util import compare, dev, make_cache, make_oracle, poison_outside, write_window

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl_name,c", [("qwen3b", 2), ("qwen3b", 6), ("qwen3b", 12),
                                       ("qwen3b", 16), ("audio8", 6), ("encoder750", 4)])
def test_tc_chunk_causal(wl_name, c):
    """From an empty window through fill, eviction and several wraps of a
    64-slot ring (2 layers): every step against the oracle."""
    base = WORKLOADS[wl_name]
    wl = base.replace(n_new=c, capacity=64, n_layers=2, window=None)
    cache = make_cache(wl, attend_impl="tc", max_chunk=c)
    orc = make_oracle(wl)
    for t in range(1, 40):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        out = cache.attend(dev(q, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        compare(out, orc.attend(q.double().numpy()))


def test_tc_qwen3b_chunk6_full_window_sampled_layers():
    """The 6-token workload (36 layers, GQA 16/2 x 128, W 4096, 1% of k rows
    doubled): full window at origin 123456, all layers in one launch (the
    benchmarked call), layers 0, 17 and 35 checked over three steps."""
    wl = WORKLOADS["qwen3b_chunk6"]
    layers = [0, 17, 35]
    cache = make_cache(wl, attend_impl="tc")
    orc = make_oracle(wl, n_layers=len(layers))
    k, v = initial_window(wl, 0, wl.capacity)
    write_window(cache, 0, 123_456, wl.capacity, k, v)
    orc.set_state(0, 123_456, wl.capacity, k[layers].double().numpy(),
                  v[layers].double().numpy())
    for t in range(1, 4):
        q, kn, vn = step_inputs(wl, t)
        cache.append(dev(kn, torch.bfloat16), dev(vn, torch.bfloat16))
        out = cache.attend(dev(q, torch.bfloat16))
        orc.append(kn[layers].double().numpy(), vn[layers].double().numpy())
        compare(out[layers], orc.attend(q[layers].double().numpy()))


@pytest.mark.parametrize("layout,style,epoch", [("pre_rope", "interleaved", 0),
                                                ("stored_rotated", "split_half", 0),
                                                ("stored_rotated", "interleaved", 64)])
def test_tc_layouts(layout, style, epoch):
    """Interleaved pairing, stored-rotated keys (re-rotated at every eviction,
    or with a re-basing epoch): 6-token chunks through fill, eviction and wrap."""
    wl = WORKLOADS["qwen3b_chunk6"].replace(n_layers=2, capacity=96)
    from rolling_kv_cache_buffer_b300 import RollingKV
    cache = RollingKV(1, 2, 16, 2, 128, 96, max_chunk=6, layout=layout, rope_style=style,
                      attend_impl="tc", rebase_epoch=epoch)
    if epoch:
        orc = O.EpochRotatedOracle(1, 2, 16, 2, 128, 96, style=style, epoch=epoch)
    else:
        cls = O.StoredRotatedOracle if layout == "stored_rotated" else O.RollingCacheOracle
        orc = cls(1, 2, 16, 2, 128, 96, style=style)
    for t in range(1, 60):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if layout == "stored_rotated":
            cache.rebase()
            orc.rebase()
        out = cache.attend(dev(q, torch.bfloat16))
        compare(out, orc.attend(q.double().numpy()))


def test_tc_partial_windows_poisoned():
    """Four streams with fills 6..256 at scattered origins, every slot outside
    the windows NaN: finite outputs, bitwise equal to those of clean pools,
    within tolerance of the oracle."""
    wl = WORKLOADS["qwen3b"].replace(n_streams=4, n_layers=3, capacity=256, n_new=6)
    cache = make_cache(wl, attend_impl="tc", max_chunk=6)
    orc = make_oracle(wl)
    origins, fills = [0, 250, 1000, 77], [6, 37, 200, 256]
    for s in range(4):
        k = random_rows((3, 2, fills[s], 128), 300 + s, torch.bfloat16)
        v = random_rows((3, 2, fills[s], 128), 400 + s, torch.bfloat16)
        write_window(cache, s, origins[s], fills[s], k, v)
        orc.set_state(s, origins[s], fills[s], k.double().numpy(), v.double().numpy())
    q = dev(random_rows((3, 4, 6, 16, 128), 7, torch.bfloat16), torch.bfloat16)
    clean = cache.attend(q).clone()
    poison_outside(cache, origins, fills)
    dirty = cache.attend(q)
    assert torch.isfinite(dirty).all()
    assert torch.equal(clean, dirty)
    compare(dirty, orc.attend(q.double().cpu().numpy()))


def test_tc_pinned_prefix_and_window():
    """A pinned prefix (32 slots, 20 pairs) in front of a ring of 224 slots
    with a retained window of 200, 4-token chunks through eviction and wraps."""
    from rolling_kv_cache_buffer_b300 import RollingKV
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=256, n_new=4)
    cache = RollingKV(1, 2, 16, 2, 128, 256, max_chunk=4, attend_impl="tc", window=200,
                      n_pinned=32)
    orc = O.RollingCacheOracle(1, 2, 16, 2, 128, 256, window=200, n_pinned=32)
    kp = random_rows((2, 20, 2, 128), 51, torch.bfloat16)
    vp = random_rows((2, 20, 2, 128), 52, torch.bfloat16)
    cache.reset_stream(0, 5_000, dev(kp, torch.bfloat16), dev(vp, torch.bfloat16))
    orc.reset(0, 5_000, kp.permute(0, 2, 1, 3).double().numpy(),
              vp.permute(0, 2, 1, 3).double().numpy(), 20)
    for t in range(1, 160):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if t % 7 == 0 or t in (1, 50, 51, 56, 57, 159):
            compare(cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy()))


def test_tc_agrees_with_mma_chunk_kernel():
    """The tcgen05 kernel and the mma.sync chunk kernel on the same full window
    (36 layers of the 6-token workload): both within tolerance of each other."""
    wl = WORKLOADS["qwen3b_chunk6"]
    outs = []
    for impl in ("tc", "auto"):
        cache = make_cache(wl, attend_impl=impl)
        k, v = initial_window(wl, 0, wl.capacity)
        write_window(cache, 0, 7_777, wl.capacity, k, v)
        q, kn, vn = step_inputs(wl, 1)
        cache.append(dev(kn, torch.bfloat16), dev(vn, torch.bfloat16))
        outs.append(cache.attend(dev(q, torch.bfloat16)).double().cpu().numpy())
    compare(outs[0], outs[1], 2e-2, 2e-3)


@pytest.mark.parametrize("c,style,window", [(6, "split_half", None), (16, "split_half", None),
                                            (6, "interleaved", 512)])
def test_tc_pair_merge(c, style, window):
    """Rings of 16-17 blocks over 2 layers x 2 KV heads: the grid is exactly
    two CTAs per unit, one 2-CTA cluster each, and rank 1's partial is merged
    into rank 0's through distributed shared memory.  Windows of 1 block (whole
    units, no merge), 9 blocks (a 4 + 5 split) and the full window, then
    steps that evict; 16-token chunks fill the 128-row tile."""
    from rolling_kv_cache_buffer_b300 import RollingKV
    W = 512 if window is None else 544
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=W, n_new=c, window=window)
    cache = RollingKV(1, 2, 16, 2, 128, W, max_chunk=c, rope_style=style, attend_impl="tc",
                      window=window or 0)
    orc = O.RollingCacheOracle(1, 2, 16, 2, 128, W, style=style, window=window)
    for i, (fill, origin) in enumerate([(20, 77), (280, 123_457), (window or W, 9_999_999)]):
        k = random_rows((2, 2, fill, 128), 500 + 2 * i, torch.bfloat16)
        v = random_rows((2, 2, fill, 128), 501 + 2 * i, torch.bfloat16)
        write_window(cache, 0, origin, fill, k, v)
        orc.set_state(0, origin, fill, k.double().numpy(), v.double().numpy())
        for t in range(1, 4):
            q, kn, vn = step_inputs(wl, 10 * i + t)
            cache.append(dev(kn, torch.bfloat16), dev(vn, torch.bfloat16))
            orc.append(kn.double().numpy(), vn.double().numpy())
            compare(cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy()))


def test_tc_pair_merge_stored_rotated_and_pinned():
    """The cluster merge with stored-rotated keys (re-rotated at every
    eviction) from an empty 512-slot ring through eviction, and with a pinned
    prefix of 20 pairs in 32 slots in front of a 512-slot ring."""
    from rolling_kv_cache_buffer_b300 import RollingKV
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=512, n_new=6)
    cache = RollingKV(1, 2, 16, 2, 128, 512, max_chunk=6, layout="stored_rotated",
                      attend_impl="tc")
    orc = O.StoredRotatedOracle(1, 2, 16, 2, 128, 512)
    for t in range(1, 100):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        cache.rebase()
        orc.rebase()
        out = cache.attend(dev(q, torch.bfloat16))
        if t % 9 == 0 or t > 95:
            compare(out, orc.attend(q.double().numpy()))
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=544, n_new=4)
    cache = RollingKV(1, 2, 16, 2, 128, 544, max_chunk=4, attend_impl="tc", n_pinned=32)
    orc = O.RollingCacheOracle(1, 2, 16, 2, 128, 544, n_pinned=32)
    kp = random_rows((2, 20, 2, 128), 61, torch.bfloat16)
    vp = random_rows((2, 20, 2, 128), 62, torch.bfloat16)
    cache.reset_stream(0, 70_000, dev(kp, torch.bfloat16), dev(vp, torch.bfloat16))
    orc.reset(0, 70_000, kp.permute(0, 2, 1, 3).double().numpy(),
              vp.permute(0, 2, 1, 3).double().numpy(), 20)
    for t in range(1, 140):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if t % 11 == 0 or t in (1, 2, 128, 129, 130, 139):
            compare(cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy()))


def test_tc_pair_merge_head_dim_64():
    """The cluster merge with D = 64 (8 KV heads of one query head each, 8
    queries per step: 8 rows per unit) over a 512-slot ring: two CTAs per
    unit, windows of 9 blocks and the full ring, then steps that evict."""
    from rolling_kv_cache_buffer_b300 import RollingKV
    wl = WORKLOADS["audio8"].replace(n_layers=2, capacity=512, n_new=8)
    cache = RollingKV(1, 2, 8, 8, 64, 512, max_chunk=8, attend_impl="tc")
    orc = O.RollingCacheOracle(1, 2, 8, 8, 64, 512)
    for i, (fill, origin) in enumerate([(280, 4_321), (512, 77_777)]):
        k = random_rows((2, 8, fill, 64), 700 + 2 * i, torch.bfloat16)
        v = random_rows((2, 8, fill, 64), 701 + 2 * i, torch.bfloat16)
        write_window(cache, 0, origin, fill, k, v)
        orc.set_state(0, origin, fill, k.double().numpy(), v.double().numpy())
        for t in range(1, 4):
            q, kn, vn = step_inputs(wl, 20 * i + t)
            cache.append(dev(kn, torch.bfloat16), dev(vn, torch.bfloat16))
            orc.append(kn.double().numpy(), vn.double().numpy())
            compare(cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy()))
