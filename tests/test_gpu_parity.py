"""CUDA path against the float64 oracle (through the C ABI).

Bookkeeping (origins, fills, evictions, slots) must be bit-exact; attention
outputs must stay within max-abs 2e-2 and mean-abs 2e-3 of the oracle on the
same bf16-rounded inputs.
"""
import os

import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, initial_window, random_rows, step_inputs
from rolling_kv_cache_buffer_b300 import RollingKV
from tests.gpu_util import (MAX_ABS, MEAN_ABS, compare, dev, make_cache, make_oracle,
                            poison_outside, write_window)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

IMPLS = ["fma", "auto"]


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [tuple(int(x) for x in line.split()) for line in f if not line.startswith("#")]


# ----------------------------------------------------------------------------
# Bookkeeping: bit-exact logs
# ----------------------------------------------------------------------------

def test_tiny_stream_every_step():
    """Tiny workload, 200 single-token steps: the GPU step log equals the
    stored closed-form log bit for bit, and the attention output of every step
    matches the oracle."""
    wl = WORKLOADS["tiny"]
    cache = make_cache(wl)
    orc = make_oracle(wl)
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    want = _golden("tiny_bookkeeping.txt")
    worst = 0.0
    for t in range(1, wl.steps + 1):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.float32), dev(v, torch.float32), step_log=log)
        out = cache.attend(dev(q, torch.float32))
        orc.append(k.double().numpy(), v.double().numpy())
        ref = orc.attend(q.double().numpy())
        assert tuple(log[0].tolist()) == want[t - 1][1:], f"step {t}"
        worst = max(worst, compare(out, ref, 1e-4, 1e-5)[0])
    o, f, st = cache.get_stream_state()
    assert (int(o[0]), int(f[0]), int(st[0])) == (168, 32, 0)


def test_chunk_bookkeeping_golden():
    """Six pairs per step from origin 999990 with 20 retained: GPU logs equal
    the stored oracle log."""
    wl = WORKLOADS["tiny"].replace(n_new=6)
    cache = make_cache(wl, max_chunk=6)
    cache.set_stream_state(0, 999_990, 20)
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    for row in _golden("chunk_bookkeeping.txt"):
        _, k, v = step_inputs(wl, row[0])
        cache.append(dev(k, torch.float32), dev(v, torch.float32), step_log=log)
        assert tuple(log[0].tolist()) == row[1:]


@pytest.mark.parametrize("impl", IMPLS)
def test_audio8_fill_evict_wrap(impl):
    """Audio8-ASR-0.1B shape (8 layers, 8/8 heads, D 64, bf16, W 1024): run
    past the fill, the first eviction and a wrap of the ring; check the logs
    every step and the outputs at sampled steps."""
    wl = WORKLOADS["audio8"]
    cache = make_cache(wl, attend_impl=impl)
    orc = make_oracle(wl)
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    o, n = 0, 0
    check = {1, 2, 31, 32, 33, 500, 1023, 1024, 1025, 1100, 2049}
    for t in range(1, 2050):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16), step_log=log)
        orc.append(k.double().numpy(), v.double().numpy())
        bk = O.bookkeep(o, n, 1, wl.capacity)
        o, n = bk.origin, bk.fill
        if t in check:
            assert tuple(log[0].tolist()) == bk.log()
            out = cache.attend(dev(q, torch.bfloat16))
            compare(out, orc.attend(q.double().numpy()))


# ----------------------------------------------------------------------------
# Full-size workloads, sampled outputs
# ----------------------------------------------------------------------------

def _seed_full_window(wl, cache, orc, s, origin, fill, layers, orc_stream=0):
    k, v = initial_window(wl, s, fill)
    write_window(cache, s, origin, fill, k, v)
    orc.set_state(orc_stream, origin, fill, k[layers].double().numpy(),
                  v[layers].double().numpy())


@pytest.mark.parametrize("impl", IMPLS)
def test_qwen3b_full_window_sampled_layers(impl):
    """36-layer GQA 16/2 x 128, W 4096, full window at origin 123456, all 36
    layers in one attend launch (the benchmarked call); layers 0, 17 and 35
    checked against the oracle over three evicting steps."""
    wl = WORKLOADS["qwen3b"]
    layers = [0, 17, 35]
    cache = make_cache(wl, attend_impl=impl)
    orc = make_oracle(wl, n_layers=len(layers))
    _seed_full_window(wl, cache, orc, 0, 123_456, wl.capacity, layers)
    for t in range(1, 4):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        out = cache.attend(dev(q, torch.bfloat16))
        orc.append(k[layers].double().numpy(), v[layers].double().numpy())
        compare(out[layers], orc.attend(q[layers].double().numpy()))
    o, f, st = cache.get_stream_state()
    assert (int(o[0]), int(f[0]), int(st[0])) == (123_459, 4096, 0)


@pytest.mark.parametrize("impl", IMPLS)
def test_batch64_sampled_streams(impl):
    """64 streams, W 8192, fills uniform in [1, 8192], origins uniform in
    [0, 1e6).  Streams 0, 1 and 63 carry seeded contents and are checked on
    layers 0 and 35; the others hold random data."""
    wl = WORKLOADS["batch64"]
    from rkv_inputs import initial_states
    origins, fills = initial_states(wl)
    cache = make_cache(wl, attend_impl=impl)
    gen = torch.Generator(device="cuda").manual_seed(7)
    cache.k_pool.normal_(generator=gen)
    cache.v_pool.normal_(generator=gen)
    for s in range(wl.n_streams):
        cache.set_stream_state(s, origins[s], fills[s])
    sample, layers = [0, 1, 63], [0, 35]
    orcs = {}
    for s in sample:
        orcs[s] = make_oracle(wl, n_layers=len(layers), n_streams=1)
        _seed_full_window(wl, cache, orcs[s], s, origins[s], fills[s], layers)
    for t in range(1, 3):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        out = cache.attend(dev(q, torch.bfloat16))
        for s in sample:
            orcs[s].append(k[layers][:, s:s + 1].double().numpy(),
                           v[layers][:, s:s + 1].double().numpy())
            ref = orcs[s].attend(q[layers][:, s:s + 1].double().numpy())
            compare(out[layers][:, s:s + 1], ref)
    o, f, st = cache.get_stream_state()
    for s in range(wl.n_streams):
        bk1 = O.bookkeep(origins[s], fills[s], 1, wl.capacity)
        bk2 = O.bookkeep(bk1.origin, bk1.fill, 1, wl.capacity)
        assert (int(o[s]), int(f[s]), int(st[s])) == (bk2.origin, bk2.fill, 0)


# ----------------------------------------------------------------------------
# Pages' invariants on the GPU
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("impl", IMPLS)
def test_evicted_slots_never_read(impl):
    """Every slot outside each stream's window holds NaN; the outputs stay
    finite and bitwise equal to those of the unpoisoned pools."""
    wl = WORKLOADS["qwen3b"].replace(n_streams=4, n_layers=3, capacity=256)
    cache = make_cache(wl, attend_impl=impl)
    origins, fills = [0, 250, 1000, 77], [1, 37, 200, 256]
    for s in range(4):
        k = random_rows((3, 2, fills[s], 128), 100 + s, torch.bfloat16)
        v = random_rows((3, 2, fills[s], 128), 200 + s, torch.bfloat16)
        write_window(cache, s, origins[s], fills[s], k, v)
    q = dev(random_rows((3, 4, 1, 16, 128), 5, torch.bfloat16), torch.bfloat16)
    clean = cache.attend(q).clone()
    poison_outside(cache, origins, fills)
    dirty = cache.attend(q)
    assert torch.isfinite(dirty).all()
    assert torch.equal(clean, dirty)


@pytest.mark.parametrize("impl", IMPLS)
def test_origin_shift_invariance(impl):
    """The same window contents at origins 0, 12345, 999999 and 10^12 give the
    same outputs: bitwise when the origins agree modulo W (same slots).
    Otherwise the slot blocks differ, which changes the summation order (the
    f32 CUDA-core path stays within 1e-5) and, on the tensor-core path, which
    rotation goes into the bf16 query operand and which into the bf16 key
    operand (within 4e-3, inside the oracle tolerance)."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=512)
    k = random_rows((2, 2, 400, 128), 11, torch.bfloat16)
    v = random_rows((2, 2, 400, 128), 12, torch.bfloat16)
    q = dev(random_rows((2, 1, 1, 16, 128), 13, torch.bfloat16), torch.bfloat16)
    outs = {}
    for origin in (0, 12345, 999_999, 512 * 7, 10 ** 12):
        cache = make_cache(wl, attend_impl=impl)
        write_window(cache, 0, origin, 400, k, v)
        outs[origin] = cache.attend(q).cpu()
    assert torch.equal(outs[0], outs[512 * 7])
    tol = 1e-5 if impl == "fma" else 4e-3
    for origin in (12345, 999_999, 10 ** 12):
        assert (outs[origin] - outs[0]).abs().max() < tol


def test_empty_window_gives_zero():
    wl = WORKLOADS["qwen3b"].replace(n_streams=2, n_layers=1, capacity=64)
    cache = make_cache(wl)
    k = random_rows((1, 2, 10, 128), 1, torch.bfloat16)
    write_window(cache, 1, 5, 10, k, k)
    q = dev(random_rows((1, 2, 1, 16, 128), 2, torch.bfloat16), torch.bfloat16)
    out = torch.full(q.shape, 7.0, device="cuda")
    cache.attend(q, out)
    assert torch.equal(out[:, 0], torch.zeros_like(out[:, 0]))
    assert torch.isfinite(out[:, 1]).all() and out[:, 1].abs().sum() > 0


# ----------------------------------------------------------------------------
# Chunked insert (causal among the chunk)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("wl_name,c,impl", [("tiny", 5, "fma"), ("audio8", 6, "fma"),
                                            ("audio8", 6, "auto"), ("qwen3b", 6, "auto"),
                                            ("qwen3b", 2, "auto"), ("qwen3b", 12, "auto")])
def test_chunk_causal(wl_name, c, impl):
    base = WORKLOADS[wl_name]
    wl = base.replace(n_new=c, capacity=min(base.capacity, 64), n_layers=min(base.n_layers, 2))
    dt = torch.bfloat16 if wl.kv_dtype == "bf16" else torch.float32
    cache = make_cache(wl, attend_impl=impl, max_chunk=c)
    orc = make_oracle(wl)
    for t in range(1, 30):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, dt), dev(v, dt))
        out = cache.attend(dev(q, dt))
        orc.append(k.double().numpy(), v.double().numpy())
        compare(out, orc.attend(q.double().numpy()))


def test_qwen3b_chunk6_full_window_sampled_layers():
    """The 6-token workload (36 layers, GQA 16/2 x 128, W 4096, 1% of k rows
    doubled): full window at origin 123456, all layers in one launch, layers
    0, 17 and 35 checked over three evicting steps."""
    wl = WORKLOADS["qwen3b_chunk6"]
    layers = [0, 17, 35]
    cache = make_cache(wl)
    orc = make_oracle(wl, n_layers=len(layers))
    _seed_full_window(wl, cache, orc, 0, 123_456, wl.capacity, layers)
    for t in range(1, 4):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        out = cache.attend(dev(q, torch.bfloat16))
        orc.append(k[layers].double().numpy(), v[layers].double().numpy())
        compare(out[layers], orc.attend(q[layers].double().numpy()))
    o, f, st = cache.get_stream_state()
    assert (int(o[0]), int(f[0]), int(st[0])) == (123_474, 4096, 0)


@pytest.mark.parametrize("layout,style", [("pre_rope", "interleaved"),
                                          ("stored_rotated", "split_half")])
def test_chunk_layouts(layout, style):
    """6-token chunks with the interleaved pairing and with stored-rotated keys,
    through fill, eviction and the ring's wrap."""
    wl = WORKLOADS["qwen3b_chunk6"].replace(n_layers=2, capacity=64)
    cache = make_cache(wl, layout=layout, style=style)
    cls = O.StoredRotatedOracle if layout == "stored_rotated" else O.RollingCacheOracle
    orc = make_oracle(wl, cls=cls, style=style)
    for t in range(1, 26):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if layout == "stored_rotated":
            cache.rebase()
            orc.rebase()
        out = cache.attend(dev(q, torch.bfloat16))
        compare(out, orc.attend(q.double().numpy()))


def test_chunk_evicted_slots_never_read():
    """Chunk attention over windows whose other slots hold NaN: finite outputs,
    bitwise equal to those of clean pools."""
    wl = WORKLOADS["qwen3b"].replace(n_streams=4, n_layers=3, capacity=256)
    cache = make_cache(wl, max_chunk=6)
    origins, fills = [0, 250, 1000, 77], [6, 37, 200, 256]
    for s in range(4):
        k = random_rows((3, 2, fills[s], 128), 300 + s, torch.bfloat16)
        v = random_rows((3, 2, fills[s], 128), 400 + s, torch.bfloat16)
        write_window(cache, s, origins[s], fills[s], k, v)
    q = dev(random_rows((3, 4, 6, 16, 128), 7, torch.bfloat16), torch.bfloat16)
    clean = cache.attend(q).clone()
    poison_outside(cache, origins, fills)
    dirty = cache.attend(q)
    assert torch.isfinite(dirty).all()
    assert torch.equal(clean, dirty)


# ----------------------------------------------------------------------------
# Stored-rotated layout
# ----------------------------------------------------------------------------

def test_stored_rotated_rerotation_within_one_ulp():
    """Per call: the GPU's re-rotation of its own stored bf16 keys equals the
    oracle's float64 rotation rounded to bf16 within one bf16 ulp."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=128)
    cache = make_cache(wl, layout="stored_rotated")
    for t in range(1, 140):
        q, k, v = step_inputs(wl, t)
        before = cache.k_pool.clone()
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        o, f, _ = cache.get_stream_state()
        after_append = cache.k_pool.clone()
        cache.rebase()
        after = cache.k_pool.clone()
        if t in (129, 130, 139):
            e = 1
            W = wl.capacity
            old = [(int(o[0]) + r) % W for r in range(int(f[0]) - 1)]
            src = after_append[0][:, :, old].double().cpu().numpy()
            want = O.rerotate(src, e, wl.rope_theta)
            got = after[0][:, :, old].double().cpu().numpy()
            ulp = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
            assert np.all(np.abs(got - want) <= ulp + 1e-30)
        del before


def test_stored_rotated_stream_matches_oracle():
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=64)
    cache = make_cache(wl, layout="stored_rotated")
    orc = make_oracle(wl, cls=O.StoredRotatedOracle)
    for t in range(1, 100):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        cache.rebase()
        orc.append(k.double().numpy(), v.double().numpy())
        orc.rebase()
        out = cache.attend(dev(q, torch.bfloat16))
        if t % 7 == 0 or t > 95:
            compare(out, orc.attend(q.double().numpy()))


@pytest.mark.parametrize("style", ["split_half", "interleaved"])
def test_stored_rotated_float32_head_dim_64(style):
    """Stored-rotated keys in float32 pools (tiny workload, D = 64), re-rotated
    at every eviction for 100 steps (three trips round the ring): each call's
    re-rotation equals the float64 rotation R(-e) of the stored keys within
    float32 rounding, and the attention equals the exact (pre-RoPE) oracle
    within the float32 path's 1e-4 / 1e-5."""
    wl = WORKLOADS["tiny"]
    cache = make_cache(wl, layout="stored_rotated", style=style)
    orc = make_oracle(wl, style=style)
    W = wl.capacity
    for t in range(1, 101):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.float32), dev(v, torch.float32))
        o, f, _ = cache.get_stream_state()
        old = [(int(o[0]) + r) % W for r in range(int(f[0]) - 1)]
        src = cache.k_pool[0][:, :, old].double().cpu().numpy()
        cache.rebase()
        if t > W:   # one eviction per step from here on
            got = cache.k_pool[0][:, :, old].double().cpu().numpy()
            want = O.rope(src, -1.0, wl.rope_theta, style)
            assert np.abs(got - want).max() <= 1e-5
        orc.append(k.double().numpy(), v.double().numpy())
        compare(cache.attend(dev(q, torch.float32)), orc.attend(q.double().numpy()), 1e-4, 1e-5)


def test_stored_rotated_bf16_head_dim_64():
    """Stored-rotated bf16 keys with D = 64 and the interleaved pairing (audio8
    shape, 2 layers, W = 64), every eviction re-rotated: each call within one
    bf16 ulp of the float64 rotation, outputs against the oracle that stores
    bf16 keys the same way."""
    wl = WORKLOADS["audio8"].replace(n_layers=2, capacity=64)
    style = "interleaved"
    cache = make_cache(wl, layout="stored_rotated", style=style)
    orc = make_oracle(wl, cls=O.StoredRotatedOracle, style=style)
    W = wl.capacity
    for t in range(1, 151):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        o, f, _ = cache.get_stream_state()
        old = [(int(o[0]) + r) % W for r in range(int(f[0]) - 1)]
        src = cache.k_pool[0][:, :, old].double().cpu().numpy()
        cache.rebase()
        if t > W and t % 5 == 0:
            got = cache.k_pool[0][:, :, old].double().cpu().numpy()
            want = O.rerotate(src, 1, wl.rope_theta, style)
            ulp = np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8)
            assert np.all(np.abs(got - want) <= ulp + 1e-30)
        orc.append(k.double().numpy(), v.double().numpy())
        orc.rebase()
        if t % 7 == 0 or t > 145:
            compare(cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy()))


# ----------------------------------------------------------------------------
# Utterance reset with a prefix
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["pre_rope", "stored_rotated"])
def test_reset_stream_with_prefix(layout):
    """Stream 1 restarts at a new origin holding a 20-pair prefix while stream 0
    keeps its window (its pools untouched): outputs match the oracle whose
    window is set to the same prefix, through the appends that later evict
    the prefix; states and logs follow the closed form; a sticky status is
    cleared by the reset; a reset without prefix leaves an empty window."""
    stored = layout == "stored_rotated"
    wl = WORKLOADS["qwen3b"].replace(n_streams=2, n_layers=2, capacity=64)
    cache = make_cache(wl, layout=layout)
    orc = make_oracle(wl, cls=O.StoredRotatedOracle if stored else O.RollingCacheOracle)

    def step(t):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if stored:
            cache.rebase()
            orc.rebase()
        return cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy())

    for t in range(1, 11):
        step(t)
    st32 = cache.state.view(torch.int32)
    st32[8 * 1 + 2] = 65     # stream 1: fill 65 > W (corrupt) ...
    st32[8 * 1 + 3] = 5      # ... and flagged
    n, origin = 20, 777_777
    kp = random_rows((2, n, 2, 128), 11, torch.bfloat16)   # [L][n][H_kv][D]
    vp = random_rows((2, n, 2, 128), 12, torch.bfloat16)
    pool0 = cache.k_pool[0].clone(), cache.v_pool[0].clone()
    cache.reset_stream(1, origin, dev(kp, torch.bfloat16), dev(vp, torch.bfloat16))
    orc.set_state(1, origin, n, kp.permute(0, 2, 1, 3).double().numpy(),
                  vp.permute(0, 2, 1, 3).double().numpy())
    assert torch.equal(cache.k_pool[0], pool0[0]) and torch.equal(cache.v_pool[0], pool0[1])
    o, f, st = cache.get_stream_state()
    assert (int(o[1]), int(f[1]), int(st[1])) == (origin, n, 0)
    assert (int(o[0]), int(f[0]), int(st[0])) == (0, 10, 0)
    for t in range(11, 11 + 60):   # stream 1 fills at 64 and then evicts the prefix
        out, ref = step(t)
        if t % 6 == 0 or t > 65:
            compare(out, ref)
    o, f, st = cache.get_stream_state()
    assert (int(o[1]), int(f[1]), int(st[1])) == (origin + 20 + 60 - 64, 64, 0)
    cache.reset_stream(1, 5)
    orc.set_state(1, 5, 0)
    o, f, st = cache.get_stream_state()
    assert (int(o[1]), int(f[1]), int(st[1])) == (5, 0, 0)
    out, ref = step(71)
    compare(out, ref)


@pytest.mark.parametrize("wl_name,layout,style,epoch", [
    ("qwen3b", "stored_rotated", "split_half", 16),
    ("qwen3b", "pre_rope", "interleaved", 0),
    ("qwen3b", "stored_rotated", "interleaved", 0),
    ("tiny", "pre_rope", "split_half", 0),
    ("tiny", "stored_rotated", "interleaved", 0)])
def test_reset_stream_with_prefix_variants(wl_name, layout, style, epoch):
    """The utterance reset on the paths the base case does not take: stored-
    rotated keys with a re-basing epoch (the reset clears the lag and stores the
    prefix keys rotated to their positions from the new origin), the
    interleaved pairing (both layouts) and float32 pools (the CUDA-core path).
    Stream 1 restarts with a prefix, then appends run until the prefix is
    evicted; every few steps the outputs are compared with the oracle whose
    window was set to the same prefix."""
    base = WORKLOADS[wl_name]
    wl = base.replace(n_streams=2, n_layers=min(base.n_layers, 2),
                      capacity=min(base.capacity, 64))
    f32 = wl.kv_dtype == "f32"
    dt = torch.float32 if f32 else torch.bfloat16
    stored = layout == "stored_rotated"
    cache = RollingKV(2, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.capacity,
                      max_chunk=1, kv_dtype=wl.kv_dtype, layout=layout, rope_style=style,
                      rope_theta=wl.rope_theta, rebase_epoch=epoch)
    args = (2, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.capacity)
    if epoch:
        orc = O.EpochRotatedOracle(*args, theta=wl.rope_theta, style=style, epoch=epoch)
    elif stored and not f32:
        orc = O.StoredRotatedOracle(*args, theta=wl.rope_theta, style=style)
    else:   # float32 keys are kept exact enough for the plain definition
        orc = O.RollingCacheOracle(*args, theta=wl.rope_theta, style=style)
    tol = (1e-4, 1e-5) if f32 else (MAX_ABS, MEAN_ABS)
    rebase_oracle = hasattr(orc, "rebase") and (epoch or (stored and not f32))

    def step(t):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, dt), dev(v, dt))
        orc.append(k.double().numpy(), v.double().numpy())
        if stored:
            cache.rebase()
            if rebase_oracle:
                orc.rebase()
        return cache.attend(dev(q, dt)), orc.attend(q.double().numpy())

    for t in range(1, 11):
        step(t)
    n, origin = 12, 424_242
    D, Hkv = wl.head_dim, wl.n_kv_heads
    kp = random_rows((wl.n_layers, n, Hkv, D), 31, dt)
    vp = random_rows((wl.n_layers, n, Hkv, D), 32, dt)
    cache.reset_stream(1, origin, dev(kp, dt), dev(vp, dt))
    orc.set_state(1, origin, n, kp.permute(0, 2, 1, 3).double().numpy(),
                  vp.permute(0, 2, 1, 3).double().numpy())
    o, f, st = cache.get_stream_state()
    assert (int(o[1]), int(f[1]), int(st[1])) == (origin, n, 0)
    W = wl.capacity
    for t in range(11, 11 + W + 16):   # past the fill and the prefix's eviction
        out, ref = step(t)
        if t % 5 == 0 or t > W + 20:
            compare(out, ref, *tol)
    o, f, st = cache.get_stream_state()
    assert (int(o[1]), int(f[1]), int(st[1])) == (origin + n + W + 16 - W, W, 0)


# ----------------------------------------------------------------------------
# Device-side error paths (no fault: a status word)
# ----------------------------------------------------------------------------

def test_corrupt_state_sets_status_and_is_skipped():
    wl = WORKLOADS["qwen3b"].replace(n_streams=2, n_layers=1, capacity=64)
    cache = make_cache(wl)
    st = cache.state.view(torch.int32)
    st[8 * 1 + 2] = 65          # stream 1: fill 65 > W = 64
    q, k, v = step_inputs(wl, 1)
    log = torch.zeros((2, 4), dtype=torch.int64, device="cuda")
    cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16), step_log=log)
    o, f, status = cache.get_stream_state()
    assert status[0] == 0 and status[1] == 5
    assert log[1, 2].item() == -1 and log[0, 1].item() == 1
    out = torch.full((1, 2, 1, 16, 128), 3.0, device="cuda")
    cache.attend(dev(q, torch.bfloat16), out)
    assert torch.equal(out[:, 1], torch.full_like(out[:, 1], 3.0))   # not written
    cache.set_stream_state(1, 0, 0)
    assert cache.get_stream_state()[2][1] == 0


def test_stored_rotated_missing_rebase_is_flagged():
    wl = WORKLOADS["qwen3b"].replace(n_layers=1, capacity=32)
    cache = make_cache(wl, layout="stored_rotated")
    for t in range(1, 35):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
    assert cache.get_stream_state()[2][0] == 5      # step 33 evicted; no re-base before 34


def test_launch_counts():
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=64)
    cache = make_cache(wl)
    q, k, v = step_inputs(wl, 1)
    cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
    assert cache.last_launch_count() == 1
    cache.rebase()
    assert cache.last_launch_count() == 0          # pre-RoPE re-base moves nothing
    cache.attend(dev(q, torch.bfloat16))
    assert cache.last_launch_count() == 1
