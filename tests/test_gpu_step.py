"""rkv_step (append + re-base + attend in one launch) against the float64
oracle and against the three separate calls (through the C ABI)."""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, initial_states, initial_window, random_rows, step_inputs
from tests.gpu_util import compare, dev, make_cache, make_oracle, write_window

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl_name,style", [("qwen3b", "split_half"), ("qwen3b", "interleaved"),
                                           ("audio8", "split_half")])
def test_step_from_empty_through_wrap(wl_name, style):
    """From an empty cache through the fill, the first eviction and two wraps
    of the ring: logs bit-exact, outputs within tolerance of the oracle, and
    pools bitwise equal to those of rkv_append + rkv_attend."""
    wl = WORKLOADS[wl_name].replace(n_layers=2, capacity=64)
    fused = make_cache(wl, style=style)
    split = make_cache(wl, style=style)
    orc = make_oracle(wl, style=style)
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    o, n = 0, 0
    for t in range(1, 140):
        q, k, v = step_inputs(wl, t)
        qd, kd, vd = dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16)
        out = fused.step(kd, vd, qd, step_log=log)
        split.append(kd, vd)
        orc.append(k.double().numpy(), v.double().numpy())
        bk = O.bookkeep(o, n, 1, wl.capacity)
        o, n = bk.origin, bk.fill
        assert tuple(log[0].tolist()) == bk.log(), f"step {t}"
        if t <= 3 or t % 9 == 0 or t in (63, 64, 65, 128, 129):
            compare(out, orc.attend(q.double().numpy()))
            # The fused kernel scores the new pair in f32 from the inputs, the
            # separate path from bf16 tensor-core operands: both sit within the
            # oracle tolerance, and within half of it of each other.
            ref = split.attend(qd)
            compare(out, ref.double().cpu().numpy(), 1e-2, 1e-3)
    assert torch.equal(fused.k_pool, split.k_pool) and torch.equal(fused.v_pool, split.v_pool)
    fo, ff, fs = fused.get_stream_state()
    so, sf, ss = split.get_stream_state()
    assert (fo.tolist(), ff.tolist(), fs.tolist()) == (so.tolist(), sf.tolist(), ss.tolist())


def test_step_qwen3b_full_window_sampled_layers():
    """The benchmarked call: 36 layers, GQA 16/2 x 128, W 4096, full window at
    origin 123456; layers 0, 17 and 35 checked over three steps."""
    wl = WORKLOADS["qwen3b"]
    layers = [0, 17, 35]
    cache = make_cache(wl)
    orc = make_oracle(wl, n_layers=len(layers))
    k, v = initial_window(wl, 0, wl.capacity)
    write_window(cache, 0, 123_456, wl.capacity, k, v)
    orc.set_state(0, 123_456, wl.capacity, k[layers].double().numpy(),
                  v[layers].double().numpy())
    for t in range(1, 4):
        q, k, v = step_inputs(wl, t)
        out = cache.step(dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.bfloat16))
        orc.append(k[layers].double().numpy(), v[layers].double().numpy())
        compare(out[layers], orc.attend(q[layers].double().numpy()))
    o, f, st = cache.get_stream_state()
    assert (int(o[0]), int(f[0]), int(st[0])) == (123_459, 4096, 0)


def test_step_many_streams():
    """Eight streams with fills 0, 1, 5, 31, 32, 33, 200, 256 (W 256) and
    scattered origins: every stream's outputs against the oracle."""
    wl = WORKLOADS["qwen3b"].replace(n_streams=8, n_layers=2, capacity=256)
    fills = [0, 1, 5, 31, 32, 33, 200, 256]
    origins = [0, 7, 250, 1000, 77, 12345, 999_999, 256 * 9 + 3]
    cache = make_cache(wl)
    orcs = []
    for s in range(8):
        k = random_rows((2, 2, fills[s], 128), 500 + s, torch.bfloat16)
        v = random_rows((2, 2, fills[s], 128), 600 + s, torch.bfloat16)
        write_window(cache, s, origins[s], fills[s], k, v)
        orc = make_oracle(wl, n_streams=1)
        orc.set_state(0, origins[s], fills[s], k.double().numpy(), v.double().numpy())
        orcs.append(orc)
    for t in range(1, 4):
        q, k, v = step_inputs(wl, t)
        out = cache.step(dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.bfloat16))
        for s in range(8):
            orcs[s].append(k[:, s:s + 1].double().numpy(), v[:, s:s + 1].double().numpy())
            compare(out[:, s:s + 1], orcs[s].attend(q[:, s:s + 1].double().numpy()))


def test_step_unsupported_layouts_are_refused():
    wl = WORKLOADS["qwen3b"].replace(n_layers=1, capacity=64)
    cache = make_cache(wl, layout="stored_rotated")
    q, k, v = step_inputs(wl, 1)
    from rolling_kv_cache_buffer_b300.rkv import RKV_ERR_UNSUPPORTED, RkvError
    with pytest.raises(RkvError) as e:
        cache.step(dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.bfloat16))
    assert e.value.status == RKV_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------
# Per-layer form of the step (rkv_step_layers), also under a CUDA graph
# ----------------------------------------------------------------------------

def _layer_calls(cache, kd, vd, qd, out, order, log=None):
    """One step as one rkv_step_layers call per layer, in `order`; the last
    call publishes."""
    for i, l in enumerate(order):
        cache.step_layers(l, kd[l:l + 1], vd[l:l + 1], qd[l:l + 1], out[l:l + 1],
                          last=(i == len(order) - 1), step_log=log)


@pytest.mark.parametrize("order", ["forward", "reverse"])
def test_step_layers_equals_step(order):
    """Per-layer calls (any order, the last one publishing) leave the same
    pools, states and logs as rkv_step, and outputs within float rounding of
    it (the two launch shapes split the windows differently)."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=4, capacity=128)
    whole = make_cache(wl)
    per = make_cache(wl)
    orc = make_oracle(wl)
    L = wl.n_layers
    seq = list(range(L)) if order == "forward" else list(reversed(range(L)))
    log_a = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    log_b = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    for t in range(1, 2 * wl.capacity + 10):
        q, k, v = step_inputs(wl, t)
        qd, kd, vd = dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16)
        a = whole.step(kd, vd, qd, step_log=log_a)
        b = torch.empty_like(a)
        # intermediate calls must leave the state alone
        st0 = per.state.clone()
        per.step_layers(seq[0], kd[seq[0]:seq[0] + 1], vd[seq[0]:seq[0] + 1],
                        qd[seq[0]:seq[0] + 1], b[seq[0]:seq[0] + 1], last=False)
        assert torch.equal(per.state, st0)
        _layer_calls(per, kd, vd, qd, b, seq[1:], log=log_b)
        orc.append(k.double().numpy(), v.double().numpy())
        assert torch.equal(log_a, log_b), f"step {t}"
        if t % 11 == 0 or t in (1, 2, 127, 128, 129):
            assert torch.allclose(a, b, atol=1e-5, rtol=0), f"step {t}"
            compare(b, orc.attend(q.double().numpy()))
    assert torch.equal(whole.k_pool, per.k_pool) and torch.equal(whole.v_pool, per.v_pool)
    assert torch.equal(whole.state, per.state)


def test_step_layers_in_a_cuda_graph():
    """A step's per-layer calls captured once in a CUDA graph and replayed
    every step (inputs copied into the graph's static buffers) give the same
    results as the same calls made eagerly."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=3, capacity=64)
    eager = make_cache(wl)
    graphed = make_cache(wl)
    L = wl.n_layers
    q0, k0, v0 = step_inputs(wl, 1)
    qs, ks, vs = dev(q0, torch.bfloat16), dev(k0, torch.bfloat16), dev(v0, torch.bfloat16)
    outs = torch.zeros(q0.shape, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _layer_calls(graphed, ks, vs, qs, outs, list(range(L)))   # warm-up (step 1)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _layer_calls(graphed, ks, vs, qs, outs, list(range(L)))
    e1 = torch.empty_like(outs)
    _layer_calls(eager, ks, vs, qs, e1, list(range(L)))           # eager step 1
    for t in range(2, 150):
        q, k, v = step_inputs(wl, t)
        qd, kd, vd = dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16)
        ref = torch.empty_like(outs)
        _layer_calls(eager, kd, vd, qd, ref, list(range(L)))
        qs.copy_(qd), ks.copy_(kd), vs.copy_(vd)
        g.replay()
        assert torch.equal(outs, ref), f"step {t}"
    assert torch.equal(eager.k_pool, graphed.k_pool) and torch.equal(eager.state, graphed.state)


def test_step_layers_bad_range():
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=64)
    cache = make_cache(wl)
    q, k, v = step_inputs(wl, 1)
    qd, kd, vd = dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    from rolling_kv_cache_buffer_b300 import RkvError
    with pytest.raises(RkvError):
        cache.step_layers(1, kd, vd, qd, out, last=True)      # layers 1..2 of 2


def test_step_layers_many_streams():
    """Per-layer calls over eight streams with fills 0 .. W and scattered
    origins (several units per CTA, split units merged through global
    partials): every stream's outputs against the oracle, states published by
    the last call only."""
    wl = WORKLOADS["qwen3b"].replace(n_streams=8, n_layers=3, capacity=256)
    fills = [0, 1, 5, 31, 32, 33, 200, 256]
    origins = [0, 7, 250, 1000, 77, 12345, 999_999, 256 * 9 + 3]
    cache = make_cache(wl)
    orcs = []
    for s in range(8):
        k = random_rows((3, 2, fills[s], 128), 700 + s, torch.bfloat16)
        v = random_rows((3, 2, fills[s], 128), 800 + s, torch.bfloat16)
        write_window(cache, s, origins[s], fills[s], k, v)
        orc = make_oracle(wl, n_streams=1)
        orc.set_state(0, origins[s], fills[s], k.double().numpy(), v.double().numpy())
        orcs.append(orc)
    for t in range(1, 4):
        q, k, v = step_inputs(wl, t)
        qd, kd, vd = dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16)
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        st0 = cache.state.clone()
        cache.step_layers(0, kd[0:2], vd[0:2], qd[0:2], out[0:2], last=False)
        assert torch.equal(cache.state, st0)
        cache.step_layers(2, kd[2:3], vd[2:3], qd[2:3], out[2:3], last=True)
        for s in range(8):
            orcs[s].append(k[:, s:s + 1].double().numpy(), v[:, s:s + 1].double().numpy())
            compare(out[:, s:s + 1], orcs[s].attend(q[:, s:s + 1].double().numpy()))
        o, f, _ = cache.get_stream_state()
        assert [int(x) for x in f] == [orcs[s].fill[0] for s in range(8)]
        assert [int(x) for x in o] == [orcs[s].origin[0] for s in range(8)]
