"""rkv_attend_static_scratch against rkv_attend, through the C ABI (GPU).

rkv_attend_static_scratch is for callers that cannot allocate device memory
where they attend (a framework-owned memory pool, a plugin callback that
forbids allocation, a real-time loop): its split-softmax scratch lives in one
static device array owned by the library instead of the caller's workspace.
It runs the same kernels on the same grid as rkv_attend, so its output must be
bitwise equal to rkv_attend's, on two calls in a row (the array keeps the
previous call's contents); one case is also checked against the float64 oracle
within the tolerance of the other GPU tests.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test; it also passes alone.
"""
import numpy as np
import pytest
import torch

import rolling_kv_cache_buffer_b300 as R
from rkv_inputs import WORKLOADS, initial_window, random_rows, step_inputs
from tests.gpu_util import MAX_ABS, MEAN_ABS, compare, dev, make_cache, make_oracle, write_window

pytestmark = pytest.mark.gpu


def _static(cache, q, out):
    stream = torch.cuda.current_stream().cuda_stream
    R.rkv_attend_static_scratch(cache.handle, q.data_ptr(), out.data_ptr(), 0, q.shape[0],
                                q.shape[2], stream)


@pytest.mark.parametrize("wl_name,impl,c", [("qwen3b", "auto", 1), ("qwen3b", "fma", 1),
                                            ("audio8", "fma", 6)])
def test_static_scratch_matches_rkv_attend_on_two_calls(wl_name, impl, c):
    """Full windows at a large origin, so units are split across CTAs and the
    partials / tickets in the static array are exercised."""
    wl = WORKLOADS[wl_name].replace(n_new=c)
    cache = make_cache(wl, attend_impl=impl, max_chunk=c)
    k, v = initial_window(wl, 0, wl.capacity)
    write_window(cache, 0, 123_456, wl.capacity, k, v)
    for t in (1, 2):                    # two steps: two calls in a row each
        q, kn, vn = step_inputs(wl, t)
        cache.append(dev(kn, torch.bfloat16), dev(vn, torch.bfloat16))
        qd = dev(q, torch.bfloat16)
        ref = cache.attend(qd)
        for _ in range(2):
            out = torch.full(qd.shape, float("nan"), dtype=torch.float32, device="cuda")
            _static(cache, qd, out)
            torch.cuda.synchronize()
            assert torch.equal(out, ref)


def test_static_scratch_multi_stream_partial_windows():
    wl = WORKLOADS["qwen3b"].replace(n_streams=5, n_layers=3, capacity=512)
    cache = make_cache(wl)
    origins, fills = [0, 700, 12345, 99, 4], [512, 37, 300, 0, 511]
    for s in range(5):
        if fills[s]:
            kk = random_rows((3, 2, fills[s], 128), 10 + s, torch.bfloat16)
            vv = random_rows((3, 2, fills[s], 128), 20 + s, torch.bfloat16)
            write_window(cache, s, origins[s], fills[s], kk, vv)
    q = dev(random_rows((3, 5, 1, 16, 128), 3, torch.bfloat16), torch.bfloat16)
    ref = cache.attend(q)
    orc = make_oracle(wl)
    for s in range(5):
        kk = random_rows((3, 2, fills[s], 128), 10 + s, torch.bfloat16) if fills[s] else None
        vv = random_rows((3, 2, fills[s], 128), 20 + s, torch.bfloat16) if fills[s] else None
        orc.set_state(s, origins[s], fills[s], None if kk is None else kk.double().numpy(),
                      None if vv is None else vv.double().numpy())
    want = orc.attend(q.double().cpu().numpy())
    for _ in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        _static(cache, q, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        compare(out, want, MAX_ABS, MEAN_ABS)


def test_static_scratch_rejects_too_many_units():
    """64 streams x 36 layers x 8 KV heads need more merge tickets than the
    static array holds: rejected before anything is enqueued."""
    cache = R.RollingKV(64, 36, 8, 8, 64, 32)
    q = torch.zeros((36, 64, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(R.RkvError) as e:
        _static(cache, q, out)
    assert e.value.status == R.rkv.RKV_ERR_UNSUPPORTED


def test_static_scratch_rejects_the_chunked_36_layer_decoder():
    """The 6-token chunk of the 36-layer GQA decoder (G = 8, D = 128) needs
    2 * #SMs * 48 * 130 * 4 bytes of partials, more than the static array
    holds: rejected before anything is enqueued (rkv_attend serves it)."""
    wl = WORKLOADS["qwen3b_chunk6"]
    cache = make_cache(wl, max_chunk=6)
    q = torch.zeros((36, 1, 6, 16, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    with pytest.raises(R.RkvError) as e:
        _static(cache, q, out)
    assert e.value.status == R.rkv.RKV_ERR_UNSUPPORTED
