"""Pinned prefix slots on the GPU (through the C ABI).

A constant prefix (the audio-independent prompt prepared once and checked
again on every silence reset, "Reza2kn/Audio8-ASR-Infinite-Compressed",
"Linux CPU") goes into P pinned slots in front of the ring; appends roll the
ring behind it and never evict it.  The window reads as a re-prefill of
"prefix, then the retained tokens" ("audio8-asr-infinite-p150",
"Limitations"): prefix pair i at position i, retained token p at
npin + (p - origin).  Step logs must equal the oracle's bookkeeping bit for bit;
outputs must stay within max-abs 2e-2 / mean-abs 2e-3 of the float64 oracle.
"""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, random_rows, step_inputs
from rolling_kv_cache_buffer_b300 import RollingKV
from tests.gpu_util import compare, dev

pytestmark = pytest.mark.gpu


def _pair(wl, layout, P, window=None, impl="auto", max_chunk=None, style="split_half"):
    kw = dict(max_chunk=max_chunk or wl.n_new, kv_dtype=wl.kv_dtype, layout=layout,
              rope_style=style, rope_theta=wl.rope_theta, attend_impl=impl,
              window=window or 0, n_pinned=P)
    cache = RollingKV(wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                      wl.capacity, **kw)
    cls = O.StoredRotatedOracle if layout == "stored_rotated" else O.RollingCacheOracle
    orc = cls(wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.capacity,
              theta=wl.rope_theta, style=style, window=window, n_pinned=P)
    return cache, orc


def _reset(cache, orc, wl, s, origin, n, seed):
    k = random_rows((wl.n_layers, n, wl.n_kv_heads, wl.head_dim), seed, torch.bfloat16)
    v = random_rows((wl.n_layers, n, wl.n_kv_heads, wl.head_dim), seed + 1, torch.bfloat16)
    cache.reset_stream(s, origin, dev(k, torch.bfloat16), dev(v, torch.bfloat16))
    kk = k.permute(0, 2, 1, 3).double().numpy()        # [L][H_kv][n][D]
    vv = v.permute(0, 2, 1, 3).double().numpy()
    orc.reset(s, origin, kk, vv, n)
    return k, v


@pytest.mark.parametrize("layout,path", [("pre_rope", "calls"), ("pre_rope", "fused"),
                                         ("stored_rotated", "calls")])
def test_pinned_decode_through_wraps(layout, path):
    """Decoder shape cut to 2 layers (8 heads x 64, W 1024 with 64 pinned slots,
    a ring of 960): a 40-pair prefix, then 2100 single tokens -- past the fill,
    the first eviction and two trips around the ring.  Logs every step,
    outputs at sampled steps, prefix slots unchanged at the end."""
    wl = WORKLOADS["audio8"].replace(n_layers=2)
    P = 64
    cache, orc = _pair(wl, layout, P)
    k_pre, v_pre = _reset(cache, orc, wl, 0, 1000, 40, 11)
    pool_k0 = cache.k_pool[0, :, :, :P].clone()
    pool_v0 = cache.v_pool[0, :, :, :P].clone()
    log = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    check = {1, 2, 900, 959, 960, 961, 1500, 1919, 1920, 1921, 2100}
    for t in range(1, 2101):
        q, k, v = step_inputs(wl, t)
        kd, vd, qd = dev(k, torch.bfloat16), dev(v, torch.bfloat16), dev(q, torch.bfloat16)
        want_log = orc.append(k.double().numpy(), v.double().numpy())[0]
        if layout == "stored_rotated":
            orc.rebase()
        if path == "fused":
            out = cache.step(kd, vd, qd, step_log=log)
        else:
            cache.append(kd, vd, step_log=log)
            cache.rebase()
            out = cache.attend(qd) if t in check else None
        assert tuple(log[0].tolist()) == tuple(want_log), f"step {t}"
        if t in check:
            compare(out, orc.attend(q.double().numpy()))
    # The pinned slots were never written after the reset.
    assert torch.equal(cache.k_pool[0, :, :, :P], pool_k0)
    assert torch.equal(cache.v_pool[0, :, :, :P], pool_v0)
    assert torch.equal(cache.v_pool[0, :, :, :40].cpu(), v_pre.permute(0, 2, 1, 3).to(torch.bfloat16))


@pytest.mark.parametrize("impl,c", [("auto", 4), ("fma", 2), ("auto", 6)])
def test_pinned_chunks_gqa(impl, c):
    """GQA 16/2 x 128 cut to 3 layers, W 512 with 32 pinned slots: a 20-pair
    prefix, then chunks of c tokens through eviction and wrap (the chunk
    kernel, or the CUDA-core kernel)."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=3, capacity=512, n_new=c)
    cache, orc = _pair(wl, "pre_rope", 32, impl=impl, max_chunk=c)
    _reset(cache, orc, wl, 0, 77, 20, 21)
    n_steps = 1200 // c
    check = {1, 2, 480 // c, 480 // c + 1, n_steps // 2, n_steps}
    for t in range(1, n_steps + 1):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if t in check:
            out = cache.attend(dev(q, torch.bfloat16))
            compare(out, orc.attend(q.double().numpy()))


def test_pinned_window_and_poison():
    """Pinned slots together with a retained window below the ring (64 pinned
    slots, a ring of 960, a window of 900), three streams with prefixes of 64,
    1 and 0 pairs, every slot outside the prefix and the window poisoned with
    NaN before each attend."""
    wl = WORKLOADS["audio8"].replace(n_layers=2, n_streams=3)
    P, Wr = 64, 900
    cache, orc = _pair(wl, "pre_rope", P, window=Wr)
    for s, (origin, n) in enumerate([(5, 64), (123_456, 1), (999, 0)]):
        _reset(cache, orc, wl, s, origin, n, 30 + 2 * s)
    npre = [64, 1, 0]
    for t in range(1, 1001):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        orc.append(k.double().numpy(), v.double().numpy())
        if t in (1, 899, 900, 901, 1000):
            o, f, st = cache.get_stream_state()
            assert list(f) == [min(t, Wr)] * 3 and list(st) == [0, 0, 0]
            ring = cache.W - P
            for s in range(3):
                keep = torch.zeros(cache.W, dtype=torch.bool)
                keep[:npre[s]] = True
                keep[P + (torch.arange(int(f[s])) + int(o[s])) % ring] = True
                bad = (~keep).nonzero().flatten().cuda()
                cache.k_pool[s][:, :, bad] = float("nan")
                cache.v_pool[s][:, :, bad] = float("nan")
            compare(cache.attend(dev(q, torch.bfloat16)), orc.attend(q.double().numpy()))


def test_pinned_config_rejects():
    import rolling_kv_cache_buffer_b300 as R
    for kw, st in [(dict(n_pinned=40), R.rkv.RKV_ERR_INVALID_ARG),     # not a multiple of 32
                   (dict(n_pinned=1024), R.rkv.RKV_ERR_INVALID_ARG),   # no ring left
                   (dict(n_pinned=64, window=961), R.rkv.RKV_ERR_INVALID_ARG),
                   (dict(n_pinned=64, layout="stored_rotated", rebase_epoch=64),
                    R.rkv.RKV_ERR_UNSUPPORTED)]:
        with pytest.raises(R.RkvError) as e:
            RollingKV(1, 1, 8, 8, 64, 1024, **kw)
        assert e.value.status == st
    cache = RollingKV(1, 1, 8, 8, 64, 1024, n_pinned=64)
    k = torch.zeros((1, 65, 8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(R.RkvError):
        cache.reset_stream(0, 0, k, k)
