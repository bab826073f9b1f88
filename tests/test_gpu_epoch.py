"""Lazy (epoch) re-basing of stored-rotated keys on the GPU against the
oracle's EpochRotatedOracle, and the drift of stored keys compared across the
three key layouts."""
import numpy as np
import pytest
import torch

from oracle import rkv_oracle as O
from rkv_inputs import WORKLOADS, step_inputs
from rolling_kv_cache_buffer_b300 import RollingKV
from tests.gpu_util import compare, dev

pytestmark = pytest.mark.gpu


def _cache(wl, epoch, layout="stored_rotated", max_chunk=None, attend_impl="auto"):
    return RollingKV(wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                     wl.capacity, max_chunk=max_chunk or wl.n_new, kv_dtype=wl.kv_dtype,
                     layout=layout, rope_theta=wl.rope_theta, attend_impl=attend_impl,
                     rebase_epoch=epoch)


def _oracle(wl, epoch):
    return O.EpochRotatedOracle(wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads,
                                wl.head_dim, wl.capacity, theta=wl.rope_theta, epoch=epoch)


def _lag(cache):
    """Per-stream lag (int32 field 4 of each 32-byte state record)."""
    return cache.state.view(torch.int32)[: 8 * cache.S].view(cache.S, 8)[:, 4].cpu().numpy()


def _ulp(x):
    return np.ldexp(1.0, np.frexp(np.abs(x))[1] - 8)


@pytest.mark.parametrize("c,impl", [(1, "auto"), (3, "auto"), (1, "fma")])
def test_epoch_stream_matches_oracle(c, impl):
    """Append, re-base, attend for several epochs: bookkeeping and lag exact,
    outputs within tolerance of the oracle's epoch model."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=64, n_new=c)
    E = wl.capacity + 1 - c
    cache = _cache(wl, E, attend_impl=impl)
    orc = _oracle(wl, E)
    for t in range(1, 3 * wl.capacity // c + 5):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        cache.rebase()
        orc.append(k.double().numpy(), v.double().numpy())
        orc.rebase()
        o, f, st = cache.get_stream_state()
        assert st[0] == 0
        assert (int(o[0]), int(f[0])) == (orc.origin[0], orc.fill[0])
        assert int(_lag(cache)[0]) == orc.lag[0]
        out = cache.attend(dev(q, torch.bfloat16))
        if t % 9 == 0 or orc.lag[0] in (0, E - 1):
            compare(out, orc.attend(q.double().numpy()))


def test_epoch_append_and_rerotation_within_one_ulp():
    """Per call: a new key is stored as R(p - o_ref) k and the due re-base turns
    every retained key by R(-lag), each within one bf16 ulp of the float64
    rotation of the GPU's own inputs."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=1, capacity=32)
    E = 32
    cache = _cache(wl, E)
    W = wl.capacity
    checked = 0
    for t in range(1, 4 * W):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
        o, f, _ = cache.get_stream_state()
        lag = int(_lag(cache)[0])
        p = t - 1
        ref = int(o[0]) - lag
        got = cache.k_pool[0][:, :, p % W].double().cpu().numpy()
        want = O.bf16_round(O.rope(k[:, 0, 0].double().numpy(), p - ref, wl.rope_theta))
        assert np.all(np.abs(got - want) <= _ulp(want) + 1e-30)
        before = cache.k_pool.clone()
        cache.rebase()
        if lag >= E:
            slots = [(int(o[0]) + r) % W for r in range(int(f[0]))]
            src = before[0][:, :, slots].double().cpu().numpy()
            want = O.rerotate(src, lag, wl.rope_theta)
            got = cache.k_pool[0][:, :, slots].double().cpu().numpy()
            assert np.all(np.abs(got - want) <= _ulp(want) + 1e-30)
            assert int(_lag(cache)[0]) == 0
            checked += 1
    assert checked >= 2


def test_epoch_missed_rebase_is_flagged():
    wl = WORKLOADS["qwen3b"].replace(n_layers=1, capacity=32)
    cache = _cache(wl, 8)
    for t in range(1, 32 + 10):
        q, k, v = step_inputs(wl, t)
        cache.append(dev(k, torch.bfloat16), dev(v, torch.bfloat16))
    # evictions start at step 33; the ninth append after that finds lag 8 = E
    assert cache.get_stream_state()[2][0] == 5


def test_drift_of_stored_keys_across_layouts():
    """The pages' hazard measured on the kernels: a stream of 12 W tokens.
    Stored keys re-rotated at every eviction drift from the exact rotation of
    the input key; with an epoch E = W they stay within three bf16 roundings;
    the attention outputs follow.  Prints the numbers."""
    wl = WORKLOADS["audio8"].replace(n_layers=1, capacity=256)
    W = wl.capacity
    caches = {"pre_rope": _cache(wl, 0, layout="pre_rope"),
              "eager": _cache(wl, 0),
              "epoch": _cache(wl, W)}
    keys = {}
    T = 12 * W
    for t in range(1, T + 1):
        q, k, v = step_inputs(wl, t)
        kb, vb = dev(k, torch.bfloat16), dev(v, torch.bfloat16)
        for c in caches.values():
            c.append(kb, vb)
            c.rebase()
        keys[t - 1] = k[:, 0, 0].double().numpy()
        keys.pop(t - 1 - W, None)
    o, f, _ = caches["eager"].get_stream_state()
    origin = int(o[0])
    # stored-key error against the float64 rotation of each input key
    kerr = {}
    for name in ("eager", "epoch"):
        c = caches[name]
        ref = origin - int(_lag(c)[0])
        worst = 0.0
        for p, kk in keys.items():
            exact = O.rope(kk, p - ref, wl.rope_theta)
            got = c.k_pool[0][:, :, p % W].double().cpu().numpy()
            worst = max(worst, float(np.max(np.linalg.norm(got - exact, axis=-1) /
                                            np.linalg.norm(exact, axis=-1))))
        kerr[name] = worst
    # attention output error against the exact pre-RoPE oracle of the final window
    orc = O.RollingCacheOracle(1, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, W,
                               theta=wl.rope_theta)
    kw = np.stack([keys[p] for p in sorted(keys)], axis=2)
    vw = np.zeros_like(kw)
    vw[...] = np.stack([step_inputs(wl, p + 1)[2][:, 0, 0].double().numpy()
                        for p in sorted(keys)], axis=2)
    orc.set_state(0, origin, W, kw, vw)
    q, _, _ = step_inputs(wl, T + 7)
    want = orc.attend(q.double().numpy())
    oerr = {}
    for name, c in caches.items():
        out = c.attend(dev(q, torch.bfloat16)).double().cpu().numpy()
        oerr[name] = float(np.abs(out - want).max())
    print(f"\ndrift after {T} tokens, W={W}: stored-key rel. error eager {kerr['eager']:.4f} "
          f"epoch {kerr['epoch']:.4f}; output max-abs pre_rope {oerr['pre_rope']:.2e} "
          f"eager {oerr['eager']:.2e} epoch {oerr['epoch']:.2e}")
    assert kerr["epoch"] <= 3 * 2.0 ** -8
    assert kerr["eager"] > 2 * kerr["epoch"]
    assert oerr["epoch"] <= 2e-2 and oerr["pre_rope"] <= 2e-2


@pytest.mark.parametrize("style", ["split_half", "interleaved"])
def test_epoch_fused_step_matches_three_calls(style):
    """rkv_step on stored-rotated keys with an epoch (then rkv_rebase) against
    rkv_append + rkv_rebase + rkv_attend and the oracle's epoch model, across
    several due re-bases: states and lag equal, V pools equal, K pools within
    one bf16 ulp, outputs within tolerance."""
    wl = WORKLOADS["qwen3b"].replace(n_layers=2, capacity=64)
    E = wl.capacity
    kw = dict(layout="stored_rotated", rope_theta=wl.rope_theta, rebase_epoch=E,
              rope_style=style)
    fused = RollingKV(1, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.capacity, **kw)
    split = RollingKV(1, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.capacity, **kw)
    orc = O.EpochRotatedOracle(1, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                               wl.capacity, theta=wl.rope_theta, epoch=E, style=style)
    for t in range(1, 3 * wl.capacity + 5):
        q, k, v = step_inputs(wl, t)
        qd, kd, vd = dev(q, torch.bfloat16), dev(k, torch.bfloat16), dev(v, torch.bfloat16)
        a = fused.step(kd, vd, qd)
        fused.rebase()
        split.append(kd, vd)
        split.rebase()
        b = split.attend(qd)
        orc.append(k.double().numpy(), v.double().numpy())
        orc.rebase()
        assert torch.equal(fused.state, split.state), f"step {t}"
        assert int(_lag(fused)[0]) == orc.lag[0]
        if t % 7 == 0 or orc.lag[0] in (0, E - 1) or t < 4:
            ref = orc.attend(q.double().numpy())
            compare(a, ref)
            compare(b, ref)
    assert torch.equal(fused.v_pool, split.v_pool)
    kf = fused.k_pool.double().cpu().numpy()
    ks = split.k_pool.double().cpu().numpy()
    assert np.all(np.abs(kf - ks) <= _ulp(ks) + 1e-30)
