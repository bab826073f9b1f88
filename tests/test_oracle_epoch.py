"""Pins of the oracle's lazy (epoch) re-basing model for stored-rotated keys
(CPU only).  The expected values are built here from other routines than the
oracle's own: complex-number rotation for RoPE, torch's bf16 conversion for
rounding, and closed-form bookkeeping (one token per step from an empty
stream: origin = max(0, t - W), one eviction per step once full)."""
import math

import numpy as np
import pytest
import torch
from hypothesis import given, settings, strategies as st

import oracle as O

RNG = np.random.default_rng(20261202)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _rot(x, pos, theta=1e6):
    """Split-half RoPE as complex multiplication: pair (x_i, x_{i+D/2})."""
    D = x.shape[-1]
    w = theta ** (-(2.0 * np.arange(D // 2)) / D)
    z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * pos * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def _ulp(x):
    return np.ldexp(1.0, np.frexp(np.abs(x))[1] - 8)


@pytest.mark.parametrize("W,E", [(8, 5), (16, 16), (8, 2)])
def test_epoch_storage_follows_the_lag(W, E):
    """Every stored key equals its own history: bf16(R(p - o_ref) k) when it
    was inserted, then one bf16(R(-lag) .) per re-base it lived through; the
    lag grows by one per eviction and returns to 0 at each re-base."""
    D = 8
    o = O.EpochRotatedOracle(1, 1, 2, 1, D, W, epoch=E)
    hist = {}          # p -> expected stored key (float64)
    lag = 0
    for t in range(1, 6 * W):
        k = _bf16(RNG.standard_normal((1, 1, 1, 1, D)))
        v = _bf16(RNG.standard_normal((1, 1, 1, 1, D)))
        o.append(k, v)
        origin = max(0, t - W)
        e = 1 if t > W else 0
        lag += e
        p = t - 1
        hist[p] = _bf16(_rot(k[0, 0, 0, 0], p - (origin - lag)))
        hist.pop(p - W, None)
        o.rebase()
        if lag >= E:
            for q in hist:
                hist[q] = _bf16(_rot(hist[q], -lag))
            lag = 0
        assert o.origin[0] == origin and o.lag[0] == lag
        assert sorted(hist) == o.retained_positions(0)
        for q, want in hist.items():
            got = o.window[0][q][0][0, 0]
            # the two rotations agree to ~1e-16; allow the rare flipped rounding
            assert np.all(np.abs(got - want) <= _ulp(want)), (t, q)


def test_epoch_attention_matches_pre_rope():
    """Attention over epoch-rotated keys equals the plain pre-RoPE attention up
    to the bf16 rounding of the stored keys, across several re-bases."""
    S, L, Hq, Hkv, D, W = 1, 1, 4, 2, 64, 16
    a = O.RollingCacheOracle(S, L, Hq, Hkv, D, W)
    b = O.EpochRotatedOracle(S, L, Hq, Hkv, D, W, epoch=W)
    errs = []
    for t in range(5 * W):
        k = _bf16(RNG.standard_normal((L, S, 1, Hkv, D)))
        v = _bf16(RNG.standard_normal((L, S, 1, Hkv, D)))
        q = _bf16(RNG.standard_normal((L, S, 1, Hq, D)))
        a.append(k, v)
        b.append(k, v)
        b.rebase()
        errs.append(np.abs(a.attend(q) - b.attend(q)).max())
    assert max(errs) < 5e-2
    assert b.lag[0] < W


def test_epoch_missed_rebase_is_an_error():
    o = O.EpochRotatedOracle(1, 1, 2, 1, 8, 8, epoch=2)
    for _ in range(10):
        kv = _bf16(RNG.standard_normal((1, 1, 1, 1, 8)))
        o.append(kv, kv)
    with pytest.raises(RuntimeError):
        o.append(kv, kv)


def test_epoch_bounds_the_drift_of_stored_keys():
    """The pages' hazard, on the oracle: after many evictions, keys re-rotated
    at every eviction have been rounded up to W times; with an epoch E = W a
    key is rounded at most three times (insert + two re-bases).  bf16 keeps 8
    significant bits, so each rounding moves a key by at most 2^-8 of its norm:
    the lazy keys stay within 3 * 2^-8 of the exact rotation, the eager ones
    drift further."""
    D, W = 64, 32
    eager = O.StoredRotatedOracle(1, 1, 2, 1, D, W)
    lazy = O.EpochRotatedOracle(1, 1, 2, 1, D, W, epoch=W)
    raw = {}
    for t in range(8 * W):
        k = _bf16(RNG.standard_normal((1, 1, 1, 1, D)))
        eager.append(k, k)
        eager.rebase()
        lazy.append(k, k)
        lazy.rebase()
        raw[t] = k[0, 0, 0, 0]

    def err(model, ref):
        worst = 0.0
        for p in model.retained_positions(0):
            exact = _rot(raw[p], p - ref)
            got = model.window[0][p][0][0, 0]
            worst = max(worst, float(np.linalg.norm(got - exact) / np.linalg.norm(exact)))
        return worst
    e_eager = err(eager, eager.origin[0])
    e_lazy = err(lazy, lazy.o_ref(0))
    assert e_lazy <= 3 * 2.0 ** -8
    assert e_eager > 4 * e_lazy



@settings(max_examples=40, deadline=None)
@given(W=st.sampled_from([8, 16, 32]), c=st.integers(1, 3), data=st.data())
def test_epoch_lag_and_positions_stay_bounded(W, c, data):
    """For any epoch E with E + c <= W + 1: after an append the lag is below
    E + c, every stored position p - o_ref lies in [0, 2W) (the RoPE table's
    rows), and a re-base leaves the lag below E; bookkeeping is the plain one."""
    E = data.draw(st.integers(2, W + 1 - c))
    steps = data.draw(st.integers(1, 5 * W // c))
    o = O.EpochRotatedOracle(1, 1, 2, 1, 4, W, epoch=E)
    origin, fill = 0, 0
    for _ in range(steps):
        kv = np.zeros((1, 1, c, 1, 4))
        o.append(kv, kv)
        bk = O.bookkeep(origin, fill, c, W)
        origin, fill = bk.origin, bk.fill
        assert (o.origin[0], o.fill[0]) == (origin, fill)
        assert 0 <= o.lag[0] < E + c
        ref = o.o_ref(0)
        assert all(0 <= p - ref < 2 * W for p in o.retained_positions(0))
        o.rebase()
        assert o.lag[0] < E
