"""Pins of the stored-rotated oracles' ``set_state`` (CPU only).

``set_state`` seeds a window (a reset with a prefix, or a benchmark's steady
state) in the two stored-rotated models.  The keys it receives are unrotated;
"Audio8 ASR Infinite: What It Actually Takes to Listen Forever" ("Inside the
Rolling KV Cache and Exact RoPE Re-Basing") places every retained key at its
position from the new zero, so the key at absolute position origin + i must be
stored as bf16(R(i) k_i).  The expected values here come from complex-number
rotation and torch's bf16 conversion, not from the oracle's ``rope`` or
``bf16_round``; the window's attention is checked against brute force over the
history "prefix, then the appended tokens".
"""
import numpy as np
import pytest
import torch

import oracle as O

RNG = np.random.default_rng(20261203)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _rot(x, pos, style, theta=1e6):
    """RoPE as complex multiplication: pair i is (x_i, x_{i+D/2}) split-half or
    (x_{2i}, x_{2i+1}) interleaved, turned by pos * theta^(-2i/D)."""
    D = x.shape[-1]
    w = theta ** (-(2.0 * np.arange(D // 2)) / D)
    if style == O.SPLIT_HALF:
        z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * pos * w)
        return np.concatenate([z.real, z.imag], axis=-1)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * pos * w)
    y = np.empty(x.shape)
    y[..., 0::2], y[..., 1::2] = z.real, z.imag
    return y


def _ulp(x):
    return np.ldexp(1.0, np.frexp(np.abs(x))[1] - 8)


def _make(kind, S, L, Hq, Hkv, D, W, style):
    if kind == "stored":
        return O.StoredRotatedOracle(S, L, Hq, Hkv, D, W, style=style)
    return O.EpochRotatedOracle(S, L, Hq, Hkv, D, W, style=style, epoch=W)


@pytest.mark.parametrize("kind", ["stored", "epoch"])
@pytest.mark.parametrize("style", [O.SPLIT_HALF, O.INTERLEAVED])
@pytest.mark.parametrize("origin,n", [(987_654, 11), (0, 16), (5, 0), (123, 1)])
def test_set_state_stores_keys_rotated_from_the_new_origin(kind, style, origin, n):
    """Key i of the seeded window (absolute position origin + i) is stored as
    bf16(R(i) k_i): representable in bf16, within one bf16 ulp of the
    complex rotation rounded by torch, and equal to it almost everywhere (the
    two float64 rotations differ by ~1e-16, which can flip a rounding tie);
    values are stored unchanged; the lag of the epoch model starts at 0."""
    L, Hkv, D, W = 2, 2, 16, 16
    o = _make(kind, 2, L, 4, Hkv, D, W, style)
    o.append(np.ones((L, 2, 3, Hkv, D)), np.ones((L, 2, 3, Hkv, D)))   # old contents
    k = _bf16(RNG.standard_normal((L, Hkv, n, D)))
    v = _bf16(RNG.standard_normal((L, Hkv, n, D)))
    o.set_state(1, origin, n, k, v)
    assert o.retained_positions(1) == [origin + i for i in range(n)]
    assert (o.origin[1], o.fill[1]) == (origin, n)
    assert o.fill[0] == 3                                   # the other stream is untouched
    assert (o.lag[1] if kind == "epoch" else o.pending[1]) == 0
    exact = 0
    for i, p in enumerate(o.retained_positions(1)):
        got, gv = o.window[1][p]
        want = _bf16(_rot(k[:, :, i], i, style))
        np.testing.assert_array_equal(_bf16(got), got)      # a bf16 value
        assert np.all(np.abs(got - want) <= _ulp(want)), (i, p)
        exact += int(np.sum(got == want))
        np.testing.assert_array_equal(gv, v[:, :, i])
    assert exact >= 0.99 * max(1, n * L * Hkv * D) or n == 0


@pytest.mark.parametrize("kind", ["stored", "epoch"])
@pytest.mark.parametrize("n_prefix,cs", [(5, [1] * 14), (8, [2, 3, 1, 3, 2]), (3, [3] * 5)])
def test_stored_reset_with_prefix_is_a_new_history(kind, n_prefix, cs):
    """A reset with a prefix in a stored-rotated model: every later step's
    attention equals brute force (float64, exact rotation, no rounding of the
    stored keys) over the history "prefix, then the appended tokens" from the
    new origin, within the bf16 rounding of the stored keys; the prefix is the
    oldest part of the window and the first to be evicted."""
    S, L, Hq, Hkv, D, W = 1, 2, 4, 2, 32, 8
    origin = 4_321
    o = _make(kind, S, L, Hq, Hkv, D, W, O.SPLIT_HALF)
    o.append(_bf16(RNG.standard_normal((L, S, 3, Hkv, D))),
             _bf16(RNG.standard_normal((L, S, 3, Hkv, D))))
    if kind == "stored":
        o.rebase()
    kp = _bf16(RNG.standard_normal((L, Hkv, n_prefix, D)))
    vp = _bf16(RNG.standard_normal((L, Hkv, n_prefix, D)))
    o.set_state(0, origin, n_prefix, kp, vp)
    hk = [kp[:, :, i] for i in range(n_prefix)]
    hv = [vp[:, :, i] for i in range(n_prefix)]
    worst = 0.0
    for c in cs:
        k = _bf16(RNG.standard_normal((L, S, c, Hkv, D)))
        v = _bf16(RNG.standard_normal((L, S, c, Hkv, D)))
        q = _bf16(RNG.standard_normal((L, S, c, Hq, D)))
        o.append(k, v)
        o.rebase()
        hk += [k[:, 0, j] for j in range(c)]
        hv += [v[:, 0, j] for j in range(c)]
        want = O.brute_force_window(np.array(hk), np.array(hv), q[:, 0], W, c, Hkv,
                                    theta=1e6, p0=origin)
        worst = max(worst, float(np.abs(o.attend(q)[:, 0] - want).max()))
    assert worst < 5e-2
    assert o.origin[0] == origin + max(0, len(hk) - W)
