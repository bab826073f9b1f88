"""Pins of the oracle's pinned prefix (CPU only).

A constant prefix -- the audio-independent prompt that the CPU runtime of
"Reza2kn/Audio8-ASR-Infinite-Compressed" prepares once and checks again on
every silence reset ("Linux CPU") -- sits in slots that no append evicts,
while the ring behind it rolls.  The positions follow a re-prefill of the
window ("audio8-asr-infinite-p150", "Limitations": the rolling context is
rebuilt by re-prefilling the window): prefix, then the retained tokens,
numbered from 0.  Expected values come from brute force over that explicit
sequence, from closed-form bookkeeping, and from complex-number rotation with
torch's bf16 rounding.
"""
import numpy as np
import pytest
import torch

import oracle as O

RNG = np.random.default_rng(4242)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _rot(x, pos, theta=1e6):
    D = x.shape[-1]
    w = theta ** (-(2.0 * np.arange(D // 2)) / D)
    z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * pos * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def _run(cls, P, W, Wr, n_pre, cs, rnd=lambda a: a, tol=1e-9):
    S, L, Hq, Hkv, D = 1, 2, 4, 2, 16
    o = cls(S, L, Hq, Hkv, D, W, window=Wr, n_pinned=P)
    o.append(rnd(RNG.standard_normal((L, S, 2, Hkv, D))), rnd(RNG.standard_normal((L, S, 2, Hkv, D))))
    kp = rnd(RNG.standard_normal((L, Hkv, n_pre, D)))
    vp = rnd(RNG.standard_normal((L, Hkv, n_pre, D)))
    origin = 55_555
    o.reset(0, origin, kp, vp, n_pre)
    pre_k = np.moveaxis(kp, 2, 0)
    pre_v = np.moveaxis(vp, 2, 0)
    hk, hv, worst = [], [], 0.0
    for c in cs:
        k = rnd(RNG.standard_normal((L, S, c, Hkv, D)))
        v = rnd(RNG.standard_normal((L, S, c, Hkv, D)))
        q = rnd(RNG.standard_normal((L, S, c, Hq, D)))
        logs = o.append(k, v)
        if hasattr(o, "rebase"):
            o.rebase()
        t0 = len(hk)
        hk += [k[:, 0, j] for j in range(c)]
        hv += [v[:, 0, j] for j in range(c)]
        # bookkeeping of the rolling part, slots after the pinned ones
        assert logs[0][3] == P + (origin + t0) % (W - P)
        assert o.fill[0] == min(len(hk), Wr) and o.origin[0] == origin + max(0, len(hk) - Wr)
        assert o.n_prefix(0) == n_pre
        want = O.brute_force_reprefill(pre_k, pre_v, np.array(hk), np.array(hv), q[:, 0], Wr,
                                       c, Hkv)
        err = float(np.abs(o.attend(q)[:, 0] - want).max())
        worst = max(worst, err)
        assert err <= tol, (len(hk), err)
    return o, worst


@pytest.mark.parametrize("P,W,Wr,n_pre,cs", [
    (8, 24, 16, 5, [1] * 40),            # prefix shorter than its slots, single tokens
    (8, 24, 12, 8, [3, 1, 4, 4, 2, 4] * 5),
    (4, 12, 8, 0, [2] * 12),             # no prefix at all
])
def test_pinned_prefix_is_a_reprefill(P, W, Wr, n_pre, cs):
    """Every step's attention equals brute force over "prefix, then the last
    W_r tokens" numbered from 0 (float64, 1e-9), through fill, eviction and
    several trips around the ring; the prefix is never evicted."""
    _run(O.RollingCacheOracle, P, W, Wr, n_pre, cs)


def test_pinned_stored_rotated_within_bf16():
    """Stored-rotated keys with a pinned prefix: within the bf16 rounding of
    the stored keys of the same brute force; prefix keys stay exactly
    bf16(R(i) k_i) through every re-rotation of the ring."""
    o, worst = _run(O.StoredRotatedOracle, 8, 24, 16, 6, [1, 2, 3] * 12, rnd=_bf16, tol=5e-2)
    assert worst > 0.0


def test_pinned_prefix_keys_are_rotated_once():
    S, L, Hkv, D = 1, 1, 1, 16
    o = O.StoredRotatedOracle(S, L, 2, Hkv, D, 24, n_pinned=8)
    kp = _bf16(RNG.standard_normal((L, Hkv, 6, D)))
    o.reset(0, 10, kp, kp, 6)
    for _ in range(50):
        kv = _bf16(RNG.standard_normal((L, S, 1, Hkv, D)))
        o.append(kv, kv)
        o.rebase()
    for i, (kk, _) in enumerate(o.prefix[0]):
        want = _bf16(_rot(kp[:, :, i], i))
        assert np.all(np.abs(kk - want) <= np.ldexp(1.0, np.frexp(np.abs(want))[1] - 8))
        np.testing.assert_array_equal(_bf16(kk), kk)


def test_pinned_rejects():
    with pytest.raises(ValueError):
        O.RollingCacheOracle(1, 1, 2, 1, 8, 16, n_pinned=16)
    with pytest.raises(ValueError):
        O.RollingCacheOracle(1, 1, 2, 1, 8, 16, n_pinned=8, window=9)
    o = O.RollingCacheOracle(1, 1, 2, 1, 8, 16, n_pinned=4)
    with pytest.raises(ValueError):
        o.reset(0, 0, np.zeros((1, 1, 5, 8)), np.zeros((1, 1, 5, 8)), 5)
    with pytest.raises(ValueError):
        O.EpochRotatedOracle(1, 1, 2, 1, 8, 16, n_pinned=4, epoch=4)


def test_pinned_mutations_are_caught(monkeypatch):
    """Retained keys placed at p - origin (the prefix's length forgotten), and a
    prefix that the ring evicts, each fail the brute-force pin."""
    class Forgot(O.RollingCacheOracle):
        """Retained tokens and queries re-based from 0 instead of npin."""
        def _attend(self, q, layer_begin, absolute):
            q = np.asarray(q, np.float64)
            out = np.zeros_like(q)
            pos = np.array(self.retained_positions(0), dtype=np.int64)
            npin, n = self.n_prefix(0), len(pos)
            r = np.concatenate([np.arange(npin), pos - self.origin[0]])
            for l in range(q.shape[0]):
                for h in range(self.Hq):
                    g = h // self.G
                    pairs = list(self.prefix[0]) + [self.window[0][p] for p in pos]
                    K = O.rope(np.stack([kv[0][l, g] for kv in pairs]), r, self.theta)
                    V = np.stack([kv[1][l, g] for kv in pairs])
                    for j in range(q.shape[2]):
                        pq = self.origin[0] + n - q.shape[2] + j
                        vis = np.concatenate([np.ones(npin, bool), pos <= pq])
                        qr = O.rope(q[l, 0, j, h], pq - self.origin[0], self.theta)
                        out[l, 0, j, h] = O.softmax_attention(qr, K[vis], V[vis], self.scale)
            return out

    with pytest.raises(AssertionError):
        _run(Forgot, 8, 24, 16, 5, [1] * 20)

    class Evicting(O.RollingCacheOracle):
        def reset(self, s, origin, k=None, v=None, n=0):
            self.set_state(s, origin, n, k, v)      # prefix in the rolling window

        def n_prefix(self, s):
            return getattr(self, "_n", 0)

    with pytest.raises(AssertionError):
        _run(Evicting, 8, 24, 16, 5, [1] * 20)
