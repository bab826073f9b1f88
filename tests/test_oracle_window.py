"""Pins of the oracle's retained window smaller than its ring (CPU only).

The causal audio encoder of "audio8-asr-infinite-p150" ("At a glance") keeps a
sliding window of 750 frames; the ring that holds it has 768 slots (a whole
number of 32-slot blocks).  The window decides eviction, the ring decides the
slot: position p lives in slot p mod 768 while the oldest frames leave once
more than 750 are held.  Expected values come from closed forms and from
brute force over the whole history (the last 750 frames with absolute RoPE
positions), not from the oracle's own bookkeeping.
"""
import numpy as np
import pytest
from hypothesis import given, settings, strategies as st

from oracle import rkv_oracle as O

RNG = np.random.default_rng(750)


def test_encoder_window_closed_form():
    """Window 750 in 768 slots, four frames per step from an empty window:
    after step t the fill is min(4t, 750), the origin max(0, 4t - 750), the
    step's first frame sits in slot 4(t - 1) mod 768 and the step evicts
    max(0, 4t - 750) - max(0, 4(t - 1) - 750) frames."""
    o, n = 0, 0
    for t in range(1, 2001):
        bk = O.bookkeep(o, n, 4, 750, 768)
        assert bk.fill == min(4 * t, 750)
        assert bk.origin == max(0, 4 * t - 750)
        assert bk.first_slot == (4 * (t - 1)) % 768
        assert bk.evicted == max(0, 4 * t - 750) - max(0, 4 * (t - 1) - 750)
        assert bk.new_slots == [(4 * (t - 1) + j) % 768 for j in range(4)]
        o, n = bk.origin, bk.fill


def test_window_rejects():
    with pytest.raises(ValueError):
        O.bookkeep(0, 0, 1, 40, 32)            # more retained pairs than slots
    with pytest.raises(ValueError):
        O.bookkeep(0, 11, 1, 10, 16)           # fill above the window
    with pytest.raises(ValueError):
        O.RollingCacheOracle(1, 1, 2, 1, 8, 16, window=17)


@settings(max_examples=200, deadline=None)
@given(Wr=st.integers(1, 40), extra=st.integers(0, 24), o0=st.integers(0, 10 ** 9),
       cs=st.lists(st.integers(0, 40), min_size=1, max_size=25))
def test_window_invariants(Wr, extra, o0, cs):
    """Brute force: the window is the last min(len, Wr) inserted positions; the
    retained positions occupy distinct slots p mod (Wr + extra)."""
    W = Wr + extra
    hist = []
    o, n = o0, 0
    for c in cs:
        c = min(c, Wr)
        bk = O.bookkeep(o, n, c, Wr, W)
        hist += list(range(o0 + len(hist), o0 + len(hist) + c))
        keep = hist[-Wr:] if hist else []
        assert bk.fill == len(keep)
        assert bk.origin == (keep[0] if keep else o0)
        slots = [p % W for p in keep]
        assert len(set(slots)) == len(slots)
        o, n = bk.origin, bk.fill


@pytest.mark.parametrize("Wr,W,cs", [(10, 16, [3] * 9), (13, 32, [4, 1, 4, 4, 2, 4, 4, 4]),
                                     (7, 8, [1] * 20)])
def test_window_attention_is_brute_force_over_last_frames(Wr, W, cs):
    """Attention of every chunk over a window of Wr pairs kept in W slots equals
    brute force over the last Wr frames of the history with absolute
    positions (causal within the chunk)."""
    S, L, Hq, Hkv, D = 1, 2, 2, 2, 8
    origin = 31_337
    cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W, theta=1e6, window=Wr)
    cache.set_state(0, origin, 0)
    hk, hv = [], []
    for c in cs:
        k = RNG.standard_normal((L, S, c, Hkv, D))
        v = RNG.standard_normal((L, S, c, Hkv, D))
        q = RNG.standard_normal((L, S, c, Hq, D))
        cache.append(k, v)
        hk += [k[:, 0, j] for j in range(c)]
        hv += [v[:, 0, j] for j in range(c)]
        want = O.brute_force_window(np.array(hk), np.array(hv), q[:, 0], Wr, c, Hkv,
                                    theta=1e6, p0=origin)
        np.testing.assert_allclose(cache.attend(q)[:, 0], want, rtol=1e-9, atol=1e-11)
        assert cache.fill[0] == min(len(hk), Wr)


def test_window_mutation_is_caught(monkeypatch):
    """Eviction at the slot count instead of the window fails the closed form."""
    orig = O.bookkeep

    def at_slots(origin, fill, n_new, capacity, slots=None):
        return orig(origin, fill, n_new, slots or capacity, slots)

    monkeypatch.setattr(O, "bookkeep", at_slots)
    with pytest.raises(AssertionError):
        test_encoder_window_closed_form()
