"""Pins of the float64 oracle against things other than itself (CPU only).

Each test names what fixes the expected value: a closed form, a library
routine, a textbook special case, brute force, or an invariant stated on
"Audio8 ASR Infinite: What It Actually Takes to Listen Forever"
("Inside the Rolling KV Cache and Exact RoPE Re-Basing").
"""

import math

import numpy as np
import pytest
import torch
from hypothesis import given, settings, strategies as st

from oracle import rkv_oracle as O

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------
# bf16 rounding: pinned to torch's float32 -> bfloat16 conversion (RNE)
# ----------------------------------------------------------------------------

def _torch_bf16(x32):
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_round_matches_torch_random():
    x = (RNG.standard_normal(200000) * np.exp(RNG.uniform(-30, 30, 200000))).astype(np.float32)
    np.testing.assert_array_equal(O.bf16_round(x.astype(np.float64)), _torch_bf16(x))


def test_bf16_round_ties_subnormals_overflow():
    # exact ties: 1 + 2^-8 (between 1 and 1+2^-7) -> even -> 1; 1 + 3*2^-8 -> 1 + 2^-6
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 + 2 ** -134,
                     3 * 2 ** -134, 2 ** -140, 0.0, -0.0, 3.3895e38, 3.4e38, -3.4e38,
                     np.float32(3.3961775e38)], dtype=np.float32)
    np.testing.assert_array_equal(O.bf16_round(ties.astype(np.float64)), _torch_bf16(ties))
    assert O.bf16_round(np.array([1 + 2 ** -8]))[0] == 1.0
    assert O.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert np.isinf(O.bf16_round(np.array([3.4e38]))[0])


# ----------------------------------------------------------------------------
# Bookkeeping: closed form of the tiny workload and invariants
# ----------------------------------------------------------------------------

def test_bookkeeping_closed_form_tiny():
    """Capacity 32, one token per step: after step t the fill is min(t, 32),
    the origin max(0, t - 32), the new token sits in slot (t - 1) mod 32 and
    from step 33 on position t - 33 is evicted."""
    o, n = 0, 0
    for t in range(1, 201):
        bk = O.bookkeep(o, n, 1, 32)
        assert bk.fill == min(t, 32)
        assert bk.origin == max(0, t - 32)
        assert bk.first_slot == (t - 1) % 32
        assert bk.new_positions == [t - 1]
        assert bk.evicted_positions == ([t - 33] if t >= 33 else [])
        assert bk.log() == (max(0, t - 32), min(t, 32), int(t >= 33), (t - 1) % 32)
        o, n = bk.origin, bk.fill


def test_bookkeeping_rejects():
    with pytest.raises(ValueError):
        O.bookkeep(0, 0, 33, 32)
    with pytest.raises(ValueError):
        O.bookkeep(0, 33, 1, 32)
    with pytest.raises(ValueError):
        O.bookkeep(-1, 0, 1, 32)


@settings(max_examples=300, deadline=None)
@given(W=st.integers(1, 64), o0=st.integers(0, 10 ** 9), n0=st.integers(0, 64),
       cs=st.lists(st.integers(0, 64), min_size=1, max_size=30))
def test_bookkeeping_invariants(W, o0, n0, cs):
    """Brute force: keep the list of every position ever inserted; the window
    is its last min(len, W) entries (FIFO), so fill <= W, the retained
    positions are contiguous from the origin and their slots are distinct."""
    n0 = min(n0, W)
    hist = list(range(o0, o0 + n0))
    o, n = o0, n0
    for c in cs:
        c = min(c, W)
        bk = O.bookkeep(o, n, c, W)
        before = hist[-n:] if n else []
        hist.extend(range(o + n, o + n + c))
        window = hist[-min(len(hist), W):] if hist else []
        # window recomputed by brute force from the full history
        assert bk.fill == len(window) <= W
        assert bk.origin == (window[0] if window else o)
        assert bk.evicted_positions == [p for p in before if p not in window]
        assert bk.new_positions == window[len(window) - c:] if c else bk.new_positions == []
        assert len({p % W for p in window}) == len(window)
        assert bk.evicted == max(0, n + c - W)
        o, n = bk.origin, bk.fill


# ----------------------------------------------------------------------------
# RoPE: closed forms, complex-number rotation, relative property
# ----------------------------------------------------------------------------

def test_inv_freq_closed_form():
    w = O.inv_freq(128, 1e6)
    assert w[0] == 1.0
    assert math.isclose(w[32], 1e-3, rel_tol=1e-14)        # 1e6^(-64/128)
    assert math.isclose(w[16], 10 ** -1.5, rel_tol=1e-14)   # 1e6^(-32/128)
    np.testing.assert_allclose(np.diff(np.log(w)), -2 * math.log(1e6) / 128, rtol=1e-12)
    w64 = O.inv_freq(64, 1e6)
    assert math.isclose(w64[16], 1e-3, rel_tol=1e-14)


@pytest.mark.parametrize("D", [2, 8, 64, 128])
def test_rope_split_half_is_complex_multiplication(D):
    """rotate_half convention: pair (x_i, x_{i+D/2}) is the complex number
    x_i + 1j*x_{i+D/2}, multiplied by exp(1j * pos * theta^(-2i/D))."""
    x = RNG.standard_normal((5, D))
    pos = np.array([0, 1, 7, 4095, 999999])
    z = x[:, : D // 2] + 1j * x[:, D // 2:]
    freq = np.array([1e6 ** (-(2.0 * i) / D) for i in range(D // 2)])
    zr = z * np.exp(1j * pos[:, None] * freq[None, :])
    want = np.concatenate([zr.real, zr.imag], axis=1)
    # angles reach 1e6 rad: one ulp of the frequency moves them by ~1e-10
    np.testing.assert_allclose(O.rope(x, pos, 1e6), want, rtol=1e-9, atol=1e-9)


def test_rope_d2_rotation_matrix():
    """D = 2: the single frequency is 1, so R(r) is the plane rotation by r rad."""
    x = np.array([0.3, -1.7])
    for r in [0, 1, 2, -3, 100]:
        R = np.array([[math.cos(r), -math.sin(r)], [math.sin(r), math.cos(r)]])
        np.testing.assert_allclose(O.rope(x, r, 1e6), R @ x, rtol=1e-13, atol=1e-13)


def test_rope_interleaved_is_permuted_split_half():
    D = 16
    x = RNG.standard_normal((3, D))
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])  # (2i,2i+1) -> (i,i+D/2)
    pos = np.array([3, 50, 1000])
    y_int = O.rope(x, pos, 1e4, O.INTERLEAVED)
    y_split = O.rope(x[:, perm], pos, 1e4, O.SPLIT_HALF)
    inv = np.argsort(perm)
    np.testing.assert_allclose(y_int, y_split[:, inv], rtol=1e-12, atol=1e-12)
    assert not np.allclose(y_int, O.rope(x, pos, 1e4, O.SPLIT_HALF))


@pytest.mark.parametrize("style", [O.SPLIT_HALF, O.INTERLEAVED])
def test_rope_invariants(style):
    x = RNG.standard_normal((4, 128))
    np.testing.assert_array_equal(O.rope(x, 0, 1e6, style), x)                      # r = 0
    np.testing.assert_allclose(np.linalg.norm(O.rope(x, 12345, 1e6, style), axis=1),
                               np.linalg.norm(x, axis=1), rtol=1e-13)               # |R k| = |k|
    np.testing.assert_allclose(O.rope(O.rope(x, 300, 1e6, style), 4000, 1e6, style),
                               O.rope(x, 4300, 1e6, style), rtol=1e-10, atol=1e-10)  # R(a)R(b)=R(a+b)
    np.testing.assert_allclose(O.rope(O.rope(x, 77, 1e6, style), -77, 1e6, style), x,
                               rtol=1e-12, atol=1e-12)                              # R(d)R(-d)=I
    q, k = RNG.standard_normal(128), RNG.standard_normal(128)
    for a, b in [(5, 9), (1000, 1003), (999990, 1000000)]:
        lhs = O.rope(q, a, 1e6, style) @ O.rope(k, b, 1e6, style)
        rhs = q @ O.rope(k, b - a, 1e6, style)
        assert math.isclose(lhs, rhs, rel_tol=1e-9, abs_tol=1e-9)


# ----------------------------------------------------------------------------
# Attention: textbook cases, torch SDPA, split merge
# ----------------------------------------------------------------------------

def test_softmax_two_keys_closed_form():
    q = np.array([1.0, 0.0, 0.0, 0.0])
    K = np.array([[2.0, 0, 0, 0], [0.0, 1, 0, 0]])
    V = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    out = O.softmax_attention(q, K, V, 1 / 2.0)     # scores 1 and 0
    w0 = math.e / (math.e + 1.0)
    np.testing.assert_allclose(out, [w0, 1 - w0, 0, 0], rtol=1e-14)


def test_softmax_special_cases():
    K = RNG.standard_normal((9, 16))
    V = RNG.standard_normal((9, 16))
    np.testing.assert_allclose(O.softmax_attention(np.zeros(16), K, V, 0.25), V.mean(0), rtol=1e-13)
    np.testing.assert_allclose(O.softmax_attention(RNG.standard_normal(16), K[:1], V[:1], 0.25),
                               V[0], rtol=1e-15)
    np.testing.assert_array_equal(O.softmax_attention(np.ones(16), K[:0], V[:0], 0.25), np.zeros(16))


def test_lse_merge_equals_unsplit():
    q = RNG.standard_normal(64)
    K = RNG.standard_normal((1000, 64)) * 3
    V = RNG.standard_normal((1000, 64))
    whole = O.softmax_attention(q, K, V, 0.125)
    cuts = [0, 1, 250, 251, 700, 1000]
    parts = [O.softmax_partial(q, K[a:b], V[a:b], 0.125) for a, b in zip(cuts[:-1], cuts[1:])]
    merged = O.lse_merge([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts])
    np.testing.assert_allclose(merged, whole, rtol=1e-12, atol=1e-14)


def _sdpa_reference(hist_k, hist_v, q_all, G, theta, causal_rows):
    """torch scaled_dot_product_attention (float64, CPU) on absolute-position RoPE."""
    T, L, Hkv, D = hist_k.shape
    pos = np.arange(T)
    outs = np.zeros_like(q_all)
    for l in range(L):
        for h in range(q_all.shape[2]):
            g = h // G
            Kr = torch.from_numpy(O.rope(hist_k[:, l, g], pos, theta))
            V = torch.from_numpy(hist_v[:, l, g])
            Qr = torch.from_numpy(O.rope(q_all[l, :, h], causal_rows, theta))
            mask = torch.from_numpy(pos[None, :] <= causal_rows[:, None])
            o = torch.nn.functional.scaled_dot_product_attention(
                Qr[None, None], Kr[None, None], V[None, None], attn_mask=mask[None, None])
            outs[l, :, h] = o[0, 0].numpy()
    return outs


@pytest.mark.parametrize("c", [1, 3])
def test_cache_matches_sdpa_without_eviction(c):
    """Capacity >= stream length: nothing is evicted, origin stays 0, so the
    re-based cache is plain causal RoPE attention (torch SDPA, float64)."""
    S, L, Hq, Hkv, D, W = 1, 2, 4, 2, 16, 64
    cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W, theta=1e4)
    hk, hv = [], []
    for step in range(6):
        k = RNG.standard_normal((L, S, c, Hkv, D))
        v = RNG.standard_normal((L, S, c, Hkv, D))
        q = RNG.standard_normal((L, S, c, Hq, D))
        cache.append(k, v)
        for j in range(c):
            hk.append(k[:, 0, j])
            hv.append(v[:, 0, j])
        out = cache.attend(q)
        T = len(hk)
        rows = np.arange(T - c, T)
        want = _sdpa_reference(np.array(hk), np.array(hv), q[:, 0], Hq // Hkv, 1e4, rows)
        np.testing.assert_allclose(out[:, 0], want, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("W,cs,style", [
    (8, [1] * 30, O.SPLIT_HALF),
    (5, [2, 3, 1, 4, 5, 1, 2, 3, 3, 1], O.SPLIT_HALF),
    (7, [3, 1, 7, 2, 6, 1, 1, 4], O.INTERLEAVED),
])
def test_cache_matches_brute_force_with_eviction(W, cs, style):
    """The ring + re-based oracle equals brute-force attention over the last W
    tokens of the full history with absolute positions, starting at a large
    absolute origin."""
    S, L, Hq, Hkv, D = 1, 2, 4, 2, 8
    p0 = 999_000
    cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W, theta=1e6, style=style)
    cache.set_state(0, p0, 0)
    hk, hv = [], []
    for c in cs:
        k = RNG.standard_normal((L, S, c, Hkv, D))
        v = RNG.standard_normal((L, S, c, Hkv, D))
        q = RNG.standard_normal((L, S, c, Hq, D))
        cache.append(k, v)
        for j in range(c):
            hk.append(k[:, 0, j])
            hv.append(v[:, 0, j])
        out = cache.attend(q)
        want = O.brute_force_window(np.array(hk), np.array(hv), q[:, 0], W, c, Hkv,
                                    theta=1e6, style=style, p0=p0)
        np.testing.assert_allclose(out[:, 0], want, rtol=1e-9, atol=1e-11)
        assert cache.fill[0] <= W
        assert all(0 <= p - cache.origin[0] < W for p in cache.retained_positions(0))


@pytest.mark.parametrize("n_prefix,cs", [(5, [1] * 12), (8, [2, 3, 1, 4]), (0, [1, 2, 1])])
def test_reset_with_prefix_is_a_new_history(n_prefix, cs):
    """Utterance reset with a prefix (the window set to n prefix pairs at a new
    origin): every later step equals brute force over the history "prefix,
    then the appended tokens" from that origin, so the prefix is the oldest
    part of the window and the first to be evicted."""
    S, L, Hq, Hkv, D, W = 1, 2, 4, 2, 8, 8
    origin = 4_321
    cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W, theta=1e6)
    cache.append(RNG.standard_normal((L, S, 3, Hkv, D)), RNG.standard_normal((L, S, 3, Hkv, D)))
    kp = RNG.standard_normal((L, Hkv, n_prefix, D))
    vp = RNG.standard_normal((L, Hkv, n_prefix, D))
    cache.set_state(0, origin, n_prefix, kp, vp)
    hk = [kp[:, :, i] for i in range(n_prefix)]
    hv = [vp[:, :, i] for i in range(n_prefix)]
    for c in cs:
        k = RNG.standard_normal((L, S, c, Hkv, D))
        v = RNG.standard_normal((L, S, c, Hkv, D))
        q = RNG.standard_normal((L, S, c, Hq, D))
        cache.append(k, v)
        hk += [k[:, 0, j] for j in range(c)]
        hv += [v[:, 0, j] for j in range(c)]
        want = O.brute_force_window(np.array(hk), np.array(hv), q[:, 0], W, c, Hkv,
                                    theta=1e6, p0=origin)
        np.testing.assert_allclose(cache.attend(q)[:, 0], want, rtol=1e-9, atol=1e-11)
    assert cache.origin[0] == origin + max(0, len(hk) - W)


def test_brute_force_window_is_last_w_tokens():
    """Brute force itself: with one key per step and q = 0 the output is the
    mean of the values of the last W tokens (closed form)."""
    T, W = 20, 6
    hk = RNG.standard_normal((T, 1, 1, 4))
    hv = RNG.standard_normal((T, 1, 1, 4))
    out = O.brute_force_window(hk, hv, np.zeros((1, 1, 1, 4)), W, 1, 1)
    np.testing.assert_allclose(out[0, 0, 0], hv[T - W:, 0, 0].mean(0), rtol=1e-13)


@pytest.mark.parametrize("origin", [0, 12345, 999_999, 123_456_789])
def test_rebasing_invariance(origin):
    """Exact re-basing: attention with re-based positions equals attention with
    absolute positions (relative distances preserved), for any origin."""
    S, L, Hq, Hkv, D, W = 1, 1, 2, 1, 64, 16
    cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W)
    k = RNG.standard_normal((L, Hkv, W, D))
    v = RNG.standard_normal((L, Hkv, W, D))
    cache.set_state(0, origin, W, k, v)
    kn = RNG.standard_normal((L, S, 2, Hkv, D))
    cache.append(kn, kn * 0.5)
    q = RNG.standard_normal((L, S, 2, Hq, D))
    a = cache.attend(q)
    b = cache.attend_absolute(q)
    # the absolute form carries angles up to origin rad, so its own float64
    # error grows like origin * 2^-52; the re-based form stays below W rad
    tol = max(1e-9, origin * 2.0 ** -52 * 64)
    np.testing.assert_allclose(a, b, rtol=tol, atol=tol)


def test_absolute_positions_lose_precision_rebased_do_not():
    """At an origin of 1e12 the absolute-position form is visibly off in
    float64 while the re-based form still equals the origin-0 result
    bit for bit: re-basing makes the result independent of the origin."""
    S, L, Hq, Hkv, D, W = 1, 1, 2, 1, 64, 16
    k = RNG.standard_normal((L, Hkv, W, D))
    v = RNG.standard_normal((L, Hkv, W, D))
    kn = RNG.standard_normal((L, S, 1, Hkv, D))
    q = RNG.standard_normal((L, S, 1, Hq, D))
    outs = []
    for origin in (0, 10 ** 12):
        cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W)
        cache.set_state(0, origin, W, k, v)
        cache.append(kn, kn)
        outs.append((cache.attend(q), cache.attend_absolute(q)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    assert np.abs(outs[1][1] - outs[1][0]).max() > 1e-9


def test_gqa_head_mapping():
    """Query head h reads KV head floor(h / G): with q = 0 the output of head h
    is the mean of KV head floor(h/G)'s values, here the constant 10*g."""
    S, L, Hq, Hkv, D, W = 1, 1, 8, 2, 8, 4
    cache = O.RollingCacheOracle(S, L, Hq, Hkv, D, W)
    k = RNG.standard_normal((L, S, 3, Hkv, D))
    v = np.zeros((L, S, 3, Hkv, D))
    v[:, :, :, 1] = 10.0
    cache.append(k, v)
    out = cache.attend(np.zeros((L, S, 3, Hq, D)))
    for h in range(Hq):
        np.testing.assert_allclose(out[0, 0, :, h], 10.0 * (h // 4))


def test_empty_window_gives_zero():
    cache = O.RollingCacheOracle(1, 1, 2, 1, 8, 4)
    np.testing.assert_array_equal(cache.attend(np.ones((1, 1, 1, 2, 8))), 0.0)


# ----------------------------------------------------------------------------
# Stored-rotated layout
# ----------------------------------------------------------------------------

def test_rerotate_identity_and_inverse():
    k = O.bf16_round(RNG.standard_normal((10, 128)))
    np.testing.assert_array_equal(O.rerotate(k, 0, 1e6), k)
    # before rounding, R(-d) undoes R(d)
    np.testing.assert_allclose(O.rope(O.rope(k, 5, 1e6), -5, 1e6), k, atol=1e-13)
    # after rounding, one re-rotation moves each element by at most half a bf16 ulp
    y = O.rerotate(k, 3, 1e6)
    exact = O.rope(k, -3, 1e6)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    assert np.all(np.abs(y - exact) <= 0.5 * ulp + 1e-300)


def test_stored_rotated_matches_pre_rope_within_bf16():
    """Stored-rotated attention equals pre-RoPE attention up to the bf16
    rounding of the stored rotated keys (the error the pages warn about)."""
    S, L, Hq, Hkv, D, W = 1, 1, 2, 1, 64, 8
    a = O.RollingCacheOracle(S, L, Hq, Hkv, D, W)
    b = O.StoredRotatedOracle(S, L, Hq, Hkv, D, W)
    errs = []
    for t in range(40):
        k = O.bf16_round(RNG.standard_normal((L, S, 1, Hkv, D)))
        v = O.bf16_round(RNG.standard_normal((L, S, 1, Hkv, D)))
        q = O.bf16_round(RNG.standard_normal((L, S, 1, Hq, D)))
        a.append(k, v)
        b.append(k, v)
        b.rebase()
        errs.append(np.abs(a.attend(q) - b.attend(q)).max())
    assert max(errs) < 5e-2
    assert max(errs) > 0.0          # rounding does leave a trace
