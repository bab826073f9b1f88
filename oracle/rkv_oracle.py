"""Oracle for the rolling KV cache with exact RoPE re-basing.

TEST INFRASTRUCTURE ONLY.  This is a plain, slow, float64 CPU statement of what
the hot path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product package (``rolling_kv_cache_buffer_b300``) never imports it, and this
module imports nothing from the product: the two share no code.

Sources, cited by page title and section:

* [LF]  "Audio8 ASR Infinite: What It Actually Takes to Listen Forever":
        the flowchart (keep / evict oldest pair / shift sliding origin /
        re-base RoPE indices / attention over window), the section
        "Inside the Rolling KV Cache and Exact RoPE Re-Basing", and
        "Failure Modes That Only Appear on Day Three of a Session".
* [A8]  "Audio8-ASR-0.1B in audio.cpp", section "Architecture":
        RoPE theta 1e6, head_dim 64.
* [MLX] "Audio8-ASR-Infinite-mlx", section "Requires a patched
        mlx-audio-swift": the checkpoint uses split-half (rotate_half)
        rotary pairing; interleaved pairing gives wrong output.
* [CPU] "Reza2kn/Audio8-ASR-Infinite-Compressed", section "Linux CPU":
        BF16 cache storage.
* [TT]  "audio8-asr-infinite-p150", section "At a glance": the decoder
        keeps a fixed rolling context.

Readings taken where the pages are silent:

* origin = absolute position of the oldest retained token; re-based
  position r = p - origin, so 0 <= r < capacity;
* eviction happens before insertion, so the fill never exceeds capacity and
  a new token is inside the window it attends over;
* slot(p) = p mod capacity;
* inverse frequencies w_i = theta^(-2i/D), no scaling;
* softmax scale 1/sqrt(D) unless given;
* GQA: query head h reads KV head floor(h / G), G = H_q / H_kv;
* a chunk of c new tokens is inserted at once; query j (absolute position
  p_j) attends over the post-insert window, keys with p <= p_j;
* an empty window attends to nothing and yields a zero output;
* stored-rotated layout: a key is stored as bf16(R(p - origin') k) when it
  is inserted; every later eviction of e pairs re-rotates each retained
  older key by R(-e) and rounds it to bf16 again (round to nearest even).

Parity pins (tests/test_oracle.py): every function below is pinned to
something other than itself -- closed forms, torch's bf16 conversion and
scaled_dot_product_attention, complex-number rotation, brute force over the
full history, and invariants the pages state.  ``rerotate`` carries the pin
"identity at delta 0, inverse of rotation before rounding"; its rounding
step is pinned separately through ``bf16_round``.  The stored-rotated models'
``set_state`` (tests/test_oracle_set_state.py) is pinned to complex-number
rotation rounded by torch's bf16 conversion (key i of a seeded window stored
as bf16(R(i) k_i)) and to brute force over the history after a reset.
"""

from __future__ import annotations

import math
from collections import OrderedDict
from dataclasses import dataclass, field

import numpy as np

SPLIT_HALF = "split_half"
INTERLEAVED = "interleaved"


# ---------------------------------------------------------------------------
# bf16 rounding (the cache stores BF16 values: [CPU] "Linux CPU")
# ---------------------------------------------------------------------------

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits.  A normal value with frexp exponent e
    (|x| in [2^(e-1), 2^e)) is quantised in steps of 2^(e-8); below the
    smallest normal 2^-126 the step stays 2^-133 (subnormals).  Values whose
    magnitude rounds to 2^128 or more become infinities.  Returns float64.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(xf)
    e = np.maximum(e, -125)
    step = np.ldexp(1.0, e - 8)
    y = np.rint(xf / step) * step          # np.rint rounds half to even
    y = np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, y), y)
    out[finite] = y
    return out


# ---------------------------------------------------------------------------
# Bookkeeping: FIFO eviction and sliding origin ([LF] flowchart, "Inside ...")
# ---------------------------------------------------------------------------

@dataclass
class Bookkeeping:
    origin: int            # origin after the step (absolute position of oldest kept)
    fill: int              # number of retained pairs after the step
    evicted: int           # pairs evicted by this step
    first_slot: int        # slot of the first new position
    new_positions: list = field(default_factory=list)
    new_slots: list = field(default_factory=list)
    evicted_positions: list = field(default_factory=list)

    def log(self):
        """The 4-word step log: (origin', fill', evicted, first_slot)."""
        return (self.origin, self.fill, self.evicted, self.first_slot)


def bookkeep(origin: int, fill: int, n_new: int, capacity: int,
             slots: int | None = None) -> Bookkeeping:
    """One append of ``n_new`` pairs to a window that retains ``capacity`` pairs.

    [LF] flowchart: a token that does not fit makes the cache "evict oldest
    pair" and "shift sliding origin forward".  Retained absolute positions
    before the step are origin .. origin+fill-1; the new tokens take the next
    positions origin+fill .. origin+fill+n_new-1.  Just enough of the oldest
    pairs are evicted that the fill never exceeds the capacity.  Position p
    lives in slot p mod ``slots`` (default: the capacity); a ring with more
    slots than retained pairs (the 750-frame encoder window of [TT] "At a
    glance" in 768 slots) keeps the same FIFO.
    """
    slots = capacity if slots is None else slots
    if capacity <= 0 or slots < capacity:
        raise ValueError("capacity must be positive and at most the slot count")
    if n_new < 0 or n_new > capacity:
        raise ValueError("n_new must be in [0, capacity]")
    if origin < 0 or not (0 <= fill <= capacity):
        raise ValueError("corrupt state")
    evicted = max(0, fill + n_new - capacity)
    first_pos = origin + fill
    new_positions = [first_pos + j for j in range(n_new)]
    return Bookkeeping(
        origin=origin + evicted,
        fill=fill + n_new - evicted,
        evicted=evicted,
        first_slot=first_pos % slots,
        new_positions=new_positions,
        new_slots=[p % slots for p in new_positions],
        evicted_positions=list(range(origin, origin + evicted)),
    )


# ---------------------------------------------------------------------------
# Rotary position embedding ([A8] "Architecture": theta 1e6; [MLX] split-half)
# ---------------------------------------------------------------------------

def inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """w_i = theta^(-2i/D) for i < D/2 (float64)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope(x, pos, theta: float, style: str = SPLIT_HALF):
    """Rotate the last axis of ``x`` (length D) to position(s) ``pos``.

    Pair i (i < D/2) is rotated by the angle pos * w_i.  Split-half pairs
    element i with element i + D/2 (rotate_half); interleaved pairs 2i with
    2i+1.  For a pair (a, b) the result is (a cos - b sin, b cos + a sin).
    ``pos`` broadcasts against x[..., 0].
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    y = np.empty(np.broadcast_shapes(x.shape, c.shape[:-1] + (d,)), dtype=np.float64)
    if style == SPLIT_HALF:
        a, b = x[..., : d // 2], x[..., d // 2:]
        y[..., : d // 2] = a * c - b * s
        y[..., d // 2:] = b * c + a * s
    elif style == INTERLEAVED:
        a, b = x[..., 0::2], x[..., 1::2]
        y[..., 0::2] = a * c - b * s
        y[..., 1::2] = b * c + a * s
    else:
        raise ValueError(style)
    return y


# ---------------------------------------------------------------------------
# Attention over the window ([LF] flowchart "Attention over window")
# ---------------------------------------------------------------------------

def softmax_attention(q, keys, values, scale: float):
    """out = sum_r softmax_r(<q, k_r> * scale) v_r, all float64.

    q: [D]; keys, values: [n, D] with keys already rotated.  An empty key set
    gives a zero vector.
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1], dtype=np.float64)
    s = (keys @ q) * scale
    s = s - s.max()
    w = np.exp(s)
    return (w / w.sum()) @ values


def lse_merge(ms, ls, os_):
    """Merge split-softmax partials: each part carries its max m_i, its sum
    l_i = sum exp(s - m_i) and its unnormalised output o_i = sum exp(s - m_i) v.
    m = max m_i; out = sum_i e^(m_i - m) o_i / sum_i e^(m_i - m) l_i."""
    ms = np.asarray(ms, dtype=np.float64)
    m = ms.max()
    w = np.exp(ms - m)
    num = sum(wi * np.asarray(oi, dtype=np.float64) for wi, oi in zip(w, os_))
    den = float(np.dot(w, np.asarray(ls, dtype=np.float64)))
    return num / den


def softmax_partial(q, keys, values, scale: float):
    """(m, l, o) of one split, as defined for ``lse_merge``."""
    s = (np.asarray(keys, np.float64) @ np.asarray(q, np.float64)) * scale
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ np.asarray(values, np.float64)


# ---------------------------------------------------------------------------
# The rolling cache, pre-RoPE layout
# ---------------------------------------------------------------------------

class RollingCacheOracle:
    """Fixed-capacity KV window per stream, keys stored before rotation.

    [LF] "Inside the Rolling KV Cache and Exact RoPE Re-Basing": capacity is
    constant; once full, the oldest pairs are evicted as new ones arrive; the
    origin shifts forward and every retained key and the query are placed at
    position (p - origin), which leaves query-key distances unchanged.

    Per stream the window is an ordered map from absolute position p to the
    pair (k[L][H_kv][D], v[L][H_kv][D]) in float64.  ``capacity`` is the
    number of slots; ``window`` (default: the ring's slot count) the number
    of pairs retained, which may be smaller (an encoder's 750-frame window
    kept in 768 slots, [TT] "At a glance").

    Pinned prefix (``n_pinned`` = P > 0 slots, the rest a ring of capacity - P
    slots): ``reset`` places a constant prefix -- the audio-independent prompt
    prepared once and checked again on every silence reset ([CPU] "Linux
    CPU") -- in the pinned slots, where no append evicts it.  The window is
    read as a re-prefill of "prefix, then the retained tokens" ([TT]
    "Limitations": the decoder's rolling context is rebuilt by re-prefilling
    the window): prefix pair i sits at position i, a retained token p at
    npin + (p - origin), the query of token p_q at npin + (p_q - origin).
    """

    def __init__(self, n_streams, n_layers, n_q_heads, n_kv_heads, head_dim,
                 capacity, theta=1e6, style=SPLIT_HALF, scale=None, window=None,
                 n_pinned=0):
        if n_q_heads % n_kv_heads:
            raise ValueError("n_q_heads must be a multiple of n_kv_heads")
        self.S, self.L = n_streams, n_layers
        self.Hq, self.Hkv, self.D = n_q_heads, n_kv_heads, head_dim
        self.G = n_q_heads // n_kv_heads
        self.W = capacity
        self.P = int(n_pinned)
        if not 0 <= self.P < capacity:
            raise ValueError("n_pinned must be in [0, capacity)")
        self.ring = capacity - self.P            # slots of the rolling part
        self.Wr = self.ring if window is None else int(window)
        if not 0 < self.Wr <= self.ring:
            raise ValueError("window must be in [1, capacity - n_pinned]")
        self.theta, self.style = theta, style
        self.scale = (1.0 / math.sqrt(head_dim)) if not scale else float(scale)
        self.origin = [0] * n_streams
        self.fill = [0] * n_streams
        self.window = [OrderedDict() for _ in range(n_streams)]
        self.prefix = [[] for _ in range(n_streams)]   # pinned (k, v) pairs

    # -- state --------------------------------------------------------------
    def set_state(self, s, origin, fill, k=None, v=None):
        """Jump stream ``s`` to (origin, fill) holding the given contents.
        k, v: [L][H_kv][fill][D] in position order (position origin + i)."""
        if origin < 0 or not (0 <= fill <= self.Wr):
            raise ValueError("corrupt state")
        self.origin[s], self.fill[s] = int(origin), int(fill)
        self.window[s] = OrderedDict()
        self.prefix[s] = []
        for i in range(fill):
            self.window[s][origin + i] = (
                np.asarray(k[:, :, i, :], np.float64).copy(),
                np.asarray(v[:, :, i, :], np.float64).copy())

    def reset(self, s, origin, k=None, v=None, n=0):
        """Utterance reset of stream ``s`` at ``origin`` with an ``n``-pair
        prefix (k, v: [L][H_kv][n][D]).  With pinned slots the prefix is
        pinned (n <= n_pinned) and the rolling window starts empty; without,
        the prefix is the rolling window's first n pairs (``set_state``)."""
        if not self.P:
            self.set_state(s, origin, n, k, v)
            return
        if not 0 <= n <= self.P:
            raise ValueError("prefix longer than the pinned slots")
        self.set_state(s, origin, 0)
        self.prefix[s] = [(np.asarray(k[:, :, i, :], np.float64).copy(),
                           np.asarray(v[:, :, i, :], np.float64).copy()) for i in range(n)]

    def retained_positions(self, s):
        return list(self.window[s].keys())

    def n_prefix(self, s):
        return len(self.prefix[s])

    # -- append ---------------------------------------------------------------
    def append(self, k_new, v_new):
        """k_new, v_new: [L][S][c][H_kv][D].  Returns the per-stream logs."""
        k_new = np.asarray(k_new, np.float64)
        v_new = np.asarray(v_new, np.float64)
        c = k_new.shape[2]
        logs = []
        for s in range(self.S):
            bk = self._bookkeep(s, c)
            for p in bk.evicted_positions:
                del self.window[s][p]
            for j, p in enumerate(bk.new_positions):
                self.window[s][p] = (k_new[:, s, j].copy(), v_new[:, s, j].copy())
            self.origin[s], self.fill[s] = bk.origin, bk.fill
            logs.append(bk.log())
        return logs

    def _bookkeep(self, s, c):
        """The append's bookkeeping in the rolling part: the ring is the slots
        after the pinned ones, so the logged first slot is P + p mod (W - P)."""
        bk = bookkeep(self.origin[s], self.fill[s], c, self.Wr, self.ring)
        bk.first_slot += self.P
        bk.new_slots = [self.P + x for x in bk.new_slots]
        return bk

    # -- attend ---------------------------------------------------------------
    def _attend(self, q, layer_begin, absolute):
        q = np.asarray(q, np.float64)
        nl, S, c, Hq, D = q.shape
        out = np.zeros_like(q)
        for s in range(S):
            pos = np.array(self.retained_positions(s), dtype=np.int64)
            n = len(pos)
            npin = self.n_prefix(s)
            if absolute and npin:
                raise ValueError("a pinned prefix has re-based positions only")
            base = 0 if absolute else self.origin[s]
            # prefix pair i at i, retained token p at npin + (p - base)
            r = np.concatenate([np.arange(npin), npin + pos - base]).astype(np.int64)
            for li in range(nl):
                l = layer_begin + li
                for g in range(self.Hkv):
                    pairs = [self.prefix[s][i] for i in range(npin)] + \
                        [self.window[s][p] for p in pos]
                    if pairs:
                        K = np.stack([kv[0][l, g] for kv in pairs])
                        V = np.stack([kv[1][l, g] for kv in pairs])
                        Kr = rope(K, r, self.theta, self.style)
                    for j in range(c):
                        pq = self.origin[s] + n - c + j   # absolute query position
                        rq = npin + pq - base
                        vis = np.concatenate([np.ones(npin, bool), pos <= pq])
                        for hh in range(self.G):
                            h = g * self.G + hh
                            if not pairs:
                                continue
                            qr = rope(q[li, s, j, h], rq, self.theta, self.style)
                            out[li, s, j, h] = softmax_attention(
                                qr, Kr[vis], V[vis], self.scale)
        return out

    def attend(self, q, layer_begin=0):
        """q: [n_layers][S][c][H_q][D] pre-RoPE queries for the c newest tokens.
        Re-based positions: key r = p - origin', query r_j = fill' - c + j."""
        return self._attend(q, layer_begin, absolute=False)

    def attend_absolute(self, q, layer_begin=0):
        """Same attention with absolute positions (no re-basing)."""
        return self._attend(q, layer_begin, absolute=True)


# ---------------------------------------------------------------------------
# Stored-rotated layout with explicit re-rotation ([LF] "Inside ...", the
# rounding hazard; "Failure Modes ..."): keys are kept rotated and re-based
# by a rotation at every eviction, each time rounded back to bf16.
# ---------------------------------------------------------------------------

def rerotate(k_stored, delta, theta, style=SPLIT_HALF):
    """Per-call re-rotation: bf16(R(-delta) k) with the rotation in float64."""
    return bf16_round(rope(np.asarray(k_stored, np.float64), -float(delta), theta, style))


class StoredRotatedOracle(RollingCacheOracle):
    """Keys are stored as bf16(R(p - origin') k) and re-rotated by R(-e)
    (then rounded to bf16 again) whenever e pairs are evicted.  With a pinned
    prefix, prefix pair i is stored as bf16(R(i) k) once and never turned
    again (its position does not move); retained keys sit at
    npin + (p - origin')."""

    def __init__(self, *a, **kw):
        super().__init__(*a, **kw)
        self.pending = [0] * self.S

    def set_state(self, s, origin, fill, k=None, v=None):
        """k holds *unrotated* keys; they are stored rotated to p - origin."""
        super().set_state(s, origin, fill, k, v)
        for i, p in enumerate(list(self.window[s].keys())):
            kk, vv = self.window[s][p]
            self.window[s][p] = (bf16_round(rope(kk, p - origin, self.theta, self.style)), vv)
        self.pending[s] = 0

    def reset(self, s, origin, k=None, v=None, n=0):
        """As the base class; pinned prefix keys are stored rotated to i."""
        super().reset(s, origin, k, v, n)
        self.prefix[s] = [(bf16_round(rope(kk, i, self.theta, self.style)), vv)
                          for i, (kk, vv) in enumerate(self.prefix[s])]
        self.pending[s] = 0

    def append(self, k_new, v_new):
        k_new = np.asarray(k_new, np.float64)
        v_new = np.asarray(v_new, np.float64)
        c = k_new.shape[2]
        logs = []
        for s in range(self.S):
            bk = self._bookkeep(s, c)
            npin = self.n_prefix(s)
            for p in bk.evicted_positions:
                del self.window[s][p]
            for j, p in enumerate(bk.new_positions):
                kt = bf16_round(rope(k_new[:, s, j], npin + p - bk.origin, self.theta,
                                     self.style))
                self.window[s][p] = (kt, v_new[:, s, j].copy())
            self.origin[s], self.fill[s] = bk.origin, bk.fill
            self.pending[s] = bk.evicted
            logs.append(bk.log())
        self._new = c
        return logs

    def rebase(self):
        """Re-rotate every retained key that predates the last append by
        R(-e), e = pairs that append evicted, and round to bf16."""
        for s in range(self.S):
            e = self.pending[s]
            if e:
                keep_new = self._new
                items = list(self.window[s].items())
                for p, (kt, vv) in items[: len(items) - keep_new]:
                    self.window[s][p] = (rerotate(kt, e, self.theta, self.style), vv)
            self.pending[s] = 0

    def attend(self, q, layer_begin=0):
        q = np.asarray(q, np.float64)
        nl, S, c, Hq, D = q.shape
        out = np.zeros_like(q)
        for s in range(S):
            pos = np.array(self.retained_positions(s), dtype=np.int64)
            n = len(pos)
            npin = self.n_prefix(s)
            if n + npin == 0:
                continue
            for li in range(nl):
                l = layer_begin + li
                for g in range(self.Hkv):
                    pairs = list(self.prefix[s]) + [self.window[s][p] for p in pos]
                    K = np.stack([kv[0][l, g] for kv in pairs])
                    V = np.stack([kv[1][l, g] for kv in pairs])
                    for j in range(c):
                        pq = self.origin[s] + n - c + j
                        vis = np.concatenate([np.ones(npin, bool), pos <= pq])
                        for hh in range(self.G):
                            h = g * self.G + hh
                            qr = rope(q[li, s, j, h], npin + pq - self.origin[s], self.theta,
                                      self.style)
                            out[li, s, j, h] = softmax_attention(qr, K[vis], V[vis], self.scale)
        return out


class EpochRotatedOracle(RollingCacheOracle):
    """Stored-rotated keys with lazy (epoch) re-basing.

    Not a scheme the pages describe: a variant of their stored-rotated layout
    that trades the every-eviction re-rotation (and its repeated rounding,
    [LF] "Failure Modes That Only Appear on Day Three of a Session") for a
    lag.  Keys are stored as bf16(R(p - o_ref) k), o_ref = origin' - lag, where
    lag counts the evictions since the last re-rotation; the query at p_q is
    turned by R(p_q - o_ref), so every query-key distance is unchanged.
    ``rebase`` turns every retained key by R(-lag) and rounds it to bf16, once
    lag >= epoch; an append with lag >= epoch is an error (a missed re-base).
    """

    def __init__(self, *a, epoch, **kw):
        super().__init__(*a, **kw)
        if epoch < 2:
            raise ValueError("epoch >= 2")
        if self.P:
            # A pinned key would need the lag in its position as well: not modelled.
            raise ValueError("no pinned prefix with a re-basing epoch")
        self.epoch = int(epoch)
        self.lag = [0] * self.S

    def set_state(self, s, origin, fill, k=None, v=None):
        """k holds *unrotated* keys; they are stored rotated to p - origin."""
        super().set_state(s, origin, fill, k, v)
        for p in list(self.window[s].keys()):
            kk, vv = self.window[s][p]
            self.window[s][p] = (bf16_round(rope(kk, p - origin, self.theta, self.style)), vv)
        self.lag[s] = 0

    def o_ref(self, s):
        return self.origin[s] - self.lag[s]

    def append(self, k_new, v_new):
        k_new = np.asarray(k_new, np.float64)
        v_new = np.asarray(v_new, np.float64)
        c = k_new.shape[2]
        logs = []
        for s in range(self.S):
            if self.lag[s] >= self.epoch:
                raise RuntimeError("append before the due re-base")
            bk = self._bookkeep(s, c)
            for p in bk.evicted_positions:
                del self.window[s][p]
            lag2 = self.lag[s] + bk.evicted
            ref = bk.origin - lag2
            for j, p in enumerate(bk.new_positions):
                kt = bf16_round(rope(k_new[:, s, j], p - ref, self.theta, self.style))
                self.window[s][p] = (kt, v_new[:, s, j].copy())
            self.origin[s], self.fill[s] = bk.origin, bk.fill
            self.lag[s] = lag2
            logs.append(bk.log())
        return logs

    def rebase(self):
        """Streams whose lag reached the epoch: every retained key turns by
        R(-lag) (float64) and is rounded to bf16; the lag returns to 0."""
        for s in range(self.S):
            lag = self.lag[s]
            if lag >= self.epoch:
                for p, (kt, vv) in list(self.window[s].items()):
                    self.window[s][p] = (rerotate(kt, lag, self.theta, self.style), vv)
                self.lag[s] = 0

    def attend(self, q, layer_begin=0):
        q = np.asarray(q, np.float64)
        nl, S, c, Hq, D = q.shape
        out = np.zeros_like(q)
        for s in range(S):
            pos = np.array(self.retained_positions(s), dtype=np.int64)
            n = len(pos)
            if n == 0:
                continue
            ref = self.o_ref(s)
            for li in range(nl):
                l = layer_begin + li
                for g in range(self.Hkv):
                    K = np.stack([self.window[s][p][0][l, g] for p in pos])
                    V = np.stack([self.window[s][p][1][l, g] for p in pos])
                    for j in range(c):
                        pq = self.origin[s] + n - c + j
                        vis = pos <= pq
                        for hh in range(self.G):
                            h = g * self.G + hh
                            qr = rope(q[li, s, j, h], pq - ref, self.theta, self.style)
                            out[li, s, j, h] = softmax_attention(qr, K[vis], V[vis], self.scale)
        return out


# ---------------------------------------------------------------------------
# Brute force over the whole history (no ring, no re-basing)
# ---------------------------------------------------------------------------

def brute_force_reprefill(pre_k, pre_v, hist_k, hist_v, q, window, n_new, n_kv_heads,
                          theta=1e6, style=SPLIT_HALF, scale=None):
    """Attention of the ``n_new`` newest tokens over a re-prefilled window:
    the sequence "prefix, then the last ``window`` tokens of the history",
    numbered 0, 1, 2, ... from its start ([TT] "Limitations": the rolling
    context rebuilt by re-prefilling the window), causal.

    pre_k, pre_v: [P][L][H_kv][D]; hist_k, hist_v: [T][L][H_kv][D];
    q: [L][n_new][H_q][D].  Returns [L][n_new][H_q][D].
    """
    pre_k = np.asarray(pre_k, np.float64).reshape((-1,) + np.shape(hist_k)[1:])
    pre_v = np.asarray(pre_v, np.float64).reshape((-1,) + np.shape(hist_v)[1:])
    hist_k = np.asarray(hist_k, np.float64)
    hist_v = np.asarray(hist_v, np.float64)
    q = np.asarray(q, np.float64)
    T, L, Hkv, D = hist_k.shape
    G = q.shape[2] // n_kv_heads
    sc = (1.0 / math.sqrt(D)) if not scale else scale
    seq_k = np.concatenate([pre_k, hist_k[max(0, T - window):]])
    seq_v = np.concatenate([pre_v, hist_v[max(0, T - window):]])
    n = seq_k.shape[0]
    out = np.zeros_like(q)
    for l in range(L):
        for h in range(q.shape[2]):
            g = h // G
            for j in range(n_new):
                iq = n - n_new + j                      # the query's index in the sequence
                K = rope(seq_k[: iq + 1, l, g], np.arange(iq + 1), theta, style)
                qr = rope(q[l, j, h], iq, theta, style)
                out[l, j, h] = softmax_attention(qr, K, seq_v[: iq + 1, l, g], sc)
    return out


def brute_force_window(hist_k, hist_v, q, capacity, n_new, n_kv_heads,
                       theta=1e6, style=SPLIT_HALF, scale=None, p0=0):
    """Attention of the ``n_new`` newest tokens over the last ``capacity``
    tokens of the full history, with absolute RoPE positions.

    hist_k, hist_v: [T][L][H_kv][D], token t at absolute position p0 + t.
    q: [L][n_new][H_q][D] for the newest n_new tokens.  The window after the
    step is the last min(T, capacity) tokens; query j (absolute position
    p0 + T - n_new + j) sees the window tokens at or before its own position.
    Returns [L][n_new][H_q][D].
    """
    hist_k = np.asarray(hist_k, np.float64)
    hist_v = np.asarray(hist_v, np.float64)
    q = np.asarray(q, np.float64)
    T, L, Hkv, D = hist_k.shape
    Hq = q.shape[2]
    G = Hq // n_kv_heads
    sc = (1.0 / math.sqrt(D)) if not scale else scale
    lo = max(0, T - capacity)
    out = np.zeros_like(q)
    for l in range(L):
        for h in range(Hq):
            g = h // G
            for j in range(n_new):
                t_q = T - n_new + j
                ts = np.arange(lo, t_q + 1)
                K = rope(hist_k[ts, l, g], p0 + ts, theta, style)
                qr = rope(q[l, j, h], p0 + t_q, theta, style)
                out[l, j, h] = softmax_attention(qr, K, hist_v[ts, l, g], sc)
    return out
