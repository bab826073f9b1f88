"""Plant plausible mistakes in the oracle (on the CPU) and check that at least
one pin catches each: a pin that a wrong sign, a dropped term or a wrong index
slips through would pin nothing."""

import math

import numpy as np
import pytest

from oracle import rkv_oracle as O
from tests import test_oracle as T

_ORIG = {name: getattr(O, name) for name in ("rope", "bookkeep", "softmax_attention")}


def _rope_sin_sign_flipped(x, pos, theta, style=O.SPLIT_HALF):
    return _ORIG['rope'](x, -np.asarray(pos, np.float64), theta, style)


def _rope_wrong_pairing(x, pos, theta, style=O.SPLIT_HALF):
    other = O.INTERLEAVED if style == O.SPLIT_HALF else O.SPLIT_HALF
    return _ORIG['rope'](x, pos, theta, other)


def _inv_freq_wrong_exponent(head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -1.0 * i / head_dim)


def _bookkeep_off_by_one(origin, fill, n_new, capacity):
    bk = _ORIG['bookkeep'](origin, fill, n_new, capacity)
    if bk.evicted:
        bk.evicted -= 1
        bk.origin -= 1
        bk.fill += 1
    return bk


def _softmax_no_scale(q, keys, values, scale):
    return _ORIG['softmax_attention'](q, keys, values, 1.0)


def _lse_merge_unweighted(ms, ls, os_):
    return sum(np.asarray(o) for o in os_) / float(np.sum(ls))


def _bf16_truncate(x):
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    e = np.maximum(e, -125)
    step = np.ldexp(1.0, e - 8)
    return np.trunc(x / step) * step


class _ShiftedQuery(O.RollingCacheOracle):
    """Query placed one position too far (off-by-one in r_q)."""

    def _attend(self, q, layer_begin, absolute):
        saved = [dict(w) for w in self.window]
        try:
            self.origin = [o - 1 for o in self.origin]
            return super()._attend(q, layer_begin, absolute)
        finally:
            self.origin = [o + 1 for o in self.origin]
            del saved


MUTATIONS = [
    ("rope", _rope_sin_sign_flipped, [T.test_rope_split_half_is_complex_multiplication], {"D": 64}),
    ("rope", _rope_wrong_pairing, [T.test_rope_split_half_is_complex_multiplication], {"D": 64}),
    ("inv_freq", _inv_freq_wrong_exponent, [T.test_inv_freq_closed_form], {}),
    ("bookkeep", _bookkeep_off_by_one, [T.test_bookkeeping_closed_form_tiny], {}),
    ("softmax_attention", _softmax_no_scale, [T.test_softmax_two_keys_closed_form], {}),
    ("lse_merge", _lse_merge_unweighted, [T.test_lse_merge_equals_unsplit], {}),
    ("bf16_round", _bf16_truncate, [T.test_bf16_round_matches_torch_random], {}),
]


@pytest.mark.parametrize("target,mutant,pins,kw", MUTATIONS,
                         ids=[m[1].__name__ for m in MUTATIONS])
def test_mutation_is_caught(monkeypatch, target, mutant, pins, kw):
    monkeypatch.setattr(O, target, mutant)
    caught = False
    for pin in pins:
        try:
            pin(**kw)
        except AssertionError:
            caught = True
    assert caught, f"no pin caught the mutated {target}"


def test_gqa_mapping_mutation_is_caught(monkeypatch):
    """h -> h % H_kv instead of h // G."""
    class Mod(O.RollingCacheOracle):
        def _attend(self, q, layer_begin, absolute):
            q = np.asarray(q, np.float64)
            out = np.zeros_like(q)
            for s in range(q.shape[1]):
                pos = np.array(self.retained_positions(s))
                for li in range(q.shape[0]):
                    for h in range(self.Hq):
                        g = h % self.Hkv
                        K = np.stack([self.window[s][p][0][li, g] for p in pos])
                        V = np.stack([self.window[s][p][1][li, g] for p in pos])
                        for j in range(q.shape[2]):
                            out[li, s, j, h] = O.softmax_attention(
                                O.rope(q[li, s, j, h], 0, 1e6), O.rope(K, pos - self.origin[s], 1e6),
                                V, self.scale)
            return out

    monkeypatch.setattr(O, "RollingCacheOracle", Mod)
    with pytest.raises(AssertionError):
        T.test_gqa_head_mapping()


def test_query_offset_mutation_is_caught(monkeypatch):
    monkeypatch.setattr(O, "RollingCacheOracle", _ShiftedQuery)
    with pytest.raises(AssertionError):
        T.test_cache_matches_brute_force_with_eviction(8, [1] * 30, O.SPLIT_HALF)


# ---- set_state of the stored-rotated models --------------------------------

def _set_state_absolute(self, s, origin, fill, k=None, v=None):
    """Keys rotated to their absolute position p instead of p - origin."""
    O.RollingCacheOracle.set_state(self, s, origin, fill, k, v)
    for p in list(self.window[s].keys()):
        kk, vv = self.window[s][p]
        self.window[s][p] = (O.bf16_round(O.rope(kk, p, self.theta, self.style)), vv)
    if hasattr(self, "lag"):
        self.lag[s] = 0
    else:
        self.pending[s] = 0


def _set_state_unrounded(self, s, origin, fill, k=None, v=None):
    """Rotated keys kept in float64 (the bf16 round forgotten)."""
    O.RollingCacheOracle.set_state(self, s, origin, fill, k, v)
    for p in list(self.window[s].keys()):
        kk, vv = self.window[s][p]
        self.window[s][p] = (O.rope(kk, p - origin, self.theta, self.style), vv)
    if hasattr(self, "lag"):
        self.lag[s] = 0
    else:
        self.pending[s] = 0


@pytest.mark.parametrize("cls", ["StoredRotatedOracle", "EpochRotatedOracle"])
@pytest.mark.parametrize("mutant", [_set_state_absolute, _set_state_unrounded],
                         ids=["absolute_position", "no_bf16_round"])
def test_set_state_mutation_is_caught(monkeypatch, cls, mutant):
    from tests import test_oracle_set_state as T2
    monkeypatch.setattr(getattr(O, cls), "set_state", mutant)
    kind = "stored" if cls == "StoredRotatedOracle" else "epoch"
    with pytest.raises(AssertionError):
        T2.test_set_state_stores_keys_rotated_from_the_new_origin(kind, O.SPLIT_HALF, 987_654, 11)
