"""The C-ABI library loads, exports every symbol include/rkv.h declares, and
rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import rolling_kv_cache_buffer_b300 as R
from rkv_inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(rkv_[a-z0-9_]+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    lib = R.load_library()
    names = _declared()
    assert {"rkv_create", "rkv_append", "rkv_attend", "rkv_rebase", "rkv_destroy"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_abi_version_and_struct_size():
    assert R.rkv_abi_version() == 2
    assert ctypes.sizeof(R.rkv_config) == 72
    assert ctypes.sizeof(R.rkv_buffers) == 40


def _cfg(**kw):
    base = dict(n_streams=1, n_layers=36, n_q_heads=16, n_kv_heads=2, head_dim=128,
                capacity=4096)
    base.update(kw)
    return R.make_config(**base)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_required_bytes_closed_form(name):
    wl = WORKLOADS[name]
    cfg = R.make_config(wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                        wl.capacity, max_chunk=wl.n_new, kv_dtype=wl.kv_dtype)
    pool, state, ws = R.rkv_required_bytes(cfg)
    assert pool == (wl.n_streams * wl.n_layers * wl.n_kv_heads * wl.capacity * wl.head_dim *
                    wl.elem_bytes)
    assert state >= 32 * wl.n_streams and state % 256 == 0
    # the float32 (cos, sin) table alone takes 2W x D/2 float2
    assert ws >= 2 * wl.capacity * (wl.head_dim // 2) * 8


@pytest.mark.parametrize("kw,status", [
    (dict(n_q_heads=15), R.rkv.RKV_ERR_INVALID_ARG),
    (dict(head_dim=96), R.rkv.RKV_ERR_UNSUPPORTED),
    (dict(capacity=100), R.rkv.RKV_ERR_UNSUPPORTED),
    (dict(capacity=32, max_chunk=33), R.rkv.RKV_ERR_CAPACITY),
    (dict(n_streams=0), R.rkv.RKV_ERR_INVALID_ARG),
    (dict(rope_theta=1.0), R.rkv.RKV_ERR_INVALID_ARG),
    (dict(n_streams=2000), R.rkv.RKV_ERR_UNSUPPORTED),
    (dict(rebase_epoch=-1), R.rkv.RKV_ERR_INVALID_ARG),
    (dict(rebase_epoch=64), R.rkv.RKV_ERR_INVALID_ARG),                       # pre-RoPE
    (dict(layout="stored_rotated", rebase_epoch=4096, max_chunk=2), R.rkv.RKV_ERR_INVALID_ARG),
    (dict(capacity=768, window=769), R.rkv.RKV_ERR_INVALID_ARG),              # window > slots
    (dict(capacity=768, window=-1), R.rkv.RKV_ERR_INVALID_ARG),
    (dict(capacity=768, window=4, max_chunk=5), R.rkv.RKV_ERR_CAPACITY),      # chunk > window
    (dict(layout="stored_rotated", capacity=768, window=750, rebase_epoch=751),
     R.rkv.RKV_ERR_INVALID_ARG),                                               # E + c > W_r + 1
])
def test_config_rejected(kw, status):
    with pytest.raises(R.RkvError) as e:
        R.rkv_required_bytes(_cfg(**kw))
    assert e.value.status == status


def test_rebase_epoch_bounds_accepted():
    # an epoch E needs E + max_chunk <= W + 1 (positions p - o_ref stay below 2W)
    R.rkv_required_bytes(_cfg(layout="stored_rotated", rebase_epoch=4096))
    R.rkv_required_bytes(_cfg(layout="stored_rotated", rebase_epoch=4090, max_chunk=7))
    R.rkv_required_bytes(_cfg(layout="stored_rotated", rebase_epoch=0))
    R.rkv_required_bytes(_cfg(layout="stored_rotated", rebase_epoch=1))   # 1 = every eviction
    R.rkv_required_bytes(_cfg(layout="stored_rotated", capacity=768, window=750,
                              rebase_epoch=750))


def test_window_accepted():
    # the encoder's 750-frame window in 768 slots, four frames per step
    pool, _, _ = R.rkv_required_bytes(_cfg(n_layers=32, n_q_heads=20, n_kv_heads=20,
                                          head_dim=64, capacity=768, window=750, max_chunk=4))
    assert pool == 32 * 20 * 768 * 64 * 2


def test_create_rejects_null_and_misaligned_buffers_without_gpu():
    cfg = _cfg()
    _, _, ws = R.rkv_required_bytes(cfg)
    with pytest.raises(R.RkvError) as e:
        R.rkv_create(cfg, R.rkv_buffers(0, 0, 0, 0, ws), 0)
    assert e.value.status == R.rkv.RKV_ERR_INVALID_ARG
    with pytest.raises(R.RkvError) as e:
        R.rkv_create(cfg, R.rkv_buffers(4096, 4096 + 8, 8192, 16384, ws), 0)
    assert e.value.status == R.rkv.RKV_ERR_INVALID_ARG
    with pytest.raises(R.RkvError) as e:
        R.rkv_create(cfg, R.rkv_buffers(4096, 8192, 8192, 16384, ws - 1), 0)
    assert e.value.status == R.rkv.RKV_ERR_INVALID_ARG


def test_null_handle_calls():
    lib = R.load_library()
    assert lib.rkv_append(None, None, None, 1, None, None) == R.rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_attend(None, None, None, 0, 1, 1, None) == R.rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_rebase(None, None) == R.rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_destroy(None) == R.rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_set_stream_state(None, 0, 0, 0, None) == R.rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_last_launch_count(None) == 0
    for s in range(6):
        assert R.status_string(s)


def test_reset_stream_rejects_bad_arguments_without_gpu():
    """rkv_reset_stream checks its arguments before touching the GPU."""
    lib = R.load_library()
    assert lib.rkv_reset_stream(None, 0, 0, None, None, 0, None) == R.rkv.RKV_ERR_INVALID_ARG
