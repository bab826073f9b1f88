"""Python binding of librkv.so (include/rkv.h), argument marshalling only.

The functions ``rkv_*`` mirror the C ABI one to one (raw device pointers as
ints, CUDA streams as ``cudaStream_t`` ints).  ``RollingKV`` is a convenience
owner of the caller-side buffers: it allocates the K/V pools, the state and
the workspace as torch CUDA tensors, checks shapes and dtypes, and forwards to
the C entry points on torch's current stream.  Every step of the hot path
runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "librkv.so")

RKV_OK, RKV_ERR_INVALID_ARG, RKV_ERR_UNSUPPORTED, RKV_ERR_CAPACITY, RKV_ERR_CUDA, \
    RKV_ERR_DEVICE_STATE = range(6)
RKV_BF16, RKV_F32 = 0, 1
RKV_PRE_ROPE, RKV_STORED_ROTATED = 0, 1
RKV_ROPE_SPLIT_HALF, RKV_ROPE_INTERLEAVED = 0, 1
RKV_ATTEND_AUTO, RKV_ATTEND_FMA, RKV_ATTEND_MMA, RKV_ATTEND_TC = 0, 1, 2, 3


class rkv_config(ctypes.Structure):
    _fields_ = [
        ("n_streams", c_int32), ("n_layers", c_int32), ("n_q_heads", c_int32),
        ("n_kv_heads", c_int32), ("head_dim", c_int32), ("capacity", c_int32),
        ("max_chunk", c_int32), ("kv_dtype", c_int32), ("q_dtype", c_int32),
        ("layout", c_int32), ("rope_style", c_int32), ("attend_impl", c_int32),
        ("rope_theta", c_double), ("softmax_scale", c_float), ("rebase_epoch", c_int32),
        ("window", c_int32), ("n_pinned", c_int32),
    ]


class rkv_buffers(ctypes.Structure):
    _fields_ = [("k_pool", c_void_p), ("v_pool", c_void_p), ("state", c_void_p),
                ("workspace", c_void_p), ("workspace_bytes", c_size_t)]


class RkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_lib = None


def load_library():
    """Loads librkv.so from the package; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m rolling_kv_cache_buffer_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P = c_void_p
    sig = {
        "rkv_required_bytes": (c_int32, [POINTER(rkv_config), POINTER(c_size_t),
                                         POINTER(c_size_t), POINTER(c_size_t)]),
        "rkv_create": (c_int32, [POINTER(rkv_config), POINTER(rkv_buffers), P, POINTER(P)]),
        "rkv_append": (c_int32, [P, P, P, c_int32, P, P]),
        "rkv_attend": (c_int32, [P, P, P, c_int32, c_int32, c_int32, P]),
        "rkv_attend_static_scratch": (c_int32, [P, P, P, c_int32, c_int32, c_int32, P]),
        "rkv_rebase": (c_int32, [P, P]),
        "rkv_step": (c_int32, [P, P, P, P, P, P, P]),
        "rkv_step_layers": (c_int32, [P, c_int32, c_int32, P, P, P, P, P, c_int32, P]),
        "rkv_destroy": (c_int32, [P]),
        "rkv_set_stream_state": (c_int32, [P, c_int32, c_int64, c_int32, P]),
        "rkv_reset_stream": (c_int32, [P, c_int32, c_int64, P, P, c_int32, P]),
        "rkv_get_stream_state": (c_int32, [P, P, P, P, P]),
        "rkv_last_launch_count": (c_int32, [P]),
        "rkv_status_string": (c_char_p, [c_int32]),
        "rkv_abi_version": (c_int32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().rkv_status_string(status).decode()


def _check(status: int, where: str):
    if status != RKV_OK:
        raise RkvError(status, where)


# --- the C ABI, one function each ------------------------------------------

def rkv_abi_version() -> int:
    return load_library().rkv_abi_version()


def rkv_required_bytes(cfg: rkv_config):
    a, b, c = c_size_t(), c_size_t(), c_size_t()
    _check(load_library().rkv_required_bytes(ctypes.byref(cfg), ctypes.byref(a),
                                             ctypes.byref(b), ctypes.byref(c)),
           "rkv_required_bytes")
    return a.value, b.value, c.value


def rkv_create(cfg: rkv_config, bufs: rkv_buffers, stream: int) -> int:
    h = c_void_p()
    _check(load_library().rkv_create(ctypes.byref(cfg), ctypes.byref(bufs), stream,
                                     ctypes.byref(h)), "rkv_create")
    return h.value


def rkv_append(h, k_new, v_new, n_new, step_log, stream):
    _check(load_library().rkv_append(h, k_new, v_new, n_new, step_log, stream), "rkv_append")


def rkv_attend(h, q, out, layer_begin, n_layers, n_q, stream):
    _check(load_library().rkv_attend(h, q, out, layer_begin, n_layers, n_q, stream),
           "rkv_attend")


def rkv_attend_static_scratch(h, q, out, layer_begin, n_layers, n_q, stream):
    """rkv_attend with its scratch in the library's static device array (for
    callers that cannot allocate device memory where they attend)."""
    _check(load_library().rkv_attend_static_scratch(h, q, out, layer_begin, n_layers, n_q,
                                                    stream), "rkv_attend_static_scratch")


def rkv_rebase(h, stream):
    _check(load_library().rkv_rebase(h, stream), "rkv_rebase")


def rkv_step_layers(h, layer_begin, n_layers, k_new, v_new, q, out, step_log, last, stream):
    _check(load_library().rkv_step_layers(h, layer_begin, n_layers, k_new, v_new, q, out,
                                          step_log, last, stream), "rkv_step_layers")


def rkv_step(h, k_new, v_new, q, out, step_log, stream):
    """Fused decode step: append one pair per stream, re-base, attend all layers."""
    _check(load_library().rkv_step(h, k_new, v_new, q, out, step_log, stream), "rkv_step")


def rkv_destroy(h):
    _check(load_library().rkv_destroy(h), "rkv_destroy")


def rkv_set_stream_state(h, s, origin, fill, stream):
    _check(load_library().rkv_set_stream_state(h, s, origin, fill, stream),
           "rkv_set_stream_state")


def rkv_reset_stream(h, s, origin, k, v, n_prefix, stream):
    """Utterance reset of stream s, with n_prefix prefix pairs (k, v) at its
    start (0: an empty window)."""
    _check(load_library().rkv_reset_stream(h, s, origin, k, v, n_prefix, stream),
           "rkv_reset_stream")


def rkv_get_stream_state(h, origins, fills, status, stream):
    _check(load_library().rkv_get_stream_state(h, origins, fills, status, stream),
           "rkv_get_stream_state")


def rkv_last_launch_count(h) -> int:
    return load_library().rkv_last_launch_count(h)


# --- convenience owner of the buffers ---------------------------------------

_DT = {"bf16": RKV_BF16, "f32": RKV_F32}
_LAYOUT = {"pre_rope": RKV_PRE_ROPE, "stored_rotated": RKV_STORED_ROTATED}
_STYLE = {"split_half": RKV_ROPE_SPLIT_HALF, "interleaved": RKV_ROPE_INTERLEAVED}
_IMPL = {"auto": RKV_ATTEND_AUTO, "fma": RKV_ATTEND_FMA, "mma": RKV_ATTEND_MMA,
         "tc": RKV_ATTEND_TC}


def make_config(n_streams, n_layers, n_q_heads, n_kv_heads, head_dim, capacity, max_chunk=1,
                kv_dtype="bf16", q_dtype=None, layout="pre_rope", rope_style="split_half",
                rope_theta=1e6, softmax_scale=0.0, attend_impl="auto",
                rebase_epoch=0, window=0, n_pinned=0) -> rkv_config:
    return rkv_config(n_streams, n_layers, n_q_heads, n_kv_heads, head_dim, capacity, max_chunk,
                      _DT[kv_dtype], _DT[q_dtype or kv_dtype], _LAYOUT[layout],
                      _STYLE[rope_style], _IMPL[attend_impl], float(rope_theta),
                      float(softmax_scale), int(rebase_epoch), int(window), int(n_pinned))


class RollingKV:
    """Owns the device buffers of one rolling cache and calls the C ABI."""

    def __init__(self, n_streams, n_layers, n_q_heads, n_kv_heads, head_dim, capacity,
                 max_chunk=1, kv_dtype="bf16", q_dtype=None, layout="pre_rope",
                 rope_style="split_half", rope_theta=1e6, softmax_scale=0.0,
                 attend_impl="auto", device="cuda", rebase_epoch=0, window=0, n_pinned=0):
        import torch
        self.torch = torch
        self.cfg = make_config(n_streams, n_layers, n_q_heads, n_kv_heads, head_dim, capacity,
                               max_chunk, kv_dtype, q_dtype, layout, rope_style, rope_theta,
                               softmax_scale, attend_impl, rebase_epoch, window, n_pinned)
        self.P = n_pinned
        self.Wr = window or capacity - n_pinned
        pool_b, state_b, ws_b = rkv_required_bytes(self.cfg)
        self.kv_dtype = torch.bfloat16 if kv_dtype == "bf16" else torch.float32
        self.q_dtype = torch.bfloat16 if (q_dtype or kv_dtype) == "bf16" else torch.float32
        self.S, self.L, self.Hq, self.Hkv = n_streams, n_layers, n_q_heads, n_kv_heads
        self.D, self.W, self.max_chunk = head_dim, capacity, max_chunk
        self.stored = layout == "stored_rotated"
        self.device = torch.device(device)
        shape = (n_streams, n_layers, n_kv_heads, capacity, head_dim)
        self.k_pool = torch.zeros(shape, dtype=self.kv_dtype, device=self.device)
        self.v_pool = torch.zeros(shape, dtype=self.kv_dtype, device=self.device)
        assert self.k_pool.numel() * self.k_pool.element_size() == pool_b
        self.state = torch.zeros(state_b, dtype=torch.uint8, device=self.device)
        self.workspace = torch.zeros(ws_b, dtype=torch.uint8, device=self.device)
        self.bufs = rkv_buffers(self.k_pool.data_ptr(), self.v_pool.data_ptr(),
                                self.state.data_ptr(), self.workspace.data_ptr(), ws_b)
        self.handle = rkv_create(self.cfg, self.bufs, self._stream())

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def _need(self, t, shape, dtype, name):
        if not t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape) or \
                not t.is_contiguous():
            raise ValueError(f"{name}: want contiguous CUDA {dtype} {tuple(shape)}, got "
                             f"{t.device} {t.dtype} {tuple(t.shape)}")

    def append(self, k_new, v_new, step_log=None):
        c = k_new.shape[2]
        shp = (self.L, self.S, c, self.Hkv, self.D)
        self._need(k_new, shp, self.kv_dtype, "k_new")
        self._need(v_new, shp, self.kv_dtype, "v_new")
        lp = 0
        if step_log is not None:
            self._need(step_log, (self.S, 4), self.torch.int64, "step_log")
            lp = step_log.data_ptr()
        rkv_append(self.handle, k_new.data_ptr(), v_new.data_ptr(), c, lp, self._stream())

    def attend(self, q, out=None, layer_begin=0):
        n_layers, c = q.shape[0], q.shape[2]
        self._need(q, (n_layers, self.S, c, self.Hq, self.D), self.q_dtype, "q")
        if out is None:
            out = self.torch.empty(q.shape, dtype=self.torch.float32, device=self.device)
        self._need(out, tuple(q.shape), self.torch.float32, "out")
        rkv_attend(self.handle, q.data_ptr(), out.data_ptr(), layer_begin, n_layers, c,
                   self._stream())
        return out

    def rebase(self):
        rkv_rebase(self.handle, self._stream())

    def step(self, k_new, v_new, q, out=None, step_log=None):
        """append(k_new, v_new) + rebase() + attend(q) for one token per stream,
        all layers, in one kernel launch (pre-RoPE bf16 caches)."""
        shp = (self.L, self.S, 1, self.Hkv, self.D)
        self._need(k_new, shp, self.kv_dtype, "k_new")
        self._need(v_new, shp, self.kv_dtype, "v_new")
        self._need(q, (self.L, self.S, 1, self.Hq, self.D), self.q_dtype, "q")
        if out is None:
            out = self.torch.empty(q.shape, dtype=self.torch.float32, device=self.device)
        self._need(out, tuple(q.shape), self.torch.float32, "out")
        lp = 0
        if step_log is not None:
            self._need(step_log, (self.S, 4), self.torch.int64, "step_log")
            lp = step_log.data_ptr()
        rkv_step(self.handle, k_new.data_ptr(), v_new.data_ptr(), q.data_ptr(), out.data_ptr(),
                 lp, self._stream())
        return out

    def step_layers(self, layer_begin, k_new, v_new, q, out, last, step_log=None):
        """The step for layers layer_begin .. layer_begin + n - 1 (n = k_new's
        first dimension): each layer range of a step once, `last` on the final
        call (it publishes the new stream states)."""
        n = k_new.shape[0]
        shp = (n, self.S, 1, self.Hkv, self.D)
        self._need(k_new, shp, self.kv_dtype, "k_new")
        self._need(v_new, shp, self.kv_dtype, "v_new")
        self._need(q, (n, self.S, 1, self.Hq, self.D), self.q_dtype, "q")
        self._need(out, tuple(q.shape), self.torch.float32, "out")
        lp = 0
        if step_log is not None:
            self._need(step_log, (self.S, 4), self.torch.int64, "step_log")
            lp = step_log.data_ptr()
        rkv_step_layers(self.handle, layer_begin, n, k_new.data_ptr(), v_new.data_ptr(),
                        q.data_ptr(), out.data_ptr(), lp, 1 if last else 0, self._stream())
        return out

    def set_stream_state(self, s, origin, fill):
        rkv_set_stream_state(self.handle, s, origin, fill, self._stream())

    def reset_stream(self, s, origin, k=None, v=None):
        """Utterance reset of stream s at `origin`, with the prefix k, v
        ([L][n][H_kv][D] of the cache type, keys before rotation) as the first
        pairs of its new window, or an empty window."""
        n, kp, vp = 0, 0, 0
        if k is not None:
            n = int(k.shape[1])
            shape = (self.L, n, self.Hkv, self.D)
            self._need(k, shape, self.kv_dtype, "k")
            self._need(v, shape, self.kv_dtype, "v")
            kp, vp = k.data_ptr(), v.data_ptr()
        rkv_reset_stream(self.handle, s, origin, kp, vp, n, self._stream())

    def get_stream_state(self):
        import numpy as np
        o = np.zeros(self.S, np.int64)
        f = np.zeros(self.S, np.int32)
        st = np.zeros(self.S, np.int32)
        rkv_get_stream_state(self.handle, o.ctypes.data, f.ctypes.data, st.ctypes.data,
                             self._stream())
        return o, f, st

    def last_launch_count(self):
        return rkv_last_launch_count(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            rkv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
