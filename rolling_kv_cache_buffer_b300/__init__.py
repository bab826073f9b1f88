"""Rolling KV cache with exact RoPE re-basing, B300-native (sm_103a).

The hot path lives in librkv.so (CUDA kernels behind the C ABI of
include/rkv.h); this package is its Python binding.
"""
from .rkv import (  # noqa: F401
    RollingKV, RkvError, load_library, make_config, rkv_config, rkv_buffers, status_string,
    rkv_abi_version, rkv_required_bytes, rkv_create, rkv_append, rkv_attend, rkv_attend_static_scratch, rkv_rebase,
    rkv_step, rkv_step_layers, rkv_destroy, rkv_set_stream_state, rkv_reset_stream,
    rkv_get_stream_state,
    rkv_last_launch_count, LIB_PATH)
