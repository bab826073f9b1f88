"""Helpers of the GPU parity tests: build a cache for a workload, seed windows,
and compare the CUDA path with the float64 oracle."""
import numpy as np
import torch

from oracle import rkv_oracle as O
from rolling_kv_cache_buffer_b300 import RollingKV

MAX_ABS, MEAN_ABS = 2e-2, 2e-3   # attention-output tolerance against the oracle


def make_cache(wl, layout="pre_rope", attend_impl="auto", max_chunk=None, style="split_half",
               n_streams=None):
    return RollingKV(n_streams or wl.n_streams, wl.n_layers, wl.n_q_heads, wl.n_kv_heads,
                     wl.head_dim, wl.capacity, max_chunk=max_chunk or wl.n_new,
                     kv_dtype=wl.kv_dtype, layout=layout, rope_style=style,
                     rope_theta=wl.rope_theta, attend_impl=attend_impl,
                     window=wl.window or 0)


def make_oracle(wl, cls=O.RollingCacheOracle, style="split_half", n_layers=None, n_streams=None):
    return cls(n_streams or wl.n_streams, n_layers or wl.n_layers, wl.n_q_heads, wl.n_kv_heads,
               wl.head_dim, wl.capacity, theta=wl.rope_theta, style=style, window=wl.window)


def dev(x, dtype):
    return x.to(dtype).cuda().contiguous()


def write_window(cache, s, origin, fill, k, v):
    """Place a window (k, v: [L][H_kv][fill][D], position order) into the
    pools at slots (origin + i) mod W and set the stream state."""
    W = cache.W
    slots = (torch.arange(fill, dtype=torch.int64) + origin) % W
    slots = slots.cuda()
    cache.k_pool[s][:, :, slots] = k.to(cache.kv_dtype).cuda()
    cache.v_pool[s][:, :, slots] = v.to(cache.kv_dtype).cuda()
    cache.set_stream_state(s, origin, fill)


def poison_outside(cache, origins, fills):
    """Fill every slot outside each stream's window with NaN."""
    W = cache.W
    for s, (o, n) in enumerate(zip(origins, fills)):
        keep = torch.zeros(W, dtype=torch.bool)
        keep[(torch.arange(n, dtype=torch.int64) + int(o)) % W] = True
        bad = (~keep).nonzero().flatten().cuda()
        if bad.numel():
            cache.k_pool[s][:, :, bad] = float("nan")
            cache.v_pool[s][:, :, bad] = float("nan")


def compare(gpu, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    g = gpu.detach().double().cpu().numpy() if torch.is_tensor(gpu) else np.asarray(gpu)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    err = np.abs(g - r)
    assert err.max() <= max_abs, f"max-abs {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"mean-abs {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())
