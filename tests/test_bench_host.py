"""Host logic of bench.py on CPU: the step's call sequence per layout, the
algorithmic bytes, and the source hash that keys the committed DRAM counters."""
import argparse

import bench
from rkv_inputs import WORKLOADS


def _args(**kw):
    a = dict(path="auto", no_fused=False, per_layer=False, graph=False, attend_impl="auto")
    a.update(kw)
    return argparse.Namespace(**a)


def test_auto_path_per_layout():
    q = WORKLOADS["qwen3b"]
    # Pre-RoPE keys: the fused step (faster on B300); the separate calls on request.
    assert bench.step_is_fused(q, "pre_rope", 0, _args())
    assert not bench.step_is_fused(q, "pre_rope", 0, _args(path="split"))
    assert bench.step_is_fused(q, "pre_rope", 0, _args(path="fused"))
    assert bench.step_is_fused(q, "pre_rope", 0, _args(per_layer=True))
    assert bench.step_is_fused(q, "pre_rope", 0, _args(graph=True))
    assert not bench.step_is_fused(q, "pre_rope", 0, _args(path="fused", no_fused=True))
    # Stored-rotated keys: fused only with a re-basing epoch.
    assert bench.step_is_fused(q, "stored_rotated", 4096, _args())
    assert not bench.step_is_fused(q, "stored_rotated", 4096, _args(path="split"))
    assert not bench.step_is_fused(q, "stored_rotated", 0, _args(path="fused"))


def test_fused_step_needs_one_bf16_pair_and_tensor_cores():
    assert not bench.step_is_fused(WORKLOADS["qwen3b_chunk6"], "pre_rope", 0, _args(path="fused"))
    assert not bench.step_is_fused(WORKLOADS["tiny"], "pre_rope", 0, _args(path="fused"))
    assert not bench.step_is_fused(WORKLOADS["qwen3b"], "pre_rope", 0,
                                   _args(path="fused", attend_impl="fma"))


def test_kv_bytes_per_step_closed_form():
    q = WORKLOADS["qwen3b"]
    # 36 layers x 2 KV heads x 4096 pairs x 128 dims x 2 bytes x (K and V)
    assert bench._kv_bytes_per_step(q, [4096]) == 36 * 2 * 4096 * 128 * 2 * 2 == 150_994_944
    assert bench._kv_bytes_per_step(q, [10, 20]) == 30 * 36 * 2 * 128 * 2 * 2


def test_code_hash_ignores_comments_and_layout_only():
    a = bench._code_only(b"int a = 1;  // note\n/* block\n comment */\nint b;\n")
    assert a == bench._code_only(b"int a = 1;\nint b;")
    assert a != bench._code_only(b"int a = 2;\nint b;")


def test_kernel_sources_include_their_headers():
    src = bench._sources(bench.KERNEL_SOURCE["attend_mma_step"])
    assert {"rkv_attend_mma.cu", "rkv_attend_pipe.cuh", "rkv_attend_common.cuh",
            "rkv_device.cuh", "rkv_api.cu"} <= set(src)
    assert "rkv_misc.cu" not in src and "rkv.h" not in src
    assert "rkv_misc.cu" in bench._sources(bench.KERNEL_SOURCE["rerotate"])


def test_pack_lays_out_aligned_views():
    """The e2e loop's packed buffer: each tensor's view starts on a 16-byte
    boundary, round-trips its contents, and the buffer holds nothing else
    beyond the alignment padding."""
    import torch
    q = torch.randn(36, 1, 1, 16, 128).bfloat16()
    k = torch.randn(36, 1, 1, 2, 128).bfloat16()
    x = torch.randn(3).bfloat16()
    flat, views = bench._pack([q, x, k], lambda n, dt: torch.empty(n, dtype=dt))
    for view, t in zip(views, (q, x, k)):
        view.copy_(t)
        assert torch.equal(view, t) and view.is_contiguous()
        assert (view.data_ptr() - flat.data_ptr()) % 16 == 0
    assert flat.numel() == q.numel() + 8 + k.numel()


def test_traffic_record_per_workload_and_scaling(tmp_path, monkeypatch):
    """`<kernel>@<workload>` wins over the plain kernel record; a record that
    names another workload or another source hash gives None; a record with
    the captured launch's algorithmic bytes scales to the line's bytes."""
    import json
    (tmp_path / "profiles").mkdir()
    d = {"k": {"bytes_per_launch": 100, "source_hash": "h", "workload": "qwen3b (--x)"},
         "k@grow": {"bytes_per_launch": 110, "algorithmic_bytes": 100, "source_hash": "h",
                    "workload": "grow"},
         "k@old": {"bytes_per_launch": 7, "source_hash": "stale", "workload": "old"}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(d))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda key: "h")
    assert bench._traffic("k", "qwen3b", 1) == 100
    assert bench._traffic("k", "audio8", 1) is None
    assert bench._traffic("k", "grow", 200) == 220
    assert bench._traffic("k", "old", 1) is None
    assert bench._traffic("other", "qwen3b", 1) is None


def test_committed_traffic_records_are_well_formed():
    """Every record in profiles/dram_traffic.json names a timed kernel and a
    workload that bench.py runs, and its bytes add up; a record keyed
    <kernel>@<workload> names that workload."""
    import json
    import os
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        d = json.load(f)
    assert d
    for key, e in d.items():
        kernel = key.split("@")[0]
        assert kernel in bench.KERNEL_SOURCE, key
        assert e["source"] == bench.KERNEL_SOURCE[kernel]
        assert e["bytes_per_launch"] == e["dram_read"] + e["dram_write"] > 0
        wl = e["workload"].split(" ")[0]
        assert wl in bench.WORKLOAD_TEXT, key
        if "@" in key:
            assert key.split("@")[1] == wl
        if "algorithmic_bytes" in e:
            assert 1.0 <= e["bytes_per_launch"] / e["algorithmic_bytes"] < 1.1, key
