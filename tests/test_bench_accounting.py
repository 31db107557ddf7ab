"""The benchmark's accounting on the CPU: the algorithmic bytes behind every GB/s and roofline
fraction, and how a capture of a workload's first sequences is scaled to the full launch."""
import os

import numpy as np

import bench
import pkv_workloads as W


def test_per_unit_bytes_follow_the_kv_layout():
    """One (cached token, KV head) reads K and V once: 2 * head_dim * element bytes (512 B for
    bf16 head_dim 128, 256 B for fp8 or for bf16 head_dim 64)."""
    expect = {"c0": 256, "c1": 512, "c2": 512, "c3": 512, "c4": 256}
    for name in W.WORKLOADS:
        w = W.make_workload(name)
        units = int(w.attend_lens.astype(np.int64).sum()) * w.Hkv
        b = bench.algorithmic_bytes(w)
        assert b["kv"] == units * expect[name], name
        assert b["attention"] >= b["kv"] and b["step"] == b["attention"] + b["append"]


def test_long_context_bytes_equal_the_closed_form():
    """c3 attends over fixed lengths 32k, 48k, ..., 128k, 128k (k = 1024) with 8 KV heads of 128
    bf16 elements: 704512 tokens x 8 heads x 512 B = 2,885,681,152 B of K/V, plus Q and out."""
    w = W.make_workload("c3")
    assert int(w.attend_lens.sum()) == 1024 * (32 + 48 + 64 + 80 + 96 + 112 + 128 + 128) == 704512
    b = bench.algorithmic_bytes(w)
    assert b["kv"] == 704512 * 8 * 2 * 128 * 2 == 2_885_681_152
    pages = int(((w.attend_lens + 63) // 64).sum())
    assert b["attention"] == b["kv"] + 2 * 8 * 64 * 128 * 2 + 4 * pages + 4 * 8
    assert b["append"] == 0


def test_fp8_bytes_include_one_scale_pair_per_page_and_head():
    w = W.make_workload("c4")
    L = w.attend_lens.astype(np.int64)
    pages = int(((L + 15) // 16).sum())
    b = bench.algorithmic_bytes(w)
    assert b["attention"] - b["kv"] == pages * w.Hkv * 8 + 2 * w.B * w.Hq * w.D * 2 + 4 * pages + 4 * w.B


def test_partial_captures_scale_by_algorithmic_bytes(tmp_path, monkeypatch):
    """A capture of a workload's first sequences ("c3[:2]") is scaled to the full launch by the
    ratio of algorithmic bytes; a capture taken on other kernel sources is not used."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "ncu_traffic.txt").write_text("# comment\nc3[:2] feedface 1000000 x.md\nc1 feedface 777 y.md\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "feedface")
    w3 = W.make_workload("c3")
    full = bench.algorithmic_bytes(w3)["attention"]
    part = bench.algorithmic_bytes(W.truncated(w3, 2))["attention"]
    got, note = bench.ncu_traffic(w3)
    assert got == int(round(1000000 * full / part)) and "scaled" in note
    assert bench.ncu_traffic(W.make_workload("c1"))[0] == 777
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0ther")
    assert bench.ncu_traffic(w3) == (None, None)
    assert os.path.exists(prof / "ncu_traffic.txt")


def test_append_launch_count_follows_the_library_paths():
    """gpu_launches counts the library's kernels: a bf16 append is one launch; a one-byte append
    one up to 1024 tokens and three above; a one-byte decode step of up to 1024 tokens appends
    inside its attention kernel (no append launch)."""
    import bench
    assert bench.append_launches("bf16", 200, in_step=True) == 1
    assert bench.append_launches("bf16", 4096) == 1
    assert bench.append_launches("fp8_e4m3", 200, in_step=True) == 0
    assert bench.append_launches("int8", 1024, in_step=True) == 0
    assert bench.append_launches("fp8_e4m3", 200) == 1
    assert bench.append_launches("int8", 1025, in_step=True) == 3
    assert bench.append_launches("fp8_e4m3", 4096) == 3
    assert bench.append_launches("fp8_e4m3", 0, in_step=True) == 0
