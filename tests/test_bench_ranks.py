"""bench.py's multi-rank arithmetic on two gloo ranks (CPU): timing is the
maximum over ranks and the reported value is the whole job's work over it."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        elapsed = [40.0, 55.5][rank]                       # this rank's timed region, ms
        slowest = bench.max_over_ranks(elapsed, dist, "cpu")
        assert slowest == 55.5
        value = bench.job_throughput(2.0e12, 10, world, slowest)
        assert abs(value - 2.0e12 * 10 * world / 0.0555 / 1e12) < 1e-9
        env_ws, env_rank, _ = bench.dist_env()
        assert (env_ws, env_rank) == (1, 0) or env_ws == world
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port), nprocs=2, join=True)


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(1e12, 5, 1, 1000.0) == pytest.approx(5.0)


def test_general_options_parse_and_count():
    """The general-forward bench options: mask defaults follow the workload,
    packed lengths are seeded, positive and sum to the token count."""
    sys.path.insert(0, ROOT)
    import argparse

    import numpy as np

    import bench
    from exact_tiled_attention_fa2_gb300 import synthetic as sy

    w = sy.WORKLOADS[4]
    ns = dict(window_left=None, window_right=None, prefix=0, seqlen_k=0, layout="bhnd", varlen_seqs=0, decode_rows=0)
    assert bench.general_mask(argparse.Namespace(**ns), w) is None
    g = bench.general_mask(argparse.Namespace(**dict(ns, window_left=4095)), w)
    assert (g["window_left"], g["window_right"], g["seqlen_k"]) == (4095, 0, w.N)   # causal workload: right edge 0
    g = bench.general_mask(argparse.Namespace(**dict(ns, seqlen_k=20000)), w)
    assert g["seqlen_k"] == 20000 and "Nk20000" in g["label"]
    lens = bench.varlen_lengths(1 << 16, 37, 5)
    assert lens.sum() == 1 << 16 and lens.min() >= 1 and lens.size == 37
    np.testing.assert_array_equal(lens, bench.varlen_lengths(1 << 16, 37, 5))
    # a 4096-key window on a causal N=16384 problem: every row past the first 4095 sees 4096 keys
    vis = sy.visible_keys(16384, 16384, 4095, 0, 0)
    assert vis.sum() == sum(range(1, 4097)) + (16384 - 4096) * 4096
    g = bench.general_mask(argparse.Namespace(**dict(ns, decode_rows=1)), w)
    assert g["seqlen_q"] == 1 and g["seqlen_k"] == w.N and g["label"].startswith("decode 1 row vs 16384 keys")
    # one causal row facing the last of N keys sees all of them: K + V read once dominate the bytes
    assert g["input_bytes"] == (1 + 2 * w.N) * w.H * w.d * 2


def test_traffic_record_matches_kernel_source_and_workload(tmp_path, monkeypatch):
    """`roofline.traffic` comes only from a record taken on the same kernel
    source (hash), kernel name and workload; any other record, or one without
    a kernel name (an earlier forward kernel's), gives null."""
    sys.path.insert(0, ROOT)
    import bench

    hashes = {}

    def fake_hash(names=None):
        key = tuple(names or bench.KERNEL_SOURCES)
        return hashes.setdefault(key, "h%d" % len(hashes))

    monkeypatch.setattr(bench, "kernel_source_hash", fake_hash)
    fwd, bwd = fake_hash(bench.KERNEL_SOURCES), fake_hash(bench.BWD_KERNEL_SOURCES)
    assert fwd != bwd
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic_per_launch.txt").write_text(
        "# comment line\n"
        "kernel_sha=%s workload=4 bytes_per_launch=111\n" % fwd +                          # no kernel name
        "kernel_sha=old0 workload=4 kernel=fa2_fwd_dbuf_kernel bytes_per_launch=222\n"
        "kernel_sha=%s workload=3 kernel=fa2_fwd_dbuf_kernel bytes_per_launch=333\n" % fwd +
        "kernel_sha=%s workload=4 kernel=fa2_fwd_dbuf_kernel bytes_per_launch=444\n" % fwd +
        "kernel_sha=%s workload=4 kernel=fa2_bwd_kernel bytes_per_launch=555\n" % fwd +       # forward hash
        "kernel_sha=%s workload=4 kernel=fa2_bwd_kernel bytes_per_launch=666\n" % bwd)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic(4) == 444.0
    assert bench.recorded_traffic(3) == 333.0
    assert bench.recorded_traffic(2) is None
    assert bench.recorded_traffic(4, "fa2_bwd_kernel") == 666.0
    assert bench.recorded_traffic(4, "fa2_decode_kernel") is None
    hashes[tuple(bench.KERNEL_SOURCES)] = "changed"          # a kernel source edited since the capture
    assert bench.recorded_traffic(4) is None
    (tmp_path / "profiles" / "traffic_per_launch.txt").unlink()
    assert bench.recorded_traffic(4, "fa2_bwd_kernel") is None


def test_l2_flush_follows_input_size():
    """Inputs that fit in the 129 MB L2 are timed after an L2 overwrite:
    workloads 1, 2 and 5 forward.  Workloads 3 and 4 are larger, and so is
    workload 2's backward step, which also reads o, dO and L."""
    sys.path.insert(0, ROOT)
    import bench
    from exact_tiled_attention_fa2_gb300 import synthetic as sy

    fwd = {i: bench.flush_l2(bench.step_input_bytes(sy.WORKLOADS[i], None, False), "auto") for i in range(1, 6)}
    assert fwd == {1: True, 2: True, 3: False, 4: False, 5: True}
    bwd = {i: bench.flush_l2(bench.step_input_bytes(sy.WORKLOADS[i], None, True), "auto") for i in range(1, 6)}
    assert bwd == {1: True, 2: False, 3: False, 4: False, 5: True}
    assert bench.step_input_bytes(sy.WORKLOADS[4], None, False) == 3 * 32 * 16384 * 128 * 2
    assert bench.flush_l2(10 ** 12, "on") and not bench.flush_l2(1, "off")


def test_profile_commands_parse():
    """Every bench command a profile summary records parses with the bench's
    own options (and keeps at least 3 warm-up steps)."""
    import glob
    import shlex

    sys.path.insert(0, ROOT)
    import bench

    found = 0
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        text = open(path).read().replace("\\\n", " ")
        for line in text.splitlines():
            if "python bench.py" not in line:
                continue
            cmd = line.split("python bench.py", 1)[1]
            for stop in ("&&", ">", "|", "`"):
                cmd = cmd.split(stop, 1)[0]
            argv = shlex.split(cmd)
            args = bench.build_parser().parse_args(argv)
            assert args.warmup >= 3, (path, argv)
            found += 1
    assert found >= 8


def test_timing_regions_and_spread():
    """Regions of K steps are repeated until they add up to >= 1 s of device
    time (at least 3, at most MAX_REGIONS); the line reports their median."""
    sys.path.insert(0, ROOT)
    import bench

    assert bench.region_count(31.0) == 33            # 20 launches of 1.55 ms
    assert bench.region_count(2000.0) == 3           # long regions: still three
    assert bench.region_count(0.01) == bench.MAX_REGIONS
    assert bench.region_count(0.0) == bench.MAX_REGIONS
    t = bench.spread([3.0, 1.0, 2.0, 100.0, 2.0])
    assert t["regions"] == 5 and t["median_ms"] == 2.0 and t["min_ms"] == 1.0 and t["max_ms"] == 100.0
    assert t["total_s"] == pytest.approx(0.108)


def test_both_arms_report_the_same_config():
    sys.path.insert(0, ROOT)
    import bench
    from exact_tiled_attention_fa2_gb300 import synthetic as sy

    for wl in (1, 2, 4):
        args = bench.build_parser().parse_args(["--workload", str(wl)])
        w = sy.WORKLOADS[wl]
        c = bench.arm_config(args, w, None, 1)
        assert c["launch"] == bench.launch_mode(bench.flush_l2(bench.step_input_bytes(w, None, False), "auto"))
        assert c == bench.arm_config(bench.build_parser().parse_args(["--workload", str(wl), "--impl", "reference"]),
                                     w, None, 1)
