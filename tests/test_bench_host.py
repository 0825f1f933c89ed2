"""Host logic of bench.py: the multi-rank path (gloo, world size 2, CPU),
the algorithmic byte count, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, world)
    q.put((rank, t, bench.rank_seed(7, rank)))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_own_seeds():
    import torch.multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    out = sorted(q.get() for _ in range(2))
    assert [t for _, t, _ in out] == [2.0, 2.0]          # max over ranks
    assert out[0][2] != out[1][2]                        # every rank its own batch


def test_algorithmic_bytes():
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_verification_25_gb300 import synth
    w = synth.make("long_draft_mixed_t", seed=0, rows=[0, 1, 2])   # row 0 greedy
    acc = np.array([3, 8, 2])
    p1, p2 = bench.algorithmic_bytes(w, acc)
    V, K = w.V, w.K
    assert p1 == 3 * (K + 1) * V * 4 + 2 * K * V * 4      # greedy row reads no draft rows
    assert p2 == (1 + 2) * V * 4                          # row 1 bonus (1 row), row 2 residual (2 rows)


def test_algorithmic_bytes_ragged_rows():
    sys.path.insert(0, ROOT)
    import dataclasses
    import bench
    from speculative_decoding_verification_25_gb300 import synth
    w = synth.make("llama3_ragged", seed=0, rows=[0, 1, 2])
    w = dataclasses.replace(w, k_per_row=np.array([0, 2, 4], np.int32))
    acc = np.array([0, 1, 4])                              # bonus, rejection at 1, bonus
    p1, p2 = bench.algorithmic_bytes(w, acc)
    V = w.V
    # rows read: K_b + 1 target rows and K_b draft rows (all rows tempered)
    assert p1 == ((0 + 1) + 0 + (2 + 1) + 2 + (4 + 1) + 4) * V * 2
    assert p2 == (1 + 2 + 1) * V * 2
    np.testing.assert_array_equal(bench.row_lengths(w), [0, 2, 4])


def test_ragged_reference_arm_counts_verified_positions():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--workload", "llama3_ragged"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0


def test_reference_arm_prints_one_json_line():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--workload", "tiny_stochastic"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_stored_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    # the hash is taken over the real sources; only the summary file is fake
    rev = bench.kernel_rev("sv_row_stats_kernel")
    (prof / "sv_row_stats_kernel_w.md").write_text(
        f"# x\n\n- kernel_rev: {rev}\n- dram_bytes_per_launch: 12345\n")
    (prof / "sv_row_stats_kernel_old.md").write_text(
        "- kernel_rev: 000000000000\n- dram_bytes_per_launch: 999\n")
    real_root = bench.ROOT
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_rev", lambda kernel="sv_row_stats_kernel": rev)
    assert bench.stored_traffic("w") == 12345
    assert bench.stored_traffic("old") is None        # taken on other sources
    assert bench.stored_traffic("missing") is None
    monkeypatch.setattr(bench, "ROOT", real_root)
    assert set(bench.KERNEL_SOURCES) == {"sv_row_stats_kernel", "sv_row_stats_compact_kernel",
                                         "sv_draw_kernel", "sv_tree_kernel"}
    csrc = os.path.join(ROOT, "speculative_decoding_verification_25_gb300", "csrc")
    for files in bench.KERNEL_SOURCES.values():
        assert all(os.path.exists(os.path.join(csrc, f)) for f in files)


def test_tree_reference_arm_runs():
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--workload", "llama3_tree"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0


def test_kernel_rev_ignores_comments_but_not_code():
    sys.path.insert(0, ROOT)
    import bench
    a = "int f(int x) {  // doubles\n  return 2 * x; /* a\n block */ }\n"
    b = "int f(int x) {\n  // another comment\n  return 2 * x;   }"
    c = "int f(int x) { return 3 * x; }"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
