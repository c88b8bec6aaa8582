"""The multi-rank path of bench.py on CPU: two gloo ranks (one process per rank, as torchrun
launches them) agree on the slowest rank's time and on the whole-job aggregate, and the
reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(None)
    try:
        # rank r "took" r + 1.5 seconds: every rank must see the slowest one
        slowest = bench.max_over_ranks(r + 1.5, w, torch.device("cpu"))
        bench.barrier(w)
        value = bench.aggregate(100.0, 4, w, slowest)
        with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
            json.dump({"rank": r, "world": w, "local": local, "slowest": slowest, "value": value,
                       "backend": dist.get_backend()}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, g in enumerate(got):
        assert g["rank"] == r and g["world"] == world and g["local"] == r
        assert g["backend"] == "gloo"
        assert g["slowest"] == pytest.approx(world - 1 + 1.5)
        # whole-job throughput: units of all ranks over the slowest rank's time
        assert g["value"] == pytest.approx(100.0 * 4 * world / (world - 1 + 1.5))


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    """bench.py reports ncu DRAM traffic only while the hash of the kernel's code (the .cu file
    and the inline PTX helpers it includes, comments and layout left out) matches the one recorded
    with the counters, and only for the workload the counters were taken on."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    csrc = tmp_path / "block_sparse_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int kernel = 1;  // a comment\n")
    (csrc / "h.cuh").write_text("/* helpers */\nint helper = 2;\n")
    digest = hashlib.sha256(b"int kernel = 1;\nint helper = 2;\n").hexdigest()[:16]
    assert bench.source_digest([csrc / "k.cu", csrc / "h.cuh"]) == digest
    prof = tmp_path / "profiles"
    prof.mkdir()
    rec = {"k": {"source": ["k.cu", "h.cuh"], "source_sha256_16": digest, "bytes_per_launch": 1234,
                 "config": "C3"}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k", "C3") == 1234
    assert bench.traffic_record("k", "C2") is None          # taken on another workload
    assert bench.traffic_record("missing", "C3") is None
    # a comment or layout edit keeps the record, a code edit drops it
    (csrc / "k.cu").write_text("// reworded\n    int kernel = 1;   // another comment\n\n")
    assert bench.traffic_record("k", "C3") == 1234
    (csrc / "h.cuh").write_text("/* helpers */\nint helper = 3;\n")
    assert bench.traffic_record("k", "C3") is None
