"""Multi-rank host logic of the benchmark, run as world-size-2 gloo process groups on CPU.

With N GPUs every rank runs its own replica of the workload (heads are independent, so
the forward shards with no exchange in the data path).  What the ranks share is control
only: the barriers around the timed region, the max-over-ranks reduction of the elapsed
time, the whole-job throughput and the rule that rank 0 alone prints.  These tests cover
that logic without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    from chunked_scan_mixer_gb300 import inputs

    d = bench.Dist("gloo")
    try:
        assert d.on and d.world == world and d.rank == rank
        d.barrier()
        local_ms = 1.25 * (rank + 1)  # rank-dependent "elapsed time"
        ms = d.max(local_ms)
        value = bench.weak_scaling_value(d.world, 1000, ms)
        w = inputs.WORKLOADS["tiny"]
        x = inputs.make(w, seed=bench.replica_seed(w.seed, d.rank))
        d.barrier()
        out_q.put({"rank": rank, "ms": ms, "value": value, "q0": float(x["q"].flatten()[0])})
    finally:
        d.close()


def test_two_rank_max_and_aggregate():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort(key=lambda r: r["rank"])
    # every rank sees the slowest rank's time, and the same whole-job throughput
    assert res[0]["ms"] == res[1]["ms"] == pytest.approx(2.5)
    assert res[0]["value"] == res[1]["value"] == pytest.approx(2 * 1000 / 2.5e-3)
    # each rank drew its own replica
    assert res[0]["q0"] != res[1]["q0"]


def test_weak_scaling_value_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.weak_scaling_value(1, 1_048_576, 0.5) == pytest.approx(1_048_576 / 0.5e-3)
    assert bench.replica_seed(3, 0) == 3 and bench.replica_seed(3, 2) == 2003


def test_torchrun_reference_arm_prints_once():
    """`bench.py --impl reference` under a 2-rank launch: rank 0 alone runs and prints one
    JSON line, the other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert abs(rec["ms_per_step"] - 1e3 * 16 * 65536 / rec["value"]) <= 1e-6 * rec["ms_per_step"]
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_survives_comment_edits(tmp_path, monkeypatch):
    """The recorded DRAM traffic stays valid through an edit of comments or blank lines in
    the kernel sources and turns null on an edit of code."""
    import shutil
    import bench

    rels = ("chunked_scan_mixer_gb300/csrc/fwd_chunk_tc.cu", "chunked_scan_mixer_gb300/csrc/tc_common.cuh",
            "chunked_scan_mixer_gb300/csrc/common.cuh")
    for rel in rels + ("profiles/traffic.json",):
        (tmp_path / rel).parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, rel), tmp_path / rel)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha()
    rec = json.loads((tmp_path / "profiles/traffic.json").read_text())
    rec["segment_summaries"]["source_sha"] = sha
    (tmp_path / "profiles/traffic.json").write_text(json.dumps(rec))
    want = rec["segment_summaries"]["bytes_per_launch"]
    assert bench.recorded_traffic("segment_summaries") == want

    src = tmp_path / rels[0]
    text = src.read_text()
    src.write_text("// an added comment line\n\n" + text.replace("\n", "   // trailing note\n", 3))
    assert bench.kernel_source_sha() == sha
    assert bench.recorded_traffic("segment_summaries") == want

    src.write_text(text + "\nstatic int added_code_line = 0;\n")
    assert bench.kernel_source_sha() != sha
    assert bench.recorded_traffic("segment_summaries") is None
