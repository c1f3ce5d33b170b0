"""bench.py's rank bookkeeping with two gloo ranks on the CPU.

Each rank scans its own batch (weak scaling): the seeds differ per rank, no
collective touches the data, and the reported time is the slowest rank's.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        seconds = 0.5 + rank                       # rank 1 is the slow one
        slowest = bench.max_over_ranks(seconds)
        seed = bench.rank_seed(1, r)
        gbs = bench.aggregate_gbs(402653184, w, 10, slowest)
        out[rank] = (r, w, local, slowest, seed, gbs)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, local, slowest, seed, gbs) in res.items():
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == pytest.approx(1.5)       # max over ranks, seen by every rank
        assert gbs == pytest.approx(402653184 * 2 * 10 / 1.5 / 1e9)
    assert res[0][4] == 1 and res[1][4] != res[0][4]  # rank 0 scans the named workload's own batch


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.aggregate_gbs(12, 1, 1, 1e-9) == pytest.approx(12.0)


def test_launches_per_step():
    """The bench's count of kernel launches per call (its gpu_launches claim) follows the plan:
    one for a single-launch mode, two for the speculative mode and the segmented register path,
    and for two-pass mode the reduce and apply launches plus those of the scan of the tile maps,
    which is itself two-pass on the long workload."""
    import linear_recurrence_scan_fp32_gb300 as lr
    plan = lr.linrec_plan_f32(1, 1 << 20, 64, sm_count=152)
    assert plan["speculative"] and bench.launches_per_step(plan, "forward") == 2
    plan = lr.linrec_plan_f32(1, 1 << 20, 64, sm_count=152, path="chunked", chunk_mode="twopass")
    inner = lr.linrec_plan_f32(1, plan["chunks"], 64, sm_count=152)
    assert inner["twopass"] and bench.launches_per_step(plan, "forward", inner) == 5
    assert bench.launches_per_step(lr.linrec_plan_f32(32, 4096, 256, sm_count=152), "forward") == 1
    plan = lr.linrec_plan_f32(7, 3000, 777, sm_count=152)
    assert plan["path_name"] == "regcarry" and plan["twopass"] and bench.launches_per_step(plan, "forward") == 2


def test_committed_traffic_follows_the_source_digest(tmp_path, monkeypatch):
    """The bench line's roofline.traffic comes from a committed capture only while the digest of the
    kernel sources it lists matches the tree; a capture on other sources is reported apart."""
    csrc = tmp_path / "linear_recurrence_scan_fp32_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.kernel_source_digest(["k.cu"])
    (tmp_path / "profiles" / "traffic_kern_work.txt").write_text(
        "# a capture\nkernel_sources: k.cu\n"
        f"kernel_source_sha256_16: {digest}\ndram_bytes_per_launch: 1234\n")
    assert bench.committed_traffic("kern", "work") == 1234
    assert bench.committed_capture("kern", "work") == (1234, True, "profiles/traffic_kern_work.txt")
    (csrc / "k.cu").write_text("kernel v2")
    assert bench.committed_traffic("kern", "work") is None
    assert bench.committed_capture("kern", "work") == (1234, False, "profiles/traffic_kern_work.txt")
    assert bench.committed_capture("kern", "other") is None


def _reference_arm(extra, env_over=None):
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env.update(env_over or {})
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3",
                        "--ref-seconds", "3"] + extra, cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    return lines


@pytest.mark.parametrize("extra", [["--workload", "pages"], ["--workload", "tiny", "--dtype", "bf16"]],
                         ids=("pages-f32", "tiny-bf16"))
def test_reference_arm_line(extra):
    """The reference arm (the oracle on host cores) prints one JSON line with the contract's keys, on a
    bounded sample of the named workload."""
    lines = _reference_arm(extra)
    assert len(lines) == 1
    line = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"]


def test_reference_arm_other_ranks_do_no_work():
    """Under torchrun only rank 0 runs the reference arm; the others exit 0 and print nothing."""
    lines = _reference_arm(["--workload", "pages"],
                           {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert lines == []
