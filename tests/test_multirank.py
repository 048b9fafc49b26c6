"""Two-rank paths of bench.py on CPU (gloo), launched the way a multi-GPU
bench run is: torchrun, one process per rank, rendezvous on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout=300):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), *args]
    env = dict(os.environ, OMP_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def test_rank_aggregation_takes_the_slowest_rank(tmp_path):
    r = _torchrun([os.path.join(ROOT, "tests", "multirank_worker.py"), str(tmp_path)])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads((tmp_path / f"rank{i}.json").read_text()) for i in range(2)]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    for d in lines:
        assert d["world"] == 2
        assert d["max_ms"] == 15.0                       # both ranks see the slower rank's time
        assert abs(d["rate"] - 2 * 1000 * 4 / 0.015) < 1e-6   # units of both ranks over that time


def test_reference_arm_runs_on_rank_zero_only():
    r = _torchrun(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
                   "--workload", "tiny", "--ref-rows", "16"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]


def test_job_rate_formula():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_rate(1, 32768, 10, 70.0) == 32768 * 10 / 0.070
    assert bench.job_rate(8, 32768, 10, 70.0) == 8 * bench.job_rate(1, 32768, 10, 70.0)


def test_reference_arm_line_keeps_the_contract():
    """One process: the reference arm's JSON line carries every key of the
    bench contract (the oracle timed on the host cores)."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1",
                        "--workload", "tiny", "--ref-rows", "16"], cwd=ROOT, capture_output=True, text=True,
                       timeout=300, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and "workload" in d["config"]
    assert set(d["cpu_baseline"]) >= {"value", "unit", "cores", "kind", "sample"}
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert abs(d["ms_per_step"] * d["steps"] / 1e3 * d["value"] - 2 * 8) < 1e-6 * d["value"] + 1e-6


def test_topk_overlap_helper():
    """bench.py's per-row top-k overlap (used by the table's MXFP8-vs-BF16
    column): ascending rows with -1 padding past each row's length."""
    import importlib.util

    import torch

    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    a = torch.tensor([[1, 3, 5, -1], [2, 4, 6, 8], [7, -1, -1, -1]], dtype=torch.int32)
    b = torch.tensor([[1, 5, 7, -1], [2, 4, 6, 8], [0, 9, -1, -1]], dtype=torch.int32)
    la = torch.tensor([3, 4, 1])
    lb = torch.tensor([3, 4, 2])
    mean, mn = bench.topk_overlap(a, la, b, lb)
    assert abs(mean - (2 / 3 + 1 + 0) / 3) < 1e-12 and mn == 0.0
    # a row against itself overlaps fully, padding never counts
    mean, mn = bench.topk_overlap(a, la, a, la)
    assert mean == 1.0 and mn == 1.0
