"""The N > 1 launch path on the CPU: bench.py under torchrun with two gloo
ranks.  The reference arm runs on rank 0 only and prints one JSON line; the
other rank exits 0 without work (the block is row-independent, so ranks never
exchange data)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, OMP_NUM_THREADS="2", MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29517", os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "3", "--ref-budget", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def _rank_main(rank, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    d, r, ws = bench.dist_setup("gloo")
    # rank 1 is the slower one: the job's time is its time
    t = bench.max_over_ranks([0.5, 2.0][r], d, "cpu")
    out.put((r, ws, t, bench.job_tflops(1e12, 10, ws, t)))
    d.barrier()
    d.destroy_process_group()


def test_coda_arm_aggregates_over_ranks_with_gloo():
    """The GPU arm's multi-rank bookkeeping (bench.dist_setup, max_over_ranks,
    job_tflops), run as two gloo ranks on the CPU: every rank sees the slowest
    rank's time, and the whole-job value counts both ranks' work."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 29531, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, ws, t, v in res:
        assert ws == 2 and t == 2.0
        assert v == 1e12 * 10 * 2 / 2.0 / 1e12
