"""Benchmark of the fused GEMM-epilogue block on GB300.

Default workload: the LLaMA-3-1B attention-out block, bf16 in / fp32
accumulate, M = 8192 tokens (batch 4 x seq 2048):
    h = R + X Wo            X [8192, 2048], Wo [2048, 2048]   coda_gemm_residual_partial_rms
    r = rms(h)                                                 coda_rms_reduce
    act = SwiGLU(r h Wg', r h Wu')   Wg, Wu [2048, 8192]       coda_gemm_swiglu
One step = one pass of that chain over one batch (3 kernel launches).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl coda|reference|unfused]

Prints ONE JSON line (rank 0).  ``value`` is the whole-job TFLOP/s with
inputs resident in HBM (3 rotating input sets of 136 MB each, so every step
reads inputs that are not in the 129 MB L2); ``e2e`` is the same metric
with the inputs copied in from pinned host memory and h and act copied back
every step; ``roofline`` is the SwiGLU GEMM (89% of the flops) timed live
with CUDA events around each of its launches; ``cpu_baseline`` is the fp64
CPU oracle timed on this host on a bounded row sample.  Multi-GPU: one
process per GPU (torchrun), each rank runs its own independent batch (weak
scaling, no collective on the data path; a barrier and a max-reduce of the
elapsed time bracket the timed region).
``--impl reference`` times the CPU oracle alone; ``--impl unfused`` times the
unfused PyTorch sequence (cuBLAS GEMM, add, RMSNorm, GEMM, silu*mul).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from coda_inputs import WORKLOADS, make_inputs  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NSETS = 3


# ------------------------------------------------------------------ helpers ----

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def flops_swiglu_chain(M, K1, N, I):
    return {"gemm_residual": 2.0 * M * N * K1, "swiglu": 2.0 * M * 2 * I * N}


def algorithmic_bytes(M, K1, N, I, T):
    """Compulsory HBM bytes of one step: every tensor read or written once."""
    b = 2  # bf16
    fused = {
        "gemm_residual": M * K1 * b + N * K1 * b + M * N * b + M * N * b + M * T * 4,  # X, Wo, R, h, P
        "rms_reduce": M * T * 4 + M * 4,
        "swiglu": M * N * b + 2 * I * N * b + M * 4 + M * I * b,  # h, Wg, Wu, r, act
    }
    unfused = (M * K1 * b + N * K1 * b + M * N * b          # X Wo -> XW
               + 3 * M * N * b                               # XW + R -> h
               + 2 * M * N * b                               # RMSNorm(h) -> y
               + M * N * b + 2 * I * N * b + 2 * M * I * b   # y [Wg Wu] -> gu
               + 2 * M * I * b + M * I * b)                  # silu(g) * u -> act
    return fused, unfused


def kernel_source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_epilogue_fusion_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", f"ncu_{kernel_tag}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_b) or m_sha.group(1) != kernel_source_sha():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.path = None
        sel = []
        try:
            uuid = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
            if uuid is not None:
                s = str(uuid)
                sel = ["-i", s if s.startswith("GPU-") else "GPU-" + s]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100"]

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        power = [num(r[2]) for r in rows]
        pmax = max([p for p in power if p is not None] or [0.0])
        loaded = [r for r, p in zip(rows, power) if p is not None and p >= 0.5 * pmax] or rows
        sm = [num(r[0]) for r in loaded if num(r[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(loaded[0][1]),
                "power_w_max": pmax, "samples": len(loaded), "reasons": reasons}


def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


# ------------------------------------------------------------- CPU oracle ----

def oracle_sample(w, inp, budget_s, min_rows=16, max_rows=8192):
    """Time the fp64 oracle on the first rows of the workload (rows of the
    block are independent).  Returns (rows, seconds, flops, threads)."""
    import oracle
    Wt = lambda t: t.double().numpy().T.copy()  # noqa: E731
    W1, Wg, Wu = Wt(inp["W1t"]), Wt(inp["Wgt"]), Wt(inp["Wut"])
    g = inp["gamma1"].double().numpy()
    X = inp["X"].double().numpy()
    R = inp["R"].double().numpy()
    per_row = 2.0 * (w.K1 * w.N + 2 * w.N * w.N2)

    def run(n):
        t0 = time.perf_counter()
        oracle.block_swiglu(X[:n], W1, R[:n], g, Wg, Wu, w.eps)
        return time.perf_counter() - t0
    run(min_rows)  # warm (thread pool, pages)
    t = run(min_rows)
    n = int(max(min_rows, min(max_rows, budget_s / max(t, 1e-6) * min_rows)))
    dt = run(n)
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    return n, dt, per_row * n, threads


# -------------------------------------------------------------- the arms ----

def run_reference(args, w):
    dist, rank, ws = dist_setup("gloo")
    if rank != 0:
        return
    inp = make_inputs(w)
    import oracle
    Wt = lambda t: t.double().numpy().T.copy()  # noqa: E731
    W1, Wg, Wu = Wt(inp["W1t"]), Wt(inp["Wgt"]), Wt(inp["Wut"])
    g = inp["gamma1"].double().numpy()
    X = inp["X"].double().numpy()
    R = inp["R"].double().numpy()
    per_row = 2.0 * (w.K1 * w.N + 2 * w.N * w.N2)
    threads = int(os.environ.get("OMP_NUM_THREADS", len(os.sched_getaffinity(0))))
    # size each step's row sample so that warm-up + timed steps end in ~2 minutes
    t0 = time.perf_counter()
    oracle.block_swiglu(X[:threads], W1, R[:threads], g, Wg, Wu, w.eps)
    t_min = time.perf_counter() - t0
    budget = args.ref_budget / max(args.steps + args.warmup, 1)
    rows = int(max(threads, min(1024, threads * budget / max(t_min, 1e-6))))
    rows = min(rows, w.M)
    for s in range(args.warmup):
        o = (s * rows) % (w.M - rows + 1)
        oracle.block_swiglu(X[o:o + rows], W1, R[o:o + rows], g, Wg, Wu, w.eps)
    t0 = time.perf_counter()
    for s in range(args.steps):
        o = (s * rows) % (w.M - rows + 1)
        oracle.block_swiglu(X[o:o + rows], W1, R[o:o + rows], g, Wg, Wu, w.eps)
    dt = time.perf_counter() - t0
    value = per_row * rows * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows of the {w.M}-row batch per step (rows are independent), "
                                   f"fp64 unfused oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "fused GEMM-epilogue chain TFLOP/s and % of GB300 dense peak; DRAM bytes vs unfused"


def config_of(w):
    return {"workload": w.name, "chain": "gemm_residual_partial_rms -> rms_reduce -> gemm_swiglu",
            "M": w.M, "hidden": w.N, "K1": w.K1, "intermediate": w.N2, "eps": w.eps, "seed": w.seed,
            "l2": f"{NSETS} rotating input sets of 136 MB each (> 129 MB L2); no flush"}


def run_coda(args, w):
    dist, rank, ws = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain

    g.load_library()
    inp = make_inputs(w)
    M, K1, N, I = w.M, w.K1, w.N, w.N2
    T = g.coda_partial_cols(N)
    # independent batches per rank: same shapes, rank-specific data
    sets = []
    for s in range(NSETS):
        d = {k: v.to(dev) for k, v in inp.items()}
        if s or rank:
            gen = torch.Generator(device=dev).manual_seed(1000 * rank + s)
            d["X"] = torch.randn(M, K1, generator=gen, device=dev).bfloat16()
            d["R"] = torch.randn(M, N, generator=gen, device=dev).bfloat16()
        Wg = g.coda_fold_gamma(d["Wgt"], d["gamma1"])
        Wu = g.coda_fold_gamma(d["Wut"], d["gamma1"])
        if s:  # distinct weight copies so each step also reads its weights from HBM
            d["W1t"] = d["W1t"].clone()
        bufs = {"h": torch.empty(M, N, dtype=torch.bfloat16, device=dev),
                "P": torch.empty(M, T, dtype=torch.float32, device=dev),
                "r": torch.empty(M, dtype=torch.float32, device=dev),
                "act": torch.empty(M, I, dtype=torch.bfloat16, device=dev)}
        sets.append((d["X"], d["W1t"], d["R"], Wg, Wu, bufs))
    torch.cuda.synchronize()

    fl = flops_swiglu_chain(M, K1, N, I)
    step_flops = sum(fl.values())
    stream = torch.cuda.current_stream(dev)

    def step(i, ev=None):
        X, W1t, R, Wg, Wu, b = sets[i % NSETS]
        h, P = g.coda_gemm_residual_partial_rms(X, W1t, R, b["h"], b["P"])
        r = g.coda_rms_reduce(P, N, w.eps, b["r"])
        if ev is not None:
            ev[0].record(stream)
        g.coda_gemm_swiglu(h, Wg, Wu, r, b["act"])
        if ev is not None:
            ev[1].record(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step(i)
    g.coda_get_device_status()
    barrier()

    # ---- timed region: K steps, inputs resident in HBM
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        t_start.record(stream)
        for i in range(args.steps):
            step(i, evs[i])
        t_end.record(stream)
        barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    sw_ms = statistics.fmean(a.elapsed_time(b) for a, b in evs)
    g.coda_get_device_status()
    elapsed_max = elapsed
    if dist is not None:
        t = torch.tensor([elapsed], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_max = float(t.item())
    value = step_flops * args.steps * ws / elapsed_max / 1e12

    # ---- end to end: pinned host inputs in, h and act out, every step
    e2e_steps = max(10, min(200, args.steps // 10))
    X, W1t, R, Wg, Wu, b = sets[0]
    hX = torch.empty(X.shape, dtype=X.dtype, pin_memory=True).copy_(X.cpu())
    hR = torch.empty(R.shape, dtype=R.dtype, pin_memory=True).copy_(R.cpu())
    hh = torch.empty(b["h"].shape, dtype=torch.bfloat16, pin_memory=True)
    hact = torch.empty(b["act"].shape, dtype=torch.bfloat16, pin_memory=True)
    dX, dR = torch.empty_like(X), torch.empty_like(R)

    def e2e_step():
        dX.copy_(hX, non_blocking=True)
        dR.copy_(hR, non_blocking=True)
        chain.swiglu_block(dX, W1t, dR, Wg, Wu, w.eps, b)
        hh.copy_(b["h"], non_blocking=True)
        hact.copy_(b["act"], non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_s = e0.elapsed_time(e1) / 1e3
    if dist is not None:
        t = torch.tensor([e2e_s], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_val = step_flops * e2e_steps * ws / e2e_s / 1e12
    h2d = hX.numel() * hX.element_size() + hR.numel() * hR.element_size()
    d2h = hh.numel() * 2 + hact.numel() * 2

    if rank != 0:
        return
    pk, pk_kind = peaks()
    achieved = fl["swiglu"] / (sw_ms / 1e3) / 1e12
    fused_b, unfused_b = algorithmic_bytes(M, K1, N, I, T)
    roof = {"kernel": "gemm_swiglu (tcgen05, bf16)", "bound": "tensor", "achieved": achieved,
            "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
            "peak_kind": f"bf16 burst, {pk_kind}",
            "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
            "traffic": recorded_traffic("gemm_swiglu_llama1b"),
            "algorithmic_bytes": fused_b["swiglu"], "avg_launch_ms": sw_ms}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w),
        "frac_of_peak": value / ws / pk["bf16_tflops"],
        "dram_bytes_algorithmic": {"fused": sum(fused_b.values()), "unfused": unfused_b},
        "roofline": roof,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        n, dt, fl_cpu, threads = oracle_sample(w, inp, args.cpu_budget)
        line["cpu_baseline"] = {"value": fl_cpu / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {n} of {M} rows of the same batch (rows are independent), "
                                          f"{dt:.1f} s of fp64 unfused oracle"}
    print(json.dumps(line), flush=True)


def run_unfused(args, w):
    """cuBLAS + PyTorch eager, unfused: XW, add, RMSNorm (fp32 math), GEMM, silu*mul."""
    dist, rank, ws = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_inputs(w)
    d = {k: v.to(dev) for k, v in inp.items()}
    Wgu = torch.cat([d["Wgt"], d["Wut"]], 0)
    gamma = d["gamma1"]

    def step():
        h = torch.matmul(d["X"], d["W1t"].t()) + d["R"]
        hf = h.float()
        y = (hf * torch.rsqrt(hf.pow(2).mean(-1, keepdim=True) + w.eps) * gamma).bfloat16()
        gu = torch.matmul(y, Wgu.t())
        g_, u = gu.chunk(2, dim=-1)
        return h, torch.nn.functional.silu(g_) * u

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    dt = a.elapsed_time(b) / 1e3
    fl = sum(flops_swiglu_chain(w.M, w.K1, w.N, w.N2).values())
    if rank == 0:
        print(json.dumps({"impl": "unfused_torch_eager", "metric": METRIC, "value": fl * args.steps / dt / 1e12,
                          "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": dt / args.steps * 1e3, "dtype": "bf16", "config": config_of(w)}),
              flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["coda", "reference", "unfused"], default="coda")
    ap.add_argument("--workload", default="llama1b_attn_out_swiglu", choices=["llama1b_attn_out_swiglu"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work for warm-up + timed steps together")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif args.impl == "unfused":
        run_unfused(args, w)
    else:
        run_coda(args, w)


if __name__ == "__main__":
    main()
