"""Benchmark of the fused GEMM-epilogue chain on GB300.

Default workload: the LLaMA-3-8B block tail, bf16 in / fp32 accumulate,
M = 16384 tokens (batch 8 x seq 2048), hidden 4096, intermediate 14336:
    h1 = R + X Wo                 X [16384, 4096], Wo [4096, 4096]   residual + partial RMS program
    act = SwiGLU(r1 h1 Wg', r1 h1 Wu')   Wg, Wu [4096, 14336]         SwiGLU program, r1 reduced in its epilogue
    h2 = h1 + act Wd              Wd [14336, 4096]                    residual + partial RMS program
    Z = r2 h2 Wq'                 Wq [4096, 6144]                     row-scale program (next layer's QKV)
7146.8 GFLOP per step.  One step = one pass of that chain over one batch.
The default ``--reduce block`` runs it as two two-phase launches
(coda_block_swiglu, then coda_block_rowscale); ``--reduce fused`` as 4
launches (each reduction in its consumer's epilogue); ``--reduce separate``
as 6 (coda_rms_reduce launches).  ``--workload`` selects the other
configurations and ``--pass backward|aux`` the backward chain or the
memory-bound kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl coda|reference|unfused]

Prints ONE JSON line (rank 0).  ``value`` is the whole-job TFLOP/s with
inputs resident in HBM (3 rotating sets of X, R and the weights, each larger
than the 129 MB L2, so every step reads inputs that are not in L2); ``e2e``
is the same metric with X and R copied in from pinned host memory and the
chain's outputs copied back every step (copies of one step overlapped with
the compute of its neighbours); ``roofline`` is the dominant kernel (the
first block kernel by default) timed live with CUDA events around each of
its launches; ``sustained`` repeats the step for a window of seconds, with
the clocks sampled inside that window, so the figure holds under the power
cap; ``cpu_baseline`` is the fp64 CPU oracle timed on this host on a bounded
row sample.  Multi-GPU: one process per GPU (torchrun), each rank runs its
own independent batch (weak scaling, no collective on the data path; a
barrier and a max-reduce of the elapsed time bracket the timed region).
``--impl reference`` times the CPU oracle alone; ``--impl unfused`` times the
unfused PyTorch sequence (cuBLAS GEMM, add, RMSNorm, GEMM, silu*mul),
``--compile`` the same under torch.compile.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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


def chain_bytes_full(w, T):
    """Compulsory HBM bytes of one step of the 8B chain (bf16), fused (the two
    one-launch blocks: every operand, residual, output, partial and row scale
    once) and unfused (cuBLAS-style GEMMs with the add, RMSNorm and silu*mul as
    separate passes, each reading its inputs and writing its output once)."""
    b, M, H, I, Q, K1 = 2, w.M, w.N, w.inter, w.N2, w.K1
    fused = (b * (M * K1 + H * K1 + 2 * M * H) + 4 * M * T                  # X, Wo, R -> h1, P1
             + b * (M * H + 2 * I * H + M * I) + 4 * M * T + 4 * M          # h1, Wg, Wu, P1 -> act, r1
             + b * (M * I + H * I + 2 * M * H) + 4 * M * T                  # act, Wd, h1 -> h2, P2
             + b * (M * H + Q * H + M * Q) + 4 * M * T + 4 * M)             # h2, Wq, P2 -> Z, r2
    unfused = b * (M * K1 + H * K1 + M * H                                  # X Wo -> XW
                   + 3 * M * H                                              # XW + R -> h1
                   + 2 * M * H                                              # RMSNorm(h1) -> y1
                   + M * H + 2 * I * H + 2 * M * I                          # y1 [Wg Wu] -> g, u
                   + 3 * M * I                                              # silu(g) * u -> act
                   + M * I + H * I + M * H                                  # act Wd -> AW
                   + 3 * M * H                                              # AW + h1 -> h2
                   + 2 * M * H                                              # RMSNorm(h2) -> y2
                   + M * H + Q * H + M * Q)                                 # y2 Wq -> Z
    return fused, unfused


def timed_kernel_bytes(w, mode, T):
    """Compulsory HBM bytes of one launch of the kernel the roofline reports:
    every operand, residual, output, partial and row scale read or written
    once (weights once per launch).  Operands are 1 byte for e4m3 and 2 for
    bf16; R, h and the outputs are bf16; P and r are fp32."""
    a = 1 if w.dtype == "e4m3" else 2
    o = 2
    M = w.M

    def residual(K, N):  # A [M, K], W [N, K], R [M, N] -> h [M, N], P [M, T]
        return M * K * a + N * K * a + 2 * M * N * o + 4 * M * T

    def consumer(N, N_out, n_weights):  # h [M, N], weights [N_out, N] -> out [M, N_out]; P -> r
        red = 4 * M * T + 4 * M if mode != "separate" else 4 * M
        return M * N * a + n_weights * N_out * N * a + M * N_out * o + red

    if w.dtype == "e4m3" and mode == "block":
        # FP8 block 1: X read (bf16) and quantised (Xq written, then read by
        # the GEMM), h1 read back and quantised (h1q written, then read)
        quant = lambda rows, cols: rows * cols * (o + 2 * a)  # noqa: E731
        return quant(M, w.K1) + residual(w.K1, w.N) + quant(M, w.N) + consumer(w.N, w.inter, 2)
    if w.chain == "swiglu":
        sw = consumer(w.N, w.N2, 2)
        return residual(w.K1, w.N) + sw if mode == "block" else sw
    if w.chain == "rowscale":
        res = residual(w.K1, w.N)
        return res + consumer(w.N, w.N2, 1) if mode == "block" else res
    sw = consumer(w.N, w.inter, 2)
    return residual(w.K1, w.N) + sw if mode == "block" else sw


# Sources each kernel family is compiled from: a recorded ncu figure is valid
# while the hash of its family's files is unchanged.
KERNEL_SOURCES = {
    "gemm": ["coda_internal.h", "gemm_epilogue.cuh", "sm103_ptx.cuh", "fp8_e4m3.cuh", "coda_gemm_bf16.cu",
             "coda_gemm_tf32.cu", "coda_gemm_e4m3.cu"],
    "aux": ["coda_internal.h", "sm103_ptx.cuh", "fp8_e4m3.cuh", "coda_aux.cu"],
}


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed, so an
    edit of the comments leaves the hash of the compiled code unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha(family="gemm"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_epilogue_fusion_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[family]):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    return recorded_traffic_with_source(kernel_tag)[0]


def recorded_traffic_with_source(kernel_tag):
    """(bytes per launch or None, where the figure comes from)."""
    rel = os.path.join("profiles", f"ncu_{kernel_tag}.md")
    p = os.path.join(ROOT, rel)
    if not os.path.exists(p):
        return None, f"no ncu summary {rel}"
    text = open(p).read()
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_b):
        return None, f"{rel} records no source_sha / dram_bytes_per_launch"
    if m_sha.group(1) != kernel_source_sha():
        return None, f"{rel} was taken on other kernel sources ({m_sha.group(1)}, now {kernel_source_sha()})"
    return float(m_b.group(1)), (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch, committed in "
                                 f"{rel} (kernel sources {m_sha.group(1)}), not measured in this run")


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


def max_over_ranks(x, dist, dev):
    """The largest of every rank's x (the job ends when its slowest rank
    does); x itself when there is one rank."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step, steps, world_size, seconds):
    """Whole-job throughput: every rank runs its own batches (weak scaling),
    so the job does world_size x steps x flops_per_step in the slowest rank's
    time."""
    return flops_per_step * steps * world_size / seconds / 1e12


def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if backend == "nccl":
            # this rank's GPU first, so NCCL's communicators bind to it
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend=backend)
        return dist, dist.get_rank(), ws
    return None, 0, 1


# ------------------------------------------------------------- CPU oracle ----

def oracle_runner(w, inp):
    """fp64 oracle of the workload's block on a contiguous row range (rows of
    the block are independent).  The FP8 chain's quantisation needs
    whole-tensor scales, so on a row sample the exact chain is timed instead
    (same GEMM shapes and work)."""
    import oracle
    Wt = lambda t: t.double().numpy().T.copy()  # noqa: E731
    W = {k: Wt(inp[k]) for k in inp if k.startswith("W")}
    G = {k: inp[k].double().numpy() for k in inp if k.startswith("gamma")}
    X = inp["X"].double().numpy()
    R = inp["R"].double().numpy()

    def run(o, n):
        x, r = X[o:o + n], R[o:o + n]
        if w.chain == "swiglu":
            oracle.block_swiglu(x, W["W1t"], r, G["gamma1"], W["Wgt"], W["Wut"], w.eps)
        elif w.chain == "rowscale":
            oracle.block_rowscale(x, W["W1t"], r, G["gamma1"], W["W2t"], w.eps)
        else:
            oracle.chain_full(x, W["W1t"], r, G["gamma1"], W["Wgt"], W["Wut"], W["Wdt"], G["gamma2"], W["Wqt"], w.eps)
    return run


def per_row_flops(w):
    return sum(gemm_flops_by_kernel(w).values()) / w.M


def oracle_sample(w, inp, budget_s, min_rows=16, max_rows=8192):
    """Time the fp64 oracle on the first rows of the workload (rows of the
    block are independent).  Returns (rows, seconds, flops, threads)."""
    run = oracle_runner(w, inp)

    def timed(n):
        t0 = time.perf_counter()
        run(0, n)
        return time.perf_counter() - t0
    timed(min_rows)  # warm (thread pool, pages)
    t = timed(min_rows)
    n = int(max(min_rows, min(max_rows, w.M, budget_s / max(t, 1e-6) * min_rows)))
    dt = timed(n)
    import oracle
    return n, dt, per_row_flops(w) * n, oracle.set_threads(0)


def cpu_model():
    """The host CPU's model name, as lscpu prints it, for the oracle baseline's
    record (the machine type if lscpu is missing)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return os.uname().machine


# -------------------------------------------------------------- the arms ----

def run_reference(args, w):
    dist, rank, ws = dist_setup("gloo")
    if rank != 0:
        return
    inp = make_inputs(w)
    run = oracle_runner(w, inp)
    import oracle
    threads = oracle.set_threads(0)
    # size each step's row sample so that warm-up + timed steps end in about
    # --ref-budget seconds, with at least one row per thread
    t0 = time.perf_counter()
    run(0, threads)
    t_min = time.perf_counter() - t0
    budget = args.ref_budget / max(args.steps + args.warmup, 1)
    rows = int(max(threads, min(1024, threads * budget / max(t_min, 1e-6))))
    rows = min(rows, w.M)
    for s in range(args.warmup):
        run((s * rows) % (w.M - rows + 1), rows)
    t0 = time.perf_counter()
    for s in range(args.steps):
        run((s * rows) % (w.M - rows + 1), rows)
    dt = time.perf_counter() - t0
    value = per_row_flops(w) * rows * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "cpu": cpu_model(),
                         "sample": f"{rows} rows of the {w.M}-row batch per step (rows are independent), "
                                   f"fp64 unfused oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "fused GEMM-epilogue chain TFLOP/s and % of GB300 dense peak; DRAM bytes vs unfused"

# Per chain: the kernel the roofline reports (the one with most of the flops)
# and the outputs an end-to-end step copies back to the host.
DOMINANT = {"swiglu": "gemm_swiglu", "rowscale": "gemm_residual_partial_rms", "full": "gemm_swiglu"}
E2E_OUT = {"swiglu": ("h", "act"), "rowscale": ("h", "Z"), "full": ("h2", "Z")}


def chain_description(w, reduce):
    if reduce == "block" and w.dtype == "e4m3":
        return ("amax(X) -> coda_block_swiglu_fp8 (quantise X, Wo + residual + partial RMS + amax(h1), quantise h1, "
                "gate/up SwiGLU with the reduction in its epilogue + amax(act), one persistent launch) -> "
                "coda_block_rowscale_fp8 (quantise act, down + residual h1 + amax(h2), quantise h2, QKV)")
    if reduce == "block":
        if w.chain == "full":
            return ("coda_block_swiglu (Wo + residual + partial RMS, then gate/up SwiGLU with the reduction in its "
                    "epilogue, one persistent launch) -> coda_block_rowscale (down + residual h1, then QKV)")
        return f"coda_block_{w.chain}: residual GEMM and its consumer in one persistent launch"
    f = reduce != "separate"
    red = " (partials reduced to r in its epilogue)"
    if w.chain == "swiglu":
        return ("gemm_residual_partial_rms -> gemm_swiglu_fused_rms" + red) if f else \
            "gemm_residual_partial_rms -> rms_reduce -> gemm_swiglu"
    if w.chain == "rowscale":
        return ("gemm_residual_partial_rms -> gemm_rowscale_fused_rms" + red) if f else \
            "gemm_residual_partial_rms -> rms_reduce -> gemm_rowscale"
    base = ("Wo: gemm_residual_partial_rms -> gate/up: gemm_swiglu -> down: gemm_residual_partial_rms (R = h1)"
            " -> QKV: gemm_rowscale" + (", reductions fused into the consumers' epilogues" if f else
                                        ", rms_reduce before each consumer"))
    if w.dtype == "e4m3":
        base = "e4m3 operands (amax + quantise of X, h1, act, h2 on the device); " + base
    return base


def set_bytes(w):
    b = 1 if w.dtype == "e4m3" else 2
    x = w.M * w.K1 * 2 + w.M * w.N * 2
    wts = {"swiglu": w.N * w.K1 + 2 * w.N2 * w.N, "rowscale": w.N * w.K1 + w.N2 * w.N,
           "full": w.N * w.K1 + 3 * w.inter * w.N + w.N2 * w.N}[w.chain] * b
    return x + wts


def config_of(w):
    """The workload alone (shapes, dtype, seed, L2 policy): identical for every
    arm that runs it, whatever launches that arm uses."""
    return {"workload": w.name, "dtype": w.dtype,
            "M": w.M, "hidden": w.N, "K1": w.K1, "out_or_intermediate": w.inter or w.N2, "N2": w.N2,
            "eps": w.eps, "seed": w.seed, "heavy_rows": w.heavy_rows,
            "l2": f"{NSETS} rotating input sets of {set_bytes(w) / 1e6:.0f} MB each (> 129 MB L2); no flush"}


def gemm_flops_by_kernel(w):
    M, H = w.M, w.N
    if w.chain == "swiglu":
        return {"gemm_residual_partial_rms": 2.0 * M * H * w.K1, "gemm_swiglu": 2.0 * M * 2 * w.N2 * H}
    if w.chain == "rowscale":
        return {"gemm_residual_partial_rms": 2.0 * M * H * w.K1, "gemm_rowscale": 2.0 * M * w.N2 * H}
    return {"gemm_residual_partial_rms(Wo)": 2.0 * M * H * w.K1, "gemm_swiglu": 2.0 * M * 2 * w.inter * H,
            "gemm_residual_partial_rms(down)": 2.0 * M * H * w.inter, "gemm_rowscale": 2.0 * M * w.N2 * H}


def prepare_set(g, C, w, inp, dev, rank, s):
    """Device tensors of one input set: inputs, folded (and for FP8 quantised)
    weights, and every output buffer, so a step allocates nothing."""
    d = {k: v.to(dev) for k, v in inp.items() if k != "heavy_idx"}
    if s or rank:  # independent batches: same shapes and distribution, other draws
        gen = torch.Generator(device=dev).manual_seed(1000 * rank + s + 1)
        X = torch.randn(w.M, w.K1, generator=gen, device=dev)
        R = torch.randn(w.M, w.N, generator=gen, device=dev)
        if "heavy_idx" in inp:
            idx = inp["heavy_idx"].to(dev)
            X[idx] *= 50.0
            R[idx] *= 50.0
        d["X"], d["R"] = X.bfloat16(), R.bfloat16()
    if s:  # distinct weight copies, so every step also reads its weights from HBM
        for k in list(d):
            if k.startswith("W"):
                d[k] = d[k].clone()
    gam = {k: d[k] for k in d if k.startswith("gamma")}
    Wd = {k: d[k] for k in d if k.startswith("W")}
    M, H = w.M, w.N
    T = g.coda_partial_cols(H)
    bf, f32 = torch.bfloat16, torch.float32
    e = lambda *shape, dt=bf: torch.empty(*shape, dtype=dt, device=dev)  # noqa: E731
    if w.chain == "swiglu":
        f = C.fold_weights("swiglu", Wd, gam)
        st = {"W1t": d["W1t"], "Wg": f["Wgt"], "Wu": f["Wut"], "h": e(M, H), "P": e(M, T, dt=f32), "r": e(M, dt=f32),
              "act": e(M, w.N2)}
    elif w.chain == "rowscale":
        f = C.fold_weights("rowscale", Wd, gam)
        st = {"W1t": d["W1t"], "W2": f["W2t"], "h": e(M, H), "P": e(M, T, dt=f32), "r": e(M, dt=f32), "Z": e(M, w.N2)}
    else:
        f = C.fold_weights("full", Wd, gam)
        st = {"h1": e(M, H), "P1": e(M, T, dt=f32), "r1": e(M, dt=f32), "act": e(M, w.inter), "h2": e(M, H),
              "P2": e(M, T, dt=f32), "r2": e(M, dt=f32), "Z": e(M, w.N2)}
        if w.dtype == "e4m3":
            st["q8"] = C.quantize_weights({"Wot": f["W1t"], "Wgt": f["Wgt"], "Wut": f["Wut"], "Wdt": f["Wdt"],
                                           "Wqt": f["Wqt"]})
            u8 = torch.uint8
            st.update({"Xq": e(w.M, w.K1, dt=u8), "h1q": e(M, H, dt=u8), "actq": e(M, w.inter, dt=u8),
                       "h2q": e(M, H, dt=u8)})
            for k in ("ax", "a1", "a2", "a3", "sx", "s1", "s2", "s3"):
                st[k] = e(1, dt=f32)
        else:
            st.update({"Wo": f["W1t"], "Wg": f["Wgt"], "Wu": f["Wut"], "Wd": f["Wdt"], "Wq": f["Wqt"]})
    st["X"], st["R"] = d["X"], d["R"]
    return st


def make_step(g, C, w, mode, eps, ws=None, fp8_x="block", fp8_act="block"):
    """One pass of the workload's chain over a set; ``ev`` (a pair of CUDA
    events) brackets the dominant kernel's launch.  mode: "separate"
    (rms_reduce launch), "fused" (reduction in the consumer's epilogue) or
    "block" (residual GEMM and consumer in one persistent launch)."""
    fused = mode != "separate"

    def mark(ev, i):
        if ev is not None:
            ev[i].record(torch.cuda.current_stream())

    if mode == "block" and w.dtype == "e4m3":
        # amax(X), then the two FP8 one-launch blocks: block 1 quantises X,
        # runs Wo, quantises h1 and runs gate/up; block 2 quantises act, runs
        # the down projection, quantises h2 and runs QKV
        x_in_block = fp8_x == "block"
        act_in_block = fp8_act == "block"

        def step(st, ev=None):
            q8 = st["q8"]
            g.coda_amax(st["X"], st["ax"])
            if not x_in_block:
                g.coda_quantize_e4m3(st["X"], st["ax"], st["Xq"], st["sx"])
            mark(ev, 0)
            g.coda_block_swiglu_fp8(st["X"] if x_in_block else None, st["ax"] if x_in_block else None,
                                    q8["Wot"][0], q8["Wot"][1], st["R"], q8["Wgt"][0],
                                    q8["Wgt"][1], q8["Wut"][0], q8["Wut"][1], eps, ws, Aq=st["Xq"], scale_a=st["sx"],
                                    H=st["h1"], P=st["P1"], r_out=st["r1"], amax_h=st["a1"], Hq=st["h1q"],
                                    scale_h=st["s1"], Act=st["act"], amax_act=st["a2"])
            mark(ev, 1)
            if not act_in_block:
                g.coda_quantize_e4m3(st["act"], st["a2"], st["actq"], st["s2"])
            g.coda_block_rowscale_fp8(st["act"] if act_in_block else None, st["a2"] if act_in_block else None,
                                      q8["Wdt"][0], q8["Wdt"][1], st["h1"], q8["Wqt"][0],
                                      q8["Wqt"][1], eps, ws, Aq=st["actq"], scale_a=st["s2"], H=st["h2"], P=st["P2"],
                                      r_out=st["r2"], amax_h=st["a3"], Hq=st["h2q"], scale_h=st["s3"], Z=st["Z"])
        return step, 3 + (0 if x_in_block else 1) + (0 if act_in_block else 1)

    if mode == "block":
        if w.chain == "swiglu":
            def step(st, ev=None):
                mark(ev, 0)
                g.coda_block_swiglu(st["X"], st["W1t"], st["R"], st["Wg"], st["Wu"], eps, ws, H=st["h"], P=st["P"],
                                    Act=st["act"], r_out=st["r"])
                mark(ev, 1)
            return step, 1
        if w.chain == "rowscale":
            def step(st, ev=None):
                mark(ev, 0)
                g.coda_block_rowscale(st["X"], st["W1t"], st["R"], st["W2"], eps, ws, H=st["h"], P=st["P"],
                                      Z=st["Z"], r_out=st["r"])
                mark(ev, 1)
            return step, 1

        def step(st, ev=None):
            mark(ev, 0)
            g.coda_block_swiglu(st["X"], st["Wo"], st["R"], st["Wg"], st["Wu"], eps, ws, H=st["h1"], P=st["P1"],
                                Act=st["act"], r_out=st["r1"])
            mark(ev, 1)
            g.coda_block_rowscale(st["act"], st["Wd"], st["h1"], st["Wq"], eps, ws, H=st["h2"], P=st["P2"],
                                  Z=st["Z"], r_out=st["r2"])
        return step, 2

    def sw(h, Wg, Wu, P, r, act, ev=None, **kw):
        mark(ev, 0)
        if fused:
            g.coda_gemm_swiglu_fused_rms(h, Wg, Wu, P, eps, act, r, **kw)
        else:
            g.coda_rms_reduce(P, h.shape[1], eps, r)
            g.coda_gemm_swiglu(h, Wg, Wu, r, act, **kw)
        mark(ev, 1)

    def rs(h, Wq, P, r, Z, **kw):
        if fused:
            g.coda_gemm_rowscale_fused_rms(h, Wq, P, eps, Z, r, **kw)
        else:
            g.coda_rms_reduce(P, h.shape[1], eps, r)
            g.coda_gemm_rowscale(h, Wq, r, Z, **kw)

    if w.chain == "swiglu":
        def step(st, ev=None):
            g.coda_gemm_residual_partial_rms(st["X"], st["W1t"], st["R"], st["h"], st["P"])
            sw(st["h"], st["Wg"], st["Wu"], st["P"], st["r"], st["act"], ev)
        return step, (2 if fused else 3)
    if w.chain == "rowscale":
        def step(st, ev=None):
            mark(ev, 0)
            g.coda_gemm_residual_partial_rms(st["X"], st["W1t"], st["R"], st["h"], st["P"])
            mark(ev, 1)
            rs(st["h"], st["W2"], st["P"], st["r"], st["Z"])
        return step, (2 if fused else 3)
    if w.dtype != "e4m3":
        def step(st, ev=None):
            g.coda_gemm_residual_partial_rms(st["X"], st["Wo"], st["R"], st["h1"], st["P1"])
            sw(st["h1"], st["Wg"], st["Wu"], st["P1"], st["r1"], st["act"], ev)
            g.coda_gemm_residual_partial_rms(st["act"], st["Wd"], st["h1"], st["h2"], st["P2"])
            rs(st["h2"], st["Wq"], st["P2"], st["r2"], st["Z"])
        return step, (4 if fused else 6)

    def step(st, ev=None):
        q8 = st["q8"]
        g.coda_amax(st["X"], st["ax"])
        g.coda_quantize_e4m3(st["X"], st["ax"], st["Xq"], st["sx"])
        g.coda_gemm_residual_partial_rms(st["Xq"], q8["Wot"][0], st["R"], st["h1"], st["P1"], scale_x=st["sx"],
                                         scale_w=q8["Wot"][1], amax_h=st["a1"])
        g.coda_quantize_e4m3(st["h1"], st["a1"], st["h1q"], st["s1"])
        sw(st["h1q"], q8["Wgt"][0], q8["Wut"][0], st["P1"], st["r1"], st["act"], ev, scale_h=st["s1"],
           scale_wg=q8["Wgt"][1], scale_wu=q8["Wut"][1], amax_act=st["a2"])
        g.coda_quantize_e4m3(st["act"], st["a2"], st["actq"], st["s2"])
        g.coda_gemm_residual_partial_rms(st["actq"], q8["Wdt"][0], st["h1"], st["h2"], st["P2"], scale_x=st["s2"],
                                         scale_w=q8["Wdt"][1], amax_h=st["a3"])
        g.coda_quantize_e4m3(st["h2"], st["a3"], st["h2q"], st["s3"])
        rs(st["h2q"], q8["Wqt"][0], st["P2"], st["r2"], st["Z"], scale_h=st["s3"], scale_w=q8["Wqt"][1])
    return step, (9 if fused else 11)


def run_coda(args, w):
    dist, rank, ws = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C

    g.load_library()
    inp = make_inputs(w)
    sets = [prepare_set(g, C, w, inp, dev, rank, s) for s in range(NSETS)]
    torch.cuda.synchronize()
    # FP8 defaults to the nine-launch chain: the FP8 blocks (one launch per
    # block, quantisation in the launch) measured up to 1% slower on GB300
    mode = args.reduce if args.reduce != "auto" else ("fused" if w.dtype == "e4m3" else "block")
    wksp = g.block_fp8_workspace(w.M, dev) if w.dtype == "e4m3" else g.block_workspace(w.M, dev)
    step, launches = make_step(g, C, w, mode, w.eps, wksp, args.fp8_x, args.fp8_act)
    fl = gemm_flops_by_kernel(w)
    step_flops = sum(fl.values())
    dom = DOMINANT[w.chain]
    dom_flops = fl[dom]
    if mode == "block":  # the timed launch holds both GEMMs of the (first) block
        if w.chain == "full":
            name = "block_swiglu_fp8 (quantise X, Wo, quantise h1, gate/up)" if w.dtype == "e4m3" else \
                "block_swiglu (Wo + gate/up)"
            dom, dom_flops = name, fl["gemm_residual_partial_rms(Wo)"] + fl["gemm_swiglu"]
        else:
            dom, dom_flops = f"block_{w.chain}", step_flops
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        step(sets[i % NSETS])
    g.coda_get_device_status()
    barrier()
    if args.profile_step:
        profile_one_step(lambda: step(sets[args.warmup % NSETS]), rank, f"coda/{mode}", launches)
        return

    # ---- timed region: K steps, inputs resident in HBM
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        t_start.record(stream)
        for i in range(args.steps):
            step(sets[i % NSETS], evs[i])
        t_end.record(stream)
        barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    dom_ms = statistics.fmean(a.elapsed_time(b) for a, b in evs)
    g.coda_get_device_status()
    elapsed_max = max_over_ranks(elapsed, dist, dev)
    value = job_tflops(step_flops, args.steps, ws, elapsed_max)

    # ---- sustained: the same step repeated for a window of seconds, so the
    # clocks sampled inside it describe the kernel under the power cap (a
    # short timed region runs at burst clocks before the cap engages)
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, math.ceil(args.sustained_s / max(elapsed / args.steps, 1e-6)))
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_sus)]
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk_s:
            barrier()
            s0.record(stream)
            for i in range(n_sus):
                step(sets[i % NSETS], sev[i])
            s1.record(stream)
            barrier()
        sus_s = s0.elapsed_time(s1) / 1e3
        sus_dom_ms = statistics.fmean(a.elapsed_time(b) for a, b in sev)
        g.coda_get_device_status()
        sus_s = max_over_ranks(sus_s, dist, dev)
        sustained = {"steps": n_sus, "seconds": sus_s, "value": job_tflops(step_flops, n_sus, ws, sus_s),
                     "ms_per_step": sus_s / n_sus * 1e3, "kernel_avg_launch_ms": sus_dom_ms,
                     "clocks": clk_s.summary()}

    # ---- end to end: pinned host X, R in and the block's outputs out, every
    # step.  Two buffer slots and three streams, so one step's copies overlap
    # the compute of its neighbours (copy engines and SMs work concurrently).
    e2e_steps = max(40, min(200, args.steps // 2))
    outs = E2E_OUT[w.chain]
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    slots = []
    for k in range(2):
        st = sets[k]
        sl = {"st": st, "in": torch.cuda.Event(), "cmp": torch.cuda.Event(), "out": torch.cuda.Event(),
              "hX": torch.empty(st["X"].shape, dtype=st["X"].dtype, pin_memory=True).copy_(st["X"].cpu()),
              "hR": torch.empty(st["R"].shape, dtype=st["R"].dtype, pin_memory=True).copy_(st["R"].cpu())}
        for o in outs:
            sl["h_" + o] = torch.empty(st[o].shape, dtype=st[o].dtype, pin_memory=True)
        slots.append(sl)

    def e2e_step(i):
        sl = slots[i % 2]
        st = sl["st"]
        if i >= 2:
            s_in.wait_event(sl["cmp"])   # step i-2 finished reading this slot's inputs
            s_cmp.wait_event(sl["out"])  # ... and its outputs were copied out
        with torch.cuda.stream(s_in):
            st["X"].copy_(sl["hX"], non_blocking=True)
            st["R"].copy_(sl["hR"], non_blocking=True)
            sl["in"].record(s_in)
        s_cmp.wait_event(sl["in"])
        with torch.cuda.stream(s_cmp):
            step(st)
            sl["cmp"].record(s_cmp)
        s_out.wait_event(sl["cmp"])
        with torch.cuda.stream(s_out):
            for o in outs:
                sl["h_" + o].copy_(st[o], non_blocking=True)
            sl["out"].record(s_out)

    for i in range(4):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)  # after every step's last copy (s_out runs the steps' copies in order)
    barrier()
    e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, dev)
    e2e_val = job_tflops(step_flops, e2e_steps, ws, e2e_s)
    sl = slots[0]
    h2d = sum(sl[k].numel() * sl[k].element_size() for k in ("hX", "hR"))
    d2h = sum(sl["h_" + o].numel() * sl["h_" + o].element_size() for o in outs)

    if rank != 0:
        return
    pk, pk_kind = peaks()
    ratio, dtname = (2.0, "e4m3 (2 x measured bf16 burst, the nominal fp8/bf16 ratio)") if w.dtype == "e4m3" else \
        (1.0, "bf16 burst")
    peak = pk["bf16_tflops"] * ratio
    peak_sus = pk["bf16_tflops_sustained"] * ratio
    achieved = dom_flops / (dom_ms / 1e3) / 1e12
    tag = f"{dom.split(' ')[0]}_{w.name}"
    traffic, traffic_src = recorded_traffic_with_source(tag)
    roof = {"kernel": f"{dom} (tcgen05, {w.dtype})", "bound": "tensor", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": f"{dtname}, {pk_kind}",
            "traffic": traffic, "traffic_source": traffic_src, "avg_launch_ms": dom_ms,
            "flops_per_launch": dom_flops,
            "algorithmic_bytes": timed_kernel_bytes(w, mode, g.coda_partial_cols(w.N))}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if w.dtype == "e4m3" else "bf16",
        "data": "synthetic", "config": config_of(w), "chain": chain_description(w, mode),
        "frac_of_peak": value / ws / peak,
        "roofline": roof,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "how": "pinned host X, R in and " + ", ".join(outs) + " out every step; "
                                           "2 buffer slots, copy-in / compute / copy-out streams overlapped"},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    if sustained is not None:
        sus_kernel = dom_flops / (sustained["kernel_avg_launch_ms"] / 1e3) / 1e12
        clk_s = sustained.pop("clocks")
        sustained.update({"frac_of_bf16_sustained": sustained["value"] / ws / peak_sus,
                          "kernel_achieved": sus_kernel, "kernel_frac_of_bf16_sustained": sus_kernel / peak_sus,
                          "peak_sustained": peak_sus, "sm_mhz_median_under_load": clk_s.get("sm_mhz"),
                          "clocks": clk_s})
        line["sustained"] = sustained
    if w.chain == "swiglu":
        fused_b, unfused_b = algorithmic_bytes(w.M, w.K1, w.N, w.N2, g.coda_partial_cols(w.N))
        line["dram_bytes_algorithmic"] = {"fused": sum(fused_b.values()), "unfused": unfused_b}
    if w.chain == "full" and w.dtype == "bf16":
        fused_b, unfused_b = chain_bytes_full(w, g.coda_partial_cols(w.N))
        line["dram_bytes_algorithmic"] = {"fused": fused_b, "unfused": unfused_b,
                                          "measured_fused": "profiles/ncu_block_swiglu_llama8b_chain.md",
                                          "measured_unfused": "profiles/dram_fused_vs_unfused_llama8b_chain.md"}
    if not args.no_cpu_baseline:
        n, dt, fl_cpu, threads = oracle_sample(w, inp, args.cpu_budget)
        line["cpu_baseline"] = {"value": fl_cpu / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "cpu": cpu_model(),
                                "sample": f"first {n} of {w.M} rows of the same batch (rows are independent), "
                                          f"{dt:.1f} s of fp64 unfused oracle"}
        # the same oracle on one core, on a smaller sample
        import oracle
        prev = oracle.set_threads(0)
        oracle.set_threads(1)
        n1, dt1, fl1, _ = oracle_sample(w, inp, args.cpu_budget / 4)
        oracle.set_threads(prev)
        line["cpu_baseline"]["value_1thread"] = fl1 / dt1 / 1e12
        line["cpu_baseline"]["sample_1thread"] = f"first {n1} rows, {dt1:.1f} s on one thread"
    print(json.dumps(line), flush=True)


def profile_one_step(step, rank, what, launches):
    """One step between cudaProfilerStart/Stop, for `ncu --profile-from-start off`."""
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    step()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    if rank == 0:
        print(json.dumps({"profile_step": what, "launches": launches}), flush=True)


def backward_flops(w):
    """The backward's GEMMs do twice the forward's work (an input and a weight gradient per GEMM)."""
    return 2.0 * sum(gemm_flops_by_kernel(w).values())


def run_coda_backward(args, w):
    """Backward of the LLaMA block-tail chain from a saved forward state (the
    forward with coda_gemm_swiglu_save): 12 launches per step."""
    dist, rank, ws = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    g.load_library()
    inp = make_inputs(w)
    sets = []
    for s in range(2):
        d = {k: v.to(dev) for k, v in inp.items() if k != "heavy_idx"}
        gen = torch.Generator(device=dev).manual_seed(100 * rank + s)
        f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")},
                           {k: d[k] for k in d if k.startswith("gamma")})
        fwd = C.full_chain_train_forward(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], d["Wdt"], f["Wqt"], w.eps)
        sets.append({"X": d["X"], "Wot": d["W1t"], "Wgut": torch.cat([d["Wgt"], d["Wut"]], 0).contiguous(),
                     "Wdt": d["Wdt"], "Wqt": d["Wqt"], "g1": d["gamma1"], "g2": d["gamma2"], "fwd": fwd,
                     "dZ": torch.randn(w.M, w.N2, generator=gen, device=dev).bfloat16(),
                     "dH2": torch.randn(w.M, w.N, generator=gen, device=dev).bfloat16(), "f": f, "R": d["R"]})
    torch.cuda.synchronize()

    def step(st):
        return C.full_chain_backward(st["X"], st["Wot"], st["Wgut"], st["Wdt"], st["Wqt"], st["g1"], st["g2"],
                                     st["fwd"], st["dZ"], st["dH2"])

    def fwd_step(st):
        f = st["f"]
        C.full_chain_train_forward(st["X"], st["Wot"], st["R"], f["Wgt"], f["Wut"], st["Wdt"], f["Wqt"], w.eps)

    for i in range(args.warmup):
        step(sets[i % 2])
    g.coda_get_device_status()
    if args.profile_step:
        profile_one_step(lambda: step(sets[0]), rank, "coda backward", 12)
        return
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    res = {}
    with ClockSampler(local) as clk:
        for name, fn, n in (("backward", step, args.steps), ("train_forward", fwd_step, max(3, args.steps // 2))):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(n):
                fn(sets[i % 2])
            b.record()
            torch.cuda.synchronize()
            res[name] = a.elapsed_time(b) / 1e3 / n
    g.coda_get_device_status()
    if rank != 0:
        return
    pk, pk_kind = peaks()
    bf = backward_flops(w)
    value = bf * ws / res["backward"] / 1e12
    print(json.dumps({
        "metric": METRIC, "pass": "backward", "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["backward"] * 1e3, "higher_is_better": True, "scaling": "weak",
        "dtype": "bf16", "data": "synthetic", "config": config_of(w),
        "frac_of_peak": value / ws / pk["bf16_tflops"],
        "train_forward_with_saves": {"value": sum(gemm_flops_by_kernel(w).values()) / res["train_forward"] / 1e12,
                                     "ms_per_step": res["train_forward"] * 1e3},
        "gpu_launches": 12 * args.steps, "clocks": clk.summary()}), flush=True)


def _compile_toolchain():
    """torch.compile's Triton kernels need a ptxas that knows this GPU's
    architecture; Triton's bundled one may predate it, so use the CUDA
    toolkit's unless the caller chose one."""
    if "TRITON_PTXAS_PATH" not in os.environ:
        for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
            cand = os.path.join(root, "bin", "ptxas") if root else None
            if cand and os.path.exists(cand):
                os.environ["TRITON_PTXAS_PATH"] = cand
                break


def run_unfused_backward(args, w):
    """PyTorch eager autograd through the unfused chain (cuBLAS GEMMs, fp32-math
    RMSNorm, silu * mul), backward only."""
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_inputs(w)
    d = {k: v.to(dev) for k, v in inp.items() if k != "heavy_idx"}
    P = {k: d[k].clone().requires_grad_(True) for k in ("X", "R", "W1t", "Wgt", "Wut", "Wdt", "Wqt")}
    G = {k: d[k].clone().requires_grad_(True) for k in ("gamma1", "gamma2")}
    gen = torch.Generator(device=dev).manual_seed(7)
    dZ = torch.randn(w.M, w.N2, generator=gen, device=dev).bfloat16()
    dH2 = torch.randn(w.M, w.N, generator=gen, device=dev).bfloat16()

    def rms(h, gam):
        hf = h.float()
        return (hf * torch.rsqrt(hf.pow(2).mean(-1, keepdim=True) + w.eps) * gam).bfloat16()

    def forward_fn(P, G):
        h1 = P["X"] @ P["W1t"].t() + P["R"]
        y1 = rms(h1, G["gamma1"])
        act = torch.nn.functional.silu(y1 @ P["Wgt"].t()) * (y1 @ P["Wut"].t())
        h2 = h1 + act @ P["Wdt"].t()
        Z = rms(h2, G["gamma2"]) @ P["Wqt"].t()
        return Z, h2

    if args.compile:
        _compile_toolchain()
    fwd = torch.compile(forward_fn) if args.compile else forward_fn

    def step():
        Z, h2 = fwd(P, G)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        torch.autograd.backward([Z, h2], [dZ, dH2])
        b.record()
        torch.cuda.synchronize()
        for t in list(P.values()) + list(G.values()):
            t.grad = None
        return a.elapsed_time(b) / 1e3

    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    t = statistics.median(times)
    print(json.dumps({"impl": "unfused_torch_compile_autograd" if args.compile else "unfused_torch_eager_autograd",
                      "pass": "backward", "metric": METRIC,
                      "value": backward_flops(w) / t / 1e12, "unit": "TFLOP/s", "ms_per_step": t * 1e3,
                      "steps": args.steps, "dtype": "bf16", "config": config_of(w)}), flush=True)


def run_unfused(args, w):
    """cuBLAS + PyTorch eager, unfused: XW, add, RMSNorm (fp32 math), GEMM, silu*mul
    (and, for the 8B chain, the down GEMM, add, RMSNorm and QKV GEMM)."""
    if w.chain not in ("swiglu", "full") or w.dtype != "bf16":
        raise SystemExit("--impl unfused covers the bf16 attention-out + SwiGLU block and the bf16 8B chain")
    dist, rank, ws = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = make_inputs(w)
    d = {k: v.to(dev) for k, v in inp.items()}
    Wgu = torch.cat([d["Wgt"], d["Wut"]], 0)

    def rms(h, gamma):
        hf = h.float()
        return (hf * torch.rsqrt(hf.pow(2).mean(-1, keepdim=True) + w.eps) * gamma).bfloat16()

    def block(X, R):
        h = torch.matmul(X, d["W1t"].t()) + R
        gu = torch.matmul(rms(h, d["gamma1"]), Wgu.t())
        g_, u = gu.chunk(2, dim=-1)
        return h, torch.nn.functional.silu(g_) * u

    def step():
        h, act = block(d["X"], d["R"])
        if w.chain == "swiglu":
            return h, act
        h2 = torch.matmul(act, d["Wdt"].t()) + h
        return h2, torch.matmul(rms(h2, d["gamma2"]), d["Wqt"].t())

    if args.compile:
        _compile_toolchain()
        step = torch.compile(step)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if args.profile_step:
        profile_one_step(step, rank, "unfused torch.compile" if args.compile else "unfused torch eager", None)
        return
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    dt = a.elapsed_time(b) / 1e3
    fl = sum(gemm_flops_by_kernel(w).values())
    if rank == 0:
        print(json.dumps({"impl": "unfused_torch_compile" if args.compile else "unfused_torch_eager", "metric": METRIC, "value": fl * args.steps / dt / 1e12,
                          "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": dt / args.steps * 1e3, "dtype": "bf16", "config": config_of(w)}),
              flush=True)


def run_aux(args, w):
    """The HBM-bound kernels of the path at this workload's sizes: GB/s and the
    fraction of the measured HBM copy bandwidth.  Bytes are algorithmic (every
    operand read and every output written once); 3 rotating input sets, each
    larger than L2 where the operands are (P and r are tiny and stay in L2)."""
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    M, N = w.M, w.N
    I = w.inter or w.N2
    T = g.coda_partial_cols(N)
    gen = torch.Generator(device=dev).manual_seed(11)
    bf = torch.bfloat16

    def rnd(*s, dt=bf):
        return torch.randn(*s, generator=gen, device=dev).to(dt)

    sets = []
    for _ in range(NSETS):
        sets.append({"W": rnd(I, N), "gam": rnd(N, dt=torch.float32).abs() + 0.5, "Wo": torch.empty(I, N, dtype=bf, device=dev),
                     "P": rnd(M, T, dt=torch.float32).abs() * N / T, "r": torch.empty(M, device=dev),
                     "H": rnd(M, N), "dY": rnd(M, N), "S": rnd(M, T, dt=torch.float32),
                     "dH": torch.empty(M, N, dtype=bf, device=dev), "Yt": torch.empty(M, N, dtype=bf, device=dev),
                     "dgam": torch.empty(N, device=dev), "amax": torch.empty(1, device=dev),
                     "q": torch.empty(M, N, dtype=torch.uint8, device=dev), "scale": torch.empty(1, device=dev)})
    ws_bytes = g.load_library().coda_rmsnorm_backward_workspace_bytes(M, N)
    wsp = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device=dev)
    for s in sets:
        s["rr"] = torch.rand(M, device=dev) + 0.5
    kernels = {
        "fold_gamma": (lambda s: g.coda_fold_gamma(s["W"], s["gam"], out=s["Wo"]), 2 * I * N * 2 + 4 * N,
                       f"W^T [{I}x{N}] bf16 -> diag(gamma)-folded copy"),
        "rms_reduce": (lambda s: g.coda_rms_reduce(s["P"], N, w.eps, r=s["r"]), 4 * M * T + 4 * M,
                       f"P [{M}x{T}] fp32 -> r [{M}] (L2-resident, latency-bound)"),
        "amax": (lambda s: g.coda_amax(s["H"], amax=s["amax"]), 2 * M * N, f"max |h| over [{M}x{N}] bf16"),
        "quantize_e4m3": (lambda s: g.coda_quantize_e4m3(s["H"], s["amax"], q=s["q"], scale=s["scale"]), 3 * M * N,
                          f"h [{M}x{N}] bf16 -> e4m3"),
        "rmsnorm_backward": (lambda s: g.coda_rmsnorm_backward(s["dY"], s["H"], s["rr"], s["gam"], s["S"], dH=s["dH"],
                                                                Yt=s["Yt"], dgamma=s["dgam"], workspace=wsp),
                             4 * M * N * 2 + 4 * M * T + 4 * M + 8 * N,
                             f"dY, h [{M}x{N}] bf16 -> dh, r h bf16, dgamma"),
    }
    for s in sets:  # amax before quantise
        g.coda_amax(s["H"], amax=s["amax"])
    if args.profile_step:
        for i in range(args.warmup):
            for fn, _, _ in kernels.values():
                fn(sets[i % NSETS])
        profile_one_step(lambda: [fn(sets[0]) for fn, _, _ in kernels.values()], 0, "coda aux kernels",
                         len(kernels) + 1)
        return
    pk, pk_kind = peaks()
    out = {}
    clk = ClockSampler(local)
    with clk:
        for name, (fn, nbytes, what) in kernels.items():
            for i in range(args.warmup):
                fn(sets[i % NSETS])
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = max(args.steps, 10)
            a.record()
            for i in range(n):
                fn(sets[i % NSETS])
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / n
            gbs = nbytes / (us * 1e-6) / 1e9
            out[name] = {"us_per_launch": us, "bytes_per_launch": nbytes, "GB/s": gbs, "frac": gbs / pk["hbm_gbs"],
                         "what": what}
    if g.coda_get_device_status() != 0:
        raise SystemExit("device status not clean")
    print(json.dumps({"pass": "aux", "metric": "HBM GB/s of the memory-bound kernels", "unit": "GB/s",
                      "peak": pk["hbm_gbs"], "peak_kind": f"HBM copy, {pk_kind}", "kernels": out,
                      "steps": n, "config": {"workload": w.name, "M": M, "N": N, "I": I, "T": T},
                      "clocks": clk.summary()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["coda", "reference", "unfused"], default="coda")
    ap.add_argument("--workload", default="llama8b_chain",
                    choices=["llama1b_attn_out_swiglu", "llama1b_mlp_down_qkv", "llama8b_chain", "llama8b_chain_fp8",
                             "llama70b_chain"],
                    help="the default is the largest bf16 configuration (the LLaMA-3-8B chain); the others "
                         "are for the per-configuration tables")
    ap.add_argument("--reduce", choices=["auto", "block", "fused", "separate"], default="auto",
                    help="block: residual GEMM and consumer in one persistent launch per block (FP8: the FP8 "
                         "blocks, which also quantise h); fused: r reduced inside the consumer GEMM's epilogue; "
                         "separate: coda_rms_reduce launch; auto: block for bf16, fused for FP8")
    ap.add_argument("--fp8-x", choices=["block", "kernel"], default="block",
                    help="FP8 block mode: X quantised by the first block's quantiser warps, or by "
                         "coda_quantize_e4m3 before it")
    ap.add_argument("--fp8-act", choices=["block", "kernel"], default="block",
                    help="FP8 block mode: act quantised by the second block's quantiser warps, or by "
                         "coda_quantize_e4m3 between the blocks")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward", "aux"], default="forward",
                    help="backward: gradients of the LLaMA-8B chain from a saved forward state; aux: GB/s of the "
                         "memory-bound kernels (fold, reduce, amax, quantise, RMSNorm backward)")
    ap.add_argument("--compile", action="store_true", help="--impl unfused: run the unfused sequence under torch.compile")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-step", action="store_true",
                    help="after warm-up run exactly one step inside cudaProfilerStart/Stop and exit (for ncu)")
    ap.add_argument("--rows", type=int, default=0,
                    help="with --profile-step: override the workload's M (tokens), for ncu captures on a smaller "
                         "case of the same kernels")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of the sustained window after the timed steps (0: none)")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work for warm-up + timed steps together")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if args.rows:
        if not args.profile_step:
            ap.error("--rows is for --profile-step captures only")
        w = w.with_rows(args.rows)
    if args.pass_ == "aux":
        if args.impl != "coda":
            ap.error("--pass aux measures this library's kernels only")
        run_aux(args, w)
    elif args.pass_ == "backward":
        if w.chain != "full" or w.dtype != "bf16":
            ap.error("--pass backward covers the bf16 LLaMA-8B chain (--workload llama8b_chain)")
        if args.impl == "unfused":
            run_unfused_backward(args, w)
        elif args.impl == "coda":
            run_coda_backward(args, w)
        else:
            ap.error("--pass backward has no reference arm")
    elif args.impl == "reference":
        run_reference(args, w)
    elif args.impl == "unfused":
        run_unfused(args, w)
    else:
        run_coda(args, w)


if __name__ == "__main__":
    main()
