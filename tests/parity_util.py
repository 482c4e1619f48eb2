"""Shared helpers for the parity tests: oracle references for a workload's
seeded inputs, and the same blocks run through the C ABI on the GPU.

The oracle sees the exact input bits the GPU sees (bf16/fp32 widened to
fp64) with weights in the mathematical orientation W = Wt^T; it never sees
anything the GPU computed.  Tolerance metric: max|gpu - ref| / (max|ref| + 1e-6).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from coda_inputs import Workload, make_inputs

TOL = {"f32": 2e-2, "bf16": 2e-2, "e4m3": 6e-2}


def W(t: torch.Tensor) -> np.ndarray:
    """nn.Linear-layout W^T [N, K] -> fp64 W [K, N]."""
    return t.double().numpy().T.copy()


def oracle_ref(w: Workload, inp: dict, rows=None) -> dict:
    """The unfused fp64 block on (a row subset of) the workload's inputs."""
    sel = (lambda t: t) if rows is None else (lambda t: t[rows])
    X, R = sel(inp["X"]), sel(inp["R"])
    if w.chain == "rowscale":
        return oracle.block_rowscale(X, W(inp["W1t"]), R, inp["gamma1"], W(inp["W2t"]), w.eps)
    if w.chain == "swiglu":
        return oracle.block_swiglu(X, W(inp["W1t"]), R, inp["gamma1"], W(inp["Wgt"]), W(inp["Wut"]), w.eps)
    if w.chain == "full":
        fn = oracle.chain_full_fp8 if (w.dtype == "e4m3" and rows is None) else oracle.chain_full
        return fn(X, W(inp["W1t"]), R, inp["gamma1"], W(inp["Wgt"]), W(inp["Wut"]), W(inp["Wdt"]), inp["gamma2"],
                  W(inp["Wqt"]), w.eps)
    raise ValueError(w.chain)


def to_device(inp: dict, dev="cuda") -> dict:
    return {k: v.to(dev) for k, v in inp.items() if k != "heavy_idx"}


def run_gpu(w: Workload, d: dict, fused_reduce: bool = False) -> dict:
    """Run the workload's block through the C ABI on device tensors ``d``;
    returns CPU copies of every output."""
    from gemm_epilogue_fusion_gb300 import chain as C
    g = {k: d[k] for k in d if k.startswith("gamma")}
    Wd = {k: d[k] for k in d if k.startswith("W")}
    if w.dtype == "e4m3":
        f = C.fold_weights("full", Wd, g)
        q8 = C.quantize_weights({"Wot": f["W1t"], "Wgt": f["Wgt"], "Wut": f["Wut"], "Wdt": f["Wdt"],
                                 "Wqt": f["Wqt"]})
        out = C.full_chain_fp8(d["X"], d["R"], q8, w.eps, fused_reduce=fused_reduce)
    else:
        f = C.fold_weights(w.chain, Wd, g)
        if w.chain == "rowscale":
            out = C.rowscale_block(d["X"], d["W1t"], d["R"], f["W2t"], w.eps, fused_reduce=fused_reduce)
        elif w.chain == "swiglu":
            out = C.swiglu_block(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], w.eps, fused_reduce=fused_reduce)
        else:
            out = C.full_chain(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], d["Wdt"], f["Wqt"], w.eps,
                             fused_reduce=fused_reduce)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items() if isinstance(v, torch.Tensor)}


# output name on the GPU side -> name in the oracle's result
PAIRS = {
    "rowscale": [("h", "h"), ("r", "r"), ("Z", "Z")],
    "swiglu": [("h", "h"), ("r", "r"), ("act", "act")],
    "full": [("h1", "h1"), ("r1", "r1"), ("act", "act"), ("h2", "h2"), ("r2", "r2"), ("Z", "Z")],
}


def compare(w: Workload, got: dict, ref: dict, rows=None, tol=None) -> dict:
    tol = TOL[w.dtype] if tol is None else tol
    errs = {}
    for g, o in PAIRS[w.chain]:
        gv = got[g] if rows is None else got[g][rows]
        errs[g] = oracle.rel_err(gv, ref[o])
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"{w.name}: parity errors above {tol}: {bad} (all: {errs})"
    return errs
