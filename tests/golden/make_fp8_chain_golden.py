"""Writes tests/golden/llama8b_chain_fp8_rows.npz: the quantisation-aware fp64
oracle (oracle.chain_full_fp8) on the full-size LLaMA-3-8B FP8 chain
(M = 32768 tokens, 5% of rows x50), stored for a seeded sample of rows.

Per-tensor FP8 scales need the amax of whole tensors (h1, act, h2), so the
oracle has to run the chain over every row once (about 12.7 TFLOP of fp64
work: 20 minutes on 8 x86 cores, ~30 GB of RAM); the GPU test then compares
its sampled rows.  torch's CPU random draws are not bit-identical across CPU
architectures and torch versions, so the file must be written on the machine
type (and software image) that runs the GPU test; the digests enforce it.  Calls only oracle/ and the seeded input generator.  Values are stored
as float32 (far below the 6e-2 tolerance); sha256 digests of the input
tensors guard against a changed generator.

    python tests/golden/make_fp8_chain_golden.py [--out PATH]
"""
import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from coda_inputs import WORKLOADS, make_inputs, sample_rows  # noqa: E402

OUT = os.path.join(HERE, "llama8b_chain_fp8_rows.npz")
KEYS = ("X", "R", "W1t", "Wgt", "Wut", "Wdt", "Wqt", "gamma1", "gamma2")


def input_digests(inp):
    d = {}
    for k in KEYS:
        t = inp[k].contiguous()
        d[k] = hashlib.sha256(t.view(-1).view(dtype=__import__("torch").uint8).numpy().tobytes()).hexdigest()
    return d


def golden_rows(inp, M):
    heavy = sorted(inp["heavy_idx"].tolist())[:2]
    return sorted(set(sample_rows(M, 6).tolist()) | set(heavy))


def main(path=OUT):
    w = WORKLOADS["llama8b_chain_fp8"]
    t0 = time.time()
    inp = make_inputs(w)
    rows = golden_rows(inp, w.M)
    T = lambda t: t.double().numpy().T.copy()  # noqa: E731
    res = oracle.chain_full_fp8(inp["X"], T(inp["W1t"]), inp["R"], inp["gamma1"], T(inp["Wgt"]), T(inp["Wut"]),
                                T(inp["Wdt"]), inp["gamma2"], T(inp["Wqt"]), w.eps, out_rows=rows)
    save = {k: np.asarray(res[k]).astype(np.float32) for k in ("h1", "r1", "act", "h2", "r2", "Z")}
    dig = input_digests(inp)
    np.savez_compressed(path, rows=np.asarray(rows, dtype=np.int64),
                        digests=np.asarray([f"{k}:{dig[k]}" for k in KEYS]), **save)
    import platform
    import torch
    print(f"wrote {path} for rows {rows} in {time.time() - t0:.0f} s on {platform.machine()}, torch {torch.__version__}")


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=OUT)
    main(ap.parse_args().out)
