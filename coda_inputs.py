"""Seeded synthetic inputs for the CODA GEMM-epilogue block.

This module is shared by the CUDA path's tests/bench and by the CPU oracle.
It only draws random numbers and casts them to the I/O dtype: it holds none of
the method's arithmetic (no GEMM, no norm, no activation).

The CODA write-ups benchmark LLaMA-3-style hidden sizes ("experimental
results" section of the CODA news write-up) but publish no dataset, so every
tensor here is synthetic:

  X, R ~ N(0, 1)               activations and residual stream
  W    ~ N(0, 1/K)             K = the weight's input width
  gamma = 1 + 0.1 * N(0, 1)    RMSNorm weight

Weights are produced in the ``nn.Linear.weight`` layout, i.e. W^T with shape
[N_out, K] row-major.  Draw order is fixed: X, R, the weights in chain order,
then the gammas, all from one ``torch.Generator`` seeded per workload.  The
fp32 draws are rounded to nearest-even into the I/O dtype, and those exact
bits are what both the GPU path and the oracle receive.
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One benchmark workload of the fused block.

    ``chain`` names the sequence of epilogue programs:
      "rowscale"  : h = R + X W1 ; r = rms(h) ; Z = diag(r) h diag(g) W2
      "swiglu"    : h = R + X Wo ; r = rms(h) ; act = silu(r h Wg') * (r h Wu')
      "full"      : Wo+R -> rms -> gate/up SwiGLU -> down+h1 -> rms -> QKV
    """
    name: str
    chain: str
    M: int
    K1: int          # width of X (input of the first GEMM)
    N: int           # hidden size = RMSNorm width = output of the first GEMM
    N2: int          # output width of the last GEMM (W2 / QKV), or I for swiglu
    inter: int       # intermediate size of the MLP (full chain only), else 0
    dtype: str       # "f32" | "bf16" | "e4m3"
    eps: float
    seed: int
    heavy_rows: float = 0.0   # fraction of rows of X and R scaled by 50

    def gemm_flops(self) -> float:
        """Dense GEMM flops (2*M*N*K summed over the chain's GEMMs)."""
        M = self.M
        if self.chain == "rowscale":
            return 2.0 * M * (self.K1 * self.N + self.N * self.N2)
        if self.chain == "swiglu":
            return 2.0 * M * (self.K1 * self.N + self.N * 2 * self.N2)
        if self.chain == "full":
            H, I, Q = self.N, self.inter, self.N2
            return 2.0 * M * (self.K1 * H + H * 2 * I + I * H + H * Q)
        raise ValueError(self.chain)

    def with_rows(self, M: int) -> "Workload":
        return dataclasses.replace(self, M=M)


# The workloads: tiny fp32 block; LLaMA-3-1B attention-out + gate/up;
# LLaMA-3-1B MLP-down + QKV; LLaMA-3-8B full chain (bf16); the same in FP8;
# and the full chain at LLaMA-3-70B shapes.
WORKLOADS: Dict[str, Workload] = {
    "tiny_f32": Workload("tiny_f32", "rowscale", 256, 512, 512, 512, 0, "f32", 1e-6, 0),
    "llama1b_attn_out_swiglu": Workload("llama1b_attn_out_swiglu", "swiglu", 8192, 2048, 2048, 8192, 0,
                                        "bf16", 1e-5, 0),
    "llama1b_mlp_down_qkv": Workload("llama1b_mlp_down_qkv", "rowscale", 8192, 8192, 2048, 3072, 0,
                                     "bf16", 1e-5, 1),
    "llama8b_chain": Workload("llama8b_chain", "full", 16384, 4096, 4096, 6144, 14336, "bf16", 1e-5, 2),
    "llama8b_chain_fp8": Workload("llama8b_chain_fp8", "full", 32768, 4096, 4096, 6144, 14336, "e4m3",
                                  1e-5, 3, heavy_rows=0.05),
    # the write-up's largest hidden size: LLaMA-3-70B shapes (hidden 8192,
    # intermediate 28672, QKV 64 query + 2 x 8 key/value heads of 128 = 10240),
    # the same 16384 tokens and distributions as the 8B chain
    "llama70b_chain": Workload("llama70b_chain", "full", 16384, 8192, 8192, 10240, 28672, "bf16", 1e-5, 4),
}


def _io_torch_dtype(dtype: str) -> torch.dtype:
    # e4m3 workloads keep bf16 activations/weights at the I/O boundary; the
    # FP8 operands are produced from them on the device.
    return torch.float32 if dtype == "f32" else torch.bfloat16


def weight_shapes(w: Workload) -> Dict[str, tuple]:
    """W^T shapes ([N_out, K]) in draw order."""
    if w.chain == "rowscale":
        return {"W1t": (w.N, w.K1), "W2t": (w.N2, w.N)}
    if w.chain == "swiglu":
        return {"W1t": (w.N, w.K1), "Wgt": (w.N2, w.N), "Wut": (w.N2, w.N)}
    if w.chain == "full":
        return {"W1t": (w.N, w.K1), "Wgt": (w.inter, w.N), "Wut": (w.inter, w.N),
                "Wdt": (w.N, w.inter), "Wqt": (w.N2, w.N)}
    raise ValueError(w.chain)


def gamma_names(w: Workload):
    return ["gamma1", "gamma2"] if w.chain == "full" else ["gamma1"]


def make_inputs(w: Workload) -> Dict[str, torch.Tensor]:
    """Draw the workload's tensors on the CPU (use ``with_rows`` for a
    smaller M; that changes the draw, so both sides must use the same one)."""
    g = torch.Generator().manual_seed(w.seed)
    dt = _io_torch_dtype(w.dtype)
    out: Dict[str, torch.Tensor] = {}
    out["X"] = torch.randn(w.M, w.K1, generator=g, dtype=torch.float32)
    out["R"] = torch.randn(w.M, w.N, generator=g, dtype=torch.float32)
    if w.heavy_rows > 0:
        n_heavy = int(w.heavy_rows * w.M)
        idx = torch.randperm(w.M, generator=g)[:n_heavy]
        out["X"][idx] *= 50.0
        out["R"][idx] *= 50.0
        out["heavy_idx"] = idx
    for name, (n_out, k) in weight_shapes(w).items():
        out[name] = torch.randn(n_out, k, generator=g, dtype=torch.float32) * (1.0 / k ** 0.5)
    for name in gamma_names(w):
        out[name] = 1.0 + 0.1 * torch.randn(w.N, generator=g, dtype=torch.float32)
    for k in list(out):
        if k.startswith("gamma") or k == "heavy_idx":
            continue
        out[k] = out[k].to(dt).contiguous()
    return out


def sample_rows(M: int, n: int, seed: int = 1234) -> torch.Tensor:
    """Seeded row sample for checking full-size outputs row by row.

    Always includes the first and the last row (the ragged tail of the last
    M-tile) and draws the rest without replacement."""
    g = torch.Generator().manual_seed(seed)
    n = min(n, M)
    rest = torch.randperm(M - 2, generator=g)[: max(n - 2, 0)] + 1 if M > 2 else torch.empty(0, dtype=torch.long)
    idx = torch.cat([torch.tensor([0, M - 1]), rest]).unique()
    return idx.sort().values
