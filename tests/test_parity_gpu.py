"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded inputs, for every workload of the block, at sizes the
oracle finishes in seconds (several tiles plus a ragged tail in every
dimension) and, at full size, on sampled rows (rows are independent in the
block, so the oracle computes them one by one)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from coda_inputs import WORKLOADS, Workload, make_inputs, sample_rows
from parity_util import compare, oracle_ref, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    g.coda_get_device_status()  # raises if any kernel timed out


def _check(w: Workload, rows=None):
    inp = make_inputs(w)
    got = run_gpu(w, to_device(inp))
    ref = oracle_ref(w, inp, rows)
    return compare(w, got, ref, rows)


def test_tiny_f32_block_exact_config():
    """The tiny fp32 workload at its own size (tf32 tensor cores, fp32 I/O)."""
    errs = _check(WORKLOADS["tiny_f32"])
    print(errs)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rowscale_ragged_every_dim(dtype):
    # M: 1 full tile + 72 rows; K: not a multiple of the k-block; N, N2: not
    # multiples of the 256-column tile or the 128-column partial group
    K = 516 if dtype == "f32" else 520
    w = Workload("ragged", "rowscale", 200, K, 264, 136, 0, dtype, 1e-5, 7)
    _check(w)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_swiglu_ragged(dtype):
    w = Workload("ragged_swiglu", "swiglu", 130, 264, 392, 200, 0, dtype, 1e-5, 8)
    _check(w)


@pytest.mark.parametrize("M", [1, 8, 127, 129])
def test_tiny_rows(M):
    w = Workload("rows", "rowscale", M, 256, 256, 256, 0, "bf16", 1e-5, 9)
    _check(w)


def test_small_k_single_partial_block():
    w = Workload("smallk", "swiglu", 256, 8, 128, 128, 0, "bf16", 1e-5, 10)
    _check(w)


def test_llama1b_attn_out_swiglu_small_m():
    _check(WORKLOADS["llama1b_attn_out_swiglu"].with_rows(264))


def test_llama1b_mlp_down_qkv_small_m():
    _check(WORKLOADS["llama1b_mlp_down_qkv"].with_rows(136))


def test_llama8b_chain_small_m():
    _check(WORKLOADS["llama8b_chain"].with_rows(130))


@pytest.mark.parametrize("name", ["llama1b_attn_out_swiglu", "llama1b_mlp_down_qkv", "llama8b_chain",
                                  "llama70b_chain"])
def test_full_size_sampled_rows(name):
    """Full workload size, the launch configuration the benchmark times;
    the oracle checks a seeded sample of rows including the first and last."""
    w = WORKLOADS[name]
    rows = sample_rows(w.M, 12 if w.chain == "full" else 24)
    errs = _check(w, rows)
    print(name, errs)


def test_m_zero_is_a_noop():
    import gemm_epilogue_fusion_gb300 as g
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(128, 64, device="cuda").bfloat16()
    R = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    h, P = g.coda_gemm_residual_partial_rms(X, W, R)
    assert h.shape == (0, 128) and P.shape == (0, 1)


def test_zero_input_gives_eps_scale():
    """X = 0, R = 0: h = 0, every partial 0, r = 1/sqrt(eps)."""
    import gemm_epilogue_fusion_gb300 as g
    X = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(384, 256, device="cuda").bfloat16()
    R = torch.zeros(256, 384, dtype=torch.bfloat16, device="cuda")
    h, P = g.coda_gemm_residual_partial_rms(X, W, R)
    r = g.coda_rms_reduce(P, 384, 0.25)
    torch.cuda.synchronize()
    assert torch.count_nonzero(h).item() == 0 and torch.count_nonzero(P).item() == 0
    assert torch.all(r == 2.0)


def test_row_scale_invariance_heavy_rows():
    """RMSNorm output does not change when a row of h is scaled by c (eps
    small against the row's mean square): rows of X and R scaled by 50 give
    the same Z as the unscaled rows, up to bf16 rounding."""
    w = Workload("inv", "rowscale", 256, 512, 512, 384, 0, "bf16", 1e-6, 11)
    inp = make_inputs(w)
    d = to_device(inp)
    base = run_gpu(w, d)
    d2 = dict(d)
    d2["X"] = (d["X"].float() * 50).bfloat16()
    d2["R"] = (d["R"].float() * 50).bfloat16()
    sc = run_gpu(w, d2)
    assert oracle.rel_err(sc["Z"], base["Z"]) < 1e-2
    np.testing.assert_allclose(sc["r"].numpy() * 50, base["r"].numpy(), rtol=1e-2)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(1, 8), (3, 24), (257, 520), (14336, 4096)])
def test_fold_gamma_bit_exact(dtype, shape):
    """W'^T = W^T diag(gamma), each product in fp32 then rounded once: equal,
    bit for bit, to the same product rounded by torch (ragged row counts,
    one-vector rows, and the 8B gate weight's full size)."""
    import gemm_epilogue_fusion_gb300 as g
    if dtype == torch.float32 and shape[1] % 4:
        pytest.skip("fp32 rows of 16 bytes need K % 4 == 0")
    gen = torch.Generator(device="cuda").manual_seed(sum(shape))
    W = torch.randn(*shape, generator=gen, device="cuda").to(dtype)
    gam = torch.rand(shape[1], generator=gen, device="cuda") + 0.5
    out = g.coda_fold_gamma(W, gam)
    torch.cuda.synchronize()
    assert torch.equal(out, (W.float() * gam).to(dtype))
