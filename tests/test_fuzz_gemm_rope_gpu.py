"""Seeded random shapes for the general two-layout GEMM (the backward's
transposed products, with row and column scales) and for RoPE in the row-scale
epilogue, against the oracle: max |gpu - ref| / max |ref| within the bf16 bar
of 2e-2, in both CTA-group forms."""
import random

import numpy as np
import pytest
import torch

import oracle
from coda_inputs import Workload, make_inputs
from test_rope_gpu import run as run_rope

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    g.coda_get_device_status()


LAYOUTS = [(False, False), (False, True), (True, True)]


@pytest.mark.parametrize("seed", range(12))
def test_gemm_layouts_random_shapes(seed, monkeypatch):
    import gemm_epilogue_fusion_gb300 as g
    rnd = random.Random(9800 + seed)
    a_mn, b_mn = LAYOUTS[seed % 3]
    monkeypatch.setenv("CODA_CTA_GROUP", "2" if seed % 2 else "1")
    # MN-major operands are stored [K, M] / [K, N]: their rows need M, N multiples of 8; K is free there
    M = 8 * rnd.randint(1, 160) if a_mn else rnd.randint(1, 1300)
    N = 8 * rnd.randint(1, 160)
    K = rnd.randint(1, 1600) if a_mn and b_mn else 8 * rnd.randint(1, 200)
    gen = torch.Generator().manual_seed(seed)
    A = torch.randn(M, K, generator=gen).bfloat16()
    B = torch.randn(N, K, generator=gen).bfloat16()
    rs = 1 + torch.rand(M, generator=gen) if seed % 4 else None
    cs = 1 + torch.rand(N, generator=gen) if seed % 3 else None
    Aa = (A.t() if a_mn else A).contiguous().cuda()
    Bb = (B.t() if b_mn else B).contiguous().cuda()
    D = g.coda_gemm(Aa, Bb, a_mn=a_mn, b_mn=b_mn, row_scale=None if rs is None else rs.cuda(),
                    col_scale=None if cs is None else cs.cuda())
    torch.cuda.synchronize()
    ref = oracle.gemm(A, B.double().numpy().T.copy())
    if rs is not None:
        ref = ref * rs.double().numpy()[:, None]
    if cs is not None:
        ref = ref * cs.double().numpy()[None, :]
    err = oracle.rel_err(D.cpu(), ref)
    assert err <= 2e-2, (M, N, K, a_mn, b_mn, err)


@pytest.mark.parametrize("seed", range(6))
def test_rope_random_heads(seed, monkeypatch):
    rnd = random.Random(9850 + seed)
    monkeypatch.setenv("CODA_CTA_GROUP", "2" if seed % 2 else "1")
    head_dim = rnd.choice([64, 128])
    q_heads, kv_heads = rnd.randint(1, 8), rnd.randint(1, 4)
    rope_cols = head_dim * (q_heads + kv_heads)
    N2 = rope_cols + head_dim * kv_heads  # V after Q and K, unrotated
    w = Workload(f"rope_fuzz_{seed}", "rowscale", rnd.randint(1, 700), 8 * rnd.randint(1, 100),
                 8 * rnd.randint(8, 100), N2, 0, "bf16", 1e-5, 850 + seed)
    n_pos = rnd.randint(1, 4096)
    positions = None if seed % 2 else np.random.default_rng(seed).integers(0, 8192, w.M)
    run_rope(w, make_inputs(w), head_dim, rope_cols, n_pos, rnd.choice([10000.0, 500000.0]), positions=positions,
             fused=seed % 3 != 0)
