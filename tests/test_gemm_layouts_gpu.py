"""coda_gemm with K-major and MN-major (transposed) operands, the products of
the backward pass, against the oracle's fp64 GEMM: both CTA-group forms,
ragged sizes, and the row/column scales of the epilogue."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    g.coda_get_device_status()


SHAPES = [(256, 512, 320), (200, 136, 520), (1024, 768, 512), (8, 64, 64), (520, 264, 1000)]


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("layouts", [(False, False), (False, True), (True, True)], ids=["NT", "NN", "TN"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_layouts(shape, layouts, cg, monkeypatch):
    import gemm_epilogue_fusion_gb300 as g
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    M, N, K = shape
    a_mn, b_mn = layouts
    gen = torch.Generator().manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=gen).bfloat16()
    B = torch.randn(N, K, generator=gen).bfloat16()
    rs = 1 + torch.rand(M, generator=gen)
    cs = 1 + torch.rand(N, generator=gen)
    Aa = (A.t() if a_mn else A).contiguous().cuda()
    Bb = (B.t() if b_mn else B).contiguous().cuda()
    D = g.coda_gemm(Aa, Bb, a_mn=a_mn, b_mn=b_mn, row_scale=rs.cuda(), col_scale=cs.cuda())
    torch.cuda.synchronize()
    ref = oracle.gemm(A, B.double().numpy().T.copy()) * rs.double().numpy()[:, None] * cs.double().numpy()[None, :]
    assert oracle.rel_err(D.cpu(), ref) <= 2e-2
