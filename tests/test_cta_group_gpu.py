"""Both GEMM forms on the same cases: one CTA per 128-row tile
(tcgen05 cta_group::1) and CTA pairs per 256-row tile (cta_group::2, the peer
CTA's half of A and B feeding the even CTA's MMA).  The form is forced with
CODA_CTA_GROUP, which the library reads on every call.  Shapes cover a pair
whose second half lies entirely beyond M, ragged K, N and N2, and the
SwiGLU split (gate rows in one CTA, up rows in the other)."""
import pytest
import torch

from coda_inputs import Workload, WORKLOADS
from parity_util import compare, oracle_ref, run_gpu, to_device
from coda_inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    g.coda_get_device_status()


CASES = [
    Workload("pair_rowscale_ragged", "rowscale", 300, 520, 264, 136, 0, "bf16", 1e-5, 31),   # 2nd tile half-empty
    Workload("pair_rowscale_f32", "rowscale", 100, 516, 392, 264, 0, "f32", 1e-5, 32),       # peer rows all >= M
    Workload("pair_swiglu", "swiglu", 520, 264, 392, 200, 0, "bf16", 1e-5, 33),
    Workload("pair_swiglu_f32", "swiglu", 257, 128, 256, 136, 0, "f32", 1e-5, 34),
    Workload("pair_many_tiles", "rowscale", 1024, 1024, 1536, 1280, 0, "bf16", 1e-5, 35),
]


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forced_cta_group(w, cg, monkeypatch):
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    inp = make_inputs(w)
    compare(w, run_gpu(w, to_device(inp)), oracle_ref(w, inp))


@pytest.mark.parametrize("cg", ["1", "2"])
def test_forced_cta_group_fp8_chain(cg, monkeypatch):
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    w = WORKLOADS["llama8b_chain_fp8"].with_rows(200)
    inp = make_inputs(w)
    compare(w, run_gpu(w, to_device(inp)), oracle_ref(w, inp))
