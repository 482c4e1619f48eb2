"""The auxiliary reduction folded into the consuming GEMM's epilogue
(coda_gemm_rowscale_fused_rms, coda_gemm_swiglu_fused_rms): every output,
r included, must equal the separate-launch path bit for bit (both reduce a
row's partials with the same routine in the same order), and match the oracle."""
import pytest
import torch

from coda_inputs import WORKLOADS, Workload, make_inputs
from parity_util import PAIRS, compare, oracle_ref, run_gpu, to_device

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
    WORKLOADS["tiny_f32"],
    Workload("ragged_rowscale", "rowscale", 300, 520, 264, 136, 0, "bf16", 1e-5, 41),
    Workload("ragged_swiglu", "swiglu", 520, 264, 392, 200, 0, "bf16", 1e-5, 42),
    WORKLOADS["llama1b_attn_out_swiglu"].with_rows(1000),
    WORKLOADS["llama8b_chain"].with_rows(300),
    WORKLOADS["llama8b_chain_fp8"].with_rows(300),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_reduce_equals_separate_launch(w):
    inp = make_inputs(w)
    d = to_device(inp)
    sep = run_gpu(w, d, fused_reduce=False)
    fus = run_gpu(w, d, fused_reduce=True)
    for g, _ in PAIRS[w.chain]:
        assert torch.equal(sep[g], fus[g]), g
    compare(w, fus, oracle_ref(w, inp))
