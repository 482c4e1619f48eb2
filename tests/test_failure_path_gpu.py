"""Failure detection without a GPU fault: every wait inside the kernels is
bounded by the GPU's global timer and, when its limit runs out, raises a
timeout bit in the device status word and returns instead of hanging.  The
self-test entry point runs that path on purpose (a wait on an mbarrier that
nothing signals, with a short limit); the host must read CODA_ERR_TIMEOUT once,
then a clean status, and the context must still compute correct results."""
import pytest
import torch

import gemm_epilogue_fusion_gb300 as g
from coda_inputs import WORKLOADS, make_inputs
from parity_util import compare, oracle_ref, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    g.load_library()
    yield


def test_bounded_wait_reports_timeout_once_and_context_survives():
    assert g.coda_get_device_status() == g.CODA_OK
    g.coda_selftest_wait_timeout(20_000_000)  # 20 ms
    with pytest.raises(g.CodaError) as err:
        g.coda_get_device_status()
    assert err.value.status == g.CODA_ERR_TIMEOUT
    assert g.coda_get_device_status() == g.CODA_OK  # read and cleared
    # the context still computes: a small block against the oracle
    w = WORKLOADS["llama1b_attn_out_swiglu"].with_rows(130)
    inp = make_inputs(w)
    compare(w, run_gpu(w, to_device(inp)), oracle_ref(w, inp))  # asserts every output within tolerance
    assert g.coda_get_device_status() == g.CODA_OK


def test_timeout_is_bounded_by_its_limit():
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.coda_selftest_wait_timeout(5_000_000)  # 5 ms
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    assert 4.0 <= ms < 500.0, ms
    with pytest.raises(g.CodaError):
        g.coda_get_device_status()
