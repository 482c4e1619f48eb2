"""coda_block_swiglu_noalloc: the one-launch SwiGLU block for callers that
cannot allocate device memory (its band counters live inside the library).
Called through the C ABI, twice in a row (the second call reuses the built-in
counters the first one left behind), its outputs must match the workspace
form coda_block_swiglu within the parity tolerance.  This file runs last, and
also passes on its own in a fresh process."""
import os
import sys

import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
from coda_inputs import Workload, make_inputs  # noqa: E402

TOL = 2e-2


def _inputs(w):
    import gemm_epilogue_fusion_gb300 as g
    inp = make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items()}
    Wg = g.coda_fold_gamma(d["Wgt"], d["gamma1"])
    Wu = g.coda_fold_gamma(d["Wut"], d["gamma1"])
    return d, Wg, Wu


@pytest.mark.gpu
@pytest.mark.parametrize("w", [Workload("noalloc_1b", "swiglu", 1000, 2048, 2048, 1024, 0, "bf16", 1e-5, 61),
                               Workload("noalloc_ragged", "swiglu", 300, 264, 392, 200, 0, "bf16", 1e-5, 62)],
                         ids=lambda w: w.name)
def test_noalloc_block_matches_workspace_block_twice(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    d, Wg, Wu = _inputs(w)
    ws = g.block_workspace(w.M, "cuda")
    h_ref, P_ref, act_ref = g.coda_block_swiglu(d["X"], d["W1t"], d["R"], Wg, Wu, w.eps, ws)
    # the caller's outputs, allocated once up front: the calls themselves must allocate nothing
    T = g.coda_partial_cols(w.N)
    h = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
    P = torch.empty(w.M, T, dtype=torch.float32, device="cuda")
    act = torch.empty(w.M, w.N2, dtype=torch.bfloat16, device="cuda")
    r = torch.empty(w.M, dtype=torch.float32, device="cuda")
    for call in range(2):
        torch.cuda.synchronize()
        allocs = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        free = torch.cuda.mem_get_info()[0]
        g.coda_block_swiglu_noalloc(d["X"], d["W1t"], d["R"], Wg, Wu, w.eps, H=h, P=P, Act=act, r_out=r)
        torch.cuda.synchronize()
        if call == 1:
            # the first call may load the kernel's code onto the device; from
            # then on a call changes neither torch's allocations nor the
            # device's free memory
            assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == allocs
            assert torch.cuda.mem_get_info()[0] == free
        for got, ref in ((h, h_ref), (P, P_ref), (act, act_ref)):
            assert oracle.rel_err(got.cpu(), ref.cpu()) <= TOL
    g.coda_get_device_status()


def test_noalloc_rejects_rows_beyond_its_counters():
    import gemm_epilogue_fusion_gb300 as g
    lib = g.load_library()
    A = 0x7F0000000000
    st = lib.coda_block_swiglu_noalloc(A, A, A, A, A, 1e-5, A, A, None, A, 131073, 512, 512, 512, 1, None)
    assert st == g.CODA_ERR_INVALID_ARG
    assert b"131072" in lib.coda_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("cg", ["1", "2"])
def test_noalloc_block_at_its_row_limit(cg, monkeypatch):
    """M = 131072, the most rows the built-in counters serve.  With one CTA per
    tile the launch uses every one of them (1024 bands of 128 rows and the
    completion counter).  The outputs equal the workspace form bit for bit, and
    sampled rows (the first, the last, and the rows of the last two bands)
    match the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    from coda_inputs import sample_rows
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    g.load_library()
    w = Workload("noalloc_max", "swiglu", 131072, 256, 256, 256, 0, "bf16", 1e-5, 63)
    inp = make_inputs(w)
    d = {k: v.cuda() for k, v in inp.items()}
    Wg = g.coda_fold_gamma(d["Wgt"], d["gamma1"])
    Wu = g.coda_fold_gamma(d["Wut"], d["gamma1"])
    ws = g.block_workspace(w.M, "cuda")
    ref = g.coda_block_swiglu(d["X"], d["W1t"], d["R"], Wg, Wu, w.eps, ws)
    got = g.coda_block_swiglu_noalloc(d["X"], d["W1t"], d["R"], Wg, Wu, w.eps)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    rows = torch.cat([sample_rows(w.M, 8), torch.arange(w.M - 256, w.M, 37)]).unique()
    Wt = lambda t: t.double().numpy().T.copy()  # noqa: E731
    o = oracle.block_swiglu(inp["X"][rows], Wt(inp["W1t"]), inp["R"][rows], inp["gamma1"], Wt(inp["Wgt"]),
                            Wt(inp["Wut"]), w.eps)
    assert oracle.rel_err(got[0].cpu()[rows], o["h"]) <= TOL
    assert oracle.rel_err(got[2].cpu()[rows], o["act"]) <= TOL
    assert g.coda_get_device_status() == g.CODA_OK
