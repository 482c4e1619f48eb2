"""FP8 one-launch blocks (coda_block_swiglu_fp8, coda_block_rowscale_fp8) on
the GPU.  Each launch quantises its operands itself: X (when asked) before
the residual GEMM, h band by band once every CTA is past the residual GEMM.
The chain of amax(X) and the two blocks must equal the nine-launch FP8 chain
(coda_amax, coda_quantize_e4m3 and the e4m3 GEMMs as separate calls) bit for
bit, e4m3 codes and scales included, and match the quantisation-aware fp64
oracle within the FP8 tolerance."""
import os

import numpy as np
import pytest
import torch

from coda_inputs import WORKLOADS, Workload, make_inputs
from parity_util import compare, oracle_ref, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    assert g.coda_get_device_status() == g.CODA_OK


def _weights(w, d):
    from gemm_epilogue_fusion_gb300 import chain as C
    f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")}, {k: d[k] for k in d if k.startswith("gamma")})
    return C.quantize_weights({"Wot": f["W1t"], "Wgt": f["Wgt"], "Wut": f["Wut"], "Wdt": f["Wdt"], "Wqt": f["Wqt"]})


def _run_both(w, d, quantize_x_in_block):
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    q8 = _weights(w, d)
    ref = C.full_chain_fp8(d["X"], d["R"], q8, w.eps, fused_reduce=True)
    ws = g.block_fp8_workspace(w.M, d["X"].device)
    got = C.full_chain_fp8_blocks(d["X"], d["R"], q8, w.eps, ws, quantize_x_in_block=quantize_x_in_block)
    torch.cuda.synchronize()
    # the launches leave the workspace zeroed for the next call
    assert int(torch.count_nonzero(ws).item()) == 0
    return got, ref


KEYS = ("Xq", "sx", "h1", "P1", "r1", "a1", "h1q", "s1", "act", "a2", "actq", "s2", "h2", "P2", "r2", "a3", "h2q",
        "s3", "Z")

RAGGED = Workload("fp8_block_ragged", "full", 300, 272, 144, 200, 336, "e4m3", 1e-5, 17, heavy_rows=0.05)


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("xq", [True, False], ids=["x_in_block", "x_by_kernel"])
@pytest.mark.parametrize("w", [WORKLOADS["llama8b_chain_fp8"].with_rows(600), RAGGED], ids=["8b_m600", "ragged"])
def test_fp8_blocks_equal_separate_launches(w, xq, cg, monkeypatch):
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    inp = make_inputs(w)
    d = to_device(inp)
    got, ref = _run_both(w, d, xq)
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), k
    # and the quantisation-aware oracle (its own codec, amax and fp64 GEMMs)
    compare(w, {k: v.cpu() for k, v in got.items() if isinstance(v, torch.Tensor)}, oracle_ref(w, inp))


@pytest.mark.parametrize("m", [1, 17, 129])
def test_fp8_blocks_tiny_m(m):
    """Fewer quantiser chunks than quantiser warps, bands of a few rows, pairs
    whose second half lies past M: still the separate launches' bits."""
    w = Workload(f"fp8_block_m{m}", "full", m, 272, 144, 200, 336, "e4m3", 1e-5, 40 + m)
    d = to_device(make_inputs(w))
    got, ref = _run_both(w, d, True)
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), k


def test_fp8_blocks_twice_reuse_the_workspace():
    """Two calls in a row on one workspace (the first leaves it zeroed) and an
    all-zero X (scale 1, every code zero) both come out as the separate calls."""
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    w = WORKLOADS["llama8b_chain_fp8"].with_rows(264)
    d = to_device(make_inputs(w))
    q8 = _weights(w, d)
    ws = g.block_fp8_workspace(w.M, "cuda")
    for X in (d["X"], torch.zeros_like(d["X"])):
        ref = C.full_chain_fp8(X, d["R"], q8, w.eps, fused_reduce=True)
        for _ in range(2):
            got = C.full_chain_fp8_blocks(X, d["R"], q8, w.eps, ws)
            torch.cuda.synchronize()
            for k in KEYS:
                assert torch.equal(got[k], ref[k]), k
    assert float(ref["sx"].item()) == 1.0


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "llama8b_chain_fp8_rows.npz")


def test_fp8_blocks_full_size_vs_quantisation_aware_oracle():
    """M = 32768 (the configuration's size, the launches the benchmark times):
    the stored rows of the quantisation-aware oracle's whole-chain run."""
    from make_fp8_chain_golden import KEYS as GKEYS, input_digests
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    gold = np.load(GOLDEN)
    w = WORKLOADS["llama8b_chain_fp8"]
    inp = make_inputs(w)
    dig = input_digests(inp)
    assert [f"{k}:{dig[k]}" for k in GKEYS] == list(gold["digests"]), "input generator changed: regenerate the golden"
    d = to_device(inp)
    ws = g.block_fp8_workspace(w.M, "cuda")
    got = C.full_chain_fp8_blocks(d["X"], d["R"], _weights(w, d), w.eps, ws)
    torch.cuda.synchronize()
    rows = torch.from_numpy(gold["rows"])
    got_c = {k: got[k].cpu() for k in ("h1", "r1", "act", "h2", "r2", "Z")}
    errs = compare(w, got_c, {k: gold[k] for k in ("h1", "r1", "act", "h2", "r2", "Z")}, rows)
    print("FP8 blocks vs quantisation-aware oracle", errs)
    for a, t in (("a1", "h1"), ("a2", "act"), ("a3", "h2")):
        assert float(got[a].item()) == float(got[t].float().abs().max()), a
