"""Seeded random shapes for the one-launch blocks and the two-block chain.

Each case draws M, K, N and the consumer's width at random (multiples of 8, so
every row is a whole number of 16-byte chunks), with a few hand-picked edge
shapes: one row, one 8-column k-block, widths just past a tile or a 128-column
partial group.  The one-launch block must equal the separate-call path bit for
bit in both CTA-group forms, leave its workspace zeroed, and match the oracle
(max |gpu - ref| / max |ref| within the bf16 / tf32 bar of 2e-2)."""
import random

import pytest
import torch

from coda_inputs import Workload, make_inputs
from parity_util import compare, oracle_ref, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    g.coda_get_device_status()


def _random_block(seed: int) -> Workload:
    rnd = random.Random(9000 + seed)
    chain = "rowscale" if seed % 2 == 0 else "swiglu"
    dtype = "f32" if seed % 5 == 4 else "bf16"
    return Workload(f"fuzz_{chain}_{dtype}_{seed}", chain, rnd.randint(1, 1300), 8 * rnd.randint(1, 300),
                    8 * rnd.randint(1, 160), 8 * rnd.randint(1, 160), 0, dtype, rnd.choice([1e-6, 1e-5]),
                    300 + seed)


EDGE = [
    Workload("edge_one_row", "rowscale", 1, 8, 8, 8, 0, "bf16", 1e-5, 401),
    Workload("edge_one_kblock", "swiglu", 257, 8, 136, 72, 0, "bf16", 1e-5, 402),
    Workload("edge_tile_plus_one", "rowscale", 257, 264, 264, 264, 0, "bf16", 1e-5, 403),
    Workload("edge_group_plus_8", "swiglu", 129, 136, 136, 136, 0, "bf16", 1e-5, 404),
    Workload("edge_f32_one_row", "swiglu", 1, 16, 24, 8, 0, "f32", 1e-6, 405),
]
CASES = [_random_block(s) for s in range(12)] + EDGE


def _run_block(w, d, ws):
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    f = C.fold_weights(w.chain, {k: d[k] for k in d if k.startswith("W")},
                       {k: d[k] for k in d if k.startswith("gamma")})
    r = torch.empty(w.M, dtype=torch.float32, device="cuda")
    if w.chain == "rowscale":
        h, P, Z = g.coda_block_rowscale(d["X"], d["W1t"], d["R"], f["W2t"], w.eps, ws, r_out=r)
        out = {"h": h, "P": P, "r": r, "Z": Z}
    else:
        h, P, act = g.coda_block_swiglu(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], w.eps, ws, r_out=r)
        out = {"h": h, "P": P, "r": r, "act": act}
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


_REFS = {}


def _ref(w, inp):
    if w.name not in _REFS:
        _REFS[w.name] = oracle_ref(w, inp)
    return _REFS[w.name]


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}_M{w.M}_K{w.K1}_N{w.N}_N2{w.N2}")
def test_block_random_shapes(w, cg, monkeypatch):
    import gemm_epilogue_fusion_gb300 as g
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    inp = make_inputs(w)
    d = to_device(inp)
    ws = g.block_workspace(w.M, "cuda")
    sep = run_gpu(w, d, fused_reduce=True)
    blk = _run_block(w, d, ws)
    assert torch.count_nonzero(ws).item() == 0, "workspace not left zeroed"
    for k in blk:
        assert torch.equal(blk[k], sep[k]), k
    compare(w, blk, _ref(w, inp))


def _random_chain(seed: int) -> Workload:
    rnd = random.Random(9500 + seed)
    return Workload(f"fuzz_chain_{seed}", "full", rnd.randint(1, 900), 8 * rnd.randint(1, 200),
                    8 * rnd.randint(1, 120), 8 * rnd.randint(1, 120), 8 * rnd.randint(1, 200), "bf16", 1e-5,
                    500 + seed)


@pytest.mark.parametrize("w", [_random_chain(s) for s in range(4)],
                         ids=lambda w: f"{w.name}_M{w.M}_K{w.K1}_H{w.N}_Q{w.N2}_I{w.inter}")
def test_chain_random_shapes(w):
    """The block tail as the bench runs it (two one-launch blocks) on random
    widths: equal to the separate calls bit for bit and to the oracle's chain."""
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    inp = make_inputs(w)
    d = to_device(inp)
    sep = run_gpu(w, d, fused_reduce=True)
    f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")},
                       {k: d[k] for k in d if k.startswith("gamma")})
    ws1, ws2 = g.block_workspace(w.M, "cuda"), g.block_workspace(w.M, "cuda")
    r1 = torch.empty(w.M, dtype=torch.float32, device="cuda")
    r2 = torch.empty(w.M, dtype=torch.float32, device="cuda")
    h1, _, act = g.coda_block_swiglu(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], w.eps, ws1, r_out=r1)
    h2, _, Z = g.coda_block_rowscale(act, d["Wdt"], h1, f["Wqt"], w.eps, ws2, r_out=r2)
    torch.cuda.synchronize()
    blk = {"h1": h1.cpu(), "r1": r1.cpu(), "act": act.cpu(), "h2": h2.cpu(), "r2": r2.cpu(), "Z": Z.cpu()}
    for k, v in blk.items():
        assert torch.equal(v, sep[k]), k
    compare(w, blk, oracle_ref(w, inp))
