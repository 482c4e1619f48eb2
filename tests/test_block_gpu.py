"""One-launch blocks (coda_block_rowscale, coda_block_swiglu): the residual
GEMM and its consumer in one persistent kernel, the consumer's row bands
waiting on per-band counters.  Every output must equal the separate-call path
bit for bit, match the oracle, and leave the workspace zeroed for reuse; both
CTA-group forms; ragged shapes; back-to-back calls on one workspace."""
import pytest
import torch

from coda_inputs import WORKLOADS, Workload, make_inputs
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


def run_block(w, d, ws):
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    gam = {k: d[k] for k in d if k.startswith("gamma")}
    Wd = {k: d[k] for k in d if k.startswith("W")}
    f = C.fold_weights(w.chain, Wd, gam)
    r = torch.empty(w.M, dtype=torch.float32, device="cuda")
    if w.chain == "rowscale":
        h, P, Z = g.coda_block_rowscale(d["X"], d["W1t"], d["R"], f["W2t"], w.eps, ws, r_out=r)
        out = {"h": h, "P": P, "r": r, "Z": Z}
    else:
        h, P, act = g.coda_block_swiglu(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], w.eps, ws, r_out=r)
        out = {"h": h, "P": P, "r": r, "act": act}
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


CASES = [
    WORKLOADS["tiny_f32"],
    Workload("block_ragged_rowscale", "rowscale", 300, 520, 264, 136, 0, "bf16", 1e-5, 51),
    Workload("block_ragged_swiglu", "swiglu", 520, 264, 392, 200, 0, "bf16", 1e-5, 52),
    Workload("block_f32_swiglu", "swiglu", 257, 128, 256, 136, 0, "f32", 1e-5, 53),
    WORKLOADS["llama1b_attn_out_swiglu"].with_rows(1000),
    WORKLOADS["llama1b_mlp_down_qkv"].with_rows(777),
    # K rows of 8192+ bytes and a small weight: the residual phase walks N-major
    # rows with the weight kept in L2; ragged M, N and N2 / I
    Workload("block_ragged_nmajor_rowscale", "rowscale", 600, 4160, 392, 200, 0, "bf16", 1e-5, 54),
    Workload("block_ragged_nmajor_swiglu", "swiglu", 450, 4104, 264, 136, 0, "bf16", 1e-5, 55),
]


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_block_equals_separate_calls(w, cg, monkeypatch):
    import gemm_epilogue_fusion_gb300 as g
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    inp = make_inputs(w)
    d = to_device(inp)
    ws = g.block_workspace(w.M, "cuda")
    sep = run_gpu(w, d, fused_reduce=True)
    for _ in range(2):  # the second call reuses the workspace the first left zeroed
        blk = run_block(w, d, ws)
        assert torch.count_nonzero(ws).item() == 0, "workspace not left zeroed"
        for k in blk:
            assert torch.equal(blk[k], sep[k]), k
    compare(w, blk, oracle_ref(w, inp))


@pytest.mark.parametrize("name", ["llama1b_attn_out_swiglu", "llama1b_mlp_down_qkv"])
def test_block_full_size_equals_separate_calls(name):
    import gemm_epilogue_fusion_gb300 as g
    w = WORKLOADS[name]
    inp = make_inputs(w)
    d = to_device(inp)
    ws = g.block_workspace(w.M, "cuda")
    sep = run_gpu(w, d, fused_reduce=True)
    blk = run_block(w, d, ws)
    for k in blk:
        assert torch.equal(blk[k], sep[k]), k
    assert torch.count_nonzero(ws).item() == 0


@pytest.mark.parametrize("name", ["llama8b_chain", "llama70b_chain"])
def test_block_full_size_chain_equals_separate_calls(name):
    """The LLaMA-8B block-tail chain as two one-launch blocks (Wo + gate/up,
    then down + QKV, the bench's default step), at full size, and the same at
    LLaMA-70B shapes.  The second 8B block has phase-A tiles of K = 14336
    against phase-B tiles of K = 4096 and 1024 phase-A tiles over 76 CTA pairs,
    so its units walk the balanced order."""
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    w = WORKLOADS[name]
    inp = make_inputs(w)
    d = to_device(inp)
    sep = run_gpu(w, d, fused_reduce=True)
    gam = {k: d[k] for k in d if k.startswith("gamma")}
    f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")}, gam)
    ws1, ws2 = g.block_workspace(w.M, "cuda"), g.block_workspace(w.M, "cuda")
    r1 = torch.empty(w.M, dtype=torch.float32, device="cuda")
    r2 = torch.empty(w.M, dtype=torch.float32, device="cuda")
    h1, P1, act = g.coda_block_swiglu(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], w.eps, ws1, r_out=r1)
    h2, P2, Z = g.coda_block_rowscale(act, d["Wdt"], h1, f["Wqt"], w.eps, ws2, r_out=r2)
    torch.cuda.synchronize()
    blk = {"h1": h1, "r1": r1, "act": act, "h2": h2, "r2": r2, "Z": Z}
    for k, v in blk.items():
        assert torch.equal(v.cpu(), sep[k]), k
    assert torch.count_nonzero(ws1).item() == 0 and torch.count_nonzero(ws2).item() == 0


def test_block_rejects_fp8_and_missing_workspace():
    import gemm_epilogue_fusion_gb300 as g
    X = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    W = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    R = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    ws = g.block_workspace(128, "cuda")
    with pytest.raises(g.CodaError, match="UNSUPPORTED"):
        g.coda_block_rowscale(X, W, R, W, 1e-5, ws, H=R.clone(), Z=R.clone())


@pytest.mark.parametrize("cg", ["1", "2"])
def test_blocks_replay_in_a_cuda_graph(cg, monkeypatch):
    """The two one-launch blocks of the block tail captured once in a CUDA graph
    and replayed: every replay equals the eager calls bit for bit, and each
    launch leaves its workspace zeroed for the next, so replays need no reset."""
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    w = Workload("graph_chain", "full", 700, 264, 392, 200, 576, "bf16", 1e-5, 61)
    inp = make_inputs(w)
    d = to_device(inp)
    f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")}, {k: d[k] for k in d if k.startswith("gamma")})
    ws1, ws2 = g.block_workspace(w.M, "cuda"), g.block_workspace(w.M, "cuda")
    M, H, I, Q = w.M, w.N, w.inter, w.N2
    e = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    out = {"h1": e(M, H), "P1": e(M, g.coda_partial_cols(H), dt=torch.float32), "act": e(M, I),
           "h2": e(M, H), "P2": e(M, g.coda_partial_cols(H), dt=torch.float32), "Z": e(M, Q)}
    s = torch.cuda.Stream()

    def step():
        g.coda_block_swiglu(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], w.eps, ws1, H=out["h1"], P=out["P1"],
                            Act=out["act"], stream=s)
        g.coda_block_rowscale(out["act"], d["Wdt"], out["h1"], f["Wqt"], w.eps, ws2, H=out["h2"], P=out["P2"],
                              Z=out["Z"], stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in out.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for _ in range(3):
        for v in out.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(out[k], eager[k]), k
        assert torch.count_nonzero(ws1).item() == 0 and torch.count_nonzero(ws2).item() == 0
