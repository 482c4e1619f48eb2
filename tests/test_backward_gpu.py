"""Backward of the block and of the LLaMA block-tail chain on the GPU
(grad-norm GEMM epilogue, RMSNorm backward kernel, MN-major GEMMs for dX and
the weight gradients, SwiGLU backward in the down projection's gradient GEMM)
against the oracle's unfused fp64 backward."""
import numpy as np
import pytest
import torch

import oracle
from coda_inputs import WORKLOADS, Workload, make_inputs, sample_rows
from parity_util import TOL, W, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    g.coda_get_device_status()


def _check(got, ref, pairs, tol=TOL["bf16"], rows=None):
    errs = {}
    for gk, rk, transpose in pairs:
        gv = got[gk].cpu()
        if rows is not None:
            gv = gv[rows]
        rv = ref[rk].T if transpose else ref[rk]
        errs[gk] = oracle.rel_err(gv, rv)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"backward parity above {tol}: {bad} (all {errs})"
    return errs


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("with_dh", [False, True])
def test_rowscale_block_backward(cg, with_dh, monkeypatch):
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    w = Workload("bwd_rowscale", "rowscale", 300, 520, 264, 392, 0, "bf16", 1e-5, 81)
    inp = make_inputs(w)
    d = to_device(inp)
    gen = torch.Generator().manual_seed(82)
    dZ = torch.randn(w.M, w.N2, generator=gen).bfloat16()
    dH = torch.randn(w.M, w.N, generator=gen).bfloat16() if with_dh else None
    W2f = g.coda_fold_gamma(d["W2t"], d["gamma1"])
    fwd = C.rowscale_block(d["X"], d["W1t"], d["R"], W2f, w.eps, fused_reduce=True)
    got = C.rowscale_block_backward(d["X"], d["W1t"], d["W2t"], d["gamma1"], fwd["h"], fwd["r"], dZ.cuda(),
                                    None if dH is None else dH.cuda())
    torch.cuda.synchronize()
    ref = oracle.block_rowscale_backward(inp["X"], W(inp["W1t"]), inp["R"], inp["gamma1"], W(inp["W2t"]), w.eps,
                                         dZ, dH)
    print(_check(got, ref, [("dX", "dX", False), ("dR", "dR", False), ("dW1t", "dW1", True),
                            ("dW2t", "dW2", True), ("dgamma", "dgamma", False)]))


def _chain_case(w, seed):
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    inp = make_inputs(w)
    d = to_device(inp)
    gen = torch.Generator().manual_seed(seed)
    dZ = torch.randn(w.M, w.N2, generator=gen).bfloat16()
    dH2 = torch.randn(w.M, w.N, generator=gen).bfloat16()
    f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")}, {k: d[k] for k in d if k.startswith("gamma")})
    fwd = C.full_chain_train_forward(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], d["Wdt"], f["Wqt"], w.eps)
    Wgut = torch.cat([d["Wgt"], d["Wut"]], 0).contiguous()
    got = C.full_chain_backward(d["X"], d["W1t"], Wgut, d["Wdt"], d["Wqt"], d["gamma1"], d["gamma2"], fwd,
                                dZ.cuda(), dH2.cuda())
    torch.cuda.synchronize()
    I = w.inter
    got["dWgt"], got["dWut"] = got["dWgut"][:I], got["dWgut"][I:]
    got["dG"], got["dU"] = got["dGU"][:, :I], got["dGU"][:, I:]
    return inp, dZ, dH2, got


CHAIN_PAIRS = [("dX", "dX", False), ("dR", "dR", False), ("dWot", "dWo", True), ("dWgt", "dWg", True),
               ("dWut", "dWu", True), ("dWdt", "dWd", True), ("dWqt", "dWq", True), ("dgamma1", "dgamma1", False),
               ("dgamma2", "dgamma2", False), ("dh2", "dh2", False), ("dG", "dG", False), ("dU", "dU", False)]


@pytest.mark.parametrize("cg", ["1", "2"])
def test_chain_backward_ragged(cg, monkeypatch):
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    # I = 576: two full 256-column tiles and one 64-column box (I must be a multiple of 64)
    w = Workload("bwd_chain", "full", 300, 264, 392, 136, 576, "bf16", 1e-5, 83)
    inp, dZ, dH2, got = _chain_case(w, 84)
    ref = oracle.chain_full_backward(inp["X"], W(inp["W1t"]), inp["R"], inp["gamma1"], W(inp["Wgt"]),
                                     W(inp["Wut"]), W(inp["Wdt"]), inp["gamma2"], W(inp["Wqt"]), w.eps, dZ, dH2)
    print(_check(got, ref, CHAIN_PAIRS))


def test_chain_backward_llama8b_shapes_small_m():
    w = WORKLOADS["llama8b_chain"].with_rows(136)
    inp, dZ, dH2, got = _chain_case(w, 85)
    ref = oracle.chain_full_backward(inp["X"], W(inp["W1t"]), inp["R"], inp["gamma1"], W(inp["Wgt"]),
                                     W(inp["Wut"]), W(inp["Wdt"]), inp["gamma2"], W(inp["Wqt"]), w.eps, dZ, dH2)
    print(_check(got, ref, CHAIN_PAIRS))


def test_chain_backward_llama8b_full_size_sampled_rows():
    """M = 16384: the activation gradients of a row depend on that row alone,
    so the oracle checks a seeded sample of rows of dX, dR, dh2, dG, dU (the
    weight gradients sum over every row; the small cases cover them)."""
    w = WORKLOADS["llama8b_chain"]
    inp, dZ, dH2, got = _chain_case(w, 86)
    rows = sample_rows(w.M, 6)
    ref = oracle.chain_full_backward(inp["X"][rows], W(inp["W1t"]), inp["R"][rows], inp["gamma1"], W(inp["Wgt"]),
                                     W(inp["Wut"]), W(inp["Wdt"]), inp["gamma2"], W(inp["Wqt"]), w.eps, dZ[rows],
                                     dH2[rows])
    print(_check(got, ref, [p for p in CHAIN_PAIRS if p[0] in ("dX", "dR", "dh2", "dG", "dU")], rows=rows))


def test_chain_backward_llama8b_full_size_weight_gradients():
    """M = 16384, the launch configuration bench.py times: each weight gradient
    (and dX) is a transposed product over all 16384 rows, which the row-sampled
    oracle cannot see.  Each is checked against an fp32 product of the very
    bf16 operands the backward fed its kernel, at the parity bar."""
    import gemm_epilogue_fusion_gb300 as g
    from gemm_epilogue_fusion_gb300 import chain as C
    w = WORKLOADS["llama8b_chain"]
    inp = make_inputs(w)
    d = to_device(inp)
    gen = torch.Generator(device="cuda").manual_seed(87)
    dZ = torch.randn(w.M, w.N2, generator=gen, device="cuda").bfloat16()
    f = C.fold_weights("full", {k: d[k] for k in d if k.startswith("W")}, {k: d[k] for k in d if k.startswith("gamma")})
    fwd = C.full_chain_train_forward(d["X"], d["W1t"], d["R"], f["Wgt"], f["Wut"], d["Wdt"], f["Wqt"], w.eps)
    Wgut = torch.cat([d["Wgt"], d["Wut"]], 0).contiguous()
    g1, g2 = d["gamma1"], d["gamma2"]
    # the backward's steps, keeping every operand of its weight-gradient products
    dy2, S2 = g.coda_gemm_grad_norm(dZ, d["Wqt"], fwd["h2"], g2)
    dh2, Yt2, _ = g.coda_rmsnorm_backward(dy2, fwd["h2"], fwd["r2"], g2, S2)
    dGU = g.coda_gemm_swiglu_backward(dh2, d["Wdt"], fwd["GU"])
    dy1, S1 = g.coda_gemm_grad_norm(dGU, Wgut, fwd["h1"], g1)
    dh1, Yt1, _ = g.coda_rmsnorm_backward(dy1, fwd["h1"], fwd["r1"], g1, S1, dh2)
    got = {"dWqt": g.coda_gemm(dZ, Yt2, a_mn=True, b_mn=True, col_scale=g2),
           "dWdt": g.coda_gemm(dh2, fwd["act"], a_mn=True, b_mn=True),
           "dWgut": g.coda_gemm(dGU, Yt1, a_mn=True, b_mn=True, col_scale=g1),
           "dWot": g.coda_gemm(dh1, d["X"], a_mn=True, b_mn=True),
           "dX": g.coda_gemm(dh1, d["W1t"], b_mn=True)}
    ref = {"dWqt": (dZ.float().t() @ Yt2.float()) * g2,
           "dWdt": dh2.float().t() @ fwd["act"].float(),
           "dWgut": (dGU.float().t() @ Yt1.float()) * g1,
           "dWot": dh1.float().t() @ d["X"].float(),
           "dX": dh1.float() @ d["W1t"].float()}
    torch.cuda.synchronize()
    errs = {k: float((got[k].float() - ref[k]).abs().max() / (ref[k].abs().max() + 1e-6)) for k in got}
    print(errs)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
    assert g.coda_get_device_status() == g.CODA_OK


@pytest.mark.parametrize("cg", ["1", "2"])
def test_swiglu_save_matches_plain_forward_and_oracle(cg, monkeypatch):
    """The saving forward's act equals coda_gemm_swiglu_fused_rms bit for bit,
    and its G || U are the oracle's pre-activations (y Wg, y Wu)."""
    import gemm_epilogue_fusion_gb300 as g
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    w = Workload("save", "swiglu", 300, 264, 392, 576, 0, "bf16", 1e-5, 87)
    inp = make_inputs(w)
    d = to_device(inp)
    Wg = g.coda_fold_gamma(d["Wgt"], d["gamma1"])
    Wu = g.coda_fold_gamma(d["Wut"], d["gamma1"])
    h, P = g.coda_gemm_residual_partial_rms(d["X"], d["W1t"], d["R"])
    act_plain = g.coda_gemm_swiglu_fused_rms(h, Wg, Wu, P, w.eps)
    act, GU = g.coda_gemm_swiglu_save(h, Wg, Wu, P=P, eps=w.eps)
    torch.cuda.synchronize()
    assert torch.equal(act.cpu(), act_plain.cpu())
    hh = oracle.gemm(inp["X"], W(inp["W1t"]), inp["R"])
    y, _ = oracle.rmsnorm(hh, inp["gamma1"], w.eps)
    I = w.N2
    assert oracle.rel_err(GU[:, :I].cpu(), oracle.gemm(y, W(inp["Wgt"]))) <= TOL["bf16"]
    assert oracle.rel_err(GU[:, I:].cpu(), oracle.gemm(y, W(inp["Wut"]))) <= TOL["bf16"]
