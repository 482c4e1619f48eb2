"""RoPE in the QKV GEMM's epilogue (coda_gemm_rowscale_rope) against the
oracle's unfused block: GEMM -> residual add -> RMSNorm -> QKV GEMM -> RoPE on
the Q and K heads (RoFormer rotation, interleaved pairs), V unrotated."""
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


def run(w, inp, head_dim, rope_cols, n_pos, base, positions=None, fused=True, rows=None):
    import gemm_epilogue_fusion_gb300 as g
    d = to_device(inp)
    W2 = g.coda_fold_gamma(d["W2t"], d["gamma1"])
    h, P = g.coda_gemm_residual_partial_rms(d["X"], d["W1t"], d["R"])
    pos_d = None if positions is None else torch.as_tensor(positions, dtype=torch.int32).cuda()
    kw = dict(seq_len=n_pos, positions=pos_d)
    if fused:
        r = torch.empty(w.M, dtype=torch.float32, device="cuda")
        Z = g.coda_gemm_rowscale_rope(h, W2, head_dim, rope_cols, base, P=P, eps=w.eps, r_out=r, **kw)
    else:
        r = g.coda_rms_reduce(P, w.N, w.eps)
        Z = g.coda_gemm_rowscale_rope(h, W2, head_dim, rope_cols, base, r=r, **kw)
    torch.cuda.synchronize()
    pos = np.arange(w.M) % n_pos if positions is None else np.asarray(positions)
    sel = slice(None) if rows is None else rows
    ref = oracle.block_rowscale_rope(inp["X"][sel], W(inp["W1t"]), inp["R"][sel], inp["gamma1"], W(inp["W2t"]),
                                     w.eps, rope_cols, head_dim, pos[sel], base)
    got_z = Z.cpu()[sel]
    errs = {"Z": oracle.rel_err(got_z, ref["Z"]), "r": oracle.rel_err(r.cpu()[sel], ref["r"])}
    assert max(errs.values()) <= TOL[w.dtype], errs
    return errs


# QKV of 4 query heads + 2 key/value heads of 64 (1B-style head size)
SMALL = Workload("rope_small", "rowscale", 300, 520, 512, 512, 0, "bf16", 1e-5, 71)


@pytest.mark.parametrize("cg", ["1", "2"])
@pytest.mark.parametrize("fused", [True, False])
def test_rope_small_both_forms(cg, fused, monkeypatch):
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    run(SMALL, make_inputs(SMALL), 64, 384, 128, 500000.0, fused=fused)


def test_rope_fp32_and_explicit_positions():
    w = Workload("rope_f32", "rowscale", 200, 256, 256, 384, 0, "f32", 1e-5, 72)
    pos = np.random.default_rng(0).integers(0, 4096, w.M)
    run(w, make_inputs(w), 32, 256, 4096, 10000.0, positions=pos)


def test_rope_llama8b_qkv_shape_large_angles():
    # hidden 4096, QKV 6144 = 32 query heads + 8 key heads of 128 rotated, 8 value heads not;
    # positions near the end of a 2048-token sequence (angles up to ~2047 rad)
    w = Workload("rope_8b", "rowscale", 130, 4096, 4096, 6144, 0, "bf16", 1e-5, 73)
    pos = 2047 - np.arange(w.M)
    run(w, make_inputs(w), 128, 5120, 2048, 500000.0, positions=pos)


def test_rope_llama8b_qkv_full_size_sampled_rows():
    # M = 16384 tokens (batch 8 x seq 2048), positions = row mod 2048
    w = dataclass_replace(WORKLOADS["llama8b_chain"])
    rows = sample_rows(w.M, 10)
    run(w, make_inputs(w), 128, 5120, 2048, 500000.0, rows=rows.numpy())


def dataclass_replace(w):
    # the 8B chain's tail as a row-scale block: h = R + X Wo, then QKV on h
    return Workload("rope_8b_full", "rowscale", w.M, w.K1, w.N, w.N2, 0, "bf16", w.eps, 74)


def run_block_vs_separate(w, head_dim, rope_cols, n_pos, base, positions=None, rows=None):
    """coda_block_rowscale_rope (one launch) against the separate calls
    (residual GEMM, then the row-scale GEMM with the reduction and RoPE in its
    epilogue) bit for bit, and against the oracle's unfused block + RoPE."""
    import gemm_epilogue_fusion_gb300 as g
    inp = make_inputs(w)
    d = to_device(inp)
    W2 = g.coda_fold_gamma(d["W2t"], d["gamma1"])
    pos_d = None if positions is None else torch.as_tensor(positions, dtype=torch.int32).cuda()
    kw = dict(seq_len=n_pos, positions=pos_d)
    h, P = g.coda_gemm_residual_partial_rms(d["X"], d["W1t"], d["R"])
    r = torch.empty(w.M, dtype=torch.float32, device="cuda")
    Z = g.coda_gemm_rowscale_rope(h, W2, head_dim, rope_cols, base, P=P, eps=w.eps, r_out=r, **kw)
    ws = g.block_workspace(w.M, "cuda")
    rb = torch.empty_like(r)
    for _ in range(2):  # the second call reuses the workspace the first left zeroed
        hb, Pb, Zb = g.coda_block_rowscale_rope(d["X"], d["W1t"], d["R"], W2, w.eps, ws, head_dim, rope_cols, base,
                                                r_out=rb, **kw)
        torch.cuda.synchronize()
        assert torch.count_nonzero(ws).item() == 0
        for a, b, k in ((hb, h, "h"), (Pb, P, "P"), (rb, r, "r"), (Zb, Z, "Z")):
            assert torch.equal(a, b), k
    pos = np.arange(w.M) % n_pos if positions is None else np.asarray(positions)
    sel = slice(None) if rows is None else rows
    ref = oracle.block_rowscale_rope(inp["X"][sel], W(inp["W1t"]), inp["R"][sel], inp["gamma1"], W(inp["W2t"]),
                                     w.eps, rope_cols, head_dim, pos[sel], base)
    errs = {"Z": oracle.rel_err(Zb.cpu()[sel], ref["Z"]), "h": oracle.rel_err(hb.cpu()[sel], ref["h"])}
    assert max(errs.values()) <= TOL[w.dtype], errs


@pytest.mark.parametrize("cg", ["1", "2"])
def test_block_rope_small_equals_separate_calls(cg, monkeypatch):
    monkeypatch.setenv("CODA_CTA_GROUP", cg)
    run_block_vs_separate(SMALL, 64, 384, 128, 500000.0)


def test_block_rope_llama8b_shape_explicit_positions():
    w = Workload("rope_block_8b", "rowscale", 300, 4096, 4096, 6144, 0, "bf16", 1e-5, 75)
    pos = np.random.default_rng(1).integers(0, 2048, w.M)
    run_block_vs_separate(w, 128, 5120, 2048, 500000.0, positions=pos)


def test_block_rope_llama8b_full_size_sampled_rows():
    """M = 16384 (the 8B chain's down projection + QKV block size): the block
    with RoPE on the 40 query and key heads, bit-equal to the separate calls,
    sampled rows against the oracle."""
    w = Workload("rope_block_8b_full", "rowscale", 16384, 14336, 4096, 6144, 0, "bf16", 1e-5, 76)
    run_block_vs_separate(w, 128, 5120, 2048, 500000.0, rows=sample_rows(w.M, 8).numpy())
