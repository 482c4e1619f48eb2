"""Every compute entry point of the C ABI once, on small sizes that leave a
partial tile in every dimension (M = 300 rows, widths that are not multiples
of the tile), in one process: each call must return CODA_OK, write finite
values, and leave the device status clean.  The parity tests check the values;
this one checks that the calls run side by side without a bounds or status
problem, which is what a memory checker would look for."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _finite(*ts):
    for t in ts:
        assert torch.isfinite(t.float()).all()


def test_every_entry_point_on_ragged_sizes():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    dev = "cuda"
    gen = torch.Generator(device=dev).manual_seed(0)

    def rn(*s):
        return torch.randn(*s, generator=gen, device=dev)

    M, N, K, I, N2, eps = 300, 264, 392, 192, 136, 1e-5
    X, R = rn(M, K).bfloat16(), rn(M, N).bfloat16()
    W1t = (rn(N, K) / K ** 0.5).bfloat16()
    gamma = 1 + 0.1 * rn(N)
    Wg = g.coda_fold_gamma((rn(I, N) / N ** 0.5).bfloat16(), gamma)
    Wu = g.coda_fold_gamma((rn(I, N) / N ** 0.5).bfloat16(), gamma)
    W2 = g.coda_fold_gamma((rn(N2, N) / N ** 0.5).bfloat16(), gamma)

    H, P = g.coda_gemm_residual_partial_rms(X, W1t, R)
    r = g.coda_rms_reduce(P, N, eps)
    outs = [H, P, r, g.coda_gemm_rowscale(H, W2, r), g.coda_gemm_swiglu(H, Wg, Wu, r),
            g.coda_gemm_rowscale_fused_rms(H, W2, P, eps), g.coda_gemm_swiglu_fused_rms(H, Wg, Wu, P, eps),
            g.coda_gemm_rowscale_rope(H, W2, 8, 64, 500000.0, seq_len=128, P=P, eps=eps)]
    ws = g.block_workspace(M, dev)
    outs += list(g.coda_block_swiglu(X, W1t, R, Wg, Wu, eps, ws))
    outs += list(g.coda_block_rowscale(X, W1t, R, W2, eps, ws))
    outs += list(g.coda_block_swiglu_noalloc(X, W1t, R, Wg, Wu, eps))
    # general GEMM in both layouts (an MN-major A needs rows of M elements in 16-byte multiples)
    Xm = rn(304, K).bfloat16()
    outs.append(g.coda_gemm(Xm.t().contiguous(), W1t.t().contiguous(), a_mn=True, b_mn=True))
    outs.append(g.coda_gemm(X, W1t.t().contiguous(), b_mn=True))
    outs.append(g.coda_gemm(X, W1t))
    # backward
    dy, S = g.coda_gemm_grad_norm(rn(M, N2).bfloat16(), W2, H, gamma)
    outs += [dy, S, *g.coda_rmsnorm_backward(dy, H, r, gamma, S)]
    act, GU = g.coda_gemm_swiglu_save(H, Wg, Wu, r=r)
    Wd = (rn(N, I) / I ** 0.5).bfloat16()
    outs += [act, GU, g.coda_gemm_swiglu_backward(rn(M, N).bfloat16(), Wd, GU)]
    # FP8 helpers, with a tail of n mod 16 elements
    x = rn(1000 * 16 + 7).bfloat16()
    amax = g.coda_amax(x)
    q, s = g.coda_quantize_e4m3(x, amax)
    torch.cuda.synchronize()
    _finite(*[o for o in outs if o.is_floating_point()], amax, s)
    assert q.numel() == x.numel()
    assert g.coda_get_device_status() == g.CODA_OK
