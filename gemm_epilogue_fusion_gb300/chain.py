"""The CODA blocks as sequences of C-ABI calls (no arithmetic here).

Each function enqueues the block's kernels on the current CUDA stream and
returns its outputs; ``bufs`` lets a caller (the benchmark) pass the output
tensors of a previous call back in so that nothing is allocated per step.

Blocks (the CODA write-up, section "CODA: the treasure hidden in the
epilogue"; SwiGLU gate/up from the same section and "five blocks"):
  rowscale_block  h = R + X W1 ; r ; Z = diag(r) h W2'            (3 launches)
  swiglu_block    h = R + X W1 ; r ; act = silu(r h Wg') (r h Wu') (3 launches)
  full_chain      LLaMA block tail and the next layer's QKV projection:
                  h1 = R + X Wo ; r1 ; act = SwiGLU(r1, h1) ;
                  h2 = h1 + act Wd ; r2 ; Z = diag(r2) h2 Wq'          (6 launches)
  full_chain_fp8  the same with every GEMM operand in per-tensor-scaled e4m3
  full_chain_fp8_blocks  the FP8 chain as amax(X) and two FP8 one-launch
                  blocks, which quantise X, h1, act and h2 themselves
                  (3 launches)
  full_chain_train_forward / full_chain_backward, rowscale_block_backward
                  the training forward that saves G || U and r, and the
                  backward from that state (12 launches for the full chain)
W' = diag(gamma) W is prepared once by ``fold_weights`` (coda_fold_gamma).
The one-launch forms of the two blocks are the binding's coda_block_rowscale
and coda_block_swiglu themselves.
With ``fused_reduce=True`` the reduction of the partials to r runs inside the
consuming GEMM's epilogue (coda_gemm_*_fused_rms) instead of its own launch;
r is still written out.
Weights are W^T [N_out, K] row-major throughout.
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import (coda_amax, coda_block_rowscale_fp8, coda_block_swiglu_fp8, coda_fold_gamma,
               coda_gemm_residual_partial_rms, coda_gemm_rowscale, coda_gemm_rowscale_fused_rms, coda_gemm_swiglu,
               coda_gemm_swiglu_fused_rms, coda_quantize_e4m3, coda_rms_reduce)


def _b(bufs, key):
    return None if bufs is None else bufs.get(key)


def fold_weights(chain: str, W: Dict[str, torch.Tensor], gammas: Dict[str, torch.Tensor]) -> Dict[str, torch.Tensor]:
    """Fold each RMSNorm weight into the GEMM that follows its norm."""
    out = dict(W)
    if chain == "rowscale":
        out["W2t"] = coda_fold_gamma(W["W2t"], gammas["gamma1"])
    elif chain == "swiglu":
        out["Wgt"] = coda_fold_gamma(W["Wgt"], gammas["gamma1"])
        out["Wut"] = coda_fold_gamma(W["Wut"], gammas["gamma1"])
    elif chain == "full":
        out["Wgt"] = coda_fold_gamma(W["Wgt"], gammas["gamma1"])
        out["Wut"] = coda_fold_gamma(W["Wut"], gammas["gamma1"])
        out["Wqt"] = coda_fold_gamma(W["Wqt"], gammas["gamma2"])
    else:
        raise ValueError(chain)
    return out


def _r_buf(bufs, key, P):
    r = _b(bufs, key)
    return torch.empty(P.shape[0], dtype=torch.float32, device=P.device) if r is None else r


def _rowscale(h, Wt, P, eps, bufs, rkey, zkey, fused, **scales):
    if fused:
        r = _r_buf(bufs, rkey, P)
        return coda_gemm_rowscale_fused_rms(h, Wt, P, eps, _b(bufs, zkey), r, **scales), r
    r = coda_rms_reduce(P, h.shape[1], eps, _b(bufs, rkey))
    return coda_gemm_rowscale(h, Wt, r, _b(bufs, zkey), **scales), r


def _swiglu(h, Wg, Wu, P, eps, bufs, rkey, akey, fused, **kw):
    if fused:
        r = _r_buf(bufs, rkey, P)
        return coda_gemm_swiglu_fused_rms(h, Wg, Wu, P, eps, _b(bufs, akey), r, **kw), r
    r = coda_rms_reduce(P, h.shape[1], eps, _b(bufs, rkey))
    return coda_gemm_swiglu(h, Wg, Wu, r, _b(bufs, akey), **kw), r


def rowscale_block(X, W1t, R, W2t_folded, eps: float, bufs: Optional[dict] = None, fused_reduce=False) -> dict:
    h, P = coda_gemm_residual_partial_rms(X, W1t, R, _b(bufs, "h"), _b(bufs, "P"))
    Z, r = _rowscale(h, W2t_folded, P, eps, bufs, "r", "Z", fused_reduce)
    return {"h": h, "P": P, "r": r, "Z": Z}


def swiglu_block(X, W1t, R, Wgt_folded, Wut_folded, eps: float, bufs: Optional[dict] = None,
                 fused_reduce=False) -> dict:
    h, P = coda_gemm_residual_partial_rms(X, W1t, R, _b(bufs, "h"), _b(bufs, "P"))
    act, r = _swiglu(h, Wgt_folded, Wut_folded, P, eps, bufs, "r", "act", fused_reduce)
    return {"h": h, "P": P, "r": r, "act": act}


def full_chain(X, Wot, R, Wgt_f, Wut_f, Wdt, Wqt_f, eps: float, bufs: Optional[dict] = None,
               fused_reduce=False) -> dict:
    h1, P1 = coda_gemm_residual_partial_rms(X, Wot, R, _b(bufs, "h1"), _b(bufs, "P1"))
    act, r1 = _swiglu(h1, Wgt_f, Wut_f, P1, eps, bufs, "r1", "act", fused_reduce)
    h2, P2 = coda_gemm_residual_partial_rms(act, Wdt, h1, _b(bufs, "h2"), _b(bufs, "P2"))
    Z, r2 = _rowscale(h2, Wqt_f, P2, eps, bufs, "r2", "Z", fused_reduce)
    return {"h1": h1, "P1": P1, "r1": r1, "act": act, "h2": h2, "P2": P2, "r2": r2, "Z": Z}


def quantize_weights(W: Dict[str, torch.Tensor]) -> Dict[str, tuple]:
    """Per-tensor e4m3 copies (q, scale) of already-folded weights."""
    out = {}
    for k, w in W.items():
        out[k] = coda_quantize_e4m3(w, coda_amax(w))
    return out


def full_chain_fp8(X, R, Wq8: Dict[str, tuple], eps: float, bufs: Optional[dict] = None,
                   fused_reduce=False) -> dict:
    """FP8 chain: X, h1, act, h2 quantised per tensor on the device (amax of
    h1, act and h2 comes out of the producing GEMM's epilogue); weights from
    ``quantize_weights`` (keys Wot, Wgt, Wut, Wdt, Wqt, gamma folded)."""
    b = bufs if bufs is not None else {}
    dev = X.device
    for k in ("ax", "a1", "a2", "a3"):
        if k not in b:
            b[k] = torch.empty(1, dtype=torch.float32, device=dev)
    Wo, so = Wq8["Wot"]
    Wg, sg = Wq8["Wgt"]
    Wu, su = Wq8["Wut"]
    Wd, sd = Wq8["Wdt"]
    Wq, sq = Wq8["Wqt"]
    coda_amax(X, b["ax"])
    Xq, sx = coda_quantize_e4m3(X, b["ax"], b.get("Xq"), b.get("sx"))
    h1, P1 = coda_gemm_residual_partial_rms(Xq, Wo, R, b.get("h1"), b.get("P1"), scale_x=sx, scale_w=so,
                                            amax_h=b["a1"])
    h1q, s1 = coda_quantize_e4m3(h1, b["a1"], b.get("h1q"), b.get("s1"))
    act, r1 = _swiglu(h1q, Wg, Wu, P1, eps, b, "r1", "act", fused_reduce, scale_h=s1, scale_wg=sg, scale_wu=su,
                      amax_act=b["a2"])
    actq, s2 = coda_quantize_e4m3(act, b["a2"], b.get("actq"), b.get("s2"))
    h2, P2 = coda_gemm_residual_partial_rms(actq, Wd, h1, b.get("h2"), b.get("P2"), scale_x=s2, scale_w=sd,
                                            amax_h=b["a3"])
    h2q, s3 = coda_quantize_e4m3(h2, b["a3"], b.get("h2q"), b.get("s3"))
    Z, r2 = _rowscale(h2q, Wq, P2, eps, b, "r2", "Z", fused_reduce, scale_h=s3, scale_w=sq)
    b.update({"Xq": Xq, "sx": sx, "h1": h1, "P1": P1, "r1": r1, "h1q": h1q, "s1": s1, "act": act, "actq": actq,
              "s2": s2, "h2": h2, "P2": P2, "r2": r2, "h2q": h2q, "s3": s3, "Z": Z})
    return b


def full_chain_fp8_blocks(X, R, Wq8: Dict[str, tuple], eps: float, workspace, bufs: Optional[dict] = None,
                          quantize_x_in_block: bool = True) -> dict:
    """The FP8 chain of ``full_chain_fp8`` in two FP8 one-launch blocks:
    amax(X); block 1 quantises X (or takes it from coda_quantize_e4m3 when
    quantize_x_in_block is False), runs Wo + residual, quantises h1 and runs
    gate/up SwiGLU; block 2 quantises act (its amax from block 1), runs the
    down projection with R = h1, quantises h2 and runs QKV.  Results equal
    ``full_chain_fp8``'s bit for bit.  ``workspace``: block_fp8_workspace(M)."""
    b = bufs if bufs is not None else {}
    dev = X.device
    for k in ("ax", "a1", "a2", "a3", "sx", "s1", "s2", "s3"):
        if k not in b:
            b[k] = torch.empty(1, dtype=torch.float32, device=dev)
    for k in ("r1", "r2"):
        if k not in b:
            b[k] = torch.empty(X.shape[0], dtype=torch.float32, device=dev)
    Wo, so = Wq8["Wot"]
    Wg, sg = Wq8["Wgt"]
    Wu, su = Wq8["Wut"]
    Wd, sd = Wq8["Wdt"]
    Wq, sq = Wq8["Wqt"]
    coda_amax(X, b["ax"])
    if quantize_x_in_block:
        xa = {"A": X, "amax_a": b["ax"], "Aq": b.get("Xq"), "scale_a": b["sx"]}
    else:
        Xq, sx = coda_quantize_e4m3(X, b["ax"], b.get("Xq"), b["sx"])
        xa = {"A": None, "amax_a": None, "Aq": Xq, "scale_a": sx}
    o1 = coda_block_swiglu_fp8(xa["A"], xa["amax_a"], Wo, so, R, Wg, sg, Wu, su, eps, workspace, Aq=xa["Aq"],
                               scale_a=xa["scale_a"], H=b.get("h1"), P=b.get("P1"), r_out=b.get("r1"),
                               amax_h=b["a1"], Hq=b.get("h1q"), scale_h=b["s1"], Act=b.get("act"), amax_act=b["a2"])
    o2 = coda_block_rowscale_fp8(o1["act"], b["a2"], Wd, sd, o1["h"], Wq, sq, eps, workspace, Aq=b.get("actq"),
                                 scale_a=b["s2"], H=b.get("h2"), P=b.get("P2"), r_out=b.get("r2"), amax_h=b["a3"],
                                 Hq=b.get("h2q"), scale_h=b["s3"], Z=b.get("Z"))
    b.update({"Xq": o1["Aq"], "h1": o1["h"], "P1": o1["P"], "h1q": o1["Hq"], "act": o1["act"], "actq": o2["Aq"],
              "h2": o2["h"], "P2": o2["P"], "h2q": o2["Hq"], "Z": o2["Z"]})
    return b


# ------------------------------------------------------------- backward ----
# Gradients of the blocks above (bf16), each step one of the library's calls:
#   coda_gemm_grad_norm      dy = dOut . W with the RMSNorm backward's row sums
#   coda_rmsnorm_backward    dh, r h, dgamma
#   coda_gemm (MN-major)     dX = dh . W1, dW = X^T dh, dW2 = (r h)^T dZ diag(gamma)
#   coda_gemm_swiglu_backward  dG, dU in the epilogue of dAct = dh2 . Wd
# Weights are the unfolded W^T [N_out, K] the forward folded gamma into.

def rowscale_block_backward(X, W1t, W2t, gamma, h, r, dZ, dH_in=None) -> dict:
    """Gradients of rowscale_block: dX, dR (= dh), dW1t, dW2t, dgamma."""
    from . import coda_gemm, coda_gemm_grad_norm, coda_rmsnorm_backward
    dy, S = coda_gemm_grad_norm(dZ, W2t, h, gamma)
    dh, Yt, dgamma = coda_rmsnorm_backward(dy, h, r, gamma, S, dH_in)
    return {"dX": coda_gemm(dh, W1t, b_mn=True), "dR": dh, "dW1t": coda_gemm(dh, X, a_mn=True, b_mn=True),
            "dW2t": coda_gemm(dZ, Yt, a_mn=True, b_mn=True, col_scale=gamma), "dgamma": dgamma}


def full_chain_train_forward(X, Wot, R, Wgt_f, Wut_f, Wdt, Wqt_f, eps: float) -> dict:
    """full_chain with the reductions in the consumers' epilogues, saving what
    the backward needs: r1, r2 and the SwiGLU pre-activations G || U."""
    from . import coda_gemm_swiglu_save
    h1, P1 = coda_gemm_residual_partial_rms(X, Wot, R)
    r1 = torch.empty(X.shape[0], dtype=torch.float32, device=X.device)
    act, GU = coda_gemm_swiglu_save(h1, Wgt_f, Wut_f, P=P1, eps=eps, r_out=r1)
    h2, P2 = coda_gemm_residual_partial_rms(act, Wdt, h1)
    r2 = torch.empty_like(r1)
    Z = coda_gemm_rowscale_fused_rms(h2, Wqt_f, P2, eps, None, r2)
    return {"h1": h1, "r1": r1, "act": act, "GU": GU, "h2": h2, "r2": r2, "Z": Z}


def full_chain_backward(X, Wot, Wgut, Wdt, Wqt, gamma1, gamma2, fwd: dict, dZ, dH2_in=None) -> dict:
    """Gradients of full_chain from the saved forward state.  Wgut is the
    unfolded gate and up weights stacked [2I, H] (Wgt above Wut)."""
    from . import coda_gemm, coda_gemm_grad_norm, coda_gemm_swiglu_backward, coda_rmsnorm_backward
    dy2, S2 = coda_gemm_grad_norm(dZ, Wqt, fwd["h2"], gamma2)
    dh2, Yt2, dgamma2 = coda_rmsnorm_backward(dy2, fwd["h2"], fwd["r2"], gamma2, S2, dH2_in)
    dWqt = coda_gemm(dZ, Yt2, a_mn=True, b_mn=True, col_scale=gamma2)
    dGU = coda_gemm_swiglu_backward(dh2, Wdt, fwd["GU"])
    dWdt = coda_gemm(dh2, fwd["act"], a_mn=True, b_mn=True)
    dy1, S1 = coda_gemm_grad_norm(dGU, Wgut, fwd["h1"], gamma1)
    dh1, Yt1, dgamma1 = coda_rmsnorm_backward(dy1, fwd["h1"], fwd["r1"], gamma1, S1, dh2)
    dWgut = coda_gemm(dGU, Yt1, a_mn=True, b_mn=True, col_scale=gamma1)
    return {"dX": coda_gemm(dh1, Wot, b_mn=True), "dR": dh1, "dWot": coda_gemm(dh1, X, a_mn=True, b_mn=True),
            "dWgut": dWgut, "dWdt": dWdt, "dWqt": dWqt, "dgamma1": dgamma1, "dgamma2": dgamma2, "dh2": dh2,
            "dGU": dGU}
