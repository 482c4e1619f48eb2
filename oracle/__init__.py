"""CPU oracle for the CODA GEMM-epilogue block -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg and ``--impl reference`` arm may import this package.  The CUDA product
path never does.

What it computes is the *plain, unfused* definition of the block that the CODA
news write-ups reparameterise ("CODA: the treasure hidden in the epilogue"):

    h  = R + X.W1                          first GEMM + residual add
    r  = 1 / sqrt(mean_j h_j^2 + eps)      RMSNorm row scale
    y  = h * r * gamma                     RMSNorm output (LLaMA form)
    Z  = y.W2                              second GEMM
 or act = silu(y.Wg) * (y.Wu)               SwiGLU gate/up ("five blocks":
                                           elementwise activation)

The GPU path computes the reparameterised form (diag(r) moved past the second
GEMM, gamma folded into its weight); the oracle deliberately does not, so that
the two meet only in their results.  All arithmetic is fp64 in the C file
``coda_oracle.c``; this module only marshals numpy arrays and composes the
steps in the order the block applies them.

Parity pins (tests/test_oracle.py): hand-derived 4x4 cases and a one-row chain
in tests/golden/, numpy fp64 matmul on a C0-sized case, the reparameterisation
identity, RMSNorm scale invariance, silu special values, the E4M3 codec
against torch's float8_e4m3fn over all 256 codes, bf16 rounding against
torch's fp32 -> bf16 cast and hand-worked ties, a hand-derived FP8 chain in
which every quantisation site (and the fold before it) changes the result,
RoPE against its complex-number form (rotation composes, depends only on the
relative position, leaves V and position 0 alone), and central finite
differences for the backward functions.

Weights are passed in the mathematical orientation W [K, N] (``nn.Linear``'s
weight transposed).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "coda_oracle.c")
_LIB = os.path.join(_HERE, "libcoda_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP; no -ffast-math, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.coda_oracle_gemm.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64]
            lib.coda_oracle_rmsnorm.argtypes = [_dp, _dp, ctypes.c_double, _i64, _i64, _dp, _dp]
            lib.coda_oracle_silu.argtypes = [ctypes.c_double]
            lib.coda_oracle_silu.restype = ctypes.c_double
            lib.coda_oracle_silu_mul.argtypes = [_dp, _dp, _i64, _dp]
            lib.coda_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.coda_oracle_e4m3_decode.restype = ctypes.c_double
            lib.coda_oracle_e4m3_encode.argtypes = [ctypes.c_double]
            lib.coda_oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.coda_oracle_amax.argtypes = [_dp, _i64]
            lib.coda_oracle_amax.restype = ctypes.c_double
            lib.coda_oracle_e4m3_fake_quant.argtypes = [_dp, _i64, _dp]
            lib.coda_oracle_e4m3_fake_quant.restype = ctypes.c_double
            lib.coda_oracle_round_bf16_array.argtypes = [_dp, _i64, _dp]
            lib.coda_oracle_round_bf16_array.restype = None
            lib.coda_oracle_rmsnorm_backward.argtypes = [_dp, _dp, ctypes.c_double, _dp, _i64, _i64, _dp, _dp]
            lib.coda_oracle_silu_mul_backward.argtypes = [_dp, _dp, _dp, _i64, _dp, _dp]
            lib.coda_oracle_threads.argtypes = [ctypes.c_int]
            lib.coda_oracle_threads.restype = ctypes.c_int
            lib.coda_oracle_rope.argtypes = [_dp, _i64, _i64, _i64, _i64, ctypes.POINTER(ctypes.c_int64),
                                             ctypes.c_double]
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: widen its exact bits
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


# ---------------------------------------------------------------- steps ----

def set_threads(n: int) -> int:
    """Threads of the oracle's OpenMP loops (n > 0 sets it); returns the count in
    effect.  Only for timing: results do not depend on it."""
    return int(_load().coda_oracle_threads(int(n)))


def gemm(A, W, R=None) -> np.ndarray:
    """C = R + A.W (R optional).  A [M,K], W [K,N]."""
    A, W = _f64(A), _f64(W)
    M, K = A.shape
    K2, N = W.shape
    assert K == K2, (A.shape, W.shape)
    C = np.empty((M, N), dtype=np.float64)
    Rp = None
    if R is not None:
        R = _f64(R)
        assert R.shape == (M, N)
        Rp = _ptr(R)
    _load().coda_oracle_gemm(_ptr(A), _ptr(W), Rp, _ptr(C), M, N, K)
    return C


def rmsnorm(H, gamma, eps: float):
    """Returns (y, rstd) with rstd_i = 1/sqrt(mean_j h_ij^2 + eps), y = h*rstd*gamma."""
    H, gamma = _f64(H), _f64(gamma)
    M, N = H.shape
    Y = np.empty_like(H)
    rstd = np.empty(M, dtype=np.float64)
    _load().coda_oracle_rmsnorm(_ptr(H), _ptr(gamma), float(eps), M, N, _ptr(Y), _ptr(rstd))
    return Y, rstd


def silu(x: float) -> float:
    return _load().coda_oracle_silu(float(x))


def silu_mul(G, U) -> np.ndarray:
    G, U = _f64(G), _f64(U)
    assert G.shape == U.shape
    out = np.empty_like(G)
    _load().coda_oracle_silu_mul(_ptr(G), _ptr(U), G.size, _ptr(out))
    return out


def swiglu(Y, Wg, Wu) -> np.ndarray:
    """act = silu(Y.Wg) * (Y.Wu)."""
    return silu_mul(gemm(Y, Wg), gemm(Y, Wu))


def e4m3_encode(x: float) -> int:
    return int(_load().coda_oracle_e4m3_encode(float(x)))


def e4m3_decode(code: int) -> float:
    return float(_load().coda_oracle_e4m3_decode(int(code)))


def round_bf16(x) -> np.ndarray:
    """x rounded to the nearest bfloat16 value (ties to even), as fp64."""
    x = _f64(x)
    out = np.empty_like(x)
    _load().coda_oracle_round_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def fake_quant_e4m3(x):
    """Per-tensor E4M3 quantise-dequantise with s = amax/448.  Returns (x~, s)."""
    x = _f64(x)
    out = np.empty_like(x)
    s = _load().coda_oracle_e4m3_fake_quant(_ptr(x), x.size, _ptr(out))
    return out, s


def rope(Z, rot_cols: int, head_dim: int, positions, base: float) -> np.ndarray:
    """RoPE (RoFormer, interleaved pairs) on the first rot_cols columns of Z,
    head by head; row i rotated for position positions[i].  Returns a copy."""
    Z = _f64(Z).copy()
    M, N = Z.shape
    assert rot_cols <= N and rot_cols % head_dim == 0 and head_dim % 2 == 0
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    assert pos.shape == (M,)
    _load().coda_oracle_rope(_ptr(Z), M, N, rot_cols, head_dim, pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                             float(base))
    return Z


def rmsnorm_backward(H, gamma, eps: float, dY):
    """(dH, dgamma) of y = RMSNorm(h) * gamma for the upstream gradient dY."""
    H, gamma, dY = _f64(H), _f64(gamma), _f64(dY)
    M, N = H.shape
    dH = np.empty_like(H)
    dg = np.empty(N, dtype=np.float64)
    _load().coda_oracle_rmsnorm_backward(_ptr(H), _ptr(gamma), float(eps), _ptr(dY), M, N, _ptr(dH), _ptr(dg))
    return dH, dg


def silu_mul_backward(G, U, dAct):
    """(dG, dU) of act = silu(G) * U."""
    G, U, dAct = _f64(G), _f64(U), _f64(dAct)
    dG, dU = np.empty_like(G), np.empty_like(G)
    _load().coda_oracle_silu_mul_backward(_ptr(G), _ptr(U), _ptr(dAct), G.size, _ptr(dG), _ptr(dU))
    return dG, dU


# --------------------------------------------------------------- blocks ----

def block_rowscale(X, W1, R, gamma, W2, eps):
    """GEMM -> residual add -> RMSNorm -> GEMM, unfused."""
    h = gemm(X, W1, R)
    y, rstd = rmsnorm(h, gamma, eps)
    return {"h": h, "r": rstd, "Z": gemm(y, W2)}


def block_swiglu(X, W1, R, gamma, Wg, Wu, eps):
    """GEMM -> residual add -> RMSNorm -> gate/up GEMMs -> SwiGLU, unfused."""
    h = gemm(X, W1, R)
    y, rstd = rmsnorm(h, gamma, eps)
    return {"h": h, "r": rstd, "act": swiglu(y, Wg, Wu)}


def block_rowscale_rope(X, W1, R, gamma, W2, eps, rot_cols, head_dim, positions, base):
    """GEMM -> residual add -> RMSNorm -> QKV GEMM -> RoPE on the Q and K
    columns (the first rot_cols), unfused."""
    out = block_rowscale(X, W1, R, gamma, W2, eps)
    out["Z"] = rope(out["Z"], rot_cols, head_dim, positions, base)
    return out


def block_rowscale_backward(X, W1, R, gamma, W2, eps, dZ, dH_in=None):
    """Gradients of GEMM -> residual add -> RMSNorm -> GEMM (unfused) for the
    upstream dZ and, optionally, dH_in flowing into h along the residual
    stream.  Returns dX, dR (= dh), dW1 [K, N], dW2 [N, N2], dgamma."""
    h = gemm(X, W1, R)
    y, r = rmsnorm(h, gamma, eps)
    dW2 = gemm(y.T.copy(), dZ)
    dy = gemm(_f64(dZ), _f64(W2).T.copy())
    dh, dgamma = rmsnorm_backward(h, gamma, eps, dy)
    if dH_in is not None:
        dh = dh + _f64(dH_in)
    return {"dX": gemm(dh, _f64(W1).T.copy()), "dR": dh, "dW1": gemm(_f64(X).T.copy(), dh), "dW2": dW2,
            "dgamma": dgamma, "h": h, "r": r}


def block_swiglu_backward(X, W1, R, gamma, Wg, Wu, eps, dAct, dH_in=None):
    """Gradients of GEMM -> residual add -> RMSNorm -> gate/up GEMMs -> SwiGLU
    (unfused).  Returns dX, dR (= dh), dW1, dWg, dWu [N, I], dgamma."""
    h = gemm(X, W1, R)
    y, r = rmsnorm(h, gamma, eps)
    G, U = gemm(y, Wg), gemm(y, Wu)
    dG, dU = silu_mul_backward(G, U, dAct)
    yT = y.T.copy()
    dy = gemm(dG, _f64(Wg).T.copy()) + gemm(dU, _f64(Wu).T.copy())
    dh, dgamma = rmsnorm_backward(h, gamma, eps, dy)
    if dH_in is not None:
        dh = dh + _f64(dH_in)
    return {"dX": gemm(dh, _f64(W1).T.copy()), "dR": dh, "dW1": gemm(_f64(X).T.copy(), dh),
            "dWg": gemm(yT, dG), "dWu": gemm(yT, dU), "dgamma": dgamma, "h": h, "r": r}


def chain_full(X, Wo, R, gamma1, Wg, Wu, Wd, gamma2, Wq, eps):
    """Pre-norm LLaMA block tail and the next layer's QKV projection:
    h1 = R + X.Wo ; y1 = RMSNorm(h1) ; act = SwiGLU(y1) ; h2 = h1 + act.Wd ;
    y2 = RMSNorm(h2) ; Z = y2.Wq."""
    h1 = gemm(X, Wo, R)
    y1, r1 = rmsnorm(h1, gamma1, eps)
    act = swiglu(y1, Wg, Wu)
    h2 = gemm(act, Wd, h1)
    y2, r2 = rmsnorm(h2, gamma2, eps)
    return {"h1": h1, "r1": r1, "act": act, "h2": h2, "r2": r2, "Z": gemm(y2, Wq)}


def chain_full_backward(X, Wo, R, gamma1, Wg, Wu, Wd, gamma2, Wq, eps, dZ, dH2_in=None):
    """Gradients of chain_full for the upstream dZ (of the QKV output) and,
    optionally, dH2_in (of the residual stream h2).  Unfused fp64: the
    forward is recomputed, then each step's derivative in reverse order."""
    f = chain_full(X, Wo, R, gamma1, Wg, Wu, Wd, gamma2, Wq, eps)
    h1, h2 = f["h1"], f["h2"]
    y1, _ = rmsnorm(h1, gamma1, eps)
    y2, _ = rmsnorm(h2, gamma2, eps)
    G, U = gemm(y1, Wg), gemm(y1, Wu)
    T = lambda a: _f64(a).T.copy()  # noqa: E731
    # Z = y2 Wq
    dWq = gemm(T(y2), dZ)
    dh2, dgamma2 = rmsnorm_backward(h2, gamma2, eps, gemm(dZ, T(Wq)))
    if dH2_in is not None:
        dh2 = dh2 + _f64(dH2_in)
    # h2 = h1 + act Wd
    dAct = gemm(dh2, T(Wd))
    dWd = gemm(T(f["act"]), dh2)
    # act = silu(G) U, G = y1 Wg, U = y1 Wu
    dG, dU = silu_mul_backward(G, U, dAct)
    dWg, dWu = gemm(T(y1), dG), gemm(T(y1), dU)
    dh1, dgamma1 = rmsnorm_backward(h1, gamma1, eps, gemm(dG, T(Wg)) + gemm(dU, T(Wu)))
    dh1 = dh1 + dh2
    # h1 = R + X Wo
    return {"dX": gemm(dh1, T(Wo)), "dR": dh1, "dWo": gemm(T(X), dh1), "dWg": dWg, "dWu": dWu, "dWd": dWd,
            "dWq": dWq, "dgamma1": dgamma1, "dgamma2": dgamma2, "dh2": dh2, "dG": dG, "dU": dU}


def chain_full_fp8(X, Wo, R, gamma1, Wg, Wu, Wd, gamma2, Wq, eps, out_rows=None):
    """Quantisation-aware FP8 chain.  FP8 changes the arithmetic, so here the
    oracle follows the reparameterised steps and quantises exactly the GEMM
    operands an FP8 implementation feeds the tensor cores: X, every weight
    (gamma folded in first), h1, act and h2, each with its own per-tensor
    scale amax/448.  R, h, r and the outputs stay unquantised.

    The quantiser reads each tensor as the block stores it, rounded to bf16:
    the folded weights, h1, act and h2 (X and the weights arrive in bf16).
    The write-up names FP8 operands but not the precision the quantiser reads;
    an e4m3 code is a decision that a rounding of its input can flip, so it is
    taken on the stored bf16 value, and so is amax, which sets every code's
    scale.

    ``out_rows``: when given, every result is returned for those rows only and
    the last GEMM (Z) is computed for them alone.  The per-tensor scales still
    come from the whole tensors, so the values equal the full computation's."""
    q = lambda t: fake_quant_e4m3(round_bf16(t))[0]
    g1, g2 = _f64(gamma1), _f64(gamma2)
    Wg_f = _f64(Wg) * g1[:, None]
    Wu_f = _f64(Wu) * g1[:, None]
    Wq_f = _f64(Wq) * g2[:, None]
    h1 = gemm(q(X), q(Wo), R)
    _, r1 = rmsnorm(h1, g1, eps)
    h1q = q(h1)
    G = gemm(h1q, q(Wg_f)) * r1[:, None]
    U = gemm(h1q, q(Wu_f)) * r1[:, None]
    act = silu_mul(G, U)
    del G, U
    h2 = gemm(q(act), q(Wd), h1)
    _, r2 = rmsnorm(h2, g2, eps)
    h2q = q(h2)
    sel = slice(None) if out_rows is None else np.asarray(out_rows)
    Z = gemm(h2q[sel], q(Wq_f)) * r2[sel][:, None]
    return {"h1": h1[sel], "r1": r1[sel], "act": act[sel], "h2": h2[sel], "r2": r2[sel], "Z": Z}


def rel_err(got, ref) -> float:
    """max |got - ref| / (max |ref| + 1e-6): the parity metric of the block."""
    got, ref = _f64(got), _f64(ref)
    return float(np.max(np.abs(got - ref)) / (np.max(np.abs(ref)) + 1e-6)) if ref.size else 0.0
