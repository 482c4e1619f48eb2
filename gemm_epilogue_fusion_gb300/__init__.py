"""Python binding of the GB300 fused GEMM-epilogue library (``include/coda.h``).

Argument marshalling only: every function here takes torch tensors, checks
that they are contiguous CUDA tensors, passes their device pointers, sizes and
the current CUDA stream to the C ABI function of the same name, and raises
``CodaError`` on a non-OK status.  All arithmetic runs in the library's
kernels; PyTorch only provides device memory and streams.  Outputs can be
passed in (pre-allocated) or are allocated with ``torch.empty``.

The library is ``libcoda_gb300.so`` next to this file, compiled for sm_103a
by ``_build.build()``.  There is no fallback: if it cannot be built or
loaded, importing a function raises.

Hot path (the CODA write-up, section "CODA: the treasure hidden in the
epilogue"):

    h, P = coda_gemm_residual_partial_rms(X, W1t, R)   # h = R + X W1, partial sums of h^2
    r    = coda_rms_reduce(P, N, eps)                  # r = 1/sqrt(mean h^2 + eps)
    Z    = coda_gemm_rowscale(h, W2t_folded, r)        # diag(r) h diag(gamma) W2
    act  = coda_gemm_swiglu(h, Wgt_folded, Wut_folded, r)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

CODA_OK, CODA_ERR_INVALID_ARG, CODA_ERR_UNSUPPORTED, CODA_ERR_CUDA, CODA_ERR_TIMEOUT = range(5)
CODA_F32, CODA_BF16, CODA_E4M3 = 0, 1, 2
CODA_K_MAJOR, CODA_MN_MAJOR = 0, 1

_STATUS_NAMES = {0: "CODA_OK", 1: "CODA_ERR_INVALID_ARG", 2: "CODA_ERR_UNSUPPORTED", 3: "CODA_ERR_CUDA",
                 4: "CODA_ERR_TIMEOUT"}

# Every symbol include/coda.h declares, with (restype, argtypes).
_vp, _fp, _i64, _i32, _f32 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "coda_version": (_i32, []),
    "coda_status_string": (ctypes.c_char_p, [_i32]),
    "coda_last_error": (ctypes.c_char_p, []),
    "coda_partial_cols": (_i64, [_i64]),
    "coda_fold_gamma": (_i32, [_vp, _fp, _vp, _i64, _i64, _i32, _vp]),
    "coda_gemm_residual_partial_rms": (_i32, [_vp, _vp, _vp, _vp, _fp, _i64, _i64, _i64, _i32, _fp, _fp, _fp, _vp]),
    "coda_rms_reduce": (_i32, [_fp, _i64, _i64, _f32, _fp, _vp]),
    "coda_gemm_rowscale": (_i32, [_vp, _vp, _fp, _vp, _i64, _i64, _i64, _i32, _fp, _fp, _vp]),
    "coda_gemm_swiglu": (_i32, [_vp, _vp, _vp, _fp, _vp, _i64, _i64, _i64, _i32, _fp, _fp, _fp, _fp, _vp]),
    "coda_gemm_rowscale_fused_rms": (_i32, [_vp, _vp, _fp, _f32, _fp, _vp, _i64, _i64, _i64, _i32, _fp, _fp, _vp]),
    "coda_gemm_swiglu_fused_rms": (_i32, [_vp, _vp, _vp, _fp, _f32, _fp, _vp, _i64, _i64, _i64, _i32, _fp, _fp, _fp,
                                          _fp, _vp]),
    "coda_block_workspace_bytes": (_i64, [_i64]),
    "coda_block_rowscale": (_i32, [_vp, _vp, _vp, _vp, _f32, _vp, _fp, _fp, _vp, _i64, _i64, _i64, _i64, _i32, _vp,
                                   _vp]),
    "coda_block_swiglu": (_i32, [_vp, _vp, _vp, _vp, _vp, _f32, _vp, _fp, _fp, _vp, _i64, _i64, _i64, _i64, _i32, _vp,
                                 _vp]),
    "coda_block_rowscale_rope": (_i32, [_vp, _vp, _vp, _vp, _f32, _vp, _fp, _fp, _vp, _i64, _i64, _i64, _i64, _i32,
                                        _i64, _i64, ctypes.c_double, _i64, _vp, _vp, _vp]),
    "coda_block_swiglu_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _f32, _vp, _fp, _fp, _vp, _i64, _i64, _i64, _i64,
                                         _i32, _vp]),
    "coda_gemm_rowscale_rope": (_i32, [_vp, _vp, _fp, _fp, _f32, _fp, _vp, _i64, _i64, _i64, _i32, _fp, _fp, _i64,
                                       _i64, ctypes.c_double, _i64, _vp, _vp]),
    "coda_gemm": (_i32, [_vp, _i32, _vp, _i32, _vp, _i64, _i64, _i64, _i32, _fp, _fp, _vp]),
    "coda_gemm_grad_norm": (_i32, [_vp, _vp, _vp, _fp, _vp, _fp, _i64, _i64, _i64, _i32, _vp]),
    "coda_rmsnorm_backward_workspace_bytes": (_i64, [_i64, _i64]),
    "coda_rmsnorm_backward": (_i32, [_vp, _vp, _fp, _fp, _fp, _vp, _vp, _vp, _fp, _fp, _i64, _i64, _vp]),
    "coda_gemm_swiglu_backward": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]),
    "coda_gemm_swiglu_save": (_i32, [_vp, _vp, _vp, _fp, _fp, _f32, _fp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]),
    "coda_block_fp8_workspace_bytes": (_i64, [_i64]),
    "coda_block_swiglu_fp8": (_i32, [_vp, _fp, _vp, _fp, _vp, _fp, _vp, _vp, _fp, _vp, _fp, _f32, _vp, _fp, _fp, _fp,
                                     _vp, _fp, _vp, _fp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "coda_block_rowscale_fp8": (_i32, [_vp, _fp, _vp, _fp, _vp, _fp, _vp, _vp, _fp, _f32, _vp, _fp, _fp, _fp, _vp, _fp,
                                       _vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "coda_amax": (_i32, [_vp, _i64, _i32, _fp, _vp]),
    "coda_quantize_e4m3": (_i32, [_vp, _i64, _i32, _fp, _vp, _fp, _vp]),
    "coda_selftest_wait_timeout": (_i32, [_i64, _vp]),
    "coda_get_device_status": (_i32, []),
}

_lock = threading.Lock()
_lib = None


class CodaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libcoda_gb300.so (compiling it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


def _check(status: int):
    if status != CODA_OK:
        raise CodaError(status, load_library().coda_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return CODA_F32
    if t.dtype == torch.bfloat16:
        return CODA_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return CODA_E4M3
    raise TypeError(f"unsupported operand dtype {t.dtype}")


def _out_dtype(code: int) -> torch.dtype:
    return torch.float32 if code == CODA_F32 else torch.bfloat16


_F32 = (torch.float32,)
_BYTE = (torch.uint8, torch.float8_e4m3fn)


def _want(t: Optional[torch.Tensor], name: str, shape=None, dtypes=None, numel=None, nbytes=None):
    """Checks that a given tensor matches the sizes the call passes to the
    library (the kernels read and write exactly those extents): its shape,
    its dtype, at least `numel` elements (scalars) or `nbytes` bytes
    (workspaces).  None passes (a NULL argument, which the library checks)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {' or '.join(str(d) for d in dtypes)}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected at least {numel}")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, expected at least {nbytes}")


def _operand_dtypes(code: int):
    return {CODA_F32: (torch.float32,), CODA_BF16: (torch.bfloat16,), CODA_E4M3: _BYTE}[code]


def _want_scalars(**scalars):
    """Per-tensor scales and amax outputs: one fp32 each."""
    for name, t in scalars.items():
        _want(t, name, dtypes=_F32, numel=1)


def _want_block(X, W1t, R, Wb, Wb2, H, P, out, r_out, workspace, n_out, code, out_name, wb_name):
    """The tensors of a one-launch block: X [M, K], W1t [N, K], R and h [M, N],
    the consumer's weights [n_out, N], P [M, T], the output [M, n_out]."""
    M, K = X.shape
    N = W1t.shape[0]
    ops, od = _operand_dtypes(code), (_out_dtype(code),)
    _want(W1t, "W1t", (N, K), ops)
    _want(R, "R", (M, N), od)
    _want(Wb, wb_name, (n_out, N), ops)
    _want(Wb2, "Wut", (n_out, N), ops)
    _want(H, "H", (M, N), od)
    _want(P, "P", (M, coda_partial_cols(N)), _F32)
    _want(out, out_name, (M, n_out), od)
    _want(r_out, "r_out", (M,), _F32)
    _want(workspace, "workspace", nbytes=coda_block_workspace_bytes(M))


def _want_fp8_block(A, amax_a, Aq, scale_a, W1t, scale_w1, R, Wb, scale_wb, Wb2, scale_wb2, H, P, r_out, amax_h, Hq,
                    scale_h, out, amax_out, workspace, M, N, K, n_out, out_name, wb_name):
    """The tensors of an FP8 one-launch block (e4m3 operands as uint8 bytes)."""
    bf = (torch.bfloat16,)
    _want(A, "A", (M, K), bf)
    _want(Aq, "Aq", (M, K), _BYTE)
    _want(W1t, "W1t", (N, K), _BYTE)
    _want(R, "R", (M, N), bf)
    _want(Wb, wb_name, (n_out, N), _BYTE)
    _want(Wb2, "Wut", (n_out, N), _BYTE)
    _want(H, "H", (M, N), bf)
    _want(P, "P", (M, coda_partial_cols(N)), _F32)
    _want(r_out, "r_out", (M,), _F32)
    _want(Hq, "Hq", (M, N), _BYTE)
    _want(out, out_name, (M, n_out), bf)
    _want_scalars(amax_a=amax_a, scale_a=scale_a, scale_w1=scale_w1, scale_w=scale_wb, scale_wu=scale_wb2,
                  amax_h=amax_h, scale_h=scale_h, amax_act=amax_out)
    _want(workspace, "workspace", nbytes=coda_block_fp8_workspace_bytes(M))


def _dev(t: Optional[torch.Tensor], name: str):
    """Device pointer of a contiguous CUDA tensor on the current device (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.index is not None and t.device.index != torch.cuda.current_device():
        # the library launches on the current device
        raise ValueError(f"{name} is on {t.device} but the current device is cuda:{torch.cuda.current_device()}")
    return t.data_ptr() or None


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def coda_partial_cols(N: int) -> int:
    return int(load_library().coda_partial_cols(N))


def coda_fold_gamma(Wt: torch.Tensor, gamma: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None):
    """W'^T = W^T diag(gamma): out[n, k] = Wt[n, k] * gamma[k]."""
    lib = load_library()
    N_out, K = Wt.shape
    out = torch.empty_like(Wt) if out is None else out
    _want(Wt, "Wt", dtypes=(torch.float32, torch.bfloat16))
    _want(gamma, "gamma", (K,), _F32)
    _want(out, "out", (N_out, K), (Wt.dtype,))
    _check(lib.coda_fold_gamma(_dev(Wt, "Wt"), _dev(gamma, "gamma"), _dev(out, "out"), N_out, K, _dtype_code(Wt),
                               _stream(Wt, stream)))
    return out


def coda_gemm_residual_partial_rms(X, W1t, R, H=None, P=None, *, scale_x=None, scale_w=None, amax_h=None,
                                   stream=None):
    """h = R + X W1 (W1t = W1^T) and P[i, g] = sum of h[i, j]^2 over 128-column group g.  Returns (h, P)."""
    lib = load_library()
    M, K = X.shape
    N = W1t.shape[0]
    code = _dtype_code(X)
    if H is None:
        H = torch.empty(M, N, dtype=_out_dtype(code), device=X.device)
    if P is None:
        P = torch.empty(M, max(coda_partial_cols(N), 0), dtype=torch.float32, device=X.device)
    ops, od = _operand_dtypes(code), (_out_dtype(code),)
    _want(W1t, "W1t", (N, K), ops)
    _want(R, "R", (M, N), od)
    _want(H, "H", (M, N), od)
    _want(P, "P", (M, coda_partial_cols(N)), _F32)
    _want_scalars(scale_x=scale_x, scale_w=scale_w, amax_h=amax_h)
    _check(lib.coda_gemm_residual_partial_rms(_dev(X, "X"), _dev(W1t, "W1t"), _dev(R, "R"), _dev(H, "H"),
                                              _dev(P, "P"), M, N, K, code, _dev(scale_x, "scale_x"),
                                              _dev(scale_w, "scale_w"), _dev(amax_h, "amax_h"), _stream(X, stream)))
    return H, P


def coda_rms_reduce(P, N: int, eps: float, r=None, stream=None):
    """r[i] = 1 / sqrt(sum_g P[i, g] / N + eps)."""
    lib = load_library()
    M = P.shape[0]
    if r is None:
        r = torch.empty(M, dtype=torch.float32, device=P.device)
    _want(P, "P", (M, coda_partial_cols(N)), _F32)
    _want(r, "r", (M,), _F32)
    _check(lib.coda_rms_reduce(_dev(P, "P"), M, N, float(eps), _dev(r, "r"), _stream(P, stream)))
    return r


def coda_gemm_rowscale(H, W2t, r, Z=None, *, scale_h=None, scale_w=None, stream=None):
    """Z = diag(r) H W2 (W2t = W2^T, gamma already folded in)."""
    lib = load_library()
    M, K = H.shape
    N2 = W2t.shape[0]
    code = _dtype_code(H)
    if Z is None:
        Z = torch.empty(M, N2, dtype=_out_dtype(code), device=H.device)
    _want(W2t, "W2t", (N2, K), _operand_dtypes(code))
    _want(r, "r", (M,), _F32)
    _want(Z, "Z", (M, N2), (_out_dtype(code),))
    _want_scalars(scale_h=scale_h, scale_w=scale_w)
    _check(lib.coda_gemm_rowscale(_dev(H, "H"), _dev(W2t, "W2t"), _dev(r, "r"), _dev(Z, "Z"), M, N2, K, code,
                                  _dev(scale_h, "scale_h"), _dev(scale_w, "scale_w"), _stream(H, stream)))
    return Z


def coda_gemm_swiglu(H, Wgt, Wut, r=None, Act=None, *, scale_h=None, scale_wg=None, scale_wu=None, amax_act=None,
                     stream=None):
    """Act = silu(diag(r) H Wg) * (diag(r) H Wu)."""
    lib = load_library()
    M, K = H.shape
    I = Wgt.shape[0]
    code = _dtype_code(H)
    if Act is None:
        Act = torch.empty(M, I, dtype=_out_dtype(code), device=H.device)
    _want(Wgt, "Wgt", (I, K), _operand_dtypes(code))
    _want(Wut, "Wut", (I, K), _operand_dtypes(code))
    _want(r, "r", (M,), _F32)
    _want(Act, "Act", (M, I), (_out_dtype(code),))
    _want_scalars(scale_h=scale_h, scale_wg=scale_wg, scale_wu=scale_wu, amax_act=amax_act)
    _check(lib.coda_gemm_swiglu(_dev(H, "H"), _dev(Wgt, "Wgt"), _dev(Wut, "Wut"), _dev(r, "r"), _dev(Act, "Act"),
                                M, I, K, code, _dev(scale_h, "scale_h"), _dev(scale_wg, "scale_wg"),
                                _dev(scale_wu, "scale_wu"), _dev(amax_act, "amax_act"), _stream(H, stream)))
    return Act


def coda_gemm_rowscale_fused_rms(H, W2t, P, eps: float, Z=None, r_out=None, *, scale_h=None, scale_w=None,
                                 stream=None):
    """Z = diag(r) H W2 with r reduced from the partials P inside the epilogue."""
    lib = load_library()
    M, K = H.shape
    N2 = W2t.shape[0]
    code = _dtype_code(H)
    if Z is None:
        Z = torch.empty(M, N2, dtype=_out_dtype(code), device=H.device)
    _want(W2t, "W2t", (N2, K), _operand_dtypes(code))
    _want(P, "P", (M, coda_partial_cols(K)), _F32)
    _want(r_out, "r_out", (M,), _F32)
    _want(Z, "Z", (M, N2), (_out_dtype(code),))
    _want_scalars(scale_h=scale_h, scale_w=scale_w)
    _check(lib.coda_gemm_rowscale_fused_rms(_dev(H, "H"), _dev(W2t, "W2t"), _dev(P, "P"), float(eps),
                                            _dev(r_out, "r_out"), _dev(Z, "Z"), M, N2, K, code,
                                            _dev(scale_h, "scale_h"), _dev(scale_w, "scale_w"), _stream(H, stream)))
    return Z


def coda_gemm_swiglu_fused_rms(H, Wgt, Wut, P, eps: float, Act=None, r_out=None, *, scale_h=None, scale_wg=None,
                               scale_wu=None, amax_act=None, stream=None):
    """Act = silu(diag(r) H Wg) * (diag(r) H Wu) with r reduced from P inside the epilogue."""
    lib = load_library()
    M, K = H.shape
    I = Wgt.shape[0]
    code = _dtype_code(H)
    if Act is None:
        Act = torch.empty(M, I, dtype=_out_dtype(code), device=H.device)
    _want(Wgt, "Wgt", (I, K), _operand_dtypes(code))
    _want(Wut, "Wut", (I, K), _operand_dtypes(code))
    _want(P, "P", (M, coda_partial_cols(K)), _F32)
    _want(r_out, "r_out", (M,), _F32)
    _want(Act, "Act", (M, I), (_out_dtype(code),))
    _want_scalars(scale_h=scale_h, scale_wg=scale_wg, scale_wu=scale_wu, amax_act=amax_act)
    _check(lib.coda_gemm_swiglu_fused_rms(_dev(H, "H"), _dev(Wgt, "Wgt"), _dev(Wut, "Wut"), _dev(P, "P"),
                                          float(eps), _dev(r_out, "r_out"), _dev(Act, "Act"), M, I, K, code,
                                          _dev(scale_h, "scale_h"), _dev(scale_wg, "scale_wg"),
                                          _dev(scale_wu, "scale_wu"), _dev(amax_act, "amax_act"),
                                          _stream(H, stream)))
    return Act


def coda_gemm_rowscale_rope(H, W2t, head_dim: int, rope_cols: int, base: float, *, seq_len: int = 0, positions=None,
                            r=None, P=None, eps: float = 0.0, r_out=None, Z=None, scale_h=None, scale_w=None,
                            stream=None):
    """Z = RoPE(diag(r) H W2) on the first rope_cols columns; r given, or reduced from P inside the epilogue.
    Positions: ``positions`` [M] int32, else row mod ``seq_len``."""
    lib = load_library()
    M, K = H.shape
    N2 = W2t.shape[0]
    code = _dtype_code(H)
    if Z is None:
        Z = torch.empty(M, N2, dtype=_out_dtype(code), device=H.device)
    _want(W2t, "W2t", (N2, K), _operand_dtypes(code))
    _want(r, "r", (M,), _F32)
    _want(P, "P", (M, coda_partial_cols(K)), _F32)
    _want(r_out, "r_out", (M,), _F32)
    _want(Z, "Z", (M, N2), (_out_dtype(code),))
    _want(positions, "positions", (M,), (torch.int32,))
    _want_scalars(scale_h=scale_h, scale_w=scale_w)
    _check(lib.coda_gemm_rowscale_rope(_dev(H, "H"), _dev(W2t, "W2t"), _dev(r, "r"), _dev(P, "P"), float(eps),
                                       _dev(r_out, "r_out"), _dev(Z, "Z"), M, N2, K, code, _dev(scale_h, "scale_h"),
                                       _dev(scale_w, "scale_w"), head_dim, rope_cols, float(base), seq_len,
                                       _dev(positions, "positions"), _stream(H, stream)))
    return Z


def coda_gemm(A, B, *, a_mn: bool = False, b_mn: bool = False, row_scale=None, col_scale=None, D=None,
              stream=None):
    """D = diag(row_scale) opA(A) opB(B)^T diag(col_scale), with opA(A) = A [M, K] or A^T for A [K, M]
    (a_mn) and opB(B) = B [N, K] or B^T for B [K, N] (b_mn)."""
    lib = load_library()
    M, K = (A.shape[1], A.shape[0]) if a_mn else (A.shape[0], A.shape[1])
    N = B.shape[1] if b_mn else B.shape[0]
    if (B.shape[0] if b_mn else B.shape[1]) != K:
        raise ValueError("inner dimensions differ")
    code = _dtype_code(A)
    if D is None:
        D = torch.empty(M, N, dtype=_out_dtype(code), device=A.device)
    _want(B, "B", dtypes=(A.dtype,))
    _want(D, "D", (M, N), (_out_dtype(code),))
    _want(row_scale, "row_scale", (M,), _F32)
    _want(col_scale, "col_scale", (N,), _F32)
    _check(lib.coda_gemm(_dev(A, "A"), int(a_mn), _dev(B, "B"), int(b_mn), _dev(D, "D"), M, N, K, code,
                         _dev(row_scale, "row_scale"), _dev(col_scale, "col_scale"), _stream(A, stream)))
    return D


def coda_gemm_grad_norm(dOut, Wt, H, gamma, dY=None, S=None, stream=None):
    """dY = dOut . Wt (Wt [K, N] as the forward stores it) and S = per-group sums of gamma dY H.  Returns (dY, S)."""
    lib = load_library()
    M, K = dOut.shape
    N = Wt.shape[1]
    if dY is None:
        dY = torch.empty(M, N, dtype=torch.bfloat16, device=dOut.device)
    if S is None:
        S = torch.empty(M, coda_partial_cols(N), dtype=torch.float32, device=dOut.device)
    bf = (torch.bfloat16,)
    _want(dOut, "dOut", dtypes=bf)
    _want(Wt, "Wt", (K, N), bf)
    _want(H, "H", (M, N), bf)
    _want(gamma, "gamma", (N,), _F32)
    _want(dY, "dY", (M, N), bf)
    _want(S, "S", (M, coda_partial_cols(N)), _F32)
    _check(lib.coda_gemm_grad_norm(_dev(dOut, "dOut"), _dev(Wt, "Wt"), _dev(H, "H"), _dev(gamma, "gamma"),
                                   _dev(dY, "dY"), _dev(S, "S"), M, N, K, _dtype_code(dOut), _stream(dOut, stream)))
    return dY, S


def coda_rmsnorm_backward(dY, H, r, gamma, S, dH_in=None, dH=None, Yt=None, dgamma=None, workspace=None,
                          stream=None):
    """dH = r gamma dY - c H (+ dH_in), Yt = r H, dgamma.  Returns (dH, Yt, dgamma)."""
    lib = load_library()
    M, N = dY.shape
    dH = torch.empty_like(dY) if dH is None else dH
    Yt = torch.empty_like(dY) if Yt is None else Yt
    if dgamma is None:
        dgamma = torch.empty(N, dtype=torch.float32, device=dY.device)
    if workspace is None:
        n = lib.coda_rmsnorm_backward_workspace_bytes(M, N)
        workspace = torch.empty(max(n // 4, 1), dtype=torch.float32, device=dY.device)
    bf = (torch.bfloat16,)
    for t, name in ((dY, "dY"), (H, "H"), (dH_in, "dH_in"), (dH, "dH"), (Yt, "Yt")):
        _want(t, name, (M, N), bf)
    _want(r, "r", (M,), _F32)
    _want(gamma, "gamma", (N,), _F32)
    _want(S, "S", (M, coda_partial_cols(N)), _F32)
    _want(dgamma, "dgamma", (N,), _F32)
    _want(workspace, "workspace", nbytes=lib.coda_rmsnorm_backward_workspace_bytes(M, N))
    _check(lib.coda_rmsnorm_backward(_dev(dY, "dY"), _dev(H, "H"), _dev(r, "r"), _dev(gamma, "gamma"), _dev(S, "S"),
                                     _dev(dH_in, "dH_in"), _dev(dH, "dH"), _dev(Yt, "Yt"), _dev(dgamma, "dgamma"),
                                     _dev(workspace, "workspace"), M, N, _stream(dY, stream)))
    return dH, Yt, dgamma


def coda_gemm_swiglu_save(H, Wgt, Wut, *, r=None, P=None, eps: float = 0.0, r_out=None, Act=None, GU=None,
                          stream=None):
    """SwiGLU GEMM that also returns the pre-activations G || U [M, 2I].  Returns (Act, GU)."""
    lib = load_library()
    M, K = H.shape
    I = Wgt.shape[0]
    if Act is None:
        Act = torch.empty(M, I, dtype=torch.bfloat16, device=H.device)
    if GU is None:
        GU = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=H.device)
    bf = (torch.bfloat16,)
    _want(H, "H", dtypes=bf)
    _want(Wgt, "Wgt", (I, K), bf)
    _want(Wut, "Wut", (I, K), bf)
    _want(r, "r", (M,), _F32)
    _want(P, "P", (M, coda_partial_cols(K)), _F32)
    _want(r_out, "r_out", (M,), _F32)
    _want(Act, "Act", (M, I), bf)
    _want(GU, "GU", (M, 2 * I), bf)
    _check(lib.coda_gemm_swiglu_save(_dev(H, "H"), _dev(Wgt, "Wgt"), _dev(Wut, "Wut"), _dev(r, "r"), _dev(P, "P"),
                                     float(eps), _dev(r_out, "r_out"), _dev(Act, "Act"), _dev(GU, "GU"), M, I, K,
                                     _dtype_code(H), _stream(H, stream)))
    return Act, GU


def coda_gemm_swiglu_backward(dOut, Wt, GU, dGU=None, stream=None):
    """dG || dU from dAct = dOut . Wt (Wt [K, I]) and the saved G || U [M, 2I]."""
    lib = load_library()
    M, K = dOut.shape
    I = Wt.shape[1]
    if dGU is None:
        dGU = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dOut.device)
    bf = (torch.bfloat16,)
    _want(dOut, "dOut", dtypes=bf)
    _want(Wt, "Wt", (K, I), bf)
    _want(GU, "GU", (M, 2 * I), bf)
    _want(dGU, "dGU", (M, 2 * I), bf)
    _check(lib.coda_gemm_swiglu_backward(_dev(dOut, "dOut"), _dev(Wt, "Wt"), _dev(GU, "GU"), _dev(dGU, "dGU"), M, I,
                                         K, _dtype_code(dOut), _stream(dOut, stream)))
    return dGU


def coda_block_workspace_bytes(M: int) -> int:
    return int(load_library().coda_block_workspace_bytes(M))


def block_workspace(M: int, device) -> torch.Tensor:
    """A zeroed workspace for the one-launch blocks (calls leave it zeroed)."""
    n = coda_block_workspace_bytes(M)
    return torch.zeros((n + 3) // 4, dtype=torch.int32, device=device)


def _block_outputs(X, R, N, n_out, H, P, out, code):
    M = X.shape[0]
    if H is None:
        H = torch.empty(M, N, dtype=_out_dtype(code), device=X.device)
    if P is None:
        P = torch.empty(M, max(coda_partial_cols(N), 0), dtype=torch.float32, device=X.device)
    if out is None:
        out = torch.empty(M, n_out, dtype=_out_dtype(code), device=X.device)
    return H, P, out


def coda_block_rowscale(X, W1t, R, W2t, eps: float, workspace, H=None, P=None, Z=None, r_out=None, stream=None):
    """One launch: h = R + X W1, P, r, Z = diag(r) h W2 (W2t gamma-folded).  Returns (h, P, Z)."""
    lib = load_library()
    M, K = X.shape
    N, N2 = W1t.shape[0], W2t.shape[0]
    code = _dtype_code(X)
    H, P, Z = _block_outputs(X, R, N, N2, H, P, Z, code)
    _want_block(X, W1t, R, W2t, None, H, P, Z, r_out, workspace, N2, code, "Z", "W2t")
    _check(lib.coda_block_rowscale(_dev(X, "X"), _dev(W1t, "W1t"), _dev(R, "R"), _dev(W2t, "W2t"), float(eps),
                                   _dev(H, "H"), _dev(P, "P"), _dev(r_out, "r_out"), _dev(Z, "Z"), M, N, K, N2, code,
                                   _dev(workspace, "workspace"), _stream(X, stream)))
    return H, P, Z


def coda_block_rowscale_rope(X, W1t, R, W2t, eps: float, workspace, head_dim: int, rope_cols: int, base: float, *,
                             seq_len: int = 0, positions=None, H=None, P=None, Z=None, r_out=None, stream=None):
    """One launch: h = R + X W1, P, r, Z = RoPE(diag(r) h W2) on the first rope_cols columns.
    Positions: ``positions`` [M] int32, else row mod ``seq_len``.  Returns (h, P, Z)."""
    lib = load_library()
    M, K = X.shape
    N, N2 = W1t.shape[0], W2t.shape[0]
    code = _dtype_code(X)
    H, P, Z = _block_outputs(X, R, N, N2, H, P, Z, code)
    _want_block(X, W1t, R, W2t, None, H, P, Z, r_out, workspace, N2, code, "Z", "W2t")
    _want(positions, "positions", (M,), (torch.int32,))
    _check(lib.coda_block_rowscale_rope(_dev(X, "X"), _dev(W1t, "W1t"), _dev(R, "R"), _dev(W2t, "W2t"), float(eps),
                                        _dev(H, "H"), _dev(P, "P"), _dev(r_out, "r_out"), _dev(Z, "Z"), M, N, K, N2,
                                        code, head_dim, rope_cols, float(base), seq_len, _dev(positions, "positions"),
                                        _dev(workspace, "workspace"), _stream(X, stream)))
    return H, P, Z


def coda_block_swiglu(X, W1t, R, Wgt, Wut, eps: float, workspace, H=None, P=None, Act=None, r_out=None,
                      stream=None):
    """One launch: h = R + X W1, P, r, Act = silu(r h Wg) * (r h Wu).  Returns (h, P, Act)."""
    lib = load_library()
    M, K = X.shape
    N, I = W1t.shape[0], Wgt.shape[0]
    code = _dtype_code(X)
    H, P, Act = _block_outputs(X, R, N, I, H, P, Act, code)
    _want_block(X, W1t, R, Wgt, Wut, H, P, Act, r_out, workspace, I, code, "Act", "Wgt")
    _check(lib.coda_block_swiglu(_dev(X, "X"), _dev(W1t, "W1t"), _dev(R, "R"), _dev(Wgt, "Wgt"), _dev(Wut, "Wut"),
                                 float(eps), _dev(H, "H"), _dev(P, "P"), _dev(r_out, "r_out"), _dev(Act, "Act"), M, N,
                                 K, I, code, _dev(workspace, "workspace"), _stream(X, stream)))
    return H, P, Act


def coda_block_swiglu_noalloc(X, W1t, R, Wgt, Wut, eps: float, H=None, P=None, Act=None, r_out=None, stream=None):
    """coda_block_swiglu without a workspace, for callers that cannot allocate
    device memory (the library keeps the counters itself; M <= 131072; calls
    must not overlap on the GPU).  Returns (h, P, Act)."""
    lib = load_library()
    M, K = X.shape
    N, I = W1t.shape[0], Wgt.shape[0]
    code = _dtype_code(X)
    H, P, Act = _block_outputs(X, R, N, I, H, P, Act, code)
    _want_block(X, W1t, R, Wgt, Wut, H, P, Act, r_out, None, I, code, "Act", "Wgt")
    _check(lib.coda_block_swiglu_noalloc(_dev(X, "X"), _dev(W1t, "W1t"), _dev(R, "R"), _dev(Wgt, "Wgt"),
                                         _dev(Wut, "Wut"), float(eps), _dev(H, "H"), _dev(P, "P"), _dev(r_out, "r_out"),
                                         _dev(Act, "Act"), M, N, K, I, code, _stream(X, stream)))
    return H, P, Act


def coda_block_fp8_workspace_bytes(M: int) -> int:
    return int(load_library().coda_block_fp8_workspace_bytes(M))


def block_fp8_workspace(M: int, device) -> torch.Tensor:
    """A zeroed workspace for the FP8 one-launch blocks (calls leave it zeroed)."""
    n = coda_block_fp8_workspace_bytes(M)
    return torch.zeros((n + 3) // 4, dtype=torch.int32, device=device)


def _fp8_block_buffers(M, N, K, n_out, dev, A, Aq, scale_a, H, P, amax_h, Hq, scale_h, out):
    f32, bf, u8 = torch.float32, torch.bfloat16, torch.uint8
    e = lambda *shape, dt: torch.empty(*shape, dtype=dt, device=dev)  # noqa: E731
    if A is not None:  # the launch quantises A: it writes Aq and scale_a
        Aq = e(M, K, dt=u8) if Aq is None else Aq
        scale_a = e(1, dt=f32) if scale_a is None else scale_a
    elif Aq is None or scale_a is None:
        raise ValueError("without A, Aq and scale_a (the e4m3 operand and its scale) must be given")
    return (Aq, scale_a, e(M, N, dt=bf) if H is None else H,
            e(M, max(coda_partial_cols(N), 0), dt=f32) if P is None else P, e(1, dt=f32) if amax_h is None else amax_h,
            e(M, N, dt=u8) if Hq is None else Hq, e(1, dt=f32) if scale_h is None else scale_h,
            e(M, n_out, dt=bf) if out is None else out)


def coda_block_swiglu_fp8(A, amax_a, W1t, scale_w1, R, Wgt, scale_wg, Wut, scale_wu, eps: float, workspace,
                          Aq=None, scale_a=None, H=None, P=None, r_out=None, amax_h=None, Hq=None, scale_h=None,
                          Act=None, amax_act=None, M=None, stream=None):
    """FP8 one-launch block: [Aq = e4m3(A)], h = R + Aq W1, Hq = e4m3(h), Act =
    silu(r Hq Wg) * (r Hq Wu).  A (bf16) may be None when Aq and scale_a are
    given.  Returns a dict of the outputs (Aq, scale_a, h, P, amax_h, Hq,
    scale_h, act, amax_act)."""
    lib = load_library()
    src = A if A is not None else Aq
    M, K = src.shape
    N, I = W1t.shape[0], Wgt.shape[0]
    dev = src.device
    Aq, scale_a, H, P, amax_h, Hq, scale_h, Act = _fp8_block_buffers(M, N, K, I, dev, A, Aq, scale_a, H, P, amax_h,
                                                                      Hq, scale_h, Act)
    _want_fp8_block(A, amax_a, Aq, scale_a, W1t, scale_w1, R, Wgt, scale_wg, Wut, scale_wu, H, P, r_out, amax_h,
                    Hq, scale_h, Act, amax_act, workspace, M, N, K, I, "Act", "Wgt")
    _check(lib.coda_block_swiglu_fp8(_dev(A, "A"), _dev(amax_a, "amax_a"), _dev(Aq, "Aq"), _dev(scale_a, "scale_a"),
                                     _dev(W1t, "W1t"), _dev(scale_w1, "scale_w1"), _dev(R, "R"), _dev(Wgt, "Wgt"),
                                     _dev(scale_wg, "scale_wg"), _dev(Wut, "Wut"), _dev(scale_wu, "scale_wu"),
                                     float(eps), _dev(H, "H"), _dev(P, "P"), _dev(r_out, "r_out"),
                                     _dev(amax_h, "amax_h"), _dev(Hq, "Hq"), _dev(scale_h, "scale_h"), _dev(Act, "Act"),
                                     _dev(amax_act, "amax_act"), M, N, K, I, _dev(workspace, "workspace"),
                                     _stream(src, stream)))
    return {"Aq": Aq, "scale_a": scale_a, "h": H, "P": P, "amax_h": amax_h, "Hq": Hq, "scale_h": scale_h,
            "act": Act, "amax_act": amax_act}


def coda_block_rowscale_fp8(A, amax_a, W1t, scale_w1, R, W2t, scale_w2, eps: float, workspace, Aq=None,
                            scale_a=None, H=None, P=None, r_out=None, amax_h=None, Hq=None, scale_h=None, Z=None,
                            stream=None):
    """FP8 one-launch block: [Aq = e4m3(A)], h = R + Aq W1, Hq = e4m3(h), Z =
    diag(r) Hq W2.  Returns a dict of the outputs (Aq, scale_a, h, P, amax_h,
    Hq, scale_h, Z)."""
    lib = load_library()
    src = A if A is not None else Aq
    M, K = src.shape
    N, N2 = W1t.shape[0], W2t.shape[0]
    dev = src.device
    Aq, scale_a, H, P, amax_h, Hq, scale_h, Z = _fp8_block_buffers(M, N, K, N2, dev, A, Aq, scale_a, H, P, amax_h,
                                                                    Hq, scale_h, Z)
    _want_fp8_block(A, amax_a, Aq, scale_a, W1t, scale_w1, R, W2t, scale_w2, None, None, H, P, r_out, amax_h,
                    Hq, scale_h, Z, None, workspace, M, N, K, N2, "Z", "W2t")
    _check(lib.coda_block_rowscale_fp8(_dev(A, "A"), _dev(amax_a, "amax_a"), _dev(Aq, "Aq"), _dev(scale_a, "scale_a"),
                                       _dev(W1t, "W1t"), _dev(scale_w1, "scale_w1"), _dev(R, "R"), _dev(W2t, "W2t"),
                                       _dev(scale_w2, "scale_w2"), float(eps), _dev(H, "H"), _dev(P, "P"),
                                       _dev(r_out, "r_out"), _dev(amax_h, "amax_h"), _dev(Hq, "Hq"),
                                       _dev(scale_h, "scale_h"), _dev(Z, "Z"), M, N, K, N2,
                                       _dev(workspace, "workspace"), _stream(src, stream)))
    return {"Aq": Aq, "scale_a": scale_a, "h": H, "P": P, "amax_h": amax_h, "Hq": Hq, "scale_h": scale_h, "Z": Z}


def coda_amax(x, amax=None, stream=None):
    """amax = max |x| (fp32 scalar tensor)."""
    lib = load_library()
    if amax is None:
        amax = torch.empty(1, dtype=torch.float32, device=x.device)
    _want(x, "x", dtypes=(torch.float32, torch.bfloat16))
    _want(amax, "amax", dtypes=_F32, numel=1)
    _check(lib.coda_amax(_dev(x, "x"), x.numel(), _dtype_code(x), _dev(amax, "amax"), _stream(x, stream)))
    return amax


def coda_quantize_e4m3(x, amax, q=None, scale=None, stream=None):
    """q = e4m3(x / s) with s = amax / 448; returns (q as uint8, s)."""
    lib = load_library()
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(1, dtype=torch.float32, device=x.device)
    _want(x, "x", dtypes=(torch.float32, torch.bfloat16))
    _want(amax, "amax", dtypes=_F32, numel=1)
    _want(q, "q", dtypes=_BYTE, numel=x.numel())
    _want(scale, "scale", dtypes=_F32, numel=1)
    _check(lib.coda_quantize_e4m3(_dev(x, "x"), x.numel(), _dtype_code(x), _dev(amax, "amax"), _dev(q, "q"),
                                  _dev(scale, "scale"), _stream(x, stream)))
    return q, scale


def coda_selftest_wait_timeout(timeout_ns: int, stream=None):
    """Enqueue the failure-path self-test: a bounded wait on an mbarrier that
    nothing signals gives up after timeout_ns and raises the timeout bit, so
    the next coda_get_device_status() raises CodaError(CODA_ERR_TIMEOUT)."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream()
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check(lib.coda_selftest_wait_timeout(int(timeout_ns), s))


def coda_get_device_status() -> int:
    """Synchronise and read/clear the device status word; raises CodaError on a timeout."""
    st = load_library().coda_get_device_status()
    _check(st)
    return st
