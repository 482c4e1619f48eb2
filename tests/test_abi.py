"""The C ABI on the host, with no GPU: the library loads, exports every
symbol include/coda.h declares, and rejects bad arguments before anything
is enqueued (fake, never-dereferenced addresses are enough for that)."""
import ctypes
import os
import re

import pytest

import gemm_epilogue_fusion_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coda.h")


@pytest.fixture(scope="module")
def lib():
    return g.load_library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CODA_API\s+[\w\s\*]+?\b(coda_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("coda_gemm_residual_partial_rms", "coda_rms_reduce", "coda_gemm_rowscale", "coda_gemm_swiglu",
              "coda_fold_gamma"):
        assert n in names
    assert set(names) == set(g.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert lib.coda_version() >= 100


def test_partial_cols_and_status_strings(lib):
    assert [lib.coda_partial_cols(n) for n in (1, 128, 129, 2048, 4096, 0)] == [1, 1, 2, 16, 32, -1]
    assert lib.coda_status_string(4) == b"CODA_ERR_TIMEOUT"


A = 0x7F0000000000  # fake 16-byte-aligned device addresses, never dereferenced
MB = 1 << 20


def _rpr(lib, X=A, W=A + 64 * MB, R=A + 128 * MB, H=A + 192 * MB, P=A + 256 * MB, M=256, N=512, K=512, dt=1,
         sx=None, sw=None, amax=None):
    return lib.coda_gemm_residual_partial_rms(X, W, R, H, P, M, N, K, dt, sx, sw, amax, None)


def test_rejects_null_and_misaligned(lib):
    assert _rpr(lib, X=None) == g.CODA_ERR_INVALID_ARG
    assert b"X is NULL" in lib.coda_last_error()
    assert _rpr(lib, H=A + 192 * MB + 8) == g.CODA_ERR_INVALID_ARG
    assert b"16-byte" in lib.coda_last_error()


def test_rejects_bad_shapes(lib):
    assert _rpr(lib, K=0) == g.CODA_ERR_INVALID_ARG
    assert _rpr(lib, N=-4) == g.CODA_ERR_INVALID_ARG
    assert _rpr(lib, K=12) == g.CODA_ERR_INVALID_ARG          # bf16 rows of 24 bytes
    assert _rpr(lib, N=100) == g.CODA_ERR_INVALID_ARG         # bf16 rows of 200 bytes
    assert _rpr(lib, K=8, dt=2, sx=A + 300 * MB, sw=A + 300 * MB + 4) == g.CODA_ERR_INVALID_ARG  # e4m3: K % 16
    assert _rpr(lib, M=1 << 31) == g.CODA_ERR_INVALID_ARG
    assert _rpr(lib, dt=7) == g.CODA_ERR_INVALID_ARG


def test_rejects_sizes_beyond_32_bit_tile_indices(lib):
    # plausible-looking but absurd sizes are refused before anything is enqueued
    big = (1 << 31) - 8
    assert _rpr(lib, M=big, N=big, K=8) == g.CODA_ERR_INVALID_ARG
    assert b"2^60" in lib.coda_last_error() or b"tile" in lib.coda_last_error()
    assert _rpr(lib, M=1 << 30, N=1 << 20, K=8) == g.CODA_ERR_INVALID_ARG
    assert b"tile" in lib.coda_last_error()


def test_every_call_bounds_its_extents(lib):
    # sizes whose byte extents would overflow int64 are refused by every call
    # that takes them, before anything is enqueued (the addresses are fake)
    big = (1 << 31) - 8
    B, D = A + 64 * MB, A + 128 * MB
    assert lib.coda_gemm(A, 0, B, 1, D, big, big, 8, 1, None, None, None) == g.CODA_ERR_INVALID_ARG
    assert b"2^60" in lib.coda_last_error()
    assert lib.coda_gemm(A, 1, B, 1, D, 1 << 30, 1 << 20, 8, 1, None, None, None) == g.CODA_ERR_INVALID_ARG
    assert b"tile" in lib.coda_last_error()
    assert lib.coda_fold_gamma(A, B, D, big, big - 7, 1, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_rmsnorm_backward(A, B, A + 128 * MB, A + 129 * MB, A + 130 * MB, None, A + 192 * MB,
                                     A + 256 * MB, A + 320 * MB, A + 321 * MB, big, big - 7, None) \
        == g.CODA_ERR_INVALID_ARG
    assert lib.coda_amax(A, 1 << 61, 1, B, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_quantize_e4m3(A, 1 << 61, 1, B, D, B + 4, None) == g.CODA_ERR_INVALID_ARG


def test_rejects_overlapping_outputs(lib):
    assert _rpr(lib, H=A + 128 * MB) == g.CODA_ERR_INVALID_ARG   # h over R
    assert b"overlaps input R" in lib.coda_last_error()
    assert _rpr(lib, P=A + 192 * MB + 4096) == g.CODA_ERR_INVALID_ARG  # P inside h
    assert lib.coda_gemm_rowscale(A, A + MB, A + 2 * MB, A + 100, 16, 64, 64, 1, None, None, None) \
        == g.CODA_ERR_INVALID_ARG


def test_fp8_scale_rules(lib):
    # scales are required for e4m3 and forbidden otherwise
    assert _rpr(lib, dt=2) == g.CODA_ERR_INVALID_ARG
    assert _rpr(lib, dt=1, sx=A + 300 * MB, sw=A + 300 * MB + 4) == g.CODA_ERR_INVALID_ARG


def test_m_zero_enqueues_nothing(lib):
    # no amax output: nothing to do, no CUDA call is made
    assert _rpr(lib, M=0) == g.CODA_OK
    assert lib.coda_rms_reduce(A, 0, 512, 1e-5, A + MB, None) == g.CODA_OK
    assert lib.coda_gemm_rowscale(A, A + MB, A + 2 * MB, A + 3 * MB, 0, 64, 64, 1, None, None, None) == g.CODA_OK


def test_rms_reduce_and_helpers_validate(lib):
    assert lib.coda_rms_reduce(A, 16, 512, -1.0, A + MB, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_rms_reduce(A, 16, 512, float("nan"), A + MB, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_rms_reduce(A, 16, 512, 1e-5, A + 16, None) == g.CODA_ERR_INVALID_ARG  # r inside P
    assert lib.coda_fold_gamma(A, A + MB, A, 16, 64, 1, None) == g.CODA_ERR_INVALID_ARG  # in place
    assert lib.coda_fold_gamma(A, A + MB, A + 2 * MB, 16, 64, 2, None) == g.CODA_ERR_INVALID_ARG  # e4m3 fold
    assert lib.coda_amax(A, 16, 2, A + MB, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_quantize_e4m3(A, 64, 1, None, A + MB, A + 2 * MB, None) == g.CODA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    X = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(8, 8, dtype=torch.bfloat16)
    P = torch.zeros(4, 1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        g.coda_gemm_residual_partial_rms(X, W, X, X, P)


def test_binding_checks_shapes_and_dtypes_before_the_library_sees_a_pointer():
    """The kernels read and write the extents the sizes imply, so a tensor of
    another shape or dtype would be read or written out of bounds: the binding
    refuses it (these checks run before the CUDA-tensor check, so CPU tensors
    show them)."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    M, K, N = 4, 16, 8
    X, W, R = torch.zeros(M, K, dtype=bf), torch.zeros(N, K, dtype=bf), torch.zeros(M, N, dtype=bf)
    P = torch.zeros(M, 1)
    cases = [
        (lambda: g.coda_gemm_residual_partial_rms(X, W, R[:, :4].contiguous()), ValueError, "R has shape"),
        (lambda: g.coda_gemm_residual_partial_rms(X, W, R.float()), TypeError, "R has dtype"),
        (lambda: g.coda_gemm_residual_partial_rms(X, W[:, :8].contiguous(), R), ValueError, "W1t has shape"),
        (lambda: g.coda_gemm_residual_partial_rms(X, W, R, P=torch.zeros(M, 2)), ValueError, "P has shape"),
        (lambda: g.coda_rms_reduce(P, N, 1e-5, r=torch.zeros(M + 1)), ValueError, "r has shape"),
        (lambda: g.coda_gemm_rowscale(X, W, torch.zeros(M, dtype=bf)), TypeError, "r has dtype"),
        (lambda: g.coda_gemm_swiglu(X, W, W[:4].contiguous()), ValueError, "Wut has shape"),
        (lambda: g.coda_gemm(X, W, D=torch.zeros(M, N + 8, dtype=bf)), ValueError, "D has shape"),
        (lambda: g.coda_gemm(X, W.float()), TypeError, "B has dtype"),
        (lambda: g.coda_gemm_grad_norm(X, torch.zeros(K, N, dtype=bf), R, torch.zeros(N + 1)), ValueError,
         "gamma has shape"),
        (lambda: g.coda_gemm_swiglu_backward(X, torch.zeros(K, 64, dtype=bf), torch.zeros(M, 64, dtype=bf)),
         ValueError, "GU has shape"),
        (lambda: g.coda_block_swiglu(X, W, R, torch.zeros(64, N, dtype=bf), torch.zeros(64, N, dtype=bf), 1e-5,
                                     torch.zeros(0, dtype=torch.int32)), ValueError, "workspace holds"),
        (lambda: g.coda_block_rowscale(X, W, R, torch.zeros(64, N + 8, dtype=bf), 1e-5,
                                       torch.zeros(8, dtype=torch.int32)), ValueError, "W2t has shape"),
        (lambda: g.coda_quantize_e4m3(X, torch.zeros(1), q=torch.zeros(M * K - 1, dtype=torch.uint8)), ValueError,
         "q has"),
        (lambda: g.coda_amax(X, amax=torch.zeros(1, dtype=bf)), TypeError, "amax has dtype"),
        (lambda: g.coda_fold_gamma(W, torch.zeros(K + 1)), ValueError, "gamma has shape"),
    ]
    for fn, exc, msg in cases:
        with pytest.raises(exc, match=msg):
            fn()


def test_block_calls_validate(lib):
    # FP8 operands are refused (h needs its per-tensor amax first); a missing workspace is an argument error
    B = A + 512 * MB
    args = [A, A + 64 * MB, A + 128 * MB, A + 192 * MB, 1e-5, A + 256 * MB, A + 320 * MB, None, A + 384 * MB,
            256, 512, 512, 512]
    assert lib.coda_block_rowscale(*args, 2, B, None) == g.CODA_ERR_UNSUPPORTED
    assert lib.coda_block_rowscale(*args, 1, None, None) == g.CODA_ERR_INVALID_ARG
    assert b"workspace" in lib.coda_last_error()
    assert lib.coda_block_rowscale(*args, 1, A + 256 * MB, None) == g.CODA_ERR_INVALID_ARG  # workspace inside h
    assert lib.coda_block_workspace_bytes(8192) == (64 + 1) * 4
    assert lib.coda_block_workspace_bytes(1) == 8


def test_swiglu_save_and_backward_need_64_column_halves(lib):
    B = A + 512 * MB
    assert lib.coda_gemm_swiglu_save(A, A + 64 * MB, A + 128 * MB, A + 192 * MB, None, 0.0, None, A + 256 * MB,
                                     A + 320 * MB, 256, 520, 512, 1, None) == g.CODA_ERR_INVALID_ARG
    assert b"multiple of 64" in lib.coda_last_error()
    assert lib.coda_gemm_swiglu_backward(A, A + 64 * MB, A + 128 * MB, B, 256, 520, 512, 1, None) \
        == g.CODA_ERR_INVALID_ARG


def test_gemm_layout_rules(lib):
    # D [M, N] = A(m,k) B(n,k); operands 16-byte rows; MN-major only in bf16 and only A-with-B
    B = A + 64 * MB
    D = A + 128 * MB
    ok_args = (A, 0, B, 1, D, 256, 512, 320, 1, None, None, None)
    assert lib.coda_gemm(*ok_args[:5], 0, *ok_args[6:]) == g.CODA_OK          # M == 0: nothing to do
    assert lib.coda_gemm(A, 1, B, 0, D, 256, 512, 320, 1, None, None, None) == g.CODA_ERR_INVALID_ARG
    assert b"MN-major A needs" in lib.coda_last_error()
    assert lib.coda_gemm(A, 0, B, 1, D, 256, 512, 320, 0, None, None, None) == g.CODA_ERR_INVALID_ARG  # fp32 MN
    assert lib.coda_gemm(A, 1, B, 1, D, 100, 512, 320, 1, None, None, None) == g.CODA_ERR_INVALID_ARG  # [K, 100] rows
    assert lib.coda_gemm(A, 0, B, 0, D, 256, 512, 300, 1, None, None, None) == g.CODA_ERR_INVALID_ARG  # K = 300
    assert lib.coda_gemm(A, 0, B, 1, A + 4096, 256, 512, 320, 1, None, None, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_gemm(A, 2, B, 1, D, 256, 512, 320, 1, None, None, None) == g.CODA_ERR_INVALID_ARG


def test_backward_calls_validate(lib):
    B = A + 64 * MB
    # grad-norm and SwiGLU backward are bf16 only
    assert lib.coda_gemm_grad_norm(A, B, A + 128 * MB, A + 192 * MB, A + 256 * MB, A + 320 * MB, 256, 512, 512, 0,
                                   None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_gemm_swiglu_backward(A, B, A + 128 * MB, A + 192 * MB, 256, 512, 512, 0, None) \
        == g.CODA_ERR_INVALID_ARG
    # RMSNorm backward: N a multiple of 8, workspace sized per 64-row chunk
    assert lib.coda_rmsnorm_backward(A, B, A + 128 * MB, A + 129 * MB, A + 130 * MB, None, A + 192 * MB,
                                     A + 256 * MB, A + 320 * MB, A + 321 * MB, 256, 100, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_rmsnorm_backward_workspace_bytes(256, 512) == 4 * 512 * 4
    assert lib.coda_rmsnorm_backward_workspace_bytes(257, 512) == 5 * 512 * 4


def test_rope_arguments_validate(lib):
    B = A + 64 * MB
    base = (A, B, A + 128 * MB, None, 0.0, None, A + 192 * MB, 256, 512, 512, 1, None, None)
    # exactly one of r and P
    assert lib.coda_gemm_rowscale_rope(A, B, None, None, 0.0, None, A + 192 * MB, 256, 512, 512, 1, None, None,
                                       64, 256, 500000.0, 2048, None, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_gemm_rowscale_rope(*base, 60, 240, 500000.0, 2048, None, None) == g.CODA_ERR_INVALID_ARG  # head 60
    assert lib.coda_gemm_rowscale_rope(*base, 64, 200, 500000.0, 2048, None, None) == g.CODA_ERR_INVALID_ARG  # cols
    assert lib.coda_gemm_rowscale_rope(*base, 64, 256, 1.0, 2048, None, None) == g.CODA_ERR_INVALID_ARG      # base
    assert lib.coda_gemm_rowscale_rope(*base, 64, 256, 500000.0, 0, None, None) == g.CODA_ERR_INVALID_ARG    # seq


def test_selftest_timeout_range(lib):
    # the failure-path self-test only takes a bounded, sensible limit
    assert lib.coda_selftest_wait_timeout(0, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_selftest_wait_timeout(999, None) == g.CODA_ERR_INVALID_ARG
    assert lib.coda_selftest_wait_timeout(10_000_000_001, None) == g.CODA_ERR_INVALID_ARG
    assert b"timeout_ns" in lib.coda_last_error()


def _fp8_block(lib, M=512, N=256, K=512, N2=384, A_bf16=A, Aq=A + 64 * MB, H=A + 128 * MB, Hq=A + 192 * MB,
               R=A + 256 * MB, Z=A + 320 * MB, P=A + 384 * MB, W1=A + 448 * MB, W2=A + 512 * MB, ws=A + 576 * MB,
               amax_h=A + 640 * MB):
    s = A + 700 * MB  # the scalars: amax_a, scale_a, scale_w1, scale_w2, scale_h
    return lib.coda_block_rowscale_fp8(A_bf16, s, Aq, s + 16, W1, s + 32, R, W2, s + 48, 1e-5, H, P, None, amax_h, Hq,
                                       s + 64, Z, M, N, K, N2, ws, None)


def test_fp8_blocks_check_their_arguments(lib):
    """The FP8 one-launch blocks: e4m3 rows of 16 bytes for K and N, scale
    pointers required, outputs disjoint from inputs; all checked before
    anything is enqueued (amax_h is zeroed only after the checks)."""
    assert _fp8_block(lib, K=520) == g.CODA_ERR_INVALID_ARG          # e4m3 A rows: K % 16
    assert _fp8_block(lib, N=264) == g.CODA_ERR_INVALID_ARG          # e4m3 h rows: N % 16
    assert _fp8_block(lib, N2=100) == g.CODA_ERR_INVALID_ARG         # bf16 Z rows: N2 % 8
    assert _fp8_block(lib, Hq=None) == g.CODA_ERR_INVALID_ARG
    assert b"Hq is NULL" in lib.coda_last_error()
    assert _fp8_block(lib, ws=None) == g.CODA_ERR_INVALID_ARG
    assert _fp8_block(lib, Hq=A + 128 * MB) == g.CODA_ERR_INVALID_ARG  # Hq over H
    assert b"overlap" in lib.coda_last_error()
    assert _fp8_block(lib, Aq=A + 16) == g.CODA_ERR_INVALID_ARG     # the launch writes Aq over its source A
    # without A the launch reads Aq: Aq may not be an output's range either
    assert _fp8_block(lib, A_bf16=None, Aq=A + 128 * MB) == g.CODA_ERR_INVALID_ARG
    # the FP8 workspace holds three counters per 128-row band and two more
    assert lib.coda_block_fp8_workspace_bytes(1000) == (3 * 8 + 2) * 4
    assert lib.coda_block_fp8_workspace_bytes(-1) == -1


def test_block_rope_checks_rope_arguments(lib):
    """coda_block_rowscale_rope rejects RoPE arguments as coda_gemm_rowscale_rope
    does, before anything is enqueued."""
    def call(head_dim=64, rope_cols=256, base=500000.0, seq_len=128, positions=None, N2=384):
        return lib.coda_block_rowscale_rope(A, A + 64 * MB, A + 128 * MB, A + 192 * MB, 1e-5, A + 256 * MB,
                                            A + 320 * MB, None, A + 384 * MB, 256, 512, 512, N2, 1, head_dim,
                                            rope_cols, base, seq_len, positions, A + 448 * MB, None)
    assert call(head_dim=60) == g.CODA_ERR_INVALID_ARG           # bf16: a multiple of 8
    assert call(rope_cols=448) == g.CODA_ERR_INVALID_ARG         # beyond N2
    assert call(rope_cols=96) == g.CODA_ERR_INVALID_ARG          # not a multiple of head_dim
    assert call(base=1.0) == g.CODA_ERR_INVALID_ARG
    assert call(seq_len=0) == g.CODA_ERR_INVALID_ARG             # no positions and no sequence length
    assert call(positions=A + 256 * MB) == g.CODA_ERR_INVALID_ARG  # positions inside the output H
    assert b"overlaps" in lib.coda_last_error()
