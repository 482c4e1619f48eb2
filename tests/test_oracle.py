"""Pins for the CPU oracle: checks against values and facts that do not come
from the oracle itself (hand-derived golden cases, numpy's fp64 matmul, the
reparameterisation identity of the CODA write-ups, RMSNorm's scale
invariance, closed forms of silu, torch's float8_e4m3fn codec)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tiny_blocks.json")))
A = np.asarray


def _close(got, want, tol=1e-12):
    got, want = A(got, dtype=np.float64), A(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    np.testing.assert_allclose(got, want, rtol=tol, atol=tol)


@pytest.mark.parametrize("case", [c for c in GOLDEN["cases"] if c["kind"] == "rowscale"],
                         ids=lambda c: c["name"])
def test_golden_rowscale(case):
    out = oracle.block_rowscale(A(case["X"]), A(case["W1"]), A(case["R"]), A(case["gamma"]),
                                A(case["W2"]), case["eps"])
    _close(out["h"], case["h"])
    _close(out["r"], case["r"])
    _close(out["Z"], case["Z"])


def test_golden_full_chain():
    c = next(c for c in GOLDEN["cases"] if c["kind"] == "full")
    args = [A(c[k]) for k in ("X", "Wo", "R", "gamma1", "Wg", "Wu", "Wd", "gamma2", "Wq")]
    out = oracle.chain_full(*args, c["eps"])
    for k in ("h1", "r1", "act", "h2", "r2", "Z"):
        _close(out[k], c[k], 1e-12)
    # every tensor of this case holds a single nonzero magnitude, so per-tensor
    # E4M3 scaling represents it exactly and the quantisation-aware chain keeps
    # the exact values, except that its quantiser reads act rounded to bf16:
    # h2 and r2 move by at most that rounding (2^-9 relative), Z not at all
    # (r2 cancels the magnitude of the one-row h2)
    out = oracle.chain_full_fp8(*args, c["eps"])
    for k in ("h1", "r1", "act", "Z"):
        _close(out[k], c[k], 1e-12)
    for k in ("h2", "r2"):
        _close(out[k], c[k], 2.0 ** -9)


def _fp8_case():
    c = next(c for c in GOLDEN["cases"] if c["kind"] == "full_fp8")
    return c, [A(c[k]) for k in ("X", "Wo", "R", "gamma1", "Wg", "Wu", "Wd", "gamma2", "Wq")]


def test_golden_fp8_quantisation_sites():
    """The quantisation-aware chain against a hand-derived case in which every
    tensor holds values whose E4M3 rounding shows: X, Wo, the folded Wg, Wu,
    Wq, Wd, h1, act and h2 are quantised (gamma folded first), R and r are not."""
    c, args = _fp8_case()
    out = oracle.chain_full_fp8(*args, c["eps"])
    for k in ("h1", "r1", "act", "h2", "r2", "Z"):
        _close(out[k], c[k], 1e-12)
    # the case is sensitive to quantisation: the exact chain differs visibly
    exact = oracle.chain_full(*args, c["eps"])
    assert max(oracle.rel_err(exact[k], c[k]) for k in ("h1", "act", "h2", "Z")) > 1e-3


def _fp8_chain_variant(args, eps, skip=(), fold_after=False, quant_R=False, r_from_q=False, resid_q=False):
    """The FP8 chain composed from the oracle's steps with one site moved, to
    show that the golden case above tells each misplacement apart."""
    X, Wo, R, g1, Wg, Wu, Wd, g2, Wq = args
    # the quantiser reads the bf16-rounded tensor, as the block stores it
    q = lambda n, t: t if n in skip else oracle.fake_quant_e4m3(oracle.round_bf16(t))[0]  # noqa: E731
    if fold_after:
        Wg_f, Wu_f, Wq_f = g1[:, None] * q("Wg", Wg), g1[:, None] * q("Wu", Wu), g2[:, None] * q("Wq", Wq)
    else:
        Wg_f, Wu_f, Wq_f = q("Wg", g1[:, None] * Wg), q("Wu", g1[:, None] * Wu), q("Wq", g2[:, None] * Wq)
    h1 = oracle.gemm(q("X", X), q("Wo", Wo), oracle.fake_quant_e4m3(oracle.round_bf16(R))[0] if quant_R else R)
    h1q = q("h1", h1)
    _, r1 = oracle.rmsnorm(h1q if r_from_q else h1, g1, eps)
    act = oracle.silu_mul(oracle.gemm(h1q, Wg_f) * r1[:, None], oracle.gemm(h1q, Wu_f) * r1[:, None])
    h2 = oracle.gemm(q("act", act), q("Wd", Wd), h1q if resid_q else h1)
    h2q = q("h2", h2)
    _, r2 = oracle.rmsnorm(h2q if r_from_q else h2, g2, eps)
    return {"h1": h1, "r1": r1, "act": act, "h2": h2, "r2": r2, "Z": oracle.gemm(h2q, Wq_f) * r2[:, None]}


@pytest.mark.parametrize("mistake", [
    {"skip": ("X",)}, {"skip": ("Wo",)}, {"skip": ("Wg",)}, {"skip": ("Wu",)}, {"skip": ("Wd",)}, {"skip": ("Wq",)},
    {"skip": ("h1",)}, {"skip": ("act",)}, {"skip": ("h2",)}, {"fold_after": True}, {"quant_R": True},
    {"r_from_q": True}, {"resid_q": True}], ids=lambda m: "-".join(f"{k}={v}" for k, v in m.items()))
def test_fp8_golden_catches_each_misplaced_quantisation(mistake):
    """A mistake planted in the composition (a quantisation dropped, the fold
    after the quantisation, R quantised, r taken from the quantised h, the
    quantised h1 as the down projection's residual) changes some output of
    the golden case by far more than the 1e-12 its pin allows."""
    c, args = _fp8_case()
    right = _fp8_chain_variant(args, c["eps"])
    for k in ("h1", "r1", "act", "h2", "r2", "Z"):
        _close(right[k], c[k], 1e-12)
    wrong = _fp8_chain_variant(args, c["eps"], **mistake)
    assert max(oracle.rel_err(wrong[k], c[k]) for k in right) > 1e-4


def test_golden_swiglu_gate_vs_up():
    c = GOLDEN["swiglu_gate_up"]
    _close(oracle.swiglu(A(c["Y"]), A(c["Wg"]), A(c["Wu"])), c["act"])


def test_silu_closed_forms():
    for x, want in GOLDEN["silu"]["points"]:
        assert oracle.silu(x) == pytest.approx(want, rel=1e-15, abs=1e-300)
    # silu(x) -> x for large x, -> 0 (from below) for very negative x
    assert oracle.silu(40.0) == pytest.approx(40.0, rel=1e-15)
    assert -1e-15 < oracle.silu(-40.0) < 0.0
    # silu(x) - silu(-x) = x (sigmoid(x) + sigmoid(-x) = 1)
    for x in (0.3, 1.7, 5.0):
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, rel=1e-14)


def test_gemm_matches_numpy_fp64():
    rng = np.random.default_rng(0)
    X = rng.standard_normal((256, 512))
    W = rng.standard_normal((512, 384)) / math.sqrt(512)
    R = rng.standard_normal((256, 384))
    np.testing.assert_allclose(oracle.gemm(X, W), X @ W, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.gemm(X, W, R), R + X @ W, rtol=1e-12, atol=1e-12)


def test_rmsnorm_matches_closed_form_on_random_rows():
    rng = np.random.default_rng(1)
    H = rng.standard_normal((7, 33)) * 3.0
    g = 1.0 + 0.1 * rng.standard_normal(33)
    y, r = oracle.rmsnorm(H, g, 1e-5)
    for i in range(7):
        want_r = 1.0 / math.sqrt(sum(v * v for v in H[i]) / 33 + 1e-5)
        assert r[i] == pytest.approx(want_r, rel=1e-13)
        np.testing.assert_allclose(y[i], H[i] * want_r * g, rtol=1e-13)


def test_reparameterisation_identity():
    """RMSNorm(h).gamma.W2 == diag(r) . h . (diag(gamma) W2): the row scale
    commutes with the next matmul ('the treasure hidden in the epilogue')."""
    rng = np.random.default_rng(2)
    M, K, N, N2 = 256, 512, 512, 384
    X = rng.standard_normal((M, K))
    R = rng.standard_normal((M, N))
    W1 = rng.standard_normal((K, N)) / math.sqrt(K)
    W2 = rng.standard_normal((N, N2)) / math.sqrt(N)
    g = 1.0 + 0.1 * rng.standard_normal(N)
    out = oracle.block_rowscale(X, W1, R, g, W2, 1e-6)
    reparam = out["r"][:, None] * (out["h"] @ (g[:, None] * W2))
    np.testing.assert_allclose(out["Z"], reparam, rtol=1e-11, atol=1e-11)
    # SwiGLU with the row scale applied to both projections before silu
    Wg = rng.standard_normal((N, 96)) / math.sqrt(N)
    Wu = rng.standard_normal((N, 96)) / math.sqrt(N)
    sw = oracle.block_swiglu(X, W1, R, g, Wg, Wu, 1e-6)
    G = out["r"][:, None] * (out["h"] @ (g[:, None] * Wg))
    U = out["r"][:, None] * (out["h"] @ (g[:, None] * Wu))
    np.testing.assert_allclose(sw["act"], G / (1 + np.exp(-G)) * U, rtol=1e-11, atol=1e-11)


def test_scale_invariance():
    """eps=0: scaling a row of h by c>0 leaves RMSNorm's output unchanged and
    divides r by c."""
    rng = np.random.default_rng(3)
    M, K, N = 8, 32, 48
    X, R = rng.standard_normal((M, K)), rng.standard_normal((M, N))
    W1, W2 = rng.standard_normal((K, N)), rng.standard_normal((N, 16))
    g = 1.0 + 0.1 * rng.standard_normal(N)
    base = oracle.block_rowscale(X, W1, R, g, W2, 0.0)
    c = np.array([1.0, 2.0, 0.5, 50.0, 1e-3, 7.0, 1.0, 3.0])
    sc = oracle.block_rowscale(X * c[:, None], W1, R * c[:, None], g, W2, 0.0)
    np.testing.assert_allclose(sc["h"], base["h"] * c[:, None], rtol=1e-12)
    np.testing.assert_allclose(sc["r"], base["r"] / c, rtol=1e-12)
    np.testing.assert_allclose(sc["Z"], base["Z"], rtol=1e-10, atol=1e-12)
    # constant row (a, ..., a) with eps=0 normalises to sign(a) * gamma
    y, _ = oracle.rmsnorm(np.full((2, 5), [[-2.5], [4.0]]), np.arange(1.0, 6.0), 0.0)
    np.testing.assert_allclose(y, [[-1, -2, -3, -4, -5], [1, 2, 3, 4, 5]], rtol=1e-14)


def test_e4m3_decode_all_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0 and np.nanmin(np.abs(got[got != 0])) == 2.0 ** -9


def test_e4m3_encode_vs_torch_rne():
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[np.abs(x) <= 448.0]
    # all midpoints between neighbouring codes: ties go to the even code
    vals = np.array(sorted(set(oracle.e4m3_decode(c) for c in range(0, 0x7F))))
    mids = (vals[1:] + vals[:-1]) / 2
    x = np.concatenate([x, mids, -mids, vals, -vals])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    # -0.0 / +0.0 may differ only in sign bit for inputs that round to zero
    zero = (ref & 0x7F) == 0
    assert np.array_equal(got[~zero], ref[~zero])
    assert np.all((got[zero] & 0x7F) == 0)


def test_round_bf16_vs_torch_and_hand_ties():
    """bf16 rounding (the quantiser's input in the FP8 chain) against torch's
    fp32 -> bf16 cast on fp32 values across the whole range, subnormals
    included (exact in fp64, so both round once), and hand-worked ties."""
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 31, 200000, dtype=np.int64).astype(np.uint32)
    x32 = bits.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    # exact midpoints between neighbouring bf16 values: the 16 low bits 0x8000
    ties = ((bits & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    x32 = np.concatenate([x32, ties[np.isfinite(ties)], -x32[:1000]])
    ref = torch.from_numpy(x32.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x32.astype(np.float64))
    assert np.array_equal(got, ref)
    hand = {1 + 2.0 ** -8: 1.0, 1 + 3 * 2.0 ** -8: 1 + 2.0 ** -6, -(1 + 2.0 ** -8): -1.0, 0.3: 0.30078125,
            2.0 ** -130: 2.0 ** -130, 3 * 2.0 ** -134: 2.0 ** -132, 2.0 ** -134: 0.0,
            255 * 2.0 ** 120: 255 * 2.0 ** 120}
    for v, want in hand.items():
        assert oracle.round_bf16(np.array([v]))[0] == want, v
    assert np.isinf(oracle.round_bf16(np.array([255.5 * 2.0 ** 120]))[0])  # a tie to 2^128: infinity


def test_e4m3_saturates_and_nan():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(470.0) == 0x7E      # would round to 480: saturate
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # tie between 0 and 2^-9: even
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02


def test_fake_quant_exact_on_representable_and_bounded_error():
    vals = np.array([oracle.e4m3_decode(c) for c in range(0, 0x7F)])
    s = 0.125
    x = np.concatenate([vals, -vals]) * s
    xq, sq = oracle.fake_quant_e4m3(x)
    assert sq == pytest.approx(448.0 * s / 448.0)
    np.testing.assert_array_equal(xq, x)
    rng = np.random.default_rng(5)
    y = rng.standard_normal(10000)
    yq, sy = oracle.fake_quant_e4m3(y)
    normal = np.abs(y) >= sy * 2.0 ** -6
    # relative rounding error of a normal E4M3 number is at most 2^-4
    assert np.max(np.abs(yq - y)[normal] / np.abs(y[normal])) <= 2.0 ** -4 + 1e-12


def test_fp8_chain_close_to_exact_chain():
    rng = np.random.default_rng(6)
    M, H, I, Q = 16, 64, 96, 48
    X, R = rng.standard_normal((M, H)), rng.standard_normal((M, H))
    Wo, Wg, Wu = (rng.standard_normal(s) / math.sqrt(s[0]) for s in ((H, H), (H, I), (H, I)))
    Wd, Wq = rng.standard_normal((I, H)) / math.sqrt(I), rng.standard_normal((H, Q)) / math.sqrt(H)
    g1, g2 = 1 + 0.1 * rng.standard_normal(H), 1 + 0.1 * rng.standard_normal(H)
    ex = oracle.chain_full(X, Wo, R, g1, Wg, Wu, Wd, g2, Wq, 1e-5)
    q8 = oracle.chain_full_fp8(X, Wo, R, g1, Wg, Wu, Wd, g2, Wq, 1e-5)
    for k in ("h1", "act", "h2", "Z"):
        e = oracle.rel_err(q8[k], ex[k])
        assert 1e-4 < e < 0.1, (k, e)   # quantisation is visible but bounded


def test_rel_err_metric():
    assert oracle.rel_err([1.0, 2.0], [1.0, 2.0]) == 0.0
    assert oracle.rel_err([1.0, 2.5], [1.0, 2.0]) == pytest.approx(0.25, rel=1e-6)


def test_fp8_chain_row_subset_equals_full_chain():
    """out_rows only narrows what is returned and which rows the last GEMM
    computes; the per-tensor scales still come from every row."""
    rng = np.random.default_rng(7)
    M, H, I, Q = 20, 32, 48, 24
    X, Wo, R = rng.standard_normal((M, H)), rng.standard_normal((H, H)), rng.standard_normal((M, H))
    X[5] *= 50.0  # a heavy row sets the scales; it is not among the returned rows
    Wg, Wu = rng.standard_normal((H, I)), rng.standard_normal((H, I))
    Wd, Wq = rng.standard_normal((I, H)), rng.standard_normal((H, Q))
    g1, g2 = 1 + 0.1 * rng.standard_normal(H), 1 + 0.1 * rng.standard_normal(H)
    full = oracle.chain_full_fp8(X, Wo, R, g1, Wg, Wu, Wd, g2, Wq, 1e-5)
    rows = [3, 7, 19]
    sub = oracle.chain_full_fp8(X, Wo, R, g1, Wg, Wu, Wd, g2, Wq, 1e-5, out_rows=rows)
    for k in full:
        np.testing.assert_array_equal(sub[k], full[k][rows])


# ----------------------------------------------------------------- RoPE ----
# RoFormer's rotary embedding in its complex form: viewing pair j of a head as
# x_2j + i x_2j+1, position p multiplies it by exp(i p base^(-2j/d)).  The
# oracle writes it as a real rotation; these pins hold it to the complex
# definition and to the properties that make it a position encoding.

def _rope_complex(Z, rot_cols, d, pos, base):
    Z = np.array(Z, dtype=np.float64)
    zc = Z[:, :rot_cols:2] + 1j * Z[:, 1:rot_cols:2]          # [M, rot_cols/2]
    j = np.arange(rot_cols // 2) % (d // 2)                    # pair index within its head
    zc = zc * np.exp(1j * np.outer(pos, base ** (-2.0 * j / d)))
    Z[:, :rot_cols:2], Z[:, 1:rot_cols:2] = zc.real, zc.imag
    return Z


def test_rope_matches_complex_multiplication_and_leaves_v():
    rng = np.random.default_rng(8)
    M, N, rot, d = 9, 48, 32, 8
    Z = rng.standard_normal((M, N))
    pos = rng.integers(0, 5000, M)
    got = oracle.rope(Z, rot, d, pos, 500000.0)
    np.testing.assert_allclose(got, _rope_complex(Z, rot, d, pos, 500000.0), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(got[:, rot:], Z[:, rot:])


def test_rope_position_zero_is_identity_and_positions_compose():
    rng = np.random.default_rng(9)
    Z = rng.standard_normal((4, 16))
    np.testing.assert_array_equal(oracle.rope(Z, 16, 8, np.zeros(4), 10000.0), Z)
    p1, p2 = np.array([1, 7, 100, 2047]), np.array([3, 0, 900, 1])
    twice = oracle.rope(oracle.rope(Z, 16, 8, p1, 10000.0), 16, 8, p2, 10000.0)
    np.testing.assert_allclose(twice, oracle.rope(Z, 16, 8, p1 + p2, 10000.0), rtol=1e-10, atol=1e-12)


def test_rope_first_pair_turns_by_the_position_in_every_head():
    # theta_0 = base^0 = 1 whatever the base, and the frequency index restarts
    # in each head: column 0 and column d of (1, 0, ...) rotate by exactly p
    d = 4
    Z = np.zeros((1, 8))
    Z[0, 0] = Z[0, d] = 1.0
    got = oracle.rope(Z, 8, d, np.array([1]), 123.0)
    for c in (0, d):
        assert got[0, c] == pytest.approx(math.cos(1.0), abs=1e-15)
        assert got[0, c + 1] == pytest.approx(math.sin(1.0), abs=1e-15)   # counter-clockwise


def test_block_rowscale_rope_rotates_only_the_qk_columns_of_the_block():
    """The composed oracle (block, then RoPE on the QKV output): at position 0
    it is the plain block; the columns past rot_cols (V) equal the plain
    block's at any position; every rotated pair keeps its length; and the
    first pair of each head turns by exactly p radians (theta_0 = 1)."""
    rng = np.random.default_rng(12)
    M, K, N, N2, rot, d = 5, 24, 16, 40, 32, 8
    X, R = rng.standard_normal((M, K)), rng.standard_normal((M, N))
    W1, W2 = rng.standard_normal((K, N)) / K ** 0.5, rng.standard_normal((N, N2)) / N ** 0.5
    gamma = 1 + 0.1 * rng.standard_normal(N)
    plain = oracle.block_rowscale(X, W1, R, gamma, W2, 1e-5)["Z"]
    at_zero = oracle.block_rowscale_rope(X, W1, R, gamma, W2, 1e-5, rot, d, np.zeros(M), 500000.0)["Z"]
    np.testing.assert_array_equal(at_zero, plain)
    pos = np.array([1, 2, 17, 300, 4095])
    got = oracle.block_rowscale_rope(X, W1, R, gamma, W2, 1e-5, rot, d, pos, 500000.0)["Z"]
    np.testing.assert_array_equal(got[:, rot:], plain[:, rot:])
    np.testing.assert_allclose(np.hypot(got[:, 0:rot:2], got[:, 1:rot:2]),
                               np.hypot(plain[:, 0:rot:2], plain[:, 1:rot:2]), rtol=1e-12)
    for c in range(0, rot, d):
        turn = np.arctan2(got[:, c + 1], got[:, c]) - np.arctan2(plain[:, c + 1], plain[:, c]) - pos
        np.testing.assert_allclose(np.mod(turn + np.pi, 2 * np.pi) - np.pi, 0, atol=1e-9)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(10)
    d = 16
    q, k = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    def score(m, n):
        return float((oracle.rope(q, d, d, np.array([m]), 500000.0) @ oracle.rope(k, d, d, np.array([n]), 500000.0).T)[0, 0])
    assert score(10, 3) == pytest.approx(score(1010, 1003), rel=1e-9)
    assert score(5, 5) == pytest.approx(float((q @ k.T)[0, 0]), rel=1e-12)
    # and each pair keeps its length
    z = oracle.rope(q, d, d, np.array([777]), 500000.0)
    np.testing.assert_allclose(z[0, ::2] ** 2 + z[0, 1::2] ** 2, q[0, ::2] ** 2 + q[0, 1::2] ** 2, rtol=1e-12)


# ------------------------------------------------------------- backward ----
# The backward oracle is pinned by central finite differences of the forward
# oracle: L = sum(dOut * out) + sum(dH_in * h), differentiated numerically in
# every input element of tiny blocks.

def _num_grad(f, arrays, name, eps=1e-6):
    a = arrays[name]
    g = np.zeros_like(a)
    for idx in np.ndindex(a.shape):
        old = a[idx]
        a[idx] = old + eps
        lp = f(arrays)
        a[idx] = old - eps
        lm = f(arrays)
        a[idx] = old
        g[idx] = (lp - lm) / (2 * eps)
    return g


@pytest.mark.parametrize("with_dh", [False, True])
def test_rowscale_backward_matches_finite_differences(with_dh):
    rng = np.random.default_rng(11)
    M, K, N, N2 = 3, 4, 5, 6
    A = {"X": rng.standard_normal((M, K)), "W1": rng.standard_normal((K, N)), "R": rng.standard_normal((M, N)),
         "gamma": 1 + 0.1 * rng.standard_normal(N), "W2": rng.standard_normal((N, N2))}
    dZ = rng.standard_normal((M, N2))
    dH = rng.standard_normal((M, N)) if with_dh else None

    def loss(a):
        o = oracle.block_rowscale(a["X"], a["W1"], a["R"], a["gamma"], a["W2"], 1e-3)
        return float(np.sum(dZ * o["Z"]) + (np.sum(dH * o["h"]) if with_dh else 0.0))
    got = oracle.block_rowscale_backward(A["X"], A["W1"], A["R"], A["gamma"], A["W2"], 1e-3, dZ, dH)
    for name, key in (("X", "dX"), ("W1", "dW1"), ("R", "dR"), ("gamma", "dgamma"), ("W2", "dW2")):
        np.testing.assert_allclose(got[key], _num_grad(loss, A, name), rtol=1e-6, atol=1e-8, err_msg=name)


def test_swiglu_backward_matches_finite_differences():
    rng = np.random.default_rng(12)
    M, K, N, I = 3, 4, 5, 6
    A = {"X": rng.standard_normal((M, K)), "W1": rng.standard_normal((K, N)), "R": rng.standard_normal((M, N)),
         "gamma": 1 + 0.1 * rng.standard_normal(N), "Wg": rng.standard_normal((N, I)),
         "Wu": rng.standard_normal((N, I))}
    dAct = rng.standard_normal((M, I))
    dH = rng.standard_normal((M, N))

    def loss(a):
        o = oracle.block_swiglu(a["X"], a["W1"], a["R"], a["gamma"], a["Wg"], a["Wu"], 1e-3)
        return float(np.sum(dAct * o["act"]) + np.sum(dH * o["h"]))
    got = oracle.block_swiglu_backward(A["X"], A["W1"], A["R"], A["gamma"], A["Wg"], A["Wu"], 1e-3, dAct, dH)
    for name, key in (("X", "dX"), ("W1", "dW1"), ("R", "dR"), ("gamma", "dgamma"), ("Wg", "dWg"),
                      ("Wu", "dWu")):
        np.testing.assert_allclose(got[key], _num_grad(loss, A, name), rtol=1e-6, atol=1e-8, err_msg=name)


def test_silu_derivative_closed_form_and_norm_gradient_orthogonal_to_h():
    # silu'(0) = 1/2, and silu' integrates back to silu (d/dG of silu(G) * 1)
    dG, dU = oracle.silu_mul_backward(np.array([0.0, 2.0]), np.array([1.0, 1.0]), np.array([1.0, 1.0]))
    assert dG[0] == pytest.approx(0.5, abs=1e-15)
    s = 1 / (1 + math.exp(-2.0))
    assert dG[1] == pytest.approx(s * (1 + 2 * (1 - s)), rel=1e-14)
    assert dU[1] == pytest.approx(oracle.silu(2.0), rel=1e-14)
    # with eps = 0 the normalised output ignores the row's scale, so the
    # input gradient has no component along h
    rng = np.random.default_rng(13)
    H, dY = rng.standard_normal((4, 7)), rng.standard_normal((4, 7))
    dH, _ = oracle.rmsnorm_backward(H, 1 + 0.1 * rng.standard_normal(7), 0.0, dY)
    np.testing.assert_allclose(np.sum(dH * H, axis=1), 0.0, atol=1e-12)


def test_chain_backward_matches_finite_differences():
    rng = np.random.default_rng(14)
    M, K, H, I, Q = 2, 3, 4, 5, 3
    A = {"X": rng.standard_normal((M, K)), "Wo": rng.standard_normal((K, H)), "R": rng.standard_normal((M, H)),
         "g1": 1 + 0.1 * rng.standard_normal(H), "Wg": rng.standard_normal((H, I)), "Wu": rng.standard_normal((H, I)),
         "Wd": rng.standard_normal((I, H)), "g2": 1 + 0.1 * rng.standard_normal(H), "Wq": rng.standard_normal((H, Q))}
    dZ, dH2 = rng.standard_normal((M, Q)), rng.standard_normal((M, H))

    def loss(a):
        o = oracle.chain_full(a["X"], a["Wo"], a["R"], a["g1"], a["Wg"], a["Wu"], a["Wd"], a["g2"], a["Wq"], 1e-3)
        return float(np.sum(dZ * o["Z"]) + np.sum(dH2 * o["h2"]))
    got = oracle.chain_full_backward(A["X"], A["Wo"], A["R"], A["g1"], A["Wg"], A["Wu"], A["Wd"], A["g2"], A["Wq"],
                                     1e-3, dZ, dH2)
    for name, key in (("X", "dX"), ("R", "dR"), ("Wo", "dWo"), ("g1", "dgamma1"), ("Wg", "dWg"), ("Wu", "dWu"),
                      ("Wd", "dWd"), ("g2", "dgamma2"), ("Wq", "dWq")):
        np.testing.assert_allclose(got[key], _num_grad(loss, A, name), rtol=1e-6, atol=1e-8, err_msg=name)
