"""Seeded random shapes for the FP8 one-launch blocks and for the backward
chain.

FP8: the chain of amax(X) and the two FP8 blocks must equal the nine-launch
FP8 chain bit for bit (codes, scales, every output) and match the
quantisation-aware oracle within the FP8 bar of 6e-2.  Widths are multiples of
16 (every e4m3 row a whole number of 16-byte chunks), 5% of the rows of X and
R scaled by 50 as in the FP8 workload.

Backward: the 12-launch backward of the block tail against the oracle's fp64
backward (which central finite differences pin), every gradient within the
bf16 bar of 2e-2; I a multiple of 64 (the SwiGLU backward's G and U boxes)."""
import random

import pytest
import torch

from coda_inputs import Workload, make_inputs
from parity_util import W, compare, oracle_ref, to_device
from test_backward_gpu import CHAIN_PAIRS, _chain_case, _check
from test_fp8_block_gpu import KEYS, _run_both

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gemm_epilogue_fusion_gb300 as g
    g.load_library()
    yield
    assert g.coda_get_device_status() == g.CODA_OK


def _random_fp8(seed: int) -> Workload:
    rnd = random.Random(9700 + seed)
    return Workload(f"fuzz_fp8_{seed}", "full", rnd.randint(1, 700), 16 * rnd.randint(1, 100),
                    16 * rnd.randint(1, 60), 16 * rnd.randint(1, 60), 16 * rnd.randint(1, 100), "e4m3", 1e-5,
                    700 + seed, heavy_rows=0.05)


@pytest.mark.parametrize("seed", range(6))
def test_fp8_blocks_random_shapes(seed, monkeypatch):
    w = _random_fp8(seed)
    monkeypatch.setenv("CODA_CTA_GROUP", "2" if seed % 2 else "1")
    inp = make_inputs(w)
    d = to_device(inp)
    got, ref = _run_both(w, d, quantize_x_in_block=seed % 3 != 0)
    for k in KEYS:
        assert torch.equal(got[k], ref[k]), (w, k)
    compare(w, {k: v.cpu() for k, v in got.items() if isinstance(v, torch.Tensor)}, oracle_ref(w, inp))


def _random_bwd(seed: int) -> Workload:
    rnd = random.Random(9900 + seed)
    return Workload(f"fuzz_bwd_{seed}", "full", rnd.randint(1, 500), 8 * rnd.randint(1, 60), 8 * rnd.randint(1, 60),
                    8 * rnd.randint(1, 60), 64 * rnd.randint(1, 8), "bf16", 1e-5, 900 + seed)


@pytest.mark.parametrize("seed", range(6))
def test_backward_random_shapes(seed, monkeypatch):
    w = _random_bwd(seed)
    monkeypatch.setenv("CODA_CTA_GROUP", "2" if seed % 2 else "1")
    inp, dZ, dH2, got = _chain_case(w, 950 + seed)
    ref = oracle.chain_full_backward(inp["X"], W(inp["W1t"]), inp["R"], inp["gamma1"], W(inp["Wgt"]),
                                     W(inp["Wut"]), W(inp["Wdt"]), inp["gamma2"], W(inp["Wqt"]), w.eps, dZ, dH2)
    print(w, _check(got, ref, CHAIN_PAIRS))
