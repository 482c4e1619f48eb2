"""The co-residency launch policy of the two-phase kernels (cooperative_action
and launch_coresident in coda_internal.h), on the host with a fake launcher:
a cooperative attempt that the runtime refuses for its form falls back to one
plain launch; any other error, a grid too large to be co-resident included,
is returned without a second attempt; a successful cooperative launch is the
only launch."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gemm_epilogue_fusion_gb300", "csrc")

PROGRAM = r"""
#include "coda_internal.h"
#include <cstdio>
#include <vector>
using namespace coda;
// attempts made with a fake launcher whose cooperative form returns `coop_err`
static int run(cudaError_t coop_err, bool try_coop, std::vector<int>* calls, bool* refused, cudaError_t* out) {
  *out = launch_coresident([&](bool coop) { calls->push_back(coop ? 1 : 0); return coop ? coop_err : cudaSuccess; },
                           try_coop, refused);
  return 0;
}
int main() {
  struct Case { cudaError_t e; const char* name; };
  const Case cases[] = {{cudaSuccess, "success"}, {cudaErrorNotSupported, "not_supported"},
                        {cudaErrorInvalidValue, "invalid_value"}, {cudaErrorInvalidConfiguration, "invalid_config"},
                        {cudaErrorCooperativeLaunchTooLarge, "too_large"},
                        {cudaErrorLaunchOutOfResources, "out_of_resources"}, {cudaErrorIllegalAddress, "illegal"}};
  for (const Case& c : cases) {
    std::vector<int> calls;
    bool refused = false;
    cudaError_t out;
    run(c.e, true, &calls, &refused, &out);
    printf("%s action=%d calls=", c.name, (int)cooperative_action(c.e));
    for (int v : calls) printf("%d", v);
    printf(" refused=%d result=%d\n", refused ? 1 : 0, (int)out);
  }
  std::vector<int> calls;
  bool refused = true;
  cudaError_t out;
  run(cudaErrorNotSupported, false, &calls, &refused, &out);
  printf("plain calls=%zu first=%d refused=%d result=%d\n", calls.size(), calls[0], refused ? 1 : 0, (int)out);
  return 0;
}
"""


def test_cooperative_attempt_falls_back_only_when_refused(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "policy.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "policy"
    r = subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                        "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=sm_103a", str(src),
                        "-o", str(exe)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    got = {l.split()[0]: l for l in out.stdout.splitlines()}
    assert got["success"].endswith("action=0 calls=1 refused=0 result=0")
    for refusal in ("not_supported", "invalid_value", "invalid_config"):
        # one cooperative attempt, then one plain launch, whose result is returned
        assert got[refusal].endswith("action=1 calls=10 refused=1 result=0"), got[refusal]
    for name in ("too_large", "out_of_resources", "illegal"):
        # never a second, plain attempt: the error is the result
        line = got[name]
        assert " action=2 calls=1 refused=0 " in line, line
        assert not line.endswith("result=0"), line
    # without the cooperative attempt: one plain launch
    assert got["plain"] == "plain calls=1 first=0 refused=0 result=0"
