"""The tile walk of the persistent GEMM (walk_tile in gemm_epilogue.cuh), on
the host: compiled from the kernel header itself with nvcc and run on the CPU.
Every tile index is dealt exactly once, each unit's walk increases, every unit
walks all its phase-A tiles before any phase-B tile (what keeps the
two-phase launch's band waits free of cycles), and on the workloads' shapes the
busiest unit gets no more k-blocks than under a plain round robin.  The
grouped raster (tile_at) maps the tile indices of each phase one to one onto
its grid of output tiles for every band width, ragged last bands included."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gemm_epilogue_fusion_gb300", "csrc")

PROGRAM = r"""
#include "gemm_epilogue.cuh"
#include <cstdio>
#include <vector>
#include <algorithm>
using coda::walk_tile;
using coda::tile_at;
// 0 if tile_at maps phase A's and phase B's indices one to one onto their grids
static int check_raster(int m_tiles, int n_a, int n_b, int g_a, int g_b, int nm_a = 0, int nm_b = 0) {
  std::vector<int> seen_a(m_tiles * n_a, 0), seen_b(m_tiles * n_b, 0);
  for (int t = 0; t < m_tiles * (n_a + n_b); ++t) {
    const coda::Tile c = tile_at(t, m_tiles, n_a, n_b, coda::Raster{g_a, nm_a, 0}, coda::Raster{g_b, nm_b, 0});
    const int nn = c.phase ? n_b : n_a;
    if (c.phase != (t >= m_tiles * n_a) || c.m < 0 || c.m >= m_tiles || c.n < 0 || c.n >= nn) return 1;
    (c.phase ? seen_b : seen_a)[c.m * nn + c.n]++;
  }
  for (int v : seen_a) if (v != 1) return 2;
  for (int v : seen_b) if (v != 1) return 2;
  return 0;
}
static int d_of(int kb_a, int kb_b) { return (kb_a + kb_b / 2) / std::max(1, kb_b); }
// 0 if every tile is dealt once, walks increase and phase A precedes phase B
static int check_cover(int U, int nA, int nB, int d, long* max_w, long* max_rr, int kb_a, int kb_b) {
  std::vector<int> seen(nA + nB, 0);
  *max_w = 0; *max_rr = 0;
  for (int u = 0; u < U; ++u) {
    int prev = -1; bool in_b = false; long w = 0;
    for (int k = 0;; ++k) {
      const int t = walk_tile(u, k, U, nA, nB, d);
      if (t >= nA + nB) break;
      if (t <= prev || (t < nA && in_b) || k > nA + nB) return 1;
      in_b = in_b || t >= nA;
      seen[t]++; prev = t; w += t < nA ? kb_a : kb_b;
    }
    *max_w = std::max(*max_w, w);
    long rr = 0;
    for (int t = u; t < nA + nB; t += U) rr += t < nA ? kb_a : kb_b;
    *max_rr = std::max(*max_rr, rr);
  }
  for (int i = 0; i < nA + nB; ++i) if (seen[i] != 1) return 2;
  return 0;
}
int main() {
  long w, rr;
  for (int m = 1; m <= 40; m += 3)
    for (int na = 1; na <= 24; na += 5)
      for (int nb = 0; nb <= 70; nb += 23)
        for (int ga = 1; ga <= 34; ga += 3)
          for (int gb = 1; gb <= 34; gb += 4)
            for (int nm = 0; nm < 4; ++nm)
              if (check_raster(m, na, nb, ga, gb, nm & 1, nm >> 1)) { printf("FAIL raster m=%d na=%d nb=%d ga=%d gb=%d nm=%d\n", m, na, nb, ga, gb, nm); return 1; }
  // N-major bands walk rows in order: the first n tiles of a band are row 0
  {
    const coda::TileCoord c0 = coda::tile_coord(0, 10, 16, 8, 1), c7 = coda::tile_coord(7, 10, 16, 8, 1),
                          c8 = coda::tile_coord(8, 10, 16, 8, 1), c80 = coda::tile_coord(80, 10, 16, 8, 1);
    if (c0.m != 0 || c0.n != 0 || c7.m != 0 || c7.n != 7 || c8.m != 1 || c8.n != 0 || c80.m != 0 || c80.n != 8) {
      printf("FAIL n-major order\n"); return 1;
    }
  }
  // the raster chosen for each phase of the LLaMA blocks (bf16, CTA pairs):
  // group, n_major, keep (0: keep A, 1: keep B)
  {
    using Res = coda::GemmCfg<coda::kKindBF16, coda::kEpiResidualPartialRms, coda::kNoPhase, 5, 4, 2>;
    using Sw = coda::GemmCfg<coda::kKindBF16, coda::kEpiSwiGLU, coda::kNoPhase, 6, 2, 2>;
    using Rs = coda::GemmCfg<coda::kKindBF16, coda::kEpiRowScale, coda::kNoPhase, 6, 2, 2>;
    const coda::Raster r[] = {
        coda::choose_raster<Res>(16384, 4096, 4096, coda::kEpiResidualPartialRms),   // 8B Wo
        coda::choose_raster<Sw>(16384, 14336, 4096, coda::kEpiSwiGLU),               // 8B gate/up
        coda::choose_raster<Res>(16384, 4096, 14336, coda::kEpiResidualPartialRms),  // 8B down
        coda::choose_raster<Rs>(16384, 6144, 4096, coda::kEpiRowScale),              // 8B QKV
        coda::choose_raster<Res>(8192, 2048, 8192, coda::kEpiResidualPartialRms),    // 1B MLP-down
        coda::choose_raster<Rs>(8192, 3072, 2048, coda::kEpiRowScale),               // 1B QKV
        coda::choose_raster<Sw>(8192, 8192, 2048, coda::kEpiSwiGLU)};                // 1B gate/up
    for (const auto& x : r) printf("raster group=%d n_major=%d keep=%d\n", x.group, x.n_major, x.keep);
  }
  for (int U = 1; U < 160; U += 3)
    for (int nA = 0; nA < 700; nA += 41)
      for (int nB = 0; nB < 900; nB += 67)
        for (int d = 0; d < 6; ++d)
          if (check_cover(U, nA, nB, d, &w, &rr, 1, 1)) { printf("FAIL U=%d nA=%d nB=%d d=%d\n", U, nA, nB, d); return 1; }
  // (pairs, phase-A tiles, phase-B tiles, k-blocks per phase-A tile, per phase-B tile) of the block launches
  const int shapes[][5] = {{76, 256, 2048, 32, 32}, {76, 256, 384, 128, 32}, {76, 1024, 7168, 64, 64},
                           {76, 1024, 1536, 224, 64}, {152, 512, 768, 128, 32}};
  for (const auto& s : shapes) {
    const int d = d_of(s[3], s[4]);
    if (check_cover(s[0], s[1], s[2], d, &w, &rr, s[3], s[4])) { printf("FAIL shape\n"); return 1; }
    printf("shape U=%d nA=%d nB=%d d=%d max=%ld round_robin_max=%ld\n", s[0], s[1], s[2], d, w, rr);
    if (w > rr) { printf("FAIL worse than round robin\n"); return 1; }
  }
  printf("all ok\n");
  return 0;
}
"""


def test_walk_tile_deals_every_tile_once_in_phase_order(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "walk.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "walk"
    r = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                        "--expt-relaxed-constexpr", "-gencode", "arch=compute_103a,code=sm_103a", str(src),
                        "-o", str(exe), "-lcuda"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and "all ok" in out.stdout, out.stdout[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("shape")]
    # the 1B MLP-down + QKV block: 4x longer phase-A tiles, balanced from 672 to 608 k-blocks
    assert "nA=256 nB=384 d=4 max=608 round_robin_max=672" in out.stdout, lines
    # the raster per phase: a phase with K rows of 8192 bytes or more whose
    # whole weight fits 40 MB keeps it (N-major rows, every N-tile in one
    # band): the 8B Wo (33.5 MB) and the 1B MLP-down (33.5 MB); every other
    # phase keeps the legacy M-major bands (8 M-tiles of 256 rows; 16 for
    # gate/up)
    rs = [l for l in out.stdout.splitlines() if l.startswith("raster")]
    assert rs == ["raster group=16 n_major=1 keep=1", "raster group=16 n_major=0 keep=2",
                  "raster group=8 n_major=0 keep=2", "raster group=8 n_major=0 keep=2",
                  "raster group=8 n_major=1 keep=1", "raster group=8 n_major=0 keep=2",
                  "raster group=16 n_major=0 keep=2"], rs
