// Persistent, warp-specialised tcgen05 GEMM with fused epilogue programs.
//
// D[M, N_out] = epilogue(A[M, K] . B[N_out, K]^T), operands K-major by default
// (activations [M, K] and weights W^T [N_out, K], row-major; MN-major for the
// backward's transposed products, see below), TMA-loaded with 128-byte swizzle
// so every k-block row of a tile is exactly 128 bytes.
//
// One CTA (or one cluster pair of CTAs, tcgen05 cta_group::2) per SM walks
// output tiles of 128 (256) rows.  Roles (warps):
//   0      TMA producer: A and B k-blocks into a STAGES-deep shared ring
//   1      TMEM owner + MMA issuer (one thread): tcgen05.mma into one of two
//          256-column TMEM accumulators, so the epilogue of tile i overlaps
//          the mainloop of tile i+1
//   2..5   epilogue: tcgen05.ld (one accumulator row per thread) -> fused
//          program -> 128B-swizzled shared slot -> TMA store, one 128-byte
//          wide column box at a time
//   6      programs that read a tile of another tensor (R of the residual,
//          H of the grad-norm, G and U of the SwiGLU backward): TMA loads of
//          those boxes into the slot ring, so the epilogue reads them from
//          shared memory and writes its result in place; in a two-phase launch
//          it also hands the slots of the second phase's boxes to the epilogue
//   7..10  FP8 one-launch blocks only: quantiser warps that write the e4m3
//          copies of phase A's input and of h, band by band, for the TMA loads
//          of the GEMMs that follow in the same launch
//
// Epilogue programs.  The CODA write-ups ("CODA: the treasure hidden in the
// epilogue") apply the memory-bound neighbours of a GEMM while its product is
// still on chip:
//   kEpiResidualPartialRms  h = R + acc ; P[row, g] = sum of h^2 over the
//                           128-column group g of the row (of the stored,
//                           rounded h).  GEMM1 of GEMM -> add -> RMSNorm -> GEMM.
//   kEpiRowScale            Z = r_row * acc: RMSNorm's row scale moved past
//                           the second GEMM (gamma is folded into its weight).
//   kEpiSwiGLU              act = silu(r g) * (r u): the gate and up
//                           accumulators of the same 128 output columns share
//                           one N=256 MMA (B tile = 128 gate rows ++ 128 up rows);
//                           two columns per instruction on the packed f32x2 pipe.
//   kEpiSwiGLUSave          SwiGLU that also stores the pre-activations G || U
//                           (the "matrix block store" of the write-up's "five
//                           blocks"), for the backward.
//   kEpiGradNorm            backward: dY = acc stored, with the RMSNorm
//                           backward's row sums sum_j gamma_j dY_j H_j (H loaded)
//   kEpiSwiGLUBwd           backward: acc = dAct; dG, dU from the loaded G, U
// The row-scale program optionally scales columns (col_scale) and applies RoPE
// to the leading columns.  E4M3 operands: acc is multiplied by the per-tensor
// scales of A and B first.  bf16 operands may be MN-major (stored transposed,
// the output dimension contiguous), for the backward's transposed products.
//
// Two-phase launch (the whole GEMM -> RMSNorm -> GEMM block in one persistent
// kernel): the tile sequence is every residual-GEMM tile (phase A), then every
// tile of the consuming row-scale or SwiGLU GEMM (phase B, its r reduced from
// P in the epilogue).  A phase-B tile of row band m waits until every phase-A
// tile of band m has stored its h and P (a per-band counter in global memory,
// released after the stores complete, acquired before the TMA loads of h), so
// the consuming GEMM fills the SMs the residual GEMM's last wave leaves idle.
// All phase-A tiles precede all phase-B tiles in every CTA's walk and the grid
// is co-resident, so the waits cannot form a cycle.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <type_traits>

#include "coda_internal.h"
#include "fp8_e4m3.cuh"
#include "sm103_ptx.cuh"

namespace coda {

// Tuning of the legacy raster (kept for the backward's MN-major programs and
// selectable with CODA_RASTER=legacy): rows of one band of consecutive tiles
// walking the band's M-tiles before moving right, for the SwiGLU programs and
// for the others; both operands loaded with the evict-last L2 policy.
#ifndef CODA_RASTER_ROWS
#define CODA_RASTER_ROWS 2048
#endif
#ifndef CODA_RASTER_ROWS_SWIGLU
#define CODA_RASTER_ROWS_SWIGLU 4096
#endif

// Per-translation-unit device status word (timeouts), read back and cleared
// by the TU's read_clear_status_* function.
namespace {
__device__ unsigned g_status;
}

constexpr int kNoPhase = -1;

// Programs whose B tile is gate rows ++ up rows (N = 128 + 128).
__host__ __device__ constexpr bool is_swiglu(int epi) { return epi == kEpiSwiGLU || epi == kEpiSwiGLUSave; }
// Rows of one legacy raster band of a program's tiles.
__host__ __device__ constexpr int raster_rows(int epi) {
  return is_swiglu(epi) ? CODA_RASTER_ROWS_SWIGLU : CODA_RASTER_ROWS;
}

// Order of one phase's output tiles and the L2 policy of its operand loads.
// Consecutive tile indices walk `group` tiles along one dimension before
// stepping along the other: M-major bands (group M-tiles down a column, then
// the next column) keep the band's A panels in L2 while the B panels stream
// past; N-major bands (group N-tiles along a row, then the next row) keep the
// band's B panels (the weights) and stream A.  The kept operand is loaded
// evict-last, the streamed one with the streaming policy.
struct Raster {
  int group;    // tiles per band along the banded dimension (>= 1)
  int n_major;  // 1: bands of N-tiles, rows walked in order
  int keep;     // 0: keep A, stream B; 1: keep B, stream A; 2: both evict-last (legacy)
};

template <int KIND, int EPI_A, int EPI_B, int STAGES_, int NSLOTS_, int CG_ = 1, bool A_MN_ = false,
          bool B_MN_ = false, int QUANT_ = 0>
struct GemmCfg {
  static constexpr int kKind = KIND;
  // FP8 one-launch block: 1 = h quantised between the phases; 2 = phase A's
  // A operand quantised first as well.  Quantiser warps 7.. do both.
  static constexpr int QUANT = QUANT_;
  static constexpr bool FP8_BLOCK = QUANT_ > 0;
  static constexpr int NUM_QUANT_WARPS = FP8_BLOCK ? 4 : 0;
  // MN-major operands: A stored [K, M] (m contiguous) / B stored [K, N], loaded
  // as 64-element-wide TMA boxes of BK k-rows each
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  static constexpr int kEpiA = EPI_A;         // program of the (first) phase
  static constexpr int kEpiB = EPI_B;         // program of the second phase, or kNoPhase
  static constexpr bool TWO_PHASE = EPI_B != kNoPhase;
  // warp 6 owns the slot ring: programs that read a tile of another tensor
  static constexpr bool HAS_LOADER =
      EPI_A == kEpiResidualPartialRms || EPI_A == kEpiGradNorm || EPI_A == kEpiSwiGLUBwd;
  // slots one output box occupies: SwiGLU backward reads G and U and writes dG and dU
  __host__ __device__ static constexpr int slots_per_box(int epi) {
    return epi == kEpiSwiGLUBwd ? 2 : (epi == kEpiSwiGLUSave ? 3 : 1);
  }
  static constexpr int CG = CG_;              // CTAs per MMA (cta_group::1 or ::2)
  static constexpr int BM = 128;              // accumulator rows per CTA
  static constexpr int TILE_M = BM * CG;      // output rows per tile (per CTA pair)
  static constexpr int BN = 256;              // MMA N (SwiGLU: 128 gate + 128 up)
  static constexpr int STAGES = STAGES_;
  static constexpr int NSLOTS = NSLOTS_;
  static constexpr int ELEM = KIND == kKindBF16 ? 2 : (KIND == kKindTF32 ? 4 : 1);
  static constexpr int BK = 128 / ELEM;     // elements per k-block (one 128-byte swizzle row)
  static constexpr int UMMA_K = 32 / ELEM;  // K of one tcgen05.mma (32 bytes)
  static constexpr int K_STEPS = BK / UMMA_K;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_ROWS = BN / CG;    // B rows held by this CTA
  static constexpr int B_BYTES = B_ROWS * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // this CTA's bytes per stage
  // output columns per tile of a program
  __host__ __device__ static constexpr int out_cols(int epi) { return is_swiglu(epi) ? BN / 2 : BN; }
  // rows of one B TMA box: SwiGLU with one CTA loads gate and up halves
  // separately; with a pair, each CTA loads one of them whole
  __host__ __device__ static constexpr int b_box_rows(int epi) { return (is_swiglu(epi) && CG == 1) ? BN / 2 : B_ROWS; }
  static constexpr int OUT_ELEM = KIND == kKindTF32 ? 4 : 2;  // fp32 out for tf32, else bf16
  static constexpr int BOX_COLS = 128 / OUT_ELEM;             // output columns per 128-byte box
  static constexpr int NC32 = BOX_COLS / 32;  // 32-column TMEM loads per box (per operand half)
  static constexpr int CHUNK_COLS = 16 / OUT_ELEM;  // columns per 16-byte chunk of a box row
  static constexpr int SLOT_BYTES = BM * 128;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int NUM_EPI_THREADS = 128;
  static constexpr int NUM_THREADS = (HAS_LOADER ? 224 : 192) + 32 * NUM_QUANT_WARPS;
  static constexpr int QUANT_WARP0 = 7;
  // shared memory: [A stages][B stages][slots][barriers][tmem slot, abort flag]
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_SLOTS = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BARS = OFF_SLOTS + NSLOTS * SLOT_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * NSLOTS + 1;
  static constexpr int SMEM_BYTES = OFF_BARS + NUM_BARS * 8 + 16 + 1024;  // + slack for 1 KB alignment
  static_assert(CG == 1 || CG == 2, "CTA group");
  static_assert(NSLOTS >= 2 * slots_per_box(EPI_A) || HAS_LOADER, "output staging needs two boxes of slots");
  static_assert(!TWO_PHASE || (EPI_A == kEpiResidualPartialRms && (EPI_B == kEpiRowScale || EPI_B == kEpiSwiGLU)),
                "a two-phase launch is residual GEMM -> row-scale or SwiGLU GEMM");
  static_assert(TMEM_COLS == 512, "two 256-column accumulators");
  static_assert((BN / 2) % BOX_COLS == 0 && BOX_COLS % 32 == 0, "box tiling");
  static_assert(kPartialCols % BOX_COLS == 0 && BN % kPartialCols == 0, "partial groups");
  static_assert(NSLOTS >= 2, "slot ring");
  static_assert(SMEM_BYTES <= 232448, "exceeds 227 KB of shared memory");
  static constexpr uint32_t FMT = KIND == kKindBF16 ? 1u : (KIND == kKindTF32 ? 2u : 0u);
  static constexpr int MN_BOX = 64;                  // MN elements per MN-major box (128 bytes of bf16)
  static constexpr int MN_BOX_BYTES = MN_BOX * 128;  // BK k-rows of 128 bytes
  static_assert(!(A_MN || B_MN) || (KIND == kKindBF16 && !TWO_PHASE), "MN-major operands: bf16, one phase");
  static_assert((EPI_A != kEpiGradNorm && EPI_A != kEpiSwiGLUBwd) || (KIND == kKindBF16 && NSLOTS % 2 == 0),
                "backward programs: bf16, an even slot ring");
  static_assert(!FP8_BLOCK || (KIND == kKindE4M3 && TWO_PHASE && HAS_LOADER), "FP8 blocks: e4m3, two phases");
  static constexpr uint32_t IDESC = make_idesc(FMT, FMT, TILE_M, BN, A_MN, B_MN);
};

// Elements of one pass of a quantiser warp: 32 lanes x 6 groups of 16.
constexpr int kQuantGroups = 6;
constexpr int64_t kQuantPass = 32 * 16 * kQuantGroups;
// Passes per chunk, the unit that is fenced and counted into its band.  The
// fence waits for the warp's stores to land; paid once per pass, it kept the
// quantiser warps waiting for most of their time (an in-launch pass over the
// 8B chain's act ran 4.6x slower than the standalone quantise kernel), so a
// chunk of several passes pays it once.  16 measured fastest of 1, 2, 4, 8,
// 16; larger chunks make a band complete later.
#ifndef CODA_QUANT_PASSES
#define CODA_QUANT_PASSES 16
#endif
constexpr int kQuantPasses = CODA_QUANT_PASSES;
constexpr int64_t kQuantChunk = kQuantPasses * kQuantPass;
// Chunks per row band of band_rows rows and `cols` columns (the last band
// counts as many, its chunks past row M being empty).
__host__ __device__ inline int quant_chunks_per_band(int band_rows, int cols) {
  return static_cast<int>((static_cast<int64_t>(band_rows) * cols + kQuantChunk - 1) / kQuantChunk);
}

// One quantiser warp's share of a bf16 [M, cols] tensor -> e4m3 bytes: chunk
// j (band j / cpb) for j = w, w + nw, ..., pass by pass; each chunk's bytes
// are made visible (to the TMA loads of other CTAs too) before its band's
// counter is released.  Software-pipelined: the loads of the next pass are in
// flight while the current one is converted and stored.  cols is a multiple
// of 16, so a group of 16 elements never crosses a row band's end.  Returns
// false if the launch was aborted.
struct QuantChunk {
  int64_t e0, e_end, band;  // first element of this lane, end of its band, band
};
// Pass p of chunk j.
__device__ __forceinline__ QuantChunk quant_chunk(int64_t j, int p, int cpb, int64_t band_elems, int64_t total) {
  const int lane = threadIdx.x & 31;
  const int64_t b = j / cpb;
  const int64_t e_band = b * band_elems;
  return {e_band + (j - b * cpb) * kQuantChunk + p * kQuantPass + 16 * lane, min(e_band + band_elems, total), b};
}
// The bf16 source is read once: streaming loads (evict first), so the
// stream does not push the GEMM's operand panels out of L2.
#ifndef CODA_QUANT_STREAMING
#define CODA_QUANT_STREAMING 1
#endif
__device__ __forceinline__ uint4 quant_ld(const uint4* p) {
#if CODA_QUANT_STREAMING
  return __ldcs(p);
#else
  return __ldcg(p);
#endif
}
__device__ __forceinline__ void quant_load(const __nv_bfloat16* __restrict__ src, const QuantChunk& c,
                                           uint4 (&v)[kQuantGroups][2]) {
#pragma unroll
  for (int g = 0; g < kQuantGroups; ++g) {
    const int64_t e = c.e0 + 512 * g;
    if (e < c.e_end) {
      const uint4* p = reinterpret_cast<const uint4*>(src + e);
      v[g][0] = quant_ld(p);
      v[g][1] = quant_ld(p + 1);
    }
  }
}
template <bool FAST>
__device__ __forceinline__ bool quantize_bands(const __nv_bfloat16* __restrict__ src, uint8_t* __restrict__ dst,
                                               int M, int cols, int band_rows, float s, float inv,
                                               unsigned* ready, int w, int nw, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int64_t band_elems = static_cast<int64_t>(band_rows) * cols;
  const int cpb = quant_chunks_per_band(band_rows, cols);
  const int64_t total = static_cast<int64_t>(M) * cols;
  const int64_t n_chunks = static_cast<int64_t>((M + band_rows - 1) / band_rows) * cpb;
  if (w >= n_chunks) return true;
  uint4 cur[kQuantGroups][2], nxt[kQuantGroups][2];
  int64_t j = w;
  int p = 0;
  QuantChunk c = quant_chunk(j, 0, cpb, band_elems, total);
  quant_load(src, c, cur);
  for (;;) {
    if (*abort_flag) return false;
    // the next pass: of this chunk, else the first of this warp's next chunk
    const bool last_pass = p == kQuantPasses - 1;
    const int64_t jn = last_pass ? j + nw : j;
    const int pn = last_pass ? 0 : p + 1;
    const bool more = jn < n_chunks;  // always true before a chunk's last pass
    QuantChunk cn = c;
    if (more) {
      cn = quant_chunk(jn, pn, cpb, band_elems, total);
      quant_load(src, cn, nxt);
    }
#pragma unroll
    for (int g = 0; g < kQuantGroups; ++g) {
      const int64_t e = c.e0 + 512 * g;
      if (e < c.e_end) {
        float f[16];
        bf16x16_to_float(cur[g][0], cur[g][1], f);
        *reinterpret_cast<uint4*>(dst + e) = e4m3x16<FAST>(f, s, inv);
      }
    }
    if (last_pass) {
      // the chunk's codes, then its band's counter: generic stores read by TMA loads
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) red_release_gpu_add(ready + c.band, 1u);
    }
    if (!more) break;
#pragma unroll
    for (int g = 0; g < kQuantGroups; ++g) {
      cur[g][0] = nxt[g][0];
      cur[g][1] = nxt[g][1];
    }
    c = cn;
    j = jn;
    p = pn;
  }
  return true;
}

struct TileCoord {
  int m, n;
};

// Grouped raster: consecutive tile indices walk `group` M-tiles down one
// column of output tiles before moving right (or, N-major, `group` N-tiles
// along one row before moving down), so the CTAs in flight share a few A and
// B panels in L2.
__host__ __device__ __forceinline__ TileCoord tile_coord(int t, int m_tiles, int n_tiles, int group,
                                                         int n_major = 0) {
  if (n_major) {
    const int per_group = group * m_tiles;
    const int g = t / per_group;
    const int first_n = g * group;
    const int gn = min(group, n_tiles - first_n);
    const int local = t - g * per_group;
    return {local / gn, first_n + local % gn};
  }
  const int per_group = group * n_tiles;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gm = min(group, m_tiles - first_m);
  const int local = t - g * per_group;
  return {first_m + local % gm, local / gm};
}

// Position of tile index t in the launch's walk: phase A tiles first.
struct Tile {
  int phase;  // 0 = A, 1 = B
  int m, n;
};
__host__ __device__ __forceinline__ Tile tile_at(int t, int m_tiles, int n_tiles_a, int n_tiles_b, Raster ra,
                                                  Raster rb) {
  const int num_a = m_tiles * n_tiles_a;
  if (t < num_a) {
    const TileCoord c = tile_coord(t, m_tiles, n_tiles_a, ra.group, ra.n_major);
    return {0, c.m, c.n};
  }
  const TileCoord c = tile_coord(t - num_a, m_tiles, n_tiles_b, rb.group, rb.n_major);
  return {1, c.m, c.n};
}

// The k-th tile index of unit u (a CTA or a CTA pair) out of U units, or a
// value >= n_a + n_b once u has no tiles left.  Phase-A tiles are dealt round
// robin, so the first r_a = n_a mod U units hold one more of them.  A phase-A
// tile costs about `d` phase-B tiles (the ratio of their k-blocks), so those
// units sit out the first d rounds of phase B, which go round robin to the
// other units; the rest of phase B is dealt round robin to every unit.  Each
// unit then ends with about the same number of k-blocks, and consecutive
// indices still run side by side (the raster's L2 reuse).  Every unit walks
// all its phase-A tiles before any phase-B tile.  One-phase launches (n_b = 0)
// get the plain round robin u, u + U, u + 2U, ...
__host__ __device__ inline int walk_tile(int u, int k, int U, int n_a, int n_b, int d) {
  const int q_a = n_a / U, r_a = n_a % U;
  const int others = U - r_a;
  // plain round robin when phase A divides evenly, when a phase-A tile costs
  // about one phase-B tile (the round robin then already hands the first
  // phase-B round to the units without the extra phase-A tile), or when there
  // is not one whole phase-B round
  if (r_a == 0 || d <= 1 || n_b < others) return u + k * U;
  const int own_a = q_a + (u < r_a ? 1 : 0);
  if (k < own_a) return u + k * U;
  int kb = k - own_a;
  const int rounds = min(d, n_b / others);  // whole head rounds only
  const int head = rounds * others;
  if (u >= r_a) {
    if (kb < rounds) return n_a + (u - r_a) + kb * others;
    kb -= rounds;
  }
  const int j = head + u + kb * U;
  return n_a + (j < n_b ? j : n_b);
}

// sigmoid of two values: 1 / (1 + e^-x), with e^-x = 2^(-x log2 e) (change of
// base) and the quotient as a reciprocal.  For x -> -inf the denominator
// overflows and its reciprocal is 0; for x -> +inf it is 1.
__device__ __forceinline__ float2 sigmoid2(float2 x) {
  constexpr float kNegLog2e = -1.44269504088896341f;
  const float2 t = fmul2(x, make_float2(kNegLog2e, kNegLog2e));
  const float2 den = fadd2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.0f, 1.0f));
  return make_float2(rcp_approx(den.x), rcp_approx(den.y));
}
// silu(x) = x * sigmoid(x), two values.
__device__ __forceinline__ float2 silu2(float2 x) { return fmul2(x, sigmoid2(x)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// sin and cos of the RoPE angle phi = p * base^(-j / half), with log2b =
// log2(base) / half.  phi is reduced by whole turns with 2*pi split into a
// float head and its remainder (Cody and Waite's two-constant reduction), so
// the fast sincos sees |x| <= pi; the error is dominated by the fp32 product
// p * inv_freq (about 1.2e-7 * phi radians).
__device__ __forceinline__ void rope_sincos(float p, int j, float log2b, float& sn, float& cn) {
  constexpr float kTwoPiHi = 6.28318548202514648f;    // 2*pi rounded to float (above 2*pi)
  constexpr float kTwoPiLo = -1.74845553146951832e-7f;  // 2*pi - kTwoPiHi
  const float phi = p * exp2f(-static_cast<float>(j) * log2b);
  const float k = rintf(phi * 0.159154943091895336f);  // whole turns
  const float x = fmaf(-k, kTwoPiLo, fmaf(-k, kTwoPiHi, phi));
  __sincosf(x, &sn, &cn);
}

// Byte offset of 16-byte chunk `c` (0..7) of row `row` inside one 128B-swizzled
// box of 128 rows x 128 B: the chunk index is XORed with the row's position in
// its 8-row atom, as TMA lays it out.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

// Let every TMA load this thread issued into a ring land before exit: stage
// s received loads in rounds 0..(issued-1-s)/N; wait for the last one.
__device__ __forceinline__ void drain_ring(uint64_t* full, int n_stages, uint32_t issued, volatile int* abort_flag) {
  for (int s = 0; s < n_stages; ++s) {
    if (issued > static_cast<uint32_t>(s)) {
      const uint32_t round = (issued - 1u - static_cast<uint32_t>(s)) / static_cast<uint32_t>(n_stages);
      (void)mbar_wait(&full[s], round & 1u, abort_flag, &g_status, false);
    }
  }
}

// Band dependency of a two-phase launch: spin (bounded) until the counter
// reaches `target`, with acquire semantics at GPU scope.
__device__ __forceinline__ bool wait_band(const unsigned* ctr, unsigned target, volatile int* abort_flag) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(ctr) >= target) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > CODA_WAIT_TIMEOUT_NS) {
        *abort_flag = 1;
        atomicOr(&g_status, kDevTimeout);
        return false;
      }
    }
  }
}

// Operands of one phase.
struct PhaseArgs {
  int N_out, K;
  EpiParams ep;
  Raster raster;  // tile order and L2 policy of the operand loads
  int stream_first;  // the streamed operand is loaded evict-first (else evict-normal)
};

template <class C>
__global__ void __launch_bounds__(C::NUM_THREADS, 1)
    gemm_epilogue_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmR,
                         const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmA_b,
                         const __grid_constant__ CUtensorMap tmB_b, const __grid_constant__ CUtensorMap tmB2_b,
                         const __grid_constant__ CUtensorMap tmD_b, int M, PhaseArgs pa, PhaseArgs pb,
                         unsigned* band_ready, const QuantArgs qa) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::OFF_B;
  uint8_t* slots = smem + C::OFF_SLOTS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BARS);
  uint64_t* full = bars;
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* r_full = acc_empty + 2;
  uint64_t* r_empty = r_full + C::NSLOTS;
  uint64_t* mma_drain = r_empty + C::NSLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pair (CG = 2): rank 0 issues the MMAs for both; each CTA loads and
  // stores its own 128 rows and half of the B tile
  const uint32_t cta_rank = C::CG == 2 ? cluster_ctarank() : 0u;
  const bool mma_cta = cta_rank == 0;
  const int unit = blockIdx.x / C::CG;     // tile-walking unit (a CTA or a CTA pair)
  const int n_units = gridDim.x / C::CG;
  const int m_tiles = (M + C::TILE_M - 1) / C::TILE_M;
  const int n_tiles_a = (pa.N_out + C::out_cols(C::kEpiA) - 1) / C::out_cols(C::kEpiA);
  const int n_tiles_b = C::TWO_PHASE ? (pb.N_out + C::out_cols(C::kEpiB) - 1) / C::out_cols(C::kEpiB) : 0;
  const int num_tiles = m_tiles * (n_tiles_a + n_tiles_b);
  // phase-B rounds that units holding an extra phase-A tile sit out.  An FP8
  // block's phase B starts on every unit at once, after the grid-wide amax
  // barrier, so there the phase-B tiles go plain round robin (sitting out
  // rounds would leave the other units with 3-4 more tiles at the end).
  const int b_rounds = (C::TWO_PHASE && !C::FP8_BLOCK)
                           ? ((pa.K + C::BK - 1) / C::BK + ((pb.K + C::BK - 1) / C::BK) / 2) /
                                 max(1, (pb.K + C::BK - 1) / C::BK)
                           : 0;
  auto walk = [&](int k) { return walk_tile(unit, k, n_units, m_tiles * n_tiles_a, m_tiles * n_tiles_b, b_rounds); };
  // a band is ready for phase B when every phase-A tile of it (one increment
  // per CTA) has stored h and P
  const unsigned band_target = static_cast<unsigned>(n_tiles_a * C::CG);
  // FP8 blocks: CTAs past phase A, bands of e4m3 h and of e4m3 A complete
  [[maybe_unused]] unsigned* const a_done = band_ready + m_tiles + 1;
  [[maybe_unused]] unsigned* const qh_ready = band_ready + m_tiles + 2;
  [[maybe_unused]] unsigned* const qa_ready = band_ready + 2 * m_tiles + 2;
  [[maybe_unused]] const unsigned qh_target = static_cast<unsigned>(quant_chunks_per_band(C::TILE_M, pa.N_out));
  [[maybe_unused]] const unsigned qa_target = static_cast<unsigned>(quant_chunks_per_band(C::TILE_M, pa.K));
  [[maybe_unused]] const int num_a_tiles = m_tiles * n_tiles_a;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], C::CG * C::NUM_EPI_THREADS / 32);
    }
    for (int s = 0; s < C::NSLOTS; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 1);
    }
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (is_swiglu(C::kEpiA)) tma_prefetch_desc(&tmB2);
    if constexpr (C::kEpiA == kEpiSwiGLUSave) tma_prefetch_desc(&tmD_b);
    if constexpr (C::HAS_LOADER) tma_prefetch_desc(&tmR);
    tma_prefetch_desc(&tmD);
    if constexpr (C::TWO_PHASE) {
      tma_prefetch_desc(&tmA_b);
      tma_prefetch_desc(&tmB_b);
      if constexpr (C::kEpiB == kEpiSwiGLU) tma_prefetch_desc(&tmB2_b);
      tma_prefetch_desc(&tmD_b);
    }
  }
  if (warp == 1) {
    tmem_alloc<C::CG>(tmem_slot, C::TMEM_COLS);
    tmem_relinquish<C::CG>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::CG == 2) cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  // Everything above overlapped the previous kernel's tail; from here on we
  // read and write global memory that it may own.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer ----
    if (lane == 0) {
      // L2 policies: keep (evict-last) for the operand whose panels the band
      // reuses; the other operand is still shared by the band's tiles in
      // flight, so it is loaded with the normal policy (or evict-first)
      const uint64_t pol_keep = l2_policy_evict_last();
      const uint64_t pol_stream = pa.stream_first ? l2_policy_evict_first() : l2_policy_evict_normal();
      auto pol_a_of = [&](const Raster& r) { return r.keep == 1 ? pol_stream : pol_keep; };
      auto pol_b_of = [&](const Raster& r) { return r.keep == 0 ? pol_stream : pol_keep; };
      // the stage's completion is counted on the MMA CTA's barrier
      const uint32_t full0 = C::CG == 2 ? mapa_shared(smem_u32(full), 0) : 0u;
      // Every box of k-block kb of tile tl that this CTA loads: f(map, x, y,
      // is_b, byte offset in the stage's A or B buffer).
      auto boxes = [&](const Tile& tl, int kb, auto&& f) {
        const bool pB = C::TWO_PHASE && tl.phase == 1;
        const CUtensorMap* mA = pB ? &tmA_b : &tmA;
        const CUtensorMap* mB = pB ? &tmB_b : &tmB;
        [[maybe_unused]] const CUtensorMap* mB2 = pB ? &tmB2_b : &tmB2;
        [[maybe_unused]] const bool swiglu = pB ? is_swiglu(C::kEpiB) : is_swiglu(C::kEpiA);
        const int kx = kb * C::BK;
        const int a_row = tl.m * C::TILE_M + static_cast<int>(cta_rank) * C::BM;
        if constexpr (C::A_MN) {
          // MN-major boxes: x = MN coordinate, y = k
#pragma unroll
          for (int i = 0; i < C::BM / C::MN_BOX; ++i) f(mA, a_row + i * C::MN_BOX, kx, false, i * C::MN_BOX_BYTES);
        } else {
          f(mA, kx, a_row, false, 0);
        }
        if constexpr (C::B_MN) {
          const int b_row = tl.n * C::BN + static_cast<int>(cta_rank) * C::B_ROWS;
#pragma unroll
          for (int i = 0; i < C::B_ROWS / C::MN_BOX; ++i) f(mB, b_row + i * C::MN_BOX, kx, true, i * C::MN_BOX_BYTES);
        } else if (swiglu) {
          if constexpr (C::CG == 1) {  // gate rows, then up rows
            f(mB, kx, tl.n * (C::BN / 2), true, 0);
            f(mB2, kx, tl.n * (C::BN / 2), true, (C::BN / 2) * 128);
          } else {  // rank 0: gate rows, rank 1: up rows
            f(cta_rank == 0 ? mB : mB2, kx, tl.n * C::B_ROWS, true, 0);
          }
        } else {
          f(mB, kx, tl.n * C::BN + static_cast<int>(cta_rank) * C::B_ROWS, true, 0);
        }
      };
      auto num_kb_of = [&](const Tile& tl) {
        return (((C::TWO_PHASE && tl.phase == 1) ? pb.K : pa.K) + C::BK - 1) / C::BK;
      };
      int stage = 0;
      uint32_t phase = 0, issued = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int t = walk(k);
        if (t >= num_tiles) break;
        const Tile tl = tile_at(t, m_tiles, n_tiles_a, n_tiles_b, pa.raster, pb.raster);
        const int num_kb = num_kb_of(tl);
        if (C::TWO_PHASE && tl.phase == 1) {
          // h and P of this band come from other CTAs of this launch (FP8:
          // the e4m3 copy of h, from the quantiser warps)
          if (!(C::FP8_BLOCK ? wait_band(&qh_ready[tl.m], qh_target, abort_flag)
                             : wait_band(&band_ready[tl.m], band_target, abort_flag)))
            break;
          fence_proxy_async_global();
        } else if (C::QUANT == 2 && qa.a != nullptr) {
          // the e4m3 copy of this band's A operand, quantised in this launch
          if (!wait_band(&qa_ready[tl.m], qa_target, abort_flag)) break;
          fence_proxy_async_global();
        }
        const Raster& rst = (C::TWO_PHASE && tl.phase == 1) ? pb.raster : pa.raster;
        const uint64_t pol_a = pol_a_of(rst), pol_b = pol_b_of(rst);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_status)) {
            ok = false;
            break;
          }
          uint8_t* a = sA + stage * C::A_BYTES;
          uint8_t* b = sB + stage * C::B_BYTES;
          if constexpr (C::CG == 1) {
            mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
            boxes(tl, kb, [&](const CUtensorMap* m, int x, int y, bool is_b, int off) {
              tma_load_2d((is_b ? b : a) + off, m, &full[stage], x, y, is_b ? pol_b : pol_a);
            });
          } else {
            // the MMA CTA expects both CTAs' bytes; the peer only issues its copies
            if (mma_cta) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
            const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
            boxes(tl, kb, [&](const CUtensorMap* m, int x, int y, bool is_b, int off) {
              tma_load_2d_pair((is_b ? b : a) + off, m, fb, x, y, is_b ? pol_b : pol_a);
            });
          }
          ++issued;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every load issued must land before the CTA may exit (for a pair, the
      // MMA CTA's ring counts both CTAs' copies)
      if (mma_cta) drain_ring(full, C::STAGES, issued, abort_flag);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer ----
    if (lane == 0 && mma_cta) {
      constexpr uint16_t kPair = C::CG == 2 ? 3 : 1;
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k, ++it) {
        const int t = walk(k);
        if (t >= num_tiles) break;
        const Tile tl = tile_at(t, m_tiles, n_tiles_a, n_tiles_b, pa.raster, pb.raster);
        const int num_kb = (((C::TWO_PHASE && tl.phase == 1) ? pb.K : pa.K) + C::BK - 1) / C::BK;
        const int buf = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait(&acc_empty[buf], use ^ 1u, abort_flag, &g_status)) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * C::BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, &g_status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_s = smem_u32(sA + stage * C::A_BYTES), b_s = smem_u32(sB + stage * C::B_BYTES);
          const uint64_t adesc = C::A_MN ? sdesc_mnmajor_sw128(a_s, C::MN_BOX_BYTES) : sdesc_kmajor_sw128(a_s);
          const uint64_t bdesc = C::B_MN ? sdesc_mnmajor_sw128(b_s, C::MN_BOX_BYTES) : sdesc_kmajor_sw128(b_s);
          // one MMA step along K: 32 bytes inside a K-major swizzle row (+2 in
          // the descriptor's 16-byte units), or UMMA_K rows of 128 bytes of an
          // MN-major tile (+UMMA_K * 8)
          constexpr uint64_t a_step = C::A_MN ? C::UMMA_K * 8u : 2u;
          constexpr uint64_t b_step = C::B_MN ? C::UMMA_K * 8u : 2u;
#pragma unroll
          for (int k = 0; k < C::K_STEPS; ++k)
            tc_mma<C::kKind, C::CG>(d_tmem, adesc + a_step * k, bdesc + b_step * k, C::IDESC, (kb | k) != 0);
          tc_commit<C::CG>(&empty[stage], kPair);  // both CTAs' stage is free again
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit<C::CG>(&acc_full[buf], kPair);
      }
      // every MMA issued must complete before TMEM is released
      tc_commit<C::CG>(mma_drain, 1);
      (void)mbar_wait(mma_drain, 0, abort_flag, &g_status, false);
    }
  } else if (warp == 6) {
    // ------------------------------------------------ slot ring (R boxes) ----
    // Residual boxes: TMA-load R into the slot.  Boxes of a second phase:
    // hand the free slot to the epilogue as output staging.
    if constexpr (C::HAS_LOADER) {
      if (lane == 0) {
        const uint64_t pol = l2_policy_evict_first();
        int slot = 0;
        uint32_t phase = 0, used = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int t = walk(k);
          if (t >= num_tiles) break;
          const Tile tl = tile_at(t, m_tiles, n_tiles_a, n_tiles_b, pa.raster, pb.raster);
          const bool pB = C::TWO_PHASE && tl.phase == 1;
          const int row0 = tl.m * C::TILE_M + static_cast<int>(cta_rank) * C::BM;
          if (row0 >= M) continue;  // this CTA's half of the tile is empty
          const int oc = pB ? C::out_cols(C::kEpiB) : C::out_cols(C::kEpiA);
          const int n_out = pB ? pb.N_out : pa.N_out;
          for (int b = 0; b < oc / C::BOX_COLS && ok; ++b) {
            const int col0 = tl.n * oc + b * C::BOX_COLS;
            if (col0 >= n_out) break;
            // SwiGLU backward: G's box, then U's box gu_off columns further
            for (int sb = 0; sb < C::slots_per_box(C::kEpiA); ++sb) {
              if (!mbar_wait(&r_empty[slot], phase ^ 1u, abort_flag, &g_status)) {
                ok = false;
                break;
              }
              if (pB) {
                mbar_arrive(&r_full[slot]);
              } else {
                mbar_arrive_expect_tx(&r_full[slot], C::SLOT_BYTES);
                tma_load_2d(slots + slot * C::SLOT_BYTES, &tmR, &r_full[slot], col0 + sb * pa.ep.gu_off, row0, pol);
              }
              ++used;
              if (++slot == C::NSLOTS) {
                slot = 0;
                phase ^= 1u;
              }
            }
          }
        }
        // every R load issued must land before exit (hand-overs complete at once)
        drain_ring(r_full, C::NSLOTS, used, abort_flag);
      }
    }
  } else if (warp >= C::QUANT_WARP0) {
    // ---------------------------------------------- quantiser (FP8 blocks) ----
    // Phase A's A operand first (if the launch quantises it), then h once
    // every CTA is past phase A.  The warps of all CTAs share each tensor's
    // chunks round robin in band order, so bands complete roughly in order.
    if constexpr (C::FP8_BLOCK) {
      const int w = static_cast<int>(blockIdx.x) * C::NUM_QUANT_WARPS + (warp - C::QUANT_WARP0);
      const int nw = static_cast<int>(gridDim.x) * C::NUM_QUANT_WARPS;
      auto quantize = [&](const void* src, uint8_t* dst, int cols, float s, unsigned* ready) {
        const auto* x = static_cast<const __nv_bfloat16*>(src);
        return e4m3_fast_scale(s)
                   ? quantize_bands<true>(x, dst, M, cols, C::TILE_M, s, __frcp_rn(s), ready, w, nw, abort_flag)
                   : quantize_bands<false>(x, dst, M, cols, C::TILE_M, s, 0.0f, ready, w, nw, abort_flag);
      };
      bool qok = true;
      if (C::QUANT == 2 && qa.a != nullptr) {
        const float s = e4m3_scale(*qa.amax_a);
        if (w == 0 && lane == 0) *qa.scale_a = s;
        qok = quantize(qa.a, qa.aq, pa.K, s, qa_ready);
      }
      // h: every CTA has stored its phase-A tiles and folded |h| into amax_h
      if (qok && wait_band(a_done, gridDim.x, abort_flag)) {
        const float s = e4m3_scale(*reinterpret_cast<volatile const float*>(qa.amax_h));
        if (w == 0 && lane == 0) *qa.scale_h = s;
        (void)quantize(qa.h, qa.hq, pa.N_out, s, qh_ready);
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue ----
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    const bool leader = (warp == 2 && lane == 0);
    // the MMA CTA's accumulator-empty barrier (a remote arrive for the peer)
    const uint32_t acc_empty0 = C::CG == 2 ? mapa_shared(smem_u32(acc_empty), 0) : 0u;
    float amax = 0.0f;
    int slot = 0;
    uint32_t sphase = 0;
    int it = 0;
    bool ok = true;

    // One tile of program EPI: TMEM -> program -> slot -> TMA store, box by box.
    auto run_tile = [&](auto epi_tag, const Tile& tl, const PhaseArgs& ph, const CUtensorMap* mD, int buf) {
      constexpr int EPI = decltype(epi_tag)::value;
      constexpr int OUT_COLS = C::out_cols(EPI);
      constexpr int NUM_BOXES = OUT_COLS / C::BOX_COLS;
      const EpiParams& ep = ph.ep;
      const int N_out = ph.N_out;
      float sab = 1.0f, sab2 = 1.0f;
      if constexpr (C::kKind == kKindE4M3) {
        float sa;
        if constexpr (C::FP8_BLOCK) {
          if (tl.phase == 1) {
            // h's scale: amax_h is final once every CTA is past phase A
            (void)wait_band(a_done, gridDim.x, abort_flag);
            sa = e4m3_scale(*reinterpret_cast<volatile const float*>(qa.amax_h));
          } else {
            sa = qa.a != nullptr ? e4m3_scale(*qa.amax_a) : *ep.scale_a;
          }
        } else {
          sa = *ep.scale_a;
        }
        sab = sa * *ep.scale_b;
        if constexpr (is_swiglu(EPI)) sab2 = sa * *ep.scale_b2;
      }
      const int row0 = tl.m * C::TILE_M + static_cast<int>(cta_rank) * C::BM;
      const int row = row0 + row_in_tile;
      const bool half_valid = row0 < M;  // uniform over the CTA
      float rs = 1.0f;
      if constexpr (EPI != kEpiResidualPartialRms) {
        if (ep.P_in != nullptr) {
          // the auxiliary reduction, folded in: this row's partials -> r
          if constexpr (C::FP8_BLOCK) (void)wait_band(a_done, gridDim.x, abort_flag);  // acquire P (all bands)
          else if constexpr (C::TWO_PHASE) (void)wait_band(&band_ready[tl.m], band_target, abort_flag);  // acquire P
          rs = row < M ? row_rstd(ep.P_in + static_cast<int64_t>(row) * ep.T_in, ep.T_in, ep.n_norm, ep.eps) : 0.0f;
          if (ep.r_out != nullptr && tl.n == 0 && row < M) ep.r_out[row] = rs;
        } else if (ep.r != nullptr) {
          rs = row < M ? ep.r[row] : 0.0f;
        }
      }
      const float sg = rs * sab, su = rs * sab2;
      // row-scale program with RoPE: this row's position
      bool rope_on = false;
      float rope_p = 0.0f;
      if constexpr (EPI == kEpiRowScale) {
        if (ep.rope_cols > 0 && row < M) {
          rope_on = true;
          rope_p = static_cast<float>(ep.rope_pos != nullptr ? ep.rope_pos[row] : row % ep.rope_seq);
        }
      }
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * C::BN);
      auto release_acc = [&]() {
        // last TMEM read of this tile: hand the accumulator back to the MMA warp
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if constexpr (C::CG == 2) mbar_arrive_cluster(acc_empty0 + static_cast<uint32_t>(buf) * 8u);
          else mbar_arrive(&acc_empty[buf]);
        }
      };
      if (!half_valid) {
        release_acc();
        // nothing to store, but the band still counts this CTA's share of the tile
        if constexpr (C::TWO_PHASE && !C::FP8_BLOCK && EPI == kEpiResidualPartialRms)
          if (leader) red_release_gpu_add(&band_ready[tl.m], 1u);
        return;
      }
      float ss = 0.0f;
#pragma unroll 1
      for (int b = 0; b < NUM_BOXES; ++b) {
        const int col0 = tl.n * OUT_COLS + b * C::BOX_COLS;
        if (col0 >= N_out) break;  // uniform over the CTA
        uint32_t g[C::NC32][32];
        uint32_t u[is_swiglu(EPI) ? C::NC32 : 1][32];
#pragma unroll
        for (int i = 0; i < C::NC32; ++i) tmem_ld32(t_row + b * C::BOX_COLS + 32 * i, g[i]);
        if constexpr (is_swiglu(EPI)) {
#pragma unroll
          for (int i = 0; i < C::NC32; ++i) tmem_ld32(t_row + C::BN / 2 + b * C::BOX_COLS + 32 * i, u[i]);
        }
        tmem_wait_ld(g[0]);
#pragma unroll
        for (int i = 1; i < C::NC32; ++i) tmem_touch(g[i]);
        if constexpr (is_swiglu(EPI)) {
#pragma unroll
          for (int i = 0; i < C::NC32; ++i) tmem_touch(u[i]);
        }
        if (b == NUM_BOXES - 1 || col0 + C::BOX_COLS >= N_out) release_acc();
        constexpr int SPB = C::slots_per_box(EPI);
        bool got = true;
        if constexpr (C::HAS_LOADER) {
#pragma unroll
          for (int sb = 0; sb < SPB; ++sb) got = got && mbar_wait(&r_full[slot + sb], sphase, abort_flag, &g_status);
        }
        uint8_t* sp = slots + slot * C::SLOT_BYTES;
        uint8_t* sp2 = sp + (SPB - 1) * C::SLOT_BYTES;  // SwiGLU backward: U in, dU out
        if (got) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float o[C::CHUNK_COLS];
            float gs[EPI == kEpiSwiGLUSave ? C::CHUNK_COLS : 1], us[EPI == kEpiSwiGLUSave ? C::CHUNK_COLS : 1];
            if constexpr (is_swiglu(EPI)) {
              // two columns per step on the packed fp32 pipe
#pragma unroll
              for (int e = 0; e < C::CHUNK_COLS; e += 2) {
                const int j = c * C::CHUNK_COLS + e;
                const float2 G = fmul2(make_float2(__uint_as_float(g[j >> 5][j & 31]),
                                                   __uint_as_float(g[(j + 1) >> 5][(j + 1) & 31])),
                                       make_float2(sg, sg));
                const float2 U = fmul2(make_float2(__uint_as_float(u[j >> 5][j & 31]),
                                                   __uint_as_float(u[(j + 1) >> 5][(j + 1) & 31])),
                                       make_float2(su, su));
                const float2 O = fmul2(silu2(G), U);
                o[e] = O.x;
                o[e + 1] = O.y;
                if constexpr (EPI == kEpiSwiGLUSave) {
                  gs[e] = G.x;
                  gs[e + 1] = G.y;
                  us[e] = U.x;
                  us[e + 1] = U.y;
                }
              }
            } else {
#pragma unroll
              for (int e = 0; e < C::CHUNK_COLS; ++e) {
                const int j = c * C::CHUNK_COLS + e;
                o[e] = __uint_as_float(g[j >> 5][j & 31]) * sg;
              }
            }
            if constexpr (EPI == kEpiSwiGLUSave) {
              // the pre-activations, for the backward: G to the second slot, U to the third
              uint32_t wg[4], wu[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                wg[e] = pack_bf16x2(gs[2 * e], gs[2 * e + 1]);
                wu[e] = pack_bf16x2(us[2 * e], us[2 * e + 1]);
              }
              *reinterpret_cast<uint4*>(sp + C::SLOT_BYTES + swz(row_in_tile, c)) = make_uint4(wg[0], wg[1], wg[2], wg[3]);
              *reinterpret_cast<uint4*>(sp + 2 * C::SLOT_BYTES + swz(row_in_tile, c)) =
                  make_uint4(wu[0], wu[1], wu[2], wu[3]);
            }
            if constexpr (EPI == kEpiRowScale) {
              if (ep.col_scale != nullptr) {  // diag(col_scale) on the right
                const int col = col0 + c * C::CHUNK_COLS;
#pragma unroll
                for (int e = 0; e < C::CHUNK_COLS; ++e) o[e] *= col + e < N_out ? __ldg(ep.col_scale + col + e) : 0.0f;
              }
            }
            if constexpr (EPI == kEpiRowScale) {
              const int col = col0 + c * C::CHUNK_COLS;
              if (rope_on && col < ep.rope_cols) {
                // RoPE on interleaved pairs; the chunk's CHUNK_COLS / 2 pairs are
                // consecutive frequencies j of one head (head_dim % CHUNK_COLS == 0)
                const int j0 = (col >> 1) % ep.rope_half;
#pragma unroll
                for (int e = 0; e < C::CHUNK_COLS / 2; ++e) {
                  float sn, cn;
                  rope_sincos(rope_p, j0 + e, ep.rope_log2b, sn, cn);
                  const float x = o[2 * e], y = o[2 * e + 1];
                  o[2 * e] = x * cn - y * sn;
                  o[2 * e + 1] = x * sn + y * cn;
                }
              }
            }
            void* p = sp + swz(row_in_tile, c);
            if constexpr (C::OUT_ELEM == 2 && EPI == kEpiGradNorm) {
              // stored dY, and sum_j gamma_j dY_j H_j over the stored values
              const uint4 hv = *reinterpret_cast<const uint4*>(p);
              const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
              const int col = col0 + c * C::CHUNK_COLS;
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                w[e] = pack_bf16x2(o[2 * e], o[2 * e + 1]);
                const float g0 = col + 2 * e < N_out ? __ldg(ep.col_scale + col + 2 * e) : 0.0f;
                const float g1 = col + 2 * e + 1 < N_out ? __ldg(ep.col_scale + col + 2 * e + 1) : 0.0f;
                ss += g0 * bf16_lo(w[e]) * bf16_lo(hw[e]) + g1 * bf16_hi(w[e]) * bf16_hi(hw[e]);
              }
              *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            } else if constexpr (C::OUT_ELEM == 2 && EPI == kEpiSwiGLUBwd) {
              // act = silu(G) U: dG = dAct U silu'(G), dU = dAct silu(G)
              void* p2 = sp2 + swz(row_in_tile, c);
              const uint4 gv = *reinterpret_cast<const uint4*>(p), uv = *reinterpret_cast<const uint4*>(p2);
              const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
              uint32_t wg[4], wu[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // two columns at a time: s = sigmoid(G), silu(G) = G s,
                // silu'(G) = s (1 + G (1 - s)) = s + silu(G) (1 - s)
                const float2 G = make_float2(bf16_lo(gw[e]), bf16_hi(gw[e]));
                const float2 U = make_float2(bf16_lo(uw[e]), bf16_hi(uw[e]));
                const float2 da = make_float2(o[2 * e], o[2 * e + 1]);
                const float2 s = sigmoid2(G);
                const float2 gs = fmul2(G, s);
                const float2 one_minus_s = ffma2(s, make_float2(-1.0f, -1.0f), make_float2(1.0f, 1.0f));
                const float2 dsilu = ffma2(gs, one_minus_s, s);
                const float2 dg = fmul2(fmul2(da, U), dsilu);
                const float2 du = fmul2(da, gs);
                wg[e] = pack_bf16x2(dg.x, dg.y);
                wu[e] = pack_bf16x2(du.x, du.y);
              }
              *reinterpret_cast<uint4*>(p) = make_uint4(wg[0], wg[1], wg[2], wg[3]);
              *reinterpret_cast<uint4*>(p2) = make_uint4(wu[0], wu[1], wu[2], wu[3]);
            } else if constexpr (C::OUT_ELEM == 2) {
              uint32_t w[4];
              if constexpr (EPI == kEpiResidualPartialRms) {
                const uint4 rv = *reinterpret_cast<const uint4*>(p);
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  w[e] = pack_bf16x2(bf16_lo(rw[e]) + o[2 * e], bf16_hi(rw[e]) + o[2 * e + 1]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(o[2 * e], o[2 * e + 1]);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // statistics of the values actually stored (bf16-rounded)
                const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
                if constexpr (EPI == kEpiResidualPartialRms) ss += lo * lo + hi * hi;
                if (ep.amax_out) amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
              }
              *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              float4 v = make_float4(o[0], o[1], o[2], o[3]);
              if constexpr (EPI == kEpiResidualPartialRms) {
                const float4 rv = *reinterpret_cast<const float4*>(p);
                v.x += rv.x;
                v.y += rv.y;
                v.z += rv.z;
                v.w += rv.w;
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
              }
              if (ep.amax_out)
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
              *reinterpret_cast<float4*>(p) = v;
            }
          }
          if constexpr (EPI == kEpiResidualPartialRms || EPI == kEpiGradNorm) {
            const int gcol = col0 + C::BOX_COLS;  // end column of this box
            if (gcol % kPartialCols == 0 || gcol >= N_out) {
              if (row < M) ep.P[static_cast<int64_t>(row) * ep.T + col0 / kPartialCols] = ss;
              ss = 0.0f;
              if constexpr (C::TWO_PHASE) __threadfence();  // P visible before the band's release
            }
          }
        }
        // shared slot -> global
        fence_proxy_async_smem();
        if (!named_bar_and(1, C::NUM_EPI_THREADS, got)) {
          ok = false;
          return;
        }
        if (leader) {
          tma_store_2d(mD, sp, col0, row0);
          if constexpr (EPI == kEpiSwiGLUBwd) tma_store_2d(mD, sp2, col0 + ep.gu_off, row0);
          if constexpr (EPI == kEpiSwiGLUSave) {
            tma_store_2d(&tmD_b, sp + C::SLOT_BYTES, col0, row0);
            tma_store_2d(&tmD_b, sp + 2 * C::SLOT_BYTES, col0 + ep.gu_off, row0);
          }
          tma_store_commit();
          tma_store_wait_read_all();  // slots readable again before anyone rewrites them
          if constexpr (C::HAS_LOADER) {
#pragma unroll
            for (int sb = 0; sb < SPB; ++sb) mbar_arrive(&r_empty[slot + sb]);
          }
        }
        slot += SPB;
        if (slot == C::NSLOTS) {
          slot = 0;
          sphase ^= 1u;
        }
      }
      if constexpr (C::TWO_PHASE && !C::FP8_BLOCK && EPI == kEpiResidualPartialRms) {
        // h of this tile is in global memory (and P, fenced above): release the band
        if (leader) {
          tma_store_wait_all();
          fence_proxy_async_global();
          red_release_gpu_add(&band_ready[tl.m], 1u);
        }
      }
    };

    // FP8 block: once this CTA's last phase-A tile is stored, fold its |h|
    // into amax_h and count the CTA past phase A (the quantiser warps of
    // every CTA wait for all of them)
    [[maybe_unused]] auto publish_phase_a = [&]() {
      if constexpr (C::FP8_BLOCK) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) atomicMax(reinterpret_cast<int*>(qa.amax_h), __float_as_int(amax));
        __threadfence();
        amax = 0.0f;  // from here on: phase B's output
        named_bar_sync(1, C::NUM_EPI_THREADS);
        if (leader) {
          tma_store_wait_all();
          fence_proxy_async_global();
          red_release_gpu_add(a_done, 1u);
        }
      }
    };
    if constexpr (C::FP8_BLOCK)
      if (walk(0) >= num_a_tiles) publish_phase_a();  // no phase-A tile in this CTA's walk
    for (int k = 0; ok; ++k, ++it) {
      const int t = walk(k);
      if (t >= num_tiles) break;
      const Tile tl = tile_at(t, m_tiles, n_tiles_a, n_tiles_b, pa.raster, pb.raster);
      const int buf = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      // one decision for all 128 threads, so no thread is left at a barrier
      if (!named_bar_and(1, C::NUM_EPI_THREADS, mbar_wait(&acc_full[buf], use, abort_flag, &g_status))) break;
      tc_fence_after_sync();
      if (C::TWO_PHASE && tl.phase == 1) {
        if constexpr (C::TWO_PHASE) run_tile(std::integral_constant<int, C::kEpiB>{}, tl, pb, &tmD_b, buf);
      } else {
        run_tile(std::integral_constant<int, C::kEpiA>{}, tl, pa, &tmD, buf);
        if constexpr (C::FP8_BLOCK)
          if (ok && walk(k + 1) >= num_a_tiles) publish_phase_a();
      }
    }
    // FP8 blocks publish phase A's amax above; the end publishes phase B's
    float* amax_dst = C::FP8_BLOCK ? pb.ep.amax_out : (pa.ep.amax_out ? pa.ep.amax_out : pb.ep.amax_out);
    if (amax_dst) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // non-negative floats order like their bit patterns; one program per
      // launch has an amax output (bf16 two-phase launches have none)
      if (lane == 0) atomicMax(reinterpret_cast<int*>(amax_dst), __float_as_int(amax));
    }
    if (leader) tma_store_wait_all();
  }

  // --------------------------------------------------------------- teardown ----
  tc_fence_before_sync();
  __syncthreads();
  // a pair leaves together: no CTA frees TMEM or shared memory that the
  // other's copies, MMAs or arrivals may still touch
  if constexpr (C::CG == 2) cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc<C::CG>(tmem_base, C::TMEM_COLS);
  if constexpr (C::TWO_PHASE) {
    // the last CTA out resets the band counters, so the workspace is zero
    // again for the next launch
    if (threadIdx.x == 0) {
      unsigned* done = band_ready + m_tiles;
      __threadfence();
      if (atomicAdd(done, 1u) == gridDim.x - 1) {
        const int n = static_cast<int>(block_counters(m_tiles, C::FP8_BLOCK));
        for (int i = 0; i < n; ++i) band_ready[i] = 0u;
        __threadfence();
      }
    }
  }
}

// ------------------------------------------------------------------ host ----

// L2 bytes a band's kept panels may fill in the CODA_RASTER=auto experiment
// (CODA_L2_BUDGET_MB, default 64 MB).
inline int64_t l2_band_budget() {
  static const int64_t b = [] {
    const char* e = getenv("CODA_L2_BUDGET_MB");
    const long mb = e ? atol(e) : 64;
    return static_cast<int64_t>(mb > 0 ? mb : 64) << 20;
  }();
  return b;
}
inline int stream_evict_first() {
  static const int f = [] {
    const char* e = getenv("CODA_L2_STREAM");
    return e != nullptr && e[0] == 'f' ? 1 : 0;
  }();
  return f;
}
inline bool legacy_raster_forced() {
  static const bool f = [] {
    const char* e = getenv("CODA_RASTER");
    return e != nullptr && e[0] == 'l';
  }();
  return f;
}
inline bool auto_raster() {
  static const bool f = [] {
    const char* e = getenv("CODA_RASTER");
    return e != nullptr && e[0] == 'a';
  }();
  return f;
}

// The tile order of one phase.  The legacy raster (M-major bands of 2048 or
// 4096 rows, both operands evict-last) measures fastest on most shapes, even
// where other orders read fewer DRAM bytes: the tiles of a band in flight
// read each B k-slice together.  One case gains from keeping the weights
// instead: a long-K phase (at least 8192 bytes of K per row) whose whole
// weight fits in a 40 MB band.  There, N-major rows with every N-tile in one
// band read the weight once, and the rows complete in order, so a two-phase
// launch's consumer starts on early rows sooner (the LLaMA-1B MLP-down block
// +1.7%, the 8B chain +0.7%).  With shorter K rows the same order measured
// 1.5% slower (the 1B attention-out Wo); a larger weight does not stay in L2
// (the 8B down projection's 117 MB weight in 58 MB bands, and M-tile bands
// kept against evict-first weights, both read more and ran slower).
// CODA_RASTER=legacy keeps the legacy raster everywhere; CODA_RASTER=auto
// picks the order with the fewest modelled DRAM bytes in
// CODA_L2_BUDGET_MB-sized bands (an experiment: slower on most shapes).
template <class C>
Raster choose_raster(int M, int N_out, int K, int epi) {
  if (epi == kNoPhase) return {1, 0, 2};
  const int g_legacy = raster_rows(epi) / C::TILE_M > 0 ? raster_rows(epi) / C::TILE_M : 1;
  const Raster legacy = {g_legacy, 0, 2};
  if (C::A_MN || C::B_MN || legacy_raster_forced()) return legacy;
  const int64_t m_tiles = (M + C::TILE_M - 1) / C::TILE_M;
  const int64_t n_tiles = (N_out + C::out_cols(epi) - 1) / C::out_cols(epi);
  const int64_t k_bytes = static_cast<int64_t>(K) * C::ELEM;
  const int64_t a_panel = static_cast<int64_t>(C::TILE_M) * k_bytes;  // A rows of one tile
  const int64_t b_panel = static_cast<int64_t>(C::BN) * k_bytes;      // B rows of one tile (gate + up)
  if (!auto_raster()) {
    if (k_bytes >= 8192 && b_panel * n_tiles <= (int64_t(40) << 20)) return {static_cast<int>(n_tiles), 1, 1};
    return legacy;
  }
  const int64_t budget = l2_band_budget();
  // the most tiles a band may keep, then spread evenly over the bands it takes
  auto band = [](int64_t g, int64_t n) {
    g = g < 1 ? int64_t(1) : (g > n ? n : g);
    const int64_t bands = (n + g - 1) / g;
    return (n + bands - 1) / bands;
  };
  const int64_t gm = band(budget / a_panel, m_tiles), gn = band(budget / b_panel, n_tiles);
  const int64_t bytes_m = a_panel * m_tiles + b_panel * n_tiles * ((m_tiles + gm - 1) / gm);
  const int64_t bytes_n = b_panel * n_tiles + a_panel * m_tiles * ((n_tiles + gn - 1) / gn);
  if (bytes_n < bytes_m || (gn == n_tiles && bytes_n == bytes_m)) return {static_cast<int>(gn), 1, 1};
  return {static_cast<int>(gm), 0, 0};
}

template <class C>
cudaError_t launch_cfg(const GemmProblem& p, const char** msg) {
  CUtensorMapDataType in_dt = C::kKind == kKindBF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                              : C::kKind == kKindTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                      : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMapDataType out_dt = C::OUT_ELEM == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tmA, tmB, tmB2, tmR, tmD, tmA_b, tmB_b, tmB2_b, tmD_b;
  // operand maps of one phase: A [M, K], B (and B2) [N_out, K], output [M, N_out]
  auto encode_phase = [&](CUtensorMap* a, CUtensorMap* b, CUtensorMap* b2, CUtensorMap* d, const void* A,
                          const void* B, const void* B2, void* D, int N_out, int K, int epi) {
    const uint64_t kbytes = static_cast<uint64_t>(K) * C::ELEM;
    const uint64_t obytes = static_cast<uint64_t>(N_out) * C::OUT_ELEM;
    const uint32_t brows = static_cast<uint32_t>(C::b_box_rows(epi));
    CUresult e = C::A_MN ? encode_tmap_2d(a, in_dt, A, p.M, K, static_cast<uint64_t>(p.M) * C::ELEM, C::MN_BOX, C::BK)
                         : encode_tmap_2d(a, in_dt, A, K, p.M, kbytes, C::BK, C::BM);
    if (e == CUDA_SUCCESS)
      e = C::B_MN ? encode_tmap_2d(b, in_dt, B, N_out, K, static_cast<uint64_t>(N_out) * C::ELEM, C::MN_BOX, C::BK)
                  : encode_tmap_2d(b, in_dt, B, K, N_out, kbytes, C::BK, brows);
    if (e == CUDA_SUCCESS) {
      if (C::B_MN || B2 == nullptr)
        *b2 = *b;  // read only by SwiGLU programs, which have a K-major up weight
      else
        e = encode_tmap_2d(b2, in_dt, B2, K, N_out, kbytes, C::BK, brows);
    }
    if (e == CUDA_SUCCESS) e = encode_tmap_2d(d, out_dt, D, N_out, p.M, obytes, C::BOX_COLS, C::BM);
    return e;
  };
  CUresult e = encode_phase(&tmA, &tmB, &tmB2, &tmD, p.A, p.B, p.B2, p.D, p.N_out, p.K, C::kEpiA);
  // SwiGLU backward reads G || U and writes dG || dU: [M, 2 N_out] tensors
  const uint64_t rd_cols = static_cast<uint64_t>(p.N_out) * (C::kEpiA == kEpiSwiGLUBwd ? 2 : 1);
  if (e == CUDA_SUCCESS)
    e = encode_tmap_2d(&tmR, out_dt, C::HAS_LOADER ? p.R : p.D, rd_cols, p.M, rd_cols * C::OUT_ELEM, C::BOX_COLS,
                       C::BM);
  if (e == CUDA_SUCCESS && C::kEpiA == kEpiSwiGLUBwd)
    e = encode_tmap_2d(&tmD, out_dt, p.D, rd_cols, p.M, rd_cols * C::OUT_ELEM, C::BOX_COLS, C::BM);
  const uint64_t gu_cols = 2 * static_cast<uint64_t>(p.N_out);  // SwiGLU save: G || U [M, 2 N_out]
  if (e == CUDA_SUCCESS) {
    if constexpr (C::TWO_PHASE) {
      e = encode_phase(&tmA_b, &tmB_b, &tmB2_b, &tmD_b, p.b.A, p.b.B, p.b.B2, p.b.D, p.b.N_out, p.b.K, C::kEpiB);
    } else {
      // unused by a one-phase launch, except that SwiGLU save stores G || U through tmD_b
      tmA_b = tmA;
      tmB_b = tmB;
      tmB2_b = tmB2;
      tmD_b = tmD;
      if constexpr (C::kEpiA == kEpiSwiGLUSave)
        e = encode_tmap_2d(&tmD_b, out_dt, p.GU, gu_cols, p.M, gu_cols * C::OUT_ELEM, C::BOX_COLS, C::BM);
    }
  }
  if (e != CUDA_SUCCESS) {
    *msg = "cuTensorMapEncodeTiled rejected an operand (pointer, stride or extent)";
    return cudaErrorInvalidValue;
  }
  auto kernel = gemm_epilogue_kernel<C>;
  // per device: shared-memory opt-in, the number of co-resident units, and
  // (two-phase) whether the device takes a cooperative launch of this form;
  // two host threads may make their first launch at once
  static std::mutex mu;
  static int configured_mask = 0;
  static int max_units[32] = {0};
  static int coop_plain_mask = 0;  // devices that refused the cooperative form
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  int units = 0;
  // CODA_NO_COOPERATIVE=1 launches two-phase grids plainly: for profilers that
  // cannot replay a cooperative clustered launch (the co-residency contract
  // then rests on the caller, as on a device that refuses the cooperative form)
  static const bool no_coop = getenv("CODA_NO_COOPERATIVE") != nullptr;
  bool cooperative = C::TWO_PHASE && !no_coop;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 32 || !(configured_mask & (1 << dev))) {
      ce = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
      if (ce != cudaSuccess) {
        *msg = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize) failed";
        return ce;
      }
      int u = device_sm_count();
      if (C::CG == 2) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * u);
        cfg.blockDim = dim3(C::NUM_THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        ce = cudaOccupancyMaxActiveClusters(&clusters, reinterpret_cast<const void*>(kernel), &cfg);
        if (ce != cudaSuccess || clusters <= 0) {
          *msg = "cudaOccupancyMaxActiveClusters failed for the CTA-pair GEMM";
          return ce != cudaSuccess ? ce : cudaErrorInvalidConfiguration;
        }
        u = clusters;
      }
      if (dev < 32) {
        max_units[dev] = u;
        configured_mask |= 1 << dev;
      }
      units = u;
    } else {
      units = max_units[dev];
    }
    if (dev < 32 && (coop_plain_mask & (1 << dev))) cooperative = false;
  }
  const int m_tiles = (p.M + C::TILE_M - 1) / C::TILE_M;
  int num_tiles = m_tiles * ((p.N_out + C::out_cols(C::kEpiA) - 1) / C::out_cols(C::kEpiA));
  if constexpr (C::TWO_PHASE) num_tiles += m_tiles * ((p.b.N_out + C::out_cols(C::kEpiB) - 1) / C::out_cols(C::kEpiB));
  // a two-phase launch needs every CTA resident (its waits span CTAs): the
  // grid never exceeds the co-resident units
  const int grid = C::CG * (num_tiles < units ? num_tiles : units);
  int M = p.M;
  PhaseArgs pa = {p.N_out, p.K, p.ep, choose_raster<C>(p.M, p.N_out, p.K, C::kEpiA), stream_evict_first()};
  PhaseArgs pb = {p.b.N_out, p.b.K, p.b.ep, choose_raster<C>(p.M, p.b.N_out, p.b.K, C::kEpiB),
                  stream_evict_first()};
  unsigned* band_ready = p.band_ready;
  QuantArgs q = p.q;
  void* args[] = {&tmA, &tmB, &tmB2, &tmR, &tmD, &tmA_b, &tmB_b, &tmB2_b, &tmD_b, &M, &pa, &pb, &band_ready, &q};
  bool refused = false;
  ce = launch_coresident(
      [&](bool coop) {
        return launch_ex(reinterpret_cast<const void*>(kernel), dim3(grid), dim3(C::NUM_THREADS), C::SMEM_BYTES,
                         p.stream, p.pdl, args, C::CG, coop);
      },
      cooperative, &refused);
  if (refused && dev < 32) {
    // this device takes no cooperative launch of a clustered grid: the grid
    // stays sized to the co-resident units of an idle GPU
    std::lock_guard<std::mutex> lock(mu);
    coop_plain_mask |= 1 << dev;
  }
  if (ce != cudaSuccess) *msg = "GEMM kernel launch failed";
  return ce;
}

// CTA pairs (cta_group::2, 256-row tiles) unless the problem is too small to
// give every pair a tile, or CODA_CTA_GROUP=1|2 forces a choice.
inline int choose_cta_group(const GemmProblem& p) {
  if (const char* f = getenv("CODA_CTA_GROUP")) {
    if (f[0] == '1') return 1;
    if (f[0] == '2') return 2;
  }
  const int out_cols = is_swiglu(p.epi) ? 128 : 256;
  const long tiles2 = static_cast<long>((p.M + 255) / 256) * ((p.N_out + out_cols - 1) / out_cols);
  return tiles2 >= device_sm_count() / 2 ? 2 : 1;
}

// Shared memory per CTA (227 KB max):
//   one CTA per MMA : 48 KB stages; residual 3 stages + 4 R slots, others 4 + 2
//   CTA pairs       : 32 KB stages; residual 5 stages + 4 R slots, others 6 + 2
//   two-phase       : as the residual program (its slot ring serves both phases)
template <int KIND>
cudaError_t launch_gemm(const GemmProblem& p, const char** msg) {
  const bool pair = choose_cta_group(p) == 2;
  if constexpr (KIND == kKindBF16) {
    // backward programs: dY = dOut . W (W's forward W^T read MN-major)
    if (p.epi == kEpiGradNorm || p.epi == kEpiSwiGLUBwd) {
      if (!p.b_mn || p.a_mn) {
        *msg = "backward programs take a K-major A and an MN-major B";
        return cudaErrorInvalidValue;
      }
      if (p.epi == kEpiGradNorm)
        return pair ? launch_cfg<GemmCfg<KIND, kEpiGradNorm, kNoPhase, 6, 2, 2, false, true>>(p, msg)
                    : launch_cfg<GemmCfg<KIND, kEpiGradNorm, kNoPhase, 3, 4, 1, false, true>>(p, msg);
      return pair ? launch_cfg<GemmCfg<KIND, kEpiSwiGLUBwd, kNoPhase, 6, 2, 2, false, true>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiSwiGLUBwd, kNoPhase, 3, 4, 1, false, true>>(p, msg);
    }
    // MN-major operands (transposed products of the backward pass): row-scale program
    if (p.a_mn || p.b_mn) {
      if (p.epi != kEpiRowScale || p.b.epi != -1) {
        *msg = "MN-major operands take the row-scale program only";
        return cudaErrorInvalidValue;
      }
      if (p.a_mn && p.b_mn)
        return pair ? launch_cfg<GemmCfg<KIND, kEpiRowScale, kNoPhase, 6, 2, 2, true, true>>(p, msg)
                    : launch_cfg<GemmCfg<KIND, kEpiRowScale, kNoPhase, 4, 2, 1, true, true>>(p, msg);
      if (p.b_mn)
        return pair ? launch_cfg<GemmCfg<KIND, kEpiRowScale, kNoPhase, 6, 2, 2, false, true>>(p, msg)
                    : launch_cfg<GemmCfg<KIND, kEpiRowScale, kNoPhase, 4, 2, 1, false, true>>(p, msg);
      *msg = "an MN-major A needs an MN-major B";
      return cudaErrorInvalidValue;
    }
  } else {
    if (p.a_mn || p.b_mn) {
      *msg = "MN-major operands are bf16 only";
      return cudaErrorInvalidValue;
    }
  }
  if constexpr (KIND == kKindE4M3) {
    // FP8 two-phase launches quantise h (and optionally phase A's A operand)
    // in the launch: the FP8 block configurations, with quantiser warps
    if (p.b.epi != -1 && !p.fp8_block) {
      *msg = "an e4m3 two-phase launch is an FP8 block";
      return cudaErrorInvalidValue;
    }
    if (p.b.epi == kEpiRowScale)
      return pair ? launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiRowScale, 5, 4, 2, false, false, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiRowScale, 3, 4, 1, false, false, 2>>(p, msg);
    if (p.b.epi == kEpiSwiGLU)
      return pair ? launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiSwiGLU, 5, 4, 2, false, false, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiSwiGLU, 3, 4, 1, false, false, 2>>(p, msg);
  } else {
    if (p.fp8_block) {
      *msg = "FP8 blocks take e4m3 operands";
      return cudaErrorInvalidValue;
    }
    if (p.b.epi == kEpiRowScale)
      return pair ? launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiRowScale, 5, 4, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiRowScale, 3, 4, 1>>(p, msg);
    if (p.b.epi == kEpiSwiGLU)
      return pair ? launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiSwiGLU, 5, 4, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kEpiSwiGLU, 3, 4, 1>>(p, msg);
  }
  switch (p.epi) {
    case kEpiResidualPartialRms:
      return pair ? launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kNoPhase, 5, 4, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiResidualPartialRms, kNoPhase, 3, 4, 1>>(p, msg);
    case kEpiRowScale:
      return pair ? launch_cfg<GemmCfg<KIND, kEpiRowScale, kNoPhase, 6, 2, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiRowScale, kNoPhase, 4, 2, 1>>(p, msg);
    case kEpiSwiGLU:
      return pair ? launch_cfg<GemmCfg<KIND, kEpiSwiGLU, kNoPhase, 6, 2, 2>>(p, msg)
                  : launch_cfg<GemmCfg<KIND, kEpiSwiGLU, kNoPhase, 4, 2, 1>>(p, msg);
    case kEpiSwiGLUSave:
      if constexpr (KIND == kKindBF16)
        return pair ? launch_cfg<GemmCfg<KIND, kEpiSwiGLUSave, kNoPhase, 4, 6, 2>>(p, msg)
                    : launch_cfg<GemmCfg<KIND, kEpiSwiGLUSave, kNoPhase, 2, 6, 1>>(p, msg);
      *msg = "saving the SwiGLU pre-activations is bf16 only";
      return cudaErrorInvalidValue;
    default:
      *msg = "unknown epilogue program";
      return cudaErrorInvalidValue;
  }
}

inline unsigned read_clear_status_impl() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return ~0u;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  return v;
}

}  // namespace coda
