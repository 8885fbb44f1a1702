// Quantizers of bf16 tensors on sm_103a: MX block quantization (row / column
// / dual orientation, E4M3 / E5M2 / E2M1, floor or ceil scales, RNE or
// Philox stochastic rounding, optional fixed-sign Hadamard-32) and the
// per-tensor FP8 quantize with fused amax and the delayed-scaling fold.
//
// Sources: "UE8M0 FP8 / MXFP8 explainer", sections 1 and 4, gap sections 1-2
// (MX blocks of 32 sharing a UE8M0 scale taken from the block amax,
// saturating element quantization, floor versus ceil scale rounding, row and
// transposed column copies); AstrAI astrai/extension/ops/fp8.py (quantize /
// quantize_dual docstrings and commit message: per-tensor multiplier, fused
// amax, one read for x8 and x8T, last-block fold with an atomic ticket);
// "Format-aware fusion for FP4" (row-gradient stochastic rounding, fixed-sign
// 32-point Hadamard, scale layout written for its consumer).
//
// Design (one kernel shape for every mode):
//  * The tensor is cut into 128-row x 64-column bf16 tiles (16 KiB).  A
//    persistent grid of 256-thread CTAs (as many per SM as fit) walks the
//    tiles; each tile arrives by one TMA load (128-byte swizzle) into a ring
//    of NSTG stages, so HBM reads of the next tiles overlap the work on the
//    current one.
//  * Every warp owns a fixed part of each tile and runs on its own: it waits
//    for the tile's stage, quantizes its part, stages its codes in its own
//    shared-memory buffers and issues its own TMA store.  There is no barrier
//    across warps in the loop.  The last warp to finish reading a stage (a
//    shared-memory counter tells which) issues the stage's next load.
//  * Dual orientation: warps 0-3 take 32 rows each (one lane per row, both
//    1 x 32 blocks of the row); warps 4-7 take a 32-row band each (one lane
//    per two adjacent columns, two 32 x 1 blocks in registers).  Row only:
//    eight warps of 16 rows (one block per lane).  Column only: warps 0-3
//    take the bands of the CTA's even tiles, warps 4-7 those of its odd
//    tiles (an even number of stages keeps each stage with one group).
//  * The column copy is staged transposed, so it leaves as rows of q_col.
//    Scales leave from the lanes that computed them, in the requested layout
//    (canonical, or the GEMM's 512-byte tensor-core chunks).
//  * One HBM read of x produces every requested output.
//  * A launch may carry up to four tensors of one format and orientation
//    (the grouped entry point): their tiles form one sequence, and each tile
//    reads its own tensor's maps and parameters.
#include <algorithm>

#include "common.cuh"

namespace mxq {

// Pipeline depth of the quantizers: NSTG input stages per CTA and NOUT
// staging buffers per warp (2 lets a warp stage a tile while the bulk store
// of its previous tile still reads shared memory).  Build-time knobs; the
// defaults are the measured best.
#ifndef MXQ_QUANT_NST
#define MXQ_QUANT_NST 3
#endif
#ifndef MXQ_QUANT_STG
#define MXQ_QUANT_STG 2
#endif
constexpr int TR = 128;                     // tile rows
constexpr int BOX_BYTES = TR * 64 * 2;      // one TMA load box: 128 rows x 64 bf16 (16 KiB)

template <int NSTG, int NOUT, bool EXTRA, int STG_ = 2048>
struct TileCfg {
  static constexpr int TC = 64;                     // tile columns
  static constexpr int THREADS = 256;
  static constexpr int NW = THREADS / 32;
  static constexpr int IN_BYTES = TR * TC * 2;      // one stage: 128 x 64 bf16
  // one staging buffer of one warp: a dual launch's 32 rows (or 64 columns)
  // of codes, 2 KiB; a row-only warp's 16 rows, 1 KiB
  static constexpr int STG = STG_;
  // every warp writes codes through its own staging buffers; a row-only
  // launch (1 KiB buffers) thereby needs 65 KB of shared memory, which fits
  // a third CTA per SM
  static constexpr int SMEM = NSTG * IN_BYTES + NW * NOUT * STG + 256 + 1024;
  // resident CTAs per SM the registers are budgeted for
  static constexpr int MIN_BLOCKS = EXTRA ? 2 : (SMEM <= 70 * 1024 ? 3 : 2);
};

// 16-byte chunk index after the TMA swizzle of a staged row of `pitch`
// bytes (128 / 64 / 32-byte swizzle: chunk bits ^= address bits 7..9 / 7..8 / 7).
__device__ __forceinline__ int swz(int row, int chunk, int pitch) {
  return chunk ^ (((row * pitch) >> 7) & (pitch / 16 - 1));
}

struct QuantParams {
  int rows, cols;
  int tiles_c, ntiles;
  int ceil_mode, rounding, hadamard, sf_mma;
  uint32_t sr_k0, sr_k1, had_k0, had_k1;
  uint8_t* s_row;
  uint8_t* s_col;
  int* status;
  // per-tensor FP8
  const float* scale;
  float* ring;
  int hist_len, hist_idx;
  float fp8_max, margin;
  float* amax_out;
  int stall_tile;     // failure-detection test hook: this tile is never loaded (-1: off)
};

// Stochastic rounding of y (float32, exact) to the element grid with the
// 32-bit draw r: magnitude y' = min(|y|, max) between grid neighbours
// lo <= y' < lo + sp rounds up iff r < floor((y' - lo) / sp * 2^32).  All
// steps are exact in float32 (power-of-two scalings and a difference of two
// nearby values).  Returns the rounded value (on the grid, sign kept).
template <int FMT>
__device__ __forceinline__ float sr_round(float y, uint32_t r) {
  const float a = fminf(fabsf(y), FmtInfo<FMT>::maxv);
  const int bexp = static_cast<int>(__float_as_uint(a) >> 23) - 127;
  const int E = max(bexp, FmtInfo<FMT>::emin);
  const float sp = __uint_as_float(static_cast<uint32_t>(E - FmtInfo<FMT>::mbits + 127) << 23);
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - (E - FmtInfo<FMT>::mbits)) << 23);
  const float n = floorf(__fmul_rn(a, inv));
  const float lo = __fmul_rn(n, sp);
  const float frac = __fmul_rn(__fsub_rn(a, lo), inv);          // in [0, 1), exact
  const uint32_t t = __float2uint_rz(__fmul_rn(frac, 4294967296.0f));
  const float mag = (r < t) ? __fadd_rn(lo, sp) : lo;
  return copysignf(mag, y);
}

// Hadamard signs: bit j of word 0 of Philox-4x32-10(key = seed, counter = 0).
__device__ __forceinline__ uint32_t hadamard_sign_mask(uint32_t k0, uint32_t k1) {
  return philox4x32_10(u32x4{0u, 0u, 0u, 0u}, k0, k1).x;
}

__device__ __forceinline__ uint32_t sr_draw(uint64_t idx, uint32_t k0, uint32_t k1) {
  return philox4x32_10(u32x4{static_cast<uint32_t>(idx), static_cast<uint32_t>(idx >> 32), 0u, 0u}, k0, k1).x;
}

// Four draws per call: word (idx & 3) of the call with counter idx >> 2.
__device__ __forceinline__ uint32_t sr_draw4(uint64_t idx, uint32_t k0, uint32_t k1) {
  const uint64_t c = idx >> 2;
  const u32x4 w = philox4x32_10(u32x4{static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), 0u, 0u}, k0, k1);
  const uint32_t j = static_cast<uint32_t>(idx) & 3u;
  return j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
}

constexpr float kHadC = 0.17677669529663688f;  // float32 nearest 1/sqrt(32)

// Fixed-sign 32-point Hadamard of one block held by one thread:
// u_j = s_j v_j; butterflies h = 1, 2, 4, 8, 16 in that order,
// (u_i, u_{i+h}) <- (u_i + u_{i+h}, u_i - u_{i+h}) for (i & h) == 0;
// y_j = RN32(u_j * c).  Every operation is a separate float32 rounding.
// From h = 2 on, elements 2k and 2k + 1 meet elements 2k + h and
// 2k + 1 + h, so those stages and the final product run on packed pairs.
__device__ __forceinline__ void hadamard32(float (&u)[32], uint32_t signs) {
#pragma unroll
  for (int j = 0; j < 32; ++j) u[j] = ((signs >> j) & 1u) ? -u[j] : u[j];
  uint64_t P[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) P[k] = f32x2_pack(__fadd_rn(u[2 * k], u[2 * k + 1]), __fsub_rn(u[2 * k], u[2 * k + 1]));
#pragma unroll
  for (int hh = 1; hh < 16; hh <<= 1) {            // h = 2 hh
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if ((k & hh) == 0) {
        const uint64_t a = P[k], b = P[k + hh];
        P[k] = f32x2_add(a, b);
        P[k + hh] = f32x2_sub(a, b);
      }
    }
  }
  const uint64_t cc = f32x2_pack(kHadC, kHadC);
#pragma unroll
  for (int k = 0; k < 16; ++k) f32x2_unpack(f32x2_mul(P[k], cc), u[2 * k], u[2 * k + 1]);
}

// Bits of the largest |v| of a block of 32 float32 values (NaN anywhere:
// NaN bits; an infinity: 0x7F800000).
__device__ __forceinline__ uint32_t amax32_float(const float (&v)[32]) {
  return amax32_tree([&](int j) { return fabsf(v[j]); });
}

// Packed bf16x2 running max of magnitudes, NaN-propagating, one instruction
// per word: each half becomes max(|m|, |w|) with the XOR of the two signs;
// callers clear the sign bits once at the end (amax_halves).
__device__ __forceinline__ uint32_t hmax2_abs(uint32_t m, uint32_t w) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w));
  return r;
}

// Sign-cleared halves of a hmax2_abs accumulator (NaN stays above Inf).
__device__ __forceinline__ uint32_t amax_halves(uint32_t m) { return m & 0x7FFF7FFFu; }

// Largest |value| of 32 bf16 held as 16 packed words, as float32 bits
// (non-negative bf16 patterns order like their values; NaN sorts above Inf).
__device__ __forceinline__ uint32_t amax_bf16x32(const uint32_t (&w)[16]) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = hmax2_abs(m, w[j]);
  m = amax_halves(m);
  return max(m & 0xFFFFu, m >> 16) << 16;
}

// RNE quantization of a 1x32 block given as 16 packed bf16 words (element
// 2j in the low half of word j), scale exponent e.  out: FP8 8 words /
// E2M1 4 words.
template <int FMT>
__device__ __forceinline__ void rne_words16(const uint32_t (&w)[16], float m, uint32_t (&out)[8]) {
  if constexpr (FMT == MXQ_E2M1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t x = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t a = w[4 * k + j];
        x |= cvt_e2m1x2(__fmul_rn(bf16lo(a), m), __fmul_rn(bf16hi(a), m)) << (8 * j);
      }
      out[k] = x;
    }
  } else {
    const uint64_t mm = f32x2_splat(m);
#pragma unroll
    for (int k = 0; k < 8; ++k) out[k] = fp8x4_rows<FMT>(w[2 * k], w[2 * k + 1], mm);
  }
}

// RNE quantization of one 32x1 column block held as the low (half = 0) or
// high (half = 1) halves of 32 words (row k in word k).
template <int FMT>
__device__ __forceinline__ void rne_col32(const uint32_t (&w)[32], int half, float m, uint32_t (&out)[8]) {
  auto x = [&](int k) { return __fmul_rn(half ? bf16hi(w[k]) : bf16lo(w[k]), m); };
  if constexpr (FMT != MXQ_E2M1) {
    const uint64_t mm = f32x2_splat(m);
    if (half) {
#pragma unroll
      for (int k = 0; k < 8; ++k) out[k] = fp8x4_col<FMT, 1>(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3], mm);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) out[k] = fp8x4_col<FMT, 0>(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3], mm);
    }
    return;
  }
  if constexpr (FMT == MXQ_E2M1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) v |= cvt_e2m1x2(x(8 * k + 2 * j), x(8 * k + 2 * j + 1)) << (8 * j);
      out[k] = v;
    }
  }
}

// A block holding NaN or Inf gets zero codes (warp-uniform branch: rare).
__device__ __forceinline__ void zero_if_bad(bool bad, uint32_t (&out)[8]) {
  if (__any_sync(0xFFFFFFFFu, bad)) {
#pragma unroll
    for (int k = 0; k < 8; ++k) out[k] = bad ? 0u : out[k];
  }
}

// Quantize one 32-element block v (float32 values, exact) whose amax bits
// are ab.  Codes go to out (FP8: 8 words, E2M1: 4 words, element 0 in the
// lowest byte / nibble); returns the UE8M0 scale byte.  idx0 / istep give
// the flat input index of element j as idx0 + j * istep (for the SR draw).
template <int FMT, bool EXTRA>
__device__ __forceinline__ uint32_t quant_block32(const float (&v)[32], uint32_t ab, const QuantParams& p,
                                                  uint64_t idx0, uint64_t istep, uint32_t (&out)[8]) {
  const bool bad = ab >= 0x7F800000u;                 // NaN or Inf in the block
  const int e = scale_exp<FMT>(bad ? 0u : ab, p.ceil_mode);
  float vm[32];                                       // v * 2^-e, packed products
  {
    const uint64_t mm = f32x2_splat(exp2_neg(e));
#pragma unroll
    for (int k = 0; k < 16; ++k) f32x2_unpack(f32x2_mul(f32x2_pack(v[2 * k], v[2 * k + 1]), mm), vm[2 * k], vm[2 * k + 1]);
  }
  float y[32];
  if (EXTRA && p.rounding == MXQ_SR4 && istep == 1) {
    // a row block: 32 consecutive indices from a multiple of 32, so the
    // eight calls with counters idx0/4 .. idx0/4 + 7 give all 32 draws
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint64_t c = (idx0 >> 2) + k;
      const u32x4 w =
          philox4x32_10(u32x4{static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), 0u, 0u}, p.sr_k0, p.sr_k1);
      y[4 * k] = sr_round<FMT>(vm[4 * k], w.x);
      y[4 * k + 1] = sr_round<FMT>(vm[4 * k + 1], w.y);
      y[4 * k + 2] = sr_round<FMT>(vm[4 * k + 2], w.z);
      y[4 * k + 3] = sr_round<FMT>(vm[4 * k + 3], w.w);
    }
  } else if (EXTRA && p.rounding == MXQ_SR4) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      y[j] = sr_round<FMT>(vm[j], sr_draw4(idx0 + j * istep, p.sr_k0, p.sr_k1));
  } else if (EXTRA && p.rounding == MXQ_SR) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      y[j] = sr_round<FMT>(vm[j], sr_draw(idx0 + j * istep, p.sr_k0, p.sr_k1));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = vm[j];
  }
  if constexpr (FMT == MXQ_E2M1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t x = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) x |= cvt_e2m1x2(y[8 * k + 2 * j], y[8 * k + 2 * j + 1]) << (8 * j);
      out[k] = bad ? 0u : x;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t x = cvt_fp8x4<FMT>(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
      out[k] = bad ? 0u : x;
    }
  }
  return bad ? 0xFFu : static_cast<uint32_t>(e + 127);
}

// Per-tensor FP8 of 32 values: RNE-saturating encode of RN32(x * mult).
template <int FMT>
__device__ __forceinline__ void pertensor32(const uint32_t (&w)[16], float mult, uint32_t (&out)[8]) {
  const uint64_t mm = f32x2_splat(mult);
#pragma unroll
  for (int k = 0; k < 8; ++k) out[k] = fp8x4_rows<FMT>(w[2 * k], w[2 * k + 1], mm);
}

// The delayed-scaling fold (AstrAI fp8.py, commit message and quantize
// docstring): ring = [hist[n] | scale | legacy | amax | done].  The tensor
// amax goes to hist[hist_idx]; M = max(hist) (a NaN entry wins); when M is
// finite and > 0 the next scale max(hist) / fp8_max / pow2_margin is
// published as RN32(RN32(M / fp8_max) / margin), and legacy = RN32(1 / scale)
// (the multiplier the next step passes in); the amax slot and the ticket
// counter are reset to zero.  One thread runs it.
__device__ __forceinline__ void fold_ring(volatile float* ring, int n, int hist_idx, float amax, float fp8_max,
                                          float margin) {
  ring[hist_idx] = amax;
  float M = ring[0];
  for (int k = 1; k < n; ++k) {
    const float a = ring[k];
    if (isnan(a) || a > M) M = a;
  }
  if (M > 0.f && isfinite(M)) {
    const float sc = __fdiv_rn(__fdiv_rn(M, fp8_max), margin);
    ring[n] = sc;
    ring[n + 1] = __frcp_rn(sc);
  }
  ring[n + 2] = 0.f;
  reinterpret_cast<volatile unsigned int*>(ring)[n + 3] = 0u;
}

// The tensors of one launch: NJ quantize jobs of one format and orientation
// (NJ = 1: a single tensor).  Their tiles form one sequence in job order: job
// j owns tiles tile_end[j - 1] .. tile_end[j] - 1 (tile_end[-1] = 0), so the
// persistent CTAs run through all jobs without a launch boundary between
// them.  Unused trailing entries repeat the total in tile_end.  Job 0's
// parameters also travel as a separate by-value kernel argument, which is
// all a single-tensor launch reads (plain parameter loads).
template <int NJ>
struct QuantLaunch {
  CUtensorMap mx[NJ];        // bf16 input boxes
  CUtensorMap mr[NJ];        // row-block codes
  CUtensorMap mc[NJ];        // transposed column-block codes
  QuantParams p[NJ];
  int tile_end[NJ];
};

// Job of a tile of the launch: the number of jobs that end at or before it.
template <int NJ>
__device__ __forceinline__ int job_of(const QuantLaunch<NJ>& L, int tile) {
  int j = 0;
#pragma unroll
  for (int k = 0; k + 1 < NJ; ++k) j += tile >= L.tile_end[k] ? 1 : 0;
  return j;
}

// EXTRA: compile the stochastic-rounding and Hadamard paths (selected at run
// time by the parameters); without it the kernel is the lean RNE variant.
template <int FMT, int ORIENT, bool PERTENSOR, bool EXTRA, int NSTG, int NOUT, int NJ>
__global__ void __launch_bounds__(256, TileCfg<NSTG, NOUT, EXTRA,
                                               ORIENT == MXQ_ROW ? 1024 : 2048>::MIN_BLOCKS)
quant_tiles_kernel(const __grid_constant__ QuantLaunch<NJ> L, const QuantParams p0) {
  using T = TileCfg<NSTG, NOUT, EXTRA, ORIENT == MXQ_ROW ? 1024 : 2048>;
  constexpr int TC = T::TC;
  constexpr bool DO_ROW = (ORIENT & MXQ_ROW) != 0;
  constexpr bool DO_COL = (ORIENT & MXQ_COL) != 0;
  constexpr bool DUAL = DO_ROW && DO_COL;
  constexpr bool FP4 = (FMT == MXQ_E2M1);
  constexpr int QBR = FP4 ? TC / 2 : TC;            // code bytes per tile row
  constexpr int QBW = FP4 ? 16 : 32;                // code bytes per column per 32-row band
  constexpr int RR = DUAL ? 32 : 16;                // rows of a row warp
  constexpr int BPL = DUAL ? 2 : 1;                 // 1 x 32 blocks per lane of a row warp
  constexpr int ROW_WARPS = DO_ROW ? (DUAL ? 4 : 8) : 0;
  constexpr int ACTIVE = ROW_WARPS + (DO_COL ? 4 : 0);   // warps that read every stage
  static_assert((!DO_ROW || RR * QBR <= T::STG) && (!DO_COL || 64 * QBW <= T::STG), "staging buffer");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* in_s = smem;                                   // NSTG x 16 KiB stages
  uint8_t* stg_s = in_s + NSTG * T::IN_BYTES;             // per warp NOUT staging buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_s + T::NW * NOUT * T::STG);   // full[NSTG]
  uint32_t* cnt = reinterpret_cast<uint32_t*>(bars + NSTG);       // readers done with each stage
  int* last_use = reinterpret_cast<int*>(cnt + NSTG);             // latest load issued into each stage
  uint32_t* red = reinterpret_cast<uint32_t*>(last_use + NSTG);   // per-warp amax (per-tensor)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + T::NW);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // p0: job 0, and what all jobs share (status, rounding, per-tensor state)
  const int ntiles = NJ == 1 ? p0.ntiles : L.tile_end[NJ - 1];
  const uint32_t signs = (EXTRA && p0.hadamard) ? hadamard_sign_mask(p0.had_k0, p0.had_k1) : 0u;
  // first tile row and column of a tile of the launch, in its job's tensor
  auto tile_origin = [&](int tile, int jb, int& r0, int& c0) {
    const QuantParams& pj = NJ == 1 ? p0 : L.p[jb];
    const int t = tile - (jb ? L.tile_end[jb - 1] : 0);
    r0 = (t / pj.tiles_c) * TR;
    c0 = (t % pj.tiles_c) * TC;
  };

  // Load of this CTA's tile i into its stage (issued by one thread).
  auto issue = [&](int i) {
    const int tile = blockIdx.x + i * gridDim.x;
    if (tile == p0.stall_tile) return;     // test hook: leave this stage's phase incomplete
    const int jb = job_of(L, tile);
    int r0, c0;
    tile_origin(tile, jb, r0, c0);
    const uint32_t bar = smem_u32(&bars[i % NSTG]);
    last_use[i % NSTG] = i;
    mbar_arrive_expect_tx(bar, T::IN_BYTES);
    tma_load_2d(smem_u32(in_s + (i % NSTG) * T::IN_BYTES), &L.mx[jb], bar, c0, r0);
  };

  if (tid == 0) {
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      cnt[s] = 0;
      last_use[s] = -1;
    }
    *abort_flag = 0;
    fence_mbar_init();
#pragma unroll
    for (int k = 0; k < NJ; ++k) {
      prefetch_tensormap(&L.mx[k]);
      if (DO_ROW) prefetch_tensormap(&L.mr[k]);
      if (DO_COL) prefetch_tensormap(&L.mc[k]);
    }
    // The first tiles' input into L2 while the previous kernel in the stream
    // may still be finishing.  L2 is where the GPU's memory is coherent: a
    // write of that kernel that lands later updates the prefetched line, and
    // the loads below are issued only after grid_dep_wait, so they see it.
    for (int i = 0; i < NSTG; ++i) {
      const int tile = blockIdx.x + i * gridDim.x;
      if (tile < ntiles) {
        const int jb = job_of(L, tile);
        int r0, c0;
        tile_origin(tile, jb, r0, c0);
        tma_prefetch_2d(&L.mx[jb], c0, r0);
      }
    }
  }
  __syncthreads();
  grid_dep_launch();
  grid_dep_wait();                 // before any other global-memory access
  const float mult = PERTENSOR ? *p0.scale : 1.0f;
  if (tid == 0) {
    for (int i = 0; i < NSTG; ++i)
      if (blockIdx.x + i * gridDim.x < ntiles) issue(i);
  }

  // This warp's part of every tile.
  const bool row_warp = warp < ROW_WARPS;
  // column only: warps 0-3 take the even tiles of the CTA, warps 4-7 the odd.
  // With an even number of stages each stage then serves one group only, so
  // a group's waits on a stage follow that stage's phases in order (with an
  // odd count a group could pass a wait on the other group's phase).
  constexpr bool SPLIT = DO_COL && !DO_ROW;
  constexpr int ISTEP = SPLIT ? 2 : 1;
  static_assert(!SPLIT || NSTG % 2 == 0, "column-only launches need an even stage count");
  const int col_band = DO_COL ? (DUAL ? warp - 4 : (DO_ROW ? -1 : (warp & 3))) : -1;
  const bool col_warp = DO_COL && col_band >= 0 && col_band < 4;
  const int ro = row_warp ? warp * RR : 0;           // first tile row of a row warp

  uint32_t amax_acc = 0;   // per-tensor: running max of |x| bits
  if (row_warp || col_warp) {
    for (int i = SPLIT ? (warp >> 2) : 0;; i += ISTEP) {
      const int tile = blockIdx.x + i * gridDim.x;
      if (tile >= ntiles || *abort_flag) break;
      const int jb = job_of(L, tile);
      const QuantParams& p = NJ == 1 ? p0 : L.p[jb];   // this tile's tensor
      int r0, c0;
      tile_origin(tile, jb, r0, c0);
      const int s = i % NSTG;
      if (!mbar_wait(smem_u32(&bars[s]), (i / NSTG) & 1, p.status)) {
        *abort_flag = 1;
        break;
      }
      const uint8_t* in = in_s + s * T::IN_BYTES;
      uint8_t* stg = stg_s + (warp * NOUT + (i / ISTEP) % NOUT) * T::STG;
      // this buffer was last read by the bulk store of this warp's tile NOUT tiles back
      if (lane == 0) {
        if constexpr (NOUT == 2) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        else bulk_wait_read_all();
      }
      __syncwarp();

      if (row_warp) {
        // ---------------------------------------------------------- row blocks
        // 16-byte shared loads, conflict-free: the 128-byte swizzle puts the
        // 8 rows of a load phase in 8 different bank groups.
        const int r = lane % RR, row = ro + r;
        uint32_t sc2 = 0;
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
          const int b = (lane / RR) * BPL + j;
          const uint8_t* src = in + row * 128;
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 q = *reinterpret_cast<const uint4*>(src + (((b * 4 + k) ^ (row & 7)) << 4));
            w[4 * k] = q.x; w[4 * k + 1] = q.y; w[4 * k + 2] = q.z; w[4 * k + 3] = q.w;
          }
          uint32_t out[8];
          uint32_t sc = 0;
          if constexpr (PERTENSOR) {
            amax_acc = max(amax_acc, amax_bf16x32(w));
            pertensor32<FMT>(w, mult, out);
          } else if constexpr (!EXTRA) {
            const uint32_t ab = amax_bf16x32(w);
            const bool bad = ab >= 0x7F800000u;
            const int e = scale_exp<FMT>(bad ? 0u : ab, p.ceil_mode);
            rne_words16<FMT>(w, exp2_neg(e), out);
            zero_if_bad(bad, out);
            sc = bad ? 0xFFu : static_cast<uint32_t>(e + 127);
          } else {
            float v[32];
#pragma unroll
            for (int q = 0; q < 16; ++q) { v[2 * q] = bf16lo(w[q]); v[2 * q + 1] = bf16hi(w[q]); }
            uint32_t ab;
            if (p.hadamard) {
              hadamard32(v, signs);
              ab = amax32_float(v);
            } else {
              ab = amax_bf16x32(w);
            }
            const uint64_t idx0 = static_cast<uint64_t>(r0 + row) * static_cast<uint64_t>(p.cols) + (c0 + 32 * b);
            sc = quant_block32<FMT, EXTRA>(v, ab, p, idx0, 1, out);
          }
          sc2 |= sc << (8 * j);
          if constexpr (FP4) {
            *reinterpret_cast<uint4*>(stg + r * QBR + (swz(r, b, QBR) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
          } else {
            *reinterpret_cast<uint4*>(stg + r * QBR + (swz(r, 2 * b, QBR) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
            *reinterpret_cast<uint4*>(stg + r * QBR + (swz(r, 2 * b + 1, QBR) << 4)) = make_uint4(out[4], out[5], out[6], out[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&L.mr[jb], smem_u32(stg), FP4 ? c0 / 2 : c0, r0 + ro);
          bulk_commit();
        }
        // row scales: the lane's BPL bytes (blocks b0 .. b0 + BPL - 1 of its row)
        if constexpr (!PERTENSOR) {
          const int b0 = c0 / 32 + (lane / RR) * BPL, kb = p.cols / 32;
          if (r0 + row < p.rows && b0 < kb) {
            uint8_t* dst;
            bool vec = BPL == 2;
            if (p.sf_mma) {   // full tiles only (rows, cols % 128 == 0)
              dst = p.s_row + (static_cast<size_t>(r0 / 128) * (p.cols / 128) + c0 / 128) * 512 + (row & 31) * 16 +
                    ((row >> 5) & 3) * 4 + (b0 & 3);
            } else {
              dst = p.s_row + static_cast<size_t>(r0 + row) * kb + b0;
              vec = vec && (kb % 2) == 0 && b0 + 2 <= kb;
            }
            if (vec) {
              *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(sc2);
            } else {
              for (int j = 0; j < BPL && b0 + j < kb; ++j) dst[j] = static_cast<uint8_t>(sc2 >> (8 * j));
            }
          }
        }
      } else {
        // ---------------------------------------------------------- column blocks
        // 4-byte shared loads: a warp reads 128 contiguous bytes of a row.
        const int rb = col_band;
        const int chk = lane >> 2, wb = (lane & 3) * 4;
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int row = rb * 32 + k;
          w[k] = *reinterpret_cast<const uint32_t*>(in + row * 128 + ((chk ^ (k & 7)) << 4) + wb);
        }
        uint32_t m2 = 0;                       // packed amax of both columns
#pragma unroll
        for (int k = 0; k < 32; ++k) m2 = hmax2_abs(m2, w[k]);
        m2 = amax_halves(m2);
        uint32_t scb[2] = {0u, 0u};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int cl = 2 * lane + half;       // tile column = staged row
          uint32_t out[8];
          const uint32_t abw = half ? (m2 & 0xFFFF0000u) : (m2 << 16);
          if constexpr (PERTENSOR) {
            if (!DO_ROW) amax_acc = max(amax_acc, abw);
            rne_col32<FMT>(w, half, mult, out);
          } else if constexpr (!EXTRA) {
            const bool bad = abw >= 0x7F800000u;
            const int e = scale_exp<FMT>(bad ? 0u : abw, p.ceil_mode);
            rne_col32<FMT>(w, half, exp2_neg(e), out);
            zero_if_bad(bad, out);
            scb[half] = bad ? 0xFFu : static_cast<uint32_t>(e + 127);
          } else {
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = half ? bf16hi(w[k]) : bf16lo(w[k]);
            uint32_t ab = abw;
            if (p.hadamard) {
              hadamard32(v, signs);
              ab = amax32_float(v);
            }
            const uint64_t idx0 = static_cast<uint64_t>(r0 + rb * 32) * static_cast<uint64_t>(p.cols) + (c0 + cl);
            scb[half] = quant_block32<FMT, EXTRA>(v, ab, p, idx0, static_cast<uint64_t>(p.cols), out);
          }
          if constexpr (FP4) {
            *reinterpret_cast<uint4*>(stg + cl * QBW) = make_uint4(out[0], out[1], out[2], out[3]);
          } else {
            *reinterpret_cast<uint4*>(stg + cl * QBW + (swz(cl, 0, QBW) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
            *reinterpret_cast<uint4*>(stg + cl * QBW + (swz(cl, 1, QBW) << 4)) = make_uint4(out[4], out[5], out[6], out[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&L.mc[jb], smem_u32(stg), FP4 ? (r0 + 32 * rb) / 2 : r0 + 32 * rb, c0);
          bulk_commit();
        }
        // column scales: one byte per column of the lane for this band
        if constexpr (!PERTENSOR) {
          const int kb = p.rows / 32, jb = r0 / 32 + rb;
          if (jb < kb) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int cl = 2 * lane + half;
              if (c0 + cl < p.cols) {
                size_t off;
                if (p.sf_mma) {   // full tiles only
                  const int cc = (c0 & 127) + cl;
                  off = (static_cast<size_t>(c0 / 128) * (p.rows / 128) + r0 / 128) * 512 + (cc & 31) * 16 +
                        ((cc >> 5) & 3) * 4 + rb;
                } else {
                  off = static_cast<size_t>(c0 + cl) * kb + jb;
                }
                p.s_col[off] = static_cast<uint8_t>(scb[half]);
              }
            }
          }
        }
      }

      // release the stage; the last of its readers issues its next load
      if (lane == 0) {
        const uint32_t old = atomicAdd(&cnt[s], 1u);
        if (old % ACTIVE == static_cast<uint32_t>(ACTIVE - 1) && blockIdx.x + (i + NSTG) * gridDim.x < ntiles)
          issue(i + NSTG);
      }
    }
    if (lane == 0) bulk_wait_all();
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    // a wait gave up: let every load still in flight land before the CTA ends
    for (int st = 0; st < NSTG; ++st)
      if (last_use[st] >= 0) (void)mbar_wait(smem_u32(&bars[st]), (last_use[st] / NSTG) & 1, p0.status);
  }

  if constexpr (PERTENSOR) {
    // block amax -> the ring's amax slot or amax_out; last block folds.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax_acc = max(amax_acc, __shfl_xor_sync(0xFFFFFFFFu, amax_acc, o));
    if (lane == 0) red[warp] = amax_acc;
    __syncthreads();
    if (tid == 0) {
      uint32_t m = 0;
      for (int k = 0; k < T::NW; ++k) m = max(m, red[k]);
      const int n = p0.hist_len;
      if (p0.ring == nullptr) {
        atomicMax(reinterpret_cast<unsigned int*>(p0.amax_out), m);
      } else {
        float* ring = p0.ring;
        atomicMax(reinterpret_cast<unsigned int*>(ring + n + 2), m);
        __threadfence();
        const unsigned int ticket = atomicAdd(reinterpret_cast<unsigned int*>(ring + n + 3), 1u);
        if (ticket == gridDim.x - 1) {
          __threadfence();
          volatile float* vr = ring;
          const float amax = vr[n + 2];
          if (p0.amax_out) *p0.amax_out = amax;
          fold_ring(vr, n, p0.hist_idx, amax, p0.fp8_max, p0.margin);
          __threadfence();
        }
      }
    }
  }
}

// The fold alone, of a given tensor amax: the step after the exchange of a
// row-sharded per-tensor quantize (each shard's amax_out, then a MAX
// reduction across the shards, then this fold on every replica of the ring).
__global__ void ring_fold_kernel(const float* __restrict__ amax, float* ring, int n, int hist_idx, float fp8_max,
                                 float margin) {
  grid_dep_wait();
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    fold_ring(ring, n, hist_idx, *amax, fp8_max, margin);
    __threadfence();
  }
}

// ---------------------------------------------------------------- dequantize
template <int FMT>
__global__ void dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t rows,
                               int64_t cols, int out_fp32, void* __restrict__ out) {
  // one thread: 16 consecutive elements of one row (inside one 32-block)
  const int64_t groups = rows * (cols / 16);
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < groups;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / (cols / 16), c = (g % (cols / 16)) * 16;
    const uint8_t sc = s[r * (cols / 32) + c / 32];
    const float X = (sc == 0xFF) ? __uint_as_float(0x7FC00000u)
                   : (sc == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(sc) << 23));
    float v[16];
    if constexpr (FMT == MXQ_E2M1) {
      const uint2 raw = *reinterpret_cast<const uint2*>(q + r * (cols / 2) + c / 2);
      const uint32_t wds[2] = {raw.x, raw.y};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint16_t b = static_cast<uint16_t>((wds[k >> 2] >> (8 * (k & 3))) & 0xFFu);
        uint32_t h2;
        asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(b));
        v[2 * k] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
        v[2 * k + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
      }
    } else {
      const uint4 raw = *reinterpret_cast<const uint4*>(q + r * cols + c);
      const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint16_t b = static_cast<uint16_t>((wds[k >> 1] >> (16 * (k & 1))) & 0xFFFFu);
        uint32_t h2;
        if constexpr (FMT == MXQ_E4M3) {
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(b));
        } else {
          asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(b));
        }
        v[2 * k] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
        v[2 * k + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
      }
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], X);
    if (out_fp32) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + r * cols + c);
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    } else {
      uint32_t b[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k]));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * k + 1]));
        b[k] = lo | (hi << 16);
      }
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + r * cols + c);
      o[0] = make_uint4(b[0], b[1], b[2], b[3]);
      o[1] = make_uint4(b[4], b[5], b[6], b[7]);
    }
  }
}

// ---------------------------------------------------------------- SF layout
__global__ void sf_to_mma_kernel(const uint8_t* __restrict__ s, int64_t rows, int64_t kb, uint8_t* __restrict__ out) {
  // one thread: the 4 scales of one row inside one 128-K chunk
  const int64_t n = rows * (kb / 4);
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < n;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / (kb / 4), kc = g % (kb / 4);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(s + r * kb + kc * 4);
    const int64_t off = ((r / 128) * (kb / 4) + kc) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4;
    *reinterpret_cast<uint32_t*>(out + off) = v;
  }
}

}  // namespace mxq

// ==================================================================== host
using namespace mxq;
using namespace mxq_host;

namespace {

constexpr int QTC = TileCfg<1, 1, false>::TC;
constexpr int QNST = MXQ_QUANT_NST;
// The stochastic-rounding / Hadamard variants are bound by their arithmetic;
// two stages serve them better than three (measured: SR, SR4 and the
// Hadamard RNE quantize of 4096 x 14336 about 3-5 % faster).
constexpr int QNST_EXTRA = 2;
constexpr int QSTG = MXQ_QUANT_STG;

template <int FMT, int ORIENT, bool PT, bool EXTRA, int NJ>
int launch_tiles(const QuantLaunch<NJ>& L, cudaStream_t st) {
  // column-only launches split the tiles between two warp groups, which
  // needs an even stage count (two per group for the lean variants)
  constexpr int NST = EXTRA ? QNST_EXTRA : (ORIENT == MXQ_COL ? 4 : QNST);
  using T = TileCfg<NST, QSTG, EXTRA, ORIENT == MXQ_ROW ? 1024 : 2048>;
  auto kern = quant_tiles_kernel<FMT, ORIENT, PT, EXTRA, NST, QSTG, NJ>;
  // stages, per-warp staging buffers, barriers and counters (256 B), alignment slack
  constexpr int smem = T::SMEM;
  static int per_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!per_sm[dev & 63]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MXQ_ERR_CUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, T::THREADS, smem) != cudaSuccess || n < 1)
      return MXQ_ERR_CUDA;
    per_sm[dev & 63] = n;
  }
  // as many rounds of tiles as the resident CTAs need, spread evenly over
  // the fewest CTAs that take them in that many rounds: every CTA then works
  // until the last round (the tail is at most one tile per CTA shorter)
  const int ntiles = L.tile_end[NJ - 1];
  const int slots = per_sm[dev & 63] * sm_count();
  const int rounds = (ntiles + slots - 1) / slots;
  const int grid = (ntiles + rounds - 1) / rounds;
  return launch_pdl(kern, dim3(grid), dim3(T::THREADS), smem, st, L, L.p[0]);
}

// A launch of one tensor (NJ = 1: every variant), or a group of RNE jobs
// (NJ > 1: the lean variants only).
template <bool PT, int NJ>
int dispatch(int fmt, int orient, const QuantLaunch<NJ>& L, cudaStream_t st) {
  const bool extra = !PT && (L.p[0].rounding != MXQ_RNE || L.p[0].hadamard);
  if (NJ > 1 && (PT || extra)) return MXQ_ERR_UNSUPPORTED;
#define MXQ_CASE(F, O)                                                                  \
  if (fmt == F && orient == O) {                                                        \
    if constexpr (NJ > 1) return launch_tiles<F, O, false, false, NJ>(L, st);          \
    else return extra ? launch_tiles<F, O, PT, !PT, 1>(L, st)                          \
                      : launch_tiles<F, O, PT, false, 1>(L, st);                       \
  }
  MXQ_CASE(MXQ_E4M3, MXQ_ROW) MXQ_CASE(MXQ_E4M3, MXQ_COL) MXQ_CASE(MXQ_E4M3, MXQ_DUAL)
  MXQ_CASE(MXQ_E5M2, MXQ_ROW) MXQ_CASE(MXQ_E5M2, MXQ_COL) MXQ_CASE(MXQ_E5M2, MXQ_DUAL)
  if constexpr (!PT) {
    MXQ_CASE(MXQ_E2M1, MXQ_ROW) MXQ_CASE(MXQ_E2M1, MXQ_COL) MXQ_CASE(MXQ_E2M1, MXQ_DUAL)
  }
#undef MXQ_CASE
  return MXQ_ERR_UNSUPPORTED;
}

bool valid_fmt(int f) { return f == MXQ_E4M3 || f == MXQ_E5M2 || f == MXQ_E2M1; }
bool valid_orient(int o) { return o == MXQ_ROW || o == MXQ_COL || o == MXQ_DUAL; }

CUtensorMapSwizzle swizzle_for(int pitch) {
  return pitch >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                      : (pitch == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                     : (pitch == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE));
}

// Tensor maps of the tile kernel: input boxes (128 rows x 64 bf16, 128-byte
// swizzle); row codes in boxes of one row warp's rows (32 in dual mode, 16
// row-only) x the tile's code bytes; transposed codes in boxes of the
// tile's 64 columns x one 32-row band of code bytes.  The staging swizzle
// follows the staged row pitch.
int make_maps(const void* x, int64_t rows, int64_t cols, int64_t ld, bool fp4, int orient, void* q_row,
              void* q_col, CUtensorMap* mx, CUtensorMap* mr, CUtensorMap* mc) {
  if (!encode_2d(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, cols, rows, ld * 2, QTC, TR, CU_TENSOR_MAP_SWIZZLE_128B))
    return MXQ_ERR_CUDA;
  *mr = *mx;
  *mc = *mx;
  if (orient & MXQ_ROW) {
    const uint64_t inner = fp4 ? cols / 2 : cols;
    const int qbr = fp4 ? QTC / 2 : QTC;
    const int rr = orient == MXQ_DUAL ? 32 : 16;
    if (!encode_2d(mr, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_row, inner, rows, inner, qbr, rr, swizzle_for(qbr)))
      return MXQ_ERR_CUDA;
  }
  if (orient & MXQ_COL) {
    const uint64_t inner = fp4 ? rows / 2 : rows;
    const int qbw = fp4 ? 16 : 32;
    if (!encode_2d(mc, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_col, inner, cols, inner, qbw, QTC, swizzle_for(qbw)))
      return MXQ_ERR_CUDA;
  }
  return MXQ_OK;
}

// Argument checks of one MX quantize of x [rows][cols] (row stride ld
// elements); the format and orientation are checked by the caller.
int check_mx_args(const void* x, int64_t rows, int64_t cols, int64_t ld, int orient, int scale_mode, int sf_layout,
                  const void* q_row, const uint8_t* s_row, const void* q_col, const uint8_t* s_col) {
  if (!x) return MXQ_ERR_BAD_ARG;
  if (scale_mode != MXQ_SCALE_FLOOR_OCP && scale_mode != MXQ_SCALE_CEIL) return MXQ_ERR_BAD_ARG;
  if (sf_layout != MXQ_SF_CANONICAL && sf_layout != MXQ_SF_MMA) return MXQ_ERR_BAD_ARG;
  if ((orient & MXQ_ROW) && (!q_row || !s_row)) return MXQ_ERR_BAD_ARG;
  if ((orient & MXQ_COL) && (!q_col || !s_col)) return MXQ_ERR_BAD_ARG;
  if (rows <= 0 || cols <= 0 || rows % 32 || cols % 32 || ld < cols) return MXQ_ERR_BAD_SHAPE;
  if (rows > (1ll << 31) - 256 || cols > (1ll << 31) - 256) return MXQ_ERR_BAD_SHAPE;
  if (sf_layout == MXQ_SF_MMA && (rows % 128 || cols % 128)) return MXQ_ERR_BAD_SHAPE;
  if (!aligned16(x) || ld % 8) return MXQ_ERR_MISALIGNED;
  if ((orient & MXQ_ROW) && !aligned16(q_row)) return MXQ_ERR_MISALIGNED;
  if ((orient & MXQ_COL) && !aligned16(q_col)) return MXQ_ERR_MISALIGNED;
  if (sf_layout == MXQ_SF_MMA && (((orient & MXQ_ROW) && !aligned16(s_row)) || ((orient & MXQ_COL) && !aligned16(s_col))))
    return MXQ_ERR_MISALIGNED;
  return MXQ_OK;
}

// Tiles of one tensor: 128-row x 64-column boxes, ragged edges included.
int64_t tile_count(int64_t rows, int64_t cols) { return ((cols + QTC - 1) / QTC) * ((rows + TR - 1) / TR); }

}  // namespace

extern "C" int mxq_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int fmt, int orient,
                            int scale_mode, int rounding, int hadamard32, uint64_t sr_key,
                            uint64_t hadamard_seed, int sf_layout, void* q_row, uint8_t* s_row, void* q_col,
                            uint8_t* s_col, void* stream) {
  if (!valid_fmt(fmt) || !valid_orient(orient)) return MXQ_ERR_BAD_ARG;
  if (rounding != MXQ_RNE && rounding != MXQ_SR && rounding != MXQ_SR4) return MXQ_ERR_BAD_ARG;
  const int rc0 = check_mx_args(x, rows, cols, ld, orient, scale_mode, sf_layout, q_row, s_row, q_col, s_col);
  if (rc0) return rc0;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;

  QuantLaunch<1> L{};
  int rc = make_maps(x, rows, cols, ld, fmt == MXQ_E2M1, orient, q_row, q_col, &L.mx[0], &L.mr[0], &L.mc[0]);
  if (rc) return rc;
  QuantParams& p = L.p[0];
  p.rows = static_cast<int>(rows);
  p.cols = static_cast<int>(cols);
  p.tiles_c = static_cast<int>((cols + QTC - 1) / QTC);
  p.ntiles = p.tiles_c * static_cast<int>((rows + TR - 1) / TR);
  p.ceil_mode = scale_mode == MXQ_SCALE_CEIL;
  p.rounding = rounding;
  p.hadamard = hadamard32 != 0;
  p.sf_mma = sf_layout == MXQ_SF_MMA;
  p.sr_k0 = static_cast<uint32_t>(sr_key);
  p.sr_k1 = static_cast<uint32_t>(sr_key >> 32);
  p.had_k0 = static_cast<uint32_t>(hadamard_seed);
  p.had_k1 = static_cast<uint32_t>(hadamard_seed >> 32);
  p.s_row = s_row;
  p.s_col = s_col;
  p.status = status_ptr();
  p.stall_tile = take_test_stall(1) ? 0 : -1;
  if (!p.status) return MXQ_ERR_CUDA;
  L.tile_end[0] = p.ntiles;
  return dispatch<false>(fmt, orient, L, static_cast<cudaStream_t>(stream));
}

extern "C" int mxq_quantize_group(const mxq_quant_job* jobs, int njobs, int fmt, int orient, int sf_layout,
                                  void* stream) {
  if (!jobs || njobs < 1 || njobs > MXQ_QUANT_GROUP_MAX || !valid_fmt(fmt) || !valid_orient(orient))
    return MXQ_ERR_BAD_ARG;
  int64_t total = 0;
  for (int j = 0; j < njobs; ++j) {
    const mxq_quant_job& J = jobs[j];
    const int rc = check_mx_args(J.x, J.rows, J.cols, J.ld, orient, J.scale_mode, sf_layout, J.q_row, J.s_row,
                                 J.q_col, J.s_col);
    if (rc) return rc;
    total += tile_count(J.rows, J.cols);
  }
  if (total > (1ll << 31) - 1) return MXQ_ERR_BAD_SHAPE;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  int* status = status_ptr();
  if (!status) return MXQ_ERR_CUDA;
  QuantLaunch<MXQ_QUANT_GROUP_MAX> L{};
  int end = 0;
  for (int j = 0; j < MXQ_QUANT_GROUP_MAX; ++j) {
    if (j >= njobs) {                          // unused: never reached (its tiles end where the last job's do)
      L.mx[j] = L.mx[0];
      L.mr[j] = L.mr[0];
      L.mc[j] = L.mc[0];
      L.p[j] = L.p[0];
      L.tile_end[j] = end;
      continue;
    }
    const mxq_quant_job& J = jobs[j];
    const int rc = make_maps(J.x, J.rows, J.cols, J.ld, fmt == MXQ_E2M1, orient, J.q_row, J.q_col, &L.mx[j],
                             &L.mr[j], &L.mc[j]);
    if (rc) return rc;
    QuantParams& p = L.p[j];
    p.rows = static_cast<int>(J.rows);
    p.cols = static_cast<int>(J.cols);
    p.tiles_c = static_cast<int>((J.cols + QTC - 1) / QTC);
    p.ntiles = static_cast<int>(tile_count(J.rows, J.cols));
    p.ceil_mode = J.scale_mode == MXQ_SCALE_CEIL;
    p.rounding = MXQ_RNE;
    p.sf_mma = sf_layout == MXQ_SF_MMA;
    p.s_row = J.s_row;
    p.s_col = J.s_col;
    p.status = status;
    p.stall_tile = -1;
    end += p.ntiles;
    L.tile_end[j] = end;
  }
  return dispatch<false>(fmt, orient, L, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_quantize_pertensor(const void* x, int64_t rows, int64_t cols, const float* scale, int fmt,
                                      int orient, float* ring_state, int hist_len, int hist_idx, float fp8_max,
                                      float pow2_margin, uint8_t* x8, uint8_t* x8T, float* amax_out,
                                      void* stream) {
  if (!x || !scale || (fmt != MXQ_E4M3 && fmt != MXQ_E5M2) || !valid_orient(orient)) return MXQ_ERR_BAD_ARG;
  if ((orient & MXQ_ROW) && !x8) return MXQ_ERR_BAD_ARG;
  if ((orient & MXQ_COL) && !x8T) return MXQ_ERR_BAD_ARG;
  if (!ring_state && !amax_out) return MXQ_ERR_BAD_ARG;
  if (ring_state && (hist_len < 1 || hist_idx < 0 || hist_idx >= hist_len)) return MXQ_ERR_BAD_ARG;
  if (rows <= 0 || cols <= 0 || cols % 16) return MXQ_ERR_BAD_SHAPE;
  if ((orient & MXQ_COL) && rows % 16) return MXQ_ERR_BAD_SHAPE;
  if (rows > (1ll << 31) - 256 || cols > (1ll << 31) - 256) return MXQ_ERR_BAD_SHAPE;
  if (!aligned16(x) || ((orient & MXQ_ROW) && !aligned16(x8)) || ((orient & MXQ_COL) && !aligned16(x8T)))
    return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  QuantLaunch<1> L{};
  int rc = make_maps(x, rows, cols, cols, false, orient, x8, x8T, &L.mx[0], &L.mr[0], &L.mc[0]);
  if (rc) return rc;
  QuantParams& p = L.p[0];
  p.rows = static_cast<int>(rows);
  p.cols = static_cast<int>(cols);
  p.tiles_c = static_cast<int>((cols + QTC - 1) / QTC);
  p.ntiles = p.tiles_c * static_cast<int>((rows + TR - 1) / TR);
  p.status = status_ptr();
  if (!p.status) return MXQ_ERR_CUDA;
  p.scale = scale;
  p.ring = ring_state;
  p.hist_len = hist_len;
  p.hist_idx = hist_idx;
  p.fp8_max = fp8_max;
  p.margin = pow2_margin;
  p.amax_out = amax_out;
  p.stall_tile = -1;
  if (!ring_state) {
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return MXQ_ERR_CUDA;
  }
  L.tile_end[0] = p.ntiles;
  return dispatch<true>(fmt, orient, L, st);
}

extern "C" int fp8_ring_fold(const float* amax, float* ring_state, int hist_len, int hist_idx, float fp8_max,
                             float pow2_margin, void* stream) {
  if (!amax || !ring_state || hist_len < 1 || hist_idx < 0 || hist_idx >= hist_len) return MXQ_ERR_BAD_ARG;
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) || (reinterpret_cast<uintptr_t>(ring_state) & 3u))
    return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  return launch_pdl(ring_fold_kernel, dim3(1), dim3(32), 0, static_cast<cudaStream_t>(stream), amax, ring_state,
                    hist_len, hist_idx, fp8_max, pow2_margin);
}

extern "C" int mxq_dequantize(const void* q, const uint8_t* s, int64_t rows, int64_t cols, int fmt, int out_fp32,
                              void* out, void* stream) {
  if (!q || !s || !out || !valid_fmt(fmt)) return MXQ_ERR_BAD_ARG;
  if (rows <= 0 || cols <= 0 || cols % 32) return MXQ_ERR_BAD_SHAPE;
  if (!aligned16(q) || !aligned16(out)) return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  const int64_t groups = rows * (cols / 16);
  const int grid = static_cast<int>(std::min<int64_t>((groups + 255) / 256, 8ll * sm_count()));
  auto st = static_cast<cudaStream_t>(stream);
  const uint8_t* qb = static_cast<const uint8_t*>(q);
  if (fmt == MXQ_E4M3) dequant_kernel<MXQ_E4M3><<<grid, 256, 0, st>>>(qb, s, rows, cols, out_fp32, out);
  else if (fmt == MXQ_E5M2) dequant_kernel<MXQ_E5M2><<<grid, 256, 0, st>>>(qb, s, rows, cols, out_fp32, out);
  else dequant_kernel<MXQ_E2M1><<<grid, 256, 0, st>>>(qb, s, rows, cols, out_fp32, out);
  return launch_status();
}

extern "C" int mxq_sf_to_mma(const uint8_t* s, int64_t rows, int64_t kb, uint8_t* out, void* stream) {
  if (!s || !out) return MXQ_ERR_BAD_ARG;
  if (rows <= 0 || kb <= 0 || rows % 128 || kb % 4) return MXQ_ERR_BAD_SHAPE;
  if ((reinterpret_cast<uintptr_t>(s) & 3) || (reinterpret_cast<uintptr_t>(out) & 3)) return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  const int64_t n = rows * (kb / 4);
  const int grid = static_cast<int>(std::min<int64_t>((n + 255) / 256, 8ll * sm_count()));
  sf_to_mma_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(s, rows, kb, out);
  return launch_status();
}
