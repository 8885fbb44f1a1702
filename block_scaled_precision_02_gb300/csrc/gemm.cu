// GEMMs on the sm_103a tensor cores, C = A * B^T with float32 accumulation
// in tensor memory (block-scaled operands K-contiguous; per-tensor FP8
// operands K-contiguous or M / N-contiguous):
//  * block-scaled (MX):
//      C[m][n] = sum_k dec(a[m][k]) 2^(sa[m][k/32]-127) dec(b[n][k]) 2^(sb[n][k/32]-127)
//    Source: "UE8M0 FP8 / MXFP8 explainer", section 1 -- tensor cores consume
//    the UE8M0 scale X and the element codes q_i of both operands, block by
//    block, and accumulate in FP32; gap section 2 -- the blocks must run
//    along the contiguous reduction dimension.  Output bf16 or float32, or
//    (format-aware fusion: the producer writes its consumer's format) MX
//    codes and scales of 1 x 32 row blocks quantized from the accumulator.
//  * per-tensor FP8 (AstrAI fp8.py, mm_fp8): C = (A * B^T) * scale + bias,
//    bf16 out, optionally batched; an operand stored [K][M] / [K][N] is read
//    in place through MN-major tiles.
//
// Two kernels share the warp roles below.
//  * CTA pair (M and N multiples of 256): clusters of two CTAs on two SMs
//    compute one 256 x 256 tile with tcgen05.mma.cta_group::2.  Each CTA
//    holds its own 128 rows of A and one 128-row half of B; the tensor cores
//    of the pair exchange the B halves, so each SM streams 32 KB of operands
//    per K step instead of 48 KB.  Scale chunks: each CTA holds its own rows
//    of A's scales and all 256 rows of B's; one tcgen05.cp.cta_group::2
//    fills both CTAs' tensor memory from the same offset.
//    Tiles run in waves of consecutive indices, ordered so the smaller
//    operand stays in L2.  A stream-K variant (a separate instantiation)
//    evens out a sparse last wave by splitting k-ranges over the pairs; cut
//    tiles meet through a caller workspace or the library's static scratch.
//  * single CTA (otherwise): 128 x BN tiles, tcgen05.mma.cta_group::1.
// Roles (one CTA per SM, persistent over output tiles):
//  * warp 0      TMA producer: per K step (128 bytes of codes per row) the
//                A and B tiles with the 128-byte swizzle, plus the matching
//                512-byte scale chunks (the quantizer already wrote them in
//                the tensor-core layout), into a ring of stages.
//  * warp 1      allocates tensor memory; one thread (of the pair's first
//                CTA) issues 4 tcgen05.mma per stage (E4M3/E5M2 block-scaled:
//                kind::mxf8f6f4, scale_vec::1X, K = 32; E2M1: kind::mxf4,
//                scale_vec::2X, K = 64; per-tensor FP8: kind::f8f6f4), then
//                tcgen05.commit to free the stage (in both CTAs of a pair).
//                The single-CTA kernel issues the tcgen05.cp of the scale
//                chunks into tensor memory from the same thread; the pair
//                kernel leaves them to warp 6, which runs ahead of the MMAs.
//  * warps 2..5  epilogue: tcgen05.ld of this CTA's 128 x N float32
//                accumulator rows (each thread owns one row), conversion,
//                and stores (TMA through two 64-byte-swizzled staging
//                buffers, one for MXFP4; the MX output is stored directly).  The pair
//                kernel's MX-output variants add warps 7..10, a second
//                epilogue group that takes the other half of the columns,
//                and read all of a group's columns into registers before
//                releasing the accumulator.
// Operands: E4M3 / E5M2 / E2M1 in any pairing.  Packed E2M1 beside an 8-bit
// operand is widened to one byte per code by its tensor map on the way into
// shared memory (the 4-bit layout of kind::mxf8f6f4), so both operands then
// share the 8-bit tile layout.
// Every wait is bounded (1 s); on expiry the status word records
// MXQ_ERR_TIMEOUT, all roles wind down, in-flight copies are awaited (with a
// limit) and tensor memory is released.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace mxq {
namespace gemm {

constexpr int BM = 128;
constexpr int BKB = 128;                 // bytes of codes per row per stage
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int PAIR_THREADS = 224;     // pair kernel: the roles above plus warp 6 (scale copies)
constexpr int STG_BYTES = BM * 64;       // one staging buffer: 128 rows x 64 B
// Transpose scratch of one epilogue warp (MX column-block output): its
// 32 x 32 chunk, row k at word k * XS_PITCH.  A pitch of 36 words keeps
// 16-byte row writes (eight lanes per access phase, banks 4 k .. 4 k + 3
// apart) and column reads (lane j at bank 4 k + j) free of bank conflicts.
constexpr int XS_PITCH = 36;
constexpr int XS_WORDS = 32 * XS_PITCH;
constexpr int XS_GROUP_BYTES = 4 * XS_WORDS * 4;    // four epilogue warps
// the staging area: two buffers, also the four epilogue warps' transpose scratch
constexpr int OUT_BYTES = std::max(2 * STG_BYTES + 512, XS_GROUP_BYTES);

// Operand kinds (a template parameter of both kernels).
constexpr int KIND_MXF8 = 0;   // block-scaled E4M3 / E5M2: kind::mxf8f6f4, scale_vec::1X
constexpr int KIND_MXF4 = 1;   // block-scaled E2M1 (packed): kind::mxf4, scale_vec::2X
constexpr int KIND_F8 = 2;     // per-tensor E4M3 / E5M2: kind::f8f6f4, no block scales

// Epilogue modes.
constexpr int EPI_BF16 = 0;    // bf16 (RNE); per-tensor kind: RN32(RN32(acc * scale) + bias) first
constexpr int EPI_FP32 = 1;    // float32 accumulator as is
constexpr int EPI_MX = 2;      // MX codes + UE8M0 scales of 1 x 32 row blocks

struct Params {
  const uint8_t* a_s;
  const uint8_t* b_s;
  int M, N, K;
  int tiles_m, tiles_n, ntiles;   // tiles_m x tiles_n per product; ntiles over all batches
  int kblocks;        // K steps of BKB bytes
  int kb4;            // 512-byte scale chunks per 128 rows (K / 128)
  int a_batched, b_batched;       // 1: operand rows advance by M (N) per batch; 0: shared
  int epi;
  const float* alpha;             // per-tensor kind: combined dequantization scale (device scalar)
  const __nv_bfloat16* bias;      // per-tensor kind: bias[N] or nullptr
  uint8_t* cq;                    // EPI_MX: codes [M][N]
  uint8_t* cs;                    // EPI_MX: scales, canonical [M][N/32] or the MMA layout
  uint8_t* cqT;                   // EPI_MX column blocks: codes of C^T [N][M] (or nullptr)
  uint8_t* csT;                   // EPI_MX column blocks: scales, canonical [N][M/32] or the MMA layout
  int mx_fmt, mx_ceil, mx_sf_mma;
  int* status;
  uint32_t a_type, b_type;   // element type codes of the instruction descriptor
  int a_mn, b_mn;     // per-tensor kind: operand stored MN-major ([K][M] / [K][N] rows), else K-major
  int m_fast;         // tile order: M index fastest (A resident in L2), else N fastest
  // stream-K (CTA-pair kernel, bf16 / float32 output of block-scaled kinds):
  // tiles [0, sk_dp) go round-robin over the pairs; the k-iterations of the
  // rest are split into even ranges, one per pair.  A tile cut by a range
  // boundary b is finished by whichever of its two pieces ends second, which
  // adds the float32 sums the other parked in workspace slot b.
  int sk;             // 1: stream-K schedule
  int sk_dp;          // tiles of the round-robin part
  float* sk_part;     // per slot and CTA half: 256 columns x 128 rows of float32 (column-major)
  uint32_t* sk_flags; // per slot and CTA half: ticket word, ready word
  uint32_t sk_epoch;  // this launch's tag (tickets and ready words never need clearing)
  uint32_t tx_bytes;  // bytes the loads of one stage complete on its "full" barrier (both CTAs of a pair)
  int stall_u;        // failure-detection test hook: CTA 0 never fills this stage use (-1: off)
};

// Batch, first row and first column of output tile `tile` (tm x tn tiles).
struct TilePos {
  int b, m0, n0;
};
// Tiles run in waves of consecutive indices.  With m_fast the index walks
// down M first, so a wave covers every M tile of a few N columns and A stays
// in L2 while B streams through once; otherwise N runs first and B stays.
// The host picks the order that keeps the smaller operand resident.
__device__ __forceinline__ TilePos tile_pos(const Params& p, int tile, int tm, int tn) {
  const int per = p.tiles_m * p.tiles_n;
  const int b = tile / per, r = tile - b * per;
  if (p.m_fast) return {b, (r % p.tiles_m) * tm, (r / p.tiles_m) * tn};
  return {b, (r / p.tiles_n) * tm, (r % p.tiles_n) * tn};
}

// One piece of work of a CTA pair: k-blocks [kb0, kb1) of output tile
// `tile`.  slot > 0: the tile is cut at range boundary `slot` (the other piece
// belongs to the neighbouring pair); slot == 0: the whole tile.
struct Seg {
  int tile, kb0, kb1, slot;
};

// The pieces of pair `pair`, in order.  Without stream-K: tiles pair,
// pair + npairs, ...  With it: those of the round-robin part, then the pair's
// contiguous range of the remaining k-iterations (iteration = tile *
// kblocks + k-block).  The host guarantees every range is at least one tile
// long, so a tile is cut at most once.
template <bool SK>
struct SegIter {
  int tile, step, dp, kblocks, pair;
  int64_t it, hi;
  __device__ __forceinline__ SegIter(const Params& p, int pair_, int npairs) {
    pair = pair_;
    tile = pair_;
    step = npairs;
    kblocks = p.kblocks;
    dp = SK ? p.sk_dp : p.ntiles;
    it = hi = 0;
    if (SK) {
      const int64_t base = static_cast<int64_t>(p.sk_dp) * p.kblocks;
      const int64_t rest = static_cast<int64_t>(p.ntiles - p.sk_dp) * p.kblocks;
      it = base + rest * pair_ / npairs;
      hi = base + rest * (pair_ + 1) / npairs;
    }
  }
  __device__ __forceinline__ bool next(Seg& sg) {
    if (tile < dp) {
      sg = Seg{tile, 0, kblocks, 0};
      tile += step;
      return true;
    }
    if (!SK || it >= hi) return false;
    const int t = static_cast<int>(it / kblocks);
    const int k0 = static_cast<int>(it - static_cast<int64_t>(t) * kblocks);
    const int k1 = static_cast<int>(min(static_cast<int64_t>(kblocks), k0 + (hi - it)));
    sg = Seg{t, k0, k1, k0 > 0 ? pair : (k1 < kblocks ? pair + 1 : 0)};
    it += k1 - k0;
    return true;
  }
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- tcgen05 wrappers
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int KIND>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
  if constexpr (KIND == KIND_MXF4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
  } else if constexpr (KIND == KIND_MXF8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
  }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// CTA-pair forms: issued by one thread of the pair's first CTA (alloc and
// dealloc by one warp of each CTA); shared-memory descriptors and tensor
// memory addresses name the same offsets in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// arrive on the mbarrier at this offset in both CTAs once the issued work is done
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
  const uint16_t mask = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_self(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
template <int KIND>
__device__ __forceinline__ void tc_mma_pair(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t acc) {
  if constexpr (KIND == KIND_MXF4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
  } else if constexpr (KIND == KIND_MXF8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
  }
}

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (>> 4), fixed version field 1 at bit 46, swizzle
// mode at bits 61-63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(swz & 7u) << 61;
  return d;
}

// Instruction descriptor of the block-scaled MMA: A and B element type codes
// at bits 7-9 and 10-12 (kind::mxf8f6f4: E4M3 0, E5M2 1; kind::mxf4: E2M1 1),
// K-major operands, N >> 3 at bits 17-22, scale type UE8M0 (bit 23), M >> 4
// at bits 24-28, scale-factor byte selectors for B (bits 4-5) and A (29-30).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t a_type, uint32_t b_type, int n, int m, uint32_t sf_id) {
  return (sf_id << 4) | (a_type << 7) | (b_type << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24) | (sf_id << 29);
}

// Instruction descriptor of the unscaled kind::f8f6f4 MMA: float32
// accumulator (bits 4-5 = 1), A / B element types at bits 7-9 / 10-12,
// A / B major-ness at bits 15 / 16 (0 K-major, 1 MN-major), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t instr_desc_f8(uint32_t a_type, uint32_t b_type, int n, int m, uint32_t a_mn,
                                                     uint32_t b_mn) {
  return (1u << 4) | (a_type << 7) | (b_type << 10) | (a_mn << 15) | (b_mn << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Shared-memory descriptor of an operand tile and the descriptor step from
// one 32-byte K slice to the next (16-byte units).  Both layouts are what a
// TMA load with the 128-byte swizzle writes: K-major -- 128-byte rows along
// K, one per M (N) index, 8-row groups 1024 bytes apart; MN-major -- 128-byte
// rows along M (N), one per K index (the tile is 128 elements wide: a single
// swizzle atom across), 8-row groups along K 1024 bytes apart, so a 32-deep
// K slice is 32 rows = 4096 bytes.  An MN-major tile has one atom across,
// so the atom stride across M (N) is never used; it is set to the 8-row
// group stride as well.
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr, int mn) {
  return mn ? smem_desc(addr, 1024, 1024, 2) : smem_desc(addr, 16, 1024, 2);
}
__device__ __forceinline__ uint32_t k_slice_step(int mn) { return mn ? 256u : 2u; }

template <int KIND>
__device__ __forceinline__ uint32_t mma_idesc(const Params& p, int n, int m, int kk) {
  if constexpr (KIND == KIND_F8)
    return instr_desc_f8(p.a_type, p.b_type, n, m, static_cast<uint32_t>(p.a_mn), static_cast<uint32_t>(p.b_mn));
  else return instr_desc(p.a_type, p.b_type, n, m, KIND == KIND_MXF4 ? (kk & 1) * 2 : kk);
}

// Bits of the largest magnitude among the 32 float32 words of a block
// (NaN anywhere: NaN bits; an infinity: 0x7F800000).
__device__ __forceinline__ uint32_t amax32_bits(const uint32_t (&v)[32]) {
  return amax32_tree([&](int j) { return fabsf(__uint_as_float(v[j])); });
}

// FP8 codes of four float32 words each multiplied by m (mm = m twice; one
// packed multiply per pair, rounded to nearest like the scalar product),
// converted RNE-saturating; the first word's code in the lowest byte.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4_scaled(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint64_t mm) {
  uint32_t r;
  if constexpr (FMT == MXQ_E4M3) {
    asm("{\n\t.reg .b64 pa, pb;\n\t.reg .b32 a0, a1, b0, b1;\n\t.reg .b16 t0, t1;\n\t"
        "mov.b64 pa, {%1, %2};\n\tmov.b64 pb, {%3, %4};\n\t"
        "mul.rn.f32x2 pa, pa, %5;\n\tmul.rn.f32x2 pb, pb, %5;\n\t"
        "mov.b64 {a0, a1}, pa;\n\tmov.b64 {b0, b1}, pb;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t0, a1, a0;\n\tcvt.rn.satfinite.e4m3x2.f32 t1, b1, b0;\n\t"
        "mov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r) : "r"(a), "r"(b), "r"(c), "r"(d), "l"(mm));
  } else {
    asm("{\n\t.reg .b64 pa, pb;\n\t.reg .b32 a0, a1, b0, b1;\n\t.reg .b16 t0, t1;\n\t"
        "mov.b64 pa, {%1, %2};\n\tmov.b64 pb, {%3, %4};\n\t"
        "mul.rn.f32x2 pa, pa, %5;\n\tmul.rn.f32x2 pb, pb, %5;\n\t"
        "mov.b64 {a0, a1}, pa;\n\tmov.b64 {b0, b1}, pb;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 t0, a1, a0;\n\tcvt.rn.satfinite.e5m2x2.f32 t1, b1, b0;\n\t"
        "mov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r) : "r"(a), "r"(b), "r"(c), "r"(d), "l"(mm));
  }
  return r;
}

// E2M1 codes of eight float32 words each multiplied by m (packed multiplies
// as above), RNE-saturating, packed two per byte: the first word's code in
// the lowest nibble.
__device__ __forceinline__ uint32_t e2m1x8_scaled(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                                  uint32_t f, uint32_t g, uint32_t h, uint64_t mm) {
  uint32_t r;
  asm("{\n\t.reg .b64 p0, p1, p2, p3;\n\t.reg .b32 x<8>;\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "mov.b64 p0, {%1, %2};\n\tmov.b64 p1, {%3, %4};\n\tmov.b64 p2, {%5, %6};\n\tmov.b64 p3, {%7, %8};\n\t"
      "mul.rn.f32x2 p0, p0, %9;\n\tmul.rn.f32x2 p1, p1, %9;\n\t"
      "mul.rn.f32x2 p2, p2, %9;\n\tmul.rn.f32x2 p3, p3, %9;\n\t"
      "mov.b64 {x0, x1}, p0;\n\tmov.b64 {x2, x3}, p1;\n\tmov.b64 {x4, x5}, p2;\n\tmov.b64 {x6, x7}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, x1, x0;\n\tcvt.rn.satfinite.e2m1x2.f32 t1, x3, x2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, x5, x4;\n\tcvt.rn.satfinite.e2m1x2.f32 t3, x7, x6;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r) : "r"(a), "r"(b), "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h), "l"(mm));
  return r;
}

// MX quantization of one 32-value row block of the accumulator: the scale
// rule of the quantizer (floor or ceil on the block amax's exponent and
// mantissa bits), then codes = RNE-saturating FP8 of v * 2^-e (exact
// product).  A block holding NaN or Inf gets scale 0xFF and zero codes.
template <int FMT>
__device__ __forceinline__ uint32_t mx_block32_fmt(const uint32_t (&v)[32], int ceil_mode, uint32_t* codes) {
  const uint32_t ab = amax32_bits(v);
  const bool bad = ab >= 0x7F800000u;
  const int e = bad ? 0 : scale_exp<FMT>(ab, ceil_mode);
  const uint64_t mm = f32x2_splat(exp2_neg(e));
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t x = fp8x4_scaled<FMT>(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3], mm);
    codes[k] = bad ? 0u : x;
  }
  return bad ? 0xFFu : static_cast<uint32_t>(e + 127);
}
__device__ __forceinline__ uint32_t mx_block32(const uint32_t (&v)[32], int fmt, int ceil_mode,
                                               uint32_t* codes /* 8 words */) {
  return fmt == MXQ_E4M3 ? mx_block32_fmt<MXQ_E4M3>(v, ceil_mode, codes)
                         : mx_block32_fmt<MXQ_E5M2>(v, ceil_mode, codes);
}

// The same for E2M1 output: codes in 4 words, eight nibbles each (element 0
// in the lowest nibble).
__device__ __forceinline__ uint32_t mx_block32_e2m1(const uint32_t (&v)[32], int ceil_mode, uint32_t* codes /* 4 words */) {
  const uint32_t ab = amax32_bits(v);
  const bool bad = ab >= 0x7F800000u;
  const int e = bad ? 0 : scale_exp<MXQ_E2M1>(ab, ceil_mode);
  const uint64_t mm = f32x2_splat(exp2_neg(e));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t x = e2m1x8_scaled(v[8 * k], v[8 * k + 1], v[8 * k + 2], v[8 * k + 3], v[8 * k + 4], v[8 * k + 5],
                                     v[8 * k + 6], v[8 * k + 7], mm);
    codes[k] = bad ? 0u : x;
  }
  return bad ? 0xFFu : static_cast<uint32_t>(e + 127);
}

// One MX block of the output format (FP4O: E2M1, else p.mx_fmt), codes
// stored at dst (32 bytes of FP8 or 16 of packed E2M1); returns the scale.
template <bool FP4O>
__device__ __forceinline__ uint32_t mx_block_store(const uint32_t (&v)[32], const Params& p, uint8_t* dst) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  if constexpr (FP4O) {
    uint32_t c[4];
    const uint32_t s = mx_block32_e2m1(v, p.mx_ceil, c);
    d[0] = make_uint4(c[0], c[1], c[2], c[3]);
    return s;
  } else {
    uint32_t c[8];
    const uint32_t s = mx_block32(v, p.mx_fmt, p.mx_ceil, c);
    d[0] = make_uint4(c[0], c[1], c[2], c[3]);
    d[1] = make_uint4(c[4], c[5], c[6], c[7]);
    return s;
  }
}

// Column `lane` of the warp's chunk, read once from the transpose scratch.
__device__ __forceinline__ void load_col32(const uint32_t* xs, int lane, uint32_t (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k) v[k] = xs[k * XS_PITCH + lane];
}

// Row-block scale words of one output row (BN / 32 scale bytes, four per
// word, scale columns n0 / 32 ..) in the canonical or the MMA layout.
template <int BN>
__device__ __forceinline__ void store_row_scales(const Params& p, size_t rg, int n0, const uint32_t (&sc)[BN / 128]) {
  const int kb = p.N / 32;                                       // scale columns
#pragma unroll
  for (int g = 0; g < BN / 128; ++g) {
    const int j0 = n0 / 32 + 4 * g;                              // first scale column of this word
    size_t off;
    if (p.mx_sf_mma)                                             // chunk (rg/128, j0/4), row rg%32, word (rg/32)%4
      off = ((rg / 128) * static_cast<size_t>(kb / 4) + j0 / 4) * 512 + (rg % 32) * 16 + ((rg / 32) % 4) * 4;
    else
      off = rg * static_cast<size_t>(kb) + j0;
    *reinterpret_cast<uint32_t*>(p.cs + off) = sc[g];
  }
}

// Epilogue of one output tile: drain this CTA's 128 x BN float32
// accumulator (tensor-memory lanes 0..127, columns 0..BN-1; the thread of
// lane quarter q and lane `lane` owns row 32 q + lane), call release() once
// it has been read completely, and store it to C[m0 .., n0 ..] (rows of the
// whole batched output) in the mode p.epi.  bf16 / float32 go through NBUF
// (two, or one) 64-byte-swizzled staging buffers and TMA stores issued by `leader`; all
// 128 epilogue threads take part (named barrier 1).
// Before a staging buffer is rewritten: with two buffers the bulk store
// issued from this one two chunks ago must have read it (at most one store
// group still reading); with one buffer the last store must have.
template <int NBUF>
__device__ __forceinline__ void bulk_wait_read_staging() {
  if constexpr (NBUF == 2) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
  else asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

template <int BN, bool PER_TENSOR, int MXOUT, int NBUF, typename Release>
__device__ __forceinline__ void store_tile(const Params& p, float alpha, uint32_t tmem, int q, int lane, bool leader,
                                           int& buf, uint8_t* sOut, const CUtensorMap* map_c, int m0, int n0,
                                           Release release) {
  // MX outputs: 1 rows, 2 rows + columns (FP8 codes); 3, 4 the same in E2M1
  constexpr int ORI = MXOUT > 2 ? MXOUT - 2 : MXOUT;
  constexpr bool FP4O = MXOUT > 2;
  constexpr int CSH = FP4O ? 1 : 0;                        // E2M1: half a byte per code
  const int row = q * 32 + lane;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
  if (MXOUT == 0 && p.epi == EPI_BF16) {
    // drain the whole accumulator row into registers first, so the MMA warp
    // can start the next tile while this one is written out (two 32-column
    // loads in flight per wait)
    uint32_t pk[BN / 2];
#pragma unroll
    for (int c = 0; c < BN / 32; c += 2) {
      uint32_t v[2][32];
      tmem_ld32(lane_addr + c * 32, v[0]);
      tmem_ld32(lane_addr + (c + 1) * 32, v[1]);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x0 = __uint_as_float(v[h][2 * j]), x1 = __uint_as_float(v[h][2 * j + 1]);
          if constexpr (PER_TENSOR) {
            x0 = __fmul_rn(x0, alpha);
            x1 = __fmul_rn(x1, alpha);
            if (p.bias) {
              const __nv_bfloat162 bb =
                  *reinterpret_cast<const __nv_bfloat162*>(p.bias + n0 + (c + h) * 32 + 2 * j);
              x0 = __fadd_rn(x0, __low2float(bb));
              x1 = __fadd_rn(x1, __high2float(bb));
            }
          }
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(x0, x1);
          pk[(c + h) * 16 + j] = *reinterpret_cast<const uint32_t*>(&b2);
        }
    }
    tc_fence_before();
    __syncwarp();
    release();
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      if (leader) bulk_wait_read_staging<NBUF>();
      named_bar(1, 128);
      uint8_t* stg = sOut + buf * STG_BYTES;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int phys = j ^ ((row >> 1) & 3);                   // 64-byte swizzle
        *reinterpret_cast<uint4*>(stg + row * 64 + phys * 16) =
            make_uint4(pk[c * 16 + 4 * j], pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2], pk[c * 16 + 4 * j + 3]);
      }
      fence_proxy_async_smem();
      named_bar(1, 128);
      if (leader) {
        tma_store_2d(map_c, smem_u32(stg), n0 + c * 32, m0);
        bulk_commit();
      }
      buf ^= NBUF - 1;
    }
    return;
  }
  if constexpr (MXOUT != 0 && BN <= 128) {
    // At most 128 columns per thread (the pair kernel's two epilogue
    // groups): read all of them into registers and release the accumulator
    // first, so the MMAs of the next tile run while this one is quantized.
    uint32_t v[BN / 32][32];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) tmem_ld32(lane_addr + c * 32, v[c]);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    release();
    uint32_t sc[BN / 128 > 0 ? BN / 128 : 1];
#pragma unroll
    for (int g = 0; g < (BN / 128 > 0 ? BN / 128 : 1); ++g) sc[g] = 0;
    uint32_t* xs = reinterpret_cast<uint32_t*>(sOut) + q * XS_WORDS;    // this warp's transpose scratch
    const size_t rg = static_cast<size_t>(m0 + row);
    const size_t rT = static_cast<size_t>(m0 + q * 32);          // first row of the warp's column blocks
    const bool rows_out = ORI == 1 || p.cq, cols_out = ORI == 2 && p.cqT;
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      if (rows_out) {
        const uint32_t s8 =
            mx_block_store<FP4O>(v[c], p, p.cq + ((rg * static_cast<size_t>(p.N) + n0 + c * 32) >> CSH));
        sc[c >> 2] |= s8 << (8 * (c & 3));
      }
      if (cols_out) {
        // a warp's 32 rows of the chunk are 32 column blocks: transposed
        // through the warp's scratch, lane j takes column j
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(xs + lane * XS_PITCH + 4 * j) =
              make_uint4(v[c][4 * j], v[c][4 * j + 1], v[c][4 * j + 2], v[c][4 * j + 3]);
        __syncwarp();
        uint32_t col[32];
        load_col32(xs, lane, col);
        __syncwarp();
        const size_t n = static_cast<size_t>(n0 + c * 32 + lane);
        const uint32_t sT = mx_block_store<FP4O>(col, p, p.cqT + ((n * static_cast<size_t>(p.M) + rT) >> CSH));
        const size_t kbT = static_cast<size_t>(p.M / 32), jT = rT / 32;
        const size_t offT = p.mx_sf_mma
                                ? ((n / 128) * (kbT / 4) + jT / 4) * 512 + (n % 32) * 16 + ((n / 32) % 4) * 4 + jT % 4
                                : n * kbT + jT;
        p.csT[offT] = static_cast<uint8_t>(sT);
      }
    }
    if (rows_out) store_row_scales<BN>(p, rg, n0, sc);
    return;
  }
  if constexpr (ORI == 1) {
    // row blocks only: each 32-column chunk of a row is one MX block, formed
    // and stored chunk by chunk; the accumulator is released at the end
    uint32_t sc[BN / 128];
    const size_t rg = static_cast<size_t>(m0 + row);
#pragma unroll
    for (int g = 0; g < BN / 128; ++g) sc[g] = 0;
#pragma unroll
    for (int c = 0; c < BN / 32; c += 2) {
      uint32_t v[2][32];
      tmem_ld32(lane_addr + c * 32, v[0]);
      tmem_ld32(lane_addr + (c + 1) * 32, v[1]);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t s8 =
            mx_block_store<FP4O>(v[h], p, p.cq + ((rg * static_cast<size_t>(p.N) + n0 + (c + h) * 32) >> CSH));
        sc[(c + h) >> 2] |= s8 << (8 * ((c + h) & 3));
      }
    }
    tc_fence_before();
    __syncwarp();
    release();
    store_row_scales<BN>(p, rg, n0, sc);
    return;
  }
  if constexpr (ORI == 2) {
    // row blocks: each 32-column chunk of a row is one MX block, formed
    // from the registers and stored at once (only the scale words are kept
    // to the end).  Column blocks: a warp's 32 rows of a chunk are 32 blocks
    // of 32 x 1; the warp transposes the chunk through its part of the (here
    // unused) staging area, rows XS_PITCH words apart so that neither the
    // 16-byte row writes nor the column reads conflict, and lane j quantizes
    // column j.
    uint32_t sc[BN / 128];
    uint32_t* xs = reinterpret_cast<uint32_t*>(sOut) + q * XS_WORDS;    // this warp's transpose scratch
    const size_t rg = static_cast<size_t>(m0 + row);
    const size_t rT = static_cast<size_t>(m0 + q * 32);          // first row of the warp's column blocks
#pragma unroll
    for (int g = 0; g < BN / 128; ++g) sc[g] = 0;
#pragma unroll
    for (int c = 0; c < BN / 32; c += 2) {
      uint32_t v[2][32];
      tmem_ld32(lane_addr + c * 32, v[0]);
      tmem_ld32(lane_addr + (c + 1) * 32, v[1]);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (p.cq) {
          const uint32_t s8 =
              mx_block_store<FP4O>(v[h], p, p.cq + ((rg * static_cast<size_t>(p.N) + n0 + (c + h) * 32) >> CSH));
          sc[(c + h) >> 2] |= s8 << (8 * ((c + h) & 3));
        }
        if (p.cqT) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(xs + lane * XS_PITCH + 4 * j) =
                make_uint4(v[h][4 * j], v[h][4 * j + 1], v[h][4 * j + 2], v[h][4 * j + 3]);
          __syncwarp();
          uint32_t col[32];
          load_col32(xs, lane, col);
          __syncwarp();
          const size_t n = static_cast<size_t>(n0 + (c + h) * 32 + lane);
          const uint32_t sT =
              mx_block_store<FP4O>(col, p, p.cqT + ((n * static_cast<size_t>(p.M) + rT) >> CSH));
          const size_t kbT = static_cast<size_t>(p.M / 32), jT = rT / 32;
          const size_t offT = p.mx_sf_mma
                                  ? ((n / 128) * (kbT / 4) + jT / 4) * 512 + (n % 32) * 16 + ((n / 32) % 4) * 4 + jT % 4
                                  : n * kbT + jT;
          p.csT[offT] = static_cast<uint8_t>(sT);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    release();
    if (p.cq) store_row_scales<BN>(p, rg, n0, sc);
    return;
  }
  // float32 output: chunk by chunk
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t v[32];
    tmem_ld32(lane_addr + c0, v);
    tmem_ld_wait();
    if (c0 + 32 == BN) {                                         // accumulator fully read
      tc_fence_before();
      __syncwarp();
      release();
    }
    for (int h = 0; h < 2; ++h) {
      if (leader) bulk_wait_read_staging<NBUF>();
      named_bar(1, 128);
      uint8_t* stg = sOut + buf * STG_BYTES;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int phys = j ^ ((row >> 1) & 3);                   // 64-byte swizzle
        *reinterpret_cast<uint4*>(stg + row * 64 + phys * 16) =
            make_uint4(v[h * 16 + 4 * j], v[h * 16 + 4 * j + 1], v[h * 16 + 4 * j + 2], v[h * 16 + 4 * j + 3]);
      }
      fence_proxy_async_smem();
      named_bar(1, 128);
      if (leader) {
        tma_store_2d(map_c, smem_u32(stg), n0 + c0 + h * 16, m0);
        bulk_commit();
      }
      buf ^= NBUF - 1;
    }
  }
}

// Stream-K: the second of a cut tile's two pieces to finish writes the tile
// (bf16 or float32) from RN32(acc + other), `other` the float32 sums the
// first parked, column-major (column j of this CTA's 128 rows at
// other[j * 128 + row]).  Chunk by chunk (32 columns), through the same
// staging buffers and TMA stores as store_tile; the accumulator is released
// once its last chunk is read.
template <int BN, typename Release>
__device__ __forceinline__ void store_tile_added(const Params& p, uint32_t tmem, int q, int lane, bool leader, int& buf,
                                                 uint8_t* sOut, const CUtensorMap* map_c, int m0, int n0,
                                                 Release release, const float* other) {
  const int row = q * 32 + lane;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
  // the other piece's sums arrive 64 columns at a time, the next batch's
  // loads in flight while the current one is added and stored
  float nxt[64];
#pragma unroll
  for (int j = 0; j < 64; ++j) nxt[j] = __ldcg(other + j * 128 + row);
#pragma unroll
  for (int cb = 0; cb < BN; cb += 64) {
    float cur[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) cur[j] = nxt[j];
    if (cb + 64 < BN) {
#pragma unroll
      for (int j = 0; j < 64; ++j) nxt[j] = __ldcg(other + (cb + 64 + j) * 128 + row);
    }
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      const int c0 = cb + 32 * hc;
      uint32_t v[32];
      tmem_ld32(lane_addr + c0, v);
      tmem_ld_wait();
      if (c0 + 32 == BN) {
        tc_fence_before();
        __syncwarp();
        release();
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__fadd_rn(__uint_as_float(v[j]), cur[32 * hc + j]));
      const int nbox = p.epi == EPI_BF16 ? 1 : 2;          // staging boxes of 64 bytes per row
      for (int h = 0; h < nbox; ++h) {
        if (leader) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        named_bar(1, 128);
        uint8_t* stg = sOut + buf * STG_BYTES;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int phys = j ^ ((row >> 1) & 3);                   // 64-byte swizzle
          uint4 w;
          if (p.epi == EPI_BF16) {
            uint32_t b[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[8 * j + 2 * k]),
                                                              __uint_as_float(v[8 * j + 2 * k + 1]));
              b[k] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            w = make_uint4(b[0], b[1], b[2], b[3]);
          } else {
            w = make_uint4(v[h * 16 + 4 * j], v[h * 16 + 4 * j + 1], v[h * 16 + 4 * j + 2], v[h * 16 + 4 * j + 3]);
          }
          *reinterpret_cast<uint4*>(stg + row * 64 + phys * 16) = w;
        }
        fence_proxy_async_smem();
        named_bar(1, 128);
        if (leader) {
          tma_store_2d(map_c, smem_u32(stg), p.epi == EPI_BF16 ? n0 + c0 : n0 + c0 + h * 16, m0);
          bulk_commit();
        }
        buf ^= 1;
      }
    }
  }
}

// Stream-K: the first of a cut tile's two pieces to finish parks this
// CTA's float32 sums (128 rows x BN columns) in its workspace slot, column
// by column (a warp's 32 rows make one 128-byte store), then releases the
// accumulator.
template <int BN, typename Release>
__device__ __forceinline__ void park_partial(uint32_t tmem, int q, int lane, float* part, Release release) {
  const int row = q * 32 + lane;
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
  for (int c = 0; c < BN / 32; c += 2) {
    uint32_t v[2][32];
    tmem_ld32(lane_addr + c * 32, v[0]);
    tmem_ld32(lane_addr + (c + 1) * 32, v[1]);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int j = 0; j < 32; ++j) __stcg(part + ((c + h) * 32 + j) * 128 + row, __uint_as_float(v[h][j]));
  }
  tc_fence_before();
  __syncwarp();
  release();
}

template <int KIND_, int BN>
struct Cfg {
  static constexpr int KIND = KIND_;
  static constexpr bool FP4 = KIND == KIND_MXF4;
  static constexpr bool SCALED = KIND != KIND_F8;
  static constexpr int A_BYTES = BM * BKB;
  static constexpr int B_BYTES = BN * BKB;
  static constexpr int SF_CHUNKS = SCALED ? (FP4 ? 2 : 1) : 0;   // 512-B chunks per 128 rows per stage
  static constexpr int SFA_BYTES = 512 * SF_CHUNKS;
  static constexpr int SFB_BYTES = 512 * SF_CHUNKS * (BN / 128);
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // tensor memory: accumulator BN columns, then per stage the scale chunks:
  // A (4 columns per chunk), then B (per chunk, BN / 32 consecutive columns:
  // column j holds rows 32 j .. 32 j + 31 of the tile)
  static constexpr int SFA_COLS = 4 * SF_CHUNKS;
  static constexpr int SFB_COLS = 4 * SF_CHUNKS * (BN / 128);
  static constexpr int SF_COLS_STAGE = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(BN + STAGES * SF_COLS_STAGE <= TMEM_COLS, "tensor memory budget");
  static constexpr int SMEM = STAGES * (STAGE_BYTES + SFA_BYTES + SFB_BYTES) + OUT_BYTES + 256 + 1024;
};

template <int KIND, int BN, int MXOUT>
__global__ void __launch_bounds__(THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_c, const Params p) {
  using C = Cfg<KIND, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                          // STAGES x A_BYTES
  uint8_t* sB = sA + STAGES * C::A_BYTES;                      // STAGES x B_BYTES
  uint8_t* sSFA = sB + STAGES * C::B_BYTES;                    // STAGES x SFA_BYTES
  uint8_t* sSFB = sSFA + STAGES * C::SFA_BYTES;                // STAGES x SFB_BYTES
  uint8_t* sOut = sSFB + STAGES * C::SFB_BYTES;                // OUT_BYTES (1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + OUT_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_full + 2;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(acc_full + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_full + 3) + 1;
  volatile int* epi_fail = reinterpret_cast<volatile int*>(acc_full + 3) + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), 4);      // one arrive per epilogue warp
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *epi_fail = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
    if (p.epi != EPI_MX) prefetch_tensormap(&map_c);
  }
  if (warp == 1) tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_launch();
  grid_dep_wait();                 // before any global-memory access
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_sf = tmem + BN;                          // column offset of the scale area

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int u = 0;                                               // stage use counter
      for (int tile = blockIdx.x; tile < p.ntiles && !*abort_flag; tile += gridDim.x) {
        const TilePos tp = tile_pos(p, tile, BM, BN);
        const int ar = tp.b * (p.a_batched ? p.M : 0) + tp.m0;   // operand rows (K-major)
        const int br = tp.b * (p.b_batched ? p.N : 0) + tp.n0;
        const int ak = tp.b * (p.a_batched ? p.K : 0);           // first K row (MN-major)
        const int bk = tp.b * (p.b_batched ? p.K : 0);
        for (int kb = 0; kb < p.kblocks; ++kb, ++u) {
          const int s = u % STAGES;
          if (!mbar_wait(smem_u32(&empty[s]), ((u / STAGES) & 1) ^ 1, p.status)) { *abort_flag = 1; break; }
          if (blockIdx.x == 0 && u == p.stall_u) continue;   // test hook: phase never completes
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, p.tx_bytes);
          if (p.a_mn) tma_load_2d(smem_u32(sA + s * C::A_BYTES), &map_a, fb, tp.m0, ak + kb * BKB);
          else tma_load_2d(smem_u32(sA + s * C::A_BYTES), &map_a, fb, kb * BKB, ar);
          if (p.b_mn) tma_load_2d(smem_u32(sB + s * C::B_BYTES), &map_b, fb, tp.n0, bk + kb * BKB);
          else tma_load_2d(smem_u32(sB + s * C::B_BYTES), &map_b, fb, kb * BKB, br);
          if constexpr (C::SCALED) {
            const uint8_t* sfa_src = p.a_s + (static_cast<size_t>(tp.m0 / 128) * p.kb4) * 512;
            bulk_load_1d(smem_u32(sSFA + s * C::SFA_BYTES), sfa_src + kb * C::SFA_BYTES, C::SFA_BYTES, fb);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h) {
              const uint8_t* src = p.b_s + (static_cast<size_t>(tp.n0 / 128 + h) * p.kb4) * 512 + kb * C::SFA_BYTES;
              bulk_load_1d(smem_u32(sSFB + s * C::SFB_BYTES + h * C::SFA_BYTES), src, C::SFA_BYTES, fb);
            }
          }
        }
      }
      // make sure no copy is still landing in shared memory when the CTA ends
      for (int s = 0; s < STAGES && u > 0; ++s) {
        int last = u - 1 - ((u - 1 - s) % STAGES + STAGES) % STAGES;   // most recent use of stage s
        if (last >= 0 && last % STAGES == s) (void)mbar_wait(smem_u32(&full[s]), (last / STAGES) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptors of stage 0, k-slice 0; every other (stage, slice) is a
      // plain add on the 14-bit start-address field (addresses stay < 256 KB).
      const uint64_t a_desc0 = operand_desc(smem_u32(sA), p.a_mn);
      const uint64_t b_desc0 = operand_desc(smem_u32(sB), p.b_mn);
      const uint32_t a_step = k_slice_step(p.a_mn), b_step = k_slice_step(p.b_mn);
      const uint64_t sfa_desc0 = smem_desc(smem_u32(sSFA), 0, 128, 0);
      const uint64_t sfb_desc0 = smem_desc(smem_u32(sSFB), 0, 128, 0);
      uint32_t idesc[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) idesc[kk] = mma_idesc<KIND>(p, BN, BM, kk);
      int u = 0, t = 0;
      for (int tile = blockIdx.x; tile < p.ntiles && !*abort_flag; tile += gridDim.x, ++t) {
        if (!mbar_wait(smem_u32(acc_empty), (t & 1) ^ 1, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < p.kblocks; ++kb, ++u) {
          const int s = u % STAGES;
          if (!mbar_wait(smem_u32(&full[s]), (u / STAGES) & 1, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sfa_t = tmem_sf + s * C::SF_COLS_STAGE;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
          if constexpr (C::SCALED) {
            // scale chunks -> tensor memory (each 512-B chunk: 32 lanes x 16 B, x4 lane groups)
#pragma unroll
            for (int c = 0; c < C::SF_CHUNKS; ++c)
              tc_cp_sf(sfa_t + 4 * c, sfa_desc0 + ((s * C::SFA_BYTES + c * 512) >> 4));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
#pragma unroll
              for (int c = 0; c < C::SF_CHUNKS; ++c)
                tc_cp_sf(sfb_t + 4 * (BN / 128) * c + 4 * h,
                         sfb_desc0 + ((s * C::SFB_BYTES + h * C::SFA_BYTES + c * 512) >> 4));
          }
          const uint64_t ad = a_desc0 + ((s * C::A_BYTES) >> 4);
          const uint64_t bd = b_desc0 + ((s * C::B_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // 32 bytes of K per MMA (32 FP8 or 64 FP4 elements).  E2M1: K = 64
            // consumes two scales per row, chunk kk / 2, byte pair (kk % 2) * 2;
            // the BN rows of B's chunk sit in BN / 32 consecutive columns.
            const uint32_t sfa = C::FP4 ? sfa_t + 4 * (kk >> 1) : sfa_t;
            const uint32_t sfb = C::FP4 ? sfb_t + 4 * (BN / 128) * (kk >> 1) : sfb_t;
            tc_mma<KIND>(tmem, ad + a_step * kk, bd + b_step * kk, idesc[kk], sfa, sfb, (kb | kk) != 0);
          }
          tc_commit(smem_u32(&empty[s]));                       // stage free when these MMAs finish
        }
        if (!ok) { *abort_flag = 1; break; }
        tc_commit(smem_u32(acc_full));                          // accumulator ready
      }
      tc_commit(smem_u32(drain));
      (void)mbar_wait(smem_u32(drain), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                                      // tensor-memory lane quarter
    const bool leader = (warp == EPI_WARP0 && lane == 0);
    const float alpha = (C::KIND == KIND_F8 && p.alpha) ? *p.alpha : 1.0f;
    int t = 0, buf = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++t) {
      const TilePos tp = tile_pos(p, tile, BM, BN);
      // the four warps decide together, so none is left alone at a named barrier
      if (!mbar_wait(smem_u32(acc_full), t & 1, p.status)) *epi_fail = 1;
      named_bar(1, 128);
      if (*epi_fail) { *abort_flag = 1; break; }
      tc_fence_after();
      store_tile<BN, C::KIND == KIND_F8, MXOUT, 2>(p, alpha, tmem, q, lane, leader, buf, sOut, &map_c, tp.b * p.M + tp.m0,
                                         tp.n0, [&] {
                                           if (lane == 0) mbar_arrive(smem_u32(acc_empty));
                                         });
    }
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- CTA pair
// 256 x 256 output tiles per cluster of two CTAs.  CTA rank r of the pair
// holds rows m0 + 128 r .. of A, rows n0 + 128 r .. of B, A's scale chunks of
// its own rows and B's of all 256 rows.  The pair's first CTA (rank 0) owns
// the stage ring's "full" barriers (both CTAs' loads complete on them), the
// accumulator-empty barrier (all epilogue warps of both CTAs arrive) and
// issues the tensor-core work (scale copies from warp 6, MMAs from warp 1);
// its MMA commits arrive on the "empty" and accumulator-full barriers of
// both CTAs.
//
// The MX outputs quantize in the epilogue, which then does far more
// arithmetic per accumulator value; with one epilogue warp per SM
// sub-partition that work is latency-bound, so these variants run two groups
// of four epilogue warps (warps 2-5 and 7-10), each draining 128 of the 256
// accumulator columns.
template <int KIND_, int MXOUT_ = 0, bool SK_ = false>
struct PairCfg {
  static constexpr int KIND = KIND_;
  static constexpr bool FP4 = KIND == KIND_MXF4;
  static constexpr bool SCALED = KIND != KIND_F8;
  static constexpr int BN = 256;                        // columns per tile (both CTAs)
  static constexpr int EPI_GROUPS = MXOUT_ ? 2 : 1;
  static constexpr int EPI_COLS = BN / EPI_GROUPS;      // accumulator columns per epilogue group
  static constexpr int THREADS = PAIR_THREADS + (EPI_GROUPS - 1) * 128;
  // the column-block output transposes through 32 x 33 words per epilogue warp
  static constexpr bool MX_COLS = MXOUT_ == 2 || MXOUT_ == 4;     // MX column blocks too
  // MXFP4 with bf16 / float32 output: one staging buffer (the epilogue runs
  // after the accumulator is released, off the MMAs' path), which leaves
  // room for a sixth stage
  static constexpr bool ONE_STG = FP4 && MXOUT_ == 0 && !SK_;
  static constexpr int NBUF = ONE_STG ? 1 : 2;
  // MX row blocks alone are stored straight from registers: no staging
  static constexpr bool MX_ROWS_ONLY = MXOUT_ == 1 || MXOUT_ == 3;
  static constexpr int OUT =
      MX_COLS ? EPI_GROUPS * XS_GROUP_BYTES : (MX_ROWS_ONLY ? 0 : (ONE_STG ? STG_BYTES + 512 : OUT_BYTES));
  static constexpr int STAGES = (ONE_STG || (FP4 && MX_ROWS_ONLY)) ? 6 : ((FP4 || MX_COLS) ? 5 : 6);
  static constexpr int A_BYTES = BM * BKB;              // this CTA's 128 rows of A
  static constexpr int B_BYTES = (BN / 2) * BKB;        // this CTA's 128 rows of B
  static constexpr int SF_CHUNKS = SCALED ? (FP4 ? 2 : 1) : 0;   // 512-B chunks per 128 rows per stage
  static constexpr int SFA_BYTES = 512 * SF_CHUNKS;
  static constexpr int SFB_BYTES = 2 * SFA_BYTES;       // both 128-row halves of B
  static constexpr int TX_CTA = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;   // shared memory per stage
  static constexpr int SFA_COLS = 4 * SF_CHUNKS;
  static constexpr int SFB_COLS = 8 * SF_CHUNKS;
  static constexpr int SF_COLS_STAGE = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_COLS = 512;
  // without block scales two accumulators fit: the epilogue drains one
  // while the MMAs fill the other
  static constexpr int NACC = SCALED ? 1 : 2;
  static_assert(NACC * BN + STAGES * SF_COLS_STAGE <= TMEM_COLS, "tensor memory budget");
  static constexpr int SMEM = STAGES * TX_CTA + OUT + 256 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int KIND, int MXOUT, bool SK = false>
__global__ void __launch_bounds__(PairCfg<KIND, MXOUT, SK>::THREADS, 1)
mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_sfa, const __grid_constant__ CUtensorMap map_sfb,
                    const __grid_constant__ CUtensorMap map_c, const Params p) {
  using C = PairCfg<KIND, MXOUT, SK>;
  constexpr int STAGES_P = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                          // STAGES x A_BYTES
  uint8_t* sB = sA + STAGES_P * C::A_BYTES;                    // STAGES x B_BYTES
  uint8_t* sSFA = sB + STAGES_P * C::B_BYTES;                  // STAGES x SFA_BYTES
  uint8_t* sSFB = sSFA + STAGES_P * C::SFA_BYTES;              // STAGES x SFB_BYTES
  uint8_t* sOut = sSFB + STAGES_P * C::SFB_BYTES;              // C::OUT bytes (1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + C::OUT);
  uint64_t* full = bars;                                       // used in rank 0
  uint64_t* empty = bars + STAGES_P;
  uint64_t* acc_full = bars + 2 * STAGES_P;
  uint64_t* acc_empty = acc_full + 1;                          // used in rank 0
  uint64_t* drain = acc_full + 2;                              // used in rank 0
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(acc_full + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(acc_full + 3) + 1;
  volatile int* epi_fail = reinterpret_cast<volatile int*>(acc_full + 3) + 2;
  volatile int* sk_first = reinterpret_cast<volatile int*>(acc_full + 3) + 3;   // stream-K ticket outcome
  uint64_t* sf_full = acc_full + 5;                            // rank 0: a slot's scales are in tensor memory
  uint64_t* sf_drain = sf_full + STAGES_P;                     // rank 0
  // accumulator buffer b: full / empty barriers (the second pair exists when NACC == 2)
  uint64_t* const acc_full1 = sf_drain + 1;
  uint64_t* const acc_empty1 = sf_drain + 2;                   // used in rank 0
  auto accf = [&](int b) { return b ? acc_full1 : acc_full; };
  auto acce = [&](int b) { return b ? acc_empty1 : acc_empty; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES_P; ++s) {
      mbar_init(smem_u32(&full[s]), 1);                        // rank 0's producer arrives (with both CTAs' bytes)
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    mbar_init(smem_u32(acc_empty), 8 * C::EPI_GROUPS);         // the epilogue warps of both CTAs
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < STAGES_P; ++s) mbar_init(smem_u32(&sf_full[s]), 1);
    mbar_init(smem_u32(sf_drain), 1);
    mbar_init(smem_u32(acc_full1), 1);
    mbar_init(smem_u32(acc_empty1), 8 * C::EPI_GROUPS);
    *abort_flag = 0;
    *epi_fail = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
    if (C::SCALED) {
      prefetch_tensormap(&map_sfa);
      prefetch_tensormap(&map_sfb);
    }
    if (p.epi != EPI_MX) prefetch_tensormap(&map_c);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
  tc_fence_before();
  cluster_sync();                  // barriers of both CTAs initialised, tensor memory allocated in both
  tc_fence_after();
  grid_dep_launch();
  grid_dep_wait();                 // before any global-memory access
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_sf = tmem + C::BN;                       // column offset of the scale area

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int u = 0;                                               // stage use counter
      SegIter<SK> segs(p, pair, npairs);
      Seg sg;
      while (!*abort_flag && segs.next(sg)) {
        const TilePos tp = tile_pos(p, sg.tile, 256, 256);
        const int m0 = tp.m0 + static_cast<int>(rank) * BM;   // this CTA's rows of the product
        const int ar = tp.b * (p.a_batched ? p.M : 0) + m0;
        const int n0r = tp.n0 + static_cast<int>(rank) * 128;  // this CTA's half of B
        const int br = tp.b * (p.b_batched ? p.N : 0) + n0r;
        const int ak = tp.b * (p.a_batched ? p.K : 0);           // first K row (MN-major operands)
        const int bk = tp.b * (p.b_batched ? p.K : 0);
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++u) {
          const int s = u % STAGES_P;
          if (!mbar_wait_suspend(smem_u32(&empty[s]), ((u / STAGES_P) & 1) ^ 1, p.status)) { *abort_flag = 1; break; }
          if (rank == 0 && blockIdx.x == 0 && u == p.stall_u) continue;   // test hook: phase never completes
          const uint32_t fb = cluster_map(smem_u32(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full[s]), p.tx_bytes);
          if (p.a_mn) tma_load_2d_pair(smem_u32(sA + s * C::A_BYTES), &map_a, fb, m0, ak + kb * BKB);
          else tma_load_2d_pair(smem_u32(sA + s * C::A_BYTES), &map_a, fb, kb * BKB, ar);
          if (p.b_mn) tma_load_2d_pair(smem_u32(sB + s * C::B_BYTES), &map_b, fb, n0r, bk + kb * BKB);
          else tma_load_2d_pair(smem_u32(sB + s * C::B_BYTES), &map_b, fb, kb * BKB, br);
          if constexpr (C::SCALED) {
            // scale maps: one 512-B chunk per row, chunk (rb, kc) at row rb * kb4 + kc
            tma_load_2d_pair(smem_u32(sSFA + s * C::SFA_BYTES), &map_sfa, fb, 0, (m0 / 128) * p.kb4 + kb * C::SF_CHUNKS);
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_2d_pair(smem_u32(sSFB + s * C::SFB_BYTES + h * C::SFA_BYTES), &map_sfb, fb, 0,
                               (tp.n0 / 128 + h) * p.kb4 + kb * C::SF_CHUNKS);
          }
        }
      }
      // rank 0: make sure no copy of either CTA is still landing when the pair ends
      // (rank 1 is held at the final cluster barrier until this has finished)
      if (rank == 0) {
        for (int s = 0; s < STAGES_P && u > 0; ++s) {
          int last = u - 1 - ((u - 1 - s) % STAGES_P + STAGES_P) % STAGES_P;
          if (last >= 0 && last % STAGES_P == s) (void)mbar_wait_suspend(smem_u32(&full[s]), (last / STAGES_P) & 1, p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    // The tensor pipe takes only a few instructions ahead, so every cycle
    // this thread spends elsewhere can idle it: it waits for a slot's scales
    // (copied by warp 6, which runs ahead) -- or, unscaled, for the slot's
    // operands -- and issues the four MMAs only.
    if (lane == 0 && rank == 0) {
      const uint64_t a_desc0 = operand_desc(smem_u32(sA), p.a_mn);
      const uint64_t b_desc0 = operand_desc(smem_u32(sB), p.b_mn);
      const uint32_t a_step = k_slice_step(p.a_mn), b_step = k_slice_step(p.b_mn);
      uint32_t idesc[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) idesc[kk] = mma_idesc<KIND>(p, C::BN, 2 * BM, kk);
      uint64_t* ready = C::SCALED ? sf_full : full;
      bool ok = true;
      int s = 0, ph = 0;
      SegIter<SK> segs(p, pair, npairs);
      Seg sg;
      for (int t = 0; ok && !*abort_flag && segs.next(sg); ++t) {
        const int ab = C::NACC == 2 ? (t & 1) : 0;            // accumulator buffer and its use parity
        const uint32_t aph = C::NACC == 2 ? ((t >> 1) & 1) : (t & 1);
        const uint32_t dacc = tmem + ab * C::BN;
        if (!mbar_wait_suspend(smem_u32(acce(ab)), aph ^ 1, p.status)) { ok = false; break; }
        tc_fence_after();
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait_suspend(smem_u32(&ready[s]), ph, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sfa_t = tmem_sf + s * C::SF_COLS_STAGE;
          const uint32_t sfb_t = sfa_t + C::SFA_COLS;
          const uint64_t ad = a_desc0 + ((s * C::A_BYTES) >> 4);
          const uint64_t bd = b_desc0 + ((s * C::B_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t sfa = C::FP4 ? sfa_t + 4 * (kk >> 1) : sfa_t;
            const uint32_t sfb = C::FP4 ? sfb_t + 8 * (kk >> 1) : sfb_t;
            tc_mma_pair<KIND>(dacc, ad + a_step * kk, bd + b_step * kk, idesc[kk], sfa, sfb,
                              (kb != sg.kb0) || (kk != 0));
          }
          tc_commit_pair_both(smem_u32(&empty[s]));            // stage free in both CTAs
          if (++s == STAGES_P) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair_both(smem_u32(accf(ab)));                // both halves of the accumulator ready
      }
      if (!ok) *abort_flag = 1;
      tc_commit_pair_self(smem_u32(drain));
      (void)mbar_wait_suspend(smem_u32(drain), 0, p.status);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ scale copies (rank 0)
    // Per stage: A's chunks and both halves of B's into the slot's own
    // tensor-memory columns (one tcgen05.cp.cta_group::2 fills both CTAs),
    // then a commit that tells the MMA issuer they have landed.  A slot is
    // rewritten only after its stage was refilled, i.e. after the MMAs that
    // read its previous scales completed.
    if (C::SCALED && lane == 0 && rank == 0) {
      const uint64_t sfa_desc0 = smem_desc(smem_u32(sSFA), 0, 128, 0);
      const uint64_t sfb_desc0 = smem_desc(smem_u32(sSFB), 0, 128, 0);
      int total = 0;                                           // stage uses of this pair
      {
        SegIter<SK> segs(p, pair, npairs);
        Seg sg;
        while (segs.next(sg)) total += sg.kb1 - sg.kb0;
      }
      int s = 0, ph = 0;
      for (int u = 0; u < total && !*abort_flag; ++u) {
        if (!mbar_wait_suspend(smem_u32(&full[s]), ph, p.status)) { *abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t sfa_t = tmem_sf + s * C::SF_COLS_STAGE;
#pragma unroll
        for (int c = 0; c < C::SF_CHUNKS; ++c)
          tc_cp_sf_pair(sfa_t + 4 * c, sfa_desc0 + ((s * C::SFA_BYTES + c * 512) >> 4));
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int c = 0; c < C::SF_CHUNKS; ++c)
            tc_cp_sf_pair(sfa_t + C::SFA_COLS + 8 * c + 4 * hh,
                          sfb_desc0 + ((s * C::SFB_BYTES + hh * C::SFA_BYTES + c * 512) >> 4));
        tc_commit_pair_self(smem_u32(&sf_full[s]));
        if (++s == STAGES_P) { s = 0; ph ^= 1; }
      }
      tc_commit_pair_self(smem_u32(sf_drain));                // no copy in flight at exit
      (void)mbar_wait_suspend(smem_u32(sf_drain), 0, p.status);
    }
  } else if ((warp >= 2 && warp <= 5) || warp >= 7) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                                    // lane quarter of tensor memory
    const int grp = warp >= 7 ? 1 : 0;                         // accumulator columns grp * EPI_COLS ..
    const bool leader = (warp == EPI_WARP0 && lane == 0);
    const uint32_t acc_empty_r0 = cluster_map(smem_u32(acc_empty), 0);
    const uint32_t acc_empty1_r0 = cluster_map(smem_u32(acc_empty1), 0);
    const float alpha = (C::KIND == KIND_F8 && p.alpha) ? *p.alpha : 1.0f;
    int t = 0, buf = 0;
    SegIter<SK> segs(p, pair, npairs);
    Seg sg;
    for (; segs.next(sg); ++t) {
      const TilePos tp = tile_pos(p, sg.tile, 256, 256);
      const int m0 = tp.b * p.M + tp.m0 + static_cast<int>(rank) * BM;   // rows of the batched output
      const int ab = C::NACC == 2 ? (t & 1) : 0;
      const uint32_t aph = C::NACC == 2 ? ((t >> 1) & 1) : (t & 1);
      if (!mbar_wait_suspend(smem_u32(accf(ab)), aph, p.status)) *epi_fail = 1;
      named_bar(1, 128 * C::EPI_GROUPS);
      if (*epi_fail) { *abort_flag = 1; break; }
      tc_fence_after();
      auto release = [&] {
        if (lane == 0) {
          if (rank == 0) mbar_arrive(smem_u32(acce(ab)));
          else mbar_arrive_remote(ab ? acc_empty1_r0 : acc_empty_r0);
        }
      };
      if constexpr (SK) {
        if (sg.slot) {
          // A cut tile: the first of its two pieces to get here parks its
          // sums; the second adds them and writes the tile.  The ticket is a
          // swap of this launch's tag into the slot's word, so nothing needs
          // clearing between launches.
          uint32_t* flags = p.sk_flags + (static_cast<size_t>(sg.slot) * 2 + rank) * 2;
          float* part = p.sk_part + (static_cast<size_t>(sg.slot) * 2 + rank) * (C::BN * 128);
          if (leader) *sk_first = atomicExch(flags, p.sk_epoch) != p.sk_epoch;
          named_bar(1, 128);
          if (*sk_first) {
            park_partial<C::BN>(tmem, q, lane, part, release);
            __threadfence();
            named_bar(1, 128);
            if (leader) st_release_gpu(flags + 1, p.sk_epoch);
            continue;
          }
          // the first piece is running its epilogue: its sums land shortly
          if (leader) {
            const unsigned long long t0 = globaltimer_ns();
            while (ld_acquire_gpu(flags + 1) != p.sk_epoch) {
              if (globaltimer_ns() - t0 > kWaitLimitNs) { record_timeout(p.status); break; }
              __nanosleep(256);
            }
          }
          named_bar(1, 128);
          store_tile_added<C::BN>(p, tmem, q, lane, leader, buf, sOut, &map_c, m0, tp.n0, release, part);
          continue;
        }
      }
      store_tile<C::EPI_COLS, C::KIND == KIND_F8, MXOUT, C::NBUF>(
          p, alpha, tmem + ab * C::BN + grp * C::EPI_COLS, q, lane, leader, buf, sOut + grp * XS_GROUP_BYTES,
          &map_c, m0, tp.n0 + grp * C::EPI_COLS, release);
    }
    if (leader) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();                  // rank 0's tensor-core work on rank 1's memory has finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

}  // namespace gemm
}  // namespace mxq

// ==================================================================== host
using namespace mxq_host;

namespace {

using mxq::gemm::Params;

// One product as the entry points describe it.
struct GemmArgs {
  const void* a_q;
  const uint8_t* a_s;
  const void* b_q;
  const uint8_t* b_s;
  int64_t batch, M, N, K;
  int a_batched, b_batched;
  uint32_t a_type, b_type;
  int fp4;                        // both operands packed E2M1: kind::mxf4
  int a_mn, b_mn;                 // per-tensor kind: operand stored [K][M] / [K][N] (MN-major)
  int a_u4, b_u4;                 // packed E2M1 beside an 8-bit operand (see encode_operand)
  int epi;
  void* c;                        // EPI_BF16 / EPI_FP32 output [batch * M][N]
  const float* alpha;
  const void* bias;
  uint8_t* cq;
  uint8_t* cs;
  uint8_t* cqT;
  uint8_t* csT;
  int mx_fmt, mx_ceil, mx_sf_mma;
  void* ws;                       // stream-K workspace (or nullptr)
  size_t ws_bytes;
};

// Stream-K workspace: per range boundary (slot) and CTA half a ticket word
// and a ready word, then per slot and half 256 x 128 float32 partial sums.
// Slots 1 .. pairs - 1 are used; the layout reserves one per pair.
constexpr size_t kSkSlotFloats = 2 * 256 * 128;
// The stream-K schedule is used when the tile schedule's last wave keeps at
// most this share of the pairs busy.  Measured on GB300: a pair's tensor
// throughput drops when every pair runs (with 76 pairs busy, a pair takes
// about twice as long per k-block as with 4), so a partial last wave runs
// faster per pair and costs less than its share of a wave; only a sparse
// last wave pays for the cut tiles (80 tiles of 8192-deep MXFP8:
// 99.9 -> 73.7 us; 104 tiles: 100.5 -> 98.3 us).
constexpr double kSkMaxLastWave = 0.25;
size_t sk_flag_bytes(int pairs) { return (static_cast<size_t>(pairs) * 16 + 255) & ~size_t(255); }
size_t sk_workspace_bytes(int pairs) { return sk_flag_bytes(pairs) + static_cast<size_t>(pairs) * kSkSlotFloats * 4; }

// A fresh tag per launch on each device, never 0 (a zero-filled workspace
// holds no valid ticket).
uint32_t next_epoch() {
  static uint32_t epoch[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(mu);
  uint32_t& e = epoch[dev & 63];
  if (++e == 0) e = 1;
  return e;
}

Params make_params(const GemmArgs& g, int tm, int tn, int64_t kbytes) {
  Params p{};
  p.a_s = g.a_s;
  p.b_s = g.b_s;
  p.M = static_cast<int>(g.M);
  p.N = static_cast<int>(g.N);
  p.K = static_cast<int>(g.K);
  p.tiles_m = static_cast<int>(g.M / tm);
  p.tiles_n = static_cast<int>(g.N / tn);
  p.ntiles = static_cast<int>(g.batch) * p.tiles_m * p.tiles_n;
  p.kblocks = static_cast<int>(kbytes / mxq::gemm::BKB);
  p.kb4 = static_cast<int>(g.K / 128);
  p.a_batched = g.a_batched;
  p.b_batched = g.b_batched;
  p.epi = g.epi;
  p.alpha = g.alpha;
  p.bias = static_cast<const __nv_bfloat16*>(g.bias);
  p.cq = g.cq;
  p.cs = g.cs;
  p.cqT = g.cqT;
  p.csT = g.csT;
  p.mx_fmt = g.mx_fmt;
  p.mx_ceil = g.mx_ceil;
  p.mx_sf_mma = g.mx_sf_mma;
  p.status = status_ptr();
  p.a_type = g.a_type;
  p.b_type = g.b_type;
  p.a_mn = g.a_mn;
  p.b_mn = g.b_mn;
  // keep the operand with fewer rows (the smaller one) resident in L2
  p.m_fast = (g.a_batched == g.b_batched) && g.M < g.N;
  p.stall_u = take_test_stall(2) ? 0 : -1;
  return p;
}

// The output map: bf16 [rows][N] boxes of 32 columns, or float32 boxes of 16,
// both 128 rows with the 64-byte swizzle; the MX output needs none.
bool encode_c(CUtensorMap* mc, const GemmArgs& g) {
  *mc = CUtensorMap{};
  if (g.epi == mxq::gemm::EPI_MX) return true;
  const uint64_t rows = static_cast<uint64_t>(g.batch * g.M);
  if (g.epi == mxq::gemm::EPI_FP32)
    return encode_2d(mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, g.c, g.N, rows, g.N * 4, 16, mxq::gemm::BM,
                     CU_TENSOR_MAP_SWIZZLE_64B);
  return encode_2d(mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.c, g.N, rows, g.N * 2, 32, mxq::gemm::BM,
                   CU_TENSOR_MAP_SWIZZLE_64B);
}

// An operand's code map: 128-byte K steps of `box_rows` rows, 128-byte
// swizzle.  Codes are bytes (8-bit formats, or packed E2M1 for kind::mxf4,
// kbytes = K / 2).  Packed E2M1 beside an 8-bit operand (kind::mxf8f6f4)
// goes through the 16 x 4-bit type that widens every 8 packed bytes to a
// 16-byte slot: a K step is then 128 elements in the same 128 bytes of
// shared memory per row as an 8-bit operand, the layout the tensor core
// reads for 4-bit elements of that kind, and the map's x coordinate counts
// elements, so the kernels' coordinates (kb * 128) are unchanged.
bool encode_operand(CUtensorMap* m, const void* q, bool u4, int64_t K, int64_t kbytes, uint64_t rows,
                    uint32_t box_rows) {
  using namespace mxq::gemm;
  if (u4)
    return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, q, K, rows, K / 2, 128, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, kbytes, rows, kbytes, BKB, box_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// An MN-major FP8 operand's code map: the operand stored row-major as
// [K][MN] (one row per K index, batch entries stacked), boxes of 128 bytes
// along MN by 128 K rows, 128-byte swizzle -- the tile layout operand_desc
// describes for MN-major operands.
bool encode_operand_mn(CUtensorMap* m, const void* q, int64_t mn, uint64_t krows) {
  return encode_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, mn, krows, mn, 128, mxq::gemm::BKB,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

// Both operand maps of a product (box_b: rows of B per tile when K-major).
bool encode_operands(CUtensorMap* ma, CUtensorMap* mb, const GemmArgs& g, int64_t kbytes, uint32_t box_b) {
  using namespace mxq::gemm;
  const int64_t nba = g.a_batched ? g.batch : 1, nbb = g.b_batched ? g.batch : 1;
  const bool a_ok = g.a_mn ? encode_operand_mn(ma, g.a_q, g.M, static_cast<uint64_t>(nba * g.K))
                           : encode_operand(ma, g.a_q, g.a_u4, g.K, kbytes, static_cast<uint64_t>(nba * g.M), BM);
  const bool b_ok = g.b_mn ? encode_operand_mn(mb, g.b_q, g.N, static_cast<uint64_t>(nbb * g.K))
                           : encode_operand(mb, g.b_q, g.b_u4, g.K, kbytes, static_cast<uint64_t>(nbb * g.N), box_b);
  return a_ok && b_ok;
}

// Transaction bytes of one operand tile: the widened E2M1 load completes the
// packed bytes it reads (half its shared-memory footprint; the padding
// slots are not written).
constexpr uint32_t tx_bytes(int smem_bytes, bool u4) { return static_cast<uint32_t>(u4 ? smem_bytes / 2 : smem_bytes); }

template <int KIND, int BN, int MXOUT>
int launch(const GemmArgs& g, cudaStream_t st) {
  using namespace mxq::gemm;
  using Cf = Cfg<KIND, BN>;
  const int64_t kbytes = Cf::FP4 ? g.K / 2 : g.K;
  CUtensorMap ma, mb, mc;
  if (!encode_operands(&ma, &mb, g, kbytes, BN)) return MXQ_ERR_CUDA;
  if (!encode_c(&mc, g)) return MXQ_ERR_CUDA;
  Params p = make_params(g, BM, BN, kbytes);
  if (!p.status) return MXQ_ERR_CUDA;
  p.tx_bytes = tx_bytes(Cf::A_BYTES, g.a_u4) + tx_bytes(Cf::B_BYTES, g.b_u4) + Cf::SFA_BYTES + Cf::SFB_BYTES;
  auto kern = mx_gemm_kernel<KIND, BN, MXOUT>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM) != cudaSuccess)
      return MXQ_ERR_CUDA;
    attr_set[dev & 63] = true;
  }
  const int grid = std::min(p.ntiles, sm_count());
  return launch_pdl(kern, dim3(grid), dim3(THREADS), Cf::SMEM, st, ma, mb, mc, p);
}

// Co-resident clusters of two for the pair kernel (cached per device and
// kernel); 0 if the device cannot hold one.
template <int KIND, int MXOUT, bool SK>
int max_pairs(void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, mxq::gemm::Params),
              int smem, int threads) {
  static int cache[64] = {};
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (cache[dev & 63]) return cache[dev & 63] > 0 ? cache[dev & 63] : 0;
  if (!attr_set[dev & 63]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    attr_set[dev & 63] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (sm_count() / 2));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[dev & 63] = n > 0 ? n : -1;
  return n > 0 ? n : 0;
}

template <int KIND, int MXOUT>
int launch_pair(const GemmArgs& g, int pairs, cudaStream_t st) {
  using namespace mxq::gemm;
  using Cf = PairCfg<KIND, MXOUT>;
  const int64_t kbytes = Cf::FP4 ? g.K / 2 : g.K;
  const int64_t kb4 = g.K / 128;
  CUtensorMap ma, mb, msa, msb, mc;
  if (!encode_operands(&ma, &mb, g, kbytes, 128)) return MXQ_ERR_CUDA;
  msa = CUtensorMap{};
  msb = CUtensorMap{};
  if (Cf::SCALED) {
    // scales in the tensor-core layout: one 512-byte chunk (128 x 32-bit words) per row
    if (!encode_2d(&msa, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.a_s, 128, (g.M / 128) * kb4, 512, 128, Cf::SF_CHUNKS,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return MXQ_ERR_CUDA;
    if (!encode_2d(&msb, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.b_s, 128, (g.N / 128) * kb4, 512, 128, Cf::SF_CHUNKS,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
      return MXQ_ERR_CUDA;
  }
  if (!encode_c(&mc, g)) return MXQ_ERR_CUDA;
  Params p = make_params(g, 256, 256, kbytes);
  if (!p.status) return MXQ_ERR_CUDA;
  p.tx_bytes = 2 * (tx_bytes(Cf::A_BYTES, g.a_u4) + tx_bytes(Cf::B_BYTES, g.b_u4) + Cf::SFA_BYTES + Cf::SFB_BYTES);
  // Stream-K when a workspace is given and the tiles do not fill whole
  // waves: all but the last full wave run round-robin, the remaining
  // pairs..2*pairs-1 tiles' k-iterations are split evenly (every range at
  // least one tile long).
  if constexpr (MXOUT == 0 && Cf::NACC == 1) {
    const int last = p.ntiles % pairs;                     // tiles in the last, partial wave
    const bool worth = p.ntiles > pairs && last > 0 && last <= kSkMaxLastWave * pairs;
    if (g.ws && worth) {
      using Ck = PairCfg<KIND, MXOUT, true>;
      auto kern = mx_gemm_pair_kernel<KIND, MXOUT, true>;
      const int sk_pairs = max_pairs<KIND, MXOUT, true>(kern, Ck::SMEM, Ck::THREADS);
      if (sk_pairs == pairs && g.ws_bytes >= sk_workspace_bytes(pairs)) {
        p.sk = 1;
        p.sk_dp = (p.ntiles / pairs - 1) * pairs;
        p.sk_flags = static_cast<uint32_t*>(g.ws);
        p.sk_part = reinterpret_cast<float*>(static_cast<uint8_t*>(g.ws) + sk_flag_bytes(pairs));
        p.sk_epoch = next_epoch();
        return launch_pdl_cluster(kern, dim3(2 * pairs), dim3(Ck::THREADS), Ck::SMEM, st, 2, ma, mb, msa, msb, mc,
                                  p);
      }
    }
  }
  const int grid = 2 * std::min(p.ntiles, pairs);
  return launch_pdl_cluster(mx_gemm_pair_kernel<KIND, MXOUT>, dim3(grid), dim3(Cf::THREADS), Cf::SMEM, st, 2, ma, mb, msa,
                            msb, mc, p);
}

// The pair kernel for M and N multiples of 256 (when the device can hold it),
// else the single-CTA kernel.
template <int KIND, int MXOUT>
int dispatch_out(const GemmArgs& g, cudaStream_t st) {
  if (g.M % 256 == 0 && g.N % 256 == 0) {
    using Cf = mxq::gemm::PairCfg<KIND, MXOUT>;
    const int pairs = max_pairs<KIND, MXOUT, false>(mxq::gemm::mx_gemm_pair_kernel<KIND, MXOUT>, Cf::SMEM, Cf::THREADS);
    if (pairs > 0) return launch_pair<KIND, MXOUT>(g, pairs, st);
  }
  // an MN-major B tile is one 128-element swizzle atom wide
  return (g.N % 256 == 0 && !g.b_mn) ? launch<KIND, 256, MXOUT>(g, st) : launch<KIND, 128, MXOUT>(g, st);
}

// The MX outputs are separate kernels (row blocks only; with column
// blocks), so their epilogue registers do not weigh on the bf16 / float32
// kernel, nor the column pass on the row-only one.
template <int KIND>
int dispatch(const GemmArgs& g, cudaStream_t st) {
  if constexpr (KIND == mxq::gemm::KIND_F8) return dispatch_out<KIND, 0>(g, st);
  else {
    if (g.epi != mxq::gemm::EPI_MX) return dispatch_out<KIND, 0>(g, st);
    if (g.mx_fmt == MXQ_E2M1) return g.cqT ? dispatch_out<KIND, 4>(g, st) : dispatch_out<KIND, 3>(g, st);
    return g.cqT ? dispatch_out<KIND, 2>(g, st) : dispatch_out<KIND, 1>(g, st);
  }
}

// Element type code of the MMA's instruction descriptor: E4M3 0 and E5M2 1
// (kind::mxf8f6f4 / f8f6f4); E2M1 1 in kind::mxf4 and 5 in kind::mxf8f6f4.
uint32_t mma_type(int fmt, bool kind_mxf4) {
  if (fmt == MXQ_E2M1) return kind_mxf4 ? 1u : 5u;
  return fmt == MXQ_E4M3 ? 0u : 1u;
}

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

bool valid_fmt(int f) { return f == MXQ_E4M3 || f == MXQ_E5M2 || f == MXQ_E2M1; }

// Checks shared by the block-scaled entry points; fills g's operand fields.
int check_mx(GemmArgs& g, const void* a_q, const uint8_t* a_s, int a_fmt, const void* b_q, const uint8_t* b_s,
             int b_fmt, int64_t M, int64_t N, int64_t K, int sf_layout) {
  if (!a_q || !a_s || !b_q || !b_s) return MXQ_ERR_BAD_ARG;
  if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt)) return MXQ_ERR_BAD_ARG;
  if (sf_layout != MXQ_SF_MMA) return sf_layout == MXQ_SF_CANONICAL ? MXQ_ERR_UNSUPPORTED : MXQ_ERR_BAD_ARG;
  // Both E2M1: kind::mxf4 on packed operands.  One E2M1 beside an 8-bit
  // operand: kind::mxf8f6f4, the E2M1 codes widened on their way into
  // shared memory (encode_operand), which wants 32-byte aligned rows.
  const bool fp4 = a_fmt == MXQ_E2M1 && b_fmt == MXQ_E2M1;
  const bool a_u4 = a_fmt == MXQ_E2M1 && !fp4, b_u4 = b_fmt == MXQ_E2M1 && !fp4;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % (fp4 ? 256 : 128)) return MXQ_ERR_BAD_SHAPE;
  if (M > (1ll << 31) - 256 || N > (1ll << 31) - 256 || K > (1ll << 31) - 256) return MXQ_ERR_BAD_SHAPE;
  if (!aligned16(a_q) || !aligned16(b_q) || !aligned16(a_s) || !aligned16(b_s)) return MXQ_ERR_MISALIGNED;
  if ((a_u4 && !aligned32(a_q)) || (b_u4 && !aligned32(b_q))) return MXQ_ERR_MISALIGNED;
  g = GemmArgs{};
  g.a_q = a_q;
  g.a_s = a_s;
  g.b_q = b_q;
  g.b_s = b_s;
  g.batch = 1;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_type = mma_type(a_fmt, fp4);
  g.b_type = mma_type(b_fmt, fp4);
  g.fp4 = fp4;
  g.a_u4 = a_u4;
  g.b_u4 = b_u4;
  return MXQ_OK;
}

int run_mx(const GemmArgs& g, void* stream) {
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  auto st = static_cast<cudaStream_t>(stream);
  return g.fp4 ? dispatch<mxq::gemm::KIND_MXF4>(g, st) : dispatch<mxq::gemm::KIND_MXF8>(g, st);
}

int gemm_checked(const void* a_q, const uint8_t* a_s, int a_fmt, const void* b_q, const uint8_t* b_s, int b_fmt,
                 int64_t M, int64_t N, int64_t K, int sf_layout, void* c, int out_fp32, void* stream,
                 void* ws = nullptr, size_t ws_bytes = 0) {
  GemmArgs g;
  const int rc = check_mx(g, a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, sf_layout);
  if (rc != MXQ_OK) return rc;
  if (!c) return MXQ_ERR_BAD_ARG;
  if (!aligned16(c)) return MXQ_ERR_MISALIGNED;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return MXQ_ERR_MISALIGNED;
  g.c = c;
  g.epi = out_fp32 ? mxq::gemm::EPI_FP32 : mxq::gemm::EPI_BF16;
  g.ws = ws;
  g.ws_bytes = ws ? ws_bytes : 0;
  return run_mx(g, stream);
}

}  // namespace

extern "C" int mxq_gemm(const void* a_q, const uint8_t* a_s, const void* b_q, const uint8_t* b_s, int64_t M,
                        int64_t N, int64_t K, int fmt, int sf_layout, void* c, int out_fp32, void* stream) {
  return gemm_checked(a_q, a_s, fmt, b_q, b_s, fmt, M, N, K, sf_layout, c, out_fp32, stream);
}

extern "C" int mxq_gemm_mixed(const void* a_q, const uint8_t* a_s, int a_fmt, const void* b_q, const uint8_t* b_s,
                              int b_fmt, int64_t M, int64_t N, int64_t K, int sf_layout, void* c, int out_fp32,
                              void* stream) {
  return gemm_checked(a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, sf_layout, c, out_fp32, stream);
}

extern "C" int mxq_gemm_workspace_size(size_t* bytes) {
  if (!bytes) return MXQ_ERR_BAD_ARG;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  *bytes = sk_workspace_bytes(sm_count() / 2);
  return MXQ_OK;
}

extern "C" int mxq_gemm_ws(const void* a_q, const uint8_t* a_s, int a_fmt, const void* b_q, const uint8_t* b_s,
                           int b_fmt, int64_t M, int64_t N, int64_t K, int sf_layout, void* c, int out_fp32,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return gemm_checked(a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, sf_layout, c, out_fp32, stream, workspace,
                      workspace_bytes);
}

// ---------------------------------------------------------------- no-allocation variant
// Scratch of mxq_gemm_noalloc: the stream-K workspace of mxq_gemm_ws, held
// in the library itself for callers that cannot allocate device memory.
// Every device that loads the library holds this array until the process
// exits.  It covers up to 80 CTA pairs (160 SMs).
constexpr size_t kNoAllocScratchBytes = MXQ_GEMM_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes >= 80 * kSkSlotFloats * 4 + 80 * 16 + 256, "scratch covers 80 pairs");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, looked up once
// per device (in host code the array's name is not a device address).
int noalloc_scratch(void** out) {
  static void* ptr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MXQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MXQ_ERR_CUDA;
    ptr[dev] = p;
  }
  *out = ptr[dev];
  return MXQ_OK;
}

extern "C" int mxq_gemm_noalloc(const void* a_q, const uint8_t* a_s, int a_fmt, const void* b_q, const uint8_t* b_s,
                                int b_fmt, int64_t M, int64_t N, int64_t K, int sf_layout, void* c, int out_fp32,
                                void* stream) {
  GemmArgs g;
  const int rc = check_mx(g, a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, sf_layout);
  if (rc != MXQ_OK) return rc;
  if (!c) return MXQ_ERR_BAD_ARG;
  if (!aligned16(c)) return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  // the scratch this device's stream-K schedule can need, against the array
  if (sk_workspace_bytes(sm_count() / 2) > kNoAllocScratchBytes) return MXQ_ERR_UNSUPPORTED;
  void* ws = nullptr;
  const int src = noalloc_scratch(&ws);
  if (src != MXQ_OK) return src;
  return gemm_checked(a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, sf_layout, c, out_fp32, stream, ws,
                      kNoAllocScratchBytes);
}

extern "C" int mxq_gemm_mx_out(const void* a_q, const uint8_t* a_s, int a_fmt, const void* b_q, const uint8_t* b_s,
                               int b_fmt, int64_t M, int64_t N, int64_t K, int sf_layout, int out_fmt,
                               int out_scale_mode, int out_sf_layout, uint8_t* c_q, uint8_t* c_s, uint8_t* c_qT,
                               uint8_t* c_sT, void* stream) {
  GemmArgs g;
  const int rc = check_mx(g, a_q, a_s, a_fmt, b_q, b_s, b_fmt, M, N, K, sf_layout);
  if (rc != MXQ_OK) return rc;
  if (!c_q != !c_s || !c_qT != !c_sT || (!c_q && !c_qT)) return MXQ_ERR_BAD_ARG;
  if ((c_q && (!aligned16(c_q) || !aligned16(c_s))) || (c_qT && (!aligned16(c_qT) || !aligned16(c_sT))))
    return MXQ_ERR_MISALIGNED;
  if (out_fmt != MXQ_E4M3 && out_fmt != MXQ_E5M2 && out_fmt != MXQ_E2M1) return MXQ_ERR_BAD_ARG;
  if (out_scale_mode != MXQ_SCALE_FLOOR_OCP && out_scale_mode != MXQ_SCALE_CEIL) return MXQ_ERR_BAD_ARG;
  if (out_sf_layout != MXQ_SF_CANONICAL && out_sf_layout != MXQ_SF_MMA) return MXQ_ERR_BAD_ARG;
  g.epi = mxq::gemm::EPI_MX;
  g.cq = c_q;
  g.cs = c_s;
  g.cqT = c_qT;
  g.csT = c_sT;
  g.mx_fmt = out_fmt;
  g.mx_ceil = out_scale_mode == MXQ_SCALE_CEIL;
  g.mx_sf_mma = out_sf_layout == MXQ_SF_MMA;
  return run_mx(g, stream);
}

extern "C" int mxq_mm_fp8(const void* a, const void* b, int64_t batch, int64_t M, int64_t N, int64_t K,
                          int a_batched, int b_batched, int trans_a, int trans_b, int fmt, const float* scale,
                          const void* bias, void* c, void* stream) {
  if (!a || !b || !scale || !c) return MXQ_ERR_BAD_ARG;
  if (fmt != MXQ_E4M3 && fmt != MXQ_E5M2) return fmt == MXQ_E2M1 ? MXQ_ERR_UNSUPPORTED : MXQ_ERR_BAD_ARG;
  if ((a_batched != 0 && a_batched != 1) || (b_batched != 0 && b_batched != 1)) return MXQ_ERR_BAD_ARG;
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return MXQ_ERR_BAD_ARG;
  if (batch <= 0 || M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % 128) return MXQ_ERR_BAD_SHAPE;
  if (batch * M > (1ll << 31) - 256 || batch * N > (1ll << 31) - 256 || batch * K > (1ll << 31) - 256)
    return MXQ_ERR_BAD_SHAPE;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || (bias && !aligned16(bias)) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  GemmArgs g{};
  g.a_q = a;
  g.b_q = b;
  g.batch = batch;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_batched = batch > 1 ? a_batched : 0;
  g.b_batched = batch > 1 ? b_batched : 0;
  g.a_type = mma_type(fmt, false);
  g.b_type = mma_type(fmt, false);
  g.a_mn = trans_a;               // a stored [K][M]: op(a) = a^T is M-contiguous
  g.b_mn = !trans_b;              // b stored [K][N]: op(b) = b is N-contiguous
  g.epi = mxq::gemm::EPI_BF16;
  g.c = c;
  g.alpha = scale;
  g.bias = bias;
  return dispatch<mxq::gemm::KIND_F8>(g, static_cast<cudaStream_t>(stream));
}
