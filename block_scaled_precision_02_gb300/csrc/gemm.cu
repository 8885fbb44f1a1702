// Block-scaled (MX) GEMM on the sm_103a tensor cores:
//   C[m][n] = sum_k dec(a[m][k]) 2^(sa[m][k/32]-127) dec(b[n][k]) 2^(sb[n][k/32]-127)
// with float32 accumulation in tensor memory and a bf16 (or float32) output.
//
// Source: "UE8M0 FP8 / MXFP8 explainer", section 1 -- tensor cores consume the
// UE8M0 scale X and the element codes q_i of both operands, block by block,
// and accumulate in FP32; gap section 2 -- the blocks must run along the
// contiguous reduction dimension (both operands K-contiguous, C = A * B^T).
//
// Kernel structure (one CTA per SM, persistent over 128 x BN output tiles):
//  * warp 0      TMA producer: per K step (128 bytes of codes per row) one
//                128 x 128 B tile of A and one BN x 128 B tile of B with the
//                128-byte swizzle, plus the matching 512-byte scale chunks
//                (bulk copies; the quantizer already wrote them in the
//                tensor-core layout), into a 4-stage ring.
//  * warp 1      allocates tensor memory; one thread issues tcgen05.cp of the
//                scale chunks into tensor memory and 4 block-scaled
//                tcgen05.mma per stage (E4M3/E5M2: kind::mxf8f6f4,
//                scale_vec::1X, K = 32; E2M1: kind::mxf4, scale_vec::2X,
//                K = 64), then tcgen05.commit to free the stage.
//  * warps 2..5  epilogue: tcgen05.ld of the 128 x BN float32 accumulator
//                (each thread owns one row), conversion, and TMA stores
//                through two 64-byte-swizzled staging buffers.
// Every wait is bounded (1 s); on expiry the status word records
// MXQ_ERR_TIMEOUT, all roles wind down, in-flight copies are awaited (with a
// limit) and tensor memory is released.
#include <algorithm>

#include "common.cuh"

namespace mxq {
namespace gemm {

constexpr int BM = 128;
constexpr int BKB = 128;                 // bytes of codes per row per stage
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int STG_BYTES = BM * 64;       // one staging buffer: 128 rows x 64 B

struct Params {
  const uint8_t* a_s;
  const uint8_t* b_s;
  int M, N, K;
  int tiles_m, tiles_n, ntiles;
  int kblocks;        // K steps of BKB bytes
  int kb4;            // 512-byte scale chunks per 128 rows (K / 128)
  int out_fp32;
  int* status;
  int stall_u;        // failure-detection test hook: CTA 0 never fills this stage use (-1: off)
};

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

template <bool FP4>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
  if constexpr (FP4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
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

// Instruction descriptor of the block-scaled MMA: A/B element type codes at
// bits 7-9 / 10-12, K-major operands, N >> 3 at bits 17-22, scale type UE8M0
// (bit 23), M >> 4 at bits 24-28, scale-factor byte selectors for B (bits 4-5)
// and A (bits 29-30).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_type, int n, int m, uint32_t sf_id) {
  return (sf_id << 4) | (ab_type << 7) | (ab_type << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(m >> 4) << 24) | (sf_id << 29);
}

template <int FMT, int BN>
struct Cfg {
  static constexpr bool FP4 = FMT == MXQ_E2M1;
  static constexpr int A_BYTES = BM * BKB;
  static constexpr int B_BYTES = BN * BKB;
  static constexpr int SF_CHUNKS = FP4 ? 2 : 1;         // 512-B chunks per 128 rows per stage
  static constexpr int SFA_BYTES = 512 * SF_CHUNKS;
  static constexpr int SFB_BYTES = 512 * SF_CHUNKS * (BN / 128);
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TX_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // tensor memory: accumulator BN columns, then per stage the scale chunks:
  // A (4 columns per chunk), then B (per chunk, BN / 32 consecutive columns:
  // column j holds rows 32 j .. 32 j + 31 of the tile)
  static constexpr int SFA_COLS = 4 * SF_CHUNKS;
  static constexpr int SFB_COLS = 4 * SF_CHUNKS * (BN / 128);
  static constexpr int SF_COLS_STAGE = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_COLS = 512;
  static_assert(BN + STAGES * SF_COLS_STAGE <= TMEM_COLS, "tensor memory budget");
  static constexpr uint32_t AB_TYPE = FMT == MXQ_E4M3 ? 0u : (FMT == MXQ_E5M2 ? 1u : 1u);  // E2M1 in kind::mxf4 is 1
  static constexpr int SMEM = STAGES * (STAGE_BYTES + SFA_BYTES + SFB_BYTES) + 2 * STG_BYTES + 256 + 1024;
};

template <int FMT, int BN>
__global__ void __launch_bounds__(THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_c, const Params p) {
  using C = Cfg<FMT, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                                          // STAGES x A_BYTES
  uint8_t* sB = sA + STAGES * C::A_BYTES;                      // STAGES x B_BYTES
  uint8_t* sSFA = sB + STAGES * C::B_BYTES;                    // STAGES x SFA_BYTES
  uint8_t* sSFB = sSFA + STAGES * C::SFA_BYTES;                // STAGES x SFB_BYTES
  uint8_t* sOut = sSFB + STAGES * C::SFB_BYTES;                // 2 x STG_BYTES (1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + 2 * STG_BYTES);
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
    prefetch_tensormap(&map_c);
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
        const int m0 = (tile / p.tiles_n) * BM, n0 = (tile % p.tiles_n) * BN;
        const uint8_t* sfa_src = p.a_s + (static_cast<size_t>(m0 / 128) * p.kb4) * 512;
        for (int kb = 0; kb < p.kblocks; ++kb, ++u) {
          const int s = u % STAGES;
          if (!mbar_wait(smem_u32(&empty[s]), ((u / STAGES) & 1) ^ 1, p.status)) { *abort_flag = 1; break; }
          if (blockIdx.x == 0 && u == p.stall_u) continue;   // test hook: phase never completes
          const uint32_t fb = smem_u32(&full[s]);
          mbar_arrive_expect_tx(fb, C::TX_BYTES);
          tma_load_2d(smem_u32(sA + s * C::A_BYTES), &map_a, fb, kb * BKB, m0);
          tma_load_2d(smem_u32(sB + s * C::B_BYTES), &map_b, fb, kb * BKB, n0);
          bulk_load_1d(smem_u32(sSFA + s * C::SFA_BYTES), sfa_src + kb * C::SFA_BYTES, C::SFA_BYTES, fb);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            const uint8_t* src = p.b_s + (static_cast<size_t>(n0 / 128 + h) * p.kb4) * 512 + kb * C::SFA_BYTES;
            bulk_load_1d(smem_u32(sSFB + s * C::SFB_BYTES + h * C::SFA_BYTES), src, C::SFA_BYTES, fb);
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
      const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(smem_u32(sB), 16, 1024, 2);
      const uint64_t sfa_desc0 = smem_desc(smem_u32(sSFA), 0, 128, 0);
      const uint64_t sfb_desc0 = smem_desc(smem_u32(sSFB), 0, 128, 0);
      uint32_t idesc[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) idesc[kk] = instr_desc(C::AB_TYPE, BN, BM, C::FP4 ? (kk & 1) * 2 : kk);
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
          // scale chunks -> tensor memory (each 512-B chunk: 32 lanes x 16 B, x4 lane groups)
#pragma unroll
          for (int c = 0; c < C::SF_CHUNKS; ++c)
            tc_cp_sf(sfa_t + 4 * c, sfa_desc0 + ((s * C::SFA_BYTES + c * 512) >> 4));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
#pragma unroll
            for (int c = 0; c < C::SF_CHUNKS; ++c)
              tc_cp_sf(sfb_t + 4 * (BN / 128) * c + 4 * h, sfb_desc0 + ((s * C::SFB_BYTES + h * C::SFA_BYTES + c * 512) >> 4));
          const uint64_t ad = a_desc0 + ((s * C::A_BYTES) >> 4);
          const uint64_t bd = b_desc0 + ((s * C::B_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // 32 bytes of K per MMA (32 FP8 or 64 FP4 elements).  E2M1: K = 64
            // consumes two scales per row, chunk kk / 2, byte pair (kk % 2) * 2;
            // the BN rows of B's chunk sit in BN / 32 consecutive columns.
            const uint32_t sfa = C::FP4 ? sfa_t + 4 * (kk >> 1) : sfa_t;
            const uint32_t sfb = C::FP4 ? sfb_t + 4 * (BN / 128) * (kk >> 1) : sfb_t;
            tc_mma<C::FP4>(tmem, ad + 2 * kk, bd + 2 * kk, idesc[kk], sfa, sfb, (kb | kk) != 0);
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
    const int row = q * 32 + lane;                               // row within the tile
    const bool leader = (warp == EPI_WARP0 && lane == 0);
    int t = 0, buf = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++t) {
      const int m0 = (tile / p.tiles_n) * BM, n0 = (tile % p.tiles_n) * BN;
      // the four warps decide together, so none is left alone at a named barrier
      if (!mbar_wait(smem_u32(acc_full), t & 1, p.status)) *epi_fail = 1;
      named_bar(1, 128);
      if (*epi_fail) { *abort_flag = 1; break; }
      tc_fence_after();
      if (!p.out_fp32) {
        // bf16: drain the whole accumulator row into registers first, so the
        // MMA warp can start the next tile while this one is written out
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            pk[c * 16 + j] = *reinterpret_cast<const uint32_t*>(&b2);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(acc_empty));
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          if (leader) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          named_bar(1, 128);
          uint8_t* stg = sOut + buf * STG_BYTES;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int phys = j ^ ((row >> 1) & 3);               // 64-byte swizzle
            *reinterpret_cast<uint4*>(stg + row * 64 + phys * 16) =
                make_uint4(pk[c * 16 + 4 * j], pk[c * 16 + 4 * j + 1], pk[c * 16 + 4 * j + 2], pk[c * 16 + 4 * j + 3]);
          }
          fence_proxy_async_smem();
          named_bar(1, 128);
          if (leader) {
            tma_store_2d(&map_c, smem_u32(stg), n0 + c * 32, m0);
            bulk_commit();
          }
          buf ^= 1;
        }
        continue;
      }
      // float32 output: chunk by chunk
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, v);
        tmem_ld_wait();
        if (c0 + 32 == BN) {                                     // accumulator fully read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(acc_empty));
        }
        for (int h = 0; h < 2; ++h) {
          if (leader) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
          named_bar(1, 128);
          uint8_t* stg = sOut + buf * STG_BYTES;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int phys = j ^ ((row >> 1) & 3);               // 64-byte swizzle
            *reinterpret_cast<uint4*>(stg + row * 64 + phys * 16) =
                make_uint4(v[h * 16 + 4 * j], v[h * 16 + 4 * j + 1], v[h * 16 + 4 * j + 2], v[h * 16 + 4 * j + 3]);
          }
          fence_proxy_async_smem();
          named_bar(1, 128);
          if (leader) {
            tma_store_2d(&map_c, smem_u32(stg), n0 + c0 + h * 16, m0);
            bulk_commit();
          }
          buf ^= 1;
        }
      }
    }
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace gemm
}  // namespace mxq

// ==================================================================== host
using namespace mxq_host;

namespace {

template <int FMT, int BN>
int launch(const void* a_q, const uint8_t* a_s, const void* b_q, const uint8_t* b_s, int64_t M, int64_t N,
           int64_t K, void* c, int out_fp32, cudaStream_t st) {
  using namespace mxq::gemm;
  using Cf = Cfg<FMT, BN>;
  const int64_t kbytes = Cf::FP4 ? K / 2 : K;
  CUtensorMap ma, mb, mc;
  if (!encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_q, kbytes, M, kbytes, BKB, BM, CU_TENSOR_MAP_SWIZZLE_128B))
    return MXQ_ERR_CUDA;
  if (!encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_q, kbytes, N, kbytes, BKB, BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return MXQ_ERR_CUDA;
  if (out_fp32) {
    if (!encode_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, c, N, M, N * 4, 16, BM, CU_TENSOR_MAP_SWIZZLE_64B))
      return MXQ_ERR_CUDA;
  } else {
    if (!encode_2d(&mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c, N, M, N * 2, 32, BM, CU_TENSOR_MAP_SWIZZLE_64B))
      return MXQ_ERR_CUDA;
  }
  Params p{};
  p.a_s = a_s;
  p.b_s = b_s;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.tiles_m = static_cast<int>(M / BM);
  p.tiles_n = static_cast<int>(N / BN);
  p.ntiles = p.tiles_m * p.tiles_n;
  p.kblocks = static_cast<int>(kbytes / BKB);
  p.kb4 = static_cast<int>(K / 128);
  p.out_fp32 = out_fp32;
  p.status = status_ptr();
  p.stall_u = take_test_stall(2) ? 0 : -1;
  if (!p.status) return MXQ_ERR_CUDA;
  auto kern = mx_gemm_kernel<FMT, BN>;
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

}  // namespace

extern "C" int mxq_gemm(const void* a_q, const uint8_t* a_s, const void* b_q, const uint8_t* b_s, int64_t M,
                        int64_t N, int64_t K, int fmt, int sf_layout, void* c, int out_fp32, void* stream) {
  if (!a_q || !a_s || !b_q || !b_s || !c) return MXQ_ERR_BAD_ARG;
  if (fmt != MXQ_E4M3 && fmt != MXQ_E5M2 && fmt != MXQ_E2M1) return MXQ_ERR_BAD_ARG;
  if (sf_layout != MXQ_SF_MMA) return sf_layout == MXQ_SF_CANONICAL ? MXQ_ERR_UNSUPPORTED : MXQ_ERR_BAD_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || M % 128 || N % 128 || K % (fmt == MXQ_E2M1 ? 256 : 128))
    return MXQ_ERR_BAD_SHAPE;
  if (M > (1ll << 31) - 256 || N > (1ll << 31) - 256 || K > (1ll << 31) - 256) return MXQ_ERR_BAD_SHAPE;
  if (!aligned16(a_q) || !aligned16(b_q) || !aligned16(a_s) || !aligned16(b_s) || !aligned16(c))
    return MXQ_ERR_MISALIGNED;
  if (!device_ok()) return MXQ_ERR_UNSUPPORTED;
  auto st = static_cast<cudaStream_t>(stream);
  const bool n256 = (N % 256) == 0;
  switch (fmt) {
    case MXQ_E4M3: return n256 ? launch<MXQ_E4M3, 256>(a_q, a_s, b_q, b_s, M, N, K, c, out_fp32, st)
                               : launch<MXQ_E4M3, 128>(a_q, a_s, b_q, b_s, M, N, K, c, out_fp32, st);
    case MXQ_E5M2: return n256 ? launch<MXQ_E5M2, 256>(a_q, a_s, b_q, b_s, M, N, K, c, out_fp32, st)
                               : launch<MXQ_E5M2, 128>(a_q, a_s, b_q, b_s, M, N, K, c, out_fp32, st);
    default: return n256 ? launch<MXQ_E2M1, 256>(a_q, a_s, b_q, b_s, M, N, K, c, out_fp32, st)
                         : launch<MXQ_E2M1, 128>(a_q, a_s, b_q, b_s, M, N, K, c, out_fp32, st);
  }
}
