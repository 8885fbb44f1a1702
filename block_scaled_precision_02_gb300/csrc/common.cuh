// Shared device helpers of the sm_103a kernels: status word, bounded
// mbarrier waits, TMA (cp.async.bulk.tensor) wrappers, tensor-map encoding.
// Every wait here gives up after a wall-clock limit, records MXQ_ERR_TIMEOUT
// in the device status word and lets the kernel wind down; nothing traps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "../../include/mxq.h"

namespace mxq {

// Wall-clock limit of one bounded wait, in nanoseconds (1 s).  No legitimate
// wait in these kernels lasts longer than a few hundred microseconds.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// The device status word (0 or a negative MXQ status) lives in api.cu; each
// kernel receives its address.
__device__ __forceinline__ void record_timeout(int* status) { atomicExch(status, MXQ_ERR_TIMEOUT); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about hint_ns elapse, instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (and records a timeout) if it did not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  // spin for the first few microseconds (fast wake-up on the critical path),
  // then sleep in the barrier between checks (no issue slots burnt)
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      const unsigned long long dt = globaltimer_ns() - t0;
      if (dt > kWaitLimitNs) {
        record_timeout(status);
        return false;
      }
      if (dt > 4000u) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
      }
    }
  }
}

// Cluster-scope variant, for barriers that other CTAs of the cluster (or
// their async copies and tensor-core commits) complete.
__device__ __forceinline__ bool mbar_try_wait_cl_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait that lets the hardware suspend the thread until the phase
// completes (no polling loop competing for issue slots and the barrier unit
// with the thread that issues tensor-core work); cluster-scope acquire.
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity, int* status) {
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cl_sleep(bar, parity, 1000000u)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_timeout(status);
      return false;
    }
  }
}

// Address of the same shared-memory object in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// Tile load of a CTA pair: the data lands in this CTA's shared memory and the
// byte count completes on `bar_cluster`, an mbarrier in either CTA of the pair
// (a shared::cluster address, see cluster_map).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All committed bulk stores have finished READING shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// All committed bulk stores have completed (writes visible).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Prefetch one tile of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Plain 1-D bulk copy global -> shared (16-B aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- dependent launch
// Kernels are launched with programmatic stream serialization: a kernel may
// start while the previous one in the stream is finishing.  Every thread
// runs grid_dep_wait() before its first global-memory access (it returns once
// the previous grid has completed and its writes are visible; a no-op when
// there is none), so ordering is as for a plain launch; only the prologue
// overlaps.  grid_dep_launch() lets the next kernel begin its own prologue.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- bf16 / fp8 bits
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Pack two float32 into FP8 (RNE, saturating to the format maximum).  The
// first element lands in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
  uint16_t r;
  if constexpr (FMT == MXQ_E4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

// Four float32 to four FP8 codes in one word (a lowest byte, d highest):
// two paired conversions whose 16-bit results are joined without shifts.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x4(float a, float b, float c, float d) {
  uint32_t r;
  if constexpr (FMT == MXQ_E4M3) {
    asm("{\n\t.reg .b16 t0, t1;\n\tcvt.rn.satfinite.e4m3x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t1, %4, %3;\n\tmov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
  } else {
    asm("{\n\t.reg .b16 t0, t1;\n\tcvt.rn.satfinite.e5m2x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 t1, %4, %3;\n\tmov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
  }
  return r;
}

// The multiplier m twice, as the 64-bit operand of a packed f32x2 multiply.
__device__ __forceinline__ uint64_t f32x2_splat(float m) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(m));
  return r;
}

// Packed pairs of float32 (first element in the low half) and the packed
// operations on them: each half rounds to nearest exactly as the scalar
// operation would.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// FP8 codes of lo(wa), hi(wa), lo(wb), hi(wb) -- four bf16 values (packed
// two per word, element 2i in the low half) each multiplied by m (RN, with
// one packed f32x2 multiply per pair) and converted RNE-saturating.  Code of
// the first element in the lowest byte.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4_rows(uint32_t wa, uint32_t wb, uint64_t mm) {
  uint32_t r;
  if constexpr (FMT == MXQ_E4M3) {
    asm("{\n\t.reg .b32 a0, a1, b0, b1;\n\t.reg .b64 pa, pb;\n\t.reg .b16 t0, t1;\n\t"
        "shl.b32 a0, %1, 16;\n\tand.b32 a1, %1, 0xFFFF0000;\n\t"
        "shl.b32 b0, %2, 16;\n\tand.b32 b1, %2, 0xFFFF0000;\n\t"
        "mov.b64 pa, {a0, a1};\n\tmov.b64 pb, {b0, b1};\n\t"
        "mul.rn.f32x2 pa, pa, %3;\n\tmul.rn.f32x2 pb, pb, %3;\n\t"
        "mov.b64 {a0, a1}, pa;\n\tmov.b64 {b0, b1}, pb;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t0, a1, a0;\n\tcvt.rn.satfinite.e4m3x2.f32 t1, b1, b0;\n\t"
        "mov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r) : "r"(wa), "r"(wb), "l"(mm));
  } else {
    asm("{\n\t.reg .b32 a0, a1, b0, b1;\n\t.reg .b64 pa, pb;\n\t.reg .b16 t0, t1;\n\t"
        "shl.b32 a0, %1, 16;\n\tand.b32 a1, %1, 0xFFFF0000;\n\t"
        "shl.b32 b0, %2, 16;\n\tand.b32 b1, %2, 0xFFFF0000;\n\t"
        "mov.b64 pa, {a0, a1};\n\tmov.b64 pb, {b0, b1};\n\t"
        "mul.rn.f32x2 pa, pa, %3;\n\tmul.rn.f32x2 pb, pb, %3;\n\t"
        "mov.b64 {a0, a1}, pa;\n\tmov.b64 {b0, b1}, pb;\n\t"
        "cvt.rn.satfinite.e5m2x2.f32 t0, a1, a0;\n\tcvt.rn.satfinite.e5m2x2.f32 t1, b1, b0;\n\t"
        "mov.b32 %0, {t0, t1};\n\t}"
        : "=r"(r) : "r"(wa), "r"(wb), "l"(mm));
  }
  return r;
}

// FP8 codes of one column of four consecutive rows: the low (HALF = 0) or
// high (HALF = 1) bf16 of words w0..w3, multiplied by m and converted as in
// fp8x4_rows.  Code of w0's element in the lowest byte.
template <int FMT, int HALF>
__device__ __forceinline__ uint32_t fp8x4_col(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint64_t mm) {
  uint32_t r;
#define MXQ_COL_BODY(EXTRACT, CVT)                                                         \
  asm("{\n\t.reg .b32 a0, a1, b0, b1;\n\t.reg .b64 pa, pb;\n\t.reg .b16 t0, t1;\n\t" \
      EXTRACT                                                                            \
      "mov.b64 pa, {a0, a1};\n\tmov.b64 pb, {b0, b1};\n\t"                             \
      "mul.rn.f32x2 pa, pa, %5;\n\tmul.rn.f32x2 pb, pb, %5;\n\t"                      \
      "mov.b64 {a0, a1}, pa;\n\tmov.b64 {b0, b1}, pb;\n\t"                             \
      CVT " t0, a1, a0;\n\t" CVT " t1, b1, b0;\n\t"                                    \
      "mov.b32 %0, {t0, t1};\n\t}"                                                      \
      : "=r"(r) : "r"(w0), "r"(w1), "r"(w2), "r"(w3), "l"(mm))
#define MXQ_LO "shl.b32 a0, %1, 16;\n\tshl.b32 a1, %2, 16;\n\tshl.b32 b0, %3, 16;\n\tshl.b32 b1, %4, 16;\n\t"
#define MXQ_HI "and.b32 a0, %1, 0xFFFF0000;\n\tand.b32 a1, %2, 0xFFFF0000;\n\tand.b32 b0, %3, 0xFFFF0000;\n\tand.b32 b1, %4, 0xFFFF0000;\n\t"
  if constexpr (FMT == MXQ_E4M3) {
    if constexpr (HALF == 0) MXQ_COL_BODY(MXQ_LO, "cvt.rn.satfinite.e4m3x2.f32");
    else MXQ_COL_BODY(MXQ_HI, "cvt.rn.satfinite.e4m3x2.f32");
  } else {
    if constexpr (HALF == 0) MXQ_COL_BODY(MXQ_LO, "cvt.rn.satfinite.e5m2x2.f32");
    else MXQ_COL_BODY(MXQ_HI, "cvt.rn.satfinite.e5m2x2.f32");
  }
#undef MXQ_LO
#undef MXQ_HI
#undef MXQ_COL_BODY
  return r;
}

// Pack two float32 into E2M1 (RNE, saturating): first element in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------- MX scale rule
// destmax = m_d * 2^E_d: exponent and 23-bit mantissa field of the largest
// finite element (E4M3 1.75*2^8, E5M2 1.75*2^15, E2M1 1.5*2^2).
template <int FMT> struct FmtInfo;
template <> struct FmtInfo<MXQ_E4M3> { static constexpr int Ed = 8;  static constexpr uint32_t md = 0x600000u; static constexpr int mbits = 3; static constexpr int emin = -6;  static constexpr float maxv = 448.f; };
template <> struct FmtInfo<MXQ_E5M2> { static constexpr int Ed = 15; static constexpr uint32_t md = 0x600000u; static constexpr int mbits = 2; static constexpr int emin = -14; static constexpr float maxv = 57344.f; };
template <> struct FmtInfo<MXQ_E2M1> { static constexpr int Ed = 2;  static constexpr uint32_t md = 0x400000u; static constexpr int mbits = 1; static constexpr int emin = 0;   static constexpr float maxv = 6.f; };

// Shared exponent e from the block amax given as float32 bits (>= 0, finite;
// bf16 values are exact float32): floor rule e = E(amax) - E(destmax); ceil
// rule adds 1 when amax's mantissa field exceeds destmax's.  A zero or
// subnormal amax has E <= -127, so with E(destmax) >= 2 the clamp to
// [-127, 127] gives -127 -- the amax == 0 rule -- without special cases.
template <int FMT>
__device__ __forceinline__ int scale_exp(uint32_t ab, int ceil_mode) {
  int e = static_cast<int>(ab >> 23) - 127 - FmtInfo<FMT>::Ed;
  if (ceil_mode && (ab & 0x7FFFFFu) > FmtInfo<FMT>::md) e += 1;
  return max(-127, min(127, e));
}

// NaN-propagating maximum of three float32 values: a NaN operand gives NaN,
// subnormals are kept.
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Bits of the largest magnitude among 32 float32 values, mag(j) = |v_j|, by
// a tree of 16 three-input maxima: a NaN anywhere gives NaN bits, an
// infinity 0x7F800000, otherwise the largest |v_j| exactly -- the same
// classification and bits as the unsigned maximum of the sign-cleared words.
template <typename Mag>
__device__ __forceinline__ uint32_t amax32_tree(Mag mag) {
  float t[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) t[i] = fmax3_nan(mag(3 * i), mag(3 * i + 1), mag(3 * i + 2));
  t[10] = fmax3_nan(mag(30), mag(31), 0.0f);
  const float u = fmax3_nan(fmax3_nan(t[0], t[1], t[2]), fmax3_nan(t[3], t[4], t[5]), fmax3_nan(t[6], t[7], t[8]));
  return __float_as_uint(fmax3_nan(u, t[9], t[10])) & 0x7FFFFFFFu;
}

// 2^-e as float32 (e in [-127, 125] here, so the result is a normal number).
__device__ __forceinline__ float exp2_neg(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// ---------------------------------------------------------------- Philox-4x32-10
// Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11),
// section 3.3: per round, two 32x32->64 multiplies; key bumped by the Weyl
// constants between rounds.
struct u32x4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ u32x4 philox4x32_10(u32x4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = u32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

}  // namespace mxq

// ---------------------------------------------------------------- host side
namespace mxq_host {

// Encode a 2-D tiled tensor map (row-major, inner dimension first).
// Returns false if the driver rejects the description.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle);

// Number of SMs of the current device (cached per device).
int sm_count();

// True if the current device is an sm_103 part.
bool device_ok();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launch_status();

// Launch kernel with programmatic stream serialization (see grid_dep_wait).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? launch_status() : MXQ_ERR_CUDA;
}

// Same, for a kernel launched in clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
int launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? launch_status() : MXQ_ERR_CUDA;
}

// Device address of the status word of the current device.
int* status_ptr();

// Failure-detection test hook: true (once) if mxq_test_stall_next_launch(which)
// armed it (which: 1 quantizer, 2 GEMM).
bool take_test_stall(int which);

}  // namespace mxq_host
