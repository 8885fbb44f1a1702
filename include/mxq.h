/*
 * mxq.h -- block-scaled (OCP MX) and per-tensor FP8 quantization of bf16
 * tensors, the block-scaled GEMM that consumes them (bf16, float32 or MX
 * output; same or mixed 8-bit formats) and the per-tensor FP8 GEMM, on NVIDIA
 * GB300 (sm_103a).  C ABI: plain pointers and sizes, int status codes, no
 * exceptions.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates or frees device memory; it keeps only a per-device
 *    cache of the SM count and a device status word.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Nothing is read back to the host.
 *  - Matrices are row-major.  "rows x cols" means cols is the contiguous
 *    dimension.
 *  - Element codes: one byte per FP8 element; E2M1 is packed two per byte,
 *    element 2i in the low nibble and 2i+1 in the high nibble.
 *  - Scale codes are UE8M0 bytes: code c means 2^(c-127); 0xFF is NaN.
 *  - Return value: MXQ_OK or a negative status (see mxq_strerror).  Argument
 *    checks happen before any launch; on error nothing is launched.
 *
 * Sources of the operations (page title, section):
 *  [MX]  "UE8M0 FP8 / MXFP8 explainer" (ag-981.com), section 1 (MX block of
 *        k = 32 elements sharing one UE8M0 scale X; quantizing V_i means
 *        finding X and q_i with q_i * X ~= V_i; tensor cores consume X and
 *        q_i of both operands), section 4 (scale from the block amax,
 *        saturating element quantization), gap section 1 (OCP round-down
 *        versus ceil(log2(amax/destmax)) scales), gap section 2 (row and
 *        column copies; blocks must run along the contiguous reduction
 *        dimension).
 *  [FP8] AstrAI astrai/extension/ops/fp8.py (commit 962c10c52b): commit
 *        message (last-block delayed-scaling fold with an atomic ticket) and
 *        the quantize / quantize_dual / mm_fp8 docstrings.
 *  [FAF] "Format-aware fusion for FP4" (theaicronicle.com): MXFP4 with
 *        row-gradient stochastic rounding and a fixed-sign 32-point
 *        Hadamard; producers emit the scale layout their consumer reads.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define MXQ_OK               0
#define MXQ_ERR_BAD_ARG     -1  /* NULL pointer, bad enum, bad ring index   */
#define MXQ_ERR_BAD_SHAPE   -2  /* size not a multiple of the block/tile    */
#define MXQ_ERR_MISALIGNED  -3  /* pointer or leading dimension not 16-B    */
#define MXQ_ERR_UNSUPPORTED -4  /* format/orientation combination, or GPU  */
#define MXQ_ERR_CUDA        -5  /* launch or driver error                   */
#define MXQ_ERR_TIMEOUT     -6  /* a bounded device wait expired            */

/* ---- enums ---------------------------------------------------------------- */
/* Element formats.  0/1 keep the E4M3/E5M2 numbering of [FP8] (_FMT_TO_INT). */
#define MXQ_E4M3 0
#define MXQ_E5M2 1
#define MXQ_E2M1 2
/* Orientation.  ROW: 1x32 blocks along cols, output q_row [rows][cols].
 * COL: 32x1 blocks along rows, output stored transposed, q_col [cols][rows]
 * (the K-contiguous copy [MX] gap section 2 asks for).  DUAL: both from one
 * read of x. */
#define MXQ_ROW  1
#define MXQ_COL  2
#define MXQ_DUAL 3
/* Scale rule [MX] gap section 1.
 * FLOOR_OCP: e = floor(log2 amax) - floor(log2 destmax).
 * CEIL:      e = ceil(log2(amax / destmax)), computed from exponent and
 *            mantissa bits (never saturates).
 * Both: amax == 0 -> e = -127; e clamped to [-127, 127]; a block holding
 * NaN/Inf gets scale 0xFF and zero codes. */
#define MXQ_SCALE_FLOOR_OCP 0
#define MXQ_SCALE_CEIL      1
/* Element rounding.  RNE: round to nearest, ties to even code, saturating
 * at the format maximum, sign kept on zero.  SR: stochastic rounding with
 * r = word 0 of Philox-4x32-10(key = sr_key, counter = (i, i >> 32, 0, 0)),
 * i = r*cols + c the element's index in x; with y' = min(|y|, max) between
 * grid neighbours lo < y' < hi, round up iff r < floor((y'-lo)/(hi-lo)*2^32).
 * SR4: the same rounding with four draws per generator call: r = word
 * (i & 3) of Philox-4x32-10(key = sr_key, counter = (c, c >> 32, 0, 0)),
 * c = i >> 2 (an option of this library, not of the pages: a quarter of the
 * generator work of SR, different draws). */
#define MXQ_RNE 0
#define MXQ_SR  1
#define MXQ_SR4 2
/* Scale-factor layout.
 * CANONICAL: row-major bytes, s_row [rows][cols/32], s_col [cols][rows/32].
 * MMA: the layout the GEMM's tensor-core scale path reads ([FAF]: the
 * producer writes its consumer's layout).  For a scale matrix of R rows and
 * KB = K/32 scale columns (R % 128 == 0, KB % 4 == 0): 512-byte chunks, chunk
 * (R/128 index rb, KB/4 index kc) at byte offset (rb*(KB/4) + kc)*512, and
 * inside a chunk the scale of row r and k-block k at byte
 * (r%32)*16 + ((r/32)%4)*4 + (k%4).  Same bytes, permuted. */
#define MXQ_SF_CANONICAL 0
#define MXQ_SF_MMA       1

/* ---- MX quantize ([MX] sections 1 and 4, gap sections 1-2; [FAF]) ----------
 * x        bf16 [rows][ld] (only the first cols of each row are read),
 *          16-byte aligned, ld % 8 == 0, ld >= cols.
 * rows, cols  positive multiples of 32 (an empty tensor is MXQ_ERR_BAD_SHAPE);
 *          rows % 128 == 0 and cols % 128 == 0 for MXQ_SF_MMA.
 * fmt      MXQ_E4M3 | MXQ_E5M2 | MXQ_E2M1.
 * orient   MXQ_ROW | MXQ_COL | MXQ_DUAL.
 * scale_mode  MXQ_SCALE_FLOOR_OCP | MXQ_SCALE_CEIL.
 * rounding MXQ_RNE | MXQ_SR | MXQ_SR4.
 * hadamard32  non-zero: before scale selection each 32-block (along its
 *          block direction) becomes y = c * H32 * D * v in float32: D holds
 *          the 32 signs given by bit j of word 0 of
 *          Philox-4x32-10(key = hadamard_seed, counter = 0) (set bit = -1),
 *          butterflies h = 1,2,4,8,16 in that order, c = RN32(1/sqrt(32)).
 * q_row, s_row  outputs for ROW/DUAL (else may be NULL): q_row
 *          [rows][cols] bytes (E2M1: [rows][cols/2]); s_row per sf_layout.
 * q_col, s_col  outputs for COL/DUAL: q_col [cols][rows] (E2M1:
 *          [cols][rows/2]); s_col per sf_layout.
 * All output pointers 16-byte aligned.  Outputs must not overlap x. */
int mxq_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                 int fmt, int orient, int scale_mode, int rounding,
                 int hadamard32, uint64_t sr_key, uint64_t hadamard_seed,
                 int sf_layout, void* q_row, uint8_t* s_row, void* q_col,
                 uint8_t* s_col, void* stream);

/* ---- Grouped MX quantize (no counterpart in the pages: a batching of
 * mxq_quantize) --------------------------------------------------------------
 * Up to MXQ_QUANT_GROUP_MAX tensors of one format and orientation, RNE
 * elements, no Hadamard, quantized in one launch: the tiles of all jobs form
 * one sequence that the persistent grid runs through, so the fill and drain
 * of a launch are paid once for the group instead of once per tensor.  Each
 * job's bytes are exactly those mxq_quantize(job.x, ..., fmt, orient,
 * job.scale_mode, MXQ_RNE, 0, 0, 0, sf_layout, ...) writes.
 * jobs     host array of njobs descriptions (read during the call only);
 *          every field as the same argument of mxq_quantize, all device
 *          pointers on the current device.
 * njobs    1 .. MXQ_QUANT_GROUP_MAX.
 * Errors: any job's argument error is returned as mxq_quantize would return
 * it, before anything is launched.  Outputs of different jobs must not
 * overlap one another or any input. */
#define MXQ_QUANT_GROUP_MAX 4
typedef struct mxq_quant_job {
  const void* x;               /* bf16 [rows][ld] */
  int64_t rows, cols, ld;
  int scale_mode;              /* MXQ_SCALE_FLOOR_OCP | MXQ_SCALE_CEIL */
  void* q_row;                 /* ROW / DUAL outputs (else NULL) */
  uint8_t* s_row;
  void* q_col;                 /* COL / DUAL outputs (else NULL) */
  uint8_t* s_col;
} mxq_quant_job;
int mxq_quantize_group(const mxq_quant_job* jobs, int njobs, int fmt,
                       int orient, int sf_layout, void* stream);

/* ---- MX dequantize ([MX] section 1: V_i ~= q_i * X) --------------------------
 * q        codes [rows][cols] (E2M1 packed [rows][cols/2]), s canonical
 *          scales [rows][cols/32].  out [rows][cols]: float32 when
 *          out_fp32 != 0 (exact product, overflow to Inf), else bf16 (RNE).
 * rows >= 1, cols % 32 == 0. */
int mxq_dequantize(const void* q, const uint8_t* s, int64_t rows, int64_t cols,
                   int fmt, int out_fp32, void* out, void* stream);

/* ---- per-tensor FP8 quantize with fused amax and delayed-scaling fold ([FP8])
 * x        bf16 [rows][cols], 16-byte aligned, cols % 16 == 0.  For COL/DUAL
 *          also rows % 16 == 0.
 * scale    device float: the quantization multiplier m; x8 = RNE-saturating
 *          FP8 of RN32(x * m).  May alias ring_state[hist_len + 1].
 * fmt      MXQ_E4M3 | MXQ_E5M2.
 * orient   MXQ_ROW -> x8 [rows][cols]; MXQ_COL -> x8T [cols][rows] only
 *          ([FP8] transposed=True); MXQ_DUAL -> both from one read.
 * ring_state  NULL, or device float[hist_len + 4] laid out
 *          [hist[hist_len] | scale | legacy | amax | done]; amax and done
 *          must be 0 on entry (the kernel leaves them 0).  The last block
 *          to finish folds the tensor amax into hist[hist_idx] and, if
 *          M = max(hist) is finite and > 0, publishes
 *          scale = RN32(RN32(M / fp8_max) / pow2_margin) and
 *          legacy = RN32(1 / scale) (the next step's multiplier).
 * amax_out NULL or device float: receives max|x| (without a ring it is
 *          zeroed on the stream first, so it must not alias x or outputs).
 *          At least one of ring_state / amax_out must be given.
 * Concurrent calls sharing a ring_state race; calls on one stream are
 * ordered. */
int fp8_quantize_pertensor(const void* x, int64_t rows, int64_t cols,
                           const float* scale, int fmt, int orient,
                           float* ring_state, int hist_len, int hist_idx,
                           float fp8_max, float pow2_margin, uint8_t* x8,
                           uint8_t* x8T, float* amax_out, void* stream);

/* ---- delayed-scaling fold of a given tensor amax ([FP8] commit message:
 * the fold takes the tensor's amax into the history and publishes the next
 * scale) ---------------------------------------------------------------------
 * The fold fp8_quantize_pertensor runs in its last block, as a call of its
 * own, for a tensor quantized in row shards (one shard per GPU, each a
 * multiple of 16 rows):
 *   1. each shard: fp8_quantize_pertensor(x_shard, scale = &ring[hist_len+1],
 *      ..., ring_state = NULL, ..., amax_out = a) -- a = the shard's amax;
 *   2. a MAX all-reduce of the 4-byte a over the shards (e.g. NCCL);
 *   3. each shard: fp8_ring_fold(a, ring, ...) on its own replica of the ring.
 * Every replica then holds the ring a single whole-tensor call would leave.
 * amax      device float: the tensor amax to fold (read by the kernel).
 * ring_state device float[hist_len + 4], [hist | scale | legacy | amax | done]:
 *           hist[hist_idx] = *amax; M = max(hist); if M is finite and > 0,
 *           scale = RN32(RN32(M / fp8_max) / pow2_margin) and
 *           legacy = RN32(1 / scale); amax and done are set to 0.
 * hist_len >= 1, 0 <= hist_idx < hist_len; both pointers 4-byte aligned.
 * One thread of the device does the fold, ordered on `stream`. */
int fp8_ring_fold(const float* amax, float* ring_state, int hist_len,
                  int hist_idx, float fp8_max, float pow2_margin,
                  void* stream);

/* ---- block-scaled GEMM ([MX] section 1: tensor cores consume X and q_i of
 * both operands, FP32 accumulation) -------------------------------------------
 * C[m][n] = sum_k dec(a[m][k]) * 2^(sa[m][k/32]-127) * dec(b[n][k]) *
 *           2^(sb[n][k/32]-127), accumulated in float32 on the tensor cores,
 * written as bf16 (RNE) or, with out_fp32 != 0, float32.
 * a_q [M][K] codes, b_q [N][K] codes (both K-contiguous; E2M1 packed
 *          [M][K/2], [N][K/2]); a_s, b_s scales in MXQ_SF_MMA layout.
 * fmt      MXQ_E4M3 | MXQ_E5M2 | MXQ_E2M1 (same for both operands).
 * M, N, K positive; M % 128 == 0, N % 128 == 0, K % 128 == 0 (E2M1:
 * K % 256 == 0).  Zero sizes are MXQ_ERR_BAD_SHAPE.
 * c [M][N], 16-byte aligned. */
int mxq_gemm(const void* a_q, const uint8_t* a_s, const void* b_q,
             const uint8_t* b_s, int64_t M, int64_t N, int64_t K, int fmt,
             int sf_layout, void* c, int out_fp32, void* stream);

/* ---- mixed-format block-scaled GEMM (same product; [MX] FP8 section: E4M3
 * for precision beside E5M2 for range, e.g. an E5M2 gradient times an E4M3
 * operand) ----------------------------------------------------------------------
 * As mxq_gemm, with a_fmt for A and b_fmt for B: any pair of E4M3 / E5M2 /
 * E2M1, e.g. MXFP8 activations times MXFP4 weights.  E2M1 with E2M1 is
 * mxq_gemm's MXFP4 product (K % 256 == 0).  E2M1 beside an 8-bit format
 * runs at the 8-bit rate and needs K % 128 == 0 and the E2M1 codes (still
 * packed [rows][K/2] in memory) 32-byte aligned, else MXQ_ERR_MISALIGNED. */
int mxq_gemm_mixed(const void* a_q, const uint8_t* a_s, int a_fmt,
                   const void* b_q, const uint8_t* b_s, int b_fmt,
                   int64_t M, int64_t N, int64_t K, int sf_layout, void* c,
                   int out_fp32, void* stream);

/* ---- block-scaled GEMM with a stream-K schedule ----------------------------
 * The product of mxq_gemm_mixed (same arguments, same output).  With a
 * workspace the CTA-pair kernel (M and N multiples of 256, bf16 or float32
 * output) balances its last waves: when the last wave of 256 x 256 output
 * tiles would keep at most a quarter of the GPU's CTA pairs busy, the
 * k-iterations of the last one to two waves of tiles are split into even
 * contiguous ranges, one per pair, and a tile cut by a
 * range boundary is finished by whichever of its two pieces ends second,
 * which adds the float32 sums the other parked in the workspace (so such a
 * tile's sum is RN32(first piece + second piece), a rounding order that
 * differs from an uncut tile within the float32 accumulation error; the
 * result does not depend on which piece ends first).
 * workspace  device memory of at least mxq_gemm_workspace_size bytes,
 *            256-byte aligned, zero-filled before its first use (the library
 *            keeps it valid afterwards).  Calls that share a workspace must
 *            not run concurrently (order them on one stream).  NULL, or
 *            fewer bytes, runs mxq_gemm_mixed's schedule.
 * Shapes and alignment as mxq_gemm_mixed. */
int mxq_gemm_workspace_size(size_t* bytes);
int mxq_gemm_ws(const void* a_q, const uint8_t* a_s, int a_fmt,
                const void* b_q, const uint8_t* b_s, int b_fmt,
                int64_t M, int64_t N, int64_t K, int sf_layout, void* c,
                int out_fp32, void* workspace, size_t workspace_bytes,
                void* stream);

/* ---- mxq_gemm_ws without a caller workspace (no counterpart on the pages:
 * an entry point of this library for callers that cannot allocate) -----------
 * Some callers cannot allocate device memory when they call: code running
 * inside another framework's executor that owns all of the device's memory,
 * or a plugin whose execute step is not allowed to allocate.  This call runs
 * the product of mxq_gemm_ws with the library's own scratch instead of a
 * caller workspace: a static array of MXQ_GEMM_NOALLOC_SCRATCH_BYTES in
 * device memory, which every device that loads the library holds until the
 * process exits.  The call itself allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before
 *    any stream capture.
 *  - Every call on a device shares the one array, which keeps what the last
 *    call left there.  Its ticket words carry a tag that is new for every
 *    launch, so nothing in it has to start at zero for a call (the array is
 *    zero when the library loads).  Calls that overlap on the GPU (on
 *    different streams, or from different threads without ordering) race
 *    on the array: order them on one stream.
 *  - The array covers the stream-K scratch of up to 80 CTA pairs (a GPU of
 *    up to 160 SMs); on a device that would need more the call returns
 *    MXQ_ERR_UNSUPPORTED and launches nothing.
 * Arguments, shapes, alignment and output as mxq_gemm_ws. */
#define MXQ_GEMM_NOALLOC_SCRATCH_BYTES ((size_t)20 * 1024 * 1024 + 4096)
int mxq_gemm_noalloc(const void* a_q, const uint8_t* a_s, int a_fmt,
                     const void* b_q, const uint8_t* b_s, int b_fmt,
                     int64_t M, int64_t N, int64_t K, int sf_layout,
                     void* c, int out_fp32, void* stream);

/* ---- block-scaled GEMM with an MX output (FAF article: producers emit the
 * format and scale layout their consumer reads, with no bf16 round trip;
 * gap section 2: row-wise and column-wise copies) -----------------------------
 * Same product as mxq_gemm_mixed.  Instead of C, writes MX codes of out_fmt
 * (MXQ_E4M3 | MXQ_E5M2 | MXQ_E2M1) with their UE8M0 scales:
 *   c_q, c_s    row blocks (1x32 along each row of C): codes [M][N] (E2M1
 *               packed [M][N/2]), scales canonical [M][N/32] or MXQ_SF_MMA
 *               (the layout mxq_gemm reads for an A operand);
 *   c_qT, c_sT  column blocks (32x1 along each column of C), stored
 *               transposed: codes [N][M] of C^T (E2M1 [N][M/2]), scales
 *               canonical [N][M/32] or MXQ_SF_MMA (the layout of a B operand
 *               along M).
 * Either pair may be NULL (both of a pair, not one), not both pairs.
 * The block scale (out_scale_mode MXQ_SCALE_FLOOR_OCP | MXQ_SCALE_CEIL) and
 * the RNE-saturating element rounding follow mxq_quantize, applied to the
 * float32 accumulator.  A block holding NaN/Inf gets scale 0xFF and zero
 * codes.  Outputs 16-byte aligned.  An E2M1 output in the MMA layout feeds
 * the next MXFP4 product directly (format-aware fusion for FP4). */
int mxq_gemm_mx_out(const void* a_q, const uint8_t* a_s, int a_fmt,
                    const void* b_q, const uint8_t* b_s, int b_fmt,
                    int64_t M, int64_t N, int64_t K, int sf_layout,
                    int out_fmt, int out_scale_mode, int out_sf_layout,
                    uint8_t* c_q, uint8_t* c_s, uint8_t* c_qT, uint8_t* c_sT,
                    void* stream);

/* ---- per-tensor FP8 GEMM (AstrAI fp8.py, mm_fp8: "a @ b * scale (+ bias)",
 * op() transposes when trans_a / trans_b is set, and a view that swaps the
 * last two axes is read where it lies, with no copy; scale is the combined
 * dequantization scale, bias is added in the fp32 epilogue, the result is
 * bf16) --------------------------------------------------------------------------
 * c[i][m][n] = bf16_RNE( RN32( RN32(acc * scale) + bias[n] ) ), acc the
 * float32 tensor-core sum over k of dec(op(a)[i][m][k]) * dec(op(b)[i][k][n]).
 * a        FP8 codes, row-major: [batch][M][K] (trans_a == 0, op(a) = a) or
 *          [batch][K][M] (trans_a == 1, op(a) = a^T); without a_batched one
 *          matrix ([M][K] or [K][M]) serves every batch entry.
 * b        FP8 codes, row-major: [batch][K][N] (trans_b == 0, op(b) = b) or
 *          [batch][N][K] (trans_b == 1, op(b) = b^T, e.g. a weight stored
 *          [out][in]); without b_batched one matrix serves every entry.
 *          All four trans_a / trans_b combinations read the operands in
 *          place (K-contiguous or M / N-contiguous rows).
 * fmt      MXQ_E4M3 | MXQ_E5M2 for both operands.
 * scale    device float (4-byte aligned), read by the kernel.
 * bias     NULL or device bf16 [N], 16-byte aligned.
 * c        bf16 [batch][M][N], 16-byte aligned.
 * batch >= 1; M, N, K multiples of 128. */
int mxq_mm_fp8(const void* a, const void* b, int64_t batch, int64_t M,
               int64_t N, int64_t K, int a_batched, int b_batched,
               int trans_a, int trans_b, int fmt, const float* scale,
               const void* bias, void* c, void* stream);

/* ---- scale layout conversion ([FAF]) -----------------------------------------
 * Canonical scales s [rows][kb] -> MMA layout (rows % 128 == 0,
 * kb % 4 == 0).  out holds rows*kb bytes; must not overlap s. */
int mxq_sf_to_mma(const uint8_t* s, int64_t rows, int64_t kb, uint8_t* out,
                  void* stream);

/* ---- diagnostics ----------------------------------------------------------
 * mxq_last_device_status: synchronizes `stream`, returns MXQ_ERR_TIMEOUT if
 * any kernel of this library on the current device gave up a bounded wait
 * since the last call (then clears the word), MXQ_ERR_CUDA on a CUDA error,
 * else MXQ_OK. */
int mxq_last_device_status(void* stream);
const char* mxq_strerror(int status);
/* Library version, major*10000 + minor*100 + patch. */
int mxq_version(void);

/* Failure-detection test hook (no counterpart on the pages).  which = 1 arms
 * the next mxq_quantize call, 2 the next mxq_gemm call, 0 disarms: in that
 * launch CTA 0 leaves one of its input stages unloaded, so the mbarrier phase
 * that stage's consumer waits on never completes.  The bounded wait expires
 * after about a second, the kernel records MXQ_ERR_TIMEOUT in the device
 * status word, winds all of its roles down (awaiting its own copies, with a
 * limit, and releasing tensor memory) and exits; the CUDA context stays
 * usable.  The launch's outputs are then unspecified.  Returns MXQ_OK, or
 * MXQ_ERR_BAD_ARG for another value of which.  Not for production use. */
int mxq_test_stall_next_launch(int which);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
