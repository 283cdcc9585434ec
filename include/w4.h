/*
 * w4.h -- C ABI of the int4 weight-only GEMV/GEMM library for GB300 (sm_103a).
 *
 * Operations (sources are the web pages on int4 weight-only quantisation,
 * cited by page title and section):
 *   quantize_pack_int4  per-column symmetric int4 quantisation of W[K][N] and
 *                       the column pack of two rows per byte
 *                       ("[PHI] add int4 weight only quant kernel, add int4
 *                       weight only permute kernel", section "int4量化kernel").
 *   permute_int4        the int4 interleave permute of the packed matrix
 *                       (same page, sections "int4 permute kernel",
 *                       "简单的位运算", "int4 row interval").
 *   gemv_w4             fused dequant GEMV / small-batch multiply,
 *                       d[c][r] = sum_k (q[r][k] - zero[r]) * scale[r] * x[c][k]
 *                       ("怎样在安卓端利用 Vulkan 编写 4-bit 专用算子", sections 1
 *                       and 2; batched form from "三值量化模型的无损压缩", section 3).
 *   gemv_w4_permuted    the same multiply over permute_int4's output (the
 *                       interleaved layout the page builds for the fast
 *                       int4 -> 16-bit dequant), symmetric per-column scale.
 *   gemm_w4             large-M bf16 x int4 dequant GEMM
 *                       ("int4 gemm kernel", the matmul_bf16_int4 example);
 *                       gemm_w4_permuted, the same over permute_int4's output.
 *   quantize_int8, permute_int8, gemv_w8, gemm_w8
 *                       the int8 weight-only counterparts (the first page's
 *                       int8 permute, from which its int4 permute derives).
 *   quantize_q8_1_pt, gemv_w4a8
 *                       x quantised to block_q8_1 in the "PT" planes, and
 *                       gemv_w4's int4 weights against it with integer dot
 *                       products ("三值量化模型的无损压缩", sections 3 and 3.1).
 *   mmvq_ptq1_0, mmvq_ptq1_1
 *                       ternary weights in PTQ1_0 blocks, or in the PTQ1_1
 *                       superblocks that pack eight of them, against x in
 *                       that form (same page, sections 2, 3 and 3.2).
 *   ptq1_1_codebook, ptq1_1_encode
 *                       host-side conversion of ternary PTQ1_0 blocks into
 *                       PTQ1_1 superblocks ("三值量化模型的无损压缩", section 2).
 *
 * Conventions shared by every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or retains them, and keeps no per-call state.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on that stream and returns; the
 *     results are ready when the stream reaches that point.
 *   - Arguments are validated on the host before anything is enqueued: a
 *     NULL pointer gives W4_ERR_NULL, an illegal size W4_ERR_SHAPE, a pointer
 *     that is not 16-byte aligned W4_ERR_ALIGN, an unknown dtype W4_ERR_DTYPE;
 *     in all those cases nothing is launched and no output is touched.  A
 *     CUDA error while launching gives W4_ERR_CUDA (the CUDA error itself is
 *     left for cudaGetLastError of the caller's runtime to report),
 *     W4_ERR_DEVICE means the current device is not an sm_103 GPU, and
 *     W4_ERR_VALUE an input value the format cannot hold (host conversions).
 *   - Sizes are int64_t; every size must be >= 0.  Outputs are fully
 *     overwritten (their prior contents never matter).  Inputs and outputs
 *     must not overlap.
 *   - Calls are re-entrant and may run concurrently on different streams.
 */
#ifndef W4_H_
#define W4_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4_OK = 0,
    W4_ERR_NULL = -1,
    W4_ERR_SHAPE = -2,
    W4_ERR_ALIGN = -3,
    W4_ERR_DTYPE = -4,
    W4_ERR_CUDA = -5,
    W4_ERR_DEVICE = -6,
    W4_ERR_VALUE = -7
} w4_status;

/* Largest K that gemv_w4 accepts. */
#define W4_GEMV_MAX_K 40960

/* Element type of gemv_w4's x, scale, zero and d (all four share it). */
typedef enum { W4_F32 = 0, W4_BF16 = 1 } w4_dtype;

/* Version of this ABI (bumped on any signature change). */
int w4_abi_version(void);

/* Static text for a status code. */
const char* w4_status_string(w4_status status);

/*
 * Device-side error word.  Kernels never trap: a wait that exceeds its
 * iteration/time limit (about two seconds) records a nonzero code here,
 * drains the work it already issued, frees its tensor memory and returns.
 * This call synchronises `stream`, then returns and clears the first code
 * recorded on the current device (0 = none, 1 = a pipeline wait timed out,
 * 2 = a PTQ1_1 superblock's pattern index named no codebook entry or escape;
 * its blocks then count as d = 0), or -1 if the synchronisation or the read
 * failed.
 */
int w4_device_error(void* stream);

/*
 * w4_selftest_wait_timeout -- test of the device error path: one CTA runs the
 * library's bounded mbarrier wait on a barrier that nothing completes.  The
 * wait gives up after its limit (about two seconds), the kernel writes 0 to
 * *waited (DEVICE int, 1 if the wait had completed) and records code 1 for
 * w4_device_error; the context stays usable.  Nothing faults, traps or hangs.
 */
w4_status w4_selftest_wait_timeout(int* waited, void* stream);

/*
 * w4_selftest_configure -- test hook for the pipelined kernels' error path
 * (no counterpart on the pages).  wait_limit_clocks > 0 sets how many SM
 * clock cycles every bounded wait of the library lasts before it gives up
 * (<= 0 restores the default 2^32, about two seconds); short_first_stage != 0
 * makes the producers of gemv_w4 / gemv_w4_permuted (the tensor-core path)
 * and of the gemm_w4 family announce 16 bytes more than they copy for their
 * first stage, so that stage's wait can never complete: the kernel then runs
 * out the limit, records code 1 for w4_device_error, stops issuing, drains
 * the copies already issued, frees its tensor memory and returns, having
 * stored (possibly meaningless) results only inside its output.  Nothing
 * faults, traps or hangs.  Synchronises the device first; the settings hold
 * for the whole process until changed.  Call (0, 0) to return to normal
 * operation.  Never needed by a user of the library.
 */
w4_status w4_selftest_configure(long long wait_limit_clocks, int short_first_stage);

/*
 * quantize_pack_int4 -- symmetric per-column int4 quantisation + column pack.
 *
 *   scale[n]  = max_k |W[k][n]| / 7                (IEEE fp32 division)
 *   q[k][n]   = clamp(round(W[k][n] / scale[n]), -8, 7)
 *               (IEEE fp32 division; round half away from zero; a column
 *               whose maximum is 0 gets scale 0 and q = 0)
 *   packed[k/2][n] = (q[k][n] & 0xF) | ((q[k+1][n] & 0xF) << 4)
 *               (two rows per byte along K, even row in the low nibble)
 *
 * W       bf16 [K][N] row-major (N contiguous), 16-byte aligned.
 * packed  int8 [K/2][N] row-major, 16-byte aligned (output).
 * scale   fp32 [N], 16-byte aligned (output).
 * K must be even; K == 0 writes scale = 0 and nothing else; N == 0 is a no-op.
 * NaN or Inf in W is undefined.  Results are bit-exact with the
 * definition above.
 */
w4_status quantize_pack_int4(const void* W, void* packed, float* scale, int64_t K, int64_t N,
                             void* stream);

/*
 * permute_int4 -- the int4 interleave permute for a fast-dequant consumer.
 *
 * For each column n, with b[j] = packed[j][n] (j < K/2, "total_k" = K/2):
 *   1. byte permute inside every 16-byte group: source byte t goes to
 *      position (0 4 8 12 2 6 10 14 1 5 9 13 3 7 11 15)[t];
 *   2. nibble swap inside every 4-byte group p0..p3 of the result:
 *      p0' = lo(p0)|lo(p2)<<4, p1' = lo(p1)|lo(p3)<<4,
 *      p2' = hi(p0)|hi(p2)<<4, p3' = hi(p1)|hi(p3)<<4;
 *   3. row interleave: byte j of the column's stream is stored at
 *      out[j%32 + (j/32)*128 + 32*(n%4) + (K/2)*4*(n/4)].
 * The result is N/4 runs of 2K bytes; every 32-byte chunk of four adjacent
 * columns is interleaved.  In each 32-bit word the nibble slots hold the
 * k-indices 0 8 16 24 1 9 17 25 (+2 per further word, +32 per 16-byte group),
 * the order a fast dequant reading slots 0 2 4 6 1 3 5 7 turns into
 * 0 1 8 9 16 17 24 25 ...
 *
 * packed  int8 [K/2][N] (the output of quantize_pack_int4), 16-byte aligned.
 * out     int8 [N*K/2], 16-byte aligned (output).
 * Requires K % 64 == 0 and N % 4 == 0 (else W4_ERR_SHAPE); K == 0 or N == 0
 * is a no-op.  Bit-exact.
 */
w4_status permute_int4(const void* packed, void* out, int64_t K, int64_t N, void* stream);

/* Largest K that quantize_pack_permute_int4 accepts (eight CTAs of a
 * cluster hold the strip of W in shared memory). */
#define W4_QUANT_PERMUTE_MAX_K 26624

/*
 * quantize_pack_permute_int4 -- quantize_pack_int4 and permute_int4 in one
 * pass: W is read from memory once and the packed matrix is never stored
 * ("[PHI] add int4 weight only quant kernel, add int4 weight only permute
 * kernel", sections "int4量化kernel", "int4 permute kernel", "简单的位运算",
 * "int4 row interval").
 *
 * Writes scale exactly as quantize_pack_int4 does, and into `permuted`
 * (N*K/2 bytes) exactly what permute_int4 would produce from
 * quantize_pack_int4's packed matrix.  Bit-exact with both definitions.
 *
 * W         bf16 [K][N] row-major, 16-byte aligned.
 * permuted  int8 [N*K/2], 16-byte aligned (output).
 * scale     fp32 [N], 16-byte aligned (output).
 * Requires K % 64 == 0, N % 8 == 0 and K <= W4_QUANT_PERMUTE_MAX_K (else
 * W4_ERR_SHAPE; the two separate calls cover every other shape).  K == 0
 * writes scale = 0 and nothing else; N == 0 is a no-op.  NaN or Inf in W is
 * undefined.
 */
w4_status quantize_pack_permute_int4(const void* W, void* permuted, float* scale, int64_t K, int64_t N,
                                     void* stream);

/*
 * gemv_w4 -- fused dequant GEMV / small-batch multiply.
 *
 *   d[c][r] = sum_k (q[r][k] - zero[r]) * scale[r] * x[c][k],  0 <= c < C
 *
 * qweight  uint32 [N][K/8] row-major: word i of row r holds q[r][8i+j] in
 *          bits 4j..4j+3 (packed = (w7<<28)|...|(w1<<4)|w0), unsigned 0..15.
 * scale, zero  [N] of `dtype`.
 * x        [C][K] of `dtype`, row-major.
 * d        [C][N] of `dtype`, row-major (output).
 * All pointers 16-byte aligned.  K % 8 == 0 (the caller pads K),
 * K <= W4_GEMV_MAX_K (x is held in the shared memory of at most eight SMs),
 * 1 <= C <= 8, N >= 0.  K == 0 gives d = 0.  Accumulation is fp32; with dtype W4_BF16 the
 * result is rounded once to bf16.  The difference from the exact value is
 * bounded by the parity tolerance of the test suite (2e-3 * sum_k |w*x|
 * for bf16, 1e-5 * sum_k |w*x| for fp32).
 */
w4_status gemv_w4(const void* qweight, const void* scale, const void* zero, const void* x, void* d,
                  int64_t N, int64_t K, int64_t C, w4_dtype dtype, void* stream);

/*
 * gemv_w4_permuted -- multiply by the quantiser's weights in the permuted
 * layout, without undoing the permute.
 *
 *   d[c][n] = sum_k q[k][n] * scale[n] * x[c][k],  0 <= c < C
 *
 * ("[PHI] add int4 weight only quant kernel, add int4 weight only permute
 * kernel", sections "int4量化kernel" and "int4 permute kernel": q is the
 * two's complement int4 of quantize_pack_int4, permute_int4 arranges it so
 * that one shift-and-mask per pair yields the values in the order the MMA
 * fragments take them.)
 *
 * permuted  N*K/2 bytes, the output of permute_int4 for the packed
 *           [K/2][N] matrix (column groups of 4, 128-byte lines of 64 k).
 * scale     fp32 [N] (quantize_pack_int4's scale).
 * x         bf16 [C][K] row-major.
 * d         bf16 [C][N] row-major (output).
 * All pointers 16-byte aligned.  K % 64 == 0 and N % 4 == 0 (the permute's
 * own requirements), K <= W4_GEMV_MAX_K, 1 <= C <= 8; else W4_ERR_SHAPE.
 * K == 0 gives d = 0.  fp32 accumulation, one bf16 rounding; the tolerance
 * is gemv_w4's (2e-3 * sum_k |w*x|).
 */
w4_status gemv_w4_permuted(const void* permuted, const float* scale, const void* x, void* d, int64_t N, int64_t K,
                           int64_t C, void* stream);

/*
 * gemm_w4 -- large-M bf16 x int4 dequant GEMM on the tcgen05 tensor cores.
 *
 *   C[m][n] = scale[n] * sum_k A[m][k] * (u[k][n] - zero[n])
 *
 * A      bf16 [M][K] row-major.
 * B      int8 [K/2][N] row-major; byte (kp, n) holds u[2kp][n] in its low
 *        nibble and u[2kp+1][n] in its high nibble, both unsigned 0..15.
 * scale, zero  bf16 [N].
 * C      bf16 [M][N] row-major (output).
 * All pointers 16-byte aligned.  Requires M, N, K >= 0 with K % 64 == 0 and
 * N % 16 == 0 (so that every row of A, B and C starts on a 16-byte
 * boundary, as the tensor-memory-access copies need); any M.  K == 0 gives C = 0.  Products are bf16 x bf16 on the
 * tensor cores with fp32 accumulation; the dequantised weight (u - zero[n])
 * is formed in bf16 (exact whenever it is representable, e.g. for integer
 * zero points) and the result is rounded once to bf16.
 */
w4_status gemm_w4(const void* A, const void* B, const void* scale, const void* zero, void* C,
                  int64_t M, int64_t N, int64_t K, void* stream);

/*
 * quantize_int8 -- symmetric per-column int8 quantisation of W[K][N] (the
 * int4 quantiser's definition with the int8 range; "[PHI] add int4 weight
 * only quant kernel, add int4 weight only permute kernel").
 *
 *   scale[n] = max_k |W[k][n]| / 127              (IEEE fp32 division)
 *   q[k][n]  = clamp(round(W[k][n] / scale[n]), -128, 127)
 *              (IEEE fp32 division; round half away from zero; a column
 *              whose maximum is 0 gets scale 0 and q = 0)
 *
 * W      bf16 [K][N] row-major, 16-byte aligned.
 * q      int8 [K][N] row-major, 16-byte aligned (output).
 * scale  fp32 [N], 16-byte aligned (output).
 * K == 0 writes scale = 0 and nothing else; N == 0 is a no-op.  NaN or Inf
 * in W is undefined.  Bit-exact with the definition above.
 */
w4_status quantize_int8(const void* W, void* q, float* scale, int64_t K, int64_t N, void* stream);

/*
 * permute_int8 -- the int8 interleave permute (same page, section
 * "如何从int8 permute转换为int4 permute" for the element order and section
 * "int4 row interval" for the interleave of two adjacent columns every 64
 * elements).  For each column n, with b[k] = q[k][n]:
 *   1. element permute inside every 16-element group: source element t goes
 *      to position (0 2 4 6 8 10 12 14 1 3 5 7 9 11 13 15)[t];
 *   2. row interleave: element kk of the column's permuted stream is stored
 *      at out[kk%64 + (kk/64)*128 + 64*(n%2) + K*2*(n/2)].
 * There is no nibble swap for int8.
 *
 * q    int8 [K][N] (the output of quantize_int8), 16-byte aligned.
 * out  int8 [N*K], 16-byte aligned (output).
 * Requires K % 64 == 0 and N % 2 == 0 (else W4_ERR_SHAPE); K == 0 or
 * N == 0 is a no-op.  Bit-exact.
 */
w4_status permute_int8(const void* q, void* out, int64_t K, int64_t N, void* stream);

/*
 * gemv_w8 -- GEMV / small-batch multiply by the int8 quantised matrix.
 *
 *   d[c][n] = sum_k q[k][n] * scale[n] * x[c][k],  0 <= c < C
 *
 * q      int8 [K][N] (quantize_int8's output), 16-byte aligned.
 * scale  fp32 [N], 16-byte aligned.
 * x      bf16 [C][K] row-major; d bf16 [C][N] row-major (output).
 * 1 <= C <= 8 (else W4_ERR_SHAPE); K == 0 gives d = 0.  fp32 accumulation,
 * one bf16 rounding; the tolerance is gemv_w4's (2e-3 * sum_k |w*x|).
 */
w4_status gemv_w8(const void* q, const float* scale, const void* x, void* d, int64_t N, int64_t K, int64_t C,
                  void* stream);

/*
 * gemm_w8 -- large-M bf16 x int8 GEMM over quantize_int8's matrix (the int8
 * counterpart of gemm_w4):
 *
 *   C[m][n] = scale[n] * sum_k A[m][k] * q[k][n]
 *
 * A      bf16 [M][K] row-major, 16-byte aligned.
 * q      int8 [K][N] row-major, 16-byte aligned.
 * scale  fp32 [N], 16-byte aligned.
 * C      bf16 [M][N] row-major (output), 16-byte aligned.
 * Requires K % 64 == 0 and N % 16 == 0 (else W4_ERR_SHAPE); K == 0 gives
 * C = 0.  bf16 tensor-core products (int8 is exact in bf16), fp32
 * accumulation, one bf16 rounding; the tolerance is gemm_w4's.
 */
w4_status gemm_w8(const void* A, const void* q, const float* scale, void* C, int64_t M, int64_t N, int64_t K,
                  void* stream);

/*
 * gemm_w4_permuted -- large-M bf16 x int4 GEMM that reads permute_int4's
 * output directly (the layout that page builds for the fast int4 -> 16-bit
 * dequant):
 *
 *   C[m][n] = scale[n] * sum_k A[m][k] * q[k][n]
 *
 * with q[k][n] the two's complement weights quantize_pack_int4 packed and
 * permute_int4 rearranged.
 * A         bf16 [M][K] row-major, 16-byte aligned.
 * permuted  N*K/2 bytes (permute_int4's output), 16-byte aligned.
 * scale     fp32 [N], 16-byte aligned.
 * C         bf16 [M][N] row-major (output), 16-byte aligned.
 * Requires K % 64 == 0 and N % 16 == 0 (else W4_ERR_SHAPE); K == 0 gives
 * C = 0.  Tolerance as gemm_w4.
 */
w4_status gemm_w4_permuted(const void* A, const void* permuted, const float* scale, void* C, int64_t M, int64_t N,
                           int64_t K, void* stream);

/* Shared memory available to one CTA on sm_103 (227 KB); gemv_w4a8 keeps all
 * of x there. */
#define W4_W4A8_MAX_SMEM 232448

/*
 * quantize_q8_1_pt -- x as block_q8_1 in the PT planes (page
 * "三值量化模型的无损压缩", section 3.1 "数据格式": 32 int8 values qs and the
 * halves (d, s) per block, s = d * sum qs).  For every 32-element block of
 * every vector:
 *   d  = max |x| / 127                            (IEEE fp32 division)
 *   qs = clamp(round(x / d), -127, 127)           (IEEE fp32 division, round
 *        half away from zero; a block whose maximum is 0 gets d = 0, qs = 0)
 *   stored: qs as int8, and d and the fp32 product d * sum qs as IEEE halves
 *   rounded to nearest even.
 * Layout of one vector (144 * K/128 bytes): element e of 128-element block i
 * is byte 16 * ((e / 16) * K/128 + i) + e % 16 (planes 0..7), and the four
 * (d, s) pairs of block i are the 16 bytes at 16 * (8 * K/128 + i) (plane 8;
 * pair j at +4j, d then s, little-endian).  Vectors follow each other.
 *
 * x   bf16 [C][K] row-major, 16-byte aligned.
 * pt  uint8 [C][144*K/128] (output), 16-byte aligned.
 * Requires K % 128 == 0 (else W4_ERR_SHAPE); C == 0 or K == 0 is a no-op.
 * NaN or Inf in x is undefined.  Bit-exact with the definition above.
 */
w4_status quantize_q8_1_pt(const void* x, void* pt, int64_t C, int64_t K, void* stream);

/*
 * gemv_w4a8 -- gemv_w4's int4 weights against activations in block_q8_1 /
 * PT form (same page, sections 3 and 3.1), with exact integer dot products
 * per 32-element block b and the zero point corrected through s:
 *
 *   d[c][r] = scale[r] * sum_b ( d_b * sum_{k in b} q[r][k] * qs[c][k]
 *                                - zero[r] * s_b )
 *
 * qweight  uint32 [N][K/8] as for gemv_w4 (nibble j of word i is k = 8i+j,
 *          unsigned), 16-byte aligned.
 * scale, zero  bf16 [N], 16-byte aligned.
 * pt       quantize_q8_1_pt's output for the C vectors, 16-byte aligned.
 * d        bf16 [C][N] row-major (output), 16-byte aligned.
 * Requires K % 128 == 0, 1 <= C <= 8 and C * K * 5/4 + 32 <= W4_W4A8_MAX_SMEM
 * (x is kept in shared memory; K <= 23168 at C = 8), else W4_ERR_SHAPE;
 * K == 0 gives d = 0.  fp32 accumulation of the exact dots; the tolerance is
 * 2e-3 * sum_k |(q - zero) * scale * d_b * qs| plus the bf16 rounding.
 */
w4_status gemv_w4a8(const void* qweight, const void* scale, const void* zero, const void* pt, void* d, int64_t N,
                    int64_t K, int64_t C, void* stream);

/*
 * mmvq_ptq1_0 -- the MMVQ product of ternary weights stored as PTQ1_0 blocks
 * with x in block_q8_1 / PT form (page "三值量化模型的无损压缩", section 2 for
 * the block, 3 for the product, 3.2 for where each trit sits):
 *
 *   d[c][r] = sum_b d_w(r, b) * sum_{j<4} d_x(c, b, j)
 *                             * sum_{e in q8_1 block j} t(r, 128 b + e) * qs(c, 128 b + e)
 *
 * A PTQ1_0 block (28 bytes) holds 128 trits and a half d_w: qs[24] with
 * five trits a byte (byte = sum_p (t_p + 1) 3^p), weight e < 80 at trit
 * e >> 4 of byte e & 15, weight 80 + e (e < 40) at trit e >> 3 of byte
 * 16 + (e & 7); qh[2], a little-endian 16-bit word whose 2-bit field j is
 * t + 1 of weight 120 + j; then d_w (little-endian half).
 *
 * blocks  N * K/128 blocks, row r's blocks back to back, rows back to back;
 *         16-byte aligned.
 * pt      quantize_q8_1_pt's output for the C vectors, 16-byte aligned.
 * d       fp32 [C][N] row-major (output), 16-byte aligned.
 * Requires K % 128 == 0, 1 <= C <= 8 and x within shared memory
 * (C * K * 5/4 <= W4_W4A8_MAX_SMEM, so K <= 23168 at C = 8), else
 * W4_ERR_SHAPE; K == 0 gives d = 0.  The integer
 * dots are exact; fp32 products and sums, within (K/128 + 5) * 2^-24 of
 * sum_k |w x| (2e-5 is the tested bound).
 */
w4_status mmvq_ptq1_0(const void* blocks, const void* pt, float* d, int64_t N, int64_t K, int64_t C, void* stream);

/*
 * mmvq_ptq1_1 -- mmvq_ptq1_0's product over the same weights packed as
 * PTQ1_1 superblocks (same page, section 2): eight consecutive blocks of a
 * row in 216 bytes,
 *   qs[192]        the eight blocks' qs bytes, block s at 24 s;
 *   qh[13]         the 64 tail trits, tail trit j of block s as base-3 digit
 *                  (8 s + j) mod 5 of byte (8 s + j) / 5; digit 4 of byte 12
 *                  is the free trit f;
 *   mantissa[8]    ten bits each, block s at bits 10 s .. 10 s + 9 of the
 *                  little-endian 80-bit string;
 *   exponents      one byte; the pattern index exponents + 256 f < 767 names
 *                  codebook entry [index], 767 the escape table entry of this
 *                  superblock (index r * ceil(K/1024) + sb).
 * Block s's d is the positive half with the pattern's exponent s and
 * mantissa s.  A row of K/128 blocks takes ceil(K/1024) superblocks; the
 * blocks past K (zero trits, d = 0) are not read.
 *
 * sblocks   N * ceil(K/1024) superblocks, row after row, 16-byte aligned.
 * codebook  uint8 [n_code][8] exponents (0 <= n_code <= 767).
 * esc_idx   int64 [n_esc] superblock indices, ascending; esc_patt uint8
 *           [n_esc][8] their exponents.
 * pt, d, C, K: as mmvq_ptq1_0 (the codebook takes 6136 bytes more shared
 * memory: K <= 22528 at C = 8).  All pointers 16-byte aligned; codebook / esc_* may be NULL when
 * n_code / n_esc is 0.  An index that names no entry records device error 2
 * (w4_device_error) and its blocks count as d = 0.
 */
w4_status mmvq_ptq1_1(const void* sblocks, const void* codebook, int64_t n_code, const void* esc_idx,
                      const void* esc_patt, int64_t n_esc, const void* pt, float* d, int64_t N, int64_t K, int64_t C,
                      void* stream);
/*
 * PTQ1_1 conversion (page "三值量化模型的无损压缩", section 2 "权重的无损压缩").
 * HOST functions: every pointer is host memory; nothing touches a GPU.
 *
 * A PTQ1_0 block (28 bytes) holds 128 trits: qs[24] five trits a byte
 * (byte = sum_p (t_p + 1) 3^p; weight e < 80 at trit e >> 4 of byte e & 15,
 * weight 80 + e at trit e >> 3 of byte 16 + (e & 7)), qh[2] a little-endian
 * word whose 2-bit field j is t + 1 of weight 120 + j, and the half d.
 * A PTQ1_1 superblock (216 bytes) holds eight consecutive blocks of a row:
 * qs[192] (block s at 24 s), qh[13] (tail trit j of block s as base-3
 * digit (8 s + j) mod 5 of byte (8 s + j) / 5; digit 4 of byte 12 is the
 * free trit f), eight 10-bit mantissas (block s at bits 10 s .. 10 s + 9 of
 * the little-endian 80-bit string at byte 205) and one exponents byte: the
 * pattern index exponents + 256 f names codebook entry [index] (< 767) or,
 * at 767, the escape-table entry of the superblock.  A row of K/128 blocks
 * takes ceil(K/1024) superblocks, the missing blocks of the last one being
 * zero trits with d = +0; superblock (r, sb) has index r * ceil(K/1024) + sb.
 *
 * ptq1_1_codebook -- the tensor's exponent patterns (eight 5-bit exponents of
 * a superblock's blocks) by descending count, ties in ascending order of the
 * pattern read as a 40-bit number with block 0's exponent most significant;
 * the first min(767, distinct) go to codebook (uint8 [767][8]) and their
 * number to *n_code.
 * blocks  N * K/128 PTQ1_0 blocks, row after row.  K % 128 == 0, else
 * W4_ERR_SHAPE.
 */
w4_status ptq1_1_codebook(const void* blocks, int64_t N, int64_t K, void* codebook, int64_t* n_code);

/*
 * ptq1_1_encode -- PTQ1_0 blocks -> PTQ1_1 superblocks (N * ceil(K/1024) *
 * 216 bytes) with the given codebook (uint8 [n_code][8], 0 <= n_code <=
 * 767; a repeated pattern resolves to its first entry).  A superblock whose
 * pattern is not in the codebook gets index 767 and an escape entry:
 * esc_idx (int64, ascending superblock indices) and esc_patt (uint8
 * [.][8]), at most max_esc of them (more: W4_ERR_SHAPE); *n_esc receives
 * their number.  W4_ERR_VALUE if a block has a negative d (PTQ1_1 keeps no
 * sign), a qs byte above 242 or a qh field of 3.
 */
w4_status ptq1_1_encode(const void* blocks, int64_t N, int64_t K, const void* codebook, int64_t n_code,
                        void* sblocks, void* esc_idx, void* esc_patt, int64_t max_esc, int64_t* n_esc);

#ifdef __cplusplus
}
#endif

#endif /* W4_H_ */
