/*
 * w4_oracle.c -- plain, slow, obviously-correct CPU oracle for the int4
 * weight-only hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library may include,
 * link or call this file; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, table, constant
 * or helper with the CUDA path.
 *
 * Every product is computed in IEEE double from the exact values of its
 * inputs (bf16 and fp32 convert to double exactly), so the only rounding
 * is the double accumulation itself.  The quantizer is the one place where
 * fp32 arithmetic is part of the definition (it decides an integer), and
 * there it is done in fp32, exactly as the reading below states.
 *
 * Sources (web pages on int4 weight-only quantisation, cited by page title
 * and section):
 *   [P1] "[PHI] add int4 weight only quant kernel, add int4 weight only
 *        permute kernel" (Paddle PR #64091): sections "int4量化kernel",
 *        "int4 permute kernel", "如何从int8 permute转换为int4 permute",
 *        "简单的位运算", "int4 row interval" (the last two also describe the
 *        int8 permute the int4 one is derived from).
 *   [P2] "怎样在安卓端利用 Vulkan 编写 4-bit 专用算子" (Vulkan 4-bit GEMV blog):
 *        section 1 "数据打包策略", section 2 "核心 GLSL 算子实现".
 *   [P3] "int4 gemm kernel" (pytorch/helion issue #508): the
 *        matmul_bf16_int4 example.
 *   [P4] "三值量化模型的无损压缩" (ternary compression blog): section 3 "MMVQ",
 *        the batched GEMV definition d[r,c] = sum_k W[r,k] x[c,k].
 *
 * Parity pins for every function live in tests/test_oracle_pins.py and
 * tests/test_oracle_ternary_pins.py; tests/test_oracle_mutants.py checks
 * that planted mistakes in this file fail them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element type codes for activations/scales/zeros. */
#define W4O_F32 0
#define W4O_BF16 1

int w4o_abi_version(void) { return 1; }

/* bf16 is the upper half of an IEEE binary32: widen by appending 16 zero
 * bits.  Exact. */
static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double load_elem(const void* base, int dtype, long i) {
    if (dtype == W4O_BF16) return (double)bf16_bits_to_float(((const uint16_t*)base)[i]);
    return (double)((const float*)base)[i];
}

/*
 * Fused dequant GEMV, batched.
 *
 * [P2 section 2]: one output per row; the row's K weights are stored as K/8
 * uint32 words, word i of row r at packed_weights[r*K/8 + i]; nibble j of a
 * word is (word >> 4j) & 0xF and holds weight k = 8i + j ([P2 section 1]:
 * packed = (w7<<28)|...|(w1<<4)|w0); the weight is dequantised as
 * (q - zero[r]) * scale[r] and multiplied by vec_in[8i + j].
 * [P4 section 3]: the batched form d[r,c] = sum_k W[r,k] x[c,k]; here x is
 * [C][K] row-major and the result is stored d[c*N + r].
 *
 * Rows [row_begin, row_end) are computed.  ref_abs (may be NULL) receives
 * sum_k |w * x| for each output, the denominator of the parity tolerance.
 */
void w4o_gemv(const uint32_t* packed_weights, const void* scales, const void* zeros,
              const void* x, int act_dtype, long N, long K, long C,
              long row_begin, long row_end, double* d, double* ref_abs) {
    long k_blocks = K / 8;
    for (long c = 0; c < C; ++c) {
        for (long row = row_begin; row < row_end; ++row) {
            double scale = load_elem(scales, act_dtype, row);
            double zero = load_elem(zeros, act_dtype, row);
            double sum = 0.0, abs_sum = 0.0;
            for (long i = 0; i < k_blocks; ++i) {
                uint32_t packed_val = packed_weights[row * k_blocks + i];
                for (int j = 0; j < 8; ++j) {
                    uint32_t val = (packed_val >> (j * 4)) & 0x0Fu;
                    double w = ((double)val - zero) * scale;
                    double xv = load_elem(x, act_dtype, c * K + i * 8 + j);
                    sum += xv * w;
                    abs_sum += fabs(xv * w);
                }
            }
            d[c * N + row] = sum;
            if (ref_abs) ref_abs[c * N + row] = abs_sum;
        }
    }
}

/*
 * Large-M dequant GEMM, evaluated at a list of output coordinates.
 *
 * [P3]: A is (M, K) bf16 row-major; B is the packed (K/2, N) int8 matrix
 * whose byte (kp, n) holds two int4 values along K: the low nibble
 * (b & 0x0F) is k = 2kp and the high nibble ((b >> 4) & 0x0F) is
 * k = 2kp + 1, both read as unsigned 0..15.  C[m, n] = sum_k A[m,k] *
 * B[k,n].  The per-column zero and scale dequantise each unpacked value as
 * (u - zero[n]) * scale[n] (the page's sketch has neither; the workload
 * definition supplies both, bf16).
 *
 * For t in [0, count): c[t] = C[m_idx[t], n_idx[t]], ref_abs[t] (may be
 * NULL) = sum_k |A * w|.
 */
void w4o_gemm_at(const uint16_t* A, const uint8_t* B, const uint16_t* scale,
                 const uint16_t* zero, long M, long N, long K, const long* m_idx,
                 const long* n_idx, long count, double* c, double* ref_abs) {
    (void)M;
    for (long t = 0; t < count; ++t) {
        long m = m_idx[t], n = n_idx[t];
        double s = (double)bf16_bits_to_float(scale[n]);
        double z = (double)bf16_bits_to_float(zero[n]);
        double acc = 0.0, abs_acc = 0.0;
        for (long kp = 0; kp < K / 2; ++kp) {
            uint8_t b = B[kp * N + n];
            uint32_t b_lo = b & 0x0Fu;         /* k = 2kp     */
            uint32_t b_hi = (b >> 4) & 0x0Fu;  /* k = 2kp + 1 */
            double a0 = (double)bf16_bits_to_float(A[m * K + 2 * kp]);
            double a1 = (double)bf16_bits_to_float(A[m * K + 2 * kp + 1]);
            double w0 = ((double)b_lo - z) * s;
            double w1 = ((double)b_hi - z) * s;
            acc += a0 * w0 + a1 * w1;
            abs_acc += fabs(a0 * w0) + fabs(a1 * w1);
        }
        c[t] = acc;
        if (ref_abs) ref_abs[t] = abs_acc;
    }
}

/*
 * Weight-only int4 quantisation and column pack.
 *
 * Workload definition (symmetric, per output column n of W[K][N]):
 *   scale[n] = max_k |W[k][n]| / 7           (fp32, IEEE division)
 *   q[k][n]  = clamp(round(W[k][n] / scale[n]), -8, 7)
 * with round = round half away from zero (C roundf) and the quotient an
 * IEEE fp32 division; a column of zeros has scale 0 and q = 0.
 * [P1 section "int4量化kernel"]: two int4 values are packed into one int8 by
 * taking an upper and a lower row, i.e. the pack runs along columns:
 * byte (k/2, n) holds rows k and k+1 of column n; the even row goes in the
 * low nibble.  Nibbles are two's complement (q & 0xF).
 */
void w4o_quantize_pack(const uint16_t* W, long K, long N, float* scale, uint8_t* packed) {
    for (long n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (long k = 0; k < K; ++k) {
            float a = fabsf(bf16_bits_to_float(W[k * N + n]));
            if (a > amax) amax = a;
        }
        float s = amax / 7.0f;
        scale[n] = s;
        for (long k = 0; k < K; k += 2) {
            int q[2];
            for (int h = 0; h < 2; ++h) {
                float w = bf16_bits_to_float(W[(k + h) * N + n]);
                float r = (s == 0.0f) ? 0.0f : roundf(w / s);
                if (r < -8.0f) r = -8.0f;
                if (r > 7.0f) r = 7.0f;
                q[h] = (int)r;
            }
            packed[(k / 2) * N + n] =
                (uint8_t)(((unsigned)q[0] & 0x0Fu) | (((unsigned)q[1] & 0x0Fu) << 4));
        }
    }
}

/*
 * GEMV over the quantiser's packed matrix (the operand the permute turns
 * into the fast-dequant layout).
 *
 * [P1 section "int4量化kernel"]: byte (k/2, n) of packed[K/2][N] holds rows
 * k (low nibble) and k+1 (high nibble) of column n as two's complement int4;
 * the column's weight is q[k][n] * scale[n] (symmetric per-column
 * quantisation, fp32 scale).  [P4 section 3]: the batched product
 * d[c][n] = sum_k W[k][n] x[c][k], x bf16 [C][K] row-major, stored d[c*N + n].
 * Columns [col_begin, col_end) are computed; ref_abs (may be NULL) receives
 * sum_k |w * x|.
 */
void w4o_gemv_packed(const uint8_t* packed, const float* scale, const uint16_t* x, long N, long K, long C,
                     long col_begin, long col_end, double* d, double* ref_abs) {
    for (long c = 0; c < C; ++c) {
        for (long n = col_begin; n < col_end; ++n) {
            double s = (double)scale[n];
            double sum = 0.0, abs_sum = 0.0;
            for (long k = 0; k < K; ++k) {
                unsigned byte = packed[(k / 2) * N + n];
                unsigned nib = (k % 2 == 0) ? (byte & 0x0Fu) : ((byte >> 4) & 0x0Fu);
                int q = (nib >= 8u) ? (int)nib - 16 : (int)nib;
                double w = (double)q * s;
                double xv = (double)bf16_bits_to_float(x[c * K + k]);
                sum += xv * w;
                abs_sum += fabs(xv * w);
            }
            d[c * N + n] = sum;
            if (ref_abs) ref_abs[c * N + n] = abs_sum;
        }
    }
}

/*
 * Large-M GEMM over the quantiser's packed matrix (the operand the permute
 * rearranges; [P3]'s C = A B with B the symmetric int4 weights):
 *   C[m][n] = sum_k A[m][k] * q[k][n] * scale[n]
 * with q[k][n] the two's complement nibble of byte (k/2, n) of packed[K/2][N]
 * (even k low) and scale fp32 [N]; at the coordinates (m_idx[t], n_idx[t]),
 * ref_abs (may be NULL) = sum_k |A * w|.
 */
void w4o_gemm_packed_at(const uint16_t* A, const uint8_t* packed, const float* scale, long M, long N, long K,
                        const long* m_idx, const long* n_idx, long count, double* c, double* ref_abs) {
    (void)M;
    for (long t = 0; t < count; ++t) {
        long m = m_idx[t], n = n_idx[t];
        double s = (double)scale[n];
        double acc = 0.0, abs_acc = 0.0;
        for (long k = 0; k < K; ++k) {
            unsigned byte = packed[(k / 2) * N + n];
            unsigned nib = (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);
            int q = (nib >= 8u) ? (int)nib - 16 : (int)nib;
            double a = (double)bf16_bits_to_float(A[m * K + k]);
            double w = (double)q * s;
            acc += a * w;
            abs_acc += fabs(a * w);
        }
        c[t] = acc;
        if (ref_abs) ref_abs[t] = abs_acc;
    }
}

/*
 * [P1 section "int4 permute kernel"]: destination of source byte t inside
 * each 16-byte group of a column's byte stream (the "coordinates" of the
 * mapping 0..15 -> 0 8 4 12 1 9 5 13 2 10 6 14 3 11 7 15).  Copied from the
 * page; tests/test_oracle_pins.py re-derives it from the int8 permute_kk by
 * the page's "% 8 * 2, add 1" steps.
 */
static const int k_permute_kk16[16] = {0, 4, 8, 12, 2, 6, 10, 14, 1, 5, 9, 13, 3, 7, 11, 15};

/*
 * int4 weight-only permute, [P1] steps in the page's order:
 *   1. byte permute: source byte kk of column n's stream moves to
 *      permute_kk = 16*(kk/16) + permute_kk16[kk%16]
 *      (section "int4 permute kernel");
 *   2. nibble swap: in each 4-byte group of the permuted stream, bytes 0/2
 *      and 1/3 exchange low and high nibbles (section "简单的位运算");
 *   3. row interleave: byte permute_kk of column n_id lands at
 *      permute_kk % 32 + permute_kk / 32 * 128 + 32 * (n_id % 4)
 *        + total_k * 4 * (n_id / 4)
 *      (section "int4 row interval"), with total_k = K/2 counted in packed
 *      bytes.
 * Input: packed[K/2][N] (the quantizer's output).  Output: N*K/2 bytes.
 * Requires K % 32 == 0 so that every 16-byte group is full; the
 * interleave assumes N % 4 == 0 and K/2 % 32 == 0.  Returns 0, or -1 if
 * the scratch stream cannot be allocated.
 */
int w4o_permute(const uint8_t* packed, long K, long N, uint8_t* out) {
    long total_k = K / 2;
    uint8_t* stream = (uint8_t*)malloc((size_t)(total_k > 0 ? total_k : 1));
    if (!stream) return -1;
    for (long n_id = 0; n_id < N; ++n_id) {
        /* step 1 */
        for (long kk = 0; kk < total_k; ++kk) {
            long permute_kk = (kk / 16) * 16 + k_permute_kk16[kk % 16];
            stream[permute_kk] = packed[kk * N + n_id];
        }
        /* step 2 */
        for (long g = 0; g < total_k; g += 4) {
            uint8_t b0 = stream[g], b1 = stream[g + 1], b2 = stream[g + 2], b3 = stream[g + 3];
            stream[g + 0] = (uint8_t)((b0 & 0x0F) | ((b2 & 0x0F) << 4));
            stream[g + 2] = (uint8_t)(((b0 >> 4) & 0x0F) | (b2 & 0xF0));
            stream[g + 1] = (uint8_t)((b1 & 0x0F) | ((b3 & 0x0F) << 4));
            stream[g + 3] = (uint8_t)(((b1 >> 4) & 0x0F) | (b3 & 0xF0));
        }
        /* step 3 */
        for (long permute_kk = 0; permute_kk < total_k; ++permute_kk) {
            long permute_index = permute_kk % 32 + permute_kk / 32 * 128 + 32 * (n_id % 4) +
                                 total_k * 4 * (n_id / 4);
            out[permute_index] = stream[permute_kk];
        }
    }
    free(stream);
    return 0;
}


/* ------------------------------------------------------------------------
 * int8 weight-only variant (the int8 counterpart of the path above).
 * ------------------------------------------------------------------------ */

/*
 * int8 weight-only quantisation: the int4 quantiser's definition with the
 * int8 range ([P1] quantises to int4 and describes the int8 permute its
 * int4 permute is derived from; the quantiser formula is the same reading):
 *   scale[n] = (float)max_k |W[k][n]| / 127.0f        (IEEE fp32 division)
 *   q[k][n]  = clamp(roundf(W[k][n] / scale[n]), -128, 127)
 * round half away from zero, an IEEE fp32 quotient, a column of zeros has
 * scale 0 and q = 0.  One weight per byte: q is int8 [K][N] row-major.
 */
void w4o_quantize_int8(const uint16_t* W, long K, long N, float* scale, int8_t* q) {
    for (long n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (long k = 0; k < K; ++k) {
            float a = fabsf(bf16_bits_to_float(W[k * N + n]));
            if (a > amax) amax = a;
        }
        float s = amax / 127.0f;
        scale[n] = s;
        for (long k = 0; k < K; ++k) {
            float w = bf16_bits_to_float(W[k * N + n]);
            float r = (s == 0.0f) ? 0.0f : roundf(w / s);
            if (r < -128.0f) r = -128.0f;
            if (r > 127.0f) r = 127.0f;
            q[k * N + n] = (int8_t)(int)r;
        }
    }
}

/*
 * [P1 section "如何从int8 permute转换为int4 permute"]: the int8 permute_kk,
 * the destination of source element t inside each group of 16 consecutive
 * elements of a column's stream.  Copied from the page;
 * tests/test_oracle_pins.py derives the int4 permute_kk from it by the
 * page's steps.
 */
static const int k_permute_kk16_int8[16] = {0, 2, 4, 6, 8, 10, 12, 14, 1, 3, 5, 7, 9, 11, 13, 15};

/*
 * int8 weight-only permute, [P1] in the page's order:
 *   1. element permute: source element kk of column n's stream (the K
 *      weights q[0..K-1][n]) moves to 16*(kk/16) + permute_kk_int8[kk%16];
 *   2. row interleave ([P1 section "int4 row interval"]: for int8 two
 *      adjacent rows -- output columns -- interleave every 64 elements):
 *      element permute_kk of column n lands at
 *      permute_kk % 64 + permute_kk / 64 * 128 + 64 * (n % 2) + total_k * 2 * (n / 2)
 *      with total_k = K (one element per byte).
 * There is no nibble swap for int8.  Input: q int8 [K][N].  Output: N*K
 * bytes.  Requires K % 64 == 0 and N % 2 == 0.  Returns 0, or -1 if the
 * scratch stream cannot be allocated.
 */
int w4o_permute_int8(const int8_t* q, long K, long N, uint8_t* out) {
    long total_k = K;
    uint8_t* stream = (uint8_t*)malloc((size_t)(total_k > 0 ? total_k : 1));
    if (!stream) return -1;
    for (long n_id = 0; n_id < N; ++n_id) {
        /* step 1 */
        for (long kk = 0; kk < total_k; ++kk) {
            long permute_kk = (kk / 16) * 16 + k_permute_kk16_int8[kk % 16];
            stream[permute_kk] = (uint8_t)q[kk * N + n_id];
        }
        /* step 2 */
        for (long permute_kk = 0; permute_kk < total_k; ++permute_kk) {
            long permute_index = permute_kk % 64 + permute_kk / 64 * 128 + 64 * (n_id % 2) +
                                 total_k * 2 * (n_id / 2);
            out[permute_index] = stream[permute_kk];
        }
    }
    free(stream);
    return 0;
}

/*
 * GEMV over the int8 quantised matrix ([P4 section 3] batched form, the
 * weight q[k][n] * scale[n] of the symmetric quantiser):
 *   d[c][n] = sum_k x[c][k] * q[k][n] * scale[n],  x bf16 [C][K], d[c*N + n].
 * Columns [col_begin, col_end) are computed; ref_abs (may be NULL) receives
 * sum_k |w * x|.
 */
void w4o_gemv_int8(const int8_t* q, const float* scale, const uint16_t* x, long N, long K, long C,
                   long col_begin, long col_end, double* d, double* ref_abs) {
    for (long c = 0; c < C; ++c) {
        for (long n = col_begin; n < col_end; ++n) {
            double s = (double)scale[n];
            double sum = 0.0, abs_sum = 0.0;
            for (long k = 0; k < K; ++k) {
                double w = (double)q[k * N + n] * s;
                double xv = (double)bf16_bits_to_float(x[c * K + k]);
                sum += xv * w;
                abs_sum += fabs(xv * w);
            }
            d[c * N + n] = sum;
            if (ref_abs) ref_abs[c * N + n] = abs_sum;
        }
    }
}

/*
 * Large-M GEMM over the int8 quantised matrix (the int8 counterpart of
 * w4o_gemm_at; [P3]'s C = A B with B the symmetric int8 weights):
 *   C[m][n] = sum_k A[m][k] * q[k][n] * scale[n],  A bf16 [M][K], q int8
 *   [K][N] row-major, scale fp32 [N],
 * evaluated at the coordinates (m_idx[t], n_idx[t]); ref_abs (may be NULL)
 * receives sum_k |A * w|.
 */
void w4o_gemm_int8_at(const uint16_t* A, const int8_t* q, const float* scale, long M, long N, long K,
                      const long* m_idx, const long* n_idx, long count, double* c, double* ref_abs) {
    (void)M;
    for (long t = 0; t < count; ++t) {
        long m = m_idx[t], n = n_idx[t];
        double s = (double)scale[n];
        double acc = 0.0, abs_acc = 0.0;
        for (long k = 0; k < K; ++k) {
            double a = (double)bf16_bits_to_float(A[m * K + k]);
            double w = (double)q[k * N + n] * s;
            acc += a * w;
            abs_acc += fabs(a * w);
        }
        c[t] = acc;
        if (ref_abs) ref_abs[t] = abs_acc;
    }
}

/* ------------------------------------------------------------------------
 * W4A8: int4 weights with activations quantised to block_q8_1 in the PT
 * plane layout ([P4] sections 3 and 3.1).
 * ------------------------------------------------------------------------ */

/* fp32 -> IEEE binary16 bits, round to nearest even (ggml_half). */
static uint16_t float_to_half_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag >= 0x7F800000u) return (uint16_t)(sign | (mag > 0x7F800000u ? 0x7E00u : 0x7C00u));
    /* |f| >= 65520 rounds to infinity */
    if (mag >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);
    if (mag < 0x38800000u) {
        /* subnormal half (or zero): value = m * 2^-24, m = round(|f| * 2^24) */
        double m = (double)f * (f < 0 ? -1.0 : 1.0) * 16777216.0;
        double fl = floor(m);
        double frac = m - fl;
        uint32_t r = (uint32_t)fl;
        if (frac > 0.5 || (frac == 0.5 && (r & 1u))) ++r;
        return (uint16_t)(sign | r);
    }
    /* normal: keep 10 mantissa bits, round to nearest even on the 13 dropped */
    uint32_t exp = ((mag >> 23) - 127 + 15);
    uint32_t man = mag & 0x7FFFFFu;
    uint32_t half = (exp << 10) | (man >> 13);
    uint32_t rest = man & 0x1FFFu;
    if (rest > 0x1000u || (rest == 0x1000u && (half & 1u))) ++half;   /* may carry into the exponent */
    return (uint16_t)(sign | half);
}

/* IEEE binary16 bits -> double (exact): exponent field 0 is m * 2^-24,
 * 31 is infinity (m == 0) or NaN, else (1024 + m) * 2^(e - 25). */
static double half_bits_to_double(uint16_t h) {
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 31) v = (m == 0) ? HUGE_VAL : NAN;
    else v = (e == 0) ? ldexp((double)m, -24) : ldexp((double)(m | 0x400), e - 25);
    return (h & 0x8000u) ? -v : v;
}

/* The two conversions over arrays, exported so that the pins can compare
 * them with an IEEE library conversion on chosen values (every tie). */
void w4o_float_to_half(const float* in, long n, uint16_t* out) {
    for (long i = 0; i < n; ++i) out[i] = float_to_half_bits(in[i]);
}

void w4o_half_to_double(const uint16_t* in, long n, double* out) {
    for (long i = 0; i < n; ++i) out[i] = half_bits_to_double(in[i]);
}

/*
 * [P4 section 3.1]: x as block_q8_1 -- 32 int8 values qs and a pair of
 * halves (d, s) per block, with s = d * sum_i qs_i.  The page gives the
 * struct, not the quantiser; the reading is the weight quantiser's:
 *   d  = max_i |x_i| / 127          (IEEE fp32 division)
 *   qs = clamp(roundf(x_i / d), -127, 127)   (d == 0: qs = 0)
 *   stored: half(d), half(d * sum_i qs_i) (fp32 product, each rounded to
 *   the nearest half).
 * PT layout ([P4] section 3.1, "排列方式称作 PT"): per vector of K elements
 * (K % 128 == 0) there are K/128 blocks of 128 (four q8_1 blocks each);
 * element e of 128-block i is the byte
 *   o = 16 * (floor(e / 16) * K/128 + i) + e % 16
 * (planes 0..7 of 16 bytes per block), and plane 8 holds each 128-block's
 * four (d, s) pairs: the 16 bytes at 16 * (8 * K/128 + i), pair j at +4j
 * (d then s, little-endian halves).  A vector takes 144 * K/128 bytes;
 * x is [C][K] bf16, pt is C vectors back to back.
 */
void w4o_quantize_q8_1_pt(const uint16_t* x, long C, long K, uint8_t* pt) {
    long bpr = K / 128;
    long vec_bytes = 144 * bpr;
    for (long c = 0; c < C; ++c) {
        uint8_t* v = pt + c * vec_bytes;
        for (long i = 0; i < bpr; ++i) {
            for (int j = 0; j < 4; ++j) {
                long k0 = i * 128 + 32 * j;
                float amax = 0.0f;
                for (int t = 0; t < 32; ++t) {
                    float a = fabsf(bf16_bits_to_float(x[c * K + k0 + t]));
                    if (a > amax) amax = a;
                }
                float d = amax / 127.0f;
                int sum = 0;
                for (int t = 0; t < 32; ++t) {
                    float xv = bf16_bits_to_float(x[c * K + k0 + t]);
                    float r = (d == 0.0f) ? 0.0f : roundf(xv / d);
                    if (r < -127.0f) r = -127.0f;
                    if (r > 127.0f) r = 127.0f;
                    int q = (int)r;
                    sum += q;
                    int e = 32 * j + t;
                    v[16 * ((e / 16) * bpr + i) + e % 16] = (uint8_t)(int8_t)q;
                }
                uint16_t dh = float_to_half_bits(d);
                uint16_t sh = float_to_half_bits(d * (float)sum);
                uint8_t* ds = v + 16 * (8 * bpr + i) + 4 * j;
                ds[0] = (uint8_t)(dh & 0xFF);
                ds[1] = (uint8_t)(dh >> 8);
                ds[2] = (uint8_t)(sh & 0xFF);
                ds[3] = (uint8_t)(sh >> 8);
            }
        }
    }
}

/*
 * W4A8 GEMV: the int4 weights of w4o_gemv ([P2] words, scale and zero per
 * row, bf16) against x in block_q8_1 / PT form.  Per q8_1 block b (32
 * elements) of row r:
 *   contribution = d_b * sum_{k in b} q[r][k] * qs[k]  -  zero[r] * s_b
 * ("correcting the zero through s": s_b = d_b * sum qs), and
 *   d[c][r] = scale[r] * sum_b contribution,
 * with d_b, s_b the stored halves; fp64 throughout (the integer dots are
 * exact).  ref_abs (may be NULL) receives sum_k |(q - zero) scale d_b qs_k|.
 */
void w4o_gemv_w4a8(const uint32_t* packed_weights, const uint16_t* scales, const uint16_t* zeros,
                   const uint8_t* pt, long N, long K, long C, long row_begin, long row_end, double* d,
                   double* ref_abs) {
    long bpr = K / 128;
    long vec_bytes = 144 * bpr;
    long k_words = K / 8;
    for (long c = 0; c < C; ++c) {
        const uint8_t* v = pt + c * vec_bytes;
        for (long row = row_begin; row < row_end; ++row) {
            double scale = (double)bf16_bits_to_float(scales[row]);
            double zero = (double)bf16_bits_to_float(zeros[row]);
            double total = 0.0, abs_total = 0.0;
            for (long i = 0; i < bpr; ++i) {
                for (int j = 0; j < 4; ++j) {
                    const uint8_t* ds = v + 16 * (8 * bpr + i) + 4 * j;
                    double db = half_bits_to_double((uint16_t)(ds[0] | (ds[1] << 8)));
                    double sb = half_bits_to_double((uint16_t)(ds[2] | (ds[3] << 8)));
                    long dot = 0;
                    for (int t = 0; t < 32; ++t) {
                        long k = i * 128 + 32 * j + t;
                        int e = 32 * j + t;
                        int qs = (int)(int8_t)v[16 * ((e / 16) * bpr + i) + e % 16];
                        unsigned q = (packed_weights[row * k_words + k / 8] >> (4 * (k % 8))) & 0xFu;
                        dot += (long)q * qs;
                        abs_total += fabs(((double)q - zero) * scale * db * qs);
                    }
                    total += db * (double)dot - zero * sb;
                }
            }
            d[c * N + row] = scale * total;
            if (ref_abs) ref_abs[c * N + row] = abs_total;
        }
    }
}

/* ------------------------------------------------------------------------
 * Ternary weights ([P4] sections 2, 3.1 and 3.2): PTQ1_0 blocks of 128
 * trits, the PTQ1_1 superblock that packs eight of them into 216 bytes, and
 * the MMVQ GEMV over either against x in block_q8_1 / PT form.
 *
 * Readings where the page is silent (each stated once, here):
 *  - a trit t in {-1, 0, +1} is stored as the digit u = t + 1 in {0, 1, 2};
 *  - a byte holding five trits is the base-3 number sum_p u_p 3^p, trit
 *    position p being the digit of weight 3^p;
 *  - PTQ1_0 (28 bytes): qs[24], qh[2], d (IEEE half, little-endian), in the
 *    struct's order; weight e < 80 is position e >> 4 of qs byte e & 15,
 *    weight 80 + e (e < 40) position e >> 3 of qs byte 16 + (e & 7) (the
 *    page's "byte e & 7" counted from the first byte after the 80-trit
 *    part), weight 120 + j the 2-bit field j of qh read as a little-endian
 *    16-bit word; the weight's value is d * t;
 *  - PTQ1_1 (216 bytes): qs[192] = the eight blocks' qs back to back (block
 *    s at 24 s); qh[13] holds the 64 tail trits, tail trit j of block s as
 *    digit (8 s + j) mod 5 of byte (8 s + j) / 5, and the 65th digit
 *    (position 4 of byte 12) is the free trit f; mantissa[8] are eight
 *    10-bit fields, field s at bits 10 s .. 10 s + 9 of the little-endian
 *    80-bit string; exponents is one byte.  The pattern index is
 *    exponents + 256 f, in [0, 768); an index below 767 names a codebook
 *    entry (eight 5-bit exponents), 767 sends the decoder to the tensor's
 *    escape table, keyed by the superblock's index r * SBPR + sb.  Block s's
 *    d is the positive half with exponent field E_s and mantissa M_s;
 *  - the codebook holds the tensor's most frequent exponent patterns, by
 *    descending count, ties in ascending order of the pattern read as the
 *    40-bit number with block 0's exponent most significant;
 *  - a row of K/128 blocks takes ceil(K/1024) superblocks; the blocks that
 *    pad the last one have every trit 0 and d = +0.
 * ------------------------------------------------------------------------ */

#define PTQ1_0_BYTES 28
#define PTQ1_1_BYTES 216
#define PTQ1_1_QH 192
#define PTQ1_1_MANT 205
#define PTQ1_1_EXP 215
#define PTQ1_1_ESCAPE 767

static const int k_pow3[5] = {1, 3, 9, 27, 81};

/* [P4 section 3.2]: where weight e of a PTQ1_0 block sits.  Returns the qs
 * byte and sets *pos to the trit position, or returns -1 for the tail
 * (qh) and sets *pos to the tail index. */
static int ptq1_0_place(int e, int* pos) {
    if (e < 80) { *pos = e >> 4; return e & 15; }
    if (e < 120) { *pos = (e - 80) >> 3; return 16 + ((e - 80) & 7); }
    *pos = e - 120;
    return -1;
}

static int trit_digit(uint8_t byte, int pos) { return (byte / k_pow3[pos]) % 3; }

/*
 * Pack ternary weights into PTQ1_0 blocks.  trits: int8 [N][K] in
 * {-1, 0, 1}; d: [N][K/128] half bit patterns; out: N * K/128 blocks of 28
 * bytes, row after row.  K % 128 == 0.  Returns 0, or -1 on a value
 * outside {-1, 0, 1}.
 */
int w4o_ptq1_0_pack(const int8_t* trits, const uint16_t* d, long N, long K, uint8_t* out) {
    long bpr = K / 128;
    for (long r = 0; r < N; ++r) {
        for (long b = 0; b < bpr; ++b) {
            uint8_t* blk = out + (r * bpr + b) * PTQ1_0_BYTES;
            memset(blk, 0, PTQ1_0_BYTES);
            unsigned qh = 0;
            for (int e = 0; e < 128; ++e) {
                int t = trits[r * K + b * 128 + e];
                if (t < -1 || t > 1) return -1;
                int pos, byte = ptq1_0_place(e, &pos);
                if (byte >= 0) blk[byte] = (uint8_t)(blk[byte] + (t + 1) * k_pow3[pos]);
                else qh |= (unsigned)(t + 1) << (2 * pos);
            }
            uint16_t h = d[r * bpr + b];
            blk[24] = (uint8_t)(qh & 0xFF);
            blk[25] = (uint8_t)(qh >> 8);
            blk[26] = (uint8_t)(h & 0xFF);
            blk[27] = (uint8_t)(h >> 8);
        }
    }
    return 0;
}

/* Decode one PTQ1_0 block into 128 trits and its half d. */
static void ptq1_0_decode(const uint8_t* blk, int8_t* t, uint16_t* d) {
    unsigned qh = (unsigned)blk[24] | ((unsigned)blk[25] << 8);
    for (int e = 0; e < 128; ++e) {
        int pos, byte = ptq1_0_place(e, &pos);
        int u = (byte >= 0) ? trit_digit(blk[byte], pos) : (int)((qh >> (2 * pos)) & 3u);
        t[e] = (int8_t)(u - 1);
    }
    *d = (uint16_t)(blk[26] | (blk[27] << 8));
}

/* PTQ1_0 blocks -> trits int8 [N][K] and d [N][K/128] (half bits). */
void w4o_ptq1_0_unpack(const uint8_t* blocks, long N, long K, int8_t* trits, uint16_t* d) {
    long bpr = K / 128;
    for (long r = 0; r < N; ++r)
        for (long b = 0; b < bpr; ++b)
            ptq1_0_decode(blocks + (r * bpr + b) * PTQ1_0_BYTES, trits + r * K + b * 128, d + r * bpr + b);
}

/* The exponent field of block b of row r, 0 for the padding past the row. */
static int block_exponent(const uint8_t* blocks, long bpr, long r, long b) {
    if (b >= bpr) return 0;
    const uint8_t* blk = blocks + (r * bpr + b) * PTQ1_0_BYTES;
    return (blk[27] >> 2) & 0x1F;
}

/* Superblock (r, sb)'s pattern as a 40-bit key, block 0's exponent on top. */
static uint64_t pattern_key(const uint8_t* blocks, long bpr, long r, long sb) {
    uint64_t key = 0;
    for (int s = 0; s < 8; ++s) key = (key << 5) | (uint64_t)block_exponent(blocks, bpr, r, 8 * sb + s);
    return key;
}

static void key_to_pattern(uint64_t key, uint8_t* p) {
    for (int s = 7; s >= 0; --s) { p[s] = (uint8_t)(key & 0x1F); key >>= 5; }
}

typedef struct { uint64_t key; long count; } pattern_count;

static int cmp_u64(const void* a, const void* b) {
    uint64_t x = *(const uint64_t*)a, y = *(const uint64_t*)b;
    return (x > y) - (x < y);
}

static int cmp_by_count(const void* a, const void* b) {
    const pattern_count* x = a;
    const pattern_count* y = b;
    if (x->count != y->count) return (x->count < y->count) - (x->count > y->count);
    return (x->key > y->key) - (x->key < y->key);
}

/*
 * Build the codebook of a tensor of PTQ1_0 blocks ([P4] section 2: eight
 * consecutive blocks' exponents take fewer than 768 patterns in practice).
 * codebook receives up to 767 patterns of eight exponents (uint8
 * [767][8]); returns how many, or -1 if memory runs out.
 */
long w4o_ptq1_1_codebook(const uint8_t* blocks, long N, long K, uint8_t* codebook) {
    long bpr = K / 128, sbpr = (bpr + 7) / 8, total = N * sbpr;
    uint64_t* keys = malloc((size_t)(total > 0 ? total : 1) * sizeof *keys);
    pattern_count* runs = malloc((size_t)(total > 0 ? total : 1) * sizeof *runs);
    if (!keys || !runs) { free(keys); free(runs); return -1; }
    for (long r = 0; r < N; ++r)
        for (long sb = 0; sb < sbpr; ++sb) keys[r * sbpr + sb] = pattern_key(blocks, bpr, r, sb);
    qsort(keys, (size_t)total, sizeof *keys, cmp_u64);
    long n_runs = 0;
    for (long i = 0; i < total; ++i) {
        if (n_runs > 0 && runs[n_runs - 1].key == keys[i]) ++runs[n_runs - 1].count;
        else { runs[n_runs].key = keys[i]; runs[n_runs].count = 1; ++n_runs; }
    }
    qsort(runs, (size_t)n_runs, sizeof *runs, cmp_by_count);
    long n_code = n_runs < PTQ1_1_ESCAPE ? n_runs : PTQ1_1_ESCAPE;
    for (long i = 0; i < n_code; ++i) key_to_pattern(runs[i].key, codebook + 8 * i);
    free(keys);
    free(runs);
    return n_code;
}

/*
 * PTQ1_0 blocks -> PTQ1_1 superblocks ([P4] section 2), with the codebook
 * from w4o_ptq1_1_codebook.  out: N * ceil(K/1024) superblocks of 216
 * bytes.  Superblocks whose pattern is not in the codebook get index 767
 * and an entry in the escape table: esc_idx (ascending superblock indices)
 * and esc_patt (their eight exponents), at most max_esc entries.  Returns
 * the number of escapes, -1 if a d is negative (PTQ1_1 stores no sign), or
 * -2 if the escape table is too small.
 */
long w4o_ptq1_1_encode(const uint8_t* blocks, long N, long K, const uint8_t* codebook, long n_code,
                       uint8_t* out, long* esc_idx, uint8_t* esc_patt, long max_esc) {
    long bpr = K / 128, sbpr = (bpr + 7) / 8, n_esc = 0;
    for (long r = 0; r < N; ++r) {
        for (long sb = 0; sb < sbpr; ++sb) {
            long g = r * sbpr + sb;
            uint8_t* o = out + g * PTQ1_1_BYTES;
            memset(o, 0, PTQ1_1_BYTES);
            uint8_t pattern[8];
            for (int s = 0; s < 8; ++s) {
                long b = 8 * sb + s;
                int8_t t[128];
                uint16_t h = 0;
                if (b < bpr) ptq1_0_decode(blocks + (r * bpr + b) * PTQ1_0_BYTES, t, &h);
                else memset(t, 0, sizeof t);
                if (h & 0x8000u) return -1;
                /* qs: the block's 24 bytes hold positions 0..119 exactly as in PTQ1_0 */
                if (b < bpr) memcpy(o + 24 * s, blocks + (r * bpr + b) * PTQ1_0_BYTES, 24);
                else memset(o + 24 * s, 1 + 3 + 9 + 27 + 81, 24);   /* every trit 0 */
                for (int j = 0; j < 8; ++j) {
                    int u = 8 * s + j;
                    o[PTQ1_1_QH + u / 5] = (uint8_t)(o[PTQ1_1_QH + u / 5] + (t[120 + j] + 1) * k_pow3[u % 5]);
                }
                unsigned m = h & 0x3FFu;
                for (int bit = 0; bit < 10; ++bit)
                    if (m & (1u << bit)) o[PTQ1_1_MANT + (10 * s + bit) / 8] |= (uint8_t)(1u << ((10 * s + bit) % 8));
                pattern[s] = (uint8_t)((h >> 10) & 0x1F);
            }
            long idx = PTQ1_1_ESCAPE;
            for (long i = 0; i < n_code; ++i)
                if (memcmp(codebook + 8 * i, pattern, 8) == 0) { idx = i; break; }
            if (idx == PTQ1_1_ESCAPE) {
                if (n_esc >= max_esc) return -2;
                esc_idx[n_esc] = g;
                memcpy(esc_patt + 8 * n_esc, pattern, 8);
                ++n_esc;
            }
            o[PTQ1_1_EXP] = (uint8_t)(idx % 256);
            o[PTQ1_1_QH + 12] = (uint8_t)(o[PTQ1_1_QH + 12] + (idx / 256) * k_pow3[4]);
        }
    }
    return n_esc;
}

/* Decode superblock g into eight blocks' trits (1024) and halves.  Returns
 * 0, or -1 if the index names no codebook entry or escape. */
static int ptq1_1_decode(const uint8_t* o, long g, const uint8_t* codebook, long n_code, const long* esc_idx,
                         const uint8_t* esc_patt, long n_esc, int8_t* t, uint16_t* d) {
    long idx = o[PTQ1_1_EXP] + 256L * trit_digit(o[PTQ1_1_QH + 12], 4);
    const uint8_t* pattern = NULL;
    if (idx < PTQ1_1_ESCAPE) {
        if (idx < n_code) pattern = codebook + 8 * idx;
    } else {
        for (long i = 0; i < n_esc; ++i)
            if (esc_idx[i] == g) { pattern = esc_patt + 8 * i; break; }
    }
    if (!pattern) return -1;
    for (int s = 0; s < 8; ++s) {
        for (int e = 0; e < 120; ++e) {
            int pos, byte = ptq1_0_place(e, &pos);
            t[128 * s + e] = (int8_t)(trit_digit(o[24 * s + byte], pos) - 1);
        }
        for (int j = 0; j < 8; ++j) {
            int u = 8 * s + j;
            t[128 * s + 120 + j] = (int8_t)(trit_digit(o[PTQ1_1_QH + u / 5], u % 5) - 1);
        }
        unsigned m = 0;
        for (int bit = 0; bit < 10; ++bit)
            if (o[PTQ1_1_MANT + (10 * s + bit) / 8] & (1u << ((10 * s + bit) % 8))) m |= 1u << bit;
        d[s] = (uint16_t)(((unsigned)pattern[s] << 10) | m);
    }
    return 0;
}

/* PTQ1_1 superblocks -> trits int8 [N][K] and d [N][K/128] (the padding
 * blocks past K are dropped).  Returns 0, or -1 on an unresolvable index. */
int w4o_ptq1_1_unpack(const uint8_t* sblocks, long N, long K, const uint8_t* codebook, long n_code,
                      const long* esc_idx, const uint8_t* esc_patt, long n_esc, int8_t* trits, uint16_t* d) {
    long bpr = K / 128, sbpr = (bpr + 7) / 8;
    int8_t t[1024];
    uint16_t h[8];
    for (long r = 0; r < N; ++r) {
        for (long sb = 0; sb < sbpr; ++sb) {
            long g = r * sbpr + sb;
            if (ptq1_1_decode(sblocks + g * PTQ1_1_BYTES, g, codebook, n_code, esc_idx, esc_patt, n_esc, t, h))
                return -1;
            for (int s = 0; s < 8 && 8 * sb + s < bpr; ++s) {
                long b = 8 * sb + s;
                memcpy(trits + r * K + b * 128, t + 128 * s, 128);
                d[r * bpr + b] = h[s];
            }
        }
    }
    return 0;
}

/*
 * The MMVQ product for one row given its trits and halves ([P4] section 3:
 * d[r,c] = sum_k W[r,k] x[c,k]); x is block_q8_1 in the PT layout.  Per
 * 32-element q8_1 block j of 128-block b:
 *   d_w(b) * d_x(b, j) * sum_{i<32} t_i qs_i
 * with the integer dot exact; fp64 throughout.
 */
static void mmvq_row(const int8_t* t, const uint16_t* dw, const uint8_t* v, long K, double* out, double* out_abs) {
    long bpr = K / 128;
    double total = 0.0, abs_total = 0.0;
    for (long b = 0; b < bpr; ++b) {
        double w = half_bits_to_double(dw[b]);
        for (int j = 0; j < 4; ++j) {
            const uint8_t* ds = v + 16 * (8 * bpr + b) + 4 * j;
            double dx = half_bits_to_double((uint16_t)(ds[0] | (ds[1] << 8)));
            long dot = 0, adot = 0;
            for (int i = 0; i < 32; ++i) {
                int e = 32 * j + i;
                int qs = (int)(int8_t)v[16 * ((e / 16) * bpr + b) + e % 16];
                dot += (long)t[128 * b + e] * qs;
                adot += labs((long)t[128 * b + e] * qs);
            }
            total += w * dx * (double)dot;
            abs_total += fabs(w * dx) * (double)adot;
        }
    }
    *out = total;
    *out_abs = abs_total;
}

/* MMVQ over PTQ1_0 blocks; pt: C vectors of 144 K/128 bytes; rows
 * [row_begin, row_end) of d[C][N] and ref_abs (may be NULL). */
void w4o_mmvq_ptq1_0(const uint8_t* blocks, const uint8_t* pt, long N, long K, long C, long row_begin, long row_end,
                     double* d, double* ref_abs) {
    long bpr = K / 128;
    int8_t* t = malloc((size_t)(K > 0 ? K : 1));
    uint16_t* dw = malloc((size_t)(bpr > 0 ? bpr : 1) * sizeof *dw);
    if (!t || !dw) { free(t); free(dw); return; }
    for (long row = row_begin; row < row_end; ++row) {
        for (long b = 0; b < bpr; ++b) ptq1_0_decode(blocks + (row * bpr + b) * PTQ1_0_BYTES, t + 128 * b, dw + b);
        for (long c = 0; c < C; ++c) {
            double v, a;
            mmvq_row(t, dw, pt + c * 144 * bpr, K, &v, &a);
            d[c * N + row] = v;
            if (ref_abs) ref_abs[c * N + row] = a;
        }
    }
    free(t);
    free(dw);
}

/* MMVQ over PTQ1_1 superblocks (decoded with the codebook and escape
 * table); as w4o_mmvq_ptq1_0 otherwise.  Returns 0, or -1 on an
 * unresolvable index. */
int w4o_mmvq_ptq1_1(const uint8_t* sblocks, const uint8_t* codebook, long n_code, const long* esc_idx,
                    const uint8_t* esc_patt, long n_esc, const uint8_t* pt, long N, long K, long C, long row_begin,
                    long row_end, double* d, double* ref_abs) {
    long bpr = K / 128, sbpr = (bpr + 7) / 8;
    int8_t* t = malloc((size_t)(sbpr > 0 ? sbpr : 1) * 1024);
    uint16_t* dw = malloc((size_t)(sbpr > 0 ? sbpr : 1) * 8 * sizeof *dw);
    if (!t || !dw) { free(t); free(dw); return -1; }
    int rc = 0;
    for (long row = row_begin; row < row_end && rc == 0; ++row) {
        for (long sb = 0; sb < sbpr; ++sb) {
            long g = row * sbpr + sb;
            if (ptq1_1_decode(sblocks + g * PTQ1_1_BYTES, g, codebook, n_code, esc_idx, esc_patt, n_esc,
                              t + 1024 * sb, dw + 8 * sb)) { rc = -1; break; }
        }
        if (rc) break;
        for (long c = 0; c < C; ++c) {
            double v, a;
            mmvq_row(t, dw, pt + c * 144 * bpr, K, &v, &a);
            d[c * N + row] = v;
            if (ref_abs) ref_abs[c * N + row] = a;
        }
    }
    free(t);
    free(dw);
    return rc;
}
