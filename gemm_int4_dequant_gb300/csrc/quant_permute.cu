// quant_permute.cu -- weight-only int4 quantise + column pack, and the int4
// interleave permute (page "[PHI] add int4 weight only quant kernel, add int4
// weight only permute kernel": sections "int4量化kernel", "int4 permute
// kernel", "简单的位运算", "int4 row interval").
//
// Both kernels are HBM-bound byte movers.  Roofline bytes per element are
// stated next to each kernel.

#include "common.cuh"

namespace w4 {

// ---------------------------------------------------------------------------
// quantize_pack_int4
//
// One CTA owns a strip of QP_COLS columns over all K.  Pass 1 finds each
// column's max |W| (compared as bf16 bit patterns with the sign cleared,
// which orders non-negative floats exactly); pass 2 re-reads the strip,
// quantises with an IEEE fp32 division and round-half-away, and writes two
// rows per byte.  Algorithmic bytes: 2 B read per weight + 0.5 B written.
// ---------------------------------------------------------------------------

constexpr int QP_COLS = 32;                    // columns per strip
constexpr int QP_THREADS = 256;
constexpr int QP_CG = QP_COLS / 8;             // 16-byte column groups per strip
constexpr int QP_RL = QP_THREADS / QP_CG;      // row lanes

__device__ __forceinline__ uint32_t quant_nibble(uint32_t wbits, float s) {
    float w = bf16_bits_to_f32(wbits & 0xFFFFu);
    float r = (s == 0.0f) ? 0.0f : roundf(__fdiv_rn(w, s));
    r = fminf(fmaxf(r, -8.0f), 7.0f);
    return static_cast<uint32_t>(static_cast<int>(r)) & 0xFu;
}

template <bool VEC>
__global__ void __launch_bounds__(QP_THREADS)
quantize_pack_kernel(const uint16_t* __restrict__ W, uint8_t* __restrict__ packed,
                     float* __restrict__ scale, int64_t K, int64_t N) {
    __shared__ uint32_t red[QP_RL][QP_COLS + 1];
    __shared__ float s_scale[QP_COLS];
    const int cg = threadIdx.x % QP_CG;
    const int rl = threadIdx.x / QP_CG;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * QP_COLS + cg * 8;

    // pass 1: column max of |W| as bit patterns
    uint32_t amax[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) amax[j] = 0;
    if (VEC) {
        if (n0 < N) {
            for (int64_t k = rl; k < K; k += QP_RL) {
                uint4 v = ldg_stream_u4(W + k * N + n0);
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    amax[2 * j] = max(amax[2 * j], w[j] & 0x7FFFu);
                    amax[2 * j + 1] = max(amax[2 * j + 1], (w[j] >> 16) & 0x7FFFu);
                }
            }
        }
    } else {
        for (int64_t k = rl; k < K; k += QP_RL) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (n0 + j < N) amax[j] = max(amax[j], static_cast<uint32_t>(W[k * N + n0 + j]) & 0x7FFFu);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) red[rl][cg * 8 + j] = amax[j];
    __syncthreads();
    if (threadIdx.x < QP_COLS) {
        uint32_t m = 0;
        for (int i = 0; i < QP_RL; ++i) m = max(m, red[i][threadIdx.x]);
        float s = __fdiv_rn(bf16_bits_to_f32(m), 7.0f);
        s_scale[threadIdx.x] = s;
        int64_t col = static_cast<int64_t>(blockIdx.x) * QP_COLS + threadIdx.x;
        if (col < N) scale[col] = s;
    }
    __syncthreads();

    // pass 2: quantise two rows per byte
    float s[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = s_scale[cg * 8 + j];
    const int64_t Kp = K / 2;
    if (VEC) {
        if (n0 >= N) return;
        for (int64_t kp = rl; kp < Kp; kp += QP_RL) {
            uint4 a = ldg_stream_u4(W + (2 * kp) * N + n0);
            uint4 b = ldg_stream_u4(W + (2 * kp + 1) * N + n0);
            uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
            uint32_t out[2] = {0, 0};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint32_t ea = (j & 1) ? (wa[j / 2] >> 16) : wa[j / 2];
                uint32_t eb = (j & 1) ? (wb[j / 2] >> 16) : wb[j / 2];
                uint32_t byte = quant_nibble(ea, s[j]) | (quant_nibble(eb, s[j]) << 4);
                out[j / 4] |= byte << (8 * (j % 4));
            }
            *reinterpret_cast<uint2*>(packed + kp * N + n0) = make_uint2(out[0], out[1]);
        }
    } else {
        for (int64_t kp = rl; kp < Kp; kp += QP_RL) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (n0 + j >= N) break;
                uint32_t ea = W[(2 * kp) * N + n0 + j];
                uint32_t eb = W[(2 * kp + 1) * N + n0 + j];
                packed[kp * N + n0 + j] =
                    static_cast<uint8_t>(quant_nibble(ea, s[j]) | (quant_nibble(eb, s[j]) << 4));
            }
        }
    }
}

w4_status run_quantize_pack(const void* W, void* packed, float* scale, int64_t K, int64_t N,
                            cudaStream_t stream) {
    const int64_t strips = (N + QP_COLS - 1) / QP_COLS;
    if (strips > 0x7FFFFFFF) return W4_ERR_SHAPE;
    const bool vec = (N % 8) == 0;
    dim3 grid(static_cast<unsigned>(strips));
    if (vec)
        quantize_pack_kernel<true><<<grid, QP_THREADS, 0, stream>>>(
            static_cast<const uint16_t*>(W), static_cast<uint8_t*>(packed), scale, K, N);
    else
        quantize_pack_kernel<false><<<grid, QP_THREADS, 0, stream>>>(
            static_cast<const uint16_t*>(W), static_cast<uint8_t*>(packed), scale, K, N);
    return launch_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// permute_int4
//
// Tile = one 32-byte chunk j of the k-byte stream (rows 32j..32j+31 of the
// packed matrix) x PM_COLS columns.  The tile is staged in shared memory;
// each thread then owns one column's 32-byte chunk, applies the byte permute
// and nibble swap to its two 16-byte groups in registers and writes the
// chunk to its interleaved position, so a warp writes 8 runs of 128
// contiguous bytes.  Algorithmic bytes: 1 B read + 1 B written per byte.
// ---------------------------------------------------------------------------

constexpr int PM_COLS = 128;
constexpr int PM_THREADS = PM_COLS;

// One 16-byte group, words w[0..3] = bytes 0-3, 4-7, 8-11, 12-15.
// Byte permute: output word i holds bytes (i, 8+i, 4+i, 12+i), i.e. the
// destination of source byte t is 4*(t%4) + 2*((t/4)%2) + t/8.
// Nibble swap: in each output word (p0,p1,p2,p3) the low nibbles of p0,p2
// and of p1,p3 pair up into bytes 0 and 1, the high nibbles into bytes 2, 3.
__device__ __forceinline__ void permute_group16(const uint32_t (&w)[4], uint32_t (&o)[4]) {
    uint32_t a01 = __byte_perm(w[0], w[2], 0x5140);  // b0 b8 b1 b9
    uint32_t b01 = __byte_perm(w[1], w[3], 0x5140);  // b4 b12 b5 b13
    uint32_t a23 = __byte_perm(w[0], w[2], 0x7362);  // b2 b10 b3 b11
    uint32_t b23 = __byte_perm(w[1], w[3], 0x7362);  // b6 b14 b7 b15
    uint32_t p[4];
    p[0] = __byte_perm(a01, b01, 0x5410);            // b0 b8 b4 b12
    p[1] = __byte_perm(a01, b01, 0x7632);            // b1 b9 b5 b13
    p[2] = __byte_perm(a23, b23, 0x5410);            // b2 b10 b6 b14
    p[3] = __byte_perm(a23, b23, 0x7632);            // b3 b11 b7 b15
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t lo = p[i] & 0x0F0F0F0Fu;
        uint32_t hi = (p[i] >> 4) & 0x0F0F0F0Fu;
        o[i] = ((lo | (lo >> 12)) & 0xFFFFu) | ((hi | (hi >> 12)) << 16);
    }
}

template <bool VEC>
__global__ void __launch_bounds__(PM_THREADS)
permute_kernel(const uint8_t* __restrict__ packed, uint8_t* __restrict__ out, int64_t K, int64_t N) {
    __shared__ __align__(16) uint8_t tile[32][PM_COLS + 4];
    const int64_t total_k = K / 2;
    const int64_t chunk = blockIdx.x;                          // 32-byte chunk of the k stream
    const int64_t n_base = static_cast<int64_t>(blockIdx.y) * PM_COLS;
    const int64_t rem = N - n_base;
    const int ncols = rem < PM_COLS ? static_cast<int>(rem) : PM_COLS;

    // stage 32 rows x ncols bytes (ncols is a multiple of 4)
    for (int i = threadIdx.x; i < 32 * (PM_COLS / 4); i += PM_THREADS) {
        int r = i / (PM_COLS / 4), c4 = (i % (PM_COLS / 4)) * 4;
        if (c4 < ncols) {
            const uint8_t* src = packed + (chunk * 32 + r) * N + n_base + c4;
            uint32_t v = VEC ? *reinterpret_cast<const uint32_t*>(src)
                             : (uint32_t)src[0] | ((uint32_t)src[1] << 8) | ((uint32_t)src[2] << 16) |
                                   ((uint32_t)src[3] << 24);
            *reinterpret_cast<uint32_t*>(&tile[r][c4]) = v;
        }
    }
    __syncthreads();
    const int c = threadIdx.x;
    if (c >= ncols) return;
    const int64_t n = n_base + c;
    uint8_t* dst = out + total_k * 4 * (n / 4) + 128 * chunk + 32 * (n % 4);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t w[4], o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)tile[16 * h + 4 * i][c] | ((uint32_t)tile[16 * h + 4 * i + 1][c] << 8) |
                   ((uint32_t)tile[16 * h + 4 * i + 2][c] << 16) | ((uint32_t)tile[16 * h + 4 * i + 3][c] << 24);
        permute_group16(w, o);
        *reinterpret_cast<uint4*>(dst + 16 * h) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

w4_status run_permute(const void* packed, void* out, int64_t K, int64_t N, cudaStream_t stream) {
    const int64_t chunks = (K / 2) / 32;
    const int64_t col_tiles = (N + PM_COLS - 1) / PM_COLS;
    if (chunks > 0x7FFFFFFF || col_tiles > 65535) return W4_ERR_SHAPE;
    dim3 grid(static_cast<unsigned>(chunks), static_cast<unsigned>(col_tiles));
    const bool vec = (N % 4) == 0;  // always true given the shape rules; rows are 4-byte aligned
    if (vec)
        permute_kernel<true><<<grid, PM_THREADS, 0, stream>>>(static_cast<const uint8_t*>(packed),
                                                              static_cast<uint8_t*>(out), K, N);
    else
        permute_kernel<false><<<grid, PM_THREADS, 0, stream>>>(static_cast<const uint8_t*>(packed),
                                                               static_cast<uint8_t*>(out), K, N);
    return launch_status(cudaGetLastError());
}

}  // namespace w4
