// int8.cu -- the int8 weight-only variant: per-column symmetric int8
// quantisation, the int8 interleave permute, and a GEMV over the quantised
// matrix (page "[PHI] add int4 weight only quant kernel, add int4 weight only
// permute kernel": section "如何从int8 permute转换为int4 permute" gives the
// int8 permute_kk, section "int4 row interval" the two-column interleave of
// 64 elements; the quantiser is the int4 one with the int8 range).
//
// First, plainly correct CUDA versions (bit-exact quantise and permute,
// fp32-accumulated GEMV); each is HBM-bound by nature and reads or writes
// its operands coalesced, but none has the TMA staging of the int4 kernels.

#include <cuda_bf16.h>

#include "common.cuh"

namespace w4 {

namespace {

constexpr int Q8_COLS = 32;    // columns per CTA (one warp-wide row segment)
constexpr int Q8_LANES = 8;    // row lanes per CTA

// q = clamp(round_half_away(w / s), -128, 127) with an IEEE fp32 quotient;
// s == 0 gives 0.
__device__ __forceinline__ int8_t quant8(float w, float s) {
    float r = (s == 0.0f) ? 0.0f : roundf(__fdiv_rn(w, s));
    r = fminf(fmaxf(r, -128.0f), 127.0f);
    return static_cast<int8_t>(static_cast<int>(r));
}

// One CTA per strip of 32 columns over all K: thread (lane c, row lane r)
// takes column n0 + c on rows r, r + 8, ...  Pass 1: max |W| per column
// (bf16 bit patterns with the sign cleared order non-negative values);
// pass 2: quantise.  Algorithmic bytes: 2 B read per weight (twice here) +
// 1 B written.
__global__ void __launch_bounds__(Q8_COLS * Q8_LANES)
quantize_int8_kernel(const uint16_t* __restrict__ W, int8_t* __restrict__ q, float* __restrict__ scale,
                     int64_t K, int64_t N) {
    __shared__ uint32_t red[Q8_LANES][Q8_COLS];
    __shared__ float s_col[Q8_COLS];
    const int c = threadIdx.x % Q8_COLS, r = threadIdx.x / Q8_COLS;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * Q8_COLS + c;
    const bool col_ok = n < N;
    uint32_t m = 0;
    if (col_ok)
        for (int64_t k = r; k < K; k += Q8_LANES) m = max(m, static_cast<uint32_t>(W[k * N + n]) & 0x7FFFu);
    red[r][c] = m;
    __syncthreads();
    if (r == 0) {
        uint32_t mm = 0;
        for (int i = 0; i < Q8_LANES; ++i) mm = max(mm, red[i][c]);
        const float s = __fdiv_rn(bf16_bits_to_f32(mm), 127.0f);
        s_col[c] = s;
        if (col_ok) scale[n] = s;
    }
    __syncthreads();
    if (!col_ok) return;
    const float s = s_col[c];
    for (int64_t k = r; k < K; k += Q8_LANES) q[k * N + n] = quant8(bf16_bits_to_f32(W[k * N + n]), s);
}

// Destination of source element t inside each group of 16 (the page's
// int8 permute_kk).
__device__ __forceinline__ int permute_kk16_int8(int t) { return t < 8 ? 2 * t : 2 * (t - 8) + 1; }

// Thread (p, j) builds the 128-byte line j of column pair p: columns 2p and
// 2p+1, rows 64j..64j+63.  Element (k, 2p + c) goes to byte
// 64c + 16*((k%64)/16) + permute_kk16_int8(k%16) of the line, and line j of
// pair p starts at K*2*p + 128*j (= P1's permute_index for int8).  Each row
// is one 2-byte load (the pair's two columns), so a warp (consecutive p)
// reads 64 contiguous bytes per row; the line is written as eight 16-byte
// stores.  Algorithmic bytes: 1 B read + 1 B written per weight.
__global__ void __launch_bounds__(128)
permute_int8_kernel(const uint8_t* __restrict__ q, uint8_t* __restrict__ out, int64_t K, int64_t N) {
    const int64_t pairs = N / 2, lines = K / 64;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= pairs * lines) return;
    const int64_t p = idx % pairs, j = idx / pairs;
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = 0;
#pragma unroll
    for (int kr = 0; kr < 64; ++kr) {
        const uint32_t two = *reinterpret_cast<const uint16_t*>(q + (64 * j + kr) * N + 2 * p);
        const int pos = 16 * (kr / 16) + permute_kk16_int8(kr % 16);   // compile-time after unrolling
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int b = 64 * c + pos;
            w[b / 4] |= ((two >> (8 * c)) & 0xFFu) << (8 * (b % 4));
        }
    }
    uint4* dst = reinterpret_cast<uint4*>(out + K * 2 * p + 128 * j);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// d[c][n] = bf16(scale[n] * sum_k q[k][n] * x[c][k]), fp32 accumulation.
// A CTA takes 32 columns; its 8 warps take every 8th row of K, so each warp
// reads 32 contiguous bytes of q per row and one broadcast x value per
// column of x; the 8 row lanes are added in a fixed order.
template <int C>
__global__ void __launch_bounds__(Q8_COLS * Q8_LANES)
gemv_w8_kernel(const int8_t* __restrict__ q, const float* __restrict__ scale, const __nv_bfloat16* __restrict__ x,
               __nv_bfloat16* __restrict__ d, int64_t N, int64_t K) {
    __shared__ float red[Q8_LANES][C][Q8_COLS];
    const int c0 = threadIdx.x % Q8_COLS, r = threadIdx.x / Q8_COLS;
    const int64_t n = static_cast<int64_t>(blockIdx.x) * Q8_COLS + c0;
    const bool col_ok = n < N;
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    if (col_ok) {
#pragma unroll 4
        for (int64_t k = r; k < K; k += Q8_LANES) {
            const float w = static_cast<float>(q[k * N + n]);
#pragma unroll
            for (int c = 0; c < C; ++c) acc[c] = fmaf(w, __bfloat162float(x[c * K + k]), acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) red[r][c][c0] = acc[c];
    __syncthreads();
    if (r == 0 && col_ok) {
        const float s = scale[n];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float v = 0.f;
            for (int i = 0; i < Q8_LANES; ++i) v += red[i][c][c0];
            d[c * N + n] = __float2bfloat16_rn(s * v);
        }
    }
}

}  // namespace

w4_status run_quantize_int8(const void* W, void* q, float* scale, int64_t K, int64_t N, cudaStream_t stream) {
    const int64_t strips = (N + Q8_COLS - 1) / Q8_COLS;
    if (strips > 0x7FFFFFFF) return W4_ERR_SHAPE;
    quantize_int8_kernel<<<static_cast<unsigned>(strips), Q8_COLS * Q8_LANES, 0, stream>>>(
        static_cast<const uint16_t*>(W), static_cast<int8_t*>(q), scale, K, N);
    return launch_status(cudaGetLastError());
}

w4_status run_permute_int8(const void* q, void* out, int64_t K, int64_t N, cudaStream_t stream) {
    const int64_t work = (N / 2) * (K / 64);
    const int64_t blocks = (work + 127) / 128;
    if (blocks > 0x7FFFFFFF) return W4_ERR_SHAPE;
    permute_int8_kernel<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(static_cast<const uint8_t*>(q),
                                                                          static_cast<uint8_t*>(out), K, N);
    return launch_status(cudaGetLastError());
}

w4_status run_gemv_w8(const void* q, const float* scale, const void* x, void* d, int64_t N, int64_t K, int64_t C,
                      cudaStream_t stream) {
    const int64_t blocks = (N + Q8_COLS - 1) / Q8_COLS;
    if (blocks > 0x7FFFFFFF) return W4_ERR_SHAPE;
    const dim3 grid(static_cast<unsigned>(blocks));
    const auto* qq = static_cast<const int8_t*>(q);
    const auto* xx = static_cast<const __nv_bfloat16*>(x);
    auto* dd = static_cast<__nv_bfloat16*>(d);
    switch (C) {
        case 1: gemv_w8_kernel<1><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 2: gemv_w8_kernel<2><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 3: gemv_w8_kernel<3><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 4: gemv_w8_kernel<4><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 5: gemv_w8_kernel<5><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 6: gemv_w8_kernel<6><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 7: gemv_w8_kernel<7><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        case 8: gemv_w8_kernel<8><<<grid, Q8_COLS * Q8_LANES, 0, stream>>>(qq, scale, xx, dd, N, K); break;
        default: return W4_ERR_SHAPE;
    }
    return launch_status(cudaGetLastError());
}

}  // namespace w4
