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

// Tiled variant (N % 16 == 0): a CTA of 128 threads takes 64 rows x 128
// columns.  The tile comes in by coalesced 16-byte loads (row-major, 16-byte
// chunks of row r at chunk c ^ 2((r / 16) % 4), so that the reads below hit
// 32 different banks).  Thread (q, m) -- column quad q, 16-row group m --
// then builds, for each of its four columns, the 16 bytes of the column's
// group m in the line: output word w holds rows 2w, 2w+8, 2w+1, 2w+9 (the
// permute_kk order), so four 32-bit reads of those rows and a 4 x 4 byte
// transpose (eight byte permutes) give word w of all four columns.  The
// four adjacent m of a warp write 64 contiguous bytes of each line.
constexpr int P8_ROWS = 64, P8_COLS = 128, P8_THREADS = 128;

__global__ void __launch_bounds__(P8_THREADS)
permute_int8_tiled_kernel(const uint8_t* __restrict__ q, uint8_t* __restrict__ out, int64_t K, int64_t N) {
    __shared__ __align__(16) uint8_t tile[P8_ROWS * P8_COLS];
    const int64_t n_tiles = (N + P8_COLS - 1) / P8_COLS;
    const int64_t tn = blockIdx.x % n_tiles, j = blockIdx.x / n_tiles;   // column tile, 64-row line
    const int64_t c0 = tn * P8_COLS;
    const int valid = static_cast<int>(N - c0 < P8_COLS ? N - c0 : P8_COLS);   // multiple of 16
#pragma unroll
    for (int i = 0; i < P8_ROWS * P8_COLS / 16 / P8_THREADS; ++i) {
        const int t = threadIdx.x + i * P8_THREADS;
        const int r = t >> 3, c = t & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (16 * c < valid) v = ldg_stream_u4(q + (64 * j + r) * N + c0 + 16 * c);
        *reinterpret_cast<uint4*>(tile + r * P8_COLS + 16 * (c ^ (2 * ((r >> 4) & 3)))) = v;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int m = lane & 3, qd = (threadIdx.x >> 5) * 8 + (lane >> 2);   // 16-row group, column quad
    const int sw = 8 * m;                                                  // word swizzle of rows 16m..
    uint32_t col[4][4];   // [column of the quad][output word]
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const int rbase = 16 * m + 2 * w;
        const uint32_t* rw = reinterpret_cast<const uint32_t*>(tile);
        const uint32_t a = rw[(rbase) * 32 + (qd ^ sw)], b = rw[(rbase + 8) * 32 + (qd ^ sw)];
        const uint32_t c = rw[(rbase + 1) * 32 + (qd ^ sw)], d = rw[(rbase + 9) * 32 + (qd ^ sw)];
        const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
        const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
        col[0][w] = __byte_perm(t0, t2, 0x5410);
        col[1][w] = __byte_perm(t0, t2, 0x7632);
        col[2][w] = __byte_perm(t1, t3, 0x5410);
        col[3][w] = __byte_perm(t1, t3, 0x7632);
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
        const int nl = 4 * qd + cc;   // column within the tile
        if (nl >= valid) break;
        const int64_t n = c0 + nl;
        uint8_t* dst = out + K * 2 * (n / 2) + 128 * j + 64 * (n % 2) + 16 * m;
        *reinterpret_cast<uint4*>(dst) = make_uint4(col[cc][0], col[cc][1], col[cc][2], col[cc][3]);
    }
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

// ---------------------------------------------------------------------------
// Fast GEMV over q[K][N] (N % 16 == 0): a CTA takes a strip of 128 columns
// -- one 128-byte line of every row it reads -- and a K-slice; the S CTAs
// of a cluster split K and the partial sums meet in the first CTA's shared
// memory.  A thread loads COLS columns of a row at once (16 for C <= 4, 8
// above, to bound the accumulators); int8 -> fp32 is exact through the
// float 2^23 + (q + 128) built by a byte permute, minus 2^23 + 128.
// ---------------------------------------------------------------------------

constexpr int W8F_THREADS = 256;
constexpr int W8F_STRIP = 128;
constexpr int W8F_WARPS = W8F_THREADS / 32;

__device__ __forceinline__ float i8_to_f32(uint32_t wx, uint32_t j) {   // wx = w ^ 0x80808080
    return __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | j)) - 8388736.0f;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t map_cluster_u32(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

template <int COLS>
struct W8Vec;
template <>
struct W8Vec<16> {
    using T = uint4;
    static __device__ __forceinline__ T load(const int8_t* p) { return ldg_stream_u4(p); }
    static __device__ __forceinline__ T zero() { return make_uint4(0, 0, 0, 0); }
    static __device__ __forceinline__ uint32_t word(const T& v, int i) {
        return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
    }
};
template <>
struct W8Vec<8> {
    using T = uint2;
    static __device__ __forceinline__ T load(const int8_t* p) {
        return make_uint2(ldg_stream_u32(p), ldg_stream_u32(p + 4));
    }
    static __device__ __forceinline__ T zero() { return make_uint2(0, 0); }
    static __device__ __forceinline__ uint32_t word(const T& v, int i) { return i == 0 ? v.x : v.y; }
};

__host__ __device__ inline size_t w8f_xs_bytes(int C, int64_t Ks) { return (size_t(C) * Ks * 2 + 15) / 16 * 16; }
__host__ __device__ inline size_t w8f_smem_bytes(int C, int64_t Ks) {
    return w8f_xs_bytes(C, Ks) + size_t(W8F_WARPS) * C * W8F_STRIP * 4 + size_t(C) * W8F_STRIP * 4;
}

template <int C, int COLS, int U>
__global__ void __launch_bounds__(W8F_THREADS)
gemv_w8_fast_kernel(const int8_t* __restrict__ q, const float* __restrict__ scale,
                    const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ d, int64_t N, int64_t K,
                    int S) {
    constexpr int LPR = W8F_STRIP / COLS;   // lanes per row
    constexpr int RL = W8F_THREADS / LPR;   // rows the CTA reads at once
    using V = W8Vec<COLS>;
    extern __shared__ __align__(16) uint8_t smem[];
    const int rank = static_cast<int>(blockIdx.x % S);   // clusters are S consecutive CTAs
    const int64_t strip = blockIdx.x / S;
    const int64_t Ks = (K + S - 1) / S, k0 = rank * Ks, k1 = (k0 + Ks < K) ? k0 + Ks : K;
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);                 // [C][Ks]
    float* red = reinterpret_cast<float*>(smem + w8f_xs_bytes(C, Ks));          // [warp][C][128]
    float* sum = red + W8F_WARPS * C * W8F_STRIP;                               // [C][128]

    for (int64_t t = threadIdx.x; t < int64_t(C) * Ks; t += W8F_THREADS) {
        const int64_t c = t / Ks, kk = t % Ks;
        if (k0 + kk < k1) xs[t] = x[c * K + k0 + kk];
    }
    __syncthreads();

    const int lc = threadIdx.x % LPR, rl = threadIdx.x / LPR;
    const int64_t n0 = strip * W8F_STRIP + lc * COLS;
    const bool live = n0 < N;   // N % 16 == 0: a live thread's COLS columns all exist
    float acc[C][COLS];
#pragma unroll
    for (int c = 0; c < C; ++c)
#pragma unroll
        for (int j = 0; j < COLS; ++j) acc[c][j] = 0.f;

    for (int64_t kb = k0 + rl; kb < k1; kb += int64_t(RL) * U) {
        typename V::T w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = kb + int64_t(u) * RL;
            w[u] = (live && k < k1) ? V::load(q + k * N + n0) : V::zero();
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = kb + int64_t(u) * RL;
            if (k >= k1) break;
            float wf[COLS];
#pragma unroll
            for (int i = 0; i < COLS / 4; ++i) {
                const uint32_t wx = V::word(w[u], i) ^ 0x80808080u;
#pragma unroll
                for (int j = 0; j < 4; ++j) wf[4 * i + j] = i8_to_f32(wx, j);
            }
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const float xv = __bfloat162float(xs[c * Ks + (k - k0)]);
#pragma unroll
                for (int j = 0; j < COLS; ++j) acc[c][j] = fmaf(wf[j], xv, acc[c][j]);
            }
        }
    }
    // the warp's rows, then the CTA's warps, in a fixed order
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
#pragma unroll
    for (int c = 0; c < C; ++c)
#pragma unroll
        for (int j = 0; j < COLS; ++j) {
            float v = acc[c][j];
#pragma unroll
            for (int o = LPR; o < 32; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane < LPR) red[(warp * C + c) * W8F_STRIP + lc * COLS + j] = v;
        }
    __syncthreads();
    for (int o = threadIdx.x; o < C * W8F_STRIP; o += W8F_THREADS) {
        const int c = o / W8F_STRIP, col = o % W8F_STRIP;
        float v = 0.f;
#pragma unroll
        for (int wi = 0; wi < W8F_WARPS; ++wi) v += red[(wi * C + c) * W8F_STRIP + col];
        sum[o] = v;
    }
    // the cluster's K-slices meet in rank 0 (a hardware cluster barrier; the
    // second keeps every CTA's shared memory alive until rank 0 has read it)
    if (S > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    } else {
        __syncthreads();
    }
    if (rank == 0) {
        for (int o = threadIdx.x; o < C * W8F_STRIP; o += W8F_THREADS) {
            const int c = o / W8F_STRIP, col = o % W8F_STRIP;
            float v = sum[o];
            const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(sum + o));
            for (int r = 1; r < S; ++r) v += ld_cluster_f32(map_cluster_u32(local, r));
            const int64_t n = strip * W8F_STRIP + col;
            if (n < N) d[c * N + n] = __float2bfloat16_rn(scale[n] * v);
        }
    }
    if (S > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
}

template <int C>
w4_status launch_w8_fast(const void* q, const float* scale, const void* x, void* d, int64_t N, int64_t K,
                         cudaStream_t stream) {
    constexpr int COLS = C <= 4 ? 16 : 8;
    constexpr int U = C <= 2 ? 8 : 4;
    const int sms = sm_count();
    if (sms <= 0) return W4_ERR_CUDA;
    const int64_t strips = (N + W8F_STRIP - 1) / W8F_STRIP;
    // about two CTAs per SM; more K-slices if x would not fit shared memory
    int64_t S = (2 * int64_t(sms) + strips - 1) / strips;
    S = S < 1 ? 1 : S > 8 ? 8 : S;
    while (S < 8 && w8f_smem_bytes(C, (K + S - 1) / S) > size_t(W4_W4A8_MAX_SMEM)) ++S;
    const size_t smem = w8f_smem_bytes(C, (K + S - 1) / S);
    if (smem > size_t(W4_W4A8_MAX_SMEM) || strips * S > 0x7FFFFFFF) return W4_ERR_SHAPE;
    auto kern = gemv_w8_fast_kernel<C, COLS, U>;
    static int smem_set[64];
    if (ensure_smem_limit(kern, static_cast<int>(smem), smem_set) != cudaSuccess) return W4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(strips * S), 1, 1);
    cfg.blockDim = dim3(W8F_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_status(cudaLaunchKernelEx(&cfg, kern, static_cast<const int8_t*>(q), scale,
                                            static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(d), N,
                                            K, static_cast<int>(S)));
}

}  // namespace

// the single-read quantiser shared with quantize_pack_int4 (quant_permute.cu)
w4_status run_quantize_int8_single_read(const void* W, void* q, float* scale, int64_t K, int64_t N,
                                        cudaStream_t stream);

w4_status run_quantize_int8(const void* W, void* q, float* scale, int64_t K, int64_t N, cudaStream_t stream) {
    const w4_status st = run_quantize_int8_single_read(W, q, scale, K, N, stream);
    if (st != W4_ERR_SHAPE) return st;
    const int64_t strips = (N + Q8_COLS - 1) / Q8_COLS;
    if (strips > 0x7FFFFFFF) return W4_ERR_SHAPE;
    quantize_int8_kernel<<<static_cast<unsigned>(strips), Q8_COLS * Q8_LANES, 0, stream>>>(
        static_cast<const uint16_t*>(W), static_cast<int8_t*>(q), scale, K, N);
    return launch_status(cudaGetLastError());
}

w4_status run_permute_int8(const void* q, void* out, int64_t K, int64_t N, cudaStream_t stream) {
    if (N % 16 == 0) {
        const int64_t tiles = (N + P8_COLS - 1) / P8_COLS * (K / 64);
        if (tiles > 0x7FFFFFFF) return W4_ERR_SHAPE;
        if (tiles == 0) return W4_OK;
        permute_int8_tiled_kernel<<<static_cast<unsigned>(tiles), P8_THREADS, 0, stream>>>(
            static_cast<const uint8_t*>(q), static_cast<uint8_t*>(out), K, N);
        return launch_status(cudaGetLastError());
    }
    const int64_t work = (N / 2) * (K / 64);
    const int64_t blocks = (work + 127) / 128;
    if (blocks > 0x7FFFFFFF) return W4_ERR_SHAPE;
    permute_int8_kernel<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(static_cast<const uint8_t*>(q),
                                                                          static_cast<uint8_t*>(out), K, N);
    return launch_status(cudaGetLastError());
}

w4_status run_gemv_w8(const void* q, const float* scale, const void* x, void* d, int64_t N, int64_t K, int64_t C,
                      cudaStream_t stream) {
    if (N % 16 == 0) {
        switch (C) {
            case 1: return launch_w8_fast<1>(q, scale, x, d, N, K, stream);
            case 2: return launch_w8_fast<2>(q, scale, x, d, N, K, stream);
            case 3: return launch_w8_fast<3>(q, scale, x, d, N, K, stream);
            case 4: return launch_w8_fast<4>(q, scale, x, d, N, K, stream);
            case 5: return launch_w8_fast<5>(q, scale, x, d, N, K, stream);
            case 6: return launch_w8_fast<6>(q, scale, x, d, N, K, stream);
            case 7: return launch_w8_fast<7>(q, scale, x, d, N, K, stream);
            case 8: return launch_w8_fast<8>(q, scale, x, d, N, K, stream);
            default: return W4_ERR_SHAPE;
        }
    }
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
