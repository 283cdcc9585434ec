// gemv.cu -- fused dequant GEMV / small-batch multiply on the CUDA cores.
//
//   d[c][r] = sum_k (q[r][k] - zero[r]) * scale[r] * x[c][k]
//
// (page "怎样在安卓端利用 Vulkan 编写 4-bit 专用算子", sections 1-2: uint32 words
// of eight nibbles, w0 in the low bits, dequant (q - zero) * scale inside the
// dot loop; batched form from "三值量化模型的无损压缩", section 3 "MMVQ").
//
// Design (GB300): the op is HBM-bound (0.5 B of weight per multiply-add at
// C = 1), so the kernel streams the packed words with 16-byte non-allocating
// loads, stages x once per CTA in shared memory as fp32, converts nibbles to
// exact fp32 with the IEEE "magic number" trick (OR the nibble into the
// mantissa of 2^23, then one FMA by a power of two removes the offset, the
// nibble's bit position and the zero point's integer part zi: q - zi comes
// out exact) and accumulates in fp32.  A weight equal to an integer zero
// point contributes exactly nothing; only a fractional rest is folded out
// of the k-sum:  sum_k (q - z) x = sum_k (q - zi) x - (z - zi) sum_k x.
// K is split across the CTAs of a thread-block cluster when x does not fit
// in shared memory; the partial sums are reduced through distributed shared
// memory, so no scratch buffer in global memory is needed.

#include <cooperative_groups.h>

#include "common.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace w4 {

constexpr int GV_THREADS = 256;
constexpr int GV_WARPS = GV_THREADS / 32;
constexpr int GV_KL = 8;                     // lanes along K per row
constexpr int GV_RL = 32 / GV_KL;            // row lanes per warp
constexpr int GV_RT = 2;                     // rows per lane
constexpr int GV_TILE = GV_RL * GV_RT;       // rows per warp tile
constexpr int GV_ROWS = GV_WARPS * GV_TILE;  // rows per CTA

// shared-memory offset of local k index i: 4 floats of padding after every
// 32, so the 8 K-lanes of a warp reading 32 consecutive floats each hit
// distinct banks.
__device__ __forceinline__ int xpad(int i) { return i + (i >> 5) * 4; }
__host__ __device__ constexpr int xpad_len(int n) { return n + ((n + 31) / 32) * 4 + 4; }

// The five offsets a row's nibbles are reduced by: -(2^(23-4j) + zi) for
// j = 0..4, zi = zint(z) (every one exact in fp32).
struct ZeroOffsets {
    float o[5];
};
__device__ __forceinline__ ZeroOffsets zero_offsets(int zi) {
    ZeroOffsets z;
    const float zf = static_cast<float>(zi);
    z.o[0] = -(8388608.0f + zf);
    z.o[1] = -(524288.0f + zf);
    z.o[2] = -(32768.0f + zf);
    z.o[3] = -(2048.0f + zf);
    z.o[4] = -(128.0f + zf);
    return z;
}

// Eight nibbles of a word -> eight exact floats q - zi: nibble j ORed into
// the mantissa of 2^23 is 2^23 + 2^(4j) q; scaled by 2^-4j (exact) it is
// 2^(23-4j) + q, and the offset leaves q - zi (a single rounding of an
// exactly representable result).  Nibbles 5..7 come from the word shifted
// by 12, reusing the offsets of positions 2..4.
__device__ __forceinline__ void nibbles_to_f32(uint32_t v, const ZeroOffsets& z, float (&q)[8]) {
    const uint32_t M = 0x4B000000u;  // 2^23
    const uint32_t h = v >> 12;
    q[0] = __uint_as_float((v & 0x0000Fu) | M) + z.o[0];
    q[1] = fmaf(__uint_as_float((v & 0x000F0u) | M), 0.0625f, z.o[1]);
    q[2] = fmaf(__uint_as_float((v & 0x00F00u) | M), 0.00390625f, z.o[2]);
    q[3] = fmaf(__uint_as_float((v & 0x0F000u) | M), 0.000244140625f, z.o[3]);
    q[4] = fmaf(__uint_as_float((v & 0xF0000u) | M), 0.0000152587890625f, z.o[4]);
    q[5] = fmaf(__uint_as_float((h & 0x00F00u) | M), 0.00390625f, z.o[2]);
    q[6] = fmaf(__uint_as_float((h & 0x0F000u) | M), 0.000244140625f, z.o[3]);
    q[7] = fmaf(__uint_as_float((h & 0xF0000u) | M), 0.0000152587890625f, z.o[4]);
}

template <int C>
__device__ __forceinline__ void word_dot(uint32_t v, const ZeroOffsets& z, const float (&xv)[C][8],
                                         float (&acc)[C]) {
    float q[8];
    nibbles_to_f32(v, z, q);
#pragma unroll
    for (int c = 0; c < C; ++c)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[c] = fmaf(q[j], xv[c][j], acc[c]);
}

template <int C>
__device__ __forceinline__ void load_x8(const float* xs, int xs_stride, int off, float (&xv)[C][8]) {
#pragma unroll
    for (int c = 0; c < C; ++c) {
        float4 a = *reinterpret_cast<const float4*>(xs + c * xs_stride + off);
        float4 b = *reinterpret_cast<const float4*>(xs + c * xs_stride + off + 4);
        xv[c][0] = a.x; xv[c][1] = a.y; xv[c][2] = a.z; xv[c][3] = a.w;
        xv[c][4] = b.x; xv[c][5] = b.y; xv[c][6] = b.z; xv[c][7] = b.w;
    }
}

// grid = (S, ceil(N / GV_ROWS)); cluster = (S, 1, 1) when S > 1.
// blockIdx.x = K-slice = rank in the cluster.  VEC: K % 32 == 0, lanes load
// 16-byte groups of four words; otherwise lanes load single words.
template <typename T, int C, bool VEC>
__global__ void __launch_bounds__(GV_THREADS)
gemv_ffma_kernel(const uint32_t* __restrict__ qw, const T* __restrict__ scale, const T* __restrict__ zero,
                 const T* __restrict__ x, T* __restrict__ d, int N, int K, int kslice, int xs_stride, int S) {
    extern __shared__ __align__(16) float smem[];
    float* xs = smem;                               // [C][xs_stride]
    float* part = xs + C * xs_stride;               // [GV_ROWS][C]
    float* xsum = part + GV_ROWS * C;               // [C]

    const int ks = blockIdx.x;
    const int row0 = blockIdx.y * GV_ROWS;
    const int k0 = ks * kslice;
    const int k1 = min(K, k0 + kslice);
    const int klen = max(0, k1 - k0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // stage x[:, k0:k1] as fp32 and its per-row sums
    for (int c = 0; c < C; ++c)
        for (int i = tid; i < klen; i += GV_THREADS)
            xs[c * xs_stride + xpad(i)] = to_f32<T>(x[static_cast<int64_t>(c) * K + k0 + i]);
    __syncthreads();
    if (warp < C) {
        float sacc = 0.f;
        for (int i = lane; i < klen; i += 32) sacc += xs[warp * xs_stride + xpad(i)];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, o);
        if (lane == 0) xsum[warp] = sacc;
    }
    __syncthreads();

    const int kl = lane % GV_KL, rl = lane / GV_KL;
    const int rows_here = min(GV_ROWS, N - row0);
    for (int tile = warp; tile * GV_TILE < rows_here; tile += GV_WARPS) {
        int lrow[GV_RT];
        bool valid[GV_RT];
        const uint32_t* rp[GV_RT];
        float zrow[GV_RT];
        ZeroOffsets zo[GV_RT];
#pragma unroll
        for (int t = 0; t < GV_RT; ++t) {
            lrow[t] = tile * GV_TILE + rl + GV_RL * t;
            valid[t] = lrow[t] < rows_here;
            rp[t] = qw + static_cast<int64_t>(row0 + (valid[t] ? lrow[t] : 0)) * (K / 8);
            zrow[t] = valid[t] ? to_f32<T>(zero[row0 + lrow[t]]) : 0.0f;
            zo[t] = zero_offsets(ptx::zint(zrow[t]));
        }
        float acc[GV_RT][C];
#pragma unroll
        for (int t = 0; t < GV_RT; ++t)
#pragma unroll
            for (int c = 0; c < C; ++c) acc[t][c] = 0.f;

        if (VEC) {
            const int u0 = k0 / 32, u1 = k1 / 32;
            int u = u0 + kl;
            uint4 cur[GV_RT];
#pragma unroll
            for (int t = 0; t < GV_RT; ++t)
                cur[t] = (valid[t] && u < u1) ? ldg_stream_u4(rp[t] + 4 * u) : make_uint4(0, 0, 0, 0);
            for (; u < u1; u += GV_KL) {
                uint4 nxt[GV_RT];
                const int un = u + GV_KL;
#pragma unroll
                for (int t = 0; t < GV_RT; ++t)
                    nxt[t] = (valid[t] && un < u1) ? ldg_stream_u4(rp[t] + 4 * un) : make_uint4(0, 0, 0, 0);
                const int off = (u - u0) * 36;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float xv[C][8];
                    load_x8<C>(xs, xs_stride, off + 8 * w, xv);
#pragma unroll
                    for (int t = 0; t < GV_RT; ++t) {
                        uint32_t v = w == 0 ? cur[t].x : w == 1 ? cur[t].y : w == 2 ? cur[t].z : cur[t].w;
                        word_dot<C>(v, zo[t], xv, acc[t]);
                    }
                }
#pragma unroll
                for (int t = 0; t < GV_RT; ++t) cur[t] = nxt[t];
            }
        } else {
            const int w0 = k0 / 8, w1 = k1 / 8;
            for (int wi = w0 + kl; wi < w1; wi += GV_KL) {
                uint32_t v[GV_RT];
#pragma unroll
                for (int t = 0; t < GV_RT; ++t) v[t] = valid[t] ? ldg_stream_u32(rp[t] + wi) : 0u;
                float xv[C][8];
                load_x8<C>(xs, xs_stride, xpad((wi - w0) * 8), xv);
#pragma unroll
                for (int t = 0; t < GV_RT; ++t) word_dot<C>(v[t], zo[t], xv, acc[t]);
            }
        }
        // reduce across the K lanes of each row
#pragma unroll
        for (int t = 0; t < GV_RT; ++t)
#pragma unroll
            for (int c = 0; c < C; ++c)
#pragma unroll
                for (int o = 1; o < GV_KL; o <<= 1) acc[t][c] += __shfl_xor_sync(0xffffffffu, acc[t][c], o);
        if (kl == 0) {
#pragma unroll
            for (int t = 0; t < GV_RT; ++t) {
                if (!valid[t]) continue;
                const float zf = zrow[t] - static_cast<float>(ptx::zint(zrow[t]));   // fractional rest
#pragma unroll
                for (int c = 0; c < C; ++c) part[lrow[t] * C + c] = fmaf(-zf, xsum[c], acc[t][c]);
            }
        }
    }
    __syncthreads();

    cg::cluster_group cluster = cg::this_cluster();
    if (S > 1) cluster.sync();
    // rank ks reduces rows ks, ks + S, ... of this CTA's row block
    for (int i = ks + S * tid; i < rows_here; i += S * GV_THREADS) {
        const float s = to_f32<T>(scale[row0 + i]);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float sum = 0.f;
            for (int r = 0; r < S; ++r) {
                const float* p = (S > 1) ? cluster.map_shared_rank(part, r) : part;
                sum += p[i * C + c];
            }
            d[static_cast<int64_t>(c) * N + row0 + i] = from_f32<T>(s * sum);
        }
    }
    if (S > 1) cluster.sync();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

constexpr int kXsBudgetBytes = 96 * 1024;

struct GemvPlan {
    int S;          // K-slices (cluster size)
    int kslice;     // k per slice
    int xs_stride;  // padded floats per x row in shared memory
    size_t smem;
};

GemvPlan plan_gemv(int K, int C, bool vec) {
    const int gran = vec ? 32 : 8;
    GemvPlan p{1, 0, 0, 0};
    for (int S = 1; S <= 8; S *= 2) {
        int ks = (K + S - 1) / S;
        ks = (ks + gran - 1) / gran * gran;
        int stride = xpad_len(ks);
        size_t bytes = (static_cast<size_t>(C) * stride + GV_ROWS * C + C) * sizeof(float);
        p = GemvPlan{S, ks, stride, bytes};
        if (bytes <= kXsBudgetBytes) break;
    }
    return p;
}

template <typename T, int C, bool VEC>
w4_status launch_gemv_t(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N, int K,
                        cudaStream_t stream) {
    const GemvPlan p = plan_gemv(K, C, VEC);
    auto kern = gemv_ffma_kernel<T, C, VEC>;
    static int smem_set[64];
    cudaError_t e = ensure_smem_limit(kern, static_cast<int>(p.smem), smem_set);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.S, (N + GV_ROWS - 1) / GV_ROWS, 1);
    cfg.blockDim = dim3(GV_THREADS, 1, 1);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint32_t*>(qw), static_cast<const T*>(scale),
                           static_cast<const T*>(zero), static_cast<const T*>(x), static_cast<T*>(d), N, K,
                           p.kslice, p.xs_stride, p.S);
    return launch_status(e);
}

template <typename T, bool VEC>
w4_status dispatch_c(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N, int K,
                     int C, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_gemv_t<T, 1, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 2: return launch_gemv_t<T, 2, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 3: return launch_gemv_t<T, 3, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 4: return launch_gemv_t<T, 4, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 5: return launch_gemv_t<T, 5, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 6: return launch_gemv_t<T, 6, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 7: return launch_gemv_t<T, 7, VEC>(qw, scale, zero, x, d, N, K, stream);
        case 8: return launch_gemv_t<T, 8, VEC>(qw, scale, zero, x, d, N, K, stream);
        default: return W4_ERR_SHAPE;
    }
}

}  // namespace

w4_status run_gemv_tma(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N, int K,
                       int C, cudaStream_t stream);

w4_status run_gemv(const void* qw, const void* scale, const void* zero, const void* x, void* d, int64_t N,
                   int64_t K, int64_t C, w4_dtype dtype, cudaStream_t stream) {
    if (N > (1 << 30) || K > (1 << 30) || (N + GV_ROWS - 1) / GV_ROWS > 65535) return W4_ERR_SHAPE;
    const bool vec = (K % 32) == 0;
    const int n = static_cast<int>(N), k = static_cast<int>(K), c = static_cast<int>(C);
    // bf16 with 16-byte aligned rows: tensor-core MMA path; otherwise the
    // CUDA-core path (fp32 inputs need fp32 products; odd K needs word loads)
    if (dtype == W4_BF16 && vec) return run_gemv_tma(qw, scale, zero, x, d, n, k, c, stream);
    if (dtype == W4_F32)
        return vec ? dispatch_c<float, true>(qw, scale, zero, x, d, n, k, c, stream)
                   : dispatch_c<float, false>(qw, scale, zero, x, d, n, k, c, stream);
    return vec ? dispatch_c<__nv_bfloat16, true>(qw, scale, zero, x, d, n, k, c, stream)
               : dispatch_c<__nv_bfloat16, false>(qw, scale, zero, x, d, n, k, c, stream);
}

}  // namespace w4
