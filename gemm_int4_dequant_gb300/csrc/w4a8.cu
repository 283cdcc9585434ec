// w4a8.cu -- int4 weights against int8 activations (page "三值量化模型的无损压缩",
// section 3.1 "数据格式": x as block_q8_1 -- 32 int8 values qs and the
// halves (d, s = d * sum qs) -- laid out in the "PT" planes; section 3: the
// batched product d[r,c] = sum_k W[r,k] x[c,k]).
//
// quantize_q8_1_pt_kernel  x bf16 [C][K] -> block_q8_1 in PT planes.
// gemv_w4a8_kernel         the int4 row-layout weights of gemv_w4 against
//                          the PT activations with integer dots:
//   d[c][r] = scale[r] * ( sum_b d_b * sum_{k in b} q[r][k] qs[c][k]
//                          - zero[r] * sum_b s_b )
// (the zero point corrected through s, which needs no per-row work).
//
// PT plane layout for one vector of K elements (K % 128 == 0, bpr = K/128):
// element e of 128-element block i is byte 16 * ((e / 16) * bpr + i) + e % 16
// (planes 0..7 of 16 bytes per block), and plane 8 holds each block's four
// (d, s) pairs at 16 * (8 * bpr + i) + 4 j (d then s, little-endian halves).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace w4 {

namespace {

constexpr int QPT_THREADS = 256;

// One warp per 128-element block (c, i); lane l takes elements 4l .. 4l+3, so
// the eight lanes 8j .. 8j+7 hold q8_1 block j.  d = max|x| / 127 (IEEE fp32
// division), qs = clamp(round_half_away(x / d), -127, 127) (d == 0: qs = 0),
// d and d * sum qs stored as halves rounded to nearest even.
__global__ void __launch_bounds__(QPT_THREADS)
quantize_q8_1_pt_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ pt, int64_t C, int64_t K) {
    const int64_t bpr = K / 128;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * QPT_THREADS + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (warp >= C * bpr) return;
    const int64_t c = warp / bpr, i = warp % bpr;
    const uint2 raw = *reinterpret_cast<const uint2*>(x + c * K + 128 * i + 4 * lane);
    float v[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16), bf16_bits_to_f32(raw.y & 0xFFFFu),
                  bf16_bits_to_f32(raw.y >> 16)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    uint32_t packed = 0;
    int sum = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float r = (d == 0.0f) ? 0.0f : roundf(__fdiv_rn(v[t], d));
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        const int q = static_cast<int>(r);
        sum += q;
        packed |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * t);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    uint8_t* vec = pt + c * 144 * bpr;
    // elements 4l .. 4l+3 lie in plane l / 4 at byte 4 (l % 4) of the block's 16
    *reinterpret_cast<uint32_t*>(vec + 16 * ((lane / 4) * bpr + i) + 4 * (lane % 4)) = packed;
    if (lane % 8 == 0) {
        const uint32_t dh = __half_as_ushort(__float2half_rn(d));
        const uint32_t sh = __half_as_ushort(__float2half_rn(__fmul_rn(d, static_cast<float>(sum))));
        *reinterpret_cast<uint32_t*>(vec + 16 * (8 * bpr + i) + 4 * (lane / 8)) = dh | (sh << 16);
    }
}

constexpr int WA_THREADS = 512;

__host__ __device__ constexpr int w4a8_rows(int64_t C) { return C <= 4 ? 4 : 2; }

// Shared memory of gemv_w4a8_kernel for C vectors of K elements: the C sums
// of s (32 bytes), then qs in word-matched order (C*K bytes) and d_b, s_b as
// floats (2 * C*K/32 * 4 bytes); once x is no longer read, the threads'
// partial sums [thread][R][C] take the space after the sums of s.
inline size_t w4a8_smem_bytes(int64_t C, int64_t K) {
    const size_t x = size_t(C) * K + size_t(C) * (K / 32) * 8;
    const size_t part = size_t(WA_THREADS) * w4a8_rows(C) * C * 4;
    return 32 + (x > part ? x : part);
}

// The x staging: every 16-byte chunk of planes 0..7 (elements k0 .. k0+15 of
// one vector) is stored with each 8-element group split into its even
// elements (k, k+2, k+4, k+6) and then its odd ones -- the order in which a
// weight word's nibbles come out of w & 0x0F0F0F0F and (w >> 4) &
// 0x0F0F0F0F.  The two 16-element halves of q8_1 block b (k0 = 32 b and
// 32 b + 16) go to c*K + 16 b and c*K + K/2 + 16 b, so that threads reading
// consecutive blocks read consecutive 16-byte words.  Plane 8 gives d_b and
// s_b (b = 4 i + j).
//
// Main loop (the MMVQ page's split, section 3: a few rows per worker, so the
// activations read from shared memory serve all of them): CTA b owns row
// groups [b G, b G + G) of R rows (R = 4 for C <= 4, else 2).  With G <= T
// threads, a group's 16-byte chunks (one chunk = eight words = 32 weights =
// q8_1 block) go to tpg = T / G threads: thread j loads chunks j, j + tpg,
// ... of the group's rows and, for each vector c, reads block b of x once
// and adds for each of the R rows
//   d_b * (dp4a(w & 0x0F0F0F0F, even) + dp4a((w >> 4) & 0x0F0F0F0F, odd))
// over its four words, in registers; the tpg partial sums of a group are
// added in thread order through shared memory (one warp per group: by a
// shuffle tree) and one thread stores bf16(scale * (sum - zero * S_c)) per
// row and vector.  With G > T every thread takes whole groups and stores
// them itself.
// (one column fits 64 registers: two CTAs per SM)
template <int C>
__global__ void __launch_bounds__(WA_THREADS, C == 1 ? 2 : 1)
gemv_w4a8_kernel(const uint32_t* __restrict__ qw, const __nv_bfloat16* __restrict__ scale,
                 const __nv_bfloat16* __restrict__ zero, const uint8_t* __restrict__ pt,
                 __nv_bfloat16* __restrict__ d, int64_t N, int64_t K, int64_t G) {
    constexpr int R = w4a8_rows(C);
    constexpr int BATCH = C == 1 ? 1 : R == 4 ? 2 : 4;   // chunks of each row a thread keeps in flight (64 registers at C = 1)
    extern __shared__ __align__(16) uint8_t smem[];
    const int64_t bpr = K / 128, nb = K / 32;
    float* S = reinterpret_cast<float*>(smem);
    uint8_t* xs = smem + 32;
    float* db = reinterpret_cast<float*>(xs + size_t(C) * K);
    float* sb = db + C * nb;
    float* part = reinterpret_cast<float*>(smem + 32);

    // stage planes 0..7
    const int64_t chunks = int64_t(C) * 8 * bpr;
    for (int64_t t = threadIdx.x; t < chunks; t += WA_THREADS) {
        const int64_t c = t / (8 * bpr), rem = t % (8 * bpr);
        const int64_t p = rem / bpr, i = rem % bpr;
        const uint4 v = *reinterpret_cast<const uint4*>(pt + c * 144 * bpr + 16 * (p * bpr + i));
        const uint4 w = make_uint4(__byte_perm(v.x, v.y, 0x6420), __byte_perm(v.x, v.y, 0x7531),
                                   __byte_perm(v.z, v.w, 0x6420), __byte_perm(v.z, v.w, 0x7531));
        *reinterpret_cast<uint4*>(xs + c * K + (p & 1) * (K / 2) + 16 * (4 * i + p / 2)) = w;
    }
    // plane 8
    for (int64_t t = threadIdx.x; t < int64_t(C) * bpr; t += WA_THREADS) {
        const int64_t c = t / bpr, i = t % bpr;
        const uint4 v = *reinterpret_cast<const uint4*>(pt + c * 144 * bpr + 16 * (8 * bpr + i));
        const uint32_t pr[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            db[c * nb + 4 * i + j] = __half2float(__ushort_as_half(static_cast<unsigned short>(pr[j] & 0xFFFFu)));
            sb[c * nb + 4 * i + j] = __half2float(__ushort_as_half(static_cast<unsigned short>(pr[j] >> 16)));
        }
    }
    __syncthreads();
    // S_c = sum_b s_b, one warp per vector, in a fixed order
    const int warp_id = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp_id < C) {
        float acc = 0.f;
        for (int64_t b = lane; b < nb; b += 32) acc += sb[warp_id * nb + b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0) S[warp_id] = acc;
    }
    __syncthreads();

    const int xstride = static_cast<int>(K), xhalf = static_cast<int>(K / 2);
    const int64_t groups = (N + R - 1) / R;
    const int64_t g0 = int64_t(blockIdx.x) * G;
    const int64_t gn = groups - g0 < G ? groups - g0 : G;   // groups of this CTA
    const int tpg = threads_per_group(WA_THREADS, gn, nb);
    const int j = static_cast<int>(threadIdx.x) % tpg;
    const int gstep = WA_THREADS / tpg;
    float acc[R][C];
    for (int64_t g = threadIdx.x / tpg; g < gn; g += gstep) {
        const int64_t r0 = (g0 + g) * R;
        const uint8_t* row0 = reinterpret_cast<const uint8_t*>(qw + r0 * (K / 8));   // row r at + r * K/2
        const int nrow = N - r0 < R ? static_cast<int>(N - r0) : R;               // rows of this group
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) acc[r][c] = 0.f;
        const int nbi = static_cast<int>(nb);
        // BATCH chunks per row in flight; with several columns the chunk
        // BATCH places ahead is requested as soon as a chunk's registers are
        // free (one column: 64 registers, load then compute)
        uint4 w[BATCH][R];
        auto fetch = [&](int u, int b) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                w[u][r] = (b < nbi && r < nrow) ? ldg_stream_u4(row0 + r * (K / 2) + 16 * b) : make_uint4(0, 0, 0, 0);
        };
        auto chunk = [&](int u, int b) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const uint4 x0 = *reinterpret_cast<const uint4*>(xs + c * xstride + 16 * b);
                const uint4 x1 = *reinterpret_cast<const uint4*>(xs + c * xstride + xhalf + 16 * b);
                const uint32_t xe[4] = {x0.x, x0.z, x1.x, x1.z};
                const uint32_t xo[4] = {x0.y, x0.w, x1.y, x1.w};
                const float dbc = db[c * nbi + b];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t ww[4] = {w[u][r].x, w[u][r].y, w[u][r].z, w[u][r].w};
                    int dot = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        dot = __dp4a(static_cast<int>(ww[q] & 0x0F0F0F0Fu), static_cast<int>(xe[q]), dot);
                        dot = __dp4a(static_cast<int>((ww[q] >> 4) & 0x0F0F0F0Fu), static_cast<int>(xo[q]), dot);
                    }
                    acc[r][c] = fmaf(dbc, static_cast<float>(dot), acc[r][c]);
                }
            }
        };
        if constexpr (C == 1) {
            for (int b0 = j; b0 < nbi; b0 += tpg * BATCH) {
#pragma unroll
                for (int u = 0; u < BATCH; ++u) fetch(u, b0 + tpg * u);
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    if (b0 + tpg * u >= nbi) break;
                    chunk(u, b0 + tpg * u);
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < BATCH; ++u) fetch(u, j + tpg * u);
            for (int b0 = j; b0 < nbi; b0 += tpg * BATCH) {
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    const int b = b0 + tpg * u;
                    if (b >= nbi) break;
                    chunk(u, b);
                    fetch(u, b + tpg * BATCH);
                }
            }
        }
        if (tpg == 32) {
            // a warp per group: its lanes' sums meet by a shuffle tree
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int c = 0; c < C; ++c)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[r][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][c], o);
        }
        if (tpg == 1 || tpg == 32) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r >= nrow || (tpg == 32 && lane != r)) continue;
                const float s = __bfloat162float(scale[r0 + r]), z = __bfloat162float(zero[r0 + r]);
#pragma unroll
                for (int c = 0; c < C; ++c) d[c * N + r0 + r] = __float2bfloat16_rn(s * fmaf(-z, S[c], acc[r][c]));
            }
        }
    }
    if (tpg == 1 || tpg == 32) return;   // (otherwise one round: T / tpg >= gn)
    __syncthreads();   // x is no longer read: its space takes the partial sums
    if (threadIdx.x / tpg < gn) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) part[(threadIdx.x * R + r) * C + c] = acc[r][c];
    }
    __syncthreads();
    for (int64_t o = threadIdx.x; o < gn * R * C; o += WA_THREADS) {
        const int64_t g = o / (R * C), r = (o / C) % R, c = o % C;
        const int64_t row = (g0 + g) * R + r;
        if (row >= N) continue;
        float sum = 0.f;
        for (int t = 0; t < tpg; ++t) sum += part[((g * tpg + t) * R + r) * C + c];
        const float s = __bfloat162float(scale[row]), z = __bfloat162float(zero[row]);
        d[c * N + row] = __float2bfloat16_rn(s * fmaf(-z, S[c], sum));
    }
}

template <int C>
w4_status launch_w4a8(const void* qw, const void* scale, const void* zero, const void* pt, void* d, int64_t N,
                      int64_t K, cudaStream_t stream) {
    static int smem_set[64];
    const size_t smem = w4a8_smem_bytes(C, K);
    auto kern = gemv_w4a8_kernel<C>;
    if (ensure_smem_limit(kern, static_cast<int>(smem), smem_set) != cudaSuccess) return W4_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, WA_THREADS, smem) != cudaSuccess || per_sm < 1)
        return W4_ERR_CUDA;
    // as many CTAs as are resident at once, each a contiguous range of row groups
    const int64_t groups = (N + w4a8_rows(C) - 1) / w4a8_rows(C);
    int64_t ctas = int64_t(sm_count()) * per_sm;
    if (ctas > groups) ctas = groups;
    if (ctas < 1) ctas = 1;
    const int64_t G = groups > 0 ? (groups + ctas - 1) / ctas : 1;
    ctas = groups > 0 ? (groups + G - 1) / G : 1;
    kern<<<static_cast<unsigned>(ctas), WA_THREADS, smem, stream>>>(
        static_cast<const uint32_t*>(qw), static_cast<const __nv_bfloat16*>(scale),
        static_cast<const __nv_bfloat16*>(zero), static_cast<const uint8_t*>(pt), static_cast<__nv_bfloat16*>(d), N,
        K, G);
    return launch_status(cudaGetLastError());
}

}  // namespace

bool w4a8_fits(int64_t C, int64_t K) { return w4a8_smem_bytes(C, K) <= size_t(W4_W4A8_MAX_SMEM); }

w4_status run_quantize_q8_1_pt(const void* x, void* pt, int64_t C, int64_t K, cudaStream_t stream) {
    const int64_t warps = C * (K / 128);
    const int64_t blocks = (warps + QPT_THREADS / 32 - 1) / (QPT_THREADS / 32);
    if (blocks > 0x7FFFFFFF) return W4_ERR_SHAPE;
    quantize_q8_1_pt_kernel<<<static_cast<unsigned>(blocks), QPT_THREADS, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(pt), C, K);
    return launch_status(cudaGetLastError());
}

w4_status run_gemv_w4a8(const void* qw, const void* scale, const void* zero, const void* pt, void* d, int64_t N,
                        int64_t K, int64_t C, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_w4a8<1>(qw, scale, zero, pt, d, N, K, stream);
        case 2: return launch_w4a8<2>(qw, scale, zero, pt, d, N, K, stream);
        case 3: return launch_w4a8<3>(qw, scale, zero, pt, d, N, K, stream);
        case 4: return launch_w4a8<4>(qw, scale, zero, pt, d, N, K, stream);
        case 5: return launch_w4a8<5>(qw, scale, zero, pt, d, N, K, stream);
        case 6: return launch_w4a8<6>(qw, scale, zero, pt, d, N, K, stream);
        case 7: return launch_w4a8<7>(qw, scale, zero, pt, d, N, K, stream);
        case 8: return launch_w4a8<8>(qw, scale, zero, pt, d, N, K, stream);
        default: return W4_ERR_SHAPE;
    }
}

}  // namespace w4
