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

constexpr int WA_THREADS = 512;   // 16 warps; a warp takes groups of whole rows

// Shared memory of gemv_w4a8_kernel for C vectors of K elements: qs in
// word-matched order (C*K bytes), d_b and s_b as floats (2 * C*K/32 * 4
// bytes), and the C sums of s.
inline size_t w4a8_smem_bytes(int64_t C, int64_t K) { return size_t(C) * K + size_t(C) * (K / 32) * 8 + 8 * 4; }

// The x staging: every 16-byte chunk of planes 0..7 (elements k0 .. k0+15 of
// one vector) is stored at byte c*K + k0 of `xs` with each 8-element group
// split into its even elements (k, k+2, k+4, k+6) and then its odd ones --
// the order in which a weight word's nibbles come out of w & 0x0F0F0F0F and
// (w >> 4) & 0x0F0F0F0F.  Plane 8 gives d_b and s_b (b = 4 i + j).
//
// Main loop (the MMVQ page's split, section 3: a few rows per worker, so the
// activations read from shared memory serve all of them): warp w takes row
// groups of R rows (R = 4 for C <= 4, else 2) w, w + total warps, ...;
// lane l loads the 16-byte chunks b = l, l + 32, ... of the group's rows
// (one chunk = eight words = 32 weights = q8_1 block b) and, for each vector
// c, reads block b of x once and adds for each of the R rows
//   d_b * (dp4a(w & 0x0F0F0F0F, even) + dp4a((w >> 4) & 0x0F0F0F0F, odd))
// over its four words; the lanes' sums are added by a shuffle tree and
// lanes 0..R-1 store bf16(scale * (sum - zero * S_c)) for their row.
template <int C>
__global__ void __launch_bounds__(WA_THREADS)
gemv_w4a8_kernel(const uint32_t* __restrict__ qw, const __nv_bfloat16* __restrict__ scale,
                 const __nv_bfloat16* __restrict__ zero, const uint8_t* __restrict__ pt,
                 __nv_bfloat16* __restrict__ d, int64_t N, int64_t K) {
    constexpr int R = C <= 4 ? 4 : 2;
    constexpr int BATCH = R == 4 ? 2 : 4;   // chunks of each row a lane keeps in flight
    extern __shared__ __align__(16) uint8_t smem[];
    const int64_t bpr = K / 128, nb = K / 32;
    uint8_t* xs = smem;
    float* db = reinterpret_cast<float*>(smem + size_t(C) * K);
    float* sb = db + C * nb;
    float* S = sb + C * nb;

    // stage planes 0..7
    const int64_t chunks = int64_t(C) * 8 * bpr;
    for (int64_t t = threadIdx.x; t < chunks; t += WA_THREADS) {
        const int64_t c = t / (8 * bpr), rem = t % (8 * bpr);
        const int64_t p = rem / bpr, i = rem % bpr;
        const uint4 v = *reinterpret_cast<const uint4*>(pt + c * 144 * bpr + 16 * (p * bpr + i));
        const uint4 w = make_uint4(__byte_perm(v.x, v.y, 0x6420), __byte_perm(v.x, v.y, 0x7531),
                                   __byte_perm(v.z, v.w, 0x6420), __byte_perm(v.z, v.w, 0x7531));
        *reinterpret_cast<uint4*>(xs + c * K + 128 * i + 16 * p) = w;
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

    const int64_t warps = int64_t(gridDim.x) * (WA_THREADS / 32);
    const int64_t groups = (N + R - 1) / R;
    for (int64_t rg = int64_t(blockIdx.x) * (WA_THREADS / 32) + warp_id; rg < groups; rg += warps) {
        const int64_t r0 = rg * R;
        const uint8_t* rows[R];
        bool have[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            have[r] = r0 + r < N;
            rows[r] = reinterpret_cast<const uint8_t*>(qw + (have[r] ? r0 + r : r0) * (K / 8));
        }
        float acc[R][C];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) acc[r][c] = 0.f;
        for (int64_t b0 = lane; b0 < nb; b0 += 32 * BATCH) {
            uint4 w[BATCH][R];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int64_t b = b0 + 32 * u;
#pragma unroll
                for (int r = 0; r < R; ++r)
                    w[u][r] = (b < nb && have[r]) ? ldg_stream_u4(rows[r] + 16 * b) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int64_t b = b0 + 32 * u;
                if (b >= nb) break;
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    const uint4* xv = reinterpret_cast<const uint4*>(xs + c * K + 32 * b);
                    const uint4 x0 = xv[0], x1 = xv[1];
                    const uint32_t xe[4] = {x0.x, x0.z, x1.x, x1.z};
                    const uint32_t xo[4] = {x0.y, x0.w, x1.y, x1.w};
                    const float dbc = db[c * nb + b];
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
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[r][c] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][c], o);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (lane == r && have[r]) {
                const float s = __bfloat162float(scale[r0 + r]), z = __bfloat162float(zero[r0 + r]);
#pragma unroll
                for (int c = 0; c < C; ++c) d[c * N + r0 + r] = __float2bfloat16_rn(s * fmaf(-z, S[c], acc[r][c]));
            }
        }
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
    const int64_t warps_needed = (N + (C <= 4 ? 4 : 2) - 1) / (C <= 4 ? 4 : 2), warps_per_cta = WA_THREADS / 32;
    int64_t blocks = int64_t(sm_count()) * per_sm;
    const int64_t max_useful = (warps_needed + warps_per_cta - 1) / warps_per_cta;
    if (blocks > max_useful) blocks = max_useful;
    if (blocks < 1) blocks = 1;
    kern<<<static_cast<unsigned>(blocks), WA_THREADS, smem, stream>>>(
        static_cast<const uint32_t*>(qw), static_cast<const __nv_bfloat16*>(scale),
        static_cast<const __nv_bfloat16*>(zero), static_cast<const uint8_t*>(pt), static_cast<__nv_bfloat16*>(d), N,
        K);
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
