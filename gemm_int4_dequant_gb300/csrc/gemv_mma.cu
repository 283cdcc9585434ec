// gemv_mma.cu -- fused dequant GEMV / small-batch multiply (bf16 x, C <= 8)
// with the inner products on the warp-level tensor-core MMA.
//
//   d[c][r] = sum_k (q[r][k] - zero[r]) * scale[r] * x[c][k]
//
// (page "怎样在安卓端利用 Vulkan 编写 4-bit 专用算子", sections 1-2: uint32 words
// of eight nibbles, w0 in the low bits, dequant (q - zero) * scale in the dot
// loop; batched form from "三值量化模型的无损压缩", section 3 "MMVQ").
//
// Why tensor cores in an HBM-bound kernel: at 0.5 B of weight per multiply,
// a GB300 has about 2.7 issue slots per weight at full HBM rate.  Converting
// a nibble to fp32 and multiplying on the CUDA cores costs about 2.3 issue
// slots per weight (and 1.1 half-rate ALU slots), which leaves no margin;
// with mma.sync.m16n8k16 the weights are dequantised two per instruction
// into bf16x2 (shift, mask-and-OR into the mantissa of 128.0, subtract
// 136.0 -> q - 8 exactly) and one MMA does 256 multiply-adds, so the
// per-weight cost drops to about 1.7 slots and the kernel stays HBM-bound
// for every C <= 8.  Accumulation is fp32 in the MMA; the zero point is
// folded exactly:  sum_k (q - z) x = sum_k (q - 8) x - (z - 8) sum_k x.
//
// Work split (GB300: 152 SMs): one CTA per SM (or per cluster rank when K
// is split across a cluster).  A CTA owns a contiguous, balanced range of
// rows; its 16-row tiles x 128-k blocks are one flat list of units that its
// warps split evenly, so every warp streams the same number of 16-byte
// loads.  A tile cut between two warps is summed in shared memory (two
// contributors, so the result is order-independent).  Each warp keeps
// PF units of loads in flight.  x is staged once per CTA in shared memory,
// already in the MMA B-fragment order.

#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace w4 {

namespace gmma {

// Tuning knobs (compile-time).
#ifndef W4_GEMV_WARPS
#define W4_GEMV_WARPS 16
#endif
#ifndef W4_GEMV_PF
#define W4_GEMV_PF 4
#endif
#ifndef W4_GEMV_MINB
#define W4_GEMV_MINB 1
#endif
constexpr int WARPS = W4_GEMV_WARPS;
constexpr int THREADS = WARPS * 32;
constexpr int PF = W4_GEMV_PF;   // units of loads in flight per warp
constexpr int KB = 128;          // k per unit

// Word of 8 nibbles -> 4 bf16x2 of (q - 8): pair h = (nibble h, nibble h+4).
// Each pair is one mask-and-OR into the mantissa of 128.0 (exact 128 + q)
// and one bf16x2 FMA (x * 1 - 136, exact).  The right shifts by 4, 8, 12 are
// done as multiply-high by 2^28, 2^24, 2^20 passed in at run time (m[0..2]),
// which keeps them on the FMA pipe and off the integer ALU pipe that the
// mask-and-ORs already load.
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

struct DequantConsts {
    uint32_t m4, m8, m12;  // 2^28, 2^24, 2^20
};

__device__ __forceinline__ void dequant_word(uint32_t w, const DequantConsts& k, uint32_t (&p)[4]) {
    const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;  // bf16x2 (128, 128)
    const uint32_t one = 0x3F803F80u;                          // bf16x2 (1, 1)
    const uint32_t neg136 = 0xC308C308u;                       // bf16x2 (-136, -136)
    const uint32_t w4 = __umulhi(w, k.m4), w8 = __umulhi(w, k.m8), w12 = __umulhi(w, k.m12);
    p[0] = bfma2((w & mask) | magic, one, neg136);
    p[1] = bfma2((w4 & mask) | magic, one, neg136);
    p[2] = bfma2((w8 & mask) | magic, one, neg136);
    p[3] = bfma2((w12 & mask) | magic, one, neg136);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared memory: x fragments [kblocks][4 words][C n-lanes][4 t4] x 16 B,
// then part[rows_cap][C] fp32 (tiles owned by one warp), then the first/last
// tile partials of every warp slot[WARPS][2][16][C], then xsum[C], then the
// first/last tile index of every warp.
__host__ __device__ constexpr size_t slot_floats(int C) { return static_cast<size_t>(WARPS) * 2 * 16 * C; }

template <int C>
__global__ void __launch_bounds__(THREADS, W4_GEMV_MINB)
gemv_mma_kernel(const uint32_t* __restrict__ qw, const __nv_bfloat16* __restrict__ scale,
                const __nv_bfloat16* __restrict__ zero, const __nv_bfloat16* __restrict__ x,
                __nv_bfloat16* __restrict__ d, int N, int K, int kslice, int groups, int rows_cap, int S,
                DequantConsts dqk) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int ks = blockIdx.x % S;           // K-slice = rank in the cluster
    const int grp = blockIdx.x / S;          // row group
    const int r0 = static_cast<int>((static_cast<int64_t>(grp) * N) / groups);
    const int r1 = static_cast<int>((static_cast<int64_t>(grp + 1) * N) / groups);
    const int nrows = r1 - r0;
    const int k0 = min(K, ks * kslice);
    const int k1 = min(K, k0 + kslice);
    const int klen = k1 - k0;                 // multiple of 32
    const int nkb = (klen + KB - 1) / KB;
    const int ntiles = (nrows + 15) / 16;

    // The layout must be identical in every CTA of a cluster (peers read
    // part/xsum at this CTA's offsets), so it is sized for the longest slice.
    uint4* xf = reinterpret_cast<uint4*>(smem);
    const int xf_entries = nkb * 4 * C * 4;
    const int xf_cap = ((kslice + KB - 1) / KB) * 4 * C * 4;
    uint4* xzero = xf + xf_cap;                     // 16 zero entries for padding lanes
    float* part = reinterpret_cast<float*>(smem + static_cast<size_t>(xf_cap + 16) * 16);
    float* slot = part + rows_cap * C;
    float* xsum = slot + slot_floats(C);
    int* tspan = reinterpret_cast<int*>(xsum + C);  // [WARPS][2]: first, last tile

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int64_t kw = K / 8;  // words per row

    // ---- this warp's share of the flat (tile, kblock) list ----
    const int units = ntiles * nkb;
    const int u_begin = static_cast<int>((static_cast<int64_t>(warp) * units) / WARPS);
    const int u_end = static_cast<int>((static_cast<int64_t>(warp + 1) * units) / WARPS);

    // Load cursor.  Rows past the end of the CTA's range and k past the end
    // of the slice are clamped to the last valid row / 16-byte group instead
    // of being predicated off: their weights then multiply zero x fragments
    // (k) or are never flushed (rows), so no select is needed per load.
    const int kw_last = klen / 8 - 4;              // last valid 16-byte group (words)
    const uint32_t* qslice = qw + k0 / 8 + 4 * t4;
    uint4 buf[PF][2];
    int ltile = nkb > 0 ? u_begin / nkb : 0;
    int lkb = u_begin - ltile * nkb;
    const uint32_t* la = nullptr;
    const uint32_t* lb = nullptr;
    auto set_rows = [&](int tile) {
        const int ra = min(tile * 16 + g, nrows - 1), rb = min(tile * 16 + g + 8, nrows - 1);
        la = qslice + static_cast<int64_t>(r0 + ra) * kw;
        lb = qslice + static_cast<int64_t>(r0 + rb) * kw;
    };
    auto load_next = [&](uint4 (&b)[2]) {
        const int wofs = min(lkb * 16, kw_last - 4 * t4);
        b[0] = ldg_stream_u4(la + wofs);
        b[1] = ldg_stream_u4(lb + wofs);
        if (++lkb == nkb) {
            lkb = 0;
            set_rows(++ltile);
        }
    };
    if (u_begin < u_end) set_rows(ltile);
#pragma unroll
    for (int p = 0; p < PF; ++p)
        if (u_begin + p < u_end) load_next(buf[p]);

    // ---- stage x as B fragments, and its per-row sums ----
    // Entries are visited batch row by batch row so every thread's partial
    // sum belongs to one row n; partials are reduced in a fixed order (lanes
    // by shuffle tree, then warps in index order), so xsum is deterministic.
    float* xsw = slot;  // [WARPS][C] warp partials (slots are free until the main loop ends)
    const int per_n = nkb * 16;                    // entries per batch row
    for (int n = 0; n < C; ++n) {
        float xs_part = 0.f;
        for (int j = tid; j < per_n; j += THREADS) {
            const int t = j & 3, p = (j >> 2) & 3, kb = j >> 4;
            const int kk = kb * KB + 32 * t + 8 * p;        // within the slice
            uint32_t r[4] = {0, 0, 0, 0};
            if (kk < klen) {
                const uint4 raw = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(n) * K + k0 + kk);
                // raw holds x[kk + 0..7] as bf16 pairs (0,1) (2,3) (4,5) (6,7)
                r[0] = __byte_perm(raw.x, raw.z, 0x5410);  // (x0, x4)
                r[1] = __byte_perm(raw.x, raw.z, 0x7632);  // (x1, x5)
                r[2] = __byte_perm(raw.y, raw.w, 0x5410);  // (x2, x6)
                r[3] = __byte_perm(raw.y, raw.w, 0x7632);  // (x3, x7)
                const uint32_t v[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    xs_part += bf16_bits_to_f32(v[q] & 0xFFFFu) + bf16_bits_to_f32(v[q] >> 16);
            }
            xf[((kb * 4 + p) * C + n) * 4 + t] = make_uint4(r[0], r[1], r[2], r[3]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) xs_part += __shfl_xor_sync(0xffffffffu, xs_part, o);
        if (lane == 0) xsw[warp * C + n] = xs_part;
    }
    if (tid < 16) xzero[tid] = make_uint4(0, 0, 0, 0);
    if (lane == 0) {
        tspan[2 * warp] = u_begin < u_end ? u_begin / nkb : -1;
        tspan[2 * warp + 1] = u_begin < u_end ? (u_end - 1) / nkb : -2;
    }
    __syncthreads();
    if (tid < C) {
        float s = 0.f;
        for (int w = 0; w < WARPS; ++w) s += xsw[w * C + tid];
        xsum[tid] = s;
    }
    __syncthreads();  // xsw lives in the slots, which the main loop reuses

    // ---- main loop ----
    // two independent accumulator chains (even / odd MMA of each word) halve
    // the dependent-MMA chain per unit; they are added at flush
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
    int ctile = nkb > 0 ? u_begin / nkb : 0;      // unit being computed
    int ckb = u_begin - ctile * nkb;
    int cur_tile = ctile;
    const bool bl = g < C;  // this lane's B column is a real batch row
    const int t_first = u_begin < u_end ? u_begin / nkb : -1;
    const int t_last = u_begin < u_end ? (u_end - 1) / nkb : -2;
    // Tiles strictly inside this warp's range belong to it alone and go
    // straight to part[]; its first and last tile may be shared with the
    // neighbouring warps and go to this warp's slots, summed later in warp
    // order so the rounding never depends on timing.
    auto flush = [&](int tile) {
        const int c0 = 2 * t4, c1 = 2 * t4 + 1;
#pragma unroll
        for (int i = 0; i < 4; ++i) { acc[i] += acc2[i]; acc2[i] = 0.f; }
        float* dst = (tile == t_first || tile == t_last)
                         ? slot + (static_cast<size_t>(warp) * 2 + (tile == t_first ? 0 : 1)) * 16 * C
                         : part + static_cast<size_t>(tile) * 16 * C;
        if (c0 < C) { dst[g * C + c0] = acc[0]; dst[(g + 8) * C + c0] = acc[2]; }
        if (c1 < C) { dst[g * C + c1] = acc[1]; dst[(g + 8) * C + c1] = acc[3]; }
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
    };

    // B fragments: lanes whose column is a real batch row read x, the others
    // read the zero block
    const uint4* xlane = bl ? xf + g * 4 + t4 : xzero + t4;
    const int xw_stride = bl ? C * 4 : 4;          // entries between words
    const int xkb_stride = bl ? 4 * C * 4 : 0;     // entries between k-blocks
    for (int ub = u_begin; ub < u_end; ub += PF) {
#pragma unroll
        for (int p = 0; p < PF; ++p) {
            const int u = ub + p;
            if (u < u_end) {
                if (ctile != cur_tile) {
                    flush(cur_tile);
                    cur_tile = ctile;
                }
                const uint4 wa = buf[p][0], wb = buf[p][1];
                if (u + PF < u_end) load_next(buf[p]);
                const uint4* xb = xlane + ckb * xkb_stride;
                const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w};
                const uint32_t wbv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint4 bx = xb[w * xw_stride];
                    uint32_t pa[4], pb[4];
                    dequant_word(wav[w], dqk, pa);
                    dequant_word(wbv[w], dqk, pb);
                    const uint32_t a0[4] = {pa[0], pb[0], pa[1], pb[1]};
                    const uint32_t a1[4] = {pa[2], pb[2], pa[3], pb[3]};
                    mma_bf16(acc, a0, bx.x, bx.y);
                    mma_bf16(acc2, a1, bx.z, bx.w);
                }
                if (++ckb == nkb) { ckb = 0; ++ctile; }
            }
        }
    }
    if (u_begin < u_end) flush(cur_tile);
    __syncthreads();

    // ---- per-CTA row totals (fixed warp order) ----
    for (int i = tid; i < nrows * C; i += THREADS) {
        const int row = i / C, c = i - row * C;
        const int t = row >> 4, rl = row & 15;
        float v = 0.f;
        for (int w = 0; w < WARPS; ++w) {
            const int tf = tspan[2 * w], tl = tspan[2 * w + 1];
            if (t == tf) v += slot[(static_cast<size_t>(w) * 2 + 0) * 16 * C + rl * C + c];
            else if (t == tl) v += slot[(static_cast<size_t>(w) * 2 + 1) * 16 * C + rl * C + c];
            else if (t > tf && t < tl) v += part[i];
        }
        part[i] = v;
    }
    __syncthreads();

    // ---- combine K-slices across the cluster, apply zero fold and scale ----
    cg::cluster_group cluster = cg::this_cluster();
    if (S > 1) cluster.sync();
    for (int i = ks + S * tid; i < nrows; i += S * THREADS) {
        const int row = r0 + i;
        const float s = __bfloat162float(scale[row]);
        const float zm8 = __bfloat162float(zero[row]) - 8.0f;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float sum = 0.f, xs = 0.f;
            for (int r = 0; r < S; ++r) {
                const float* pp = (S > 1) ? cluster.map_shared_rank(part, r) : part;
                const float* xx = (S > 1) ? cluster.map_shared_rank(xsum, r) : xsum;
                sum += pp[i * C + c];
                xs += xx[c];
            }
            d[static_cast<int64_t>(c) * N + row] = __float2bfloat16_rn(s * fmaf(-zm8, xs, sum));
        }
    }
    if (S > 1) cluster.sync();
}

}  // namespace gmma

namespace {

constexpr size_t kXfBudget = 48 * 1024;

template <int C>
w4_status launch_gemv_mma_t(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N,
                            int K, cudaStream_t stream) {
    using namespace gmma;
    const int sms = sm_count();
    if (sms <= 0) return W4_ERR_CUDA;
    // K-slices: smallest power of two (<= 8) whose x fragments fit the budget
    int S = 1;
    auto slice_of = [&](int s) { return ((K + s - 1) / s + 31) / 32 * 32; };
    auto xf_bytes = [&](int s) { return static_cast<size_t>((slice_of(s) + KB - 1) / KB) * 4 * C * 4 * 16; };
    while (S < 8 && xf_bytes(S) > kXfBudget) S *= 2;
    const int kslice = slice_of(S);
    int groups = sms / S;  // one CTA per SM
    if (groups < 1) groups = 1;
    // no more row groups than 16-row tiles
    groups = static_cast<int>(std::min<int64_t>(groups, (static_cast<int64_t>(N) + 15) / 16));
    const int rows_cap = (N + groups - 1) / groups;
    const size_t smem = xf_bytes(S) + 256 + (static_cast<size_t>(rows_cap) * C + slot_floats(C) + C) * 4 + WARPS * 2 * 4;
    if (smem > 220 * 1024) return W4_ERR_SHAPE;
    auto kern = gemv_mma_kernel<C>;
    static int smem_set[64];
    cudaError_t e = ensure_smem_limit(kern, static_cast<int>(smem), smem_set);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (S > 1) {
        // all clusters must be resident at once (one wave): cap the row
        // groups by the number of clusters the GPCs can hold together
        static int max_clusters[64][4];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W4_ERR_CUDA;
        const int si = S == 2 ? 0 : S == 4 ? 1 : 2;
        if (max_clusters[dev][si] == 0) {
            cfg.gridDim = dim3(S * groups, 1, 1);
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return W4_ERR_CUDA;
            max_clusters[dev][si] = n;
        }
        groups = std::min(groups, max_clusters[dev][si]);
    }
    const int rows_cap2 = (N + groups - 1) / groups;
    if (rows_cap2 != rows_cap) {
        // fewer groups than planned: recompute the per-CTA row capacity
        const size_t smem2 = xf_bytes(S) + 256 + (static_cast<size_t>(rows_cap2) * C + slot_floats(C) + C) * 4 + WARPS * 2 * 4;
        if (smem2 > 220 * 1024) return W4_ERR_SHAPE;
        e = ensure_smem_limit(kern, static_cast<int>(smem2), smem_set);
        if (e != cudaSuccess) return W4_ERR_CUDA;
        cfg.dynamicSmemBytes = smem2;
    }
    cfg.gridDim = dim3(S * groups, 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint32_t*>(qw), static_cast<const __nv_bfloat16*>(scale),
                           static_cast<const __nv_bfloat16*>(zero), static_cast<const __nv_bfloat16*>(x),
                           static_cast<__nv_bfloat16*>(d), N, K, kslice, groups, rows_cap2, S,
                           DequantConsts{1u << 28, 1u << 24, 1u << 20});
    return launch_status(e);
}

}  // namespace

// bf16 GEMV on the MMA path; requires K % 32 == 0 (16-byte aligned rows).
w4_status run_gemv_mma(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N, int K,
                       int C, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_gemv_mma_t<1>(qw, scale, zero, x, d, N, K, stream);
        case 2: return launch_gemv_mma_t<2>(qw, scale, zero, x, d, N, K, stream);
        case 3: return launch_gemv_mma_t<3>(qw, scale, zero, x, d, N, K, stream);
        case 4: return launch_gemv_mma_t<4>(qw, scale, zero, x, d, N, K, stream);
        case 5: return launch_gemv_mma_t<5>(qw, scale, zero, x, d, N, K, stream);
        case 6: return launch_gemv_mma_t<6>(qw, scale, zero, x, d, N, K, stream);
        case 7: return launch_gemv_mma_t<7>(qw, scale, zero, x, d, N, K, stream);
        case 8: return launch_gemv_mma_t<8>(qw, scale, zero, x, d, N, K, stream);
        default: return W4_ERR_SHAPE;
    }
}

}  // namespace w4
