// gemv_tma.cu -- fused dequant GEMV / small-batch multiply for bf16 x (C <= 8),
// weights streamed by the tensor memory accelerator (TMA) into a shared-memory
// ring and multiplied on the warp-level tensor-core MMA.
//
//   d[c][r] = sum_k (q[r][k] - zero[r]) * scale[r] * x[c][k]
//
// (page "怎样在安卓端利用 Vulkan 编写 4-bit 专用算子", sections 1-2: uint32 words
// of eight nibbles, w0 in the low bits, dequant (q - zero) * scale in the dot
// loop; batched form from "三值量化模型的无损压缩", section 3 "MMVQ".)
//
// GB300 design.  The op reads 0.5 B of weight per multiply-add, so HBM
// bandwidth is the roofline.  One CTA per SM owns a contiguous range of whole
// 16-row tiles (and, when x does not fit, one K-slice of a thread-block
// cluster); the grid is the smallest that keeps the busiest range as short,
// so SMs left over take the next launch's CTAs while this one finishes:
//   * warp NC (producer) streams 16-row tiles with the TMA.  The copy engine
//     has a fixed cost per copy, so a stage is one copy: the weights are
//     viewed as a 3-D tensor (8-byte words x 64-byte chunks x rows) and a box
//     of 16 rows x an ODD number of chunks lands at a row pitch of 64 mod
//     128 bytes, which keeps the consumers' fragment loads on distinct banks
//     (chunks past the end of a row are zero-filled, not fetched).  A tile
//     with fewer rows (the end of a CTA's range) takes 4-row boxes so that no
//     neighbour's rows are read.  Rows that are not whole 64-byte chunks
//     (K % 128 != 0) fall back to 1-D bulk copies: one per tile when its rows
//     are contiguous, else one per row into a padded pitch.  The ring holds
//     as many stages as shared memory allows (about 200 KB in flight per SM,
//     no registers spent);
//   * warps 0..NC-1 (consumers) share out the 128-k blocks of every stage
//     round-robin (continuing across stages, so the split stays balanced):
//     two 16-byte shared loads give a lane its rows g and g+8, each uint32
//     word becomes four 16-bit pairs (nibbles j, j+4) of q - zi, zi the
//     zero point's integer part, and two mma.sync.m16n8k16 per word
//     accumulate in fp32 against x, which was staged once per CTA in
//     B-fragment order.  The zero point leaves the weights before any
//     product, exactly: a row whose nibbles all equal z gives exactly 0.
//     In bf16 one mask-and-OR per pair puts the nibble into the mantissa of
//     128.0 (exactly 128 + q, after a shift by 4j) and one packed subtract
//     of 128 + zi leaves q - zi.  With one column of x the pairs are fp16,
//     whose ten mantissa bits take a nibble at bits 0-3 or 4-7 unshifted:
//     one mask-and-OR gives 1024 + q (nibbles 0, 2; the second after a
//     single shift by 8), minus 1024 + zi, or 1024 + 16q (nibbles 1, 3),
//     times 1/16 minus 64 + zi in one packed FMA; the two MMAs of a word
//     cover even and odd k.  x is scaled by a power of two (largest |x| in
//     [2^14, 2^15)) before its fp16 conversion, which is exact for every
//     element within 2^30 of the largest; a CTA whose slice of x spans more
//     (or whose largest |x| is below 2^-86) runs the bf16 loop instead, with
//     x scaled up by a power of two when its largest |x| is below 2^14.
//     The scaling is undone in fp32;
//   * the NC warps' partial sums of a row are added in warp order (each warp
//     keeps its own row partials, or per 16-row tile through a named
//     barrier when those do not fit), so results never depend on timing;
//   * only a fractional zero point leaves a term for the end:
//       sum_k (q - z) x = sum_k (q - zi) x - (z - zi) sum_k x;
//   * K-slices of a cluster meet at the row's owner: every rank pushes its
//     partials of the rows the others own into their shared memory
//     (st.async), and owners add the slices in rank order.
// Every mbarrier wait is bounded (about two seconds); on timeout the kernel
// records an error code (w4_device_error), stops issuing copies, drains the
// ones in flight and returns.

#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace w4 {

namespace gtma {

using namespace ptx;

// Test switch (w4_selftest_configure): when set, the producer announces 16
// bytes more than it copies for a CTA's first stage, so that stage's wait
// cannot complete and runs out -- the error path (error word, abort, drain)
// runs without any bad access.  Always 0 in normal use.
static __device__ int g_short_first_stage;

#ifndef W4_GEMV_NC
#define W4_GEMV_NC 12                           // three consumer warps per SM sub-partition
#endif
constexpr int NC = W4_GEMV_NC;                // consumer warps
constexpr int THREADS = (NC + 1) * 32;        // + one producer warp
constexpr int CT = NC * 32;                   // consumer threads
constexpr int KB = 128;                       // k per unit (one consumer warp per unit)
constexpr int MAX_NST = 8;                    // stages in the ring (at most)
#ifndef W4_GEMV_KCHUNK
#define W4_GEMV_KCHUNK 8192
#endif
constexpr int KCHUNK_MAX = W4_GEMV_KCHUNK;    // k per stage at most (4 KB per row)
#ifndef W4_GEMV_MINB
#define W4_GEMV_MINB 1
#endif
#ifndef W4_GEMV_SMEM
#define W4_GEMV_SMEM (227 * 1024)
#endif
#ifndef W4_GEMV_XR
#define W4_GEMV_XR 14                           // x fragments staged per consumer thread at most
#endif
constexpr int XR_MAX = W4_GEMV_XR;
#ifndef W4_GEMV_PREFETCH_STAGES
#define W4_GEMV_PREFETCH_STAGES 3               // stages warmed in L2 before the wait (one column of x)
#endif

// Nibble mask and bf16 magic passed at run time so they stay in registers and
// each mask-and-OR is a single three-input logic op.
struct MaskMagic {
    uint32_t mask, magic, magic_bf16;   // magic: of the loop with one column of x (fp16); bf16 loop
};

// Run-time shape of the pipeline, identical for every CTA of a launch (peers
// in a cluster read each other's shared memory at the same offsets).
struct Plan {
    int S;          // K-slices (cluster size)
    int kslice;     // k per slice (multiple of 32)
    int kchunk;     // k per stage (multiple of 128, <= kslice rounded up)
    int dense;      // 1: a stage is one copy of 16 contiguous full rows
    int pitch;      // bytes between rows of a stage in shared memory
    int nst;        // stages in the ring
    int groups;     // row groups
    int rows_cap;   // rows per CTA at most
    int perwarp;    // 1: every warp keeps its own row partials (no per-tile barrier)
    int tmap;       // 1: a stage is one (or, for a partial tile, a few) 3-D tensor copies
    int nbox;       // 64-byte chunks per row in a tensor box (odd: pitch = 64 mod 128)
    int xpitch;     // permuted layout: bytes per row of x in shared memory (16 mod 128); 0 otherwise
};

// Base alignment of the dynamic shared memory layout: tensor copies land at
// 128-byte aligned addresses (every stage and box offset is a multiple of 256)
constexpr int kSmemAlign = 128;

struct Layout {
    int stage_bytes, xf, xzero, red, part, partw, xsw, xsum, sz, zz, rcv, rxs, bars, abort, total;
};

__host__ __device__ inline Layout make_layout(int C, const Plan& P) {
    Layout L;
    L.stage_bytes = 16 * P.pitch;
    const int nkb_cap = (P.kslice + KB - 1) / KB;
    int o = P.nst * L.stage_bytes;
    o = (o + 127) & ~127;
    L.xf = o;        o += P.xpitch ? C * P.xpitch : nkb_cap * 16 * C * 16;
    L.xzero = o;     o += 16 * C * 16;
    L.red = o;       o += P.perwarp ? 0 : 2 * NC * 16 * C * 4;
    L.part = o;      o += P.rows_cap * C * 4;
    L.partw = o;     o += P.perwarp ? NC * ((P.rows_cap + 15) / 16 * 16) * C * 4 : 0;
    L.xsw = o;       o += NC * C * 2 * 4;
    // per column: [0, 8) this CTA's sum of x (unscaled), [8] the smallest
    // nonzero |x| (bf16 bits, one column), [16, 24) the largest |x| (bf16
    // bits), later 0, [24, 32) the factor that undoes the scaling of x
    L.xsum = o;      o += 32 * 4;
    // (scale, z - zint(z)) per row as fp32; with one column and no K split
    // each thread finishes the rows whose scale and zero point it holds in
    // registers, and the table is not needed
    L.sz = o;        o += (C > 1 || P.S > 1) ? P.rows_cap * 8 : 0;
    o = (o + 15) & ~15;
    // per row, what the main loop subtracts after the unpack (zi = zint(z)):
    // fp16 (1024 + zi, even k) and the addend -(64 + zi) of the odd-k FMA,
    // bf16 128 + zi, each in both halves
    L.zz = o;        o += P.rows_cap * 16;
    // K split: the other slices' partials of the rows this rank owns (rows
    // ks, ks+S, ...) and their sums of x, pushed in by the peers
    L.rcv = o;       o += P.S > 1 ? P.S * ((P.rows_cap + P.S - 1) / P.S) * C * 4 : 0;
    L.rxs = o;       o += P.S > 1 ? 8 * 8 * 4 : 0;
    o = (o + 7) & ~7;
    L.bars = o;      o += (2 * MAX_NST + 2) * 8;   // full[], empty[], x copied, pushes received
    L.abort = o;     o += 16;
    L.total = o;
    return L;
}

// PERM = false: weights uint32 [N][K/8] (rows of eight nibbles per word),
// bf16 scale and zero per row.  PERM = true: weights in the permuted layout
// of permute_int4 (column groups of 4, 128-byte lines of 64 k, two's
// complement nibbles), fp32 scale per column and no zero point.
template <int C, bool PERM>
__global__ void __launch_bounds__(THREADS, W4_GEMV_MINB)
gemv_tma_kernel(const uint8_t* __restrict__ qw, const void* __restrict__ scale,
                const void* __restrict__ zero, const __nv_bfloat16* __restrict__ x,
                __nv_bfloat16* __restrict__ d, int N, int K, Plan P, MaskMagic dq,
                const __grid_constant__ CUtensorMap tm16, const __grid_constant__ CUtensorMap tm4) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    constexpr uint32_t kAl = kSmemAlign;
    uint8_t* sm = smem_raw + (((raw_addr + (kAl - 1)) & ~(kAl - 1)) - raw_addr);
    const uint32_t sm_addr = smem_u32(sm);
    const Layout L = make_layout(C, P);
    const int S = P.S, NST = P.nst, pitch = P.pitch;

    const int ks = blockIdx.x % S;        // K-slice = rank in the cluster
    const int grp = blockIdx.x / S;       // row group
    // whole 16-row tiles per row group; the first (tiles % groups) groups
    // take one more (they are dispatched first)
    const int64_t tiles = (static_cast<int64_t>(N) + 15) / 16;
    const int64_t tb = tiles / P.groups, te = tiles % P.groups;
    const int64_t t0 = grp * tb + (grp < te ? grp : te);
    const int64_t r1t = 16 * (t0 + tb + (grp < te ? 1 : 0));
    const int r0 = static_cast<int>(16 * t0);
    const int r1 = static_cast<int>(N < r1t ? static_cast<int64_t>(N) : r1t);
    const int nrows = max(0, r1 - r0);
    const int k0 = min(K, ks * P.kslice);
    const int klen = min(K, k0 + P.kslice) - k0;      // multiple of 32
    const int nch = (klen + P.kchunk - 1) / P.kchunk;
    const int ntiles = (nrows + 15) / 16;
    const int nstages = ntiles * nch;

    uint4* xf = reinterpret_cast<uint4*>(sm + L.xf);
    uint4* xzero = reinterpret_cast<uint4*>(sm + L.xzero);
    float* red = reinterpret_cast<float*>(sm + L.red);
    float* part = reinterpret_cast<float*>(sm + L.part);
    float* partw = reinterpret_cast<float*>(sm + L.partw);
    float* xsw = reinterpret_cast<float*>(sm + L.xsw);
    float* xsum = reinterpret_cast<float*>(sm + L.xsum);
    float2* sz = reinterpret_cast<float2*>(sm + L.sz);
    const uint32_t bar_full = sm_addr + L.bars;
    const uint32_t bar_empty = bar_full + MAX_NST * 8;
    const uint32_t bar_x = bar_full + 2 * MAX_NST * 8;
    const uint32_t bar_rcv = bar_x + 8;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L.abort);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // one column of the row layout runs on fp16 MMAs (x scaled by a power of
    // two, weights unpacked with five logic ops per word) when the CTA's
    // slice of x fits fp16's range; everything else on bf16
    constexpr bool CAN_F16 = !PERM && C == 1;
    // scale of output row r and its zero point split into the integer part
    // taken out of the weights and the rest folded out at the end; the
    // permuted operand is symmetric (zero point 0)
    auto load_z = [&](int r) -> float {
        return PERM ? 0.0f : __bfloat162float(static_cast<const __nv_bfloat16*>(zero)[r]);
    };
    auto load_s = [&](int r) -> float {
        return PERM ? static_cast<const float*>(scale)[r]
                    : __bfloat162float(static_cast<const __nv_bfloat16*>(scale)[r]);
    };
    uint4* zz_s = reinterpret_cast<uint4*>(sm + L.zz);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, NC);
        }
        mbar_init(bar_x, 1);
        *abort_flag = 0;
        for (int c = 0; c < 8; ++c) reinterpret_cast<uint32_t*>(xsum)[16 + c] = 0;   // column maxima of |x|
        reinterpret_cast<uint32_t*>(xsum)[8] = 0xFFFFu;                              // (smallest nonzero |x|) - 1
        reinterpret_cast<uint32_t*>(xsum)[9] = 0u;                                   // a fractional zero point seen
        if (S > 1) {
            // every peer pushes its partials of the rows this rank owns and its
            // C sums of x; they complete bytes on this barrier
            const int own = nrows > ks ? (nrows - ks + S - 1) / S : 0;
            mbar_init(bar_rcv, 1);
            mbar_arrive_expect_tx(bar_rcv, static_cast<uint32_t>((S - 1) * (own * C + C) * 4));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // first half of a cluster barrier: this CTA's barriers are initialised
    // (the second half is waited for just before the first push to a peer)
    if (S > 1) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    // Launched with programmatic stream serialisation.  The next kernel in
    // the stream may be scheduled at once: its CTAs take SMs as they come
    // free (idle SMs first) and prepare while this grid finishes, and its own
    // wait still orders all of its reads after this grid has completed.
    pdl_launch_dependents();
    // Before waiting for the previous kernel, warm L2 with this CTA's first
    // stage(s): L2 is the device's point of coherence, so a prefetch cannot
    // yield stale data even if the previous kernel writes these bytes; every
    // load into shared memory or registers is issued only after the wait.
    if (PERM && warp == NC && lane == 0 && nstages > 0) {
        // the first stage: each column group's first lines
        const uint32_t gbytes = (min(P.kchunk, klen) + 63) / 64 * 128;
        for (int gi = 0; gi < min(16, nrows) / 4; ++gi)
            bulk_prefetch_l2(qw + static_cast<int64_t>(r0 / 4 + gi) * 2 * K + (k0 / 64) * 128, gbytes);
    } else if (warp == NC && lane == 0) {
        const int64_t row_bytes = K / 2;
        const uint8_t* src0 = qw + static_cast<int64_t>(r0) * row_bytes + k0 / 2;
        int tile = 0, ch = 0;
        // one column: three stages (measured best); several columns: one, since
        // their larger x copy follows the wait and competes with the prefetch
        constexpr int kPrefetch = C == 1 ? W4_GEMV_PREFETCH_STAGES : 1;
        for (int s = 0; s < min(nstages, kPrefetch); ++s) {
            const int rows_here = min(16, nrows - tile * 16);
            const int seg = min(P.kchunk, klen - ch * P.kchunk) / 2;
            const uint8_t* src = src0 + static_cast<int64_t>(tile) * 16 * row_bytes + ch * (P.kchunk / 2);
            if (P.dense) {
                bulk_prefetch_l2(src, rows_here * seg);
            } else {
                for (int r = 0; r < rows_here; ++r) bulk_prefetch_l2(src + r * row_bytes, seg);
            }
            if (++ch == nch) { ch = 0; ++tile; }
        }
    }
    pdl_wait();
    __syncthreads();

    if (warp == NC) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // x rows of this slice, first thing (every CTA reads the same x:
            // default L2 policy): rows of xpitch bytes for the permuted
            // layout, dense rows of klen elements for the row layout (which
            // the consumers then rearrange in place)
            const int xrow = PERM ? P.xpitch : klen * 2;
            mbar_arrive_expect_tx(bar_x, C * klen * 2);
            if (klen > 0)
                for (int n = 0; n < C; ++n)
                    bulk_load(smem_u32(xf) + n * xrow, x + static_cast<int64_t>(n) * K + k0, klen * 2, bar_x);
        }
        if (lane == 0 && nstages > 0) {
            const uint64_t policy = l2_evict_first_policy();
            const int64_t row_bytes = K / 2;
            const uint8_t* src0 = qw + static_cast<int64_t>(r0) * row_bytes + k0 / 2;
            const uint32_t short0 = g_short_first_stage ? 16u : 0u;
            int tile = 0, ch = 0, issued = 0, slot = 0, round = 0;
            for (int s = 0; s < nstages; ++s) {
                if (round > 0 && !mbar_wait_fast(bar_empty + 8 * slot, (round - 1) & 1, abort_flag)) break;
                // after an abort the consumers still release their slots, but a
                // stage whose copy never completed must not be armed again
                if (*abort_flag) break;
                const uint32_t extra = s == 0 ? short0 : 0u;
                const int rows_here = min(16, nrows - tile * 16);
                const int seg = min(P.kchunk, klen - ch * P.kchunk) / 2;   // bytes per row (multiple of 16)
                const uint32_t dst = sm_addr + slot * L.stage_bytes;
                const uint8_t* src = src0 + static_cast<int64_t>(tile) * 16 * row_bytes + ch * (P.kchunk / 2);
                if constexpr (PERM) {
                    // one bulk copy per column group: its lines of this K-chunk
                    // (128 bytes = 64 k of 4 columns each), at a group stride of
                    // 16 mod 128 bytes so that ldmatrix rows hit distinct banks
                    const int len = min(P.kchunk, klen - ch * P.kchunk);   // multiple of 64
                    const uint32_t gbytes = len / 64 * 128;
                    const int ng = rows_here / 4;
                    const uint8_t* g0 = qw + static_cast<int64_t>(r0 / 4 + tile * 4) * 2 * K +
                                        ((k0 + ch * P.kchunk) / 64) * 128;
                    mbar_arrive_expect_tx(bar_full + 8 * slot, ng * gbytes + extra);
                    for (int gi = 0; gi < ng; ++gi)
                        bulk_load_hint(dst + gi * 4 * pitch, g0 + static_cast<int64_t>(gi) * 2 * K, gbytes,
                                       bar_full + 8 * slot, policy);
                } else if (P.tmap) {
                    const int c0 = (k0 + ch * P.kchunk) / 128, row0 = r0 + tile * 16;
                    if (rows_here == 16) {
                        mbar_arrive_expect_tx(bar_full + 8 * slot, 16 * pitch + extra);
                        tma_load_3d_hint(dst, &tm16, 0, c0, row0, bar_full + 8 * slot, policy);
                    } else {
                        const int nb = (rows_here + 3) / 4;
                        mbar_arrive_expect_tx(bar_full + 8 * slot, nb * 4 * pitch + extra);
                        for (int b = 0; b < nb; ++b)
                            tma_load_3d_hint(dst + b * 4 * pitch, &tm4, 0, c0, row0 + 4 * b, bar_full + 8 * slot,
                                             policy);
                    }
                } else if (P.dense) {
                    mbar_arrive_expect_tx(bar_full + 8 * slot, rows_here * seg + extra);
                    bulk_load_hint(dst, src, rows_here * seg, bar_full + 8 * slot, policy);
                } else {
                    mbar_arrive_expect_tx(bar_full + 8 * slot, rows_here * seg + extra);
                    for (int r = 0; r < rows_here; ++r)
                        bulk_load_hint(dst + r * pitch, src + r * row_bytes, seg, bar_full + 8 * slot, policy);
                }
                issued = s + 1;
                if (++ch == nch) { ch = 0; ++tile; }
                if (++slot == NST) { slot = 0; ++round; }
            }
            // copies still landing if a consumer aborted
            for (int s = max(0, issued - NST); s < issued; ++s) mbar_drain(bar_full + 8 * (s % NST), (s / NST) & 1);
        }
        if (lane == 0) mbar_drain(bar_x, 0);
    } else {
        // ------------------------------------------------------------ consumers
        // scale / zero point of this CTA's rows: the first two per thread are
        // loaded now into registers (nothing waits on them); zint(z) goes to
        // shared memory once x has arrived (the main loop subtracts it from
        // the weights), the scale and z - zint(z) after the main loop
        float sc_pf[2], z_pf[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = tid + j * CT;
            if (i < nrows) {
                sc_pf[j] = load_s(r0 + i);
                z_pf[j] = load_z(r0 + i);
            }
        }
        auto zconsts = [](int zi) {
            const uint32_t u = static_cast<uint32_t>(zi);
            return make_uint4((0x6400u + u) * 0x10001u, (0xD400u + 16u * u) * 0x10001u, (0x4300u + u) * 0x10001u, 0u);
        };
        // (also notes whether any row's zero point has a fractional part: only
        // then do the sums of x enter the result)
        volatile uint32_t* frac_seen = reinterpret_cast<volatile uint32_t*>(xsum) + 9;
        auto store_zint = [&]() {
            if constexpr (!PERM) {
                bool frac = false;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int i = tid + j * CT;
                    if (i < nrows) {
                        const int zi = zint(z_pf[j]);
                        zz_s[i] = zconsts(zi);
                        frac |= static_cast<float>(zi) != z_pf[j];
                    }
                }
                for (int i = tid + 2 * CT; i < nrows; i += CT) {
                    const float z = load_z(r0 + i);
                    const int zi = zint(z);
                    zz_s[i] = zconsts(zi);
                    frac |= static_cast<float>(zi) != z;
                }
                if (frac) *frac_seen = 1u;
            }
        };
        bool f16 = false;   // this CTA's main loop runs on fp16 MMAs
        // x as B fragments.  Row layout: entry (kb, word p, n, t4) holds, for
        // kk = kb*128 + 32*t4 + 8*p, the pairs (x[kk], x[kk+4]) (x[kk+1],
        // x[kk+5]) (x[kk+2], x[kk+6]) (x[kk+3], x[kk+7]) in bf16 -- the b0b1 /
        // b2b3 registers of the two MMAs that consume word p (nibbles 0, 1 and
        // 2, 3).  On fp16 (one column) the order is (x[kk], x[kk+4]) (x[kk+2],
        // x[kk+6]) (x[kk+1], x[kk+5]) (x[kk+3], x[kk+7]): one MMA over the
        // word's nibbles 0 and 2 (even k), one over 1 and 3 (odd k); x is
        // multiplied by a power of two first (its largest |x| lands in
        // [2^14, 2^15)).
        const int g = lane >> 2, t4 = lane & 3;
        const bool bl = g < C;
        const uint4* xlane = bl ? xf + g * 4 + t4 : xzero + t4;
        constexpr int xw_stride = C * 4;
        // permuted layout: x is kept as rows; this lane gives the ldmatrix row
        // address for row n = lane % 8 of matrix lane / 8 (k + 8 * matrix
        // within each 32-k group); rows past C read a zero block
        const int xrow = lane & 7;
        const uint32_t xa = xrow < C ? smem_u32(xf) + xrow * P.xpitch + (lane >> 3) * 16 : smem_u32(xzero);
        const uint32_t xs = xrow < C ? 64 : 0;   // bytes per 32-k group
        {
            // thread tid stages entries tid, tid + CT, ... (n-major), stepping
            // (n, j) without dividing; the column sums are left to the tensor
            // cores
            const int nkb = (klen + KB - 1) / KB;
            if constexpr (PERM) {
                // permuted operand: x arrives by bulk copies (issued by the
                // producer) as rows of xpitch bytes; ldmatrix reads it as B
                // fragments directly.  Zero the tail of a half unit, then wait.
                const int tail = (nkb * KB - klen) * 2;   // bytes past the slice in the last unit
                for (int i = tid; i < C * (tail / 16); i += CT) {
                    const int n = i / (tail / 16), q = i - n * (tail / 16);
                    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(xf) + n * P.xpitch + klen * 2 + q * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                mbar_wait_fast(bar_x, 0, abort_flag);
                store_zint();
            } else {
                // x arrived by bulk copies as dense rows (row n at n*klen*2
                // bytes) in the fragment buffer itself: every thread reads its
                // entries' sources into registers (with one column noting the
                // largest and the smallest nonzero |x|: warp extremes meet in
                // shared memory); after a barrier it writes them in fragment
                // order (fp16: scaled and converted; bf16 with one column:
                // scaled by a power of two when the largest |x| is below
                // 2^14).  At most XR entries per thread: the plan keeps the
                // fragments within XR entries per consumer thread.
                const int per_n = nkb * 16;
                constexpr int XR = XR_MAX;
                const int dn = per_n > 0 ? CT / per_n : 0, dj = CT - dn * per_n;
                const int n_cur = per_n > 0 ? tid / per_n : C, j_cur = tid - n_cur * per_n;
                const int mine = (C * per_n - tid + CT - 1) / CT;   // entries of this thread (<= XR)
                const uint8_t* rows = reinterpret_cast<const uint8_t*>(xf);
                uint32_t* xmax = reinterpret_cast<uint32_t*>(xsum) + 16;   // max |x| bits, zeroed at entry
                uint32_t* xmin = reinterpret_cast<uint32_t*>(xsum) + 8;    // min nonzero |x| bits - 1
                uint4 v[XR];
                uint32_t mx = 0, mn = 0xFFFFu;
                mbar_wait_fast(bar_x, 0, abort_flag);
                store_zint();
                int n = n_cur, j = j_cur;
#pragma unroll
                for (int b = 0; b < XR; ++b) {
                    if (b >= mine) break;
                    v[b] = make_uint4(0, 0, 0, 0);
                    if (n < C) {
                        const int kk = (j >> 4) * KB + 32 * (j & 3) + 8 * ((j >> 2) & 3);
                        if (kk < klen) v[b] = *reinterpret_cast<const uint4*>(rows + (n * klen + kk) * 2);
                        if constexpr (CAN_F16) {
                            // |x| as bf16 bit patterns with the sign cleared
                            // (ordered as integers); |x| - 1 wraps 0 to 0xFFFF
                            const uint32_t a0 = v[b].x & 0x7FFF7FFFu, a1 = v[b].y & 0x7FFF7FFFu;
                            const uint32_t a2 = v[b].z & 0x7FFF7FFFu, a3 = v[b].w & 0x7FFF7FFFu;
                            const uint32_t m2 = __vmaxu2(__vmaxu2(a0, a1), __vmaxu2(a2, a3));
                            mx = max(mx, max(m2 & 0xFFFFu, m2 >> 16));
                            const uint32_t n2 = __vminu2(__vminu2(__vsub2(a0, 0x00010001u), __vsub2(a1, 0x00010001u)),
                                                         __vminu2(__vsub2(a2, 0x00010001u), __vsub2(a3, 0x00010001u)));
                            mn = min(mn, min(n2 & 0xFFFFu, n2 >> 16));
                        }
                    }
                    j += dj;
                    n += dn;
                    if (j >= per_n) { j -= per_n; ++n; }
                }
                if constexpr (CAN_F16) {
                    const uint32_t wm = __reduce_max_sync(0xffffffffu, mx);
                    const uint32_t wn = __reduce_min_sync(0xffffffffu, mn);
                    if (lane == 0) {
                        if (wm != 0) atomicMax(&xmax[0], wm);
                        if (wn != 0xFFFFu) atomicMin(&xmin[0], wn);
                    }
                }
                named_barrier(1, CT);   // every source read (and the extremes of |x| final)
                // fp16 when every nonzero |x| lies within 2^30 of the largest
                // and the largest is at least 2^-86: x is scaled by 2^e, e =
                // 141 - (biased bf16 exponent of max|x|) <= 100, so that
                // max|x| 2^e lies in [2^14, 2^15) and every element stays an
                // exact fp16 (normal, or subnormal with 8 significant bits).
                // Otherwise bf16, scaled by 2^min(126, e) only when e > 0
                // (exact: bf16 has fp32's exponent range).  se / so: sums of
                // the converted x over even / odd k (fp16).
                const int emax = static_cast<int>(xmax[0] >> 7), emin = static_cast<int>((xmin[0] + 1) >> 7);
                f16 = CAN_F16 && (xmax[0] == 0 || (emax >= 41 && emax - emin <= 30));
                const float sc = f16 ? __int_as_float((127 + min(100, 141 - emax)) << 23)
                                 : CAN_F16 ? __int_as_float((127 + min(126, max(0, 141 - emax))) << 23)
                                           : 1.0f;
                float se = 0.f, so = 0.f;
                n = n_cur;
                j = j_cur;
#pragma unroll
                for (int b = 0; b < XR; ++b) {
                    if (b >= mine) break;
                    if (n < C) {
                        const int t = j & 3, p = (j >> 2) & 3, kb = j >> 4;
                        uint4 r = v[b];
                        if (!f16) {
                            if (CAN_F16 && sc != 1.0f) {
                                // times a power of two, exact in bf16
                                auto up = [&](uint32_t w2) {
                                    const uint32_t lo = __float_as_uint(bf16_bits_to_f32(w2 & 0xFFFFu) * sc) >> 16;
                                    const uint32_t hi = __float_as_uint(bf16_bits_to_f32(w2 >> 16) * sc) >> 16;
                                    return lo | (hi << 16);
                                };
                                r = make_uint4(up(r.x), up(r.y), up(r.z), up(r.w));
                            }
                            xf[((kb * 4 + p) * C + n) * 4 + t] =
                                make_uint4(__byte_perm(r.x, r.z, 0x5410), __byte_perm(r.x, r.z, 0x7632),
                                           __byte_perm(r.y, r.w, 0x5410), __byte_perm(r.y, r.w, 0x7632));
                        } else {
                            auto h2 = [&](uint32_t lo_bits, uint32_t hi_bits) {
                                return __floats2half2_rn(bf16_bits_to_f32(lo_bits) * sc,
                                                         bf16_bits_to_f32(hi_bits) * sc);
                            };
                            // r holds x[kk..kk+7] as (x0,x1) (x2,x3) (x4,x5) (x6,x7)
                            const __half2 h04 = h2(r.x & 0xFFFFu, r.z & 0xFFFFu);
                            const __half2 h26 = h2(r.y & 0xFFFFu, r.w & 0xFFFFu);
                            const __half2 h15 = h2(r.x >> 16, r.z >> 16), h37 = h2(r.y >> 16, r.w >> 16);
                            xf[((kb * 4 + p) * C + n) * 4 + t] = make_uint4(
                                *reinterpret_cast<const uint32_t*>(&h04), *reinterpret_cast<const uint32_t*>(&h26),
                                *reinterpret_cast<const uint32_t*>(&h15), *reinterpret_cast<const uint32_t*>(&h37));
                            const float2 f04 = __half22float2(h04), f26 = __half22float2(h26);
                            const float2 f15 = __half22float2(h15), f37 = __half22float2(h37);
                            se += (f04.x + f04.y) + (f26.x + f26.y);
                            so += (f15.x + f15.y) + (f37.x + f37.y);
                        }
                    }
                    j += dj;
                    n += dn;
                    if (j >= per_n) { j -= per_n; ++n; }
                }
                if (f16) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        se += __shfl_xor_sync(0xffffffffu, se, o);
                        so += __shfl_xor_sync(0xffffffffu, so, o);
                    }
                    if (lane == 0) {
                        xsw[warp * 2] = se;
                        xsw[warp * 2 + 1] = so;
                    }
                }
            }
            for (int i = tid; i < 16 * C; i += CT) xzero[i] = make_uint4(0, 0, 0, 0);
            named_barrier(1, CT);

            // bf16: sums of x on the tensor cores -- an all-ones A operand turns
            // each MMA over a staged fragment into column sums (fp32
            // accumulation, as in the main product).  Warps take the (kb, word)
            // pairs round-robin, two at a time on independent accumulators.
            // They are needed only to fold out a fractional zero point, so
            // they are skipped when no row of this CTA has one.
            const bool need_sums = *frac_seen != 0u;
            if (!f16 && need_sums) {
                const uint32_t ones = 0x3F803F80u;   // bf16x2 (1.0, 1.0)
                const uint32_t a1s[4] = {ones, ones, ones, ones};
                float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
                float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
                const int nq = nkb * 4, qstride = bl ? xw_stride : 0;
                for (int q = warp; q < nq; q += 2 * NC) {
                    uint4 b0, b1 = make_uint4(0, 0, 0, 0);
                    if constexpr (PERM) {
                        ldmatrix_x4(xa + q * xs, b0.x, b0.y, b0.z, b0.w);
                        if (q + NC < nq) ldmatrix_x4(xa + (q + NC) * xs, b1.x, b1.y, b1.z, b1.w);
                    } else {
                        b0 = xlane[q * qstride];
                        if (q + NC < nq) b1 = xlane[(q + NC) * qstride];
                    }
                    mma_bf16(s0, a1s, b0.x, b0.y);
                    mma_bf16(s1, a1s, b0.z, b0.w);
                    mma_bf16(s2, a1s, b1.x, b1.y);
                    mma_bf16(s3, a1s, b1.z, b1.w);
                }
                // every row of the product holds the same sums: lanes of row 0
                // own columns 2*t4 and 2*t4 + 1
                if (g == 0) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = 2 * t4 + h;
                        if (c < C) {
                            xsw[(warp * C + c) * 2] = (s0[h] + s1[h]) + (s2[h] + s3[h]);
                            xsw[(warp * C + c) * 2 + 1] = 0.f;
                        }
                    }
                }
                named_barrier(1, CT);
            }   // (fp16: the sums were stored before the last barrier)
            if (tid < C) {
                float se = 0.f, so = 0.f;
                if (f16 || need_sums) {
                    for (int w = 0; w < NC; ++w) {
                        se += xsw[(w * C + tid) * 2];
                        so += xsw[(w * C + tid) * 2 + 1];
                    }
                }
                // the accumulators hold sum (q - zi) x in the units of the
                // staged x: undo its scaling by 2^e (one column only)
                const int emax = static_cast<int>(reinterpret_cast<const uint32_t*>(xsum)[16 + tid] >> 7);
                const int e = f16 ? min(100, 141 - emax) : CAN_F16 ? min(126, max(0, 141 - emax)) : 0;
                const float inv = __int_as_float((127 - e) << 23);   // 2^-e
                xsum[24 + tid] = inv;
                xsum[16 + tid] = 0.0f;
                xsum[tid] = (se + so) * inv;
            }
        }

        // main loop: units of each stage go round-robin to the warps, the
        // rotation carrying over from stage to stage
        const int xkb_stride = bl ? 4 * xw_stride : 0;   // next unit
        const uint32_t mask = dq.mask, mask_hi = dq.mask << 4;
        const int row_off_a = g * pitch + 16 * t4, row_off_b = (g + 8) * pitch + 16 * t4;
        // permuted operand: this lane's ldmatrix row -- column r + 8*(i & 1)
        // of matrix i = lane / 8 (r = lane % 8), 32-k group +(i >> 1); the
        // column groups sit 4*pitch apart, lines of 128 bytes, 32 bytes per column
        const int ldm_col = (lane & 7) + 8 * ((lane >> 3) & 1);
        const uint32_t ldm_off = (ldm_col >> 2) * 4 * pitch + (ldm_col & 3) * 32 + (lane >> 4) * 16;
        int slot = 0, round = 0, first = warp;   // first unit of this warp in the current stage
        const int rows16 = (P.rows_cap + 15) / 16 * 16;
        // this lane's partial sums: warp's rows, row g, columns 2*t4, 2*t4 + 1
        float* const pw_lane = partw + (warp * rows16 + g) * C + 2 * t4;
        // H: fp16 MMAs (one column of x, within fp16's range), else bf16
        auto main_loop = [&](auto mode) {
            constexpr bool H = decltype(mode)::value;
            const uint32_t magic = H ? dq.magic : dq.magic_bf16;
            // nibble -> bf16 128 + q (row layout) or 136 + q (two's complement
            // nibbles of the permuted layout, whose zero point is 0)
            auto unpack = [&](uint32_t v) { return PERM ? pass_flip_or(v, mask, magic) : and_or(v, mask, magic); };
            // what is left above q - zi after the unpack, for local row r: bf16
            // 128 + zi (136 on the permuted layout); fp16 1024 + zi (even k) and
            // the addend -(64 + zi) of the odd-k FMA by 1/16
            auto zconst = [&](int r, uint32_t& ze, uint32_t& zo) {
                if constexpr (PERM) {
                    ze = 0x43084308u;
                    zo = 0u;
                } else if (r >= nrows) {   // rows past the range: never stored
                    ze = H ? 0x64006400u : 0x43004300u;
                    zo = 0xD400D400u;
                } else if constexpr (H) {
                    const uint2 v = *reinterpret_cast<const uint2*>(&zz_s[r]);
                    ze = v.x;
                    zo = v.y;
                } else {
                    ze = zz_s[r].z;
                    zo = 0u;
                }
            };
            constexpr uint32_t kSixteenth = 0x2C002C00u;   // fp16x2 (1/16, 1/16)
            // RT consecutive 16-row tiles at once (RT = 2 only when a tile is
            // one stage): the warp's units of both stages share the x
            // fragments and the per-stage bookkeeping
            auto run = [&](auto rt_tag, int tile) {
                constexpr int RT = decltype(rt_tag)::value;
                uint32_t ze_a[RT], ze_b[RT], zo_a[RT], zo_b[RT];
#pragma unroll
                for (int t = 0; t < RT; ++t) {
                    zconst((tile + t) * 16 + g, ze_a[t], zo_a[t]);
                    zconst((tile + t) * 16 + g + 8, ze_b[t], zo_b[t]);
                }
                float acc[RT][4], acc2[RT][4];
#pragma unroll
                for (int t = 0; t < RT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[t][i] = acc2[t][i] = 0.f;
                for (int ch = 0; ch < nch; ++ch) {
                    const int units = (min(P.kchunk, klen - ch * P.kchunk) + KB - 1) / KB;
                    int sl[RT], rd[RT];
                    {
                        int s2 = slot, r2 = round;
#pragma unroll
                        for (int t = 0; t < RT; ++t) {
                            sl[t] = s2;
                            rd[t] = r2;
                            if (++s2 == NST) { s2 = 0; ++r2; }
                        }
                        slot = s2;
                        round = r2;
                    }
                    bool ok = true;
#pragma unroll
                    for (int t = 0; t < RT; ++t) ok = ok && mbar_wait_fast(bar_full + 8 * sl[t], rd[t] & 1, abort_flag);
                    if (ok) {
                        for (int u = first; u < units; u += NC) {
                            [[maybe_unused]] const uint4* xb = xlane + (ch * (P.kchunk / KB) + u) * xkb_stride;
                            uint32_t wav[RT][4], wbv[RT][4];
#pragma unroll
                            for (int t = 0; t < RT; ++t) {
                                const uint8_t* st = sm + sl[t] * L.stage_bytes;
                                if constexpr (PERM) {
                                    // words of columns g and g+8 for the unit's four 32-k groups
                                    const uint32_t a = smem_u32(st) + ldm_off + u * 256;
                                    ldmatrix_x4(a, wav[t][0], wbv[t][0], wav[t][1], wbv[t][1]);
                                    ldmatrix_x4(a + 128, wav[t][2], wbv[t][2], wav[t][3], wbv[t][3]);
                                } else {
                                    const uint4 wa = *reinterpret_cast<const uint4*>(st + row_off_a + u * 64);
                                    const uint4 wb = *reinterpret_cast<const uint4*>(st + row_off_b + u * 64);
                                    wav[t][0] = wa.x; wav[t][1] = wa.y; wav[t][2] = wa.z; wav[t][3] = wa.w;
                                    wbv[t][0] = wb.x; wbv[t][1] = wb.y; wbv[t][2] = wb.z; wbv[t][3] = wb.w;
                                }
                            }
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                uint4 bx;
                                if constexpr (PERM) {
                                    ldmatrix_x4(xa + ((ch * (P.kchunk / KB) + u) * 4 + w) * xs, bx.x, bx.y, bx.z,
                                                bx.w);
                                } else {
                                    bx = xb[w * xw_stride];
                                }
#pragma unroll
                                for (int t = 0; t < RT; ++t) {
                                    const uint32_t va = wav[t][w], vb = wbv[t][w];
                                    if constexpr (!H) {
                                        const uint32_t a0[4] = {sub_bf16x2(unpack(va), ze_a[t]),
                                                                sub_bf16x2(unpack(vb), ze_b[t]),
                                                                sub_bf16x2(unpack(va >> 4), ze_a[t]),
                                                                sub_bf16x2(unpack(vb >> 4), ze_b[t])};
                                        const uint32_t a1[4] = {sub_bf16x2(unpack(va >> 8), ze_a[t]),
                                                                sub_bf16x2(unpack(vb >> 8), ze_b[t]),
                                                                sub_bf16x2(unpack(va >> 12), ze_a[t]),
                                                                sub_bf16x2(unpack(vb >> 12), ze_b[t])};
                                        mma_bf16(acc[t], a0, bx.x, bx.y);
                                        mma_bf16(acc2[t], a1, bx.z, bx.w);
                                    } else {
                                        // fp16 1024 + q from nibbles 0 and 2 (bits 0-3 of
                                        // each half, after one shift by 8 for nibble 2),
                                        // 1024 + 16q from nibbles 1 and 3 (bits 4-7)
                                        const uint32_t va8 = va >> 8, vb8 = vb >> 8;
                                        const uint32_t a0[4] = {sub_f16x2(and_or(va, mask, magic), ze_a[t]),
                                                                sub_f16x2(and_or(vb, mask, magic), ze_b[t]),
                                                                sub_f16x2(and_or(va8, mask, magic), ze_a[t]),
                                                                sub_f16x2(and_or(vb8, mask, magic), ze_b[t])};
                                        const uint32_t a1[4] = {
                                            fma_f16x2(and_or(va, mask_hi, magic), kSixteenth, zo_a[t]),
                                            fma_f16x2(and_or(vb, mask_hi, magic), kSixteenth, zo_b[t]),
                                            fma_f16x2(and_or(va8, mask_hi, magic), kSixteenth, zo_a[t]),
                                            fma_f16x2(and_or(vb8, mask_hi, magic), kSixteenth, zo_b[t])};
                                        mma_f16(acc[t], a0, bx.x, bx.y);
                                        mma_f16(acc2[t], a1, bx.z, bx.w);
                                    }
                                }
                            }
                        }
                    }
                    // rotate: this warp's first unit of the next stage (the RT
                    // tiles of one step share the unit assignment)
                    first -= units % NC;
                    if (first < 0) first += NC;
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int t = 0; t < RT; ++t) mbar_arrive(bar_empty + 8 * sl[t]);
                    }
                }
                const int c0 = 2 * t4, c1 = 2 * t4 + 1;
#pragma unroll
                for (int t = 0; t < RT; ++t) {
                    if (P.perwarp) {
                        // this warp's partial of the tile; warps are added at the end
                        float* pw = pw_lane + (tile + t) * 16 * C;
                        if (c0 < C) {
                            pw[0] = acc[t][0] + acc2[t][0];
                            pw[8 * C] = acc[t][2] + acc2[t][2];
                        }
                        if (c1 < C) {
                            pw[1] = acc[t][1] + acc2[t][1];
                            pw[8 * C + 1] = acc[t][3] + acc2[t][3];
                        }
                    } else {
                        // tile partials, added in warp order now (bounded shared memory)
                        const int tl = tile + t;
                        float* rbuf = red + ((tl & 1) * NC + warp) * 16 * C;
                        if (c0 < C) {
                            rbuf[g * C + c0] = acc[t][0] + acc2[t][0];
                            rbuf[(g + 8) * C + c0] = acc[t][2] + acc2[t][2];
                        }
                        if (c1 < C) {
                            rbuf[g * C + c1] = acc[t][1] + acc2[t][1];
                            rbuf[(g + 8) * C + c1] = acc[t][3] + acc2[t][3];
                        }
                        named_barrier(1, CT);
                        for (int i = tid; i < 16 * C; i += CT) {
                            const int r = i / C;
                            if (tl * 16 + r < nrows) {
                                float v = 0.f;
                                for (int w = 0; w < NC; ++w) v += red[((tl & 1) * NC + w) * 16 * C + i];
                                const int c = i - r * C;
                                part[(tl * 16) * C + i] = v * xsum[24 + c];
                            }
                        }
                    }
                }
            };
            int tile = 0;
            while (tile < ntiles) {
                if (nch == 1 && P.perwarp && NST >= 2 && tile + 1 < ntiles) {
                    run(std::integral_constant<int, 2>{}, tile);
                    tile += 2;
                } else {
                    run(std::integral_constant<int, 1>{}, tile);
                    tile += 1;
                }
            }
        };
        if constexpr (CAN_F16) {
            if (f16) main_loop(std::true_type{});
            else main_loop(std::false_type{});
        } else {
            main_loop(std::false_type{});
        }
        const bool row_regs = C == 1 && S == 1;   // rows finished by the threads holding their s, z
        if (!row_regs) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = tid + j * CT;
                if (i < nrows) sz[i] = make_float2(sc_pf[j], z_pf[j] - static_cast<float>(zint(z_pf[j])));
            }
            for (int i = tid + 2 * CT; i < nrows; i += CT) {
                const float z = load_z(r0 + i);
                sz[i] = make_float2(load_s(r0 + i), z - static_cast<float>(zint(z)));
            }
        }
        if (row_regs) {
            // one column, no K split: thread tid finishes rows tid, tid + CT
            // (scale and zero point still in its registers), then every
            // further CT-th row (loaded again)
            named_barrier(1, CT);
            auto finish = [&](int r, float sc, float z) {
                float v;
                if (P.perwarp) {
                    v = 0.f;
                    for (int w = 0; w < NC; ++w) v += partw[static_cast<size_t>(w) * rows16 + r];
                    v *= xsum[24];
                } else {
                    v = part[r];
                }
                const float zf = z - static_cast<float>(zint(z));
                d[r0 + r] = __float2bfloat16_rn(sc * fmaf(-zf, xsum[0], v));
            };
            if (tid < nrows) finish(tid, sc_pf[0], z_pf[0]);
            if (tid + CT < nrows) finish(tid + CT, sc_pf[1], z_pf[1]);
            for (int r = tid + 2 * CT; r < nrows; r += CT) finish(r, load_s(r0 + r), load_z(r0 + r));
        } else if (S == 1) {
            // no K split: add the warps' partials (or take the tile sums),
            // fold the zero point, scale and store straight away
            named_barrier(1, CT);
            for (int i = tid; i < nrows * C; i += CT) {
                const int r = i / C, c = i - r * C;
                float v;
                if (P.perwarp) {
                    v = 0.f;
                    for (int w = 0; w < NC; ++w) v += partw[static_cast<size_t>(w) * rows16 * C + i];
                    v *= xsum[24 + c];
                } else {
                    v = part[i];
                }
                const float2 s_z = sz[r];
                d[static_cast<int64_t>(c) * N + r0 + r] = __float2bfloat16_rn(s_z.x * fmaf(-s_z.y, xsum[c], v));
            }
        } else if (P.perwarp) {
            named_barrier(1, CT);
            for (int i = tid; i < nrows * C; i += CT) {
                float v = 0.f;
                for (int w = 0; w < NC; ++w) v += partw[static_cast<size_t>(w) * rows16 * C + i];
                const int c = i % C;
                part[i] = v * xsum[24 + c];
            }
        }
    }
    if (S == 1) return;   // (the producer has drained its copies)
    __syncthreads();

    // part[] holds sum_k q x per (row, column) over this CTA's K-slice, in
    // the units of x (offset folded out, scaling undone); xsum[0, C) the
    // slice's sum of x.  Rank ks owns rows ks, ks+S, ...: every rank pushes
    // its partials of the rows the others own, and its sums of x, into their
    // shared memory (st.async, completing bytes on the owner's barrier); an
    // owner adds the S slices in rank order, folds the zero point, scales
    // and stores.  No CTA reads another's shared memory, so CTAs do not meet
    // at exit; each waits (bounded) until every push into it has landed.
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // every peer is initialised
    float* rcv = reinterpret_cast<float*>(sm + L.rcv);
    float* rxs = reinterpret_cast<float*>(sm + L.rxs);
    const int own_cap = (P.rows_cap + S - 1) / S;
    {
        const uint32_t rcv_l = smem_u32(rcv), rxs_l = smem_u32(rxs);
        for (int j = tid; j < nrows * C; j += THREADS) {
            const int i = j / C, c = j - i * C;
            const int owner = i % S;
            if (owner == ks) continue;
            const uint32_t dst = map_cluster(rcv_l + ((ks * own_cap + i / S) * C + c) * 4, owner);
            asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(dst),
                         "r"(__float_as_uint(part[j])), "r"(map_cluster(bar_rcv, owner))
                         : "memory");
        }
        if (tid < C) {
            for (int r = 0; r < S; ++r) {
                if (r == ks) continue;
                asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
                                 map_cluster(rxs_l + (ks * 8 + tid) * 4, r)),
                             "r"(__float_as_uint(xsum[tid])), "r"(map_cluster(bar_rcv, r))
                             : "memory");
            }
        }
    }
    if (!mbar_wait(bar_rcv, 0, abort_flag)) {
        mbar_drain(bar_rcv, 0);   // a slow peer's push may still be on its way
        return;
    }
    const int my_rows = nrows > ks ? (nrows - ks + S - 1) / S : 0;
    for (int j = tid; j < my_rows * C; j += THREADS) {
        const int il = j / C, c = j - il * C, i = ks + S * il;
        float sum = 0.f, xt = 0.f;
        for (int r = 0; r < S; ++r) {
            sum += r == ks ? part[i * C + c] : rcv[(r * own_cap + il) * C + c];
            xt += r == ks ? xsum[c] : rxs[r * 8 + c];
        }
        const float2 s_z = sz[i];
        d[static_cast<int64_t>(c) * N + r0 + i] = __float2bfloat16_rn(s_z.x * fmaf(-s_z.y, xt, sum));
    }
}

}  // namespace gtma

namespace {

using namespace gtma;

constexpr int kSmemMax = W4_GEMV_SMEM;
// x fragments: at most XR_MAX 16-byte entries per consumer thread (the
// staging pass keeps them in registers)
constexpr size_t kXfBudget = static_cast<size_t>(XR_MAX) * CT * 16;

// Pipeline shape for (N, K, C) on `sms` SMs; nst == 0 if nothing fits.
template <int C, bool PERM>
Plan make_plan(int N, int K, int sms, int max_clusters_for_S /* 0: unknown */, int S_forced) {
    Plan P{};
    const int tm = (!PERM && K % 128 == 0) ? 1 : 0;   // rows are whole 64-byte chunks
    const int sgran = (tm || PERM) ? 128 : 32;
    auto slice_of = [&](int s) { return ((K + s - 1) / s + sgran - 1) / sgran * sgran; };
    auto xf_bytes = [&](int s) { return static_cast<size_t>((slice_of(s) + KB - 1) / KB) * 16 * C * 16; };
    int S = 1;
#ifdef W4_GEMV_FORCE_S
    if (!S_forced) S_forced = W4_GEMV_FORCE_S;
#endif
    if (S_forced) {
        S = S_forced;
    } else {
        while (S < 8 && xf_bytes(S) > kXfBudget) S *= 2;
        // one more split halves every CTA's x staging; worth it when the staging
        // holds more than 8 entries per consumer thread and a stage still gives
        // every consumer warp 2.5 units or more (N=5120 K=17280 C=4: 15.2 ->
        // 14.4 us; thinner stages cost more than the staging saved)
        if (!PERM && S < 8 && xf_bytes(S) > static_cast<size_t>(8) * CT * 16 && 2 * (slice_of(2 * S) / KB) >= 5 * NC)
            S *= 2;
    }
    P.S = S;
    P.kslice = slice_of(S);
    // Row groups own whole 16-row tiles (a partial tile costs a full stage of
    // consumer time, so a finer split would not shorten the busiest group),
    // one group (or cluster) per SM: every SM streams, and the CTAs with one
    // tile fewer finish early, letting the next launch's CTAs in (measured
    // faster on every workload shape than the smallest grid with the same
    // busiest group).
    const int64_t tiles = (static_cast<int64_t>(N) + 15) / 16;
    int groups = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(sms / S, tiles)));
    if (max_clusters_for_S > 0) groups = std::min(groups, max_clusters_for_S);
    const int64_t per = std::max<int64_t>(1, (tiles + groups - 1) / groups);
#ifdef W4_GEMV_MINGRID
    groups = static_cast<int>(std::max<int64_t>(1, (tiles + per - 1) / per));
#endif
    P.groups = groups;
    P.rows_cap = static_cast<int>(16 * std::max<int64_t>(1, per));
    // stage: one 16-row tile over a K-chunk
    {
        const int nch0 = (P.kslice + KCHUNK_MAX - 1) / KCHUNK_MAX;  // chunks of about equal size
        P.kchunk = ((P.kslice + nch0 - 1) / nch0 + KB - 1) / KB * KB;
    }
    P.dense = (!PERM && S == 1 && P.kchunk >= K) ? 1 : 0;
    P.tmap = tm;
    if (PERM) {
        // four column groups of kchunk/64 lines each, 16 mod 128 bytes apart;
        // x rows of whole units, 16 mod 128 bytes apart
        P.pitch = 32 * (P.kchunk / 64) + 4;
        P.xpitch = (P.kslice + KB - 1) / KB * KB * 2 + 16;
    } else if (tm) {
        P.nbox = (P.kchunk / 128) | 1;
        P.pitch = P.nbox * 64;
    } else if (P.dense) {
        P.pitch = K / 2;
    } else {
        const int seg = P.kchunk / 2;
        P.pitch = (seg + 127) / 128 * 128 + 64;   // 64 mod 128: conflict-free fragment loads
    }
    // prefer per-warp partials (no per-tile barrier) when they leave room
    // for at least 3 stages; otherwise reduce each tile across warps at once
    for (int pw = 1; pw >= 0; --pw) {
        P.perwarp = pw;
        P.nst = MAX_NST;
        while (P.nst >= 2 && make_layout(C, P).total + kSmemAlign > kSmemMax) --P.nst;
        if (P.nst >= (pw ? 3 : 2)) return P;
    }
    P.nst = 0;
    return P;
}

template <int C, bool PERM>
w4_status launch_gemv_tma_t(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N,
                            int K, cudaStream_t stream) {
    const int sms = sm_count();
    if (sms <= 0) return W4_ERR_CUDA;
    Plan P = make_plan<C, PERM>(N, K, sms, 0, 0);
    if (P.nst == 0) return W4_ERR_SHAPE;
    auto kern = gemv_tma_kernel<C, PERM>;
    static int smem_set[64];
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = ensure_smem_limit(kern, make_layout(C, P).total + kSmemAlign, smem_set);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    if (P.S > 1) {
        // every cluster must be resident at once: cap the row groups by the
        // number of clusters the GPCs can hold together
        static int max_clusters[64][4];
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W4_ERR_CUDA;
        const int si = P.S == 2 ? 0 : P.S == 4 ? 1 : 2;
        if (max_clusters[dev][si] == 0) {
            cfg.gridDim = dim3(P.S * P.groups, 1, 1);
            cfg.dynamicSmemBytes = make_layout(C, P).total + kSmemAlign;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return W4_ERR_CUDA;
            max_clusters[dev][si] = n;
        }
        P = make_plan<C, PERM>(N, K, sms, max_clusters[dev][si], P.S);
        if (P.nst == 0) return W4_ERR_SHAPE;
        e = ensure_smem_limit(kern, make_layout(C, P).total + kSmemAlign, smem_set);
        if (e != cudaSuccess) return W4_ERR_CUDA;
    }
    cfg.gridDim = dim3(P.S * P.groups, 1, 1);
    cfg.dynamicSmemBytes = make_layout(C, P).total + kSmemAlign;
    CUtensorMap tm16, tm4;
    memset(&tm16, 0, sizeof(tm16));
    memset(&tm4, 0, sizeof(tm4));
    if (P.tmap) {
        auto encode = tensor_map_encoder();
        if (!encode) return W4_ERR_CUDA;
        cuuint64_t dims[3] = {8, static_cast<cuuint64_t>(K / 128), static_cast<cuuint64_t>(N)};
        cuuint64_t strides[2] = {64, static_cast<cuuint64_t>(K / 2)};
        cuuint32_t estr[3] = {1, 1, 1};
        for (int b = 0; b < 2; ++b) {
            cuuint32_t box[3] = {8, static_cast<cuuint32_t>(P.nbox), b == 0 ? 16u : 4u};
            if (encode(b == 0 ? &tm16 : &tm4, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<void*>(qw), dims, strides,
                       box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return W4_ERR_CUDA;
        }
    }
    // row layout: (v & 0x000F000F) | 0x43004300; permuted (two's complement):
    // pass bits 0-2, invert bit 3, set the exponent of 128.0
    const MaskMagic dq = PERM      ? MaskMagic{0x43074307u, 0x43084308u, 0x43084308u}
                         : C == 1 ? MaskMagic{0x000F000Fu, 0x64006400u, 0x43004300u}   // fp16 1024 + q
                                  : MaskMagic{0x000F000Fu, 0x43004300u, 0x43004300u};  // bf16 128 + q
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint8_t*>(qw), scale, zero,
                           static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(d), N, K, P, dq, tm16,
                           tm4);
    return launch_status(e);
}

}  // namespace

// bf16 GEMV, TMA-fed tensor-core path; requires K % 32 == 0 (16-byte rows).
w4_status run_gemv_tma(const void* qw, const void* scale, const void* zero, const void* x, void* d, int N, int K,
                       int C, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_gemv_tma_t<1, false>(qw, scale, zero, x, d, N, K, stream);
        case 2: return launch_gemv_tma_t<2, false>(qw, scale, zero, x, d, N, K, stream);
        case 3: return launch_gemv_tma_t<3, false>(qw, scale, zero, x, d, N, K, stream);
        case 4: return launch_gemv_tma_t<4, false>(qw, scale, zero, x, d, N, K, stream);
        case 5: return launch_gemv_tma_t<5, false>(qw, scale, zero, x, d, N, K, stream);
        case 6: return launch_gemv_tma_t<6, false>(qw, scale, zero, x, d, N, K, stream);
        case 7: return launch_gemv_tma_t<7, false>(qw, scale, zero, x, d, N, K, stream);
        case 8: return launch_gemv_tma_t<8, false>(qw, scale, zero, x, d, N, K, stream);
        default: return W4_ERR_SHAPE;
    }
}

// bf16 GEMV over permute_int4's output; requires K % 64 == 0, N % 4 == 0.
w4_status run_gemv_permuted(const void* permuted, const float* scale, const void* x, void* d, int N, int K, int C,
                            cudaStream_t stream) {
    switch (C) {
        case 1: return launch_gemv_tma_t<1, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 2: return launch_gemv_tma_t<2, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 3: return launch_gemv_tma_t<3, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 4: return launch_gemv_tma_t<4, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 5: return launch_gemv_tma_t<5, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 6: return launch_gemv_tma_t<6, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 7: return launch_gemv_tma_t<7, true>(permuted, scale, nullptr, x, d, N, K, stream);
        case 8: return launch_gemv_tma_t<8, true>(permuted, scale, nullptr, x, d, N, K, stream);
        default: return W4_ERR_SHAPE;
    }
}

int take_device_error_gemv() { return take_unit_device_error(); }
int set_wait_limit_gemv(long long clocks) { return set_unit_wait_limit(clocks); }
int set_short_first_stage_gemv(int on) {
    const int v = on ? 1 : 0;
    return cudaMemcpyToSymbol(gtma::g_short_first_stage, &v, sizeof(v)) == cudaSuccess ? 0 : -1;
}

}  // namespace w4
