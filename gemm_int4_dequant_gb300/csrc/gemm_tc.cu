// gemm_tc.cu -- large-M bf16 x int4 dequant GEMM on the 5th-generation
// (tcgen05) tensor cores of sm_103a.
//
//   C[m][n] = scale[n] * sum_k A[m][k] * (u[k][n] - zero[n])
//
// (page "int4 gemm kernel", the matmul_bf16_int4 example: A (M,K) bf16 and B
// packed (K/2, N) int8 with the low nibble for even k; one packed k-tile of B
// feeds an A k-tile twice as long.)
//
// Persistent CTA pairs: each thread-block cluster of two CTAs (two SMs)
// computes 256 x 256 output tiles (tile, tile + pairs, ...) with
// tcgen05.mma.cta_group::2 (M256 N256 K16).  CTA r holds A rows
// [128r, 128r+128) and B columns [128r, 128r+128) of a tile in its shared
// memory and the pair's MMA reads both halves, so each SM loads, dequantises
// and serves only half of B per FLOP.  Per CTA, 14 warps:
//   warp 0       TMA producer: A tile [128 x 64] bf16 (128B-swizzled, K-major)
//                and the packed B half [32 x 128] bytes, one mbarrier per stage,
//                running across tile boundaries;
//   warp 1       TMEM allocator (both CTAs); in the even CTA the MMA issuer (one
//                thread): 4 MMAs per k-tile into one of two fp32 accumulators in
//                TMEM (tiles alternate), the commit frees the stage in both CTAs;
//                in the odd CTA the forwarder of "stage ready" to the even CTA;
//   warps 2..9   dequant: packed bytes -> (u - zero) bf16, written straight into
//                the canonical 128B-swizzled MN-major operand layout;
//   warps 10..13 epilogue, one per TMEM lane quarter: tcgen05.ld of the
//                finished accumulator's 128 rows, * scale, -> bf16, then the
//                accumulator is handed back to the MMA issuer; the epilogue of
//                one tile overlaps the main loop of the next.
// Inside every group of four columns the shared-memory (and so TMEM) column
// order is n0 n2 n1 n3: one mask of a packed 32-bit word then yields the
// nibbles of bytes 0 and 2 (or 1 and 3) as a bf16 pair, so unpacking eight
// weights costs three shifts and four three-input logic ops.  The epilogue
// puts the columns back in order.
// Every wait is bounded; on timeout the kernel records an error code in a
// device word (w4_device_error), stops issuing work, drains and frees TMEM.
//
// The kernel is a template over the format of B:
//   FMT_INT4  the packed uint4 [K/2][N] above, bf16 scale and zero point;
//   FMT_INT8  the symmetric int8 matrix of quantize_int8 (q[K][N], fp32
//             scale per column, no zero point): B tiles of 64 rows x 128
//             bytes, five stages; each int8 becomes bf16 exactly through the
//             float 2^23 + (q + 128) built by a byte permute (bf16's seven
//             fraction bits cannot hold q + 128 at one exponent);
//   FMT_PERM  permute_int4's output (page "[PHI] add int4 weight only quant
//             kernel ...": two's complement nibbles, fp32 scale, no zero
//             point).  A 64-k tile of a group of four columns is exactly one
//             128-byte line of that layout (32 bytes a column), so the tile's
//             32 groups arrive as one 3-D TMA box, 128B-swizzled.  In word q
//             of a column's 32 bytes, byte b holds the nibbles of
//             k = 32 (q / 4) + 2 (q % 4) + {0, 8} (b = 0), {16, 24} (b = 1),
//             {1, 9} (b = 2), {17, 25} (b = 3), low nibble first (P1's byte
//             permute and nibble swap).

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace w4 {

namespace gemm {

using namespace ptx;

// Test switch (w4_selftest_configure): when set, the producer announces 16
// bytes more than it copies for its first stage, so that stage's wait runs
// out and the error path (error word, abort, drain, TMEM freed) runs
// without any bad access.  Always 0 in normal use.
static __device__ int g_short_first_stage;

constexpr int BM = 128;                      // A rows per CTA (the pair covers 256)
constexpr int BN = 256;                      // tile columns (the pair's MMA N)
constexpr int BNH = BN / 2;                  // B columns held by each CTA
constexpr int BK = 64;
constexpr int THREADS = 448;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int BD_BYTES = BK * BNH * 2;       // 16 KB dequantised

// Shared-memory layout per B format: packed int4 (4 KB a stage, six
// stages) or int8 (8 KB a stage, five stages).
constexpr int FMT_INT4 = 0, FMT_INT8 = 1, FMT_PERM = 2;

template <int FMT>
struct Lay {
    static constexpr bool I8 = FMT == FMT_INT8;
    static constexpr int STAGES = I8 ? 5 : 6;
    static constexpr int BP_BYTES = I8 ? BK * BNH : (BK / 2) * BNH;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_BD = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_BP = OFF_BD + STAGES * BD_BYTES;
    static constexpr int OFF_BAR = OFF_BP + STAGES * BP_BYTES;
    static constexpr int NUM_BARS = 4 * STAGES + 4;
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
    static constexpr int SMEM_BYTES = OFF_ABORT + 4 + 1024;   // slack to align the base to 1 KB
};
constexpr uint32_t TMEM_COLS = 512;            // two accumulators of 256 columns
constexpr int EPI_WARP0 = 10;                   // warps 10..13
constexpr int DEQ_WARPS = 8;
constexpr int DEQ_THREADS = DEQ_WARPS * 32;

// Instruction descriptor, kind::f16: D fp32, A bf16 K-major, B bf16 MN-major,
// N = 256, M = 256 (CTA pair).
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>((2 * BM) >> 4) << 24);

// Byte offset of element (k, n) of this CTA's dequantised B half: atoms of 8
// k-rows x 64 n (1 KB, 16-byte chunks XOR-swizzled by k % 8), atom (n/64,
// k/8) at ((n/64) * (BK/8) + k/8) KB.  n is a multiple of 8 (one 16-byte chunk).
__device__ __forceinline__ uint32_t bd_offset(int k, int n) {
    const int atom = (n >> 6) * (BK / 8) + (k >> 3);
    const int r = k & 7, chunk = (n & 63) >> 3;
    return static_cast<uint32_t>(atom * 1024 + r * 128 + ((chunk ^ r) << 4));
}

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// One packed word (bytes b0..b3 = columns c0..c3; low nibble = even k) ->
// bf16 pairs in shared-memory column order (c0, c2) and (c1, c3):
// e0/e1 for the even k, o0/o1 for the odd k, each 128 + u.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t& e0, uint32_t& e1, uint32_t& o0, uint32_t& o1) {
    const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;  // bf16x2 (128, 128)
    e0 = and_or(w, mask, magic);
    e1 = and_or(w >> 8, mask, magic);
    o0 = and_or(w >> 4, mask, magic);
    o1 = and_or(w >> 12, mask, magic);
}

// Four int8 (one word) -> bf16 pairs in shared-memory column order (c0, c2)
// and (c1, c3), exact.
__device__ __forceinline__ void i8_word_to_bf16(uint32_t w, uint32_t& p02, uint32_t& p13) {
    const uint32_t wx = w ^ 0x80808080u;
    float f[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | j)) - 8388736.0f;
    const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[2]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f[1], f[3]);
    p02 = *reinterpret_cast<const uint32_t*>(&a);
    p13 = *reinterpret_cast<const uint32_t*>(&b);
}

// 3-D tiled TMA load into this CTA's shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

template <int FMT>
__global__ void __launch_bounds__(THREADS, 1)
gemm_w4_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  const void* __restrict__ scale_p, const __nv_bfloat16* __restrict__ zero,
                  __nv_bfloat16* __restrict__ C, int M, int N, int K, int tiles_n, int num_tiles) {
    using L = Lay<FMT>;
    constexpr bool I8 = FMT == FMT_INT8, PERM = FMT == FMT_PERM;
    constexpr int STAGES = L::STAGES, BP_BYTES = L::BP_BYTES;
    constexpr int OFF_A = L::OFF_A, OFF_BD = L::OFF_BD, OFF_BP = L::OFF_BP, OFF_BAR = L::OFF_BAR;
    constexpr int OFF_TMEM_SLOT = L::OFF_TMEM_SLOT, OFF_ABORT = L::OFF_ABORT;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + OFF_BAR;
    auto full_tma = [&](int s) { return bar0 + 8u * s; };
    auto full_deq = [&](int s) { return bar0 + 8u * (STAGES + s); };     // this CTA's dequant warps
    auto empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto peer_deq = [&](int s) { return bar0 + 8u * (3 * STAGES + s); };  // even CTA: the odd CTA's stage is ready
    auto acc_full = [&](int b) { return bar0 + 8u * (4 * STAGES + b); };  // accumulator b finished
    auto acc_empty = [&](int b) { return bar0 + 8u * (4 * STAGES + 2 + b); };   // even CTA: b read out by both
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sbase + OFF_TMEM_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + OFF_ABORT);

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());     // 0: issues the pair's MMAs
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_kt = K / BK;
    const int my_tiles = pair < num_tiles ? (num_tiles - pair + pairs - 1) / pairs : 0;
    const int total_kt = my_tiles * num_kt;   // k-tiles this pair works through (stage ring position)
    // tile it of this pair: row block, column block (column blocks fastest, so
    // concurrently running pairs share rows of A)
    auto tile_m = [&](int it) { return (pair + it * pairs) / tiles_n; };
    auto tile_n = [&](int it) { return (pair + it * pairs) % tiles_n; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_tma(s), 1);
            mbar_init(full_deq(s), DEQ_WARPS);
            mbar_init(empty(s), 1);
            mbar_init(peer_deq(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full(b), 1);
            mbar_init(acc_empty(b), 2 * 4);   // four epilogue warps in each CTA
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), TMEM_COLS);
    tc_fence_before();
    cluster.sync();   // both CTAs' barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_a) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_b) : "memory");
            int issued = 0;
            bool ok = true;
            const uint32_t short0 = g_short_first_stage ? 16u : 0u;
            for (int it = 0; it < my_tiles && ok; ++it) {
                const int mr = tile_m(it) * (2 * BM) + rank * BM;   // this CTA's first A row
                const int nh = tile_n(it) * BN + rank * BNH;        // this CTA's first B column
                // an A or B half wholly outside the matrix (ragged M or N) is not
                // copied: its rows / columns of the tile are never stored
                const bool load_a = mr < M, load_b = nh < N;
                const uint32_t bytes = (load_a ? A_BYTES : 0) + (load_b ? BP_BYTES : 0);
                for (int kt = 0; kt < num_kt; ++kt) {
                    const int g = it * num_kt + kt, s = g % STAGES, round = g / STAGES;
                    if (round > 0 && !mbar_wait_fast(empty(s), (round - 1) & 1, abort_flag)) { ok = false; break; }
                    if (*abort_flag) { ok = false; break; }
                    mbar_arrive_expect_tx(full_tma(s), bytes + (g == 0 ? short0 : 0u));
                    if (load_a) tma_load_2d(base + OFF_A + s * A_BYTES, &tmap_a, kt * BK, mr, full_tma(s));
                    if (load_b && PERM)
                        tma_load_3d(base + OFF_BP + s * BP_BYTES, &tmap_b, 0, kt, nh / 4, full_tma(s));
                    else if (load_b)
                        tma_load_2d(base + OFF_BP + s * BP_BYTES, &tmap_b, nh, kt * (I8 ? BK : BK / 2), full_tma(s));
                    issued = g + 1;
                }
            }
            // the last copies may still be landing if a consumer aborted
            for (int g = max(0, issued - STAGES); g < issued; ++g)
                mbar_drain(full_tma(g % STAGES), (g / STAGES) & 1);
        }
    } else if (warp == 1 && rank == 1) {
        // ---------------- odd CTA: forward "stage ready" to the even CTA ----------------
        // The stage data are this CTA's shared memory (TMA-written A, the
        // dequant warps' B half): a release fence restricted to shared::cta
        // at cluster scope, then a relaxed remote arrive per stage.  Stages
        // that became ready meanwhile share one fence.
        if (lane == 0) {
            const uint32_t remote0 = map_cluster(peer_deq(0), 0);
            int g = 0;
            while (g < total_kt) {
                if (!mbar_wait_fast(full_deq(g % STAGES), (g / STAGES) & 1, abort_flag)) break;
                int end = g + 1;
                while (end < total_kt && mbar_try_wait(full_deq(end % STAGES), (end / STAGES) & 1)) ++end;
                fence_release_smem_cluster();
                for (; g < end; ++g) mbar_arrive_cluster_relaxed(remote0 + 8u * (g % STAGES));
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (even CTA) ----------------
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < my_tiles && ok; ++it) {
                const int b = it & 1;
                // accumulator b was read out by both CTAs' epilogues (tile it - 2)
                if (it >= 2 && !mbar_wait_cluster(acc_empty(b), ((it >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int kt = 0; kt < num_kt; ++kt) {
                    const int g = it * num_kt + kt, s = g % STAGES, round = g / STAGES;
                    ok = mbar_wait_fast(full_deq(s), round & 1, abort_flag) &&
                         mbar_wait_cluster(peer_deq(s), round & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a_addr = base + OFF_A + s * A_BYTES;
                    const uint32_t b_addr = base + OFF_BD + s * BD_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // A: K-major SW128, +32 B per 16-element k step; SBO = 8 rows * 128 B.
                        const uint64_t adesc = sw128_desc(a_addr + kk * 32, 16, 1024);
                        // B: MN-major SW128, k-groups of 8 rows 1 KB apart (SBO),
                        // 64-column atoms (BK/8) KB apart (LBO).
                        const uint64_t bdesc = sw128_desc(b_addr + kk * 2 * 1024, (BK / 8) * 1024, 1024);
                        umma_bf16_pair(d_tmem, adesc, bdesc, kIdesc, (kt > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit_pair(empty(s), 0x3);
                }
                if (ok) umma_commit_pair(acc_full(b), 0x3);
            }
        }
    } else if (warp < EPI_WARP0 && I8) {
        // ---------------- dequant, int8 (warps 2..9) ----------------
        // thread: 8 of this CTA's 128 columns, every 16th of the tile's 64 rows
        const int t = threadIdx.x - 64;          // 0..255
        const int nl = (t & 15) * 8;
        const int k_lane = t >> 4;               // 0..15
        bool ok = true;
        for (int it = 0; it < my_tiles && ok; ++it) {
            for (int kt = 0; kt < num_kt; ++kt) {
                const int g = it * num_kt + kt, s = g % STAGES, round = g / STAGES;
                if (round > 0 && !mbar_wait_fast(empty(s), (round - 1) & 1, abort_flag)) { ok = false; break; }
                if (!mbar_wait_fast(full_tma(s), round & 1, abort_flag)) { ok = false; break; }
                const uint8_t* bp = sbase + OFF_BP + s * BP_BYTES;
                uint8_t* bd = sbase + OFF_BD + s * BD_BYTES;
#pragma unroll
                for (int i = 0; i < BK / 16; ++i) {
                    const int k = k_lane + 16 * i;
                    const uint2 v = *reinterpret_cast<const uint2*>(bp + k * BNH + nl);
                    uint32_t h[4];
                    i8_word_to_bf16(v.x, h[0], h[1]);
                    i8_word_to_bf16(v.y, h[2], h[3]);
                    *reinterpret_cast<uint4*>(bd + bd_offset(k, nl)) = make_uint4(h[0], h[1], h[2], h[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_deq(s));
            }
        }
    } else if (warp < EPI_WARP0 && PERM) {
        // ---------------- dequant, permuted layout (warps 2..9) ----------------
        // warp w takes groups 8 (w % 4) .. + 7 and words 4 (w / 4) .. + 3 of
        // their lines; with the 128B swizzle the 32 lanes read 32 different
        // banks for each column
        const int dw = warp - 2;
        const int G = 8 * (dw & 3) + (lane & 7);   // column group (4 columns) of this CTA's 32
        const int q = 4 * (dw >> 2) + (lane >> 3); // word of each column's 32 bytes
        const uint32_t flip = 0x43084308u, pass = 0x43074307u;   // 136 + q, q two's complement
        // k of the low / high nibble of byte b of word q
        const int kb = 32 * (q >> 2) + 2 * (q & 3);
        const int klo[4] = {kb, kb + 16, kb + 1, kb + 17};
        bool ok = true;
        for (int it = 0; it < my_tiles && ok; ++it) {
            for (int kt = 0; kt < num_kt; ++kt) {
                const int g = it * num_kt + kt, s = g % STAGES, round = g / STAGES;
                if (round > 0 && !mbar_wait_fast(empty(s), (round - 1) & 1, abort_flag)) { ok = false; break; }
                if (!mbar_wait_fast(full_tma(s), round & 1, abort_flag)) { ok = false; break; }
                const uint8_t* row = sbase + OFF_BP + s * BP_BYTES + 128 * G;
                uint8_t* bd = sbase + OFF_BD + s * BD_BYTES;
                uint32_t w[4];
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    w[c] = *reinterpret_cast<const uint32_t*>(row + 16 * ((2 * c + (q >> 2)) ^ (G & 7)) + 4 * (q & 3));
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const uint32_t sel = static_cast<uint32_t>(b) | (static_cast<uint32_t>(4 + b) << 8);
                    const uint32_t z02 = __byte_perm(w[0], w[2], sel), z13 = __byte_perm(w[1], w[3], sel);
                    const uint32_t lo02 = bsub2(pass_flip_or(z02, pass, flip), flip);
                    const uint32_t lo13 = bsub2(pass_flip_or(z13, pass, flip), flip);
                    const uint32_t hi02 = bsub2(pass_flip_or(z02 >> 4, pass, flip), flip);
                    const uint32_t hi13 = bsub2(pass_flip_or(z13 >> 4, pass, flip), flip);
                    const int k0 = klo[b], k1 = klo[b] + 8;
                    *reinterpret_cast<uint2*>(bd + bd_offset(k0, 8 * (G >> 1)) + 8 * (G & 1)) = make_uint2(lo02, lo13);
                    *reinterpret_cast<uint2*>(bd + bd_offset(k1, 8 * (G >> 1)) + 8 * (G & 1)) = make_uint2(hi02, hi13);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_deq(s));
            }
        }
    } else if (warp < EPI_WARP0) {
        // ---------------- dequant (warps 2..9) ----------------
        const int t = threadIdx.x - 64;          // 0..255
        const int nl = (t & 15) * 8;             // 8 of this CTA's 128 columns
        const int kp_lane = t >> 4;              // 0..15
        const uint32_t k128 = 0x43004300u;
        bool ok = true;
        for (int it = 0; it < my_tiles && ok; ++it) {
            const int nh = tile_n(it) * BN + rank * BNH;
            // zero-point pairs in shared-memory column order: (z0,z2) (z1,z3) (z4,z6) (z5,z7).
            // Fast path: 128 + z exact in bf16 (integer zero points) -> one subtract.
            uint32_t zz[4], zraw[4];
            bool fast = true;
            {
                float zf[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int n = nh + nl + j;
                    zf[j] = n < N ? __bfloat162float(zero[n]) : 0.f;
                }
                const int pa[4] = {0, 1, 4, 5}, pb[4] = {2, 3, 6, 7};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a = 128.0f + zf[pa[j]], c = 128.0f + zf[pb[j]];
                    const __nv_bfloat162 h = __floats2bfloat162_rn(a, c);
                    fast = fast && __low2float(h) == a && __high2float(h) == c;
                    zz[j] = *reinterpret_cast<const uint32_t*>(&h);
                    const __nv_bfloat162 r = __floats2bfloat162_rn(zf[pa[j]], zf[pb[j]]);
                    zraw[j] = *reinterpret_cast<const uint32_t*>(&r);
                }
            }
            for (int kt = 0; kt < num_kt; ++kt) {
                const int g = it * num_kt + kt, s = g % STAGES, round = g / STAGES;
                if (round > 0 && !mbar_wait_fast(empty(s), (round - 1) & 1, abort_flag)) { ok = false; break; }
                if (!mbar_wait_fast(full_tma(s), round & 1, abort_flag)) { ok = false; break; }
                const uint8_t* bp = sbase + OFF_BP + s * BP_BYTES;
                uint8_t* bd = sbase + OFF_BD + s * BD_BYTES;
#pragma unroll
                for (int i = 0; i < (BK / 2) / 16; ++i) {
                    const int kp = kp_lane + 16 * i;
                    const uint2 v = *reinterpret_cast<const uint2*>(bp + kp * BNH + nl);
                    uint32_t e[4], o[4];
                    unpack_word(v.x, e[0], e[1], o[0], o[1]);
                    unpack_word(v.y, e[2], e[3], o[2], o[3]);
                    if (fast) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) { e[j] = bsub2(e[j], zz[j]); o[j] = bsub2(o[j], zz[j]); }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            e[j] = bsub2(bsub2(e[j], k128), zraw[j]);
                            o[j] = bsub2(bsub2(o[j], k128), zraw[j]);
                        }
                    }
                    *reinterpret_cast<uint4*>(bd + bd_offset(2 * kp, nl)) = make_uint4(e[0], e[1], e[2], e[3]);
                    *reinterpret_cast<uint4*>(bd + bd_offset(2 * kp + 1, nl)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_deq(s));
            }
        }
    } else {
        // ---------------- epilogue (warps 10..13) ----------------
        // TMEM lane quarter = warp % 4; each warp stores its 32 rows x 256
        // columns of the tile.  Decisions are warp-uniform (tcgen05.ld is
        // warp-collective).
        const int quarter = warp & 3;
        const uint32_t release = map_cluster(acc_empty(0), 0);
        for (int it = 0; it < my_tiles; ++it) {
            const int b = it & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(acc_full(b), (it >> 1) & 1, abort_flag))) break;
            tc_fence_after();
            const int n0 = tile_n(it) * BN;
            const int m = tile_m(it) * (2 * BM) + rank * BM + quarter * 32 + lane;
            for (int cb = 0; cb < BN / 32; ++cb) {
                uint32_t r[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * BN + cb * 32, r);
                const int nb = n0 + cb * 32;
                if (m < M && nb < N) {
                    // TMEM column order inside each group of 4 is n0 n2 n1 n3
                    uint32_t packed[16];
#pragma unroll
                    for (int g4 = 0; g4 < 8; ++g4) {
                        const int na = nb + 4 * g4;
                        float sc[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            sc[q] = na + q >= N ? 0.f
                                    : (I8 || PERM) ? static_cast<const float*>(scale_p)[na + q]
                                         : __bfloat162float(static_cast<const __nv_bfloat16*>(scale_p)[na + q]);
                        const float v0 = __uint_as_float(r[4 * g4 + 0]) * sc[0];
                        const float v1 = __uint_as_float(r[4 * g4 + 2]) * sc[1];
                        const float v2 = __uint_as_float(r[4 * g4 + 1]) * sc[2];
                        const float v3 = __uint_as_float(r[4 * g4 + 3]) * sc[3];
                        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v0, v1);
                        const __nv_bfloat162 h23 = __floats2bfloat162_rn(v2, v3);
                        packed[2 * g4] = *reinterpret_cast<const uint32_t*>(&h01);
                        packed[2 * g4 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
                    }
                    __nv_bfloat16* dst = C + static_cast<int64_t>(m) * N + nb;
                    if (nb + 32 <= N) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            reinterpret_cast<uint4*>(dst)[q] =
                                make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    } else {
                        for (int q = 0; q < (N - nb) / 8; ++q)
                            reinterpret_cast<uint4*>(dst)[q] =
                                make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    }
                }
            }
            // accumulator b is read out (tcgen05.ld waited): hand it back to the even CTA
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(release + 8u * b);
        }
    }

    // every MMA of the pair is complete (the epilogues waited for the last
    // accumulator, or everything timed out) before either CTA frees its TMEM
    if (warp == 1 && rank == 0 && lane == 0 && my_tiles > 0)
        mbar_drain(acc_full((my_tiles - 1) & 1), ((my_tiles - 1) >> 1) & 1);
    tc_fence_before();
    cluster.sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace gemm

namespace gemm {

template <int FMT>
w4_status run_gemm_t(const void* A, const void* B, const void* scale, const void* zero, void* C, int64_t M,
                     int64_t N, int64_t K, cudaStream_t stream) {
    constexpr bool I8 = FMT == FMT_INT8;
    constexpr int SMEM_BYTES = Lay<FMT>::SMEM_BYTES;
    auto kern = gemm_w4_tc_kernel<FMT>;
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return W4_ERR_SHAPE;
    const int64_t tiles_m = (M + 2 * BM - 1) / (2 * BM), tiles_n = (N + BN - 1) / BN;
    if (tiles_m * tiles_n > 0x7FFFFFFF) return W4_ERR_SHAPE;
    auto encode = tensor_map_encoder();
    if (!encode) return W4_ERR_CUDA;

    CUtensorMap ta, tb;
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        cuuint32_t box[2] = {BK, BM};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4_ERR_CUDA;
    }
    if (FMT == FMT_PERM) {
        // permute_int4's output as [N/4 groups][K/64 lines][128 bytes]
        cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(K / 64), static_cast<cuuint64_t>(N / 4)};
        cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(K / 2) * 4};
        cuuint32_t box[3] = {128, 1, BNH / 4};
        cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(B), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4_ERR_CUDA;
    } else {
        // int4: packed [K/2][N] bytes; int8: q [K][N]
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(I8 ? K : K / 2)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(N)};
        cuuint32_t box[2] = {BNH, I8 ? BK : BK / 2};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(B), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4_ERR_CUDA;
    }
    static int smem_set[64];
    cudaError_t e = ensure_smem_limit(kern, SMEM_BYTES, smem_set);
    if (e != cudaSuccess) return W4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: as many CTA pairs as can be resident at once
    static int max_pairs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return W4_ERR_CUDA;
    if (max_pairs[dev] == 0) {
        cfg.gridDim = dim3(static_cast<unsigned>(2 * std::max(1, sm_count() / 2)), 1, 1);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return W4_ERR_CUDA;
        max_pairs[dev] = n;
    }
    const int64_t num_tiles = tiles_m * tiles_n;
    const int pairs = static_cast<int>(std::min<int64_t>(num_tiles, max_pairs[dev]));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    return launch_status(cudaLaunchKernelEx(&cfg, kern, ta, tb, scale, static_cast<const __nv_bfloat16*>(zero),
                                            static_cast<__nv_bfloat16*>(C),
                                            static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                            static_cast<int>(tiles_n), static_cast<int>(num_tiles)));
}

}  // namespace gemm

w4_status run_gemm(const void* A, const void* B, const void* scale, const void* zero, void* C, int64_t M,
                   int64_t N, int64_t K, cudaStream_t stream) {
    return gemm::run_gemm_t<gemm::FMT_INT4>(A, B, scale, zero, C, M, N, K, stream);
}

w4_status run_gemm_w8(const void* A, const void* q, const float* scale, void* C, int64_t M, int64_t N, int64_t K,
                      cudaStream_t stream) {
    return gemm::run_gemm_t<gemm::FMT_INT8>(A, q, scale, nullptr, C, M, N, K, stream);
}

w4_status run_gemm_w4_permuted(const void* A, const void* permuted, const float* scale, void* C, int64_t M,
                               int64_t N, int64_t K, cudaStream_t stream) {
    return gemm::run_gemm_t<gemm::FMT_PERM>(A, permuted, scale, nullptr, C, M, N, K, stream);
}

int take_device_error_gemm() { return take_unit_device_error(); }
int set_wait_limit_gemm(long long clocks) { return set_unit_wait_limit(clocks); }
int set_short_first_stage_gemm(int on) {
    const int v = on ? 1 : 0;
    return cudaMemcpyToSymbol(gemm::g_short_first_stage, &v, sizeof(v)) == cudaSuccess ? 0 : -1;
}

}  // namespace w4
