// quant_permute.cu -- weight-only int4 quantise + column pack, and the int4
// interleave permute (page "[PHI] add int4 weight only quant kernel, add int4
// weight only permute kernel": sections "int4量化kernel", "int4 permute
// kernel", "简单的位运算", "int4 row interval").
//
// Both kernels are HBM-bound byte movers.  Roofline bytes per element are
// stated next to each kernel.

#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace w4 {

// ---------------------------------------------------------------------------
// quantize_pack_int4, single HBM read (N % 8 == 0, K <= QC_MAX_K)
//
// A thread-block cluster of cs CTAs (up to 16, a non-portable cluster size)
// owns a strip of 32 columns over all K;
// CTA r holds rows [r*R, r*R + R) of the strip in shared memory, loaded once
// with 2-D TMA boxes (64 bytes x up to 256 rows).  Each CTA reduces its rows
// to a per-column max |W| (bf16 bit patterns with the sign cleared order
// non-negative values exactly), the CTAs read each other's partial maxima
// through distributed shared memory, and every CTA then quantises the rows it
// already holds.  W is read from HBM exactly once.  Algorithmic bytes: 2 B
// read per weight + 0.5 B written.  32 KB per CTA for K = 8192 (sixteen
// CTAs of 512 rows), so several CTAs share an SM and one's copy overlaps
// another's arithmetic (eight CTAs of 64 KB measured 3.5% slower).
// ---------------------------------------------------------------------------

constexpr int QC_COLS = 32;                      // columns per strip (64-byte rows)
constexpr int QC_THREADS = 256;
constexpr int QC_RL = QC_THREADS / 4;            // row lanes (4 threads of 8 columns per row)
constexpr int QC_CS = 8;                         // K limit: eight CTAs of QC_MAX_R rows
constexpr int QC_CS_USE = 16;                    // CTAs per cluster at most (non-portable size)
constexpr int QC_BPC = 2;                        // TMA boxes per CTA aimed for (512 rows, 32 KB)
constexpr int QC_CS_ALLOC = QC_CS_USE > QC_CS ? QC_CS_USE : QC_CS;
constexpr int QC_BOXR = 256;                     // rows per TMA box
constexpr int QC_SMEM = 208 * 1024;              // strip rows per CTA at most (bytes)
constexpr int QC_MAX_R = QC_SMEM / (QC_COLS * 2) / QC_BOXR * QC_BOXR;
constexpr int64_t QC_MAX_K = static_cast<int64_t>(QC_CS) * QC_MAX_R;
static_assert(QC_MAX_K == W4_QUANT_PERMUTE_MAX_K, "the header's K limit is the single-read kernel's");

// q = clamp(round_half_away(w / s), -8, 7) as a nibble; s == 0 gives 0.
__device__ __forceinline__ uint32_t quant_nibble(uint32_t wbits, float s) {
    float w = bf16_bits_to_f32(wbits & 0xFFFFu);
    float r = (s == 0.0f) ? 0.0f : roundf(__fdiv_rn(w, s));
    r = fminf(fmaxf(r, -8.0f), 7.0f);
    return static_cast<uint32_t>(static_cast<int>(r)) & 0xFu;
}

// The same nibble from one FMA, for all but near-ties.
//   u = fl(w * inv + C),  inv = fl(1/s) (0 when s = 0),  C = 192.5 + 2^-15.
// |w| <= max|w| = 7 s, so u lies in [128, 256) where the fp32 ulp is 2^-16:
// mantissa bits 16..19 hold floor(w*inv + 0.5) mod 16 (192 = 0 mod 16) and
// the low 16 bits its fraction, lifted by 2^-15.  Unless those low bits are
// < 4 (the fraction is within 2^-14 of an integer), the exact product
// w * inv -- within 1e-6 of the IEEE quotient fl(w / s) -- is clear of every
// half-integer by more than that error, so floor(w*inv + 0.5) equals
// round-half-away(fl(w / s)); |q| <= 7, so no clamp.  Near-ties (exact ties
// such as w = max|w| / 2 recur in real columns) are flagged for the exact
// division.
__device__ __forceinline__ uint32_t quant_u(uint32_t wbits16_hi, float inv) {
    return __float_as_uint(__fmaf_rn(__uint_as_float(wbits16_hi), inv, 192.50003051757812f));
}
__device__ __forceinline__ bool quant_near(uint32_t u) { return (u & 0xFFFCu) == 0; }

// Bracketed variant: u_hi / u_lo = fl(w * inv + 192.5 +/- 2^-15).  If both
// have the same integer part F, then w * inv + 192.5 lies at least 3*2^-17
// inside (F, F + 1); the IEEE quotient fl(w / s) differs from w * inv by less
// than 2^-21 (|w / s| <= 7), so fl(w / s) + 0.5 is not an integer and
// round-half-away(fl(w / s)) = floor(fl(w / s) + 0.5) = F - 192, whose low
// four bits are bits 16..19 of u (F - 128 fills bits 16..22 of the
// mantissa; 128 and 192 are 0 mod 16).  Different integer parts flag the
// weight for the exact division.
constexpr float QB_HI = 192.50003051757812f;   // 192.5 + 2^-15
constexpr float QB_LO = 192.49996948242188f;   // 192.5 - 2^-15

// int8 (quantize_int8: s = max|w| / 127, q = clamp(round_half_away(w / s),
// -128, 127)) with the same bracket one binade higher:
//   u_hi / u_lo = fl(w * inv + 384.5 +/- 2^-13),  inv = fl(1/s).
// |w / s| <= 127 (1 + 2^-23), so u lies in [256, 512), ulp 2^-15, and the
// integer part F of u sits in mantissa bits 15..22 (F - 256).  w * inv is
// within 127 * 2^-24 of w / s and fl(w / s) within 2^-18 of it, and each FMA
// rounds by at most 2^-16: if both brackets have the integer part F, then
// fl(w / s) + 0.5 lies strictly inside (F - 384, F - 383), so
// round_half_away(fl(w / s)) = F - 384 (never 128: |fl(w / s)| < 127.5), the
// byte ((u >> 15) & 0xFF) ^ 0x80.  Otherwise the weight takes the exact
// division.
constexpr float QB8_HI = 384.50012207031250f;   // 384.5 + 2^-13
constexpr float QB8_LO = 384.49987792968750f;   // 384.5 - 2^-13

__device__ __forceinline__ uint32_t quant_byte_exact(uint32_t wbits, float s) {
    const float w = bf16_bits_to_f32(wbits & 0xFFFFu);
    float r = (s == 0.0f) ? 0.0f : roundf(__fdiv_rn(w, s));
    r = fminf(fmaxf(r, -128.0f), 127.0f);
    return static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu;
}

// Byte 2 of a and byte 2 of b in bytes 0, 1 (sel 0x0062) or 2, 3 (sel 0x6200).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

// The nibbles (bits 16..19) of x0..x3 and y0..y3 as one word with nibble
// order x0 y0 x1 y1 x2 y2 x3 y3 (x0 in bits 0..3).
__device__ __forceinline__ uint32_t pack_nibbles(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t y0,
                                                 uint32_t y1, uint32_t y2, uint32_t y3) {
    const uint32_t X = prmt(prmt(x0, x1, 0x0062), prmt(x2, x3, 0x6200), 0x7610);
    const uint32_t Y = prmt(prmt(y0, y1, 0x0062), prmt(y2, y3, 0x6200), 0x7610);
    return (X & 0x0F0F0F0Fu) | ((Y << 4) & 0xF0F0F0F0u);
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// R = rows per CTA (a multiple of box); box = TMA box height;
// grid = strips * cs with clusters of cs CTAs.
// PERMUTED = false: `out` is the packed [K/2][N] matrix.  PERMUTED = true:
// `out` is permute_int4's layout of it (N*K/2 bytes; K % 64 == 0), written
// directly: for column n and 32-row group t the 16 bytes at
// (K/2)*4*(n/4) + (t/2)*128 + 32*(n%4) + 16*(t%2), whose 32-bit word i holds
// in nibble slots 0..7 the rows 32t + 2i + (0, 8, 16, 24, 1, 9, 17, 25).
// INT8 = true (quantize_int8): `out` is q int8 [K][N], scale = max / 127.
template <bool PERMUTED, bool INT8 = false>
__global__ void __launch_bounds__(QC_THREADS)
quantize_pack_cluster_kernel(const __grid_constant__ CUtensorMap tmap, uint8_t* __restrict__ out,
                             float* __restrict__ scale, int K, int N, int R, int box) {
    uint8_t* __restrict__ packed = out;
    extern __shared__ __align__(128) uint8_t qtile[];   // [R][32] bf16
    __shared__ __align__(8) uint64_t bar;
    __shared__ __align__(8) uint64_t pm_bar;          // every rank's partial maxima have landed
    __shared__ uint32_t pm_all[QC_CS_ALLOC][QC_COLS]; // partial maxima, one row per rank
    __shared__ uint32_t wmax[QC_THREADS / 32][QC_COLS];
    __shared__ float s_scale[QC_COLS], s_inv[QC_COLS];
    __shared__ int abort_word;
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = static_cast<int>(cluster.num_blocks());
    const int rank = static_cast<int>(cluster.block_rank());
    const int n0 = (blockIdx.x / cs) * QC_COLS;
    const int k0 = rank * R;
    const int rows = max(0, min(R, K - k0));      // even
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = tid & 3, rl = tid >> 2;          // 8-column group, row lane
    const uint32_t b = ptx::smem_u32(&bar);
    const uint32_t pb = ptx::smem_u32(&pm_bar);

    if (tid == 0) {
        ptx::mbar_init(b, 1);
        ptx::mbar_init(pb, 1);
        abort_word = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the peers' pushes (cs x 32 words) complete this phase
        ptx::mbar_arrive_expect_tx(pb, static_cast<uint32_t>(cs) * QC_COLS * 4);
    }
    __syncthreads();
    // first half of a cluster barrier: this CTA's barriers are initialised
    // (the second half is waited for just before pushing to the peers)
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    const int nbox = (rows + box - 1) / box;
    if (tid == 0 && nbox > 0) {
        ptx::mbar_arrive_expect_tx(b, static_cast<uint32_t>(nbox) * box * QC_COLS * 2);
        for (int i = 0; i < nbox; ++i)
            ptx::tma_load_2d(ptx::smem_u32(qtile + static_cast<size_t>(i) * box * QC_COLS * 2), &tmap, n0,
                             k0 + i * box, b);
    }

    // column max of |W| over this CTA's rows; word j of a 16-byte group holds
    // columns 2j (low half) and 2j+1 (high half), reduced packed
    uint32_t amax[4] = {0, 0, 0, 0};
    bool ok = nbox == 0 || ptx::mbar_wait(b, 0, &abort_word);
    if (!ok && tid == 0) ptx::mbar_drain(b, 0);   // copies still landing
    if (ok) {
#pragma unroll 4
        for (int r = rl; r < rows; r += QC_RL) {
            const uint4 v = *reinterpret_cast<const uint4*>(qtile + r * (QC_COLS * 2) + g * 16);
            amax[0] = max_u16x2(amax[0], v.x & 0x7FFF7FFFu);
            amax[1] = max_u16x2(amax[1], v.y & 0x7FFF7FFFu);
            amax[2] = max_u16x2(amax[2], v.z & 0x7FFF7FFFu);
            amax[3] = max_u16x2(amax[3], v.w & 0x7FFF7FFFu);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) amax[j] = max_u16x2(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
    }
    if (lane < 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            wmax[warp][lane * 8 + 2 * j] = amax[j] & 0xFFFFu;
            wmax[warp][lane * 8 + 2 * j + 1] = amax[j] >> 16;
        }
    }
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");   // every peer is initialised
    if (tid < QC_COLS) {
        // push this CTA's partial maximum of column tid into every rank's
        // pm_all[rank][tid]; each store completes 4 bytes on that rank's pm_bar
        uint32_t m = 0;
        for (int w = 0; w < QC_THREADS / 32; ++w) m = max(m, wmax[w][tid]);
        const uint32_t slot = ptx::smem_u32(&pm_all[rank][tid]);
        for (int r = 0; r < cs; ++r)
            asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(
                             ptx::map_cluster(slot, r)),
                         "r"(m), "r"(ptx::map_cluster(pb, r))
                         : "memory");
    }
    // wait for every rank's push (bounded); afterwards no peer touches this
    // CTA's shared memory again, so no cluster barrier is needed at exit
    if (!ptx::mbar_wait(pb, 0, &abort_word)) {
        ok = false;
        if (tid == 0) ptx::mbar_drain(pb, 0);   // a slow peer's push may still be on its way
    }
    if (tid < QC_COLS) {
        uint32_t m = 0;
        for (int r = 0; r < cs; ++r) m = max(m, pm_all[r][tid]);
        const float sc = __fdiv_rn(bf16_bits_to_f32(m), INT8 ? 127.0f : 7.0f);
        s_scale[tid] = sc;
        s_inv[tid] = sc == 0.0f ? 0.0f : __frcp_rn(sc);
        if (rank == 0 && n0 + tid < N) scale[n0 + tid] = sc;
    }
    __syncthreads();

    if constexpr (PERMUTED) {
        // quantise 64 rows (two 32-row groups) per warp iteration: lane
        // (cp, par) takes columns 2cp, 2cp+1 on rows 2i + par of a group
        // (one 32-bit shared load per row), brackets each weight with two
        // FMAs, and packs the nibbles of its 16 rows into four half-words per
        // column; the partner lane (par ^ 1) holds the other half of each
        // output word.
        if (__all_sync(0xffffffffu, ok)) {
            const int cp = lane & 15, par = lane >> 4;
            const float inv0 = s_inv[2 * cp], inv1 = s_inv[2 * cp + 1];
            // a scale below about 2^-128 (column maximum below about 7 * 2^-128)
            // has no finite reciprocal: every weight of such a column takes the
            // exact path below (its bracket test cannot pass by accident:
            // |w| <= 7 s rules out the tie m s with the bogus m it reads)
            const uint32_t force0 = isinf(inv0) ? ~0u : 0u, force1 = isinf(inv1) ? ~0u : 0u;
            const int mycol = 2 * cp + par;                       // the column this lane stores
            const bool col_ok = n0 + mycol < N;
            // output: 128-byte lines of the column's group of four, this
            // CTA's first line; + 16 * (t % 2) and 128 per group pair
            uint8_t* dst = out + static_cast<int64_t>(K / 2) * 4 * ((n0 + mycol) / 4) +
                           static_cast<int64_t>(k0 / 64) * 128 + 32 * (mycol % 4);
            const uint32_t sel_lo = par ? 0x1054u : 0x5410u, sel_hi = par ? 0x3276u : 0x7632u;
            const int npairs = rows / 64;
            for (int pr = warp; pr < npairs; pr += QC_THREADS / 32) {
                uint4 res[2];
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const uint8_t* base = qtile + (64 * pr + 32 * tt + par) * (QC_COLS * 2) + 4 * cp;
                    // z[col][h]: h = 0 holds half-words 0, 1 (rows i = 0,4,8,12 | 1,5,9,13),
                    // h = 1 half-words 2, 3 (i + 2); zb: the same from the lower bracket
                    uint32_t z[2][2], zb[2][2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // rows i in nibble order x0 y0 x1 y1 x2 y2 x3 y3
                        constexpr int ix[4] = {0, 8, 1, 9}, iy[4] = {4, 12, 5, 13};
                        uint32_t wx[4], wy[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            wx[k] = *reinterpret_cast<const uint32_t*>(base + (2 * (ix[k] + 2 * h)) * (QC_COLS * 2));
                            wy[k] = *reinterpret_cast<const uint32_t*>(base + (2 * (iy[k] + 2 * h)) * (QC_COLS * 2));
                        }
#pragma unroll
                        for (int col = 0; col < 2; ++col) {
                            const float inv = col ? inv1 : inv0;
                            uint32_t ux[4], uy[4], vx[4], vy[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float fx = __uint_as_float(col ? (wx[k] & 0xFFFF0000u) : (wx[k] << 16));
                                const float fy = __uint_as_float(col ? (wy[k] & 0xFFFF0000u) : (wy[k] << 16));
                                ux[k] = __float_as_uint(__fmaf_rn(fx, inv, QB_HI));
                                uy[k] = __float_as_uint(__fmaf_rn(fy, inv, QB_HI));
                                vx[k] = __float_as_uint(__fmaf_rn(fx, inv, QB_LO));
                                vy[k] = __float_as_uint(__fmaf_rn(fy, inv, QB_LO));
                            }
                            z[col][h] = pack_nibbles(ux[0], ux[1], ux[2], ux[3], uy[0], uy[1], uy[2], uy[3]);
                            zb[col][h] = pack_nibbles(vx[0], vx[1], vx[2], vx[3], vy[0], vy[1], vy[2], vy[3]);
                        }
                    }
                    // Weights whose brackets disagree lie within 2^-15 of a tie
                    // m = k + 1/2 (k = integer part of the lower bracket - 192).
                    // Exact ties (w = m s, the usual case: the FMA residual is
                    // then exactly 0) round away from zero; the rest take the
                    // exact IEEE division.  One weight per trip of a lane.
                    uint32_t f0 = (z[0][0] ^ zb[0][0]) | force0, f1 = (z[0][1] ^ zb[0][1]) | force0;
                    uint32_t f2 = (z[1][0] ^ zb[1][0]) | force1, f3 = (z[1][1] ^ zb[1][1]) | force1;
                    if (__any_sync(0xffffffffu, (f0 | f1 | f2 | f3) != 0)) {
                        while ((f0 | f1 | f2 | f3) != 0) {
                            const int wsel = f0 ? 0 : f1 ? 1 : f2 ? 2 : 3;   // word: col = wsel / 2, h = wsel % 2
                            const uint32_t f = wsel == 0 ? f0 : wsel == 1 ? f1 : wsel == 2 ? f2 : f3;
                            const int nib = (__ffs(f) - 1) >> 2;              // nibble slot 0..7
                            const int col = wsel >> 1, h = wsel & 1;
                            // slot -> row i: even slots ix[slot/2], odd iy[slot/2] (+ 2h)
                            const int kk = nib >> 1;
                            const int i = (kk >> 1) + 8 * (kk & 1) + 4 * (nib & 1) + 2 * h;
                            const uint32_t e = reinterpret_cast<const uint16_t*>(base + (2 * i) * (QC_COLS * 2))[col];
                            const float wf = bf16_bits_to_f32(e);
                            const float sc = s_scale[2 * cp + col];
                            const uint32_t ulo = __float_as_uint(__fmaf_rn(wf, col ? inv1 : inv0, QB_LO));
                            const int k = 128 + static_cast<int>((ulo >> 16) & 0x7Fu) - 192;
                            const float m = static_cast<float>(k) + 0.5f;
                            uint32_t nibv;
                            if (__fmaf_rn(-m, sc, wf) == 0.0f) nibv = static_cast<uint32_t>(m > 0.0f ? k + 1 : k) & 0xFu;
                            else nibv = quant_nibble(e, sc);
                            const uint32_t keep = ~(0xFu << (4 * nib)), put = nibv << (4 * nib);
                            if (wsel == 0) { f0 &= keep; z[0][0] = (z[0][0] & keep) | put; }
                            else if (wsel == 1) { f1 &= keep; z[0][1] = (z[0][1] & keep) | put; }
                            else if (wsel == 2) { f2 &= keep; z[1][0] = (z[1][0] & keep) | put; }
                            else { f3 &= keep; z[1][1] = (z[1][1] & keep) | put; }
                        }
                    }
                    // lane par = 0 keeps column 2cp, par = 1 column 2cp+1: trade the
                    // other column's half-words with the partner lane
                    const uint32_t send0 = par ? z[0][0] : z[1][0], send1 = par ? z[0][1] : z[1][1];
                    const uint32_t own0 = par ? z[1][0] : z[0][0], own1 = par ? z[1][1] : z[0][1];
                    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, send0, 16);
                    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, send1, 16);
                    // word i: half-word i of the even rows (low) and of the odd rows (high)
                    res[tt] = make_uint4(__byte_perm(own0, r0, sel_lo), __byte_perm(own0, r0, sel_hi),
                                         __byte_perm(own1, r1, sel_lo), __byte_perm(own1, r1, sel_hi));
                }
                if (col_ok) {
                    uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(pr) * 128);
                    d[0] = res[0];
                    d[1] = res[1];
                }
            }
        }
        return;
    }

    if constexpr (INT8) {
        // int8: thread (g, rl) takes the 8 columns of group g on rows rl,
        // rl + QC_RL, ... (a warp: 8 consecutive rows), brackets each weight
        // with two FMAs and stores 8 bytes per row; near-ties and columns
        // whose scale has no finite reciprocal take the exact division.
        // Control flow is warp-uniform, as below.
        if (__all_sync(0xffffffffu, ok)) {
            const bool col_ok = n0 + 8 * g < N;
            float inv[8];
            uint32_t tinymask = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                inv[j] = s_inv[8 * g + j];
                if (isinf(inv[j])) tinymask |= 1u << j;
            }
            for (int r0 = rl & ~7; r0 < rows; r0 += QC_RL) {
                const int r = r0 + (rl & 7);
                const uint8_t* ra = qtile + min(r, rows - 1) * (QC_COLS * 2) + g * 16;
                const uint4 a = *reinterpret_cast<const uint4*>(ra);
                const uint32_t wa[4] = {a.x, a.y, a.z, a.w};
                uint32_t res[2] = {0, 0}, nearmask = tinymask;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float w = __uint_as_float((j & 1) ? (wa[j / 2] & 0xFFFF0000u) : (wa[j / 2] << 16));
                    const uint32_t uh = __float_as_uint(__fmaf_rn(w, inv[j], QB8_HI));
                    const uint32_t ul = __float_as_uint(__fmaf_rn(w, inv[j], QB8_LO));
                    res[j / 4] |= (((uh >> 15) & 0xFFu) ^ 0x80u) << (8 * (j % 4));
                    nearmask |= ((uh >> 15) != (ul >> 15) ? 1u : 0u) << j;
                }
                if (__any_sync(0xffffffffu, nearmask != 0)) {
                    while (nearmask != 0) {
                        const int j = __ffs(nearmask) - 1;
                        nearmask &= nearmask - 1;
                        const uint32_t e = reinterpret_cast<const uint16_t*>(ra)[j];
                        const int pos = 8 * (j & 3);
                        res[j / 4] = (res[j / 4] & ~(0xFFu << pos)) | (quant_byte_exact(e, s_scale[8 * g + j]) << pos);
                    }
                }
                if (col_ok && r < rows)
                    *reinterpret_cast<uint2*>(out + (static_cast<int64_t>(k0) + r) * N + n0 + 8 * g) =
                        make_uint2(res[0], res[1]);
            }
        }
        return;
    }

    // quantise the resident rows two at a time (low nibble = even row).
    // Control flow is warp-uniform: the trip count is the warp's, lanes past
    // the last pair redo a valid pair without storing, and the exact fix-up
    // of near-ties runs under a warp vote.
    if (__all_sync(0xffffffffu, ok)) {
        const bool col_ok = n0 + 8 * g < N;
        float inv[8];
        // columns whose scale has no finite reciprocal (below about 2^-128):
        // all their weights take the exact division of the fix-up
        uint32_t tinymask = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            inv[j] = s_inv[8 * g + j];
            if (isinf(inv[j])) tinymask |= 3u << (2 * j);
        }
        const int pairs = rows / 2;
        for (int p0 = rl & ~7; p0 < pairs; p0 += QC_RL) {   // rl & ~7: the warp's first row lane
            const int p = p0 + (rl & 7);
            const int pc = min(p, pairs - 1);
            const uint8_t* ra = qtile + (2 * pc) * (QC_COLS * 2) + g * 16;
            const uint4 a = *reinterpret_cast<const uint4*>(ra);
            const uint4 c = *reinterpret_cast<const uint4*>(ra + QC_COLS * 2);
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {c.x, c.y, c.z, c.w};
            // nibble of (row, column j) goes to bit 8*(j%4) + 4*row of word j/4
            uint32_t out[2] = {0, 0}, nearmask = tinymask;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t ha = (j & 1) ? (wa[j / 2] & 0xFFFF0000u) : (wa[j / 2] << 16);
                const uint32_t hb = (j & 1) ? (wb[j / 2] & 0xFFFF0000u) : (wb[j / 2] << 16);
                const uint32_t ua = quant_u(ha, inv[j]), ub = quant_u(hb, inv[j]);
                const int pa = 8 * (j % 4), pb = pa + 4;
                out[j / 4] |= ((ua >> 16) & 0xFu) << pa;
                out[j / 4] |= ((ub >> 16) & 0xFu) << pb;
                nearmask |= (quant_near(ua) ? 1u : 0u) << (2 * j);
                nearmask |= (quant_near(ub) ? 1u : 0u) << (2 * j + 1);
            }
            if (__any_sync(0xffffffffu, nearmask != 0)) {
                while (nearmask != 0) {
                    const int bit = __ffs(nearmask) - 1;
                    nearmask &= nearmask - 1;
                    const int j = bit >> 1, row = bit & 1;
                    const uint32_t e = reinterpret_cast<const uint16_t*>(ra + row * (QC_COLS * 2))[j];
                    const int pos = 8 * (j & 3) + 4 * row;
                    const uint32_t nib = quant_nibble(e, s_scale[8 * g + j]) << pos;
                    if (j < 4) out[0] = (out[0] & ~(0xFu << pos)) | nib;
                    else out[1] = (out[1] & ~(0xFu << pos)) | nib;
                }
            }
            if (col_ok && p < pairs)
                *reinterpret_cast<uint2*>(packed + (static_cast<int64_t>(k0 / 2) + p) * N + n0 + 8 * g) =
                    make_uint2(out[0], out[1]);
        }
    }
}

// ---------------------------------------------------------------------------
// quantize_pack_int4, two passes (fallback: N % 8 != 0 or K > QC_MAX_K)
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

namespace {

// Single-read path; W4_ERR_SHAPE means "use the two-pass kernel".
// mode 0: packed int4; 1: permute_int4's layout (requires K % 64 == 0);
// 2: int8 (quantize_int8).
w4_status launch_quantize_cluster(const void* W, void* packed, float* scale, int64_t K, int64_t N,
                                  cudaStream_t stream, int mode) {
    if ((N % 8) != 0 || K > QC_MAX_K || N > 0x7FFFFFFF) return W4_ERR_SHAPE;
    const int64_t strips = (N + QC_COLS - 1) / QC_COLS;
    // rows per CTA: whole TMA boxes, 1024 rows (64 KB) per CTA while the
    // cluster has room, more rows per CTA beyond that
    int cs = 1, R = 0, box = 0;
    const int64_t Keven = (K + 1) / 2 * 2;
    if (Keven <= QC_BOXR) {
        R = static_cast<int>(Keven);
        box = R;
    } else {
        const int64_t boxes = (K + QC_BOXR - 1) / QC_BOXR;
        cs = static_cast<int>(std::min<int64_t>(QC_CS_USE, (boxes + QC_BPC - 1) / QC_BPC));
        const int64_t bpc = (boxes + cs - 1) / cs;
        R = static_cast<int>(bpc * QC_BOXR);
        box = QC_BOXR;
    }
    if (R * QC_COLS * 2 > QC_SMEM || strips * cs > 0x7FFFFFFF) return W4_ERR_SHAPE;
    auto encode = tensor_map_encoder();
    if (!encode) return W4_ERR_CUDA;
    CUtensorMap tmap;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
    cuuint32_t boxd[2] = {QC_COLS, static_cast<cuuint32_t>(box)};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, boxd, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return W4_ERR_CUDA;
    const int smem = R * QC_COLS * 2;
    static int smem_set[3][64];
    auto kern = mode == 1 ? quantize_pack_cluster_kernel<true>
                : mode == 2 ? quantize_pack_cluster_kernel<false, true> : quantize_pack_cluster_kernel<false>;
    if (ensure_smem_limit(kern, smem, smem_set[mode]) != cudaSuccess) return W4_ERR_CUDA;
    if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return W4_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(strips * cs), 1, 1);
    cfg.blockDim = dim3(QC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return launch_status(cudaLaunchKernelEx(&cfg, kern, tmap, static_cast<uint8_t*>(packed), scale,
                                            static_cast<int>(K), static_cast<int>(N), R, box));
}

}  // namespace

w4_status run_quantize_pack(const void* W, void* packed, float* scale, int64_t K, int64_t N,
                            cudaStream_t stream) {
    const w4_status st = launch_quantize_cluster(W, packed, scale, K, N, stream, 0);
    if (st != W4_ERR_SHAPE) return st;
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
// A thread owns four adjacent columns (one group of the interleave) over one
// 32-byte chunk of the k-byte stream (rows 32j..32j+31 of the packed matrix):
// it loads the 32 rows x 4 bytes, transposes 4x4 byte blocks in registers so
// that each column's bytes are contiguous, applies the byte permute and
// nibble swap to each 16-byte group and writes the group's four 32-byte
// chunks, which are adjacent in the output (128 contiguous bytes).  A warp
// covers 8 groups x 4 chunks, so each row load is 4 whole 32-byte sectors,
// and a CTA (8 warps) covers 32 consecutive chunks of 8 groups, so each
// output run receives 4 KB of contiguous writes.  No shared memory.
// Algorithmic bytes: 1 B read + 1 B written per byte.
// ---------------------------------------------------------------------------

constexpr int PM_THREADS = 256;   // 8 warps x (8 groups x 4 chunks)
constexpr int PM_GROUPS = 8;      // column groups per CTA
constexpr int PM_CHUNKS = 32;     // 32-byte chunks per CTA

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

// 4x4 byte transpose: r[i] holds bytes (row i, columns 0..3); c[j] gets
// (column j, rows 0..3).
__device__ __forceinline__ void transpose4x4(const uint32_t (&r)[4], uint32_t (&c)[4]) {
    const uint32_t t01 = __byte_perm(r[0], r[1], 0x5140);  // r0b0 r1b0 r0b1 r1b1
    const uint32_t t23 = __byte_perm(r[2], r[3], 0x5140);
    const uint32_t u01 = __byte_perm(r[0], r[1], 0x7362);  // r0b2 r1b2 r0b3 r1b3
    const uint32_t u23 = __byte_perm(r[2], r[3], 0x7362);
    c[0] = __byte_perm(t01, t23, 0x5410);
    c[1] = __byte_perm(t01, t23, 0x7632);
    c[2] = __byte_perm(u01, u23, 0x5410);
    c[3] = __byte_perm(u01, u23, 0x7632);
}

// grid = (ceil(N/4 / PM_GROUPS), ceil(K/64 / PM_CHUNKS)); lane = group (lane % 8)
// of chunk 4*warp + lane / 8.
__global__ void __launch_bounds__(PM_THREADS)
permute_kernel(const uint8_t* __restrict__ packed, uint8_t* __restrict__ out, int64_t K, int64_t N) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t grp = static_cast<int64_t>(blockIdx.x) * PM_GROUPS + (lane & 7);          // columns 4grp..+3
    const int64_t chunk = static_cast<int64_t>(blockIdx.y) * PM_CHUNKS + 4 * warp + (lane >> 3);
    if (grp >= N / 4 || chunk >= K / 64) return;
    const uint8_t* src = packed + chunk * 32 * N + 4 * grp;
    uint32_t rw[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) rw[r] = ldg_stream_u32(src + r * N);
    // col[c][i] = bytes of column c, rows 4i..4i+3
    uint32_t col[4][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t rr[4] = {rw[4 * i], rw[4 * i + 1], rw[4 * i + 2], rw[4 * i + 3]};
        uint32_t cc[4];
        transpose4x4(rr, cc);
#pragma unroll
        for (int c = 0; c < 4; ++c) col[c][i] = cc[c];
    }
    uint4* dst = reinterpret_cast<uint4*>(out + (K / 2) * 4 * grp + 128 * chunk);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t w[4] = {col[c][4 * h], col[c][4 * h + 1], col[c][4 * h + 2], col[c][4 * h + 3]};
            uint32_t o[4];
            permute_group16(w, o);
            dst[2 * c + h] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// The same tile (8 groups x 32 chunks) with its 32 KB of input brought in by
// four 2-D TMA boxes (32 columns x 256 rows) instead of 32 four-byte loads
// per thread (which kept the load/store unit's queue full), and its 32 KB of
// output staged in shared memory so that every warp store writes 512
// contiguous bytes (whole 128-byte lines) instead of sixteen bytes into each
// of 32 lines.  The 16-byte pieces of a group's 128-byte unit are stored at
// position piece ^ group, which keeps both the per-thread writes and the
// per-warp reads of the staging buffer free of bank conflicts.  Requires
// N % 16 == 0 (16-byte row stride of the tensor map).
constexpr int PM_SMEM = PM_CHUNKS * 32 * PM_GROUPS * 4 * 2 + 16;   // in + out + barrier

__global__ void __launch_bounds__(PM_THREADS)
permute_tma_kernel(const __grid_constant__ CUtensorMap tmap, uint8_t* __restrict__ out, int64_t K, int64_t N) {
    extern __shared__ __align__(128) uint8_t pm_smem[];
    uint8_t (*tile)[PM_GROUPS * 4] = reinterpret_cast<uint8_t (*)[PM_GROUPS * 4]>(pm_smem);   // [1024][32]
    uint4* staged = reinterpret_cast<uint4*>(pm_smem + PM_CHUNKS * 32 * PM_GROUPS * 4);       // [8][32][8]
    uint64_t* bar_p = reinterpret_cast<uint64_t*>(pm_smem + 2 * PM_CHUNKS * 32 * PM_GROUPS * 4);
    __shared__ int abort_word;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gl = lane & 7, cl = 4 * warp + (lane >> 3);                   // local group, local chunk
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) * PM_GROUPS;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * PM_CHUNKS;
    const uint32_t b = ptx::smem_u32(bar_p);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        abort_word = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    constexpr int BOX_ROWS = 256, NBOX = PM_CHUNKS * 32 / BOX_ROWS;
    if (threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(b, PM_CHUNKS * 32 * PM_GROUPS * 4);
        for (int i = 0; i < NBOX; ++i)
            ptx::tma_load_2d(ptx::smem_u32(&tile[i * BOX_ROWS][0]), &tmap, blockIdx.x * PM_GROUPS * 4,
                             blockIdx.y * PM_CHUNKS * 32 + i * BOX_ROWS, b);
    }
    const bool ok = ptx::mbar_wait(b, 0, &abort_word);
    if (!__syncthreads_and(ok)) {
        if (threadIdx.x == 0) ptx::mbar_drain(b, 0);
        return;
    }
    // this thread's unit: group gl, chunk cl -> 8 pieces of 16 bytes
    uint32_t col[4][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t rr[4], cc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) rr[k] = *reinterpret_cast<const uint32_t*>(&tile[32 * cl + 4 * i + k][4 * gl]);
        transpose4x4(rr, cc);
#pragma unroll
        for (int c = 0; c < 4; ++c) col[c][i] = cc[c];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t w[4] = {col[c][4 * h], col[c][4 * h + 1], col[c][4 * h + 2], col[c][4 * h + 3]};
            uint32_t o[4];
            permute_group16(w, o);
            staged[(gl * PM_CHUNKS + cl) * 8 + ((2 * c + h) ^ gl)] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    __syncthreads();
    // a warp writes 4 chunks x 8 pieces of one group: 512 contiguous bytes
    const int64_t ngroups = N / 4, nchunks = K / 64;
    for (int e = threadIdx.x; e < PM_GROUPS * PM_CHUNKS * 8; e += PM_THREADS) {
        const int g = e / (PM_CHUNKS * 8), rest = e % (PM_CHUNKS * 8), c = rest >> 3, p = rest & 7;
        if (g0 + g < ngroups && c0 + c < nchunks)
            *reinterpret_cast<uint4*>(out + (K / 2) * 4 * (g0 + g) + 128 * (c0 + c) + 16 * p) =
                staged[(g * PM_CHUNKS + c) * 8 + (p ^ g)];
    }
}

w4_status run_permute(const void* packed, void* out, int64_t K, int64_t N, cudaStream_t stream) {
    const int64_t cblocks = ((K / 2) / 32 + PM_CHUNKS - 1) / PM_CHUNKS;
    const int64_t gblocks = (N / 4 + PM_GROUPS - 1) / PM_GROUPS;
    if (cblocks > 65535 || gblocks > 0x7FFFFFFF) return W4_ERR_SHAPE;
    dim3 grid(static_cast<unsigned>(gblocks), static_cast<unsigned>(cblocks));
    if ((N % 16) == 0) {
        auto encode = tensor_map_encoder();
        if (!encode) return W4_ERR_CUDA;
        CUtensorMap tmap;
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K / 2)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(N)};
        cuuint32_t boxd[2] = {PM_GROUPS * 4, 256};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(packed), dims, strides, boxd, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return W4_ERR_CUDA;
        static int smem_set[64];
        if (ensure_smem_limit(permute_tma_kernel, PM_SMEM, smem_set) != cudaSuccess) return W4_ERR_CUDA;
        permute_tma_kernel<<<grid, PM_THREADS, PM_SMEM, stream>>>(tmap, static_cast<uint8_t*>(out), K, N);
        return launch_status(cudaGetLastError());
    }
    permute_kernel<<<grid, PM_THREADS, 0, stream>>>(static_cast<const uint8_t*>(packed), static_cast<uint8_t*>(out),
                                                    K, N);
    return launch_status(cudaGetLastError());
}

// quantize_pack_int4 followed by permute_int4 in one pass over W (the
// single-read kernel writing the permuted layout); W4_ERR_SHAPE unless
// N % 8 == 0, K % 64 == 0 and K <= QC_MAX_K.
w4_status run_quantize_pack_permute(const void* W, void* out, float* scale, int64_t K, int64_t N,
                                    cudaStream_t stream) {
    if ((K % 64) != 0) return W4_ERR_SHAPE;
    return launch_quantize_cluster(W, out, scale, K, N, stream, 1);
}

// quantize_int8 through the single-read kernel; W4_ERR_SHAPE: the caller's
// two-pass kernel (N % 8 != 0 or K > W4_QUANT_PERMUTE_MAX_K)
w4_status run_quantize_int8_single_read(const void* W, void* q, float* scale, int64_t K, int64_t N,
                                        cudaStream_t stream) {
    return launch_quantize_cluster(W, q, scale, K, N, stream, 2);
}

int take_device_error_quant() { return take_unit_device_error(); }
int set_wait_limit_quant(long long clocks) { return set_unit_wait_limit(clocks); }

}  // namespace w4
