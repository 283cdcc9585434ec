// ptq1.cu -- the MMVQ product of ternary weights in PTQ1_0 blocks with x in
// block_q8_1 / PT form (page "三值量化模型的无损压缩": section 2 gives the
// PTQ1_0 block -- qs[24] holding 120 trits five to a byte, qh[2] holding
// 8 trits two bits each, a half scale d -- section 3 the product
// d[r,c] = sum_k W[r,k] x[c,k], section 3.1 the PT planes of x and section
// 3.2 where each trit sits: weight e < 80 at trit e >> 4 of byte e & 15,
// weight 80 + e at trit e >> 3 of byte 16 + (e & 7), the last eight in qh).
//
// Encoding read where the page is silent: trit t is the digit u = t + 1 and
// a byte is sum_p u_p 3^p; qh's 2-bit field j is tail trit j.
//
// Work split: as on the page, a thread's unit of work is one 128-weight
// block i of R rows (R = 4 for C <= 4, else 2), so the x of block i is read
// once for R rows.  GB300 layout of the work: each resident CTA (one of 512
// threads per SM; two of 256 with one column) stages x once and owns a
// contiguous range of row groups; its threads share the groups
// out, a group's blocks split over T / G threads (or one warp) that each
// keep their R x C sums in registers, added at the end in thread order (a
// warp's by a shuffle tree).
// Digit p of a qs byte lines up with PT plane p: for head word m (qs bytes
// 4m .. 4m+3) digit p of its four bytes are elements 16p + 4m .. 16p + 4m + 3,
// i.e. word m of plane p -- one dp4a each.  The integer dots are taken on
// the digits u (0..2) and corrected by the q8_1 block's sum of qs:
//   sum t qs = sum u qs - sum qs.
// Per q8_1 block j (32 elements): d_w * d_x[j] * (sum u qs - sum qs).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace w4 {

namespace {

// threads per CTA: 512, or 256 with one column (two CTAs per SM)
__host__ __device__ constexpr int pq_threads(int64_t C) { return C == 1 ? 256 : 512; }
constexpr int PQ_BLOCK_BYTES = 28;

// Base-3 digits of two values 0..242 held in the 16-bit lanes of x: u[p] is
// digit p of each lane.  floor(q / 3) = (q * 171) >> 9 for q <= 242 (the
// product of one lane never reaches the other; the mask drops what the
// shift brings down from the upper lane).
__device__ __forceinline__ void digits16(uint32_t x, uint32_t (&u)[5]) {
    uint32_t q = x;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t n = ((q * 171u) >> 9) & 0x007F007Fu;
        u[p] = q - 3u * n;
        q = n;
    }
    u[4] = q;
}

// Digit p of each byte of w (bytes 0..242), as the bytes of u[p]: bytes 0, 2
// and 1, 3 go to the low bytes of two words' 16-bit lanes, and the digit
// words are interleaved back, each by one byte permute.
__device__ __forceinline__ void trit_digits(uint32_t w, uint32_t (&u)[5]) {
    uint32_t ue[5], uo[5];
    digits16(__byte_perm(w, 0u, 0x4240), ue);
    digits16(__byte_perm(w, 0u, 0x4341), uo);
#pragma unroll
    for (int p = 0; p < 5; ++p) u[p] = __byte_perm(ue[p], uo[p], 0x6240);
}

// The four 2-bit fields of b (bits 0..7) as the four bytes of a word.
__device__ __forceinline__ uint32_t spread2(uint32_t b) {
    const uint32_t t = b | (b << 6);
    return (t | (t << 12)) & 0x03030303u;
}

__device__ __forceinline__ int dp4(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Shared memory: x transposed so that lanes reading consecutive blocks read
// consecutive words -- xs[c][plane][word][block] (C*K bytes) -- the q8_1
// scales dx[c][block][j] and sums of qs sq[c][block][j]; once every thread
// is done with x, the threads' partial sums part[thread][R][C] take the same
// space.  PTQ1_1's codebook follows both.
struct PqLayout {
    size_t xs, dx, sq, part, code, total;
};

__host__ __device__ inline PqLayout pq_layout(int64_t C, int64_t K, int R, bool super) {
    const int64_t bpr = K / 128;
    PqLayout L;
    L.xs = 0;
    L.dx = size_t(C) * K;
    L.sq = L.dx + size_t(C) * bpr * 4 * 4;
    L.part = 0;
    const size_t x_end = L.sq + size_t(C) * bpr * 4 * 4;
    const size_t part_end = size_t(pq_threads(C)) * R * C * 4;
    L.code = ((x_end > part_end ? x_end : part_end) + 15) / 16 * 16;
    L.total = L.code + (super ? size_t(767 * 8) : 0);
    return L;
}

// Stage x for the CTA: words of planes 0..7 transposed, d of each q8_1
// block as float, and each q8_1 block's sum of qs.
template <int C>
__device__ void stage_x(const uint8_t* __restrict__ pt, uint32_t* xs, float* dx, int* sq, int64_t bpr) {
    const int64_t chunks = int64_t(C) * 8 * bpr;
    for (int64_t t = threadIdx.x; t < chunks; t += pq_threads(C)) {
        const int64_t c = t / (8 * bpr), rem = t % (8 * bpr), p = rem / bpr, i = rem % bpr;
        const uint4 v = *reinterpret_cast<const uint4*>(pt + c * 144 * bpr + 16 * (p * bpr + i));
        uint32_t* dst = xs + ((c * 8 + p) * 4) * bpr + i;
        dst[0] = v.x;
        dst[bpr] = v.y;
        dst[2 * bpr] = v.z;
        dst[3 * bpr] = v.w;
    }
    for (int64_t t = threadIdx.x; t < int64_t(C) * bpr; t += pq_threads(C)) {
        const int64_t c = t / bpr, i = t % bpr;
        const uint4 v = *reinterpret_cast<const uint4*>(pt + c * 144 * bpr + 16 * (8 * bpr + i));
        const uint32_t pr[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            dx[(c * bpr + i) * 4 + j] = __half2float(__ushort_as_half(static_cast<unsigned short>(pr[j] & 0xFFFFu)));
    }
    __syncthreads();
    for (int64_t t = threadIdx.x; t < int64_t(C) * bpr; t += pq_threads(C)) {
        const int64_t c = t / bpr, i = t % bpr;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int s = 0;
#pragma unroll
            for (int pp = 0; pp < 2; ++pp)
#pragma unroll
                for (int m = 0; m < 4; ++m) s = dp4(xs[((c * 8 + 2 * j + pp) * 4 + m) * bpr + i], 0x01010101u, s);
            sq[(c * bpr + i) * 4 + j] = s;
        }
    }
}

// Digit p (0..4) of a byte b (0..242) for a p known only at run time:
// floor(b / 3^p) = (b * ceil(2^15 / 3^p)) >> 15 (exact for b <= 242), then
// mod 3 by the same rule for 3.
__device__ __forceinline__ uint32_t digit_of(uint32_t b, uint32_t p) {
    constexpr uint64_t kRecip = 10923ull | (3641ull << 16) | (1214ull << 32) | (405ull << 48);
    const uint32_t m = p == 0 ? 32768u : static_cast<uint32_t>(kRecip >> (16 * (p - 1))) & 0xFFFFu;
    const uint32_t q = (b * m) >> 15;
    return q - 3u * ((q * 10923u) >> 15);
}

// One item of R rows of the same block i: qs[r] are the block's six qs
// words of row r, tail[r] the digits (0..2) of weights 120 .. 127 as two
// words, dw[r] the block's scale.  Writes the R*C partial sums.
template <int C, int R>
__device__ __forceinline__ void mmvq_item(const uint32_t (&qs)[R][6], const uint32_t (&tail)[R][2],
                                          const float (&dw)[R], const uint32_t* xs, const float* dx, const int* sq,
                                          int64_t bpr, int64_t i, float (&acc)[R][C]) {
    int dot[R][C][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j) dot[r][c][j] = 0;

    // head: qs words 0..3, digit p -> plane p, word m; q8_1 block p / 2
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t u[R][5];
#pragma unroll
        for (int r = 0; r < R; ++r) trit_digits(qs[r][m], u[r]);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uint32_t xw[5];
#pragma unroll
            for (int p = 0; p < 5; ++p) xw[p] = xs[((c * 8 + p) * 4 + m) * bpr + i];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int p = 0; p < 5; ++p) dot[r][c][p / 2] = dp4(u[r][p], xw[p], dot[r][c][p / 2]);
        }
    }
    // middle: qs words 4, 5 (m2 = 0, 1); digit p -> element 80 + 8p + 4 m2,
    // i.e. plane 5 + p / 2, word 2 (p % 2) + m2; q8_1 block 2 for p < 2, else 3
#pragma unroll
    for (int m2 = 0; m2 < 2; ++m2) {
        uint32_t u[R][5];
#pragma unroll
        for (int r = 0; r < R; ++r) trit_digits(qs[r][4 + m2], u[r]);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uint32_t xw[5];
#pragma unroll
            for (int p = 0; p < 5; ++p) xw[p] = xs[((c * 8 + 5 + p / 2) * 4 + 2 * (p % 2) + m2) * bpr + i];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int p = 0; p < 5; ++p) dot[r][c][p < 2 ? 2 : 3] = dp4(u[r][p], xw[p], dot[r][c][p < 2 ? 2 : 3]);
        }
    }
    // tail: weights 120 .. 127 are plane 7, words 2 and 3
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const uint32_t x2 = xs[((c * 8 + 7) * 4 + 2) * bpr + i], x3 = xs[((c * 8 + 7) * 4 + 3) * bpr + i];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            dot[r][c][3] = dp4(tail[r][0], x2, dot[r][c][3]);
            dot[r][c][3] = dp4(tail[r][1], x3, dot[r][c][3]);
        }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) {
        // the block's four scales and sums of qs: one 16-byte load each
        const float4 dx4 = *reinterpret_cast<const float4*>(dx + (c * bpr + i) * 4);
        const int4 sq4 = *reinterpret_cast<const int4*>(sq + (c * bpr + i) * 4);
        const float dxj[4] = {dx4.x, dx4.y, dx4.z, dx4.w};
        const int sqj[4] = {sq4.x, sq4.y, sq4.z, sq4.w};
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) a = fmaf(dxj[j], static_cast<float>(dot[r][c][j] - sqj[j]), a);
            acc[r][c] = fmaf(dw[r], a, acc[r][c]);
        }
    }
}

// PTQ1_0: the block's seven words are qs (0..5), then qh | d << 16.
template <int C, int R>
__device__ __forceinline__ void ptq1_0_item(const uint8_t* __restrict__ blocks, const uint32_t* xs,
                                             const float* dx, const int* sq, int64_t N, int64_t bpr, int64_t row0,
                                             int64_t i, float (&acc)[R][C]) {
    uint32_t qs[R][6], tail[R][2];
    float dw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + r;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(blocks + (row * bpr + i) * PQ_BLOCK_BYTES);
#pragma unroll
        for (int q = 0; q < 6; ++q) qs[r][q] = row < N ? __ldg(src + q) : 0u;
        const uint32_t w6 = row < N ? __ldg(src + 6) : 0u;   // a missing row has d = 0
        tail[r][0] = spread2(w6 & 0xFFu);
        tail[r][1] = spread2((w6 >> 8) & 0xFFu);
        dw[r] = __half2float(__ushort_as_half(static_cast<unsigned short>(w6 >> 16)));
    }
    mmvq_item<C, R>(qs, tail, dw, xs, dx, sq, bpr, i, acc);
}

// PTQ1_1 superblock (216 bytes): qs[192] (block s at 24 s), qh[13] at 192,
// eight 10-bit mantissas at 205, the exponents byte at 215.  Block s's tail
// trit j is digit (8 s + j) mod 5 of qh byte (8 s + j) / 5; digit 4 of qh
// byte 12 is the free trit f; the pattern index exponents + 256 f names a
// codebook entry (< 767) or, at 767, the escape table entry of the
// superblock's index.  A pattern that cannot be found records ERR_PATTERN
// and gives d = 0.
constexpr int ERR_PATTERN = 2;
constexpr int PTQ1_1_BYTES = 216;

__device__ __forceinline__ const uint8_t* find_escape(const int64_t* __restrict__ esc_idx,
                                                      const uint8_t* __restrict__ esc_patt, int64_t n_esc,
                                                      int64_t g) {
    int64_t lo = 0, hi = n_esc;   // esc_idx ascending
    while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (esc_idx[mid] < g) lo = mid + 1;
        else hi = mid;
    }
    return (lo < n_esc && esc_idx[lo] == g) ? esc_patt + 8 * lo : nullptr;
}

template <int C, int R>
__device__ __forceinline__ void ptq1_1_item(const uint8_t* __restrict__ sblocks, const uint8_t* code,
                                             int64_t n_code, const int64_t* __restrict__ esc_idx,
                                             const uint8_t* __restrict__ esc_patt, int64_t n_esc,
                                             const uint32_t* xs, const float* dx, const int* sq, int64_t N,
                                             int64_t bpr, int64_t row0, int64_t i, float (&acc)[R][C]) {
    const int64_t sbpr = (bpr + 7) / 8, sb = i / 8;
    const uint32_t s = static_cast<uint32_t>(i % 8);
    uint32_t qs[R][6], tail[R][2];
    float dw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = row0 + r;
        const int64_t g = row * sbpr + sb;
        const uint32_t* base = reinterpret_cast<const uint32_t*>(sblocks + g * PTQ1_1_BYTES);
        uint32_t h[6];
#pragma unroll
        for (int q = 0; q < 6; ++q) qs[r][q] = row < N ? __ldg(base + 6 * s + q) : 0u;
#pragma unroll
        for (int q = 0; q < 6; ++q) h[q] = row < N ? __ldg(base + 48 + q) : 0u;   // bytes 192 .. 215
        // tail digits: trit u = 8 s + j is digit u % 5 of qh byte u / 5
        uint32_t t0 = 0, t1 = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t u = 8 * s + j, n = (u * 205u) >> 10, p = u - 5 * n;
            const uint32_t hw = n < 4 ? h[0] : n < 8 ? h[1] : n < 12 ? h[2] : h[3];
            const uint32_t dg = digit_of((hw >> (8 * (n & 3))) & 0xFFu, p);
            if (j < 4) t0 |= dg << (8 * j);
            else t1 |= dg << (8 * (j - 4));
        }
        tail[r][0] = t0;
        tail[r][1] = t1;
        // mantissa s: bits 10 s .. 10 s + 9 of bytes 205 .. 214
        const uint64_t lo64 = uint64_t(h[3] >> 8) | (uint64_t(h[4]) << 24) | (uint64_t(h[5] & 0xFFu) << 56);
        const uint64_t hi16 = (h[5] >> 8) & 0xFFFFu;
        const uint32_t o = 10 * s;
        const uint64_t v = o < 64 ? ((lo64 >> o) | (o > 54 ? (hi16 << (64 - o)) : 0ull)) : (hi16 >> (o - 64));
        const uint32_t mant = static_cast<uint32_t>(v) & 0x3FFu;
        // exponent from the pattern
        const uint32_t idx = (h[5] >> 24) + 256u * digit_of(h[3] & 0xFFu, 4);
        const uint8_t* pat = nullptr;
        if (row < N) {
            if (idx < 767u) pat = int64_t(idx) < n_code ? code + 8 * idx : nullptr;
            else pat = find_escape(esc_idx, esc_patt, n_esc, g);
            if (!pat) atomicCAS(&g_device_error, 0, ERR_PATTERN);
        }
        const uint32_t e = pat ? pat[s] : 0u;
        dw[r] = pat ? __half2float(__ushort_as_half(static_cast<unsigned short>((e << 10) | mant))) : 0.f;
    }
    mmvq_item<C, R>(qs, tail, dw, xs, dx, sq, bpr, i, acc);
}

// CTA b takes the row groups [b G, b G + G) (R rows each).  With G <= T
// threads, group g goes to threads [g tpg, g tpg + tpg), tpg = T / G (or 32,
// a warp per group, when that is not slower; see threads_per_group): thread
// j of them takes blocks j, j + tpg, ... in order and keeps R*C sums in
// registers.  A warp's sums meet by a shuffle tree; otherwise, after a
// barrier, the sums go to shared memory (over the staged x) and the group's
// first thread adds them in thread order.  With G > T every thread takes
// whole groups (tpg = 1) and stores them itself.  d is fp32 [C][N].
// PTQ1_1 also copies the codebook into shared memory.
template <int C, int R, bool SUPER>
__global__ void __launch_bounds__(pq_threads(C))
mmvq_ptq1_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ codebook, int64_t n_code,
                 const int64_t* __restrict__ esc_idx, const uint8_t* __restrict__ esc_patt, int64_t n_esc,
                 const uint8_t* __restrict__ pt, float* __restrict__ d, int64_t N, int64_t K, int64_t G) {
    constexpr int PQ_THREADS = pq_threads(C);
    extern __shared__ __align__(16) uint8_t smem[];
    const int64_t bpr = K / 128, groups = (N + R - 1) / R;
    const PqLayout L = pq_layout(C, K, R, SUPER);
    uint32_t* xs = reinterpret_cast<uint32_t*>(smem + L.xs);
    float* dx = reinterpret_cast<float*>(smem + L.dx);
    int* sq = reinterpret_cast<int*>(smem + L.sq);
    float* part = reinterpret_cast<float*>(smem + L.part);
    uint8_t* code = smem + L.code;
    if (SUPER)
        for (int64_t t = threadIdx.x; t < 8 * n_code; t += PQ_THREADS) code[t] = codebook[t];
    stage_x<C>(pt, xs, dx, sq, bpr);
    __syncthreads();
    const int64_t g0 = int64_t(blockIdx.x) * G;
    const int64_t gn = groups - g0 < G ? groups - g0 : G;   // groups of this CTA
    const int tpg = threads_per_group(PQ_THREADS, gn, bpr);
    const int j = static_cast<int>(threadIdx.x) % tpg;
    const int gstep = PQ_THREADS / tpg;
    float acc[R][C];
    for (int64_t g = threadIdx.x / tpg; g < gn; g += gstep) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) acc[r][c] = 0.f;
        const int64_t row0 = (g0 + g) * R;
        for (int64_t i = j; i < bpr; i += tpg) {
            if (SUPER)
                ptq1_1_item<C, R>(w, code, n_code, esc_idx, esc_patt, n_esc, xs, dx, sq, N, bpr, row0, i, acc);
            else
                ptq1_0_item<C, R>(w, xs, dx, sq, N, bpr, row0, i, acc);
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
        if (tpg == 1 || (tpg == 32 && j == 0)) {
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int c = 0; c < C; ++c)
                    if (row0 + r < N) d[c * N + row0 + r] = acc[r][c];
        }
    }
    if (tpg == 1 || tpg == 32) return;   // (otherwise one round: T / tpg >= gn)
    __syncthreads();   // every thread is done with x: its space takes the partial sums
    if (threadIdx.x / tpg < gn) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) part[(threadIdx.x * R + r) * C + c] = acc[r][c];
    }
    __syncthreads();
    for (int64_t o = threadIdx.x; o < gn * R * C; o += PQ_THREADS) {
        const int64_t g = o / (R * C), r = (o / C) % R, c = o % C;
        const int64_t row = (g0 + g) * R + r;
        if (row >= N) continue;
        float sum = 0.f;
        for (int t = 0; t < tpg; ++t) sum += part[((g * tpg + t) * R + r) * C + c];
        d[c * N + row] = sum;
    }
}

template <int C, bool SUPER>
w4_status launch_ptq1(const void* w, const void* codebook, int64_t n_code, const void* esc_idx,
                      const void* esc_patt, int64_t n_esc, const void* pt, float* d, int64_t N, int64_t K,
                      cudaStream_t stream) {
    constexpr int R = C <= 4 ? 4 : 2;
    static int smem_set[64];
    const int64_t groups = (N + R - 1) / R;
    const int sms = sm_count();
    if (sms <= 0) return W4_ERR_CUDA;
    const size_t smem = pq_layout(C, K, R, SUPER).total;
    if (smem > size_t(W4_W4A8_MAX_SMEM)) return W4_ERR_SHAPE;
    auto kern = mmvq_ptq1_kernel<C, R, SUPER>;
    if (ensure_smem_limit(kern, static_cast<int>(smem), smem_set) != cudaSuccess) return W4_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, pq_threads(C), smem) != cudaSuccess || per_sm < 1)
        return W4_ERR_CUDA;
    // as many CTAs as are resident at once, each a contiguous range of row groups
    int64_t ctas = int64_t(sms) * per_sm;
    if (ctas > groups) ctas = groups;
    if (ctas < 1) ctas = 1;
    const int64_t G = groups > 0 ? (groups + ctas - 1) / ctas : 1;
    ctas = groups > 0 ? (groups + G - 1) / G : 1;
    kern<<<static_cast<unsigned>(ctas), pq_threads(C), smem, stream>>>(
        static_cast<const uint8_t*>(w), static_cast<const uint8_t*>(codebook), n_code,
        static_cast<const int64_t*>(esc_idx), static_cast<const uint8_t*>(esc_patt), n_esc,
        static_cast<const uint8_t*>(pt), d, N, K, G);
    return launch_status(cudaGetLastError());
}

template <bool SUPER>
w4_status run_ptq1(const void* w, const void* codebook, int64_t n_code, const void* esc_idx, const void* esc_patt,
                   int64_t n_esc, const void* pt, float* d, int64_t N, int64_t K, int64_t C, cudaStream_t stream) {
    switch (C) {
#define W4_PTQ1_CASE(CC) \
    case CC: return launch_ptq1<CC, SUPER>(w, codebook, n_code, esc_idx, esc_patt, n_esc, pt, d, N, K, stream);
        W4_PTQ1_CASE(1) W4_PTQ1_CASE(2) W4_PTQ1_CASE(3) W4_PTQ1_CASE(4)
        W4_PTQ1_CASE(5) W4_PTQ1_CASE(6) W4_PTQ1_CASE(7) W4_PTQ1_CASE(8)
#undef W4_PTQ1_CASE
        default: return W4_ERR_SHAPE;
    }
}

}  // namespace

bool ptq1_fits(int64_t C, int64_t K, bool super) {
    const int R = C <= 4 ? 4 : 2;
    return pq_layout(C, K, R, super).total <= size_t(W4_W4A8_MAX_SMEM);
}

w4_status run_mmvq_ptq1_0(const void* blocks, const void* pt, float* d, int64_t N, int64_t K, int64_t C,
                          cudaStream_t stream) {
    return run_ptq1<false>(blocks, nullptr, 0, nullptr, nullptr, 0, pt, d, N, K, C, stream);
}

w4_status run_mmvq_ptq1_1(const void* sblocks, const void* codebook, int64_t n_code, const void* esc_idx,
                          const void* esc_patt, int64_t n_esc, const void* pt, float* d, int64_t N, int64_t K,
                          int64_t C, cudaStream_t stream) {
    return run_ptq1<true>(sblocks, codebook, n_code, esc_idx, esc_patt, n_esc, pt, d, N, K, C, stream);
}

int take_device_error_ptq1() { return take_unit_device_error(); }
int set_wait_limit_ptq1(long long clocks) { return set_unit_wait_limit(clocks); }

}  // namespace w4
