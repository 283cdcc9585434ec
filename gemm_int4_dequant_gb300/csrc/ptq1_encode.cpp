// ptq1_encode.cpp -- host-side conversion of ternary PTQ1_0 blocks into
// PTQ1_1 superblocks (page "三值量化模型的无损压缩", section 2 "权重的无损压缩":
// eight blocks share one 216-byte superblock; their 64 tail trits are
// re-packed five to a byte, the sign of every d is dropped, the mantissas
// kept, and the eight exponents replaced by an index into a per-tensor
// table of exponent patterns, with 767 sending the reader to an escape
// table).  This is offline model conversion: it runs on host memory.
//
// Layout read where the page is silent (the same reading as the MMVQ
// kernels): superblock fields in the struct's order (qs at 0, qh at 192,
// mantissas at 205, exponents at 215); block s's qs at 24 s; tail trit j of
// block s as base-3 digit (8 s + j) mod 5 of qh byte (8 s + j) / 5, digit 4
// of qh byte 12 being the free trit f; mantissa s at bits 10 s .. 10 s + 9
// of the little-endian 80-bit string; pattern index = exponents + 256 f.
// The table holds the most frequent patterns (ties: the smaller pattern,
// read as a 40-bit number with block 0's exponent on top).  Rows of K/128
// blocks are padded to whole superblocks with zero trits and d = +0.

#include <algorithm>
#include <cstring>
#include <unordered_map>
#include <utility>
#include <vector>

#include "w4.h"

namespace {

constexpr int64_t kBlockBytes = 28;
constexpr int64_t kSuperBytes = 216;
constexpr int kQh = 192, kMant = 205, kExp = 215;
constexpr int kEscape = 767;
constexpr int kPow3[5] = {1, 3, 9, 27, 81};

struct Block {
    const uint8_t* p;   // nullptr: a padding block past the row's end
    uint16_t d() const { return p ? static_cast<uint16_t>(p[26] | (p[27] << 8)) : 0; }
    uint32_t exponent() const { return (d() >> 10) & 0x1Fu; }
    // digit (t + 1) of tail weight j: the 2-bit field j of qh
    uint32_t tail(int j) const { return p ? ((p[24] | (p[25] << 8)) >> (2 * j)) & 3u : 1u; }
};

Block block_at(const uint8_t* blocks, int64_t bpr, int64_t r, int64_t b) {
    return Block{b < bpr ? blocks + (r * bpr + b) * kBlockBytes : nullptr};
}

uint64_t pattern_key(const uint8_t* blocks, int64_t bpr, int64_t r, int64_t sb) {
    uint64_t key = 0;
    for (int s = 0; s < 8; ++s) key = (key << 5) | block_at(blocks, bpr, r, 8 * sb + s).exponent();
    return key;
}

bool valid_blocks(const uint8_t* blocks, int64_t n_blocks) {
    for (int64_t i = 0; i < n_blocks; ++i) {
        const uint8_t* p = blocks + i * kBlockBytes;
        for (int q = 0; q < 24; ++q)
            if (p[q] > 242) return false;   // five base-3 digits
        const uint32_t qh = p[24] | (p[25] << 8);
        for (int j = 0; j < 8; ++j)
            if (((qh >> (2 * j)) & 3u) == 3u) return false;
    }
    return true;
}

bool checked_dims(int64_t N, int64_t K) { return N >= 0 && K >= 0 && K % 128 == 0; }

}  // namespace

extern "C" {

w4_status ptq1_1_codebook(const void* blocks, int64_t N, int64_t K, void* codebook, int64_t* n_code) {
    if (!checked_dims(N, K)) return W4_ERR_SHAPE;
    if (!n_code || !codebook || (N > 0 && K > 0 && !blocks)) return W4_ERR_NULL;
    const int64_t bpr = K / 128, sbpr = (bpr + 7) / 8;
    const auto* b = static_cast<const uint8_t*>(blocks);
    std::unordered_map<uint64_t, int64_t> count;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t sb = 0; sb < sbpr; ++sb) ++count[pattern_key(b, bpr, r, sb)];
    std::vector<std::pair<int64_t, uint64_t>> order;   // (count, pattern)
    order.reserve(count.size());
    for (const auto& kv : count) order.emplace_back(kv.second, kv.first);
    std::sort(order.begin(), order.end(), [](const auto& a, const auto& c) {
        return a.first != c.first ? a.first > c.first : a.second < c.second;
    });
    const int64_t n = std::min<int64_t>(static_cast<int64_t>(order.size()), kEscape);
    auto* out = static_cast<uint8_t*>(codebook);
    for (int64_t i = 0; i < n; ++i)
        for (int s = 0; s < 8; ++s) out[8 * i + s] = static_cast<uint8_t>((order[i].second >> (5 * (7 - s))) & 0x1Fu);
    *n_code = n;
    return W4_OK;
}

w4_status ptq1_1_encode(const void* blocks, int64_t N, int64_t K, const void* codebook, int64_t n_code,
                        void* sblocks, void* esc_idx, void* esc_patt, int64_t max_esc, int64_t* n_esc) {
    if (!checked_dims(N, K) || n_code < 0 || n_code > kEscape || max_esc < 0) return W4_ERR_SHAPE;
    if (!n_esc || (n_code > 0 && !codebook) || (max_esc > 0 && (!esc_idx || !esc_patt))) return W4_ERR_NULL;
    const int64_t bpr = K / 128, sbpr = (bpr + 7) / 8;
    if (N > 0 && K > 0 && (!blocks || !sblocks)) return W4_ERR_NULL;
    const auto* b = static_cast<const uint8_t*>(blocks);
    if (N > 0 && K > 0 && !valid_blocks(b, N * bpr)) return W4_ERR_VALUE;
    for (int64_t i = 0; i < N * bpr; ++i)
        if (b[i * kBlockBytes + 27] & 0x80u) return W4_ERR_VALUE;   // the superblock keeps no sign

    const auto* code = static_cast<const uint8_t*>(codebook);
    std::unordered_map<uint64_t, int64_t> index_of;
    for (int64_t i = 0; i < n_code; ++i) {
        uint64_t key = 0;
        for (int s = 0; s < 8; ++s) key = (key << 5) | (code[8 * i + s] & 0x1Fu);
        index_of.emplace(key, i);   // the first entry of a repeated pattern wins
    }
    auto* out = static_cast<uint8_t*>(sblocks);
    auto* eidx = static_cast<int64_t*>(esc_idx);
    auto* epat = static_cast<uint8_t*>(esc_patt);
    int64_t escapes = 0;
    for (int64_t r = 0; r < N; ++r) {
        for (int64_t sb = 0; sb < sbpr; ++sb) {
            const int64_t g = r * sbpr + sb;
            uint8_t* o = out + g * kSuperBytes;
            std::memset(o, 0, kSuperBytes);
            uint64_t mant = 0;   // bits 0..63 of the 80-bit mantissa string
            uint32_t mant_hi = 0;
            for (int s = 0; s < 8; ++s) {
                const Block blk = block_at(b, bpr, r, 8 * sb + s);
                if (blk.p) std::memcpy(o + 24 * s, blk.p, 24);
                else std::memset(o + 24 * s, 1 + 3 + 9 + 27 + 81, 24);   // every trit 0
                for (int j = 0; j < 8; ++j) {
                    const int t = 8 * s + j;
                    o[kQh + t / 5] = static_cast<uint8_t>(o[kQh + t / 5] + blk.tail(j) * kPow3[t % 5]);
                }
                const uint64_t m = blk.d() & 0x3FFu;
                const int at = 10 * s;
                if (at + 10 <= 64) {
                    mant |= m << at;
                } else if (at < 64) {
                    mant |= m << at;   // the low bits that fit
                    mant_hi |= static_cast<uint32_t>(m >> (64 - at));
                } else {
                    mant_hi |= static_cast<uint32_t>(m << (at - 64));
                }
            }
            for (int k = 0; k < 8; ++k) o[kMant + k] = static_cast<uint8_t>(mant >> (8 * k));
            o[kMant + 8] = static_cast<uint8_t>(mant_hi & 0xFFu);
            o[kMant + 9] = static_cast<uint8_t>((mant_hi >> 8) & 0xFFu);
            const uint64_t key = pattern_key(b, bpr, r, sb);
            const auto it = index_of.find(key);
            int64_t idx = kEscape;
            if (it != index_of.end()) {
                idx = it->second;
            } else {
                if (escapes >= max_esc) return W4_ERR_SHAPE;
                eidx[escapes] = g;
                for (int s = 0; s < 8; ++s) epat[8 * escapes + s] = static_cast<uint8_t>((key >> (5 * (7 - s))) & 0x1Fu);
                ++escapes;
            }
            o[kExp] = static_cast<uint8_t>(idx % 256);
            o[kQh + 12] = static_cast<uint8_t>(o[kQh + 12] + (idx / 256) * kPow3[4]);
        }
    }
    *n_esc = escapes;
    return W4_OK;
}

}  // extern "C"
