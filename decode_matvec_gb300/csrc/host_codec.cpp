// Host-side codec of the decode-and-multiply library: dictionary generation
// (QMoE page, Algorithm 1), the greedy longest-match packer ("Encoding
// (compression time)"), the kernel-private compact dictionary and the RVQ
// encoder ("Quantization as Cache Amplification", section "Codec").
//
// Built with -ffp-contract=off: the float64 arithmetic of the RVQ encoder must
// round exactly as written so that independent exact encoders agree bit for bit.

#include <algorithm>
#include <array>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "qmoe.h"
#include "host_common.h"

namespace qmoe {

static thread_local std::string g_last_error;

int fail(int status, const std::string& msg) {
    g_last_error = msg;
    return status;
}

const char* last_error() { return g_last_error.c_str(); }
void clear_error() { g_last_error.clear(); }

}  // namespace qmoe

using qmoe::fail;

extern "C" const char* qmoe_last_error(void) { return qmoe::last_error(); }

// ---------------------------------------------------------------------------
// Algorithm 1
// ---------------------------------------------------------------------------
namespace {

// A sequence of up to 28 ternary symbols.  `key` holds symbol i at bits
// [55-2i : 54-2i] (first symbol most significant), zero-padded, so comparing
// (key, len) orders sequences lexicographically with a prefix first.
struct Seq {
    double prio;
    uint64_t key;
    int len;
    int n0;
};

struct HeapLess {
    // std::priority_queue pops the "largest": the highest priority, then the
    // lexicographically smallest sequence.
    bool operator()(const Seq& a, const Seq& b) const {
        if (a.prio != b.prio) return a.prio < b.prio;
        if (a.key != b.key) return a.key > b.key;
        return a.len > b.len;
    }
};

inline int sym_at(uint64_t key, int i) { return (int)((key >> (54 - 2 * i)) & 3u); }

}  // namespace

extern "C" int qmoe_encode_dictionary(const int8_t* symbols, size_t n, double p0,
                                      uint32_t* dict_words, double* p0_used) {
    qmoe::clear_error();
    if (!dict_words) return fail(QMOE_EINVAL, "qmoe_encode_dictionary: dict_words is NULL");
    if (symbols) {
        if (n == 0) return fail(QMOE_EINVAL, "qmoe_encode_dictionary: no symbols given");
        size_t zeros = 0;
        for (size_t i = 0; i < n; ++i) {
            int8_t v = symbols[i];
            if (v < -1 || v > 1) return fail(QMOE_EINVAL, "qmoe_encode_dictionary: symbol outside {-1,0,1}");
            zeros += (v == 0);
        }
        p0 = (double)zeros / (double)n;
    }
    if (!(p0 > 0.0 && p0 < 1.0)) return fail(QMOE_EINVAL, "qmoe_encode_dictionary: p0 must lie in (0,1)");
    if (p0_used) *p0_used = p0;

    const double lp0 = std::log(p0);
    const double lq = std::log((1.0 - p0) / 2.0);
    std::priority_queue<Seq, std::vector<Seq>, HeapLess> heap;
    heap.push(Seq{-0.0, 0, 0, 0});
    int count = 0;
    while (count < QMOE_DICT_ENTRIES) {
        Seq s = heap.top();
        heap.pop();
        if (s.len >= 1 && s.len <= QMOE_MAX_RUN) {
            uint32_t pairs = (uint32_t)(s.len / 2);
            uint32_t w[2] = {pairs, pairs};
            for (int i = 0; i < s.len; ++i)
                w[i / 14] |= (uint32_t)sym_at(s.key, i) << (4 + 2 * (i % 14));
            dict_words[2 * count] = w[0];
            dict_words[2 * count + 1] = w[1];
            ++count;
        }
        if (s.len < QMOE_MAX_RUN) {
            for (int t1 = 0; t1 < 3; ++t1)
                for (int t2 = 0; t2 < 3; ++t2) {
                    Seq c;
                    c.len = s.len + 2;
                    c.key = s.key | ((uint64_t)t1 << (54 - 2 * s.len)) | ((uint64_t)t2 << (52 - 2 * s.len));
                    c.n0 = s.n0 + (t1 == 0) + (t2 == 0);
                    // recomputed from the counts, as the priority of equal-count
                    // sequences must tie exactly
                    c.prio = (double)c.n0 * lp0 + (double)(c.len - c.n0) * lq;
                    heap.push(c);
                }
        }
    }
    return QMOE_OK;
}

// ---------------------------------------------------------------------------
// Packer: a trie over ternary pairs (9 children per node)
// ---------------------------------------------------------------------------
namespace {

struct Trie {
    std::vector<int32_t> child;   // [node*9 + pair]
    std::vector<int32_t> code;    // codeword of the node's sequence, or -1
    uint64_t hash = 0;
    bool ok = false;
};

uint64_t fnv1a(const uint32_t* w, size_t n) {
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= w[i];
        h *= 1099511628211ull;
    }
    return h;
}

int build_trie(const uint32_t* words, Trie& t) {
    t.child.assign(9, -1);
    t.code.assign(1, -1);
    for (int e = 0; e < QMOE_DICT_ENTRIES; ++e) {
        uint32_t w0 = words[2 * e], w1 = words[2 * e + 1];
        int pairs = (int)(w0 & 15u);
        if ((w1 & 15u) != (uint32_t)pairs || pairs < 1 || pairs > 14)
            return fail(QMOE_EFORMAT, "qmoe_pack: dictionary entry with a bad pair count");
        int node = 0;
        for (int p = 0; p < pairs; ++p) {
            int i0 = 2 * p, i1 = 2 * p + 1;
            uint32_t a = ((i0 < 14 ? w0 : w1) >> (4 + 2 * (i0 % 14))) & 3u;
            uint32_t b = ((i1 < 14 ? w0 : w1) >> (4 + 2 * (i1 % 14))) & 3u;
            if (a == 3 || b == 3) return fail(QMOE_EFORMAT, "qmoe_pack: dictionary symbol 3");
            int pr = (int)(a * 3 + b);
            int nxt = t.child[(size_t)node * 9 + pr];
            if (nxt < 0) {
                nxt = (int)t.code.size();
                t.code.push_back(-1);
                t.child.insert(t.child.end(), 9, -1);
                t.child[(size_t)node * 9 + pr] = nxt;
            }
            node = nxt;
        }
        if (t.code[node] < 0) t.code[node] = e;   // first (most probable) code wins
    }
    t.ok = true;
    return QMOE_OK;
}

std::mutex g_trie_mu;
std::shared_ptr<Trie> g_trie;

int get_trie(const uint32_t* words, std::shared_ptr<Trie>& out) {
    uint64_t h = fnv1a(words, QMOE_DICT_WORDS);
    std::lock_guard<std::mutex> lk(g_trie_mu);
    if (g_trie && g_trie->ok && g_trie->hash == h) {
        out = g_trie;
        return QMOE_OK;
    }
    auto t = std::make_shared<Trie>();
    int st = build_trie(words, *t);
    if (st) return st;
    t->hash = h;
    g_trie = t;
    out = t;
    return QMOE_OK;
}

}  // namespace

extern "C" int qmoe_pack(const int8_t* tern, int rows, int cols, int block,
                         const uint32_t* dict_words, uint16_t* codes, size_t codes_cap,
                         size_t* n_codes, uint32_t* blk_off) {
    qmoe::clear_error();
    if (!tern && (size_t)rows * (size_t)cols != 0) return fail(QMOE_EINVAL, "qmoe_pack: tern is NULL");
    if (!dict_words || !n_codes) return fail(QMOE_EINVAL, "qmoe_pack: NULL argument");
    if (rows < 0 || cols <= 0 || (cols & 1) || block <= 0 || (block & 1))
        return fail(QMOE_EINVAL, "qmoe_pack: rows >= 0, cols > 0 even and block > 0 even required");
    if (codes && !blk_off) return fail(QMOE_EINVAL, "qmoe_pack: blk_off is NULL");
    std::shared_ptr<Trie> trie;
    int st = get_trie(dict_words, trie);
    if (st) return st;
    const int nb = (cols + block - 1) / block;
    size_t count = 0;
    bool overflow = false;
    for (int r = 0; r < rows; ++r) {
        const int8_t* row = tern + (size_t)r * cols;
        for (int b = 0; b < nb; ++b) {
            if (blk_off && !overflow) blk_off[(size_t)r * nb + b] = (uint32_t)count;
            const int c_end = std::min(cols, (b + 1) * block);
            int pos = b * block;
            while (pos < c_end) {
                int node = 0, best = -1, best_len = 0;
                for (int p = 0; p < 14 && pos + 2 * p + 2 <= c_end; ++p) {
                    int8_t va = row[pos + 2 * p], vb = row[pos + 2 * p + 1];
                    if (va < -1 || va > 1 || vb < -1 || vb > 1)
                        return fail(QMOE_EINVAL, "qmoe_pack: weight outside {-1,0,1}");
                    int a = va == 0 ? 0 : (va < 0 ? 1 : 2);
                    int bb = vb == 0 ? 0 : (vb < 0 ? 1 : 2);
                    int nxt = trie->child[(size_t)node * 9 + a * 3 + bb];
                    if (nxt < 0) break;
                    node = nxt;
                    if (trie->code[node] >= 0) {
                        best = trie->code[node];
                        best_len = 2 * p + 2;
                    }
                }
                if (best < 0) return fail(QMOE_EFORMAT, "qmoe_pack: the dictionary cannot express a pair");
                if (codes) {
                    if (count < codes_cap) codes[count] = (uint16_t)best;
                    else overflow = true;
                }
                ++count;
                pos += best_len;
            }
        }
    }
    if (blk_off && !overflow) blk_off[(size_t)rows * nb] = (uint32_t)count;
    *n_codes = count;
    if (count > 0xFFFFFFFFull && blk_off) return fail(QMOE_EINVAL, "qmoe_pack: more than 2^32 codewords in one matrix");
    if (codes && overflow) return fail(QMOE_ECAPACITY, "qmoe_pack: codes buffer too small");
    return QMOE_OK;
}

// ---------------------------------------------------------------------------
// Compact block offsets: per-row uint32 starts and per-block uint8 codeword counts
// ---------------------------------------------------------------------------
extern "C" int qmoe_offsets_compact(const uint32_t* blk_off, int rows, int nb, uint32_t* row_off, uint8_t* blk_len) {
    qmoe::clear_error();
    if (!blk_off || !row_off || rows < 1 || nb < 1 || (nb > 1 && !blk_len))
        return fail(QMOE_EINVAL, "qmoe_offsets_compact: bad arguments");
    if (blk_off[0] != 0) return fail(QMOE_EFORMAT, "qmoe_offsets_compact: offsets must start at 0");
    for (int r = 0; r < rows; ++r) {
        const uint32_t* o = blk_off + (size_t)r * nb;
        row_off[r] = o[0];
        for (int b = 0; b < nb; ++b) {
            if (o[b + 1] < o[b]) return fail(QMOE_EFORMAT, "qmoe_offsets_compact: offsets decrease");
            if (o[b + 1] - o[b] > 255u) return fail(QMOE_EFORMAT, "qmoe_offsets_compact: a block of more than 255 codewords");
            if (b < nb - 1) blk_len[(size_t)r * (nb - 1) + b] = (uint8_t)(o[b + 1] - o[b]);
        }
    }
    row_off[rows] = blk_off[(size_t)rows * nb];
    return QMOE_OK;
}

// ---------------------------------------------------------------------------
// Compact dictionary: uint16 plane [65536], uint8 plane [65536], then both again as one
// uint32 plane [65536] (uint16 entry | uint8 entry << 16) for reads from global memory;
// slot = 2*position + (1 if the weight is w_min).
//   up to three nonzeros:      A [3:0] pair count, [9:4] slot 0, [15:10] slot 1 (63 = empty)
//                              B [5:0] slot 2 (63 = empty), [7:6] = 0
//   four nonzeros, all in the  A [3:0] pair count, [7:4] slot 0, [11:8] slot 1, [15:12] slot 2
//   first eight positions:     B [3:0] slot 3, [6] = 1 (four 4-bit slots), [7] = 0
//   anything else:             A [3:0] pair count, [15:4] = 0xFFF; B = 0xBF ([7] = 1: the kernels
//                              read the entry's canonical words)
// ---------------------------------------------------------------------------
extern "C" int qmoe_dict_compact(const uint32_t* dict_words, void* compact) {
    qmoe::clear_error();
    if (!dict_words || !compact) return fail(QMOE_EINVAL, "qmoe_dict_compact: NULL argument");
    uint16_t* pa = (uint16_t*)compact;
    uint8_t* pb = (uint8_t*)compact + 2 * QMOE_DICT_ENTRIES;
    uint32_t* pw = (uint32_t*)((uint8_t*)compact + 3 * QMOE_DICT_ENTRIES);
    for (int e = 0; e < QMOE_DICT_ENTRIES; ++e) {
        uint32_t w0 = dict_words[2 * e], w1 = dict_words[2 * e + 1];
        uint32_t pairs = w0 & 15u;
        if ((w1 & 15u) != pairs || pairs < 1 || pairs > 14)
            return fail(QMOE_EFORMAT, "qmoe_dict_compact: bad pair count");
        int slots[4] = {63, 63, 63, 63};
        int nnz = 0;
        for (int i = 0; i < 28; ++i) {
            uint32_t s = ((i < 14 ? w0 : w1) >> (4 + 2 * (i % 14))) & 3u;
            if (s == 3) return fail(QMOE_EFORMAT, "qmoe_dict_compact: symbol 3");
            if (i >= (int)(2 * pairs)) {
                if (s) return fail(QMOE_EFORMAT, "qmoe_dict_compact: nonzero symbol in an unused field");
                continue;
            }
            if (s) {
                if (nnz < 4) slots[nnz] = 2 * i + (s == 1 ? 1 : 0);
                ++nnz;
            }
        }
        if (nnz <= 3) {
            pa[e] = (uint16_t)(pairs | ((uint32_t)slots[0] << 4) | ((uint32_t)slots[1] << 10));
            pb[e] = (uint8_t)slots[2];
        } else if (nnz == 4 && slots[3] < 16) {
            pa[e] = (uint16_t)(pairs | ((uint32_t)slots[0] << 4) | ((uint32_t)slots[1] << 8) |
                               ((uint32_t)slots[2] << 12));
            pb[e] = (uint8_t)(slots[3] | 0x40);
        } else {
            pa[e] = (uint16_t)(pairs | 0xFFF0u);
            pb[e] = 0xBF;
        }
        pw[e] = (uint32_t)pa[e] | ((uint32_t)pb[e] << 16);
    }
    return QMOE_OK;
}

// ---------------------------------------------------------------------------
// RVQ encoder
// ---------------------------------------------------------------------------
namespace {

double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, man = h & 1023;
    double v;
    if (ex == 0) v = std::ldexp((double)man, -24);
    else if (ex == 31) v = man ? NAN : INFINITY;
    else v = std::ldexp((double)(man | 1024), ex - 25);
    return sign ? -v : v;
}

// float64 -> IEEE binary16, round to nearest even (finite, non-NaN inputs).
uint16_t double_to_half(double v) {
    uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    double a = std::fabs(v);
    if (a == 0.0) return sign;
    if (a >= 65520.0) return sign | 0x7C00;   // rounds to infinity
    int e;
    std::frexp(a, &e);                          // a = m * 2^e, m in [0.5, 1)
    int ex = std::max(e, -13);                  // subnormal quantum 2^-24
    double q = std::nearbyint(std::ldexp(a, 11 - ex));   // 11 significant bits
    double r = std::ldexp(q, ex - 11);
    // re-encode r (exactly representable in binary16)
    int e2;
    std::frexp(r, &e2);
    if (e2 <= -14) return sign | (uint16_t)std::ldexp(r, 24);              // subnormal
    uint16_t man = (uint16_t)(std::ldexp(r, 11 - e2) - 1024.0);
    return sign | (uint16_t)((e2 + 14) << 10) | man;
}

void fwht_strided(double* a, int n, size_t stride) {
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double x = a[(size_t)j * stride], y = a[(size_t)(j + h) * stride];
                a[(size_t)j * stride] = x + y;
                a[(size_t)(j + h) * stride] = x - y;
            }
    double s = std::sqrt((double)n);
    for (int i = 0; i < n; ++i) a[(size_t)i * stride] = a[(size_t)i * stride] / s;
}

int nearest8(const double* u, const double* cb) {
    int best = 0;
    double bestd = INFINITY;
    for (int j = 0; j < QMOE_RVQ_CODES; ++j) {
        const double* c = cb + j * 8;
        double d = 0.0;
        int k = 0;
        for (; k < 8; ++k) {
            double diff = u[k] - c[k];
            d = d + diff * diff;
            if (d > bestd) break;     // partial sums of squares only grow: cannot win
        }
        if (k == 8 && d < bestd) {
            bestd = d;
            best = j;
        }
    }
    return best;
}

bool pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

// W' = H_rows D_out W D_in H_cols (columns first, then rows); false on a sign outside +-1.
bool rotate(const double* w, int rows, int cols, const int8_t* sign_out, const int8_t* sign_in,
            std::vector<double>& a) {
    a.assign((size_t)rows * cols, 0.0);
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c) {
            if (std::abs(sign_out[r]) != 1 || std::abs(sign_in[c]) != 1) return false;
            a[(size_t)r * cols + c] = w[(size_t)r * cols + c] * (double)sign_out[r] * (double)sign_in[c];
        }
    for (int c = 0; c < cols; ++c) fwht_strided(a.data() + c, rows, (size_t)cols);
    for (int r = 0; r < rows; ++r) fwht_strided(a.data() + (size_t)r * cols, cols, 1);
    return true;
}

// sqrt(sum_c row[c]^2 / cols), the sum taken left to right.
double row_rms(const double* row, int cols) {
    double sum = 0.0;
    for (int c = 0; c < cols; ++c) sum = sum + row[c] * row[c];
    return std::sqrt(sum / (double)cols);
}

}  // namespace

extern "C" int rvq_pack_stages(const double* w, int rows, int cols, const int8_t* sign_out,
                               const int8_t* sign_in, const uint16_t* codebooks, int n_stages, uint8_t* idx,
                               uint16_t* scale_f16) {
    qmoe::clear_error();
    if (!w || !sign_out || !sign_in || !codebooks || !idx || !scale_f16)
        return fail(QMOE_EINVAL, "rvq_pack: NULL argument");
    if (!pow2(rows) || !pow2(cols) || cols % 8 || rows > 8192 || cols > 8192)
        return fail(QMOE_EINVAL, "rvq_pack: rows and cols must be powers of two in [8, 8192]");
    if (n_stages < 1 || n_stages > QMOE_RVQ_MAX_STAGES)
        return fail(QMOE_EINVAL, "rvq_pack: stage count outside 1 .. QMOE_RVQ_MAX_STAGES");
    std::vector<double> a;
    if (!rotate(w, rows, cols, sign_out, sign_in, a)) return fail(QMOE_EINVAL, "rvq_pack: signs must be +1 or -1");
    std::vector<double> cb((size_t)n_stages * QMOE_RVQ_CODES * 8);
    for (size_t i = 0; i < cb.size(); ++i) cb[i] = half_to_double(codebooks[i]);
    for (int r = 0; r < rows; ++r) {
        const double* row = a.data() + (size_t)r * cols;
        uint16_t sh = double_to_half(row_rms(row, cols));
        double s = half_to_double(sh);
        if (s == 0.0) return fail(QMOE_EINVAL, "rvq_pack: a row's scale rounds to zero");
        scale_f16[r] = sh;
        for (int v = 0; v < cols / 8; ++v) {
            double res[8];
            for (int k = 0; k < 8; ++k) res[k] = row[v * 8 + k] / s;
            for (int st = 0; st < n_stages; ++st) {
                const double* c = cb.data() + (size_t)st * QMOE_RVQ_CODES * 8;
                const int i = nearest8(res, c);
                for (int k = 0; k < 8; ++k) res[k] = res[k] - c[i * 8 + k];
                idx[((size_t)r * (cols / 8) + v) * n_stages + st] = (uint8_t)i;
            }
        }
    }
    return QMOE_OK;
}

extern "C" int rvq_pack(const double* w, int rows, int cols, const int8_t* sign_out,
                        const int8_t* sign_in, const uint16_t* codebooks, uint8_t* idx,
                        uint16_t* scale_f16) {
    return rvq_pack_stages(w, rows, cols, sign_out, sign_in, codebooks, 2, idx, scale_f16);
}

extern "C" int rvq_stage_allocation(const double* popularity, int E, int s_bar, uint8_t* stages) {
    qmoe::clear_error();
    if (!popularity || !stages || E < 1) return fail(QMOE_EINVAL, "rvq_stage_allocation: NULL argument or E < 1");
    const int third = E / 3;
    if (s_bar < 1 || s_bar > QMOE_RVQ_MAX_STAGES || (third > 0 && (s_bar < 2 || s_bar + 1 > QMOE_RVQ_MAX_STAGES)))
        return fail(QMOE_EINVAL, "rvq_stage_allocation: s_bar - 1 and s_bar + 1 must be valid stage counts");
    std::vector<int> order(E);
    for (int e = 0; e < E; ++e) order[e] = e;
    // most popular first; equal popularity: lower expert id first
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return popularity[x] > popularity[y]; });
    for (int q = 0; q < E; ++q) {
        const int e = order[q];
        stages[e] = (uint8_t)(q < third ? s_bar + 1 : q >= E - third ? s_bar - 1 : s_bar);
    }
    return QMOE_OK;
}

// ---------------------------------------------------------------- E8P lattice code
// "M8.5 - Extreme Weight Compression and Representations", 0x06E: a 16-bit
// code word names a point of E8 + 1/4 = (D8^ + 1/4) u (D8^ - 1/4), where D8^
// (= D8 + 1/2) holds the half-integer vectors with an even coordinate sum:
// bits 0-7 pick one of 256 absolute patterns, bits 8-14 the signs of
// coordinates 0-6, bit 15 the shift; coordinate 7's sign makes the sum even.
namespace {

constexpr double kE8pAbs[3] = {0.5, 1.5, 2.5};

struct E8pTable {
    uint32_t words[QMOE_E8P_PATTERNS];          // nibble j = 2|a_j|
    uint8_t q[QMOE_E8P_PATTERNS][8];            // |a_j| = kE8pAbs[q]
    uint8_t parity[QMOE_E8P_PATTERNS];          // (sum_j |a_j|) mod 2
    int16_t index_of[6561];                     // sum_j q_j 3^j -> pattern, or -1
};

const E8pTable& e8p_table() {
    static const E8pTable t = [] {
        E8pTable t{};
        // every 8-tuple over {1, 3, 5} (= 2|a|) by squared norm, then lexicographically
        std::vector<std::array<uint8_t, 8>> all;
        for (int n = 0; n < 6561; ++n) {
            std::array<uint8_t, 8> d{};
            for (int j = 0, m = n; j < 8; ++j, m /= 3) d[7 - j] = (uint8_t)(1 + 2 * (m % 3));
            all.push_back(d);
        }
        auto norm = [](const std::array<uint8_t, 8>& d) {
            int s = 0;
            for (int v : d) s += v * v;
            return s;
        };
        std::sort(all.begin(), all.end(), [&](const std::array<uint8_t, 8>& x, const std::array<uint8_t, 8>& y) {
            const int nx = norm(x), ny = norm(y);
            return nx != ny ? nx < ny : x < y;
        });
        std::fill(std::begin(t.index_of), std::end(t.index_of), (int16_t)-1);
        for (int p = 0; p < QMOE_E8P_PATTERNS; ++p) {
            uint32_t w = 0;
            int sum2 = 0, key = 0, pw = 1;
            for (int j = 0; j < 8; ++j) {
                const int v = all[p][j];
                w |= (uint32_t)v << (4 * j);
                t.q[p][j] = (uint8_t)(v >> 1);
                sum2 += v;
                key += (v >> 1) * pw;
                pw *= 3;
            }
            t.words[p] = w;
            t.parity[p] = (uint8_t)((sum2 / 2) & 1);   // sum2 = 2 sum|a|, a sum of 8 odd numbers
            t.index_of[key] = (int16_t)p;
        }
        return t;
    }();
    return t;
}

struct E8pBest {
    double d = INFINITY;
    uint32_t code = 0x10000u;
};

// Codeword of code word `code` (pattern p, coordinate signs neg[], shift c) and its squared
// distance to u, summed over j = 0..7 in order; kept when (d, code) is the smallest so far.
void e8p_consider(const double* u, int p, const bool* neg, int b, E8pBest& best) {
    const E8pTable& t = e8p_table();
    const double c = b ? 0.25 : -0.25;
    double d = 0.0;
    uint32_t code = (uint32_t)p | ((uint32_t)b << 15);
    for (int j = 0; j < 8; ++j) {
        const double a = kE8pAbs[t.q[p][j]];
        const double v = (neg[j] ? -a : a) + c;
        const double diff = u[j] - v;
        d = d + diff * diff;
        if (j < 7 && neg[j]) code |= 1u << (8 + j);
    }
    if (d < best.d || (d == best.d && code < best.code)) {
        best.d = d;
        best.code = code;
    }
}

// Nearest point of D8^ + c (Conway and Sloane's decoder for D8, on the half-integer grid);
// false when the rounding or the parity repair is ambiguous or the pattern is not in the table.
bool e8p_lattice(const double* u, int b, int& p_out, bool (&neg)[8]) {
    const E8pTable& t = e8p_table();
    const double c = b ? 0.25 : -0.25;
    double h[8], err[8], sum = 0.0;
    for (int j = 0; j < 8; ++j) {
        const double w = u[j] - c;
        const double fl = std::floor(w);
        if (w == fl) return false;                      // equidistant from two half-integers
        h[j] = fl + 0.5;
        err[j] = w - h[j];
        sum += h[j];
    }
    if (std::fmod(std::fabs(sum), 2.0) != 0.0) {        // odd sum: move the worst coordinate
        int k = 0;
        for (int j = 1; j < 8; ++j)
            if (std::fabs(err[j]) > std::fabs(err[k])) k = j;
        for (int j = 0; j < 8; ++j)
            if (j != k && std::fabs(err[j]) == std::fabs(err[k])) return false;
        h[k] += err[k] > 0 ? 1.0 : -1.0;
    }
    int key = 0, pw = 1;
    for (int j = 0; j < 8; ++j) {
        const double a = std::fabs(h[j]);
        const int q = a == 0.5 ? 0 : a == 1.5 ? 1 : a == 2.5 ? 2 : -1;
        if (q < 0) return false;
        key += q * pw;
        pw *= 3;
        neg[j] = h[j] < 0;
    }
    p_out = t.index_of[key];
    return p_out >= 0;
}

// Nearest codeword of shift b over all 256 patterns: per pattern the optimal signs (each
// coordinate takes the sign of u_j - c; a wrong parity flips the coordinate where that
// costs least, 4 |u_j - c| |a_j|), then the exact distances of the near-best candidates.
void e8p_search(const double* u, int b, E8pBest& best) {
    const E8pTable& t = e8p_table();
    const double c = b ? 0.25 : -0.25;
    double m[8], e[8][3], f[8][3];
    bool neg0[8];
    int n_neg = 0;
    for (int j = 0; j < 8; ++j) {
        const double w = u[j] - c;
        neg0[j] = w < 0;
        n_neg += neg0[j];
        m[j] = std::fabs(w);
        for (int q = 0; q < 3; ++q) {
            const double dq = m[j] - kE8pAbs[q];
            e[j][q] = dq * dq;
            f[j][q] = m[j] * kE8pAbs[q];
        }
    }
    double D[QMOE_E8P_PATTERNS], dmin = INFINITY;
    for (int p = 0; p < QMOE_E8P_PATTERNS; ++p) {
        double s = 0.0;
        for (int j = 0; j < 8; ++j) s += e[j][t.q[p][j]];
        if ((n_neg + t.parity[p]) & 1) {
            double fm = f[0][t.q[p][0]];
            for (int j = 1; j < 8; ++j) fm = std::min(fm, f[j][t.q[p][j]]);
            s += 4.0 * fm;
        }
        D[p] = s;
        dmin = std::min(dmin, s);
    }
    const double cut = dmin + 1e-9 * (1.0 + dmin);
    for (int p = 0; p < QMOE_E8P_PATTERNS; ++p) {
        if (D[p] > cut) continue;
        if (!((n_neg + t.parity[p]) & 1)) {
            e8p_consider(u, p, neg0, b, best);
            continue;
        }
        double fm = f[0][t.q[p][0]];
        for (int j = 1; j < 8; ++j) fm = std::min(fm, f[j][t.q[p][j]]);
        for (int k = 0; k < 8; ++k) {
            if (f[k][t.q[p][k]] != fm) continue;
            bool neg[8];
            for (int j = 0; j < 8; ++j) neg[j] = neg0[j] != (j == k);
            e8p_consider(u, p, neg, b, best);
        }
    }
}

uint16_t e8p_encode8(const double* u) {
    E8pBest best;
    for (int b = 0; b < 2; ++b) {
        int p;
        bool neg[8];
        if (e8p_lattice(u, b, p, neg)) e8p_consider(u, p, neg, b, best);
        else e8p_search(u, b, best);
    }
    return (uint16_t)best.code;
}

}  // namespace

extern "C" int e8p_base_table(uint32_t* table) {
    qmoe::clear_error();
    if (!table) return fail(QMOE_EINVAL, "e8p_base_table: NULL argument");
    std::memcpy(table, e8p_table().words, sizeof(e8p_table().words));
    return QMOE_OK;
}

extern "C" int e8p_pack(const double* w, int rows, int cols, const int8_t* sign_out, const int8_t* sign_in,
                        uint16_t* codes, uint16_t* scale_f16) {
    qmoe::clear_error();
    if (!w || !sign_out || !sign_in || !codes || !scale_f16) return fail(QMOE_EINVAL, "e8p_pack: NULL argument");
    if (!pow2(rows) || !pow2(cols) || cols % 8 || rows > 8192 || cols > 8192)
        return fail(QMOE_EINVAL, "e8p_pack: rows and cols must be powers of two in [8, 8192]");
    std::vector<double> a;
    if (!rotate(w, rows, cols, sign_out, sign_in, a)) return fail(QMOE_EINVAL, "e8p_pack: signs must be +1 or -1");
    const double kappa = std::sqrt(2450.0 / 2048.0);
    for (int r = 0; r < rows; ++r) {
        const double* row = a.data() + (size_t)r * cols;
        const uint16_t sh = double_to_half(row_rms(row, cols) / kappa);
        const double s = half_to_double(sh);
        if (s == 0.0) return fail(QMOE_EINVAL, "e8p_pack: a row's scale rounds to zero");
        scale_f16[r] = sh;
        for (int v = 0; v < cols / 8; ++v) {
            double u[8];
            for (int k = 0; k < 8; ++k) u[k] = row[v * 8 + k] / s;
            codes[(size_t)r * (cols / 8) + v] = e8p_encode8(u);
        }
    }
    return QMOE_OK;
}

extern "C" int e8p_nearest(const double* u, size_t n, uint16_t* codes) {
    qmoe::clear_error();
    if ((!u || !codes) && n) return fail(QMOE_EINVAL, "e8p_nearest: NULL argument");
    for (size_t i = 0; i < n; ++i) {
        for (int j = 0; j < 8; ++j)
            if (!std::isfinite(u[i * 8 + j])) return fail(QMOE_EINVAL, "e8p_nearest: non-finite input");
        codes[i] = e8p_encode8(u + i * 8);
    }
    return QMOE_OK;
}
