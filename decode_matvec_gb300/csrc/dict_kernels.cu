// Dictionary-coded ternary path: fused decode-and-multiply kernels for sm_103a.
//
// The format is QMoE's (QMoE paper-summary page, "The Fixed-to-Variable
// Dictionary Code"): 16-bit codewords index a shared 2^16-entry dictionary of
// runs of 2..28 ternary weights; rows are independent, cut into blocks with
// start offsets.  QMoE's own kernel (its Listing 1, written for sm_86) gives a
// whole warp to one codeword at a time and multiplies all 28 lanes.  This
// design instead gives each lane its own codeword: the lane looks the codeword
// up in a compact derived table that lists only the run length and the (at
// most three) nonzero positions and signs, a warp-wide prefix sum of the run
// lengths places every run in its row, and each lane adds +-x only at its
// nonzero positions (about 2.4 per codeword instead of 28 multiplies).  The
// compact table (192 KB) is staged in shared memory for large launches and read
// through the L1/L2 path for small ones.  Several tokens that share an expert
// are handled in the same pass (the "inner loop over tokens" the QMoE page
// proposes for batched experts): activations are staged in shared memory as
// [column][token] so that one nonzero reads all of its tokens in one access.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "tc_common.cuh"

namespace {

__device__ int g_dict_error;

__device__ __forceinline__ void set_error(int code) { atomicCAS(&g_dict_error, 0, code); }

constexpr int kDictA = 2 * QMOE_DICT_ENTRIES;          // bytes of the uint16 plane
constexpr int kDictBytes = 3 * QMOE_DICT_ENTRIES;       // the uint16 and uint8 planes (staged in SMEM)
constexpr int kDictWordsOff = 3 * QMOE_DICT_ENTRIES;    // byte offset of the uint32 plane
constexpr int kSlotEmpty = 63;
constexpr int kSmemMax = 232448;                        // 227 KB opt-in per block
constexpr int kBudgetSmemDict = kSmemMax - kDictBytes - 256;   // activations + row sums, dictionary in SMEM
constexpr int kBudgetGlobalDict = 56 * 1024;                    // activations + row sums, dictionary via L1/L2
constexpr int kSaccBytes = 8192;                                // per-tile row sums (rows x tokens x 4 B), at least
#ifndef QMOE_SACC_MAX
#define QMOE_SACC_MAX 16384                                     // ... and at most, where the SMEM budget allows
#endif
// launches with at most this many token slots take row-sum buffers up to twice as large (longer
// tiles: fewer tile starts per expert; measured on the c2048-shaped layer: T = 64 0.341 -> 0.300 ms,
// while T = 4096 is 1 % faster with the smaller cap)
#ifndef QMOE_SACC_SMALL_SLOTS
#define QMOE_SACC_SMALL_SLOTS 1024
#endif
constexpr int kTcMinTokens = 32;                                // experts this busy use the tensor-core kernel
#ifndef QMOE_TC_MIN_SLOTS
#define QMOE_TC_MIN_SLOTS 256
#endif
constexpr int kTcMinSlots = QMOE_TC_MIN_SLOTS;                 // ... in launches with at least this many slots
// Threads of a block with the dictionary in SMEM, by the launch's largest
// token class: fewer accumulators per thread leave registers for more warps,
// which hide more of the shared-memory gather latency (measured on the
// c2048-shaped layer: 512 threads for every class 6.69 ms per T=4096 step,
// 640 / 768 threads for the 4- / 2-token classes 6.33 ms).
#ifndef QMOE_THREADS_NT1
#define QMOE_THREADS_NT1 512
#endif
#ifndef QMOE_THREADS_NT2
#define QMOE_THREADS_NT2 768
#endif
#ifndef QMOE_THREADS_NT4
#define QMOE_THREADS_NT4 640
#endif
__host__ __device__ constexpr int threads_smem_dict(int nt_max) {
    return nt_max == 1 ? QMOE_THREADS_NT1 : nt_max == 2 ? QMOE_THREADS_NT2 : nt_max == 4 ? QMOE_THREADS_NT4 : 512;
}
template <bool DICT_SMEM, int NTMAX>
struct GemmBounds {
    static constexpr int threads = DICT_SMEM ? threads_smem_dict(NTMAX) : 256;
    static constexpr int blocks = DICT_SMEM ? 1 : 2;
};
constexpr int kThreadsGlobalDict = 256;

struct MatDev {
    const uint16_t* codes;
    const uint64_t* code_base;
    const uint32_t* row_off;     // [count][rows + 1]
    const uint8_t* blk_len;      // [count][rows][nb - 1]
    const uint16_t* scale;
    int count, rows, cols, block, nb;
};

using qmoe::Job;
using qmoe::kPlanMaxE;

enum OutMode : int {
    OUT_PLAIN = 0,     // y[token][row] = s * acc              (fp32 or bf16)
    OUT_RELU_H = 1,    // h[slot][row] = bf16(relu(s * acc))
    OUT_GATED = 2,     // y[slot / k][row] = gate[slot] * s * acc   (k == 1 only)
    OUT_SLOT_F32 = 3,  // o[slot][row] = s * acc  (fp32)
};

struct GemmArgs {
    const uint16_t* dictA;       // compact plane A (uint16 per entry)
    const uint8_t* dictB;        // compact plane B (uint8 per entry)
    const uint32_t* words;       // canonical entries (for escape entries)
    const uint32_t* dictW;       // compact entries as one uint32 each (reads from global memory)
    MatDev m;
    const uint16_t* x;           // bf16 rows of `cols` values
    int x_div;                   // source row of slot s is s / x_div
    // jobs: either a device table (jobs != nullptr, count in *n_jobs_dev) or
    // implicit chunks of nt_max tokens over tokens [0, T) of matrix 0
    const Job* jobs;
    const int* n_jobs_dev;
    const int* slots;            // slot list (perm) for table jobs
    int T_implicit;
    int nt_max;
    int rows_per_tile;
    int row_tiles;
    int xs_bytes;                // staged-activation bytes (the row accumulators follow)
    float inv_cols;              // 1 / cols, for row = P / cols
    int mode;
    int y_is_f32;
    void* out;
    const float* gates;
};

__device__ __forceinline__ int nt_class(int n) { return n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8; }

// Dynamic shared memory of the expert kernels.  Every region is addressed by a
// 32-bit byte offset from this symbol, so that the compiler always emits
// shared-space loads and atomics for the hot loop.
extern __shared__ __align__(16) unsigned char g_smem[];

// Staged activations of one token chunk.  One token: bf16 pairs (x, -x) per
// column, so that a compact-table slot value 2*position + negative is directly
// the element offset from 2*column (no sign arithmetic); several tokens: bf16
// [column][token].  kPadCols zero columns follow the row; with cols >= 224 a
// lane's codeword can never start past column cols-1+... so every slot read
// stays inside them even for a corrupt stream (see stream_rows).
constexpr int kPadCols = 32;

struct SmemMap {
    uint32_t dict_a, dict_b, xs, sacc;
};

template <int NT>
__device__ __forceinline__ void load_x(uint32_t xs, int c, uint32_t (&w)[NT / 2]) {
    if constexpr (NT == 2) {
        w[0] = *(const uint32_t*)(g_smem + xs + 4u * c);
    } else if constexpr (NT == 4) {
        const uint2 v = *(const uint2*)(g_smem + xs + 8u * c);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        const uint4 v = *(const uint4*)(g_smem + xs + 16u * c);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    }
}

// Mixed-precision accumulation (sm_100+): acc + bf16 and acc + bf16 * bf16 in
// one instruction each, the bf16 operand taken from either half of a 32-bit
// register; the bf16 -> fp32 widening is exact, so each is one fp32 rounding.
__device__ __forceinline__ float acc_add_lo(float acc, uint32_t w) {
    float d;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %1;\n add.rn.f32.bf16 %0, l, %2;\n}" : "=f"(d) : "r"(w), "f"(acc));
    return d;
}
__device__ __forceinline__ float acc_fma_lo(float acc, uint32_t w, uint32_t sgn) {
    float d;
    asm("{\n .reg .b16 l, h, s, t;\n mov.b32 {l, h}, %1;\n mov.b32 {s, t}, %3;\n fma.rn.f32.bf16 %0, l, s, %2;\n}"
        : "=f"(d) : "r"(w), "f"(acc), "r"(sgn));
    return d;
}
__device__ __forceinline__ float acc_fma_hi(float acc, uint32_t w, uint32_t sgn) {
    float d;
    asm("{\n .reg .b16 l, h, s, t;\n mov.b32 {l, h}, %1;\n mov.b32 {s, t}, %3;\n fma.rn.f32.bf16 %0, h, s, %2;\n}"
        : "=f"(d) : "r"(w), "f"(acc), "r"(sgn));
    return d;
}
// +1 or -1 as bf16 (low half) for a compact slot: bit 0 set = negative weight.
__device__ __forceinline__ uint32_t slot_sign(uint32_t s) { return 0x3F80u | ((s & 1u) << 15); }

template <bool DICT_SMEM>
__device__ __forceinline__ void lookup(const GemmArgs& a, const SmemMap& sm, uint32_t code, uint32_t& ea,
                                       uint32_t& eb) {
    if constexpr (DICT_SMEM) {
        ea = *(const uint16_t*)(g_smem + sm.dict_a + 2u * code);
        eb = *(const uint8_t*)(g_smem + sm.dict_b + code);
    } else {
        ea = __ldg(a.dictA + code);
        eb = __ldg(a.dictB + code);
    }
}

// The compact slots of one entry: three 6-bit slots, or (ESC, flag 0x40) four
// 4-bit slots of an entry with four nonzeros in its first eight positions.
// Entries read through their canonical words have every slot empty (63).
template <bool ESC>
__device__ __forceinline__ void entry_slots(uint32_t ea, uint32_t eb, uint32_t (&sl)[4]) {
    if constexpr (ESC) {
        const bool four = (eb & 0x40u) != 0u;
        sl[0] = four ? (ea >> 4) & 15u : (ea >> 4) & 63u;
        sl[1] = four ? (ea >> 8) & 15u : ea >> 10;
        sl[2] = four ? ea >> 12 : eb & 63u;
        sl[3] = four ? eb & 15u : 63u;
    } else {
        sl[0] = (ea >> 4) & 63u;
        sl[1] = ea >> 10;
        sl[2] = eb & 63u;
        sl[3] = 63u;
    }
}

// Adds one codeword's weights (at most three nonzeros, four with ESC, from the
// compact slots) times the staged activations to the per-token sums; the run
// starts at column cj.  Empty slots read nothing and add zero.
template <int NT, bool ESC>
__device__ __forceinline__ void code_acc(uint32_t ea, uint32_t eb, int cj, uint32_t xs, float (&acc)[NT]) {
    constexpr int NS = ESC ? 4 : 3;
    uint32_t sl[4];
    entry_slots<ESC>(ea, eb, sl);
    if constexpr (NT == 1) {
        const uint32_t base = xs + 4u * (uint32_t)cj;
        uint32_t r[NS];
#pragma unroll
        for (int z = 0; z < NS; ++z) r[z] = sl[z] != 63u ? (uint32_t)*(const uint16_t*)(g_smem + base + 2u * sl[z]) : 0u;
#pragma unroll
        for (int z = 0; z < NS; ++z) acc[0] = acc_add_lo(acc[0], r[z]);
    } else {
        constexpr int W = NT / 2;
        uint32_t w[NS][W];
#pragma unroll
        for (int z = 0; z < NS; ++z) {
#pragma unroll
            for (int q = 0; q < W; ++q) w[z][q] = 0u;
            if (sl[z] != 63u) load_x<NT>(xs, cj + (int)(sl[z] >> 1), w[z]);
        }
#pragma unroll
        for (int z = 0; z < NS; ++z) {
            const uint32_t g = slot_sign(sl[z]);
#pragma unroll
            for (int q = 0; q < W; ++q) {
                acc[2 * q] = acc_fma_lo(acc[2 * q], w[z][q], g);
                acc[2 * q + 1] = acc_fma_hi(acc[2 * q + 1], w[z][q], g);
            }
        }
    }
}

// Entry outside the compact slots (flag 0x80; its slots are all empty): add
// its weights from the canonical words.
template <int NT>
__device__ void escape_dot(const GemmArgs& a, uint32_t code, int len, int cj, uint32_t xs, float (&t)[NT]) {
    const uint32_t c0 = __ldg(a.words + 2 * code), c1 = __ldg(a.words + 2 * code + 1);
    for (int q = 0; q < len; ++q) {
        const uint32_t s = ((q < 14 ? c0 : c1) >> (4 + 2 * (q % 14))) & 3u;
        if (s == 0u) continue;
        if constexpr (NT == 1) {
            const uint32_t r = *(const uint16_t*)(g_smem + xs + 4u * (uint32_t)(cj + q) + (s == 1u ? 2u : 0u));
            t[0] += __uint_as_float(r << 16);
        } else {
            uint32_t w[NT / 2];
            load_x<NT>(xs, cj + q, w);
            const uint32_t g = s == 1u ? 0xBF80u : 0x3F80u;
#pragma unroll
            for (int z = 0; z < NT / 2; ++z) {
                t[2 * z] = acc_fma_lo(t[2 * z], w[z], g);
                t[2 * z + 1] = acc_fma_hi(t[2 * z + 1], w[z], g);
            }
        }
    }
}

template <int NT>
__device__ __forceinline__ void flush_row(uint32_t sacc, int row_local, const float (&acc)[NT]) {
#pragma unroll
    for (int t = 0; t < NT; ++t) atomicAdd((float*)(g_smem + sacc) + row_local * NT + t, acc[t]);
}

template <int CPL>
__device__ __forceinline__ uint4 load_codes(const uint16_t* p) {
    if constexpr (CPL == 8) return __ldg((const uint4*)p);
    else return make_uint4((uint32_t)__ldg(p), 0u, 0u, 0u);
}

// Accumulates a lane's CPL codewords: `total` over all of them, `lo` over those
// that start in the lane's first row (a prefix: codewords are in stream order).
template <int NT, int CPL, bool ESC>
__device__ __forceinline__ void acc_codes(const uint32_t (&ea)[CPL], const uint32_t (&eb)[CPL], int col, int cols,
                                          int cross, uint32_t xs, float (&total)[NT], float (&lo)[NT]) {
    int pre = 0;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const bool second = pre >= cross;
        const int cj = second ? col + pre - cols : col + pre;
        code_acc<NT, ESC>(ea[j], eb[j], cj, xs, total);
        if (!second) {
#pragma unroll
            for (int z = 0; z < NT; ++z) lo[z] = total[z];
        }
        pre += (int)(ea[j] & 15u) * 2;
    }
}

// One window: CPL consecutive codewords per lane starting at stream index
// `my`; `valid_lo`/`valid_hi` bound the lane-relative codeword indices that
// belong to the warp's rows (only edge windows need them).
template <int NT, int CPL, bool DICT_SMEM, bool EDGE>
__device__ __forceinline__ void window(const GemmArgs& a, const SmemMap& sm, uint4 cur, int valid_lo, int valid_hi,
                                       uint32_t& P, int cols, float inv_cols, int n_rows, uint32_t sacc, bool& bad,
                                       int lane) {
    const uint32_t cw[4] = {cur.x, cur.y, cur.z, cur.w};
    uint32_t ea[CPL], eb[CPL];
    int sum = 0;
    uint32_t esc = 0;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const uint32_t code = (cw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
        if (!EDGE || (j >= valid_lo && j < valid_hi)) {
            lookup<DICT_SMEM>(a, sm, code, ea[j], eb[j]);
        } else {
            ea[j] = (kSlotEmpty << 4) | (kSlotEmpty << 10);
            eb[j] = kSlotEmpty;
        }
        sum += (int)(ea[j] & 15u) * 2;
        esc |= eb[j];
    }
    const int incl = warp_incl_scan(sum, lane);
    const uint32_t start = P + (uint32_t)(incl - sum);
    int row = (int)((float)start * inv_cols);
    if ((uint32_t)row * (uint32_t)cols > start) --row;
    else if ((uint32_t)(row + 1) * (uint32_t)cols <= start) ++row;
    const int col = (int)(start - (uint32_t)row * (uint32_t)cols);
    const int cross = cols - col;                 // prefix from which codewords start in the next row
    bad |= (col + sum > 2 * cols) | (row >= n_rows && sum > 0);
    // total: all of the lane's codewords; lo: those that start in the first row
    // (a prefix, since the codewords are in stream order)
    float total[NT], lo[NT];
#pragma unroll
    for (int z = 0; z < NT; ++z) total[z] = lo[z] = 0.0f;
    // windows holding an entry with four nonzeros (flag 0x40; dictionaries for p0 below ~0.88)
    // take the four-slot accumulation, the others the three-slot one
    if (__any_sync(QMOE_FULL_MASK, esc & 0x40u))
        acc_codes<NT, CPL, true>(ea, eb, col, cols, cross, sm.xs, total, lo);
    else
        acc_codes<NT, CPL, false>(ea, eb, col, cols, cross, sm.xs, total, lo);
    if (esc & 0x80u) {
        // entries outside the compact slots (five or more nonzeros, or a fourth one past the
        // eighth position): taken from the canonical words
        int p2 = 0;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int len = (int)(ea[j] & 15u) * 2;
            if (eb[j] & 0x80u) {
                const bool second = p2 >= cross;
                const int cj = second ? col + p2 - cols : col + p2;
                float t[NT];
#pragma unroll
                for (int z = 0; z < NT; ++z) t[z] = 0.0f;
                escape_dot<NT>(a, (cw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, len, cj, sm.xs, t);
#pragma unroll
                for (int z = 0; z < NT; ++z) {
                    total[z] += t[z];
                    if (!second) lo[z] += t[z];
                }
            }
            p2 += len;
        }
    }
    // a lane whose codewords reached the next row hands its first-row sums over now
    const bool crossed = sum > cross;
    if (crossed && row < n_rows) flush_row<NT>(sacc, row, lo);
    const int orow = crossed ? row + 1 : row;
    float v[NT];
#pragma unroll
    for (int z = 0; z < NT; ++z) v[z] = crossed ? total[z] - lo[z] : total[z];
    // segmented reduction of the open rows (lanes are in row order)
    const int rr = min(orow, n_rows - 1);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int r_from = __shfl_down_sync(QMOE_FULL_MASK, rr, d);
        const bool take = lane + d < 32 && r_from == rr;
#pragma unroll
        for (int z = 0; z < NT; ++z) {
            const float o = __shfl_down_sync(QMOE_FULL_MASK, v[z], d);
            if (take) v[z] += o;
        }
    }
    const int r_prev = __shfl_up_sync(QMOE_FULL_MASK, rr, 1);
    if ((lane == 0 || r_prev != rr) && orow < n_rows) flush_row<NT>(sacc, rr, v);
    P += (uint32_t)__shfl_sync(QMOE_FULL_MASK, incl, 31);
}

// A warp streams the codewords of rows [wr0, wr1) of one matrix as one flat
// sequence, CPL consecutive codewords per lane per window (16-byte loads; the
// next window is held in registers while this one is decoded).  Every row
// expands to exactly `cols` weights, so the running expansion P of a codeword
// gives its row and column: row = P / cols, column = P % cols.  With
// cols >= 224 the 8 codewords of a lane (at most 224 weights) touch at most
// two rows; each lane keeps its window total and its first-row part.  A lane
// that crossed adds its first-row part to the shared accumulators; then a
// segmented warp reduction (lanes are in row order) lets the first lane of
// each row segment add that segment's open-row total.  Rows belong to one
// warp; lanes of the warp may add to the same row, so the adds are
// shared-memory atomics.  Narrower matrices take one codeword per lane
// (CPL = 1), which can never reach a second row.  For a corrupt stream every
// column index still stays below max(cols, 224) + 28, inside the staged
// buffer and its zero padding; the kernel records QMOE_EFORMAT.
template <int NT, int CPL, bool DICT_SMEM>
__device__ void stream_rows(const GemmArgs& a, const SmemMap& sm, const uint16_t* codes, uint64_t g_lo,
                            uint64_t g_hi, int cols, float inv_cols, int n_rows, uint32_t sacc, int lane) {
    constexpr int WIN = 32 * CPL;
    bool bad = false;
    uint32_t P = 0;
    const uint64_t w0 = g_lo & ~(uint64_t)(CPL - 1);
    const uint16_t* p = codes + w0 + CPL * lane;
    const int64_t n = (int64_t)(g_hi - w0);       // codewords from w0 to the end of the warp's rows
    const int head = (int)(g_lo - w0);            // codewords before g_lo in the first window
    uint4 nxt = make_uint4(0, 0, 0, 0);
    if (CPL * lane < n) nxt = load_codes<CPL>(p);
    for (int64_t w = 0; w < n; w += WIN) {
        const uint4 cur = nxt;
        const int64_t mine = w + CPL * lane;      // stream index of this lane's first codeword, from w0
        if (mine + WIN < n) nxt = load_codes<CPL>(p + w + WIN);
        // keep about four windows of this warp's stream in flight towards L2
        // (one prefetch per 128-byte line)
        if (CPL == 8 && (lane & 7) == 0 && mine + 4 * WIN < n)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(p + w + 4 * WIN));
        if (w > 0 && w + WIN <= n) {
            window<NT, CPL, DICT_SMEM, false>(a, sm, cur, 0, CPL, P, cols, inv_cols, n_rows, sacc, bad, lane);
        } else {
            const int64_t lo64 = (int64_t)head - mine, hi64 = n - mine;
            const int lo = lo64 > 0 ? (int)lo64 : 0;
            const int hi = hi64 < CPL ? (int)hi64 : CPL;
            window<NT, CPL, DICT_SMEM, true>(a, sm, cur, lo, hi, P, cols, inv_cols, n_rows, sacc, bad, lane);
        }
    }
    if (lane == 0 && P != (uint32_t)n_rows * (uint32_t)cols) bad = true;
    if (__any_sync(QMOE_FULL_MASK, bad) && lane == 0) set_error(QMOE_EFORMAT);
}

__device__ __forceinline__ void job_of(const GemmArgs& a, int j, Job& job) {
    if (a.jobs) {
        job = a.jobs[j];
    } else {
        job.matrix = 0;
        job.slot_begin = j * a.nt_max;
        job.n_tok = min(a.nt_max, a.T_implicit - j * a.nt_max);
    }
}

__device__ __forceinline__ int slot_at(const GemmArgs& a, const Job& job, int i) {
    return a.slots ? a.slots[job.slot_begin + i] : job.slot_begin + i;
}

// Loads of G columns per thread are issued together, then stored: the
// staging costs a couple of memory round trips rather than one per column.
template <int NT>
__device__ void stage_x(const GemmArgs& a, const Job& job, uint32_t xs, int tid, int nthreads) {
    constexpr int G = 8;
    const int cols = a.m.cols, total = cols + kPadCols;
    const uint16_t* src[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t)
        src[t] = t < job.n_tok ? a.x + (size_t)(slot_at(a, job, t) / a.x_div) * cols : nullptr;
    for (int c0 = tid; c0 < total; c0 += nthreads * G) {
        uint32_t v[G][NT];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int c = c0 + g * nthreads;
#pragma unroll
            for (int t = 0; t < NT; ++t) v[g][t] = (src[t] && c < cols) ? (uint32_t)__ldg(src[t] + c) : 0u;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int c = c0 + g * nthreads;
            if (c >= total) break;
            if constexpr (NT == 1) {
                // (x, -x) as one 32-bit word per column
                *(uint32_t*)(g_smem + xs + 4u * c) = v[g][0] | ((v[g][0] ^ 0x8000u) << 16);
            } else if constexpr (NT == 2) {
                *(uint32_t*)(g_smem + xs + 4u * c) = v[g][0] | (v[g][1] << 16);
            } else if constexpr (NT == 4) {
                *(uint2*)(g_smem + xs + 8u * c) = make_uint2(v[g][0] | (v[g][1] << 16), v[g][2] | (v[g][3] << 16));
            } else {
                *(uint4*)(g_smem + xs + 16u * c) = make_uint4(v[g][0] | (v[g][1] << 16), v[g][2] | (v[g][3] << 16),
                                                              v[g][4] | (v[g][5] << 16), v[g][6] | (v[g][7] << 16));
            }
        }
    }
}

// Scale, activation and store of the tile's rows (threads over rows, per token).
template <int NT>
__device__ void tile_epilogue(const GemmArgs& a, const Job& job, int r0, int nr, uint32_t sacc, int tid,
                              int nthreads) {
    const int rows = a.m.rows;
    const uint16_t* scale = a.m.scale + (size_t)job.matrix * rows;
    const float* acc = (const float*)(g_smem + sacc);
    for (int i = tid; i < nr * job.n_tok; i += nthreads) {
        const int t = i / nr, rl = i - t * nr, row = r0 + rl;
        const int slot = slot_at(a, job, t);
        const float v = f16_to_f32(scale[row]) * acc[rl * NT + t];
        const size_t o = (size_t)slot * rows + row;
        switch (a.mode) {
            case OUT_PLAIN:
                if (a.y_is_f32) ((float*)a.out)[o] = v;
                else ((uint16_t*)a.out)[o] = f32_to_bf16(v);
                break;
            case OUT_RELU_H:
                ((uint16_t*)a.out)[o] = f32_to_bf16(fmaxf(v, 0.0f));
                break;
            case OUT_GATED: {
                const float g = a.gates[slot] * v;
                if (a.y_is_f32) ((float*)a.out)[o] = g;
                else ((uint16_t*)a.out)[o] = f32_to_bf16(g);
                break;
            }
            default:
                ((float*)a.out)[o] = v;
                break;
        }
    }
}

__device__ __forceinline__ void tile_rows_of(const GemmArgs& a, int tile, Job& job, int& r0, int& r1) {
    job_of(a, tile / a.row_tiles, job);
    r0 = (tile % a.row_tiles) * a.rows_per_tile;
    r1 = min(a.m.rows, r0 + a.rows_per_tile);
}

// Warms L2 with the code range of a tile this block will process later.
__device__ void prefetch_tile(const GemmArgs& a, int tile, int n_tiles) {
    if (tile >= n_tiles) return;
    Job job;
    int r0, r1;
    tile_rows_of(a, tile, job, r0, r1);
    const MatDev& m = a.m;
    const uint32_t* ro = m.row_off + (size_t)job.matrix * (m.rows + 1);
    const uint64_t base = m.code_base ? m.code_base[job.matrix] : 0ull;
    const uint64_t lo = (base + ro[r0]) & ~7ull;
    const uint64_t hi = (base + ro[r1] + 7) & ~7ull;
    if (hi <= lo) return;
    const char* p = (const char*)(m.codes + lo);
    uint64_t bytes = (hi - lo) * 2;
    while (bytes) {
        const uint32_t n = (uint32_t)(bytes < (1ull << 20) ? bytes : (1ull << 20));
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
        p += n;
        bytes -= n;
    }
}

template <int NT, bool DICT_SMEM>
__device__ void run_tile(const GemmArgs& a, const SmemMap& sm, const Job& job, int r0, int r1, int tid, int nthreads,
                         int warp, int nwarps, int lane, int prefetch, int n_tiles, bool restage) {
    const MatDev& m = a.m;
    if (restage) stage_x<NT>(a, job, sm.xs, tid, nthreads);
    const int nr = r1 - r0;
    for (int i = tid; i < nr * NT; i += nthreads) ((float*)(g_smem + sm.sacc))[i] = 0.0f;
    __syncthreads();
    const uint32_t* ro = m.row_off + (size_t)job.matrix * (m.rows + 1);
    const uint64_t base = m.code_base ? m.code_base[job.matrix] : 0ull;
    const int per = (nr + nwarps - 1) / nwarps;
    const int wr0 = r0 + warp * per, wr1 = min(r1, wr0 + per);
    if (wr0 < wr1) {
        const uint32_t lo = ro[wr0], hi = ro[wr1];
        if (hi < lo) {
            if (lane == 0) set_error(QMOE_EFORMAT);
        } else {
            const uint32_t sacc = sm.sacc + 4u * (uint32_t)((wr0 - r0) * NT);
            if (m.cols >= 8 * QMOE_MAX_RUN)
                stream_rows<NT, 8, DICT_SMEM>(a, sm, m.codes, base + lo, base + hi, m.cols, a.inv_cols, wr1 - wr0,
                                              sacc, lane);
            else
                stream_rows<NT, 1, DICT_SMEM>(a, sm, m.codes, base + lo, base + hi, m.cols, a.inv_cols, wr1 - wr0,
                                              sacc, lane);
        }
    }
    // the last warp, usually done first (it has the fewest rows), warms L2 for a later tile
    if (warp == nwarps - 1 && lane == 0) prefetch_tile(a, prefetch, n_tiles);
    __syncthreads();
    tile_epilogue<NT>(a, job, r0, nr, sm.sacc, tid, nthreads);
    __syncthreads();
}

// NTMAX: the largest token class of the launch (its chunk size); a kernel
// compiled for fewer classes needs fewer registers.
template <bool DICT_SMEM, int NTMAX>
__global__ void __launch_bounds__(GemmBounds<DICT_SMEM, NTMAX>::threads, GemmBounds<DICT_SMEM, NTMAX>::blocks)
    dict_gemm_kernel(const GemmArgs a) {
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
    SmemMap sm;
    sm.dict_a = 0;
    sm.dict_b = kDictA;
    sm.xs = DICT_SMEM ? (uint32_t)kDictBytes : 0u;
    sm.sacc = sm.xs + (uint32_t)a.xs_bytes;
    const int n_jobs = a.jobs ? *a.n_jobs_dev : (a.T_implicit + a.nt_max - 1) / a.nt_max;
    const int n_tiles = n_jobs * a.row_tiles;
    // each block takes a contiguous range of tiles: consecutive tiles of one job
    // reuse the staged activations
    const int per_block = (n_tiles + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per_block, t_end = min(n_tiles, t_begin + per_block);
    if (tid == 0) {
        prefetch_tile(a, t_begin, t_end);
        prefetch_tile(a, t_begin + 1, t_end);
    }
    if constexpr (DICT_SMEM) {
        const uint4* srcA = (const uint4*)a.dictA;
        const uint4* srcB = (const uint4*)a.dictB;
        uint4* dst = (uint4*)g_smem;
        for (int i = tid; i < kDictA / 16; i += nthreads) dst[i] = __ldg(srcA + i);
        for (int i = tid; i < QMOE_DICT_ENTRIES / 16; i += nthreads) dst[kDictA / 16 + i] = __ldg(srcB + i);
    }
    __syncthreads();
    int staged = -1;
    for (int tile = t_begin; tile < t_end; ++tile) {
        Job job;
        int r0, r1;
        tile_rows_of(a, tile, job, r0, r1);
        const int j = tile / a.row_tiles;
        const bool restage = j != staged;
        staged = j;
        const int c = nt_class(job.n_tok);
        if (c == 1 || NTMAX == 1) {
            run_tile<1, DICT_SMEM>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, tile + 2, t_end, restage);
        } else if (c == 2 || NTMAX == 2) {
            if constexpr (NTMAX >= 2)
                run_tile<2, DICT_SMEM>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, tile + 2, t_end, restage);
        } else if (c == 4 || NTMAX == 4) {
            if constexpr (NTMAX >= 4)
                run_tile<4, DICT_SMEM>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, tile + 2, t_end, restage);
        } else {
            if constexpr (NTMAX >= 8)
                run_tile<8, DICT_SMEM>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, tile + 2, t_end, restage);
        }
    }
}

// ------------------------------------------------------------ row-per-lane variant (compact table in SMEM)
// Each lane owns one row of the tile and walks its codewords in stream order,
// 8 per step from aligned 16-byte chunks (the next chunk loaded while this one
// is decoded), so the running column of a codeword is a per-lane sum: no warp
// scan, no row/column division, no segmented reduction and no shared-memory
// row sums.  The per-token sums stay in registers until the row's last
// codeword; the lane then applies the row scale and the activation or gate
// and stores.  A warp takes 32 consecutive rows at a time; lanes whose row
// ends first idle (with empty entries) until the warp's last row ends.  For a
// corrupt stream the column of a run is clamped to the row end, so every
// activation read stays inside the staged row and its zero padding; the
// kernel records QMOE_EFORMAT.
template <int NT>
__device__ __forceinline__ void row_store(const GemmArgs& a, const Job& job, int row, const float (&acc)[NT]) {
    const int rows = a.m.rows;
    const float s = f16_to_f32(a.m.scale[(size_t)job.matrix * rows + row]);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        if (t >= job.n_tok) break;
        const int slot = slot_at(a, job, t);
        const float v = s * acc[t];
        const size_t o = (size_t)slot * rows + row;
        switch (a.mode) {
            case OUT_PLAIN:
                if (a.y_is_f32) ((float*)a.out)[o] = v;
                else ((uint16_t*)a.out)[o] = f32_to_bf16(v);
                break;
            case OUT_RELU_H:
                ((uint16_t*)a.out)[o] = f32_to_bf16(fmaxf(v, 0.0f));
                break;
            case OUT_GATED: {
                const float g = a.gates[slot] * v;
                if (a.y_is_f32) ((float*)a.out)[o] = g;
                else ((uint16_t*)a.out)[o] = f32_to_bf16(g);
                break;
            }
            default:
                ((float*)a.out)[o] = v;
                break;
        }
    }
}

template <int NT>
__device__ __forceinline__ void row_walk(const GemmArgs& a, const SmemMap& sm, const Job& job, int row, bool live,
                                         bool& bad) {
    const MatDev& m = a.m;
    const int c_hi = m.cols;
    uint64_t lo = 0, hi = 0;
    if (live) {
        const uint32_t* ro = m.row_off + (size_t)job.matrix * (m.rows + 1);
        const uint64_t base = m.code_base ? m.code_base[job.matrix] : 0ull;
        lo = base + __ldg(ro + row);
        hi = base + __ldg(ro + row + 1);
        if (hi < lo || hi - lo > (uint64_t)(c_hi / 2)) {
            bad = true;
            hi = lo;
        }
    }
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    int col = 0;
    // k: index of the current chunk's first codeword relative to lo (-7 .. 0 for the first chunk);
    // the range's codewords are k + j in [0, n)
    const uint16_t* p = m.codes + (lo & ~7ull);
    const int n = (int)(hi - lo);
    int k = -(int)(lo & 7ull);
    uint4 cur = k < n ? __ldg((const uint4*)p) : make_uint4(0, 0, 0, 0);
    while (__any_sync(QMOE_FULL_MASK, k < n)) {
        const uint4 nxt = k + 8 < n ? __ldg((const uint4*)(p + 8)) : make_uint4(0, 0, 0, 0);
        const uint32_t cw[4] = {cur.x, cur.y, cur.z, cur.w};
        uint32_t ea[8], eb[8], esc = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t code = (cw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
            if ((unsigned)(k + j) < (unsigned)n) {
                lookup<true>(a, sm, code, ea[j], eb[j]);
            } else {
                ea[j] = (kSlotEmpty << 4) | (kSlotEmpty << 10);      // length 0, slots empty
                eb[j] = kSlotEmpty;
            }
            esc |= eb[j];
        }
        // entries with four nonzeros (flag 0x40) take the four-slot accumulation
        const bool four = __any_sync(QMOE_FULL_MASK, esc & 0x40u);
        int cj = col;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = min(cj, c_hi);
            if (four) code_acc<NT, true>(ea[j], eb[j], c, sm.xs, acc);
            else code_acc<NT, false>(ea[j], eb[j], c, sm.xs, acc);
            cj += (int)(ea[j] & 15u) * 2;
        }
        if (esc & 0x80u) {
            // entries outside the compact slots: from their canonical words (rare)
            int q = col;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int len = (int)(ea[j] & 15u) * 2;
                if (eb[j] & 0x80u)
                    escape_dot<NT>(a, (cw[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, len, min(q, c_hi), sm.xs, acc);
                q += len;
            }
        }
        col = cj;
        cur = nxt;
        p += 8;
        k += 8;
    }
    if (live) {
        if (col != c_hi) bad = true;
        row_store<NT>(a, job, row, acc);
    }
}

// Rows [r0, r1) of a job: warp w takes rows r0 + 32 (w + i * nwarps) + lane.
template <int NT>
__device__ void run_rows(const GemmArgs& a, const SmemMap& sm, const Job& job, int r0, int r1, int tid, int nthreads,
                         int warp, int nwarps, int lane, bool restage, bool& bad) {
    if (restage) {
        __syncthreads();                                    // every warp is done with the previous job's rows
        stage_x<NT>(a, job, sm.xs, tid, nthreads);
        __syncthreads();
    }
    for (int g = r0 + 32 * warp; g < r1; g += 32 * nwarps) {
        const int row = g + lane;
        row_walk<NT>(a, sm, job, row, row < r1, bad);
    }
}

template <int NTMAX>
__global__ void __launch_bounds__(GemmBounds<true, NTMAX>::threads, 1) dict_rows_kernel(const GemmArgs a) {
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
    SmemMap sm;
    sm.dict_a = 0;
    sm.dict_b = kDictA;
    sm.xs = (uint32_t)kDictBytes;
    sm.sacc = 0;
    const int n_jobs = a.jobs ? *a.n_jobs_dev : (a.T_implicit + a.nt_max - 1) / a.nt_max;
    const int n_tiles = n_jobs * a.row_tiles;
    const int per_block = (n_tiles + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per_block, t_end = min(n_tiles, t_begin + per_block);
    if (tid == 0) {
        prefetch_tile(a, t_begin, t_end);
        prefetch_tile(a, t_begin + 1, t_end);
    }
    {
        const uint4* srcA = (const uint4*)a.dictA;
        const uint4* srcB = (const uint4*)a.dictB;
        uint4* dst = (uint4*)g_smem;
        for (int i = tid; i < kDictA / 16; i += nthreads) dst[i] = __ldg(srcA + i);
        for (int i = tid; i < QMOE_DICT_ENTRIES / 16; i += nthreads) dst[kDictA / 16 + i] = __ldg(srcB + i);
    }
    bool bad = false;
    int staged = -1;
    for (int tile = t_begin; tile < t_end; ++tile) {
        Job job;
        int r0, r1;
        tile_rows_of(a, tile, job, r0, r1);
        const int j = tile / a.row_tiles;
        const bool restage = j != staged;
        staged = j;
        // codes of a later tile travel towards L2 meanwhile
        if (tid == 0) prefetch_tile(a, tile + 2, t_end);
        const int c = nt_class(job.n_tok);
        if (c == 1 || NTMAX == 1) {
            run_rows<1>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, restage, bad);
        } else if (c == 2 || NTMAX == 2) {
            if constexpr (NTMAX >= 2) run_rows<2>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, restage, bad);
        } else if (c == 4 || NTMAX == 4) {
            if constexpr (NTMAX >= 4) run_rows<4>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, restage, bad);
        } else {
            if constexpr (NTMAX >= 8) run_rows<8>(a, sm, job, r0, r1, tid, nthreads, warp, nwarps, lane, restage, bad);
        }
    }
    if (__any_sync(QMOE_FULL_MASK, bad) && lane == 0) set_error(QMOE_EFORMAT);
}

// ------------------------------------------------------------ tensor-core path for experts with many tokens
// An expert that receives many tokens is a real dense contraction, and the
// QMoE page's own suggestion for large token counts is to decompress first and
// then multiply.  Here the decompression goes to shared memory only, in a
// warp-specialised pipeline (one persistent CTA per SM):
//  * 8 decoder warps, in two groups of 128 threads, expand the codewords of a
//    256-column block of 128 rows into a dense bf16 tile of exact {-1, 0, +1}
//    (one thread per row: its row is zeroed, then its nonzeros written); the
//    groups take alternate blocks, so two blocks are decoded at once;
//  * a loader warp stages the activations of up to 256 tokens, 64 columns (an
//    atom) at a time, into three atom stages (bf16, 16-byte asynchronous
//    copies, zero past the tokens and columns that exist), so an expert's
//    tiles are decoded once per 256 of its tokens;
//  * one thread issues tcgen05.mma (M=128, N = tokens rounded up to 16, up to
//    256, K=16, bf16 x bf16 -> fp32 in tensor memory) and commits each atom to
//    the barrier that frees its B stage and each block to the one that frees
//    its A stage;
//  * 4 epilogue warps read a finished tile's accumulators (two accumulators in
//    tensor memory alternate between tiles), apply the row scale and the
//    activation or gate, and store.
// Tiles are 128-byte-swizzled K-major (64-column atoms of 8-row groups
// 1024 bytes apart), the layout the tensor core reads at full rate.  The row
// scale is applied in the epilogue, so the product is the same s * sum(+-x)
// as the CUDA-core kernel, summed in another order.  Every wait is bounded:
// on expiry the kernel records QMOE_ETIMEOUT, waits (bounded) for its
// outstanding MMAs, frees its tensor memory and returns.
constexpr int kDtcM = 128, kDtcN = 256, kDtcK = 256;
constexpr int kDtcStageA = kDtcM * kDtcK * 2;                 // 64 KB per A stage
constexpr int kDtcAtomA = kDtcM * 128;                        // one 64-column atom of A (16 KB)
constexpr int kDtcAtomB = kDtcN * 128;                        // ... of B (32 KB): one B stage
constexpr int kDtcDecWarps = 8, kDtcEpiWarp = 8, kDtcLoadWarp = 12, kDtcMmaWarp = 13;
constexpr int kDtcThreads = 14 * 32;
constexpr int kDtcTmemCols = 2 * kDtcN;                       // two accumulators
constexpr int kDtcStagesB = 3;                                 // activation atom stages (the loader runs ahead)
constexpr int kDtcSmem = 1024 + 2 * kDtcStageA + kDtcStagesB * kDtcAtomB + 192;
static_assert(kDtcSmem <= kSmemMax && kDtcTmemCols <= 512, "tensor-core kernel resources");
constexpr uint32_t kDtcSpin = 1u << 22;
constexpr uint16_t kBf16One = 0x3F80, kBf16MinusOne = 0xBF80;

// Byte offset of element (r, c) in a 128-byte-swizzled K-major bf16 tile whose
// 64-column atoms are atom_bytes apart: 16-byte chunk (c / 8) % 8 of row r sits at
// chunk position ((c / 8) % 8) ^ (r % 8) of its 128-byte line.
__device__ __forceinline__ uint32_t sw128_off(int r, int c, uint32_t atom_bytes) {
    return (uint32_t)(c >> 6) * atom_bytes + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
           ((uint32_t)(((c >> 3) & 7) ^ (r & 7)) << 4) + (uint32_t)(c & 7) * 2u;
}

// Descriptor of a 128-byte-swizzled K-major operand (tcgen05 version 1, 8-row groups 1024 B apart).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;                   // leading byte offset: unused for swizzled K-major
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;                                    // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(qmoe_tc::smem_u32(bar)) : "memory");
}

// Component q (0..3, a constant after unrolling) of a uint4.
__device__ __forceinline__ uint32_t u4_at(const uint4& v, int q) { return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w; }

// Bounded wait for the phase of the given parity; a thread whose phase has not
// completed is suspended (up to about a microsecond per try) instead of
// spinning, so waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t limit) {
    const uint32_t b = qmoe_tc::smem_u32(bar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(b), "r"(parity), "r"(1000u)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// 8 consecutive fp32 accumulator columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}


// Weights of an entry outside the compact slots, from its canonical words (rare: five or more
// nonzeros, or a fourth one past the eighth position).
__device__ __forceinline__ void canonical_to_row(const uint32_t* words, uint32_t code, int len, int col, unsigned char* A,
                                              int rl) {
    const uint32_t c0 = __ldg(words + 2 * code), c1 = __ldg(words + 2 * code + 1);
    for (int q = 0; q < len; ++q) {
        const uint32_t s = ((q < 14 ? c0 : c1) >> (4 + 2 * (q % 14))) & 3u;
        if (s) *(uint16_t*)(A + sw128_off(rl, col + q, kDtcAtomA)) = s == 1u ? kBf16MinusOne : kBf16One;
    }
}

// The codeword range of one (row, 256-column block) and its first two aligned
// 16-byte chunks of codewords, loaded one block ahead of its decoding.  `ok` is
// false for a range no valid block can have (every codeword covers at least two
// weights); nothing is loaded then.
struct RowBlk {
    uint64_t lo, hi;
    uint4 ch0, ch1;
    bool ok;
};

__device__ __forceinline__ RowBlk load_rowblk(const uint16_t* codes, uint2 range, uint64_t cbase, int blen) {
    RowBlk p;
    p.lo = cbase + range.x;
    p.hi = cbase + range.y;
    p.ok = !(p.hi < p.lo || p.hi - p.lo > (uint64_t)(blen / 2));
    const uint64_t c8 = p.lo & ~7ull;
    const uint4 z = make_uint4(0, 0, 0, 0);
    p.ch0 = p.ok && c8 < p.hi ? __ldg((const uint4*)(codes + c8)) : z;
    p.ch1 = p.ok && c8 + 8 < p.hi ? __ldg((const uint4*)(codes + c8 + 8)) : z;
    return p;
}

// One thread expands the codewords of one (row, block) into the tile row `rl`
// (bf16 +-1 at the nonzeros of an already zeroed row).  The codewords come 16 at
// a time as two aligned 16-byte chunks (the first two preloaded); the 16 compact
// entries are gathered with unconditional loads (out-of-range positions read
// entry 0 and are ignored) so that they are all in flight at once: a block costs
// about one memory round trip.  `bad` is set for a block that does not expand
// to exactly blen weights.
__device__ __forceinline__ void decode_row_block(const GemmArgs& a, const uint16_t* codes, const RowBlk& p, int blen,
                                                 unsigned char* A, int rl, bool& bad) {
    if (!p.ok) {
        bad = true;
        return;
    }
    const uint32_t arow = qmoe_tc::smem_u32(A) + (uint32_t)(rl >> 3) * 1024u + (uint32_t)(rl & 7) * 128u;
    const uint32_t rsw = (uint32_t)(rl & 7) << 4;
    int col = 0;
    for (uint64_t c8 = p.lo & ~7ull; c8 < p.hi; c8 += 16) {
        const bool first = c8 == (p.lo & ~7ull);
        const uint4 ch0 = first ? p.ch0 : __ldg((const uint4*)(codes + c8));
        const uint4 ch1 = first ? p.ch1 : c8 + 8 < p.hi ? __ldg((const uint4*)(codes + c8 + 8)) : make_uint4(0, 0, 0, 0);
        uint32_t code[16], e[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t w = u4_at(k < 8 ? ch0 : ch1, (k >> 1) & 3);
            code[k] = (w >> (16 * (k & 1))) & 0xFFFFu;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) e[k] = __ldg(a.dictW + code[k]);
        // run starts of the 16 positions (out-of-range positions have length 0), then every store of
        // the batch independently of the others
        int start[16];
        uint32_t esc = 0;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const bool in = c8 + k >= p.lo && c8 + k < p.hi;
            if (!in) e[k] = 0x3F0000u | 0xFFF0u;          // length 0, empty slots
            start[k] = col;
            col += (int)(e[k] & 15u) * 2;
            esc |= e[k];
        }
        if (col > blen) {
            bad = true;
            return;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t ea = e[k] & 0xFFFFu, eb = e[k] >> 16;
            // the entry's slots as four 6-bit fields (63 = empty)
            const uint32_t w = (eb & 0x40u) ? (((ea >> 4) & 15u) | (((ea >> 8) & 15u) << 6) | ((ea >> 12) << 12) |
                                               ((eb & 15u) << 18))
                                            : ((ea >> 4) | ((eb & 63u) << 12) | (63u << 18));
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const uint32_t sl = (w >> (6 * z)) & 63u;
                if (z == 3 && !(esc & 0x400000u)) break;      // no entry of the batch has a fourth slot
                if (sl != 63u) {
                    const uint32_t c = (uint32_t)start[k] + (sl >> 1);
                    const uint32_t sa = arow + (c >> 6) * (uint32_t)kDtcAtomA + (((c << 1) & 127u) ^ rsw);
                    const uint16_t v = (uint16_t)(kBf16One | ((sl & 1u) << 15));
                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(sa), "h"(v) : "memory");
                }
            }
        }
        if (esc & 0x800000u) {
            // entries outside the compact slots: from their canonical words (rare)
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if ((e[k] >> 16) & 0x80u) canonical_to_row(a.words, code[k], (int)(e[k] & 15u) * 2, start[k], A, rl);
        }
    }
    if (col != blen) bad = true;
}


// Scale, activation or gate, and store of one token column of a finished tile.
template <int MODE>
__device__ __forceinline__ void tc_store(const GemmArgs& a, int slot, int row, float v) {
    const size_t o = (size_t)slot * a.m.rows + row;
    if constexpr (MODE == OUT_RELU_H) {
        ((uint16_t*)a.out)[o] = f32_to_bf16(fmaxf(v, 0.0f));
    } else if constexpr (MODE == OUT_SLOT_F32) {
        ((float*)a.out)[o] = v;
    } else {
        const float g = MODE == OUT_GATED ? a.gates[slot] * v : v;
        if (a.y_is_f32) ((float*)a.out)[o] = g;
        else ((uint16_t*)a.out)[o] = f32_to_bf16(g);
    }
}

// A finished tile's outputs: lane i of the warp holds the slots of tokens i, i + 32, ... and hands
// each to the whole warp when its column is stored.
template <int MODE>
__device__ __forceinline__ void tc_epilogue_tile(const GemmArgs& a, uint32_t taddr, const int (&slot)[kDtcN / 32],
                                                 int n_tok, int row, float s) {
#pragma unroll
    for (int i = 0; i < kDtcN / 32; ++i) {
        if (32 * i >= n_tok) break;
        for (int n1 = 0; n1 < 32 && 32 * i + n1 < n_tok; n1 += 8) {
            uint32_t r[8];
            tmem_ld8(taddr + (uint32_t)(32 * i + n1), r);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int n = 32 * i + n1 + q;
                const int sl = __shfl_sync(QMOE_FULL_MASK, slot[i], n1 + q);
                if (n < n_tok && row < a.m.rows) tc_store<MODE>(a, sl, row, s * __uint_as_float(r[q]));
            }
        }
    }
}

__global__ void __launch_bounds__(kDtcThreads, 1) dict_tc_kernel(const GemmArgs a) {
    using namespace qmoe_tc;
    unsigned char* smem = (unsigned char*)(((uintptr_t)g_smem + 1023) & ~(uintptr_t)1023);
    unsigned char* stA = smem;                                   // 2 stages
    unsigned char* stB = smem + 2 * kDtcStageA;                  // 2 stages
    uint64_t* bars = (uint64_t*)(stB + kDtcStagesB * kDtcAtomB);
    uint64_t* full_a = bars;          // [2] decoders of a stage's group (4 warp arrivals)
    uint64_t* empty_a = bars + 2;     // [2] MMA commit: the A stage was read
    uint64_t* acc_full = bars + 4;    // [2] MMA commit: a tile's accumulator is final
    uint64_t* acc_empty = bars + 6;   // [2] epilogue warps (4 arrivals): the accumulator was read
    uint64_t* full_b = bars + 8;      // [3] loader (1 arrival)
    uint64_t* empty_b = bars + 11;    // [3] MMA commit: the B stage was read
    uint32_t* tmem_slot = (uint32_t*)(bars + 14);
    int* abort_flag = (int*)(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const MatDev& m = a.m;
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(full_a + s, 4);
            mbar_init(empty_a + s, 1);
            mbar_init(acc_full + s, 1);
            mbar_init(acc_empty + s, 4);
        }
        for (int s = 0; s < kDtcStagesB; ++s) {
            mbar_init(full_b + s, 1);
            mbar_init(empty_b + s, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_slot, kDtcTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_v = abort_flag;
    const int n_jobs = *a.n_jobs_dev;
    const int n_tiles = n_jobs * a.row_tiles;
    const int nb = m.nb;
    bool timed_out = false, bad = false;

    if (warp < kDtcDecWarps) {
        // ---------------- decoders: group g fills stage g for the global blocks g, g + 2, ...
        const int group = warp >> 2, rl = tid & (kDtcM - 1);
        uint32_t gb = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x) {
            const Job job = a.jobs[tile / a.row_tiles];
            const int row = (tile % a.row_tiles) * kDtcM + rl;
            const bool live = row < m.rows;
            const uint32_t* ro = m.row_off + (size_t)job.matrix * (m.rows + 1);
            const uint8_t* bl = m.blk_len + ((size_t)job.matrix * m.rows + (live ? row : 0)) * (nb - 1);
            const uint64_t cbase = m.code_base ? m.code_base[job.matrix] : 0ull;
            // the group's blocks of the tile are b_first, b_first + 2, ...; the memory reads run ahead of
            // the decoding: the block lengths that give a block's codeword range three of the group's
            // blocks ahead, the range two ahead, its first codewords one ahead, so that decoding a block
            // waits only for its dictionary entries.  Block b < nb - 1 has a stored length; the last
            // block ends at the row end.
            const int b_first = (int)((group - (int)(gb & 1u)) & 1);
            const uint2 z2 = make_uint2(0u, 0u);
            uint32_t re = 0, pl1 = 0, pl2 = 0;
            uint2 r_cur = z2, r_ahead = z2;
            RowBlk cur{};
            if (live && b_first < nb) {
                const uint32_t rs = __ldg(ro + row);
                re = __ldg(ro + row + 1);
                const uint32_t s0 = rs + (b_first == 1 ? (uint32_t)__ldg(bl) : 0u);
                r_cur = make_uint2(s0, b_first < nb - 1 ? s0 + __ldg(bl + b_first) : re);
                if (b_first + 2 < nb) {
                    const uint32_t s2 = r_cur.y + __ldg(bl + b_first + 1);
                    r_ahead = make_uint2(s2, b_first + 2 < nb - 1 ? s2 + __ldg(bl + b_first + 2) : re);
                }
                pl1 = b_first + 4 < nb ? __ldg(bl + b_first + 3) : 0u;
                pl2 = b_first + 4 < nb - 1 ? __ldg(bl + b_first + 4) : 0u;
                cur = load_rowblk(m.codes, r_cur, cbase, min(kDtcK, m.cols - b_first * kDtcK));
            }
            for (int b = 0; b < nb; ++b, ++gb) {
                if ((int)(gb & 1u) != group) continue;
                RowBlk nxt{};
                if (live && b + 2 < nb) {
                    nxt = load_rowblk(m.codes, r_ahead, cbase, min(kDtcK, m.cols - (b + 2) * kDtcK));
                    const uint32_t s4 = r_ahead.y + pl1;
                    r_ahead = b + 4 < nb ? make_uint2(s4, b + 4 < nb - 1 ? s4 + pl2 : re) : z2;
                    pl1 = b + 6 < nb ? __ldg(bl + b + 5) : 0u;
                    pl2 = b + 6 < nb - 1 ? __ldg(bl + b + 6) : 0u;
                }
                if (!mbar_wait_sleep(empty_a + group, ((gb >> 1) & 1u) ^ 1u, kDtcSpin) || *abort_v) {
                    timed_out = true;
                    break;
                }
                unsigned char* A = stA + group * kDtcStageA;
                // zero this thread's row: chunk j of each 128-byte line at swizzled position j ^ (row % 8),
                // so the 32 rows of a warp write 32 different banks per store
#pragma unroll 8
                for (int j = 0; j < kDtcK / 8; ++j) {
                    const uint32_t pos = (uint32_t)((j ^ rl) & 7);
                    *(uint4*)(A + (uint32_t)(j >> 3) * kDtcAtomA + (uint32_t)(rl >> 3) * 1024u + (uint32_t)(rl & 7) * 128u +
                              (pos << 4)) = make_uint4(0, 0, 0, 0);
                }
                if (live) decode_row_block(a, m.codes, cur, min(kDtcK, m.cols - b * kDtcK), A, rl, bad);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a + group);
                cur = nxt;
            }
        }
    } else if (warp < kDtcEpiWarp + 4) {
        // ---------------- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        const int ew = warp - kDtcEpiWarp;
        uint32_t t = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x, ++t) {
            const Job job = a.jobs[tile / a.row_tiles];
            const int row = (tile % a.row_tiles) * kDtcM + 32 * ew + lane;
            const uint32_t acc = t & 1u;
            int slot[kDtcN / 32];
#pragma unroll
            for (int i = 0; i < kDtcN / 32; ++i)
                slot[i] = lane + 32 * i < job.n_tok ? a.slots[job.slot_begin + lane + 32 * i] : 0;
            const float s = row < m.rows ? f16_to_f32(m.scale[(size_t)job.matrix * m.rows + row]) : 0.0f;
            if (!mbar_wait_sleep(acc_full + acc, (t >> 1) & 1u, kDtcSpin) || *abort_v) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(32 * ew) << 16) + acc * kDtcN;
            switch (a.mode) {
                case OUT_RELU_H: tc_epilogue_tile<OUT_RELU_H>(a, taddr, slot, job.n_tok, row, s); break;
                case OUT_GATED: tc_epilogue_tile<OUT_GATED>(a, taddr, slot, job.n_tok, row, s); break;
                case OUT_SLOT_F32: tc_epilogue_tile<OUT_SLOT_F32>(a, taddr, slot, job.n_tok, row, s); break;
                default: tc_epilogue_tile<OUT_PLAIN>(a, taddr, slot, job.n_tok, row, s); break;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + acc);
        }
    } else if (warp == kDtcLoadWarp) {
        // ---------------- loader: activations of atom g (64 columns of up to 256 tokens) into stage
        // g % 3; a stage is announced once the copies of the next atom are issued (so its own copies
        // have had an atom's time to land).  Lane l copies the rows of tokens l, l + 32, ...; rows past
        // the tokens (up to the MMA's N) are zero-filled, rows past N are not touched.
        uint32_t ga = 0;
        int pending = -1;                                   // atom whose copies are in flight
        for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x) {
            const Job job = a.jobs[tile / a.row_tiles];
            const int n16 = min(kDtcN, (job.n_tok + 15) & ~15);
            const uint16_t* src[kDtcN / 32];
#pragma unroll
            for (int i = 0; i < kDtcN / 32; ++i) {
                const int n = lane + 32 * i;
                src[i] = n < job.n_tok ? a.x + (size_t)(a.slots[job.slot_begin + n] / a.x_div) * m.cols : nullptr;
            }
            const uint32_t rowo = (uint32_t)(lane >> 3) * 1024u + (uint32_t)(lane & 7) * 128u, sw = (uint32_t)(lane & 7);
            for (int b = 0; b < nb && !timed_out; ++b) {
                const int kcols = min(kDtcK, m.cols - b * kDtcK);
                for (int at = 0; at < (kcols + 63) / 64; ++at, ++ga) {
                    const uint32_t s = ga % kDtcStagesB, use = ga / kDtcStagesB;
                    if (!mbar_wait_sleep(empty_b + s, (use & 1u) ^ 1u, kDtcSpin) || *abort_v) {
                        timed_out = true;
                        break;
                    }
                    const uint32_t B = smem_u32(stB + s * kDtcAtomB);
                    const int c0 = b * kDtcK + 64 * at;
                    const int live_ch = min(64, m.cols - c0) / 8;     // whole 16-byte chunks of the atom
#pragma unroll
                    for (int i = 0; i < kDtcN / 32; ++i) {
                        if (32 * i >= n16) break;
                        const uint16_t* p = src[i] ? src[i] + c0 : a.x;
                        const uint32_t rb = B + (uint32_t)(4 * i) * 1024u + rowo;   // token lane + 32 i
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const bool live = src[i] && ch < live_ch;
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(rb + ((((uint32_t)ch ^ sw) & 7u) << 4)),
                                         "l"(live ? p + ch * 8 : a.x), "r"(live ? 16 : 0)
                                         : "memory");
                        }
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    if (pending >= 0) {
                        asm volatile("cp.async.wait_group 1;" ::: "memory");
                        fence_async_shared();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(full_b + (uint32_t)pending % kDtcStagesB);
                    }
                    pending = (int)ga;
                }
            }
        }
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (pending >= 0) {
            fence_async_shared();
            __syncwarp();
            if (lane == 0) mbar_arrive(full_b + (uint32_t)pending % kDtcStagesB);
        }
    } else if (warp == kDtcMmaWarp && lane == 0) {
        // ---------------- MMA issuer
        uint32_t gb = 0, ga = 0, t = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x, ++t) {
            const Job job = a.jobs[tile / a.row_tiles];
            const uint32_t acc = t & 1u;
            if (!mbar_wait_sleep(acc_empty + acc, ((t >> 1) & 1u) ^ 1u, kDtcSpin) || *abort_v) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const int n16 = min(kDtcN, (job.n_tok + 15) & ~15);
            const uint32_t idesc = idesc_f16(kDtcM, n16, true, true);
            for (int b = 0; b < nb && !timed_out; ++b, ++gb) {
                const uint32_t s = gb & 1u;
                if (!mbar_wait_sleep(full_a + s, (gb >> 1) & 1u, kDtcSpin) || *abort_v) {
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = smem_u32(stA + s * kDtcStageA);
                const int kcols = min(kDtcK, m.cols - b * kDtcK);
                for (int at = 0; at < (kcols + 63) / 64; ++at, ++ga) {
                    const uint32_t sb = ga % kDtcStagesB;
                    if (!mbar_wait_sleep(full_b + sb, (ga / kDtcStagesB) & 1u, kDtcSpin) || *abort_v) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b0 = smem_u32(stB + sb * kDtcAtomB);
                    const int ksteps = min(4, (kcols - 64 * at + 15) / 16);
                    for (int k = 0; k < ksteps; ++k)
                        mma_f16(tmem + acc * kDtcN, umma_desc_sw128(a0 + (uint32_t)at * kDtcAtomA + (uint32_t)k * 32u),
                                umma_desc_sw128(b0 + (uint32_t)k * 32u), idesc, b > 0 || at > 0 || k > 0);
                    mma_commit(empty_b + sb);
                }
                if (timed_out) break;
                mma_commit(empty_a + s);
            }
            if (timed_out) break;
            mma_commit(acc_full + acc);
        }
        if (timed_out) {
            *abort_v = 1;
            // the tensor core may still be working on committed atoms: wait (bounded) for the commit
            // of the last one (it follows every earlier MMA) before the memory is released
            if (ga > 0) mbar_wait_sleep(empty_b + (ga - 1) % kDtcStagesB, ((ga - 1) / kDtcStagesB) & 1u, kDtcSpin);
        }
    }
    if (timed_out) *abort_v = 1;
    if (bad) set_error(QMOE_EFORMAT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && *abort_v) set_error(QMOE_ETIMEOUT);
    if (warp == 0) tmem_dealloc(tmem, kDtcTmemCols);
}

int launch_dict_tc(GemmArgs a, cudaStream_t st, long long tiles_hint) {
    int rc = qmoe::smem_attr((const void*)dict_tc_kernel, kDtcSmem, "dict tc attr");
    if (rc) return rc;
    a.rows_per_tile = kDtcM;
    a.row_tiles = (a.m.rows + kDtcM - 1) / kDtcM;
    const long long grid = std::max(1LL, std::min(tiles_hint, (long long)qmoe::sm_count()));
    dict_tc_kernel<<<(unsigned)grid, kDtcThreads, kDtcSmem, st>>>(a);
    return qmoe::launch_check("dict_tc_kernel");
}

// ------------------------------------------------------------ decode (test)
__global__ void decode_dense_kernel(const uint32_t* __restrict__ words, MatDev m, float* __restrict__ out) {
    const int gw = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= m.rows * m.nb) return;
    const int r = gw / m.nb, b = gw % m.nb;
    const int c0 = b * m.block, blen = min(m.cols, c0 + m.block) - c0;
    float* o = out + (size_t)r * m.cols + c0;
    for (int p = lane; p < blen; p += 32) o[p] = 0.0f;
    __syncwarp();
    // block b starts after the stored lengths of blocks 0 .. b-1 of the row; the last block ends at the
    // row end
    const uint8_t* bl = m.blk_len + (size_t)r * (m.nb - 1);
    uint32_t pre = 0;
    for (int j = lane; j < b; j += 32) pre += bl[j];
    pre = (uint32_t)warp_sum_int((int)pre);
    const uint32_t lo = m.row_off[r] + pre;
    const uint32_t hi = b < m.nb - 1 ? lo + bl[b] : m.row_off[r + 1];
    const float s = f16_to_f32(m.scale[r]);
    bool bad = hi < lo;
    int base = 0;
    for (uint32_t i = lo; i < hi && !bad; i += 32) {
        const bool valid = i + lane < hi;
        uint32_t w0 = 0, w1 = 0;
        int len = 0;
        if (valid) {
            const uint32_t code = m.codes[i + lane];
            w0 = __ldg(words + 2 * code);
            w1 = __ldg(words + 2 * code + 1);
            len = 2 * (int)(w0 & 15u);
            if ((w1 & 15u) != (w0 & 15u) || len == 0) {
                bad = true;
                len = 0;
            }
        }
        const int incl = warp_incl_scan(len, lane);
        const int start = base + incl - len;
        for (int q = 0; q < len; ++q) {
            const int p = start + q;
            const uint32_t sym = ((q < 14 ? w0 : w1) >> (4 + 2 * (q % 14))) & 3u;
            if (p >= blen || sym == 3u) {
                bad = true;
                break;
            }
            o[p] = sym == 0u ? 0.0f : (sym == 1u ? -s : s);
        }
        base += __shfl_sync(QMOE_FULL_MASK, incl, 31);
        bad = __any_sync(QMOE_FULL_MASK, bad);
    }
    if (base != blen) bad = true;
    if (bad && lane == 0) set_error(QMOE_EFORMAT);
}

// ------------------------------------------------------------ router
// Router for E > 256 and many tokens: one warp per token (more tokens per block than
// route_kernel_block); the chosen experts are kept in a per-thread array.
__global__ void route_kernel_warp(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                             float* __restrict__ gates) {
    const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    int chosen[32];
    float chosen_v[32];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        // loads first and unconditional, eight iterations unrolled: the loads go out together
#pragma unroll 8
        for (int e = lane; e < E; e += 32) {
            const float v = row[e];
            bool taken = false;
            for (int q = 0; q < j; ++q) taken |= (chosen[q] == e);
            if (taken) continue;
            if (v > bv || (v == bv && e < bi)) {
                bv = v;
                bi = e;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(QMOE_FULL_MASK, bv, d);
            const int oi = __shfl_xor_sync(QMOE_FULL_MASK, bi, d);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        chosen[j] = bi;
        chosen_v[j] = bv;
    }
    const float mx = chosen_v[0];
    float sum = 0.0f;
#pragma unroll 8
    for (int e = lane; e < E; e += 32) sum += expf(row[e] - mx);
    sum = warp_sum(sum);
    if (lane == 0) {
        for (int j = 0; j < k; ++j) {
            ids[(size_t)t * k + j] = chosen[j];
            gates[(size_t)t * k + j] = expf(chosen_v[j] - mx) / sum;
        }
    }
}

// Router for 256 < E <= 8192: one block of 256 threads per token; thread i keeps logits
// i, i + 256, ... (up to 32) and a taken mask in registers; each of the k passes is a block-wide
// argmax (highest logit, ties to the lower expert id).  Gates: softmax over all E logits read at
// the chosen experts.
constexpr int kRouteBlock = 256;
// up to this many tokens a block per token (latency); beyond, a warp per token (throughput)
constexpr int kRouteBlockMaxT = 512;

__global__ void __launch_bounds__(kRouteBlock) route_kernel_block(const float* __restrict__ logits, int T, int E,
                                                                  int k, int32_t* __restrict__ ids,
                                                                  float* __restrict__ gates) {
    __shared__ float wv[kRouteBlock / 32], s_v[32], s_sum[kRouteBlock / 32];
    __shared__ int wi[kRouteBlock / 32], s_id[32];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* row = logits + (size_t)t * E;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = tid + kRouteBlock * i < E ? row[tid + kRouteBlock * i] : -INFINITY;
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int e = tid + kRouteBlock * i;
            if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(QMOE_FULL_MASK, bv, d);
            const int oi = __shfl_xor_sync(QMOE_FULL_MASK, bi, d);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            wv[warp] = bv;
            wi[warp] = bi;
        }
        __syncthreads();
        if (warp == 0) {
            bv = lane < kRouteBlock / 32 ? wv[lane] : -INFINITY;
            bi = lane < kRouteBlock / 32 ? wi[lane] : 0x7FFFFFFF;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const float ov = __shfl_xor_sync(QMOE_FULL_MASK, bv, d);
                const int oi = __shfl_xor_sync(QMOE_FULL_MASK, bi, d);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (lane == 0) {
                s_v[j] = bv;
                s_id[j] = bi;
            }
        }
        __syncthreads();
        const int c = s_id[j];
        if (c < E && (c % kRouteBlock) == tid) taken |= 1u << (c / kRouteBlock);
    }
    const float mx = s_v[0];
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (tid + kRouteBlock * i < E) sum += expf(v[i] - mx);
    sum = warp_sum(sum);
    if (lane == 0) s_sum[warp] = sum;
    __syncthreads();
    if (warp == 0) {
        const float tot = warp_sum(lane < kRouteBlock / 32 ? s_sum[lane] : 0.0f);
        if (lane < k) {
            ids[(size_t)t * k + lane] = s_id[lane];
            gates[(size_t)t * k + lane] = expf(s_v[lane] - mx) / tot;
        }
    }
}

// Router for E <= 256: one warp per token; a lane keeps its (up to) 8 logits and a taken mask in
// registers, and lane j keeps the j-th choice.  Same selection, tie-breaking and gates as
// route_kernel_block.
__global__ void route_kernel_small(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                                   float* __restrict__ gates) {
    const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float* row = logits + (size_t)t * E;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = lane + 32 * i < E ? row[lane + 32 * i] : -INFINITY;
    uint32_t taken = 0;
    int my_id = 0;
    float my_v = 0.0f, first_v = 0.0f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(QMOE_FULL_MASK, bv, d);
            const int oi = __shfl_xor_sync(QMOE_FULL_MASK, bi, d);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane && bi < E) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
        if (j == 0) first_v = bv;
    }
    const float mx = first_v;
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (lane + 32 * i < E) sum += expf(v[i] - mx);
    sum = warp_sum(sum);
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        gates[(size_t)t * k + lane] = expf(my_v - mx) / sum;
    }
}

// ------------------------------------------------------------ planner
// One block: histogram, exclusive scan, stable placement (one warp, in slot
// order) and the job tables of both matrices of the layer.
constexpr int kPlanThreads = 1024;

__device__ int block_excl_scan(int v, int* sbuf) {
    // sbuf: at least 32 ints
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31) sbuf[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int s = lane < nw ? sbuf[lane] : 0;
        const int si = warp_incl_scan(s, lane);
        sbuf[lane] = si - s;
    }
    __syncthreads();
    const int res = sbuf[warp] + incl - v;
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ ids, int n_slots, int E,
                                                            int nt_a, int nt_b, int tc_min, int nt_tc,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                                            Job* __restrict__ jobs_a, Job* __restrict__ jobs_b,
                                                            Job* __restrict__ jobs_tc, int* __restrict__ n_jobs) {
    // shared memory: hist[E] (counts, then running positions) and off[E + 1] (exclusive offsets);
    // thread i owns experts [i per, (i + 1) per), so one block scan covers all E
    extern __shared__ int psm[];
    int* hist = psm;
    int* off = psm + E;
    __shared__ int sbuf[32];
    const int tid = threadIdx.x;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    for (int e = e0; e < e1; ++e) hist[e] = 0;
    __syncthreads();
    for (int i = tid; i < n_slots; i += blockDim.x) {
        const int e = ids[i];
        if (e < 0 || e >= E) set_error(QMOE_EINVAL);
        else atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    int local = 0;
    for (int e = e0; e < e1; ++e) local += hist[e];
    const int ex = block_excl_scan(local, sbuf);
    int run = ex;
    for (int e = e0; e < e1; ++e) {
        const int c = hist[e];
        counts[e] = c;
        offsets[e] = run;
        off[e] = run;
        hist[e] = run;                                 // running position for the placement
        run += c;
    }
    if (tid == blockDim.x - 1) {
        offsets[E] = ex + local;
        off[E] = ex + local;
    }
    __syncthreads();
    // stable placement: warp 0 walks the slots in order
    if (tid < 32) {
        const int lane = tid;
        for (int base = 0; base < n_slots; base += 32) {
            const int i = base + lane;
            int e = i < n_slots ? ids[i] : -1;
            if (e >= E) e = -1;
            const unsigned act = __ballot_sync(QMOE_FULL_MASK, e >= 0);
            const unsigned same = __match_any_sync(QMOE_FULL_MASK, e);
            if (e >= 0) {
                const unsigned lower = same & act & ((1u << lane) - 1u);
                const int rank = __popc(lower);
                const int cur = hist[e];
                perm[cur + rank] = i;
                __syncwarp(same);
                if (lower == 0) hist[e] = cur + __popc(same & act);
            }
            __syncwarp();
        }
    }
    if (!jobs_a) return;
    // job tables in expert order: chunks of nt tokens of the experts each kernel takes
    // (experts with at least tc_min tokens go to the tensor-core kernel when tc_min > 0); counts
    // and offsets come from shared memory
    for (int which = 0; which < 3; ++which) {
        const int nt = which == 0 ? nt_a : which == 1 ? nt_b : nt_tc;
        Job* jobs = which == 0 ? jobs_a : which == 1 ? jobs_b : jobs_tc;
        if (which == 2 && !jobs_tc) {
            if (tid == 0) n_jobs[2] = 0;
            break;
        }
        int nj_local = 0;
        for (int e = e0; e < e1; ++e) {
            int c = off[e + 1] - off[e];
            const bool tc = tc_min > 0 && c >= tc_min;
            if (tc != (which == 2)) c = 0;
            nj_local += (c + nt - 1) / nt;
        }
        const int first0 = block_excl_scan(nj_local, sbuf);
        int first = first0;
        for (int e = e0; e < e1; ++e) {
            int c = off[e + 1] - off[e];
            const bool tc = tc_min > 0 && c >= tc_min;
            if (tc != (which == 2)) c = 0;
            const int nj = (c + nt - 1) / nt;
            for (int q = 0; q < nj; ++q) {
                Job jb;
                jb.matrix = e;
                jb.slot_begin = off[e] + q * nt;
                jb.n_tok = min(nt, c - q * nt);
                jb.pad = 0;
                jobs[first + q] = jb;
            }
            first += nj;
        }
        if (tid == blockDim.x - 1) n_jobs[which] = first0 + nj_local;
        __syncthreads();                               // sbuf is reused by the next scan
    }
}

// ------------------------------------------------------------ combine
__global__ void combine_kernel(const float* __restrict__ o, const float* __restrict__ gates, int T, int k, int d,
                               void* __restrict__ y, int y_is_f32) {
    const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (i >= (size_t)T * d) return;
    const size_t t = i / d, c = i % d;
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) acc = fmaf(gates[t * k + j], o[(t * k + j) * d + c], acc);
    if (y_is_f32) ((float*)y)[i] = acc;
    else ((uint16_t*)y)[i] = f32_to_bf16(acc);
}

// ------------------------------------------------------------ host side
int g_sm_count[64];

// One token: (x, -x) bf16 pairs; several: bf16 [col][token]; plus kPadCols zero columns.
size_t xs_bytes(int cols, int nt) {
    const size_t c = (size_t)cols + kPadCols;
    return ((nt == 1 ? c * 4 : c * nt * 2) + 15) & ~(size_t)15;
}

size_t tile_smem(int cols, int nt) { return xs_bytes(cols, nt) + kSaccBytes; }

// Largest token chunk (8, 4, 2, 1) whose staged activations and row sums fit the budget.
int nt_max_for(int cols, int budget) {
    for (int nt = 8; nt >= 1; nt >>= 1)
        if (tile_smem(cols, nt) <= (size_t)budget) return nt;
    return 0;
}

// Row-sum bytes of a tile: the SMEM the staged activations leave, within
// [kSaccBytes, cap].
int sacc_bytes_for(int cols, int nt, int budget, int cap = QMOE_SACC_MAX) {
    const long long left = (long long)budget - (long long)xs_bytes(cols, nt);
    return (int)std::max<long long>(kSaccBytes, std::min<long long>(cap, left) & ~15LL);
}

// Rows per tile: as many as the row-sum buffer holds for nt tokens, split evenly,
// a multiple of the warp count; at least `min_tiles` tiles when given.
int rows_per_tile_for(int rows, int nt, int nwarps, long long n_jobs, long long min_tiles, int sacc_bytes) {
    int cap = sacc_bytes / (4 * nt);
    if (min_tiles > 0) {
        const long long per_job = (min_tiles + std::max(1LL, n_jobs) - 1) / std::max(1LL, n_jobs);
        cap = (int)std::max<long long>(nwarps, std::min<long long>(cap, (rows + per_job - 1) / per_job));
    }
    // the cap in whole warps, then tiles as equal as whole warps allow
    const int cap_w = std::max(nwarps, cap / nwarps * nwarps);
    const int n = (rows + cap_w - 1) / cap_w;
    const int rpt = ((rows + n - 1) / n + nwarps - 1) / nwarps * nwarps;
    return std::min(rpt, cap_w);
}

bool valid_set(const qmoe_matrix_set* s) {
    if (!s || !s->codes || !s->row_off || !s->scale_f16 || s->count < 1 || s->rows < 1 || s->cols < 2 ||
        (s->cols % 2) != 0 || s->block < 2 || (s->block % 2) != 0 || s->block > 510 || (s->count > 1 && !s->code_base))
        return false;
    const int nb = (s->cols + s->block - 1) / s->block;
    return nb == 1 || s->blk_len;
}

MatDev to_dev(const qmoe_matrix_set* s) {
    MatDev m;
    m.codes = s->codes;
    m.code_base = s->code_base;
    m.row_off = s->row_off;
    m.blk_len = s->blk_len;
    m.scale = s->scale_f16;
    m.count = s->count;
    m.rows = s->rows;
    m.cols = s->cols;
    m.block = s->block;
    m.nb = (s->cols + s->block - 1) / s->block;
    return m;
}

template <int NTMAX>
int launch_rows_as(const GemmArgs& a, unsigned grid, int threads, size_t smem, cudaStream_t st) {
    int rc = qmoe::smem_attr((const void*)dict_rows_kernel<NTMAX>, kSmemMax, "dict rows attr");
    if (rc) return rc;
    dict_rows_kernel<NTMAX><<<grid, threads, smem, st>>>(a);
    return QMOE_OK;
}

// Share of a block's warps busy over the rounds of a job's 32-row groups in the row-per-lane kernel.
double row_round_efficiency(int rows, int nt_max) {
    const int max_w = threads_smem_dict(nt_max) / 32;
    const long long groups = (rows + 31) / 32, rounds = (groups + max_w - 1) / max_w;
    return (double)groups / (double)(rounds * max_w);
}

// Launches with the compact table in shared memory take the row-per-lane kernel when a job's rows
// fill the block's warps in nearly whole rounds (>= 95 % busy), else the flat-stream kernel, which
// spreads a job's codewords evenly over its warps.  Measured on GB300: c2048 wi (6144 rows, 96 %)
// 2.61 -> 2.21 ms on the row kernel, c2048 wo (2080 rows, 90 %) 2.29 ms flat against 2.43 ms.
bool use_row_kernel(int rows, int nt_max) { return row_round_efficiency(rows, nt_max) >= 0.95; }

// The row-per-lane kernel (compact table in shared memory): a tile is one 32-row group per warp of
// the block, so a warp done with its group moves on to the next tile of the same job at once.
int launch_rows(GemmArgs a, int nt_max, cudaStream_t st) {
    const int sms = qmoe::sm_count();
    const int rows = a.m.rows;
    const int max_w = threads_smem_dict(nt_max) / 32;
    const int rpt = std::min(32 * max_w, (rows + 31) / 32 * 32);
    a.nt_max = nt_max;
    a.rows_per_tile = rpt;
    a.row_tiles = (rows + rpt - 1) / rpt;
    a.xs_bytes = (int)xs_bytes(a.m.cols, nt_max);
    a.inv_cols = 1.0f / (float)a.m.cols;
    const size_t smem = (size_t)kDictBytes + xs_bytes(a.m.cols, nt_max);
    if (smem > (size_t)kSmemMax) return qmoe::fail(QMOE_EUNSUPPORTED, "dict_rows: staged activations do not fit");
    const int threads = rpt;
    int rc;
    switch (nt_max) {
        case 1: rc = launch_rows_as<1>(a, (unsigned)sms, threads, smem, st); break;
        case 2: rc = launch_rows_as<2>(a, (unsigned)sms, threads, smem, st); break;
        case 4: rc = launch_rows_as<4>(a, (unsigned)sms, threads, smem, st); break;
        case 8: rc = launch_rows_as<8>(a, (unsigned)sms, threads, smem, st); break;
        default: return qmoe::fail(QMOE_EINVAL, "dict_rows: token chunk must be 1, 2, 4 or 8");
    }
    if (rc) return rc;
    return qmoe::launch_check("dict_rows_kernel");
}

template <bool DICT_SMEM, int NTMAX>
int launch_gemm_as(const GemmArgs& a, unsigned grid, int threads, size_t smem, cudaStream_t st) {
    int rc = qmoe::smem_attr((const void*)dict_gemm_kernel<DICT_SMEM, NTMAX>, kSmemMax, "dict gemm attr");
    if (rc) return rc;
    dict_gemm_kernel<DICT_SMEM, NTMAX><<<grid, threads, smem, st>>>(a);
    return QMOE_OK;
}

int launch_gemm(GemmArgs a, bool dict_smem, int nt_max, int rows_per_tile, cudaStream_t st, long long tiles_hint) {
    const int sms = qmoe::sm_count();
    if (dict_smem && use_row_kernel(a.m.rows, nt_max)) return launch_rows(a, nt_max, st);
    a.nt_max = nt_max;
    a.rows_per_tile = rows_per_tile;
    a.row_tiles = (a.m.rows + rows_per_tile - 1) / rows_per_tile;
    a.xs_bytes = (int)xs_bytes(a.m.cols, nt_max);
    a.inv_cols = 1.0f / (float)a.m.cols;
    const size_t smem = (dict_smem ? (size_t)kDictBytes : 0) + xs_bytes(a.m.cols, nt_max) +
                        std::max<size_t>(kSaccBytes, ((size_t)rows_per_tile * nt_max * 4 + 15) & ~(size_t)15);
    if (smem > (size_t)kSmemMax) return qmoe::fail(QMOE_EUNSUPPORTED, "dict_gemm: tile does not fit in shared memory");
    const unsigned grid = dict_smem ? (unsigned)sms : (unsigned)std::max(1LL, std::min(tiles_hint, (long long)sms * 4));
    const int threads = dict_smem ? threads_smem_dict(nt_max) : kThreadsGlobalDict;
    int rc;
    switch ((dict_smem ? 16 : 0) + nt_max) {
        case 16 + 1: rc = launch_gemm_as<true, 1>(a, grid, threads, smem, st); break;
        case 16 + 2: rc = launch_gemm_as<true, 2>(a, grid, threads, smem, st); break;
        case 16 + 4: rc = launch_gemm_as<true, 4>(a, grid, threads, smem, st); break;
        case 16 + 8: rc = launch_gemm_as<true, 8>(a, grid, threads, smem, st); break;
        case 1: rc = launch_gemm_as<false, 1>(a, grid, threads, smem, st); break;
        case 2: rc = launch_gemm_as<false, 2>(a, grid, threads, smem, st); break;
        case 4: rc = launch_gemm_as<false, 4>(a, grid, threads, smem, st); break;
        case 8: rc = launch_gemm_as<false, 8>(a, grid, threads, smem, st); break;
        default: return qmoe::fail(QMOE_EINVAL, "dict_gemm: token chunk must be 1, 2, 4 or 8");
    }
    if (rc) return rc;
    return qmoe::launch_check("dict_gemm_kernel");
}

}  // namespace

namespace qmoe {

void* current_context() {
    using GetCurrent = int (*)(void**);
    static GetCurrent fn = []() -> GetCurrent {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return (GetCurrent)f;
    }();
    void* ctx = nullptr;
    if (!fn || fn(&ctx) != 0) return nullptr;
    return ctx;
}

int smem_attr(const void* kernel, int bytes, const char* where) {
    struct Entry {
        const void* kernel;
        int dev;
        void* ctx;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> set;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    void* ctx = current_context();
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : set)
        if (ctx && e.kernel == kernel && e.dev == dev && e.ctx == ctx && e.bytes >= bytes) return QMOE_OK;
    const int rc = cuda_check(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), where);
    if (rc || !ctx) return rc;
    for (Entry& e : set)
        if (e.kernel == kernel && e.dev == dev && e.ctx == ctx) {
            e.bytes = bytes;
            return QMOE_OK;
        }
    set.push_back({kernel, dev, ctx, bytes});
    return QMOE_OK;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_sm_count[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 148;
    }
    return g_sm_count[dev];
}

int launch_plan(const int32_t* ids, int n_slots, int E, int nt_a, int nt_b, int32_t* counts, int32_t* offsets,
                int32_t* perm, Job* jobs_a, Job* jobs_b, int* n_jobs, cudaStream_t st, int tc_min, int nt_tc,
                Job* jobs_tc) {
    const size_t smem = (size_t)(2 * E + 1) * sizeof(int);
    if (smem > 48 * 1024) {
        const int rc = smem_attr((const void*)plan_kernel, (int)smem, "plan attr");
        if (rc) return rc;
    }
    plan_kernel<<<1, kPlanThreads, smem, st>>>(ids, n_slots, E, nt_a, nt_b, tc_min, nt_tc, counts, offsets, perm, jobs_a,
                                               jobs_b, jobs_tc, n_jobs);
    return launch_check("plan_kernel");
}

static cudaEvent_t g_phase[8];
static int g_n_phase = 0;

void phase_event(int i, cudaStream_t st) {
    if (i < g_n_phase) cudaEventRecord(g_phase[i], st);
}

int dict_take_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dict_error, sizeof(int)) != cudaSuccess) return QMOE_ECUDA;
    const int z = 0;
    if (cudaMemcpyToSymbol(g_dict_error, &z, sizeof(int)) != cudaSuccess) return QMOE_ECUDA;
    return v;
}

}  // namespace qmoe

using qmoe::fail;

extern "C" int qmoe_decode_dense(const qmoe_dict* dict, const qmoe_matrix_set* mat, float* w_out, void* stream) {
    qmoe::clear_error();
    if (!dict || !dict->words || !w_out || !valid_set(mat) || mat->count != 1)
        return fail(QMOE_EINVAL, "qmoe_decode_dense: bad arguments (count must be 1)");
    MatDev m = to_dev(mat);
    const long long warps = (long long)m.rows * m.nb;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    decode_dense_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(dict->words, m, w_out);
    return qmoe::launch_check("qmoe_decode_dense");
}

extern "C" int qmoe_expert_matvec(const qmoe_dict* dict, const qmoe_matrix_set* mat, const void* x_bf16, int T,
                                  void* y, int y_is_f32, void* stream) {
    qmoe::clear_error();
    if (!dict || !dict->words || !dict->compact || !valid_set(mat) || mat->count != 1)
        return fail(QMOE_EINVAL, "qmoe_expert_matvec: bad dictionary or matrix (count must be 1)");
    if (T < 0) return fail(QMOE_EINVAL, "qmoe_expert_matvec: T < 0");
    if (T == 0) return QMOE_OK;
    if (!x_bf16 || !y) return fail(QMOE_EINVAL, "qmoe_expert_matvec: NULL x or y");
    const int nt_max = nt_max_for(mat->cols, kBudgetGlobalDict);
    if (!nt_max) return fail(QMOE_EUNSUPPORTED, "qmoe_expert_matvec: cols too large");
    GemmArgs a{};
    a.dictA = (const uint16_t*)dict->compact;
    a.dictB = (const uint8_t*)dict->compact + kDictA;
    a.dictW = (const uint32_t*)((const uint8_t*)dict->compact + kDictWordsOff);
    a.words = dict->words;
    a.m = to_dev(mat);
    a.x = (const uint16_t*)x_bf16;
    a.x_div = 1;
    a.jobs = nullptr;
    a.slots = nullptr;
    a.T_implicit = T;
    a.mode = OUT_PLAIN;
    a.y_is_f32 = y_is_f32 ? 1 : 0;
    a.out = y;
    const long long jobs = (T + nt_max - 1) / nt_max;
    const int rpt = rows_per_tile_for(mat->rows, nt_max, kThreadsGlobalDict / 32, jobs, 2LL * qmoe::sm_count(),
                                      kSaccBytes);
    return launch_gemm(a, false, nt_max, rpt, (cudaStream_t)stream, jobs * ((mat->rows + rpt - 1) / rpt));
}

extern "C" int qmoe_route(const float* logits, int T, int E, int k, int32_t* ids, float* gates, void* stream) {
    qmoe::clear_error();
    if (T < 0 || E < 1 || E > kPlanMaxE || k < 1 || k > E || k > 32)
        return fail(QMOE_EINVAL, "qmoe_route: need 1 <= k <= min(E, 32), E <= 8192, T >= 0");
    if (T == 0) return QMOE_OK;
    if (!logits || !ids || !gates) return fail(QMOE_EINVAL, "qmoe_route: NULL pointer");
    const int threads = 256;
    const long long blocks = ((long long)T * 32 + threads - 1) / threads;
    if (E <= 256) route_kernel_small<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(logits, T, E, k, ids, gates);
    else if (T <= kRouteBlockMaxT)
        route_kernel_block<<<(unsigned)T, kRouteBlock, 0, (cudaStream_t)stream>>>(logits, T, E, k, ids, gates);
    else route_kernel_warp<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(logits, T, E, k, ids, gates);
    return qmoe::launch_check("qmoe_route");
}

namespace {
struct MoeWs {
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    Job* jobs_a;
    Job* jobs_b;
    Job* jobs_tc;
    int* n_jobs;
    uint16_t* h;
    float* o;
    size_t bytes;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

MoeWs moe_ws_layout(void* base, int E, int d_model, int d_ff, int T, int k) {
    MoeWs w{};
    size_t off = 0;
    const size_t slots = (size_t)T * k;
    auto take = [&](size_t bytes) {
        void* p = base ? (void*)((char*)base + off) : nullptr;
        off += align256(bytes);
        return p;
    };
    w.counts = (int32_t*)take(sizeof(int32_t) * E);
    w.offsets = (int32_t*)take(sizeof(int32_t) * (E + 1));
    w.perm = (int32_t*)take(sizeof(int32_t) * std::max<size_t>(slots, 1));
    w.jobs_a = (Job*)take(sizeof(Job) * std::max<size_t>(slots, 1));
    w.jobs_b = (Job*)take(sizeof(Job) * std::max<size_t>(slots, 1));
    w.jobs_tc = (Job*)take(sizeof(Job) * std::max<size_t>(slots, 1));
    w.n_jobs = (int*)take(sizeof(int) * 4);
    w.h = (uint16_t*)take(sizeof(uint16_t) * slots * d_ff);
    w.o = k > 1 ? (float*)take(sizeof(float) * slots * d_model) : nullptr;
    w.bytes = off;
    return w;
}
}  // namespace

extern "C" int qmoe_bucketise(const int32_t* ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                              int32_t* perm, void* stream) {
    qmoe::clear_error();
    if (T < 0 || k < 1 || E < 1 || E > kPlanMaxE) return fail(QMOE_EINVAL, "qmoe_bucketise: bad sizes");
    if (!counts || !offsets || (T > 0 && (!ids || !perm))) return fail(QMOE_EINVAL, "qmoe_bucketise: NULL pointer");
    return qmoe::launch_plan(ids, T * k, E, 1, 1, counts, offsets, perm, nullptr, nullptr, nullptr,
                             (cudaStream_t)stream);
}

extern "C" int qmoe_moe_layer_ws_size(int E, int d_model, int d_ff, int T, int k, size_t* bytes) {
    qmoe::clear_error();
    if (!bytes || E < 1 || E > kPlanMaxE || d_model < 2 || d_ff < 2 || T < 0 || k < 1 || k > E)
        return fail(QMOE_EINVAL, "qmoe_moe_layer_ws_size: bad sizes");
    *bytes = moe_ws_layout(nullptr, E, d_model, d_ff, T, k).bytes;
    return QMOE_OK;
}

// launches with this many token slots stage the compact dictionary in shared memory; smaller
// ones read it through L1/L2
#ifndef QMOE_SMEM_DICT_MIN_SLOTS
#define QMOE_SMEM_DICT_MIN_SLOTS 16
#endif

extern "C" int qmoe_moe_layer_kernels(int E, int d_model, int d_ff, int T, int k, int* wi_kernel, int* wo_kernel,
                                      int* tc) {
    qmoe::clear_error();
    if (!wi_kernel || !wo_kernel || !tc || E < 1 || E > kPlanMaxE || d_model < 2 || d_ff < 2 || T < 0 || k < 1 ||
        k > E)
        return fail(QMOE_EINVAL, "qmoe_moe_layer_kernels: bad sizes or NULL outputs");
    const long long slots = (long long)T * k;
    const bool big = slots >= QMOE_SMEM_DICT_MIN_SLOTS;
    const int budget = big ? kBudgetSmemDict : kBudgetGlobalDict;
    const int nt_wi = nt_max_for(d_model, budget), nt_wo = nt_max_for(d_ff, budget);
    if (!nt_wi || !nt_wo) return fail(QMOE_EUNSUPPORTED, "qmoe_moe_layer_kernels: d_model or d_ff too large");
    *wi_kernel = !big ? QMOE_KERNEL_FLAT_L2 : use_row_kernel(d_ff, nt_wi) ? QMOE_KERNEL_ROWS : QMOE_KERNEL_FLAT;
    *wo_kernel = !big ? QMOE_KERNEL_FLAT_L2 : use_row_kernel(d_model, nt_wo) ? QMOE_KERNEL_ROWS : QMOE_KERNEL_FLAT;
    *tc = big && slots >= kTcMinSlots && d_model % 8 == 0 && d_ff % 8 == 0 ? 1 : 0;
    return QMOE_OK;
}

extern "C" int qmoe_moe_layer(const qmoe_dict* dict, const qmoe_matrix_set* wi, const qmoe_matrix_set* wo,
                              const void* x_bf16, int T, int k, const int32_t* ids, const float* gates, void* y,
                              int y_is_f32, void* workspace, size_t ws_bytes, void* stream) {
    qmoe::clear_error();
    if (!dict || !dict->words || !dict->compact || !valid_set(wi) || !valid_set(wo))
        return fail(QMOE_EINVAL, "qmoe_moe_layer: bad dictionary or matrix sets");
    const int E = wi->count, d_model = wi->cols, d_ff = wi->rows;
    if (wo->count != E || wo->rows != d_model || wo->cols != d_ff)
        return fail(QMOE_EINVAL, "qmoe_moe_layer: wo must be d_model x d_ff with the same expert count as wi");
    if (E > kPlanMaxE || T < 0 || k < 1 || k > E) return fail(QMOE_EINVAL, "qmoe_moe_layer: bad E, T or k");
    if (T == 0) return QMOE_OK;
    if (!x_bf16 || !ids || !gates || !y || !workspace) return fail(QMOE_EINVAL, "qmoe_moe_layer: NULL pointer");
    MoeWs w = moe_ws_layout(workspace, E, d_model, d_ff, T, k);
    if (ws_bytes < w.bytes) return fail(QMOE_ECAPACITY, "qmoe_moe_layer: workspace too small");
    const long long slots = (long long)T * k;
    // launches with at least QMOE_SMEM_DICT_MIN_SLOTS token slots stage the compact dictionary in
    // shared memory; smaller ones read it through L1/L2
    const bool big = slots >= QMOE_SMEM_DICT_MIN_SLOTS;
    const int budget = big ? kBudgetSmemDict : kBudgetGlobalDict;
    const int nt_wi = nt_max_for(d_model, budget), nt_wo = nt_max_for(d_ff, budget);
    const int nw_wi = (big ? threads_smem_dict(nt_wi) : kThreadsGlobalDict) / 32;
    const int nw_wo = (big ? threads_smem_dict(nt_wo) : kThreadsGlobalDict) / 32;
#ifndef QMOE_MIN_TILES_PER_SM
#define QMOE_MIN_TILES_PER_SM 2
#endif
    const long long min_tiles = (long long)QMOE_MIN_TILES_PER_SM * qmoe::sm_count();
    const int sacc_cap = slots <= QMOE_SACC_SMALL_SLOTS ? 2 * QMOE_SACC_MAX : QMOE_SACC_MAX;
    const int rpt_wi = nt_wi ? rows_per_tile_for(d_ff, nt_wi, nw_wi, slots, min_tiles,
                                                 big ? sacc_bytes_for(d_model, nt_wi, budget, sacc_cap) : kSaccBytes) : 0;
    const int rpt_wo = nt_wo ? rows_per_tile_for(d_model, nt_wo, nw_wo, slots, min_tiles,
                                                 big ? sacc_bytes_for(d_ff, nt_wo, budget, sacc_cap) : kSaccBytes) : 0;
    if (!nt_wi || !nt_wo) return fail(QMOE_EUNSUPPORTED, "qmoe_moe_layer: d_model or d_ff too large");
    cudaStream_t st = (cudaStream_t)stream;
    // experts with at least kTcMinTokens tokens take the tensor-core kernel
    // (below kTcMinSlots token slots every expert takes the CUDA-core kernel: an expert of such a
    // batch rarely reaches kTcMinTokens, and an empty tensor-core launch costs a few microseconds)
    const bool use_tc = big && slots >= kTcMinSlots && d_model % 8 == 0 && d_ff % 8 == 0;
    qmoe::phase_event(0, st);
    int rc = qmoe::launch_plan(ids, (int)slots, E, nt_wi, nt_wo, w.counts, w.offsets, w.perm, w.jobs_a, w.jobs_b,
                               w.n_jobs, st, use_tc ? kTcMinTokens : 0, kDtcN, use_tc ? w.jobs_tc : nullptr);
    if (rc) return rc;
    qmoe::phase_event(1, st);
    GemmArgs a{};
    a.dictA = (const uint16_t*)dict->compact;
    a.dictB = (const uint8_t*)dict->compact + kDictA;
    a.dictW = (const uint32_t*)((const uint8_t*)dict->compact + kDictWordsOff);
    a.words = dict->words;
    a.slots = w.perm;
    a.T_implicit = 0;
    a.y_is_f32 = y_is_f32 ? 1 : 0;
    a.gates = gates;
    // wi: h[slot] = bf16(relu(Wi x[slot / k]))
    a.m = to_dev(wi);
    a.x = (const uint16_t*)x_bf16;
    a.x_div = k;
    a.jobs = w.jobs_a;
    a.n_jobs_dev = w.n_jobs;
    a.mode = OUT_RELU_H;
    a.out = w.h;
    rc = launch_gemm(a, big, nt_wi, rpt_wi, st, slots * ((d_ff + rpt_wi - 1) / rpt_wi));
    if (rc) return rc;
    qmoe::phase_event(2, st);
    if (use_tc) {
        GemmArgs t = a;
        t.jobs = w.jobs_tc;
        t.n_jobs_dev = w.n_jobs + 2;
        if ((rc = launch_dict_tc(t, st, 2LL * qmoe::sm_count()))) return rc;
    }
    qmoe::phase_event(3, st);
    // wo: o[slot] = Wo h[slot]; gated straight into y when k == 1
    a.m = to_dev(wo);
    a.x = w.h;
    a.x_div = 1;
    a.jobs = w.jobs_b;
    a.n_jobs_dev = w.n_jobs + 1;
    a.mode = k == 1 ? OUT_GATED : OUT_SLOT_F32;
    a.out = k == 1 ? y : (void*)w.o;
    rc = launch_gemm(a, big, nt_wo, rpt_wo, st, slots * ((d_model + rpt_wo - 1) / rpt_wo));
    if (rc) return rc;
    qmoe::phase_event(4, st);
    if (use_tc) {
        GemmArgs t = a;
        t.jobs = w.jobs_tc;
        t.n_jobs_dev = w.n_jobs + 2;
        if ((rc = launch_dict_tc(t, st, 2LL * qmoe::sm_count()))) return rc;
    }
    if (k > 1) {
        const size_t n = (size_t)T * d_model;
        combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w.o, gates, T, k, d_model, y, y_is_f32 ? 1 : 0);
        rc = qmoe::launch_check("combine_kernel");
    }
    qmoe::phase_event(5, st);
    return rc;
}

extern "C" int qmoe_set_phase_events(void* const* events, int n) {
    qmoe::clear_error();
    if (!events || n == 0) {
        qmoe::g_n_phase = 0;
        return QMOE_OK;
    }
    if (n < 6 || n > 8) return fail(QMOE_EINVAL, "qmoe_set_phase_events: need 6..8 events");
    for (int i = 0; i < n; ++i) qmoe::g_phase[i] = (cudaEvent_t)events[i];
    qmoe::g_n_phase = n;
    return QMOE_OK;
}

extern "C" int qmoe_check_status(void* stream) {
    qmoe::clear_error();
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return qmoe::cuda_check(e, "qmoe_check_status");
    const int a = qmoe::dict_take_error();
    const int b = qmoe::rvq_take_error();
    const int c = qmoe::pack_take_error();
    if (a == QMOE_ECUDA || b == QMOE_ECUDA || c == QMOE_ECUDA)
        return fail(QMOE_ECUDA, "qmoe_check_status: reading the error word failed");
    if (a) return fail(a, "device reported an error (dictionary kernels)");
    if (b) return fail(b, "device reported an error (RVQ kernels)");
    if (c) return fail(c, "device reported an error (device encoder)");
    return QMOE_OK;
}

// ---------------------------------------------------------------------------
// qmoe_moe_layer_noalloc: the MoE layer with its scratch in a static device array.
//
// Some callers cannot allocate device memory at all: code hosted inside
// another framework that owns every byte of device memory through its own
// pool, or a serving loop that forbids cudaMalloc/cudaFree after start-up
// because they can synchronise the device and stall every stream.  For them
// this entry point takes its scratch from g_noalloc_scratch, a file-scope
// device array of kNoAllocScratchBytes that every GPU loading this library
// holds until the process exits.  The caller still provides inputs and
// outputs.  The array's address is looked up once per device and context
// (with that device current) on the first call made there, and again after a
// device reset; that first call should come before any stream capture.  All calls share the array: calls whose work
// overlaps on the GPU (different streams, or different host threads) race on
// it and must be serialised by the caller.  Nothing in the scratch has to
// start at zero: every byte a call reads was written earlier in the same call.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
std::mutex g_noalloc_mu;
struct NoAllocAddr {
    void* ctx;
    void* ptr;
};
NoAllocAddr g_noalloc_addr[64];
}  // namespace

extern "C" int qmoe_moe_layer_noalloc(const qmoe_dict* dict, const qmoe_matrix_set* wi, const qmoe_matrix_set* wo,
                                      const void* x_bf16, int T, int k, const int32_t* ids, const float* gates,
                                      void* y, int y_is_f32, void* stream) {
    qmoe::clear_error();
    if (!wi || !wo) return fail(QMOE_EINVAL, "qmoe_moe_layer_noalloc: NULL matrix set");
    if (wi->count < 1 || wi->count > kPlanMaxE || wi->cols < 2 || wi->rows < 2 || T < 0 || k < 1 || k > wi->count)
        return fail(QMOE_EINVAL, "qmoe_moe_layer_noalloc: bad sizes (E, d_model, d_ff, T or k)");
    size_t need = 0;
    int rc = qmoe_moe_layer_ws_size(wi->count, wi->cols, wi->rows, T, k, &need);
    if (rc) return fail(rc, "qmoe_moe_layer_noalloc: " + std::string(qmoe_last_error()));
    if (need > kNoAllocScratchBytes)
        return fail(QMOE_ECAPACITY, "qmoe_moe_layer_noalloc: this layer call needs " + std::to_string(need) +
                                        " bytes of scratch; the static scratch holds " +
                                        std::to_string(kNoAllocScratchBytes) +
                                        " (use qmoe_moe_layer with a workspace)");
    int dev = 0;
    rc = qmoe::cuda_check(cudaGetDevice(&dev), "qmoe_moe_layer_noalloc: cudaGetDevice");
    if (rc) return rc;
    if (dev < 0 || dev >= 64) return fail(QMOE_EUNSUPPORTED, "qmoe_moe_layer_noalloc: device index above 63");
    // the array's device address, looked up once per device and context (a device reset or a
    // caller-created context gets its own lookup)
    void* const ctx = qmoe::current_context();
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        NoAllocAddr& c = g_noalloc_addr[dev];
        if (!c.ptr || !ctx || c.ctx != ctx) {
            void* p = nullptr;
            rc = qmoe::cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                                  "qmoe_moe_layer_noalloc: cudaGetSymbolAddress");
            if (rc) return rc;
            c.ctx = ctx;
            c.ptr = p;
        }
        ptr = c.ptr;
    }
    return qmoe_moe_layer(dict, wi, wo, x_bf16, T, k, ids, gates, y, y_is_f32, ptr, kNoAllocScratchBytes, stream);
}
