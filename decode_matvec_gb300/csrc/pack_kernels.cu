// On-device dictionary encoder: the greedy longest-match encoding of the QMoE
// paper-summary page ("Encoding (compression time)") run on the GPU, with the
// same output as the host encoder qmoe_pack, bit for bit.
//
// The host encoder walks a trie of the dictionary.  Here the dictionary is a
// hash table keyed by the canonical 64-bit entry (both words, pair count in
// bits [3:0] of each, unused symbol fields zero), built in the caller's
// workspace on every call.  One thread encodes one (row, block): at each
// position it builds the key of the next min(14, remaining pairs) pairs and
// probes the table for the longest prefix that is an entry, shortening the
// key one pair at a time; the first hit is the greedy choice.  A first pass
// writes each block's codewords to a per-block scratch slot and its count; an
// exclusive scan of the counts gives the block offsets; a last pass copies
// the codewords into place.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "device_common.cuh"

namespace {

__device__ int g_pack_error;

__device__ __forceinline__ void pack_set_error(int code) { atomicCAS(&g_pack_error, 0, code); }

constexpr int kHashBits = 18;                       // 2^18 slots for 2^16 entries (load 1/4)
constexpr uint32_t kHashSlots = 1u << kHashBits;
constexpr uint32_t kNoCode = 0xFFFFFFFFu;
constexpr int kScanThreads = 1024;

__device__ __forceinline__ uint32_t hash_key(uint64_t k) {
    k ^= k >> 33;
    k *= 0xFF51AFD7ED558CCDull;
    k ^= k >> 33;
    return (uint32_t)k & (kHashSlots - 1u);
}

// Symbols 0..2p-1 of the two words with the pair count p in bits [3:0] of both.
__device__ __forceinline__ uint64_t prefix_key(uint32_t w0, uint32_t w1, int p) {
    const int n = 2 * p;                                          // symbols kept
    const uint32_t m0 = n >= 14 ? 0xFFFFFFF0u : ((1u << (2 * n)) - 1u) << 4;
    const uint32_t m1 = n <= 14 ? 0u : ((1u << (2 * (n - 14))) - 1u) << 4;
    return (uint64_t)((w0 & m0) | (uint32_t)p) | ((uint64_t)((w1 & m1) | (uint32_t)p) << 32);
}

__global__ void hash_clear_kernel(unsigned long long* keys, uint32_t* codes) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < kHashSlots) {
        keys[i] = 0ull;
        codes[i] = kNoCode;
    }
}

// Inserts every entry; an entry that repeats an earlier one keeps the smaller
// codeword (the host trie keeps the first).
__global__ void hash_build_kernel(const uint32_t* __restrict__ words, unsigned long long* keys, uint32_t* codes) {
    const uint32_t e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= QMOE_DICT_ENTRIES) return;
    const uint32_t w0 = words[2 * e], w1 = words[2 * e + 1];
    const int p = (int)(w0 & 15u);
    if ((int)(w1 & 15u) != p || p < 1 || p > 14) {
        pack_set_error(QMOE_EFORMAT);
        return;
    }
    for (int i = 0; i < 2 * p; ++i) {
        if ((((i < 14 ? w0 : w1) >> (4 + 2 * (i % 14))) & 3u) == 3u) {
            pack_set_error(QMOE_EFORMAT);
            return;
        }
    }
    const uint64_t key = prefix_key(w0, w1, p);
    uint32_t h = hash_key(key);
    for (uint32_t probe = 0; probe < kHashSlots; ++probe) {
        const unsigned long long old = atomicCAS(keys + h, 0ull, (unsigned long long)key);
        if (old == 0ull || old == key) {
            atomicMin(codes + h, e);
            return;
        }
        h = (h + 1u) & (kHashSlots - 1u);
    }
    pack_set_error(QMOE_ECAPACITY);
}

__device__ __forceinline__ uint32_t hash_find(const unsigned long long* __restrict__ keys,
                                              const uint32_t* __restrict__ codes, uint64_t key) {
    uint32_t h = hash_key(key);
    for (uint32_t probe = 0; probe < kHashSlots; ++probe) {
        const unsigned long long k = __ldg(keys + h);
        if (k == key) return __ldg(codes + h);
        if (k == 0ull) return kNoCode;
        h = (h + 1u) & (kHashSlots - 1u);
    }
    return kNoCode;
}

// Symbol of a weight: 0 -> 0, -1 -> 1 (w_min), +1 -> 2 (w_max); 3 = invalid.
__device__ __forceinline__ uint32_t symbol_of(int8_t v) { return v == 0 ? 0u : v == -1 ? 1u : v == 1 ? 2u : 3u; }

// Pass 1: one thread per (row, block) encodes into its scratch slot of
// block/2 codewords and records the count.
__global__ void encode_blocks_kernel(const int8_t* __restrict__ tern, int rows, int cols, int block, int nb,
                                     const unsigned long long* __restrict__ keys,
                                     const uint32_t* __restrict__ codes_tab, uint16_t* __restrict__ scratch,
                                     uint32_t* __restrict__ counts) {
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t >= (long long)rows * nb) return;
    const int r = (int)(t / nb), b = (int)(t - (long long)r * nb);
    const int8_t* row = tern + (size_t)r * cols;
    const int c_end = min(cols, (b + 1) * block);
    uint16_t* out = scratch + (size_t)t * (block / 2);
    int pos = b * block;
    uint32_t n = 0;
    while (pos < c_end) {
        // symbols of the next up to 14 pairs
        const int pmax = min(14, (c_end - pos) / 2);
        uint32_t w0 = 0, w1 = 0;
        bool bad = false;
        for (int i = 0; i < 2 * pmax; ++i) {
            const uint32_t s = symbol_of(row[pos + i]);
            bad |= s == 3u;
            if (i < 14) w0 |= s << (4 + 2 * i);
            else w1 |= s << (4 + 2 * (i - 14));
        }
        if (bad) {
            pack_set_error(QMOE_EINVAL);
            break;
        }
        uint32_t code = kNoCode;
        int p = pmax;
        for (; p >= 1; --p) {
            code = hash_find(keys, codes_tab, prefix_key(w0, w1, p));
            if (code != kNoCode) break;
        }
        if (code == kNoCode) {
            pack_set_error(QMOE_EFORMAT);
            break;
        }
        out[n++] = (uint16_t)code;
        pos += 2 * p;
    }
    counts[t] = n;
}

// Exclusive scan of n counts in three passes: per-block sums, a scan of the
// block sums in one block, then per-block scans plus their base.
__device__ __forceinline__ unsigned long long block_scan_excl(unsigned long long v, unsigned long long* sh,
                                                              unsigned long long& total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(QMOE_FULL_MASK, x, d);
        if (lane >= d) x += o;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned long long y = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0ull;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long o = __shfl_up_sync(QMOE_FULL_MASK, y, d);
            if (lane >= d) y += o;
        }
        sh[lane] = y;
    }
    __syncthreads();
    const unsigned long long before = (warp > 0 ? sh[warp - 1] : 0ull) + x - v;
    total = sh[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kScanThreads) scan_sums_kernel(const uint32_t* __restrict__ counts, long long n,
                                                                 unsigned long long* __restrict__ sums) {
    __shared__ unsigned long long sh[32];
    const long long i = blockIdx.x * (long long)kScanThreads + threadIdx.x;
    unsigned long long total;
    block_scan_excl(i < n ? counts[i] : 0u, sh, total);
    if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) scan_base_kernel(unsigned long long* sums, int nblk) {
    __shared__ unsigned long long sh[32];
    __shared__ unsigned long long carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < nblk; base += kScanThreads) {
        const int i = base + threadIdx.x;
        const unsigned long long v = i < nblk ? sums[i] : 0ull;
        unsigned long long total;
        const unsigned long long ex = block_scan_excl(v, sh, total);
        if (i < nblk) sums[i] = carry + ex;
        __syncthreads();
        if (threadIdx.x == 0) carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) sums[nblk] = carry;
}

__global__ void __launch_bounds__(kScanThreads) scan_apply_kernel(const uint32_t* __restrict__ counts, long long n,
                                                                  const unsigned long long* __restrict__ sums,
                                                                  int nblk, uint32_t* __restrict__ blk_off) {
    __shared__ unsigned long long sh[32];
    const long long i = blockIdx.x * (long long)kScanThreads + threadIdx.x;
    unsigned long long total;
    const unsigned long long ex = block_scan_excl(i < n ? counts[i] : 0u, sh, total);
    const unsigned long long v = sums[blockIdx.x] + ex;
    if (v > 0xFFFFFFFFull) pack_set_error(QMOE_EINVAL);
    if (i < n) blk_off[i] = (uint32_t)v;
    if (i == 0) {
        const unsigned long long all = sums[nblk];
        if (all > 0xFFFFFFFFull) pack_set_error(QMOE_EINVAL);
        blk_off[n] = (uint32_t)all;
    }
}

// Pass 3: copy each block's codewords to its offset (those past codes_cap are
// dropped and reported as QMOE_ECAPACITY).
__global__ void place_kernel(const uint16_t* __restrict__ scratch, const uint32_t* __restrict__ counts,
                             const uint32_t* __restrict__ blk_off, long long n, int half_block,
                             uint16_t* __restrict__ codes, unsigned long long codes_cap) {
    const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t >= n) return;
    const uint32_t c = counts[t];
    const unsigned long long o = blk_off[t];
    if (o + c > codes_cap) pack_set_error(QMOE_ECAPACITY);
    const uint16_t* src = scratch + (size_t)t * half_block;
    for (uint32_t i = 0; i < c; ++i)
        if (o + i < codes_cap) codes[o + i] = src[i];
}

struct PackWs {
    unsigned long long* keys;
    uint32_t* codes_tab;
    uint32_t* counts;
    unsigned long long* sums;
    uint16_t* scratch;
    size_t bytes;
};

size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

PackWs pack_ws_layout(void* base, int rows, int cols, int block) {
    PackWs w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        void* p = base ? (void*)((char*)base + off) : nullptr;
        off += align256(bytes);
        return p;
    };
    const long long nb = (cols + block - 1) / block;
    const long long n = (long long)rows * nb;
    const long long nblk = (n + kScanThreads - 1) / kScanThreads;
    w.keys = (unsigned long long*)take(sizeof(unsigned long long) * kHashSlots);
    w.codes_tab = (uint32_t*)take(sizeof(uint32_t) * kHashSlots);
    w.counts = (uint32_t*)take(sizeof(uint32_t) * std::max(1LL, n));
    w.sums = (unsigned long long*)take(sizeof(unsigned long long) * (nblk + 1));
    w.scratch = (uint16_t*)take(sizeof(uint16_t) * std::max(1LL, n) * (block / 2));
    w.bytes = off;
    return w;
}

bool pack_shape_ok(int rows, int cols, int block) {
    return rows >= 0 && cols > 0 && (cols % 2) == 0 && block > 0 && (block % 2) == 0;
}

}  // namespace

namespace qmoe {
int pack_take_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pack_error, sizeof(int)) != cudaSuccess) return QMOE_ECUDA;
    const int z = 0;
    if (cudaMemcpyToSymbol(g_pack_error, &z, sizeof(int)) != cudaSuccess) return QMOE_ECUDA;
    return v;
}
}  // namespace qmoe

extern "C" int qmoe_pack_device_ws_size(int rows, int cols, int block, size_t* bytes) {
    qmoe::clear_error();
    if (!bytes || !pack_shape_ok(rows, cols, block))
        return qmoe::fail(QMOE_EINVAL, "qmoe_pack_device_ws_size: rows >= 0, cols > 0 even, block > 0 even");
    *bytes = pack_ws_layout(nullptr, rows, cols, block).bytes;
    return QMOE_OK;
}

extern "C" int qmoe_pack_device(const qmoe_dict* dict, const int8_t* tern, int rows, int cols, int block,
                                uint16_t* codes, size_t codes_cap, uint32_t* blk_off, void* workspace,
                                size_t ws_bytes, void* stream) {
    qmoe::clear_error();
    if (!dict || !dict->words) return qmoe::fail(QMOE_EINVAL, "qmoe_pack_device: dictionary is NULL");
    if (!pack_shape_ok(rows, cols, block))
        return qmoe::fail(QMOE_EINVAL, "qmoe_pack_device: rows >= 0, cols > 0 even, block > 0 even");
    if (!blk_off || !workspace || (rows > 0 && (!tern || !codes)))
        return qmoe::fail(QMOE_EINVAL, "qmoe_pack_device: NULL pointer");
    const PackWs w = pack_ws_layout(workspace, rows, cols, block);
    if (ws_bytes < w.bytes) return qmoe::fail(QMOE_ECAPACITY, "qmoe_pack_device: workspace too small");
    cudaStream_t st = (cudaStream_t)stream;
    const long long nb = (cols + block - 1) / block;
    const long long n = (long long)rows * nb;
    const long long nblk = (n + kScanThreads - 1) / kScanThreads;
    if (nblk > 0x7FFFFFFFLL) return qmoe::fail(QMOE_EINVAL, "qmoe_pack_device: matrix too large");
    hash_clear_kernel<<<kHashSlots / 256, 256, 0, st>>>(w.keys, w.codes_tab);
    hash_build_kernel<<<QMOE_DICT_ENTRIES / 256, 256, 0, st>>>(dict->words, w.keys, w.codes_tab);
    int rc = qmoe::launch_check("qmoe_pack_device: dictionary table");
    if (rc) return rc;
    if (n > 0) {
        encode_blocks_kernel<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(tern, rows, cols, block, (int)nb, w.keys,
                                                                          w.codes_tab, w.scratch, w.counts);
        scan_sums_kernel<<<(unsigned)nblk, kScanThreads, 0, st>>>(w.counts, n, w.sums);
        scan_base_kernel<<<1, kScanThreads, 0, st>>>(w.sums, (int)nblk);
        scan_apply_kernel<<<(unsigned)nblk, kScanThreads, 0, st>>>(w.counts, n, w.sums, (int)nblk, blk_off);
        place_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w.scratch, w.counts, blk_off, n, block / 2, codes,
                                                                  (unsigned long long)codes_cap);
    } else {
        rc = qmoe::cuda_check(cudaMemsetAsync(blk_off, 0, sizeof(uint32_t), st), "qmoe_pack_device");
        if (rc) return rc;
    }
    return qmoe::launch_check("qmoe_pack_device");
}
