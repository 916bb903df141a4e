// Residual-VQ path: randomized Hadamard transforms and the fused codebook
// decode-and-multiply for sm_103a.
//
// Format ("Quantization as Cache Amplification", section "Codec"): the weight
// is rotated, W' = H_o D_out W D_in H_i, rows of W' carry one fp16 RMS scale,
// and every 8 consecutive weights of a row are coded by two 8-bit indices into
// two 256-entry fp16 codebooks (residual stages).  At run time the rotation is
// applied to the activations, y = D_out H_o (W' (H_i D_in x)) (the page's
// runtime formula; "M8.5" section 0x06H fixes the same sign order), so the
// expert kernel only ever sees codebook indices: it decodes each 8-vector as
// C1[i1] + C2[i2] in registers from shared-memory codebooks and multiplies it
// into the staged rotated activations; the row scale multiplies the
// accumulated dot product once.  The Walsh-Hadamard transforms are in-shared-
// memory butterflies (O(n log n)), one block per activation row (the output
// transform: one block per slot, the slots of a token on one cluster).
//
// The same kernels run the E8P lattice code ("M8.5 - Extreme Weight
// Compression and Representations", 0x06E) when the matrix set's format says
// so: one 16-bit code word per 8 weights, decoded from a 256-entry table of
// absolute patterns with explicit signs, a parity-implied last sign and a
// +-1/4 shift (see e8p_half8).  Frequency-conditioned sets give each matrix
// 1 to 3 residual stages ("Quantization as Cache Amplification",
// Frequency-Conditioned Bit Allocation).

#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "device_common.cuh"

using qmoe::Job;

namespace {

__device__ int g_rvq_error;

struct RvqDev {
    const uint8_t* idx;
    const uint16_t* cb;
    const uint16_t* scale;
    const int8_t* so;
    const int8_t* si;
    int count, rows, cols;
    const uint8_t* stages;     // per matrix stage count, or NULL (2)
    const uint64_t* idx_base;  // per matrix byte offset of its codes, or NULL
    int n_st;                  // codebooks in the set (0 for E8P)
    int e8p;                   // E8P lattice code words instead of codebook indices
};

RvqDev to_dev(const rvq_matrix_set* s) {
    const bool e8p = s->format == QMOE_VQ_E8P;
    return RvqDev{s->idx, s->codebooks, s->scale_f16, s->sign_out, s->sign_in, s->count, s->rows, s->cols,
                  s->stages, s->idx_base, e8p ? 0 : s->n_stages ? s->n_stages : 2, e8p ? 1 : 0};
}

// Stage count of matrix e, or 0 for a count outside 1 .. n_st: that records
// QMOE_EFORMAT, and the kernels then read none of the matrix's codes (its
// layout is unknown) and leave its outputs unwritten (decode: zeros).
__device__ __forceinline__ int stages_of(const RvqDev& m, int e) {
    if (!m.stages) return 2;
    const int st = m.stages[e];
    if (st < 1 || st > m.n_st) {
        atomicCAS(&g_rvq_error, 0, QMOE_EFORMAT);
        return 0;
    }
    return st;
}

// First code byte of matrix e: [rows][cols/8][stages] bytes from here.
__device__ __forceinline__ const uint8_t* codes_of(const RvqDev& m, int e) {
    return m.idx + (m.idx_base ? m.idx_base[e] : (uint64_t)e * m.rows * (m.cols / 8) * 2);
}

bool pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

bool valid_set(const rvq_matrix_set* s) {
    return s && s->idx && s->codebooks && s->scale_f16 && s->sign_out && s->sign_in && s->count >= 1 &&
           pow2(s->rows) && pow2(s->cols) && s->cols >= 8 && s->rows <= 8192 && s->cols <= 8192 &&
           s->n_stages >= 0 && s->n_stages <= QMOE_RVQ_MAX_STAGES && (s->stages || s->n_stages != 1) &&
           (s->format == QMOE_VQ_RVQ || (s->format == QMOE_VQ_E8P && !s->stages && s->n_stages == 0));
}

// ---------------------------------------------------------------- E8P decode
// ("M8.5 - Extreme Weight Compression and Representations", 0x06E.)  The base
// table arrives as 256 words of 8 nibbles 2|a_j|; shared memory holds it as
// 8 bytes per pattern (byte j = 2|a_j|), replicated so that the lanes of a
// warp read different banks.  A code word's 8 coordinates come out as four
// exact fp16 pairs: a byte permute puts 2|a_j| under the fp16 exponent of
// 1024 (the value 1024 + 2|a_j|), one fp16x2 multiply-add makes |a_j|, the
// sign bits are spread onto the two halves' sign bits with one multiply, and
// one fp16x2 add applies the +-1/4 shift.  Every coordinate is a multiple of
// 1/4 below 3, so every step is exact.
constexpr int kE8pRepGemm = 16;   // table replicas in rvq_gemm_kernel (8-byte entries: 16 bank pairs)
constexpr int kE8pRepTc = 4;      // table replicas in rvq_tc_kernel

__device__ __forceinline__ uint2 e8p_bytes(uint32_t w) {
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        lo |= ((w >> (4 * j)) & 15u) << (8 * j);
        hi |= ((w >> (16 + 4 * j)) & 15u) << (8 * j);
    }
    return make_uint2(lo, hi);
}

// table[p * kRep + r] = pattern p's bytes, r = 0 .. kRep-1, by a block of kThreads threads (all
// call it); the loads are issued together.
template <int kRep, int kThreads>
__device__ __forceinline__ void e8p_stage_table(const uint32_t* __restrict__ g, uint2* t) {
    constexpr int kPer = 256 * kRep / kThreads;
    static_assert(kPer * kThreads == 256 * kRep, "table entries per thread");
    uint32_t w[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) w[j] = __ldg(g + (threadIdx.x + j * kThreads) / kRep);
#pragma unroll
    for (int j = 0; j < kPer; ++j) t[threadIdx.x + j * kThreads] = e8p_bytes(w[j]);
}

// Codebooks [n_st][256] x 16 bytes into shared memory by 256 threads, the loads issued together.
__device__ __forceinline__ void rvq_stage_codebooks(const uint4* __restrict__ g, uint4* t, int n_st) {
    uint4 c[QMOE_RVQ_MAX_STAGES];
#pragma unroll
    for (int j = 0; j < QMOE_RVQ_MAX_STAGES; ++j) c[j] = j < n_st ? __ldg(g + threadIdx.x + j * 256) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < QMOE_RVQ_MAX_STAGES; ++j)
        if (j < n_st) t[threadIdx.x + j * 256] = c[j];
}

__device__ __forceinline__ void e8p_half8(uint2 pb, uint32_t code, uint32_t (&h)[4]) {
    // sum_j 2|a_j| = 2 sum_j |a_j|; coordinate 7 is negative when the explicit negatives
    // leave sum_j s_j |a_j| odd
    const uint32_t two_sum = __dp4a(pb.x, 0x01010101u, __dp4a(pb.y, 0x01010101u, 0u));
    const uint32_t sg = (code >> 8) & 127u;
    const uint32_t neg = sg | ((((two_sum >> 1) + (uint32_t)__popc(sg)) & 1u) << 7);
    const uint32_t c2 = (code & 0x8000u) ? 0x34003400u : 0xB400B400u;   // (+1/4, +1/4) or (-1/4, -1/4)
    const __half2 half = __floats2half2_rn(0.5f, 0.5f), m512 = __floats2half2_rn(-512.0f, -512.0f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t src = q < 2 ? pb.x : pb.y;
        // fp16 lanes 0x64nn = 1024 + n: bytes (n_2q, 0x64, n_2q+1, 0x64), 0x64 from byte 1 / 3 of the constant
        const uint32_t sel = (uint32_t)((2 * q) & 3) | (5u << 4) | ((uint32_t)((2 * q + 1) & 3) << 8) | (7u << 12);
        const uint32_t m = __byte_perm(src, 0x64006400u, sel);
        const __half2 a = __hfma2(*reinterpret_cast<const __half2*>(&m), half, m512);
        // (y * 0x40008000) & 0x80008000 moves bit 0 of y to bit 15 and bit 1 to bit 31
        const uint32_t sm = ((neg >> (2 * q)) * 0x40008000u) & 0x80008000u;
        const uint32_t sa = *reinterpret_cast<const uint32_t*>(&a) ^ sm;
        const __half2 v = __hadd2(*reinterpret_cast<const __half2*>(&sa), *reinterpret_cast<const __half2*>(&c2));
        h[q] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

__device__ __forceinline__ void e8p_float8(uint2 pb, uint32_t code, float (&w)[8]) {
    uint32_t h[4];
    e8p_half8(pb, code, h);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
        w[2 * q] = f.x;
        w[2 * q + 1] = f.y;
    }
}

// Normalised Walsh-Hadamard transform of n floats in shared memory, in place.
// Every thread of the block must call it.
__device__ void fwht_smem(float* s, int n, float norm) {
    for (int h = 1; h < n; h <<= 1) {
        for (int b = threadIdx.x; b < (n >> 1); b += blockDim.x) {
            const int i = ((b & ~(h - 1)) << 1) | (b & (h - 1));
            const float a = s[i], c = s[i + h];
            s[i] = a + c;
            s[i + h] = a - c;
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) s[i] *= norm;
    __syncthreads();
}

// `count` normalised Walsh-Hadamard transforms of n floats each, stored back
// to back in shared memory, in place: every butterfly stage of all of them
// between the same two barriers.  Every thread of the block must call it.
__device__ void fwht_smem_batch(float* s, int n, int count, float norm) {
    const int half = n >> 1, lg = 31 - __clz(half);
    for (int h = 1; h < n; h <<= 1) {
        for (int b = threadIdx.x; b < count * half; b += blockDim.x) {
            const int c = b >> lg, bb = b & (half - 1);
            const int i = c * n + (((bb & ~(h - 1)) << 1) | (bb & (h - 1)));
            const float a = s[i], d = s[i + h];
            s[i] = a + d;
            s[i + h] = a - d;
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < count * n; i += blockDim.x) s[i] *= norm;
    __syncthreads();
}

// Staging scale of one rotated activation row for the tensor-core kernel, which
// splits each value into an fp16 high part and the fp16 of the remainder: the
// power of two 2^k that brings the row's largest magnitude into [2^14, 2^15).
// Both parts then stay inside fp16's range (|v| < 65504 after scaling), and a
// value loses low bits only when it is below 2^-25 of the row's largest one.
// Multiplying by 2^k is exact in fp32, so the kernel's output, divided by 2^k
// again, is what an unbounded split would give.  An all-zero (or non-finite)
// row keeps 1.  k is kept inside [-126, 126], where 2^k and 2^-k are normal.
__device__ __forceinline__ float stage_scale_of_max(float mx) {
    if (!(mx > 0.0f) || !(mx <= 3.402823466e38f)) return 1.0f;
    int ex;
    frexpf(mx, &ex);                                   // mx = f * 2^ex, f in [0.5, 1)
    const int k = max(-126, min(126, 15 - ex));
    return __int_as_float((127 + k) << 23);
}

// Largest |v| over a block's values (every thread passes its own maximum); red: 32 floats.
__device__ __forceinline__ float block_max_abs(float v, float* red) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(QMOE_FULL_MASK, v, d));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();                                   // red may still be read by an earlier call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
    return r;
}

// x'[row] = H (D_in x[src]) for one or two sign vectors (gate and up share the input).
__global__ void in_transform_kernel(const uint16_t* __restrict__ x, int x_div, const int32_t* __restrict__ expert_of,
                                    int k_of, const int8_t* __restrict__ si0, const int8_t* __restrict__ si1, int n,
                                    float norm, float* __restrict__ out0, float* __restrict__ out1,
                                    float* __restrict__ sc0, float* __restrict__ sc1) {
    __shared__ float red[32];
    extern __shared__ float sm[];
    const int row = blockIdx.x;
    const int e = expert_of ? expert_of[row] : 0;
    const uint16_t* src = x + (size_t)(row / x_div) * n;
    float* s0 = sm;
    float* s1 = sm + n;
#pragma unroll 4
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = bf16_to_f32(src[i]);
        s0[i] = v * (float)si0[(size_t)e * n + i];
        if (si1) s1[i] = v * (float)si1[(size_t)e * n + i];
    }
    __syncthreads();
    fwht_smem_batch(s0, n, si1 ? 2 : 1, norm);
    float m0 = 0.0f, m1 = 0.0f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        out0[(size_t)row * n + i] = s0[i];
        m0 = fmaxf(m0, fabsf(s0[i]));
        if (si1) {
            out1[(size_t)row * n + i] = s1[i];
            m1 = fmaxf(m1, fabsf(s1[i]));
        }
    }
    if (sc0) {
        const float a0 = block_max_abs(m0, red);
        if (threadIdx.x == 0) sc0[row] = stage_scale_of_max(a0);
        if (sc1 && si1) {
            const float a1 = block_max_abs(m1, red);
            if (threadIdx.x == 0) sc1[row] = stage_scale_of_max(a1);
        }
    }
    (void)k_of;
}

// h = bf16(silu(g) * u) with g = D_out,g H g', u = D_out,u H u'; then the down
// matrix's input transform h' = H (D_in,down h).
__global__ void swiglu_transform_kernel(const float* __restrict__ gp, const float* __restrict__ up,
                                        const int32_t* __restrict__ expert_of, const int8_t* __restrict__ so_g,
                                        const int8_t* __restrict__ so_u, const int8_t* __restrict__ si_d, int n,
                                        float norm, float* __restrict__ out, float* __restrict__ sc) {
    __shared__ float red[32];
    extern __shared__ float sm[];
    const int row = blockIdx.x;
    const int e = expert_of[row];
    float* sg = sm;
    float* su = sm + n;
#pragma unroll 4
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        sg[i] = gp[(size_t)row * n + i];
        su[i] = up[(size_t)row * n + i];
    }
    __syncthreads();
    fwht_smem_batch(sg, n, 2, norm);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float g = sg[i] * (float)so_g[(size_t)e * n + i];
        const float u = su[i] * (float)so_u[(size_t)e * n + i];
        const float silu = g / (1.0f + expf(-g));
        const float h = bf16_to_f32(f32_to_bf16(silu * u));
        sg[i] = h * (float)si_d[(size_t)e * n + i];
    }
    __syncthreads();
    fwht_smem(sg, n, norm);
    float mx = 0.0f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        out[(size_t)row * n + i] = sg[i];
        mx = fmaxf(mx, fabsf(sg[i]));
    }
    if (sc) {
        const float a = block_max_abs(mx, red);
        if (threadIdx.x == 0) sc[row] = stage_scale_of_max(a);
    }
}

// y[t] = sum_j gate[t][j] * D_out H y'[t*k + j]  (k == 1 and gates == NULL: plain output transform).
// The slots of a token are transformed kg at a time (kg * n floats of shared
// memory, plus n for the sum).
__global__ void out_transform_kernel(const float* __restrict__ yp, const int32_t* __restrict__ expert_of,
                                     const int8_t* __restrict__ so, const float* __restrict__ gates, int k, int kg,
                                     int n, float norm, void* __restrict__ y, int y_is_f32) {
    extern __shared__ float sm[];
    float* acc = sm + (size_t)kg * n;
    const int t = blockIdx.x;
    for (int i = threadIdx.x; i < n; i += blockDim.x) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += kg) {
        const int cnt = min(kg, k - j0);
        __syncthreads();                                  // the previous group is consumed
        for (int i = threadIdx.x; i < cnt * n; i += blockDim.x) sm[i] = yp[((size_t)t * k + j0) * n + i];
        __syncthreads();
        fwht_smem_batch(sm, n, cnt, norm);
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            float a = acc[i];
            for (int j = 0; j < cnt; ++j) {
                const int slot = t * k + j0 + j;
                const int e = expert_of ? expert_of[slot] : 0;
                const float g = gates ? gates[slot] : 1.0f;
                a = fmaf(g, sm[(size_t)j * n + i] * (float)so[(size_t)e * n + i], a);
            }
            acc[i] = a;                                   // the same thread reads it back
        }
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (y_is_f32) ((float*)y)[(size_t)t * n + i] = acc[i];
        else ((uint16_t*)y)[(size_t)t * n + i] = f32_to_bf16(acc[i]);
    }
}

// The same output transform with the k slots of a token on the k CTAs of one thread-block cluster
// (2 <= k <= 8): CTA j transforms slot j in its own shared memory and multiplies by D_out; after a
// cluster barrier CTA j sums columns [j n / k, (j+1) n / k) over the slots in slot order, reading
// the other CTAs' shared memory, with the per-element arithmetic of out_transform_kernel.
__global__ void out_transform_cluster_kernel(const float* __restrict__ yp, const int32_t* __restrict__ expert_of,
                                             const int8_t* __restrict__ so, const float* __restrict__ gates, int k,
                                             int n, float norm, void* __restrict__ y, int y_is_f32) {
    extern __shared__ float sm[];
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int j = (int)cluster.block_rank();
    const int t = blockIdx.x / k;
    const int slot = t * k + j;
#pragma unroll 4
    for (int i = threadIdx.x; i < n; i += blockDim.x) sm[i] = yp[(size_t)slot * n + i];
    __syncthreads();
    fwht_smem(sm, n, norm);
    const int e = expert_of ? expert_of[slot] : 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) sm[i] = sm[i] * (float)so[(size_t)e * n + i];
    cluster.sync();
    const int c0 = (int)((long long)j * n / k), c1 = (int)((long long)(j + 1) * n / k);
    for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
        float a = 0.0f;
        for (int q = 0; q < k; ++q) {
            const float* peer = cluster.map_shared_rank(sm, q);
            a = fmaf(gates ? gates[t * k + q] : 1.0f, peer[i], a);
        }
        if (y_is_f32) ((float*)y)[(size_t)t * n + i] = a;
        else ((uint16_t*)y)[(size_t)t * n + i] = f32_to_bf16(a);
    }
    cluster.sync();                                       // peers may still read this block's memory
}

// ---------------------------------------------------------------- decode-multiply (CUDA cores)
struct RvqGemmArgs {
    RvqDev m;
    const float* xr;      // rotated activations, fp32 [slot][cols]
    const float* xs;      // per-slot power-of-two staging scale of xr for the tensor-core kernel
    const Job* jobs;
    const int* n_jobs_dev;
    const int* slots;
    int T_implicit;
    int nt_max;
    int rows_per_tile;
    int row_tiles;
    float* out;           // rotated outputs, fp32 [slot][rows]
};

// w = C1 (+ C2 (+ C3)) of one 8-weight vector, fp32 adds left to right.
template <int S>
__device__ __forceinline__ void decode_vec(const uint4* cb, const uint32_t (&code)[S], float (&w)[8]) {
    const uint4 c1 = cb[code[0]];
    const uint32_t a[4] = {c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&a[q]));
        w[2 * q] = f.x;
        w[2 * q + 1] = f.y;
    }
#pragma unroll
    for (int st = 1; st < S; ++st) {
        const uint4 c = cb[256 * st + code[st]];
        const uint32_t b[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&b[q]));
            w[2 * q] = w[2 * q] + f.x;
            w[2 * q + 1] = w[2 * q + 1] + f.y;
        }
    }
}

// vectors a lane loads ahead: 8 (a whole row for cols <= 2048) for one token with one or two
// stages, 2 for eight tokens, else 4 (the accumulators and codes share 128 registers)
__host__ __device__ constexpr int rvq_batch(int nt, int s) { return nt == 1 && s < 3 ? 8 : nt == 8 ? 2 : 4; }

// E8: the codes are E8P code words (S = 2 bytes each) and scb holds the staged E8P table.
// The codes of kB vectors v0, v0 + 32, ... of one row (ip = the row's first code byte); 0 past nv.
template <int S, bool E8, int kB>
__device__ __forceinline__ void rvq_load_codes(const uint8_t* ip, int nv, int v0, uint32_t (&dst)[kB][E8 ? 1 : S]) {
#pragma unroll
    for (int u = 0; u < kB; ++u) {
        const int v = v0 + 32 * u;
        if constexpr (E8 || S == 2) {
            dst[u][0] = v < nv ? __ldg((const uint16_t*)ip + v) : 0u;
        } else {
#pragma unroll
            for (int st = 0; st < S; ++st) dst[u][st] = v < nv ? __ldg(ip + (size_t)v * S + st) : 0u;
        }
    }
}

// One vector's 8 decoded weights from its loaded code word(s).
template <int S, bool E8>
__device__ __forceinline__ void rvq_decode_one(const uint4* scb, const uint32_t (&cw)[E8 ? 1 : S], int lane,
                                               float (&w)[8]) {
    if constexpr (E8) {
        e8p_float8(((const uint2*)scb)[(cw[0] & 255u) * kE8pRepGemm + (lane & (kE8pRepGemm - 1))], cw[0], w);
    } else {
        uint32_t code[S];
        if constexpr (S == 2) {
            code[0] = cw[0] & 255u;
            code[1] = cw[0] >> 8;
        } else {
#pragma unroll
            for (int st = 0; st < S; ++st) code[st] = cw[st];
        }
        decode_vec<S>(scb, code, w);
    }
}

// acc[t] += w . x_t over the vector's 8 columns (activations staged [token][column]).
template <int NT>
__device__ __forceinline__ void rvq_fma_tokens(const float* xs, int cols, int v, const float (&w)[8], float (&acc)[NT]) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float4* xt = (const float4*)(xs + (size_t)t * cols) + 2 * v;
        const float4 x0 = xt[0], x1 = xt[1];
        acc[t] = fmaf(w[0], x0.x, acc[t]);
        acc[t] = fmaf(w[1], x0.y, acc[t]);
        acc[t] = fmaf(w[2], x0.z, acc[t]);
        acc[t] = fmaf(w[3], x0.w, acc[t]);
        acc[t] = fmaf(w[4], x1.x, acc[t]);
        acc[t] = fmaf(w[5], x1.y, acc[t]);
        acc[t] = fmaf(w[6], x1.z, acc[t]);
        acc[t] = fmaf(w[7], x1.w, acc[t]);
    }
}

template <int NT, int S, bool E8 = false>
__device__ void rvq_tile_rows(const RvqGemmArgs& a, const uint4* scb, const float* xs, const Job& job, int r0,
                              int warp, int nwarps, int lane) {
    const RvqDev& m = a.m;
    const int nv = m.cols / 8;
    const int r1 = min(m.rows, r0 + a.rows_per_tile);
    const uint8_t* codes = codes_of(m, job.matrix);
    for (int r = r0 + warp; r < r1; r += nwarps) {
        const uint8_t* ip = codes + (size_t)r * nv * S;
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
        // up to kRvqBatch vectors per lane: all their code loads are issued before the first decode
        constexpr int kRvqBatch = rvq_batch(NT, S);
        for (int v0 = lane; v0 < nv; v0 += 32 * kRvqBatch) {
            uint32_t cwb[kRvqBatch][E8 ? 1 : S];
#pragma unroll
            for (int u = 0; u < kRvqBatch; ++u) {
                const int v = v0 + 32 * u;
                if constexpr (E8 || S == 2) {
                    cwb[u][0] = v < nv ? __ldg((const uint16_t*)ip + v) : 0u;
                } else {
#pragma unroll
                    for (int st = 0; st < S; ++st) cwb[u][st] = v < nv ? __ldg(ip + (size_t)v * S + st) : 0u;
                }
            }
#pragma unroll
            for (int u = 0; u < kRvqBatch; ++u) {
                const int v = v0 + 32 * u;
                if (v >= nv) break;
                float w[8];
                rvq_decode_one<S, E8>(scb, cwb[u], lane, w);
                rvq_fma_tokens<NT>(xs, m.cols, v, w, acc);
            }
        }
        const float s = f16_to_f32(m.scale[(size_t)job.matrix * m.rows + r]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float v = warp_sum(acc[t]);
            if (lane == t && t < job.n_tok) {
                const int slot = a.slots ? a.slots[job.slot_begin + t] : job.slot_begin + t;
                a.out[(size_t)slot * m.rows + r] = s * v;
            }
        }
    }
}

constexpr int kRvqThreads = 256;

// The job's activation rows [token][column] into shared memory (zeros past its tokens); rows are
// copied as float4, two per thread at a time with the loads issued together (a 2048-column row
// in one round trip).
template <int NT>
__device__ void rvq_stage(const RvqGemmArgs& a, const Job& job, float* xs) {
    const int n4 = a.m.cols / 4;
    for (int t = 0; t < NT; ++t) {
        const int slot = t >= job.n_tok ? -1 : a.slots ? a.slots[job.slot_begin + t] : job.slot_begin + t;
        const float4* src = (const float4*)(a.xr + (size_t)(slot < 0 ? 0 : slot) * a.m.cols);
        float4* dst = (float4*)(xs + (size_t)t * a.m.cols);
        for (int c0 = threadIdx.x; c0 < n4; c0 += 2 * blockDim.x) {
            float4 v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int c = c0 + u * blockDim.x;
                v[u] = slot >= 0 && c < n4 ? src[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (c0 + u * blockDim.x < n4) dst[c0 + u * blockDim.x] = v[u];
        }
    }
}

// two blocks per SM (the launch grid): up to 128 registers a thread
__global__ void __launch_bounds__(kRvqThreads, 2) rvq_gemm_kernel(const RvqGemmArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint4* scb = (uint4*)smem;                  // [n_st][256] x 8 fp16, or the replicated E8P table
    float* xs = (float*)(smem + (a.m.e8p ? (size_t)256 * kE8pRepGemm * 8 : (size_t)a.m.n_st * 256 * 16));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    if (a.m.e8p) e8p_stage_table<kE8pRepGemm, kRvqThreads>((const uint32_t*)a.m.cb, (uint2*)smem);
    else rvq_stage_codebooks((const uint4*)a.m.cb, scb, a.m.n_st);
    __syncthreads();
    const int n_jobs = a.jobs ? *a.n_jobs_dev : (a.T_implicit + a.nt_max - 1) / a.nt_max;
    const int n_tiles = n_jobs * a.row_tiles;
    // each block takes a contiguous range of tiles: consecutive row ranges of one job reuse the
    // staged activations
    const int per_block = (n_tiles + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per_block, t_end = min(n_tiles, t_begin + per_block);
    int staged = -1;
    for (int tile = t_begin; tile < t_end; ++tile) {
        Job job;
        const int j = tile / a.row_tiles;
        if (a.jobs) {
            job = a.jobs[j];
        } else {
            job.matrix = 0;
            job.slot_begin = j * a.nt_max;
            job.n_tok = min(a.nt_max, a.T_implicit - j * a.nt_max);
        }
        const int r0 = (tile % a.row_tiles) * a.rows_per_tile;
        const int nt = job.n_tok <= 1 ? 1 : job.n_tok <= 4 ? 4 : 8;
        if (j != staged) {
            if (nt == 1) rvq_stage<1>(a, job, xs);
            else if (nt == 4) rvq_stage<4>(a, job, xs);
            else rvq_stage<8>(a, job, xs);
            staged = j;
        }
        __syncthreads();
        const int S = stages_of(a.m, job.matrix);
        if (a.m.e8p) {
            if (nt == 1) rvq_tile_rows<1, 2, true>(a, scb, xs, job, r0, warp, nwarps, lane);
            else if (nt == 4) rvq_tile_rows<4, 2, true>(a, scb, xs, job, r0, warp, nwarps, lane);
            else rvq_tile_rows<8, 2, true>(a, scb, xs, job, r0, warp, nwarps, lane);
        } else if (S == 0) {
            // nothing
        } else if (S == 2) {
            if (nt == 1) rvq_tile_rows<1, 2>(a, scb, xs, job, r0, warp, nwarps, lane);
            else if (nt == 4) rvq_tile_rows<4, 2>(a, scb, xs, job, r0, warp, nwarps, lane);
            else rvq_tile_rows<8, 2>(a, scb, xs, job, r0, warp, nwarps, lane);
        } else if (S == 1) {
            if (nt == 1) rvq_tile_rows<1, 1>(a, scb, xs, job, r0, warp, nwarps, lane);
            else if (nt == 4) rvq_tile_rows<4, 1>(a, scb, xs, job, r0, warp, nwarps, lane);
            else rvq_tile_rows<8, 1>(a, scb, xs, job, r0, warp, nwarps, lane);
        } else {
            if (nt == 1) rvq_tile_rows<1, 3>(a, scb, xs, job, r0, warp, nwarps, lane);
            else if (nt == 4) rvq_tile_rows<4, 3>(a, scb, xs, job, r0, warp, nwarps, lane);
            else rvq_tile_rows<8, 3>(a, scb, xs, job, r0, warp, nwarps, lane);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- decode-multiply (tcgen05 tensor cores)
// E8P sets: rvq_tc_kernel below.  Codebook (RVQ) sets: rvq_ws_kernel further
// down, a warp-specialised form that is faster where a K chunk takes several
// decode steps (one per residual stage); with E8P's single step per chunk the
// per-step handoff of its ring costs more than it hides (OLMoE-shaped layer at
// T = 32: E8P 0.27 ms here, 0.30 ms there; 2-stage RVQ 0.42 ms here, 0.38 there).
//
// For T >= 16 the product is a real dense contraction per expert: a CTA
// takes 128 output rows of one expert matrix and up to 32 of its tokens.  For
// every 128-wide K chunk, 256 threads decode the 128 x 128 weight tile
// (C1[i1] + C2[i2] in fp32, rounded to fp16) and the 32 x 128 activation tile
// (fp32 -> fp16) into shared memory in the canonical no-swizzle K-major layout
// (8-row x 16-byte core matrices; neighbours along K 128 B apart, along M/N
// 2048 B apart); one thread issues eight tcgen05.mma (M=128, N=32, K=16,
// fp16 x fp16 -> fp32 in tensor memory) and commits them to the buffer's
// mbarrier, while the threads decode the next chunk into the other buffer.
// The row scale is applied in the epilogue (tcgen05.ld of the accumulator).
// Every mbarrier wait is bounded: on expiry the kernel records QMOE_ETIMEOUT,
// still frees its tensor memory and returns.

constexpr int kTcM = 128, kTcN = 32, kTcK = 128;
constexpr int kTcThreads = 256;
constexpr int kTcVpt = kTcM * (kTcK / 8) / kTcThreads;   // 8-weight vectors each thread decodes per chunk (8)
constexpr int kTcBpt = kTcN * kTcK / kTcThreads;         // activations each thread stages per chunk (16)
static_assert(kTcVpt == 8 && kTcBpt == 16, "thread mapping of rvq_tc_kernel");
constexpr int kTcLBO = 128;                       // core matrices adjacent along K
constexpr int kTcSBO = (kTcK / 8) * 128;          // core matrices adjacent along M / N (2048 B)
constexpr int kTcABytes = kTcM * kTcK * 2;        // 32 KB
constexpr int kTcBBytes = kTcN * kTcK * 2;        // 8 KB
constexpr int kTcCbBytes = QMOE_RVQ_MAX_STAGES * 256 * 16;
// two weight tiles (steps alternate), and per chunk parity the activations' fp16 high and low parts
constexpr int kTcSmem = 1024 /*align*/ + kTcCbBytes + 2 * kTcABytes + 4 * kTcBBytes + 64;
constexpr uint32_t kTcSpinLimit = 1u << 20;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(kTcLBO >> 4) << 16;
    d |= (uint64_t)(kTcSBO >> 4) << 32;
    d |= 1ull << 46;                              // descriptor version for tcgen05
    return d;                                     // base offset 0, swizzle none
}

// kind::f16 instruction descriptor: D fp32, A and B fp16, both K-major, N = 64, M = 128.
// MMA N = 2 * kTcN: the activations' fp16 high parts are B rows 0..31, their low parts rows 32..63
constexpr int kTcNM = 2 * kTcN;
constexpr uint32_t kTcIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kTcNM >> 3) << 17) |
                              ((uint32_t)(kTcM >> 4) << 24);

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kTcSpinLimit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// 32 consecutive fp32 accumulator columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32_at(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Copies a thread's kTcVpt consecutive stage-`st` codewords (exact fp16 rows
// of codebook st; the vectors' S code bytes each are in cw) to consecutive
// core matrices along K of its weight-tile row.
__device__ __forceinline__ void stage_run(const uint4* scb, const uint2 (&cw)[QMOE_RVQ_MAX_STAGES], int S, int st,
                                          unsigned char* dst) {
    const uint64_t c0 = ((uint64_t)cw[0].y << 32) | cw[0].x;
    const uint64_t c1 = ((uint64_t)cw[1].y << 32) | cw[1].x;
    const uint64_t c2 = ((uint64_t)cw[2].y << 32) | cw[2].x;
#pragma unroll
    for (int q = 0; q < kTcVpt; ++q) {
        const int byte = q * S + st;                      // < 8 * QMOE_RVQ_MAX_STAGES
        const uint64_t c = byte < 8 ? c0 : byte < 16 ? c1 : c2;
        const uint32_t code = (uint32_t)(c >> (8 * (byte & 7))) & 255u;
        *(uint4*)(dst + q * kTcLBO) = scb[256 * st + code];
    }
}

// A thread's kTcVpt consecutive E8P code words (16 bytes in cw[0], cw[1]) decoded to exact
// fp16 rows of its weight-tile row.
__device__ __forceinline__ void e8p_run(const uint2* tab, const uint2 (&cw)[QMOE_RVQ_MAX_STAGES], int lane,
                                        unsigned char* dst) {
#pragma unroll
    for (int q = 0; q < kTcVpt; ++q) {
        const uint32_t word = q < 4 ? (q < 2 ? cw[0].x : cw[0].y) : (q < 6 ? cw[1].x : cw[1].y);
        const uint32_t code = (word >> (16 * (q & 1))) & 0xFFFFu;
        uint32_t h[4];
        e8p_half8(tab[(code & 255u) * kE8pRepTc + (lane & (kE8pRepTc - 1))], code, h);
        *(uint4*)(dst + q * kTcLBO) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// fp16 high part of 8 values, and the fp16 of what the high part leaves.
__device__ __forceinline__ void store_hi_lo8(uint8_t* hi, uint8_t* lo, const float (&v)[8]) {
    __half2 h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        h[q] = __floats2half2_rn(v[2 * q], v[2 * q + 1]);
        const float2 hf = __half22float2(h[q]);
        l[q] = __floats2half2_rn(v[2 * q] - hf.x, v[2 * q + 1] - hf.y);
    }
    *(uint4*)hi = *(const uint4*)h;
    *(uint4*)lo = *(const uint4*)l;
}

__global__ void __launch_bounds__(kTcThreads) rvq_tc_kernel(const RvqGemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint4* scb = (uint4*)smem;
    uint8_t* abuf = smem + kTcCbBytes;                            // 2 x 32 KB
    uint8_t* bbuf = abuf + 2 * kTcABytes;                         // 2 chunks x (high, low) x 8 KB
    uint64_t* bars = (uint64_t*)(bbuf + 4 * kTcBBytes);           // 2 mbarriers
    uint32_t* tmem_slot = (uint32_t*)(bars + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const RvqDev& m = a.m;

    if (m.e8p) e8p_stage_table<kE8pRepTc, kTcThreads>((const uint32_t*)m.cb, (uint2*)scb);
    else rvq_stage_codebooks((const uint4*)m.cb, scb, m.n_st);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bars + b)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTcNM)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    // weight-tile steps issued by this block (step j uses tile and barrier j & 1, its commit
    // completes barrier phase j >> 1); every step up to done - 1 is known to have completed
    uint32_t gs = 0, done = 0;
    bool timed_out = false;
    const int nv = m.cols / 8;
    const int nk = m.cols / kTcK;
    const int n_jobs = a.jobs ? *a.n_jobs_dev : (a.T_implicit + kTcN - 1) / kTcN;
    const int n_tiles = n_jobs * a.row_tiles;

    for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x) {
        Job job;
        const int j = tile / a.row_tiles;
        if (a.jobs) {
            job = a.jobs[j];
        } else {
            job.matrix = 0;
            job.slot_begin = j * kTcN;
            job.n_tok = min(kTcN, a.T_implicit - j * kTcN);
        }
        const int r0 = (tile % a.row_tiles) * kTcM;
        // per thread: A part (row, half of a chunk's 16 vectors), B part (token, two 8-wide K groups);
        // the 8 lanes of a quarter-warp take 8 consecutive rows (tokens), so their 16-byte tile stores
        // fill one 128-byte core matrix: no shared-memory bank conflict
        const int rl = (tid & 7) | ((tid >> 4) << 3), part = (tid >> 3) & 1;
        const int arow = r0 + rl;
        const int S = stages_of(m, job.matrix);              // code bytes per vector (8-byte aligned runs of kTcVpt)
        if (S == 0) continue;                                 // uniform over the block: skip the tile
        const uint8_t* ip = codes_of(m, job.matrix) + ((size_t)(arow < m.rows ? arow : 0) * nv + part * kTcVpt) * S;
        const int bn = (tid & 7) | ((tid >> 6) << 3), bg = (tid >> 3) & 7;
        const int bslot = bn < job.n_tok ? (a.slots ? a.slots[job.slot_begin + bn] : job.slot_begin + bn) : -1;
        const float* bp = a.xr + (size_t)(bslot < 0 ? 0 : bslot) * m.cols + bg * 16;
        // the token's staging scale: a power of two, applied before the fp16 split and undone in
        // the epilogue (exact)
        const float bscale = bslot >= 0 && a.xs ? __ldg(a.xs + bslot) : 1.0f;
        // the global loads of chunk kc + 1 are issued before chunk kc is decoded
        // a thread's kTcVpt vectors of a chunk: 8 * S code bytes, as S 8-byte loads
        uint2 cw_n[QMOE_RVQ_MAX_STAGES];
#pragma unroll
        for (int q = 0; q < QMOE_RVQ_MAX_STAGES; ++q)
            cw_n[q] = arow < m.rows && q < S ? __ldg((const uint2*)ip + q) : make_uint2(0u, 0u);
        float4 xv_n[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) xv_n[q] = bslot >= 0 ? __ldg((const float4*)bp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        // Steps: for every chunk, one per stage.  A step copies the stage's exact fp16
        // codewords into a weight tile (two tiles alternate) and issues its MMAs
        // against the chunk's activations, split as fp16 high + low parts (staged
        // at the chunk's first step, two chunk buffers alternate), so the product
        // carries neither the fp16 rounding of a stage sum nor of x'.
        for (int kc = 0; kc < nk && !timed_out; ++kc) {
            uint2 cw[QMOE_RVQ_MAX_STAGES];
#pragma unroll
            for (int q = 0; q < QMOE_RVQ_MAX_STAGES; ++q) cw[q] = cw_n[q];
            float4 xv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) xv[q] = xv_n[q];
            if (kc + 1 < nk) {
                if (arow < m.rows) {
                    const uint2* nx = (const uint2*)(ip + (size_t)(kc + 1) * (kTcK / 8) * S);
#pragma unroll
                    for (int q = 0; q < QMOE_RVQ_MAX_STAGES; ++q)
                        if (q < S) cw_n[q] = __ldg(nx + q);
                }
                if (bslot >= 0) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) xv_n[q] = __ldg((const float4*)(bp + (size_t)(kc + 1) * kTcK) + q);
                }
            }
            uint8_t* Bh = bbuf + (kc & 1) * 2 * kTcBBytes;           // N = 64 rows: high parts, then low
            uint8_t* Bl = Bh + 4 * kTcSBO;
            const int n_steps = m.e8p ? 1 : S;                // E8P: one exact fp16 tile per chunk
            for (int st = 0; st < n_steps; ++st) {
                const int b = gs & 1u;
                if (gs >= 2 && done + 1 < gs) {
                    // step gs - 2 (and so every earlier step: chunk kc - 2 included) has finished
                    // reading this weight tile and the chunk buffer about to be rewritten
                    if (!mbar_wait(smem_u32(bars + b), ((gs - 2) >> 1) & 1u)) timed_out = true;
                    done = gs - 1;
                }
                uint8_t* A = abuf + b * kTcABytes;
                unsigned char* arow_base = A + (rl >> 3) * kTcSBO + (rl & 7) * 16 + part * kTcVpt * kTcLBO;
                if (arow >= m.rows) {
#pragma unroll
                    for (int q = 0; q < kTcVpt; ++q) *(uint4*)(arow_base + q * kTcLBO) = make_uint4(0, 0, 0, 0);
                } else if (m.e8p) {
                    e8p_run((const uint2*)scb, cw, lane, arow_base);
                } else {
                    stage_run(scb, cw, S, st, arow_base);
                }
                if (st == 0) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int c8 = bg * 2 + h2;
                        const float v[8] = {xv[2 * h2].x * bscale,     xv[2 * h2].y * bscale,
                                            xv[2 * h2].z * bscale,     xv[2 * h2].w * bscale,
                                            xv[2 * h2 + 1].x * bscale, xv[2 * h2 + 1].y * bscale,
                                            xv[2 * h2 + 1].z * bscale, xv[2 * h2 + 1].w * bscale};
                        const int o = (bn >> 3) * kTcSBO + c8 * kTcLBO + (bn & 7) * 16;
                        store_hi_lo8(Bh + o, Bl + o, v);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                if (__syncthreads_or(timed_out)) {
                    timed_out = true;
                    break;
                }
                if (tid == 0) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t a0 = smem_u32(A), b0 = smem_u32(Bh);
#pragma unroll
                    for (int k = 0; k < kTcK / 16; ++k) {
                        const uint32_t acc = (kc > 0 || st > 0 || k > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                            " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                            "l"(umma_desc(a0 + k * 2 * kTcLBO)), "l"(umma_desc(b0 + k * 2 * kTcLBO)), "r"(kTcIdesc),
                            "r"(acc)
                            : "memory");
                    }
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     smem_u32(bars + b))
                                 : "memory");
                }
                ++gs;
            }
        }
        // wait for the outstanding steps (the last two at most), oldest first
        for (uint32_t j = (done + 2 > gs ? done : gs - 2); j < gs; ++j)
            if (!mbar_wait(smem_u32(bars + (j & 1u)), (j >> 1) & 1u)) timed_out = true;
        done = gs;
        timed_out = __syncthreads_or(timed_out);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (warp < 4 && !timed_out) {
            uint32_t r[32], rl2[32];
            const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
            tmem_ld32_at(taddr + kTcN, rl2);                      // the low parts' columns
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                  "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                  "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                  "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                  "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const int row = r0 + 32 * warp + lane;
            if (row < m.rows) {
                const float s = f16_to_f32(m.scale[(size_t)job.matrix * m.rows + row]);
#pragma unroll
                for (int n = 0; n < kTcN; ++n) {
                    if (n < job.n_tok) {
                        const int slot = a.slots ? a.slots[job.slot_begin + n] : job.slot_begin + n;
                        const float inv = a.xs ? 1.0f / __ldg(a.xs + slot) : 1.0f;     // exact: a power of two
                        a.out[(size_t)slot * m.rows + row] =
                            s * ((__uint_as_float(r[n]) + __uint_as_float(rl2[n])) * inv);
                    }
                }
            }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
    }
    if (timed_out) {
        // give the tensor core one more bounded chance to finish before the memory is freed
        for (uint32_t j = (done + 2 > gs ? done : gs - 2); j < gs; ++j)
            mbar_wait(smem_u32(bars + (j & 1u)), (j >> 1) & 1u);
        if (tid == 0) atomicCAS(&g_rvq_error, 0, QMOE_ETIMEOUT);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcNM) : "memory");
}

int launch_rvq_ws(RvqGemmArgs a, cudaStream_t st, long long tiles_hint);

int launch_rvq_tc(RvqGemmArgs a, cudaStream_t st, long long tiles_hint) {
    if (!a.m.e8p) return launch_rvq_ws(a, st, tiles_hint);
    int rc = qmoe::smem_attr((const void*)rvq_tc_kernel, kTcSmem, "rvq tc attr");
    if (rc) return rc;
    a.rows_per_tile = kTcM;
    a.row_tiles = (a.m.rows + kTcM - 1) / kTcM;
    const long long grid = std::max(1LL, std::min(tiles_hint, (long long)qmoe::sm_count() * 2));
    rvq_tc_kernel<<<(unsigned)grid, kTcThreads, kTcSmem, st>>>(a);
    return qmoe::launch_check("rvq_tc_kernel");
}

// ---------------------------------------------------------------- decode-multiply, warp-specialised (codebook sets)
// A tile is 128 output rows of one expert matrix and up to 32 of its tokens.
// One persistent CTA per SM, warp-specialised:
//  * 16 producer warps decode, for every 128-wide K chunk and every residual
//    stage (a "step"), the stage's exact fp16 codewords of the tile's rows into
//    a weight tile of a ring of three, in the canonical no-swizzle K-major
//    layout (8-row x 16-byte core matrices; neighbours along K 128 B apart,
//    along M/N 2048 B apart), and at a chunk's first step the chunk's rotated
//    activations as fp16 high parts and fp16 remainders (one N=64 operand,
//    two chunk buffers alternate).  The codebooks sit in shared memory eight
//    times, replica j holding every entry in 16-byte bank group j, and the
//    eight lanes of a quarter-warp read replicas 0..7: the gathers are free of
//    bank conflicts, as are the tile stores (a quarter-warp fills one core
//    matrix);
//  * one thread issues the step's eight tcgen05.mma (M=128, N=64, K=16, fp16 x
//    fp16 -> fp32 in tensor memory) once the step's barrier completes, and
//    commits them to the barriers that free the weight tile and, after the
//    chunk's last step, its activations;
//  * 4 epilogue warps read a finished tile's accumulator (two alternate, so the
//    next tile's MMAs run meanwhile), add the high and low parts' columns,
//    undo the staging scale, apply the row scale and store.
// Every wait is bounded: on expiry the kernel records
// QMOE_ETIMEOUT, waits (bounded) for its outstanding MMAs, frees its tensor
// memory and returns.

constexpr int kWsM = 128, kWsN = 32, kWsK = 128;
constexpr int kWsProd = 512;                               // producer threads (16 warps)
constexpr int kWsMmaWarp = kWsProd / 32;                   // then 4 epilogue warps
constexpr int kWsThreads = kWsProd + 5 * 32;
constexpr int kWsVpt = kWsM * (kWsK / 8) / kWsProd;        // 8-weight vectors each producer decodes per step (4)
constexpr int kWsBpt = kWsN * kWsK / kWsProd;              // activations each producer stages per chunk (8)
static_assert(kWsVpt == 4 && kWsBpt == 8, "thread mapping of rvq_ws_kernel");
constexpr int kWsLBO = 128;                       // core matrices adjacent along K
constexpr int kWsSBO = (kWsK / 8) * 128;          // core matrices adjacent along M / N (2048 B)
constexpr int kWsABytes = kWsM * kWsK * 2;        // 32 KB
constexpr int kWsBBytes = kWsN * kWsK * 2;        // 8 KB (high parts; the low parts follow)
constexpr int kWsRing = 3;                        // weight tiles
constexpr int kWsCbRep = 8;                       // codebook replicas (one per 16-byte bank group)
constexpr int kWsCbBytes = QMOE_RVQ_MAX_STAGES * 256 * kWsCbRep * 16;
constexpr int kWsBarBytes = 128;
constexpr int kWsSmem = 1024 /*align*/ + kWsCbBytes + kWsRing * kWsABytes + 4 * kWsBBytes + kWsBarBytes;
static_assert(kWsSmem <= 232448, "rvq_ws_kernel shared memory");
constexpr uint32_t kWsSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t ws_smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t ws_umma_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(kWsLBO >> 4) << 16;
    d |= (uint64_t)(kWsSBO >> 4) << 32;
    d |= 1ull << 46;                              // descriptor version for tcgen05
    return d;                                     // base offset 0, swizzle none
}

// kind::f16 instruction descriptor: D fp32, A and B fp16, both K-major, N = 64, M = 128.
// MMA N = 2 * kWsN: the activations' fp16 high parts are B rows 0..31, their low parts rows 32..63
constexpr int kWsNM = 2 * kWsN;
constexpr uint32_t kWsIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kWsNM >> 3) << 17) |
                              ((uint32_t)(kWsM >> 4) << 24);
constexpr int kWsTmemCols = 2 * kWsNM;            // two accumulators

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(ws_smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ws_smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mma_commit_to(uint64_t* b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(ws_smem_u32(b))
                 : "memory");
}

// Bounded wait for the phase of the given parity (suspending between tries); false when the bound ran out.
__device__ __forceinline__ bool ws_mbar_wait(uint64_t* b, uint32_t parity) {
    const uint32_t bar = ws_smem_u32(b);
    for (uint32_t it = 0; it < kWsSpinLimit; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(1000u)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// 16 consecutive fp32 accumulator columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld16_at(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Codebooks [n_st][256] x 16 bytes into shared memory, entry e of stage s in
// all replicas: replica j at 16-byte slot j of the 128-byte line (s * 256 + e).
// Run by the 256 producer threads (thread i loads entry i of every stage).
__device__ __forceinline__ void rvq_stage_codebooks_rep(const uint4* __restrict__ g, uint4* t, int n_st, int tid) {
    uint4 c[QMOE_RVQ_MAX_STAGES];
#pragma unroll
    for (int s = 0; s < QMOE_RVQ_MAX_STAGES; ++s) c[s] = s < n_st ? __ldg(g + tid + s * 256) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int s = 0; s < QMOE_RVQ_MAX_STAGES; ++s) {
        if (s < n_st) {
#pragma unroll
            for (int j = 0; j < kWsCbRep; ++j) t[(s * 256 + tid) * kWsCbRep + j] = c[s];
        }
    }
}

// Copies a thread's kWsVpt consecutive stage-`st` codewords (exact fp16 rows
// of codebook st, from replica j; the vectors' S code bytes each are in the S
// words of cw) to consecutive core matrices along K of its weight-tile row.
__device__ __forceinline__ void ws_stage_run(const uint4* scb, const uint32_t (&cw)[QMOE_RVQ_MAX_STAGES], int S, int st,
                                          int j, unsigned char* dst) {
#pragma unroll
    for (int q = 0; q < kWsVpt; ++q) {
        const int byte = q * S + st;                      // < 4 * QMOE_RVQ_MAX_STAGES
        const uint32_t w = byte < 4 ? cw[0] : byte < 8 ? cw[1] : cw[2];
        const uint32_t code = (w >> (8 * (byte & 3))) & 255u;
        *(uint4*)(dst + q * kWsLBO) = scb[(256 * st + code) * kWsCbRep + j];
    }
}

// The job of tile `tile` and its first row.
__device__ __forceinline__ Job rvq_tile_job(const RvqGemmArgs& a, int tile, int& r0) {
    Job job;
    const int j = tile / a.row_tiles;
    if (a.jobs) {
        job = a.jobs[j];
    } else {
        job.matrix = 0;
        job.slot_begin = j * kWsN;
        job.n_tok = min(kWsN, a.T_implicit - j * kWsN);
    }
    r0 = (tile % a.row_tiles) * kWsM;
    return job;
}

// Warms L2 with the code bytes of tile `tile` (its rows are contiguous: 128 rows x cols/8 x S
// bytes), rounded inwards to 16-byte boundaries.
__device__ void rvq_prefetch_tile(const RvqGemmArgs& a, int tile, int n_tiles) {
    if (tile >= n_tiles) return;
    int r0;
    const Job job = rvq_tile_job(a, tile, r0);
    const RvqDev& m = a.m;
    if (m.stages && (m.stages[job.matrix] < 1 || m.stages[job.matrix] > m.n_st)) return;
    const int S = m.stages ? m.stages[job.matrix] : 2;
    const size_t row_bytes = (size_t)(m.cols / 8) * S;
    const int r1 = min(m.rows, r0 + kWsM);
    const uintptr_t lo = ((uintptr_t)(codes_of(m, job.matrix) + (size_t)r0 * row_bytes) + 15) & ~(uintptr_t)15;
    const uintptr_t hi = (uintptr_t)(codes_of(m, job.matrix) + (size_t)r1 * row_bytes) & ~(uintptr_t)15;
    for (uintptr_t p = lo; p < hi;) {
        const uint32_t n = (uint32_t)min((uintptr_t)(1u << 20), hi - p);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
        p += n;
    }
}

__global__ void __launch_bounds__(kWsThreads, 1) rvq_ws_kernel(const RvqGemmArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint4* scb = (uint4*)smem;
    uint8_t* ring = smem + kWsCbBytes;                            // kWsRing weight tiles
    uint8_t* bbuf = ring + kWsRing * kWsABytes;                   // 2 chunks x (high, low)
    uint64_t* bars = (uint64_t*)(bbuf + 4 * kWsBBytes);
    uint64_t* a_full = bars;                     // [kWsRing] producers (one arrival per warp)
    uint64_t* a_empty = bars + kWsRing;          // [kWsRing] MMA commit: the weight tile was read
    uint64_t* b_full = bars + 2 * kWsRing;       // [2] producers (one arrival per warp)
    uint64_t* b_empty = b_full + 2;              // [2] MMA commit after the chunk's last step
    uint64_t* acc_full = b_full + 4;             // [2] MMA commit: the tile's accumulator is final
    uint64_t* acc_empty = b_full + 6;            // [2] epilogue warps (4 arrivals)
    uint32_t* tmem_slot = (uint32_t*)(b_full + 8);
    int* abort_flag = (int*)(tmem_slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const RvqDev& m = a.m;

    if (tid < 256) rvq_stage_codebooks_rep((const uint4*)m.cb, scb, m.n_st, tid);
    if (tid == 0) {
        for (int s = 0; s < kWsRing; ++s) {
            bar_init(a_full + s, kWsProd / 32);
            bar_init(a_empty + s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            bar_init(b_full + s, kWsProd / 32);
            bar_init(b_empty + s, 1);
            bar_init(acc_full + s, 1);
            bar_init(acc_empty + s, 4);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(ws_smem_u32(tmem_slot)),
                     "r"(kWsTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    volatile int* abort_v = abort_flag;

    bool timed_out = false;
    const int nv = m.cols / 8;
    const int nk = m.cols / kWsK;
    const int n_jobs = a.jobs ? *a.n_jobs_dev : (a.T_implicit + kWsN - 1) / kWsN;
    const int n_tiles = n_jobs * a.row_tiles;

    if (warp < kWsProd / 32) {
        // ---------------- producers: weight tiles of every step, activations of every chunk
        // per thread: A part (row, a quarter of a chunk's 16 vectors), B part (token, one 8-wide K
        // group); the 8 lanes of a quarter-warp take 8 consecutive rows (tokens), so their 16-byte tile
        // stores fill one 128-byte core matrix, and read codebook replicas 0..7
        const int rl = (tid & 7) | ((tid >> 5) << 3), part = (tid >> 3) & 3, rep = tid & 7;
        const int bn = (tid & 7) | ((tid >> 7) << 3), bg = (tid >> 3) & 15;
        uint32_t gs = 0, gc = 0;
        if (tid == 0) rvq_prefetch_tile(a, blockIdx.x, n_tiles);
        for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x) {
            // the next tile's codes travel towards L2 while this one is decoded
            if (tid == 0) rvq_prefetch_tile(a, tile + gridDim.x, n_tiles);
            int r0;
            const Job job = rvq_tile_job(a, tile, r0);
            const int S = stages_of(m, job.matrix);          // code bytes per vector
            if (S == 0) continue;                             // every role skips the tile
            const int arow = r0 + rl;
            const uint8_t* ip = codes_of(m, job.matrix) + ((size_t)(arow < m.rows ? arow : 0) * nv + part * kWsVpt) * S;
            const int bslot = bn < job.n_tok ? (a.slots ? a.slots[job.slot_begin + bn] : job.slot_begin + bn) : -1;
            const float* bp = a.xr + (size_t)(bslot < 0 ? 0 : bslot) * m.cols + bg * 8;
            // the token's staging scale: a power of two, applied before the fp16 split and undone in
            // the epilogue (exact)
            const float bscale = bslot >= 0 && a.xs ? __ldg(a.xs + bslot) : 1.0f;
            // the global loads of chunk kc + 1 are issued before chunk kc is decoded; a thread's
            // kWsVpt vectors of a chunk are 4 * S code bytes, as S 4-byte loads
            uint32_t cw_n[QMOE_RVQ_MAX_STAGES];
#pragma unroll
            for (int q = 0; q < QMOE_RVQ_MAX_STAGES; ++q)
                cw_n[q] = arow < m.rows && q < S ? __ldg((const uint32_t*)ip + q) : 0u;
            float4 xv_n[2];
#pragma unroll
            for (int q = 0; q < 2; ++q)
                xv_n[q] = bslot >= 0 ? __ldg((const float4*)bp + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            const int n_steps = S;
            for (int kc = 0; kc < nk && !timed_out; ++kc, ++gc) {
                uint32_t cw[QMOE_RVQ_MAX_STAGES];
#pragma unroll
                for (int q = 0; q < QMOE_RVQ_MAX_STAGES; ++q) cw[q] = cw_n[q];
                float4 xv[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) xv[q] = xv_n[q];
                if (kc + 1 < nk) {
                    if (arow < m.rows) {
                        const uint32_t* nx = (const uint32_t*)(ip + (size_t)(kc + 1) * (kWsK / 8) * S);
#pragma unroll
                        for (int q = 0; q < QMOE_RVQ_MAX_STAGES; ++q)
                            if (q < S) cw_n[q] = __ldg(nx + q);
                    }
                    if (bslot >= 0) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) xv_n[q] = __ldg((const float4*)(bp + (size_t)(kc + 1) * kWsK) + q);
                    }
                }
                uint8_t* Bh = bbuf + (gc & 1u) * 2 * kWsBBytes;        // N = 64 rows: high parts, then low
                uint8_t* Bl = Bh + 4 * kWsSBO;
                for (int st = 0; st < n_steps; ++st, ++gs) {
                    const uint32_t slot = gs % kWsRing;
                    bool ok = ws_mbar_wait(a_empty + slot, ((gs / kWsRing) & 1u) ^ 1u);
                    if (st == 0) ok = ok && ws_mbar_wait(b_empty + (gc & 1u), ((gc >> 1) & 1u) ^ 1u);
                    ok = ok && !*abort_v;
                    if (__any_sync(QMOE_FULL_MASK, !ok)) {
                        timed_out = true;
                        break;
                    }
                    uint8_t* A = ring + slot * kWsABytes;
                    unsigned char* arow_base = A + (rl >> 3) * kWsSBO + (rl & 7) * 16 + part * kWsVpt * kWsLBO;
                    if (arow >= m.rows) {
#pragma unroll
                        for (int q = 0; q < kWsVpt; ++q) *(uint4*)(arow_base + q * kWsLBO) = make_uint4(0, 0, 0, 0);
                    } else {
                        ws_stage_run(scb, cw, S, st, rep, arow_base);
                    }
                    if (st == 0) {
                        const float v[8] = {xv[0].x * bscale, xv[0].y * bscale, xv[0].z * bscale, xv[0].w * bscale,
                                            xv[1].x * bscale, xv[1].y * bscale, xv[1].z * bscale, xv[1].w * bscale};
                        const int o = (bn >> 3) * kWsSBO + bg * kWsLBO + (bn & 7) * 16;
                        store_hi_lo8(Bh + o, Bl + o, v);
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        bar_arrive(a_full + slot);
                        if (st == 0) bar_arrive(b_full + (gc & 1u));
                    }
                }
            }
        }
    } else if (warp == kWsMmaWarp) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t gs = 0, gc = 0, t = 0;
            for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x) {
                int r0;
                const Job job = rvq_tile_job(a, tile, r0);
                const int S = stages_of(m, job.matrix);
                if (S == 0) continue;
                const uint32_t acc = t & 1u;
                if (!ws_mbar_wait(acc_empty + acc, ((t >> 1) & 1u) ^ 1u) || *abort_v) {
                    timed_out = true;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + acc * (uint32_t)kWsNM;
                const int n_steps = S;
                for (int kc = 0; kc < nk && !timed_out; ++kc, ++gc) {
                    const uint32_t b0 = ws_smem_u32(bbuf + (gc & 1u) * 2 * kWsBBytes);
                    for (int st = 0; st < n_steps; ++st) {
                        const uint32_t slot = gs % kWsRing;
                        bool ok = ws_mbar_wait(a_full + slot, (gs / kWsRing) & 1u);
                        if (st == 0) ok = ok && ws_mbar_wait(b_full + (gc & 1u), (gc >> 1) & 1u);
                        if (!ok || *abort_v) {
                            timed_out = true;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const uint32_t a0 = ws_smem_u32(ring + slot * kWsABytes);
#pragma unroll
                        for (int k = 0; k < kWsK / 16; ++k) {
                            const uint32_t accf = (kc > 0 || st > 0 || k > 0) ? 1u : 0u;
                            asm volatile(
                                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
                                "l"(ws_umma_desc(a0 + k * 2 * kWsLBO)), "l"(ws_umma_desc(b0 + k * 2 * kWsLBO)), "r"(kWsIdesc),
                                "r"(accf)
                                : "memory");
                        }
                        mma_commit_to(a_empty + slot);
                        if (st == n_steps - 1) mma_commit_to(b_empty + (gc & 1u));
                        ++gs;
                    }
                }
                if (timed_out) break;
                mma_commit_to(acc_full + acc);
                ++t;
            }
            if (timed_out) {
                *abort_v = 1;
                // the tensor core may still be working on committed steps: wait (bounded) for the
                // last one before the memory is released
                if (gs > 0) ws_mbar_wait(a_empty + (gs - 1) % kWsRing, ((gs - 1) / kWsRing) & 1u);
            }
        }
    } else {
        // ---------------- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        const int qw = warp & 3;
        uint32_t t = 0;
        for (int tile = blockIdx.x; tile < n_tiles && !timed_out; tile += gridDim.x) {
            int r0;
            const Job job = rvq_tile_job(a, tile, r0);
            const int S = stages_of(m, job.matrix);
            if (S == 0) continue;
            const uint32_t acc = t & 1u;
            // lane n holds token n's slot and the inverse of its staging scale (exact: a power of
            // two); they and the row scale are read while the tile's MMAs run
            const int row = r0 + 32 * qw + lane;
            const int my_slot = lane < job.n_tok ? (a.slots ? a.slots[job.slot_begin + lane] : job.slot_begin + lane) : 0;
            const float my_inv = lane < job.n_tok && a.xs ? 1.0f / __ldg(a.xs + my_slot) : 1.0f;
            const float s = row < m.rows ? f16_to_f32(m.scale[(size_t)job.matrix * m.rows + row]) : 0.0f;
            const bool ok = ws_mbar_wait(acc_full + acc, (t >> 1) & 1u) && !*abort_v;
            if (__any_sync(QMOE_FULL_MASK, !ok)) {
                timed_out = true;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

            const uint32_t taddr = tmem + ((uint32_t)(32 * qw) << 16) + acc * (uint32_t)kWsNM;
#pragma unroll
            for (int h = 0; h < kWsN / 16; ++h) {
                uint32_t r[16], rl2[16];
                tmem_ld16_at(taddr + 16 * h, r);                    // the high parts' columns
                tmem_ld16_at(taddr + kWsN + 16 * h, rl2);           // the low parts' columns
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int n = 16 * h + q;
                    const int slot = __shfl_sync(QMOE_FULL_MASK, my_slot, n);
                    const float inv = __shfl_sync(QMOE_FULL_MASK, my_inv, n);
                    if (n < job.n_tok && row < m.rows)
                        a.out[(size_t)slot * m.rows + row] = s * ((__uint_as_float(r[q]) + __uint_as_float(rl2[q])) * inv);
                }
            }
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) bar_arrive(acc_empty + acc);
            ++t;
        }
    }
    if (timed_out) *abort_v = 1;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (tid == 0 && *abort_v) atomicCAS(&g_rvq_error, 0, QMOE_ETIMEOUT);
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kWsTmemCols) : "memory");
}

int launch_rvq_ws(RvqGemmArgs a, cudaStream_t st, long long tiles_hint) {
    int rc = qmoe::smem_attr((const void*)rvq_ws_kernel, kWsSmem, "rvq tc attr");
    if (rc) return rc;
    a.rows_per_tile = kWsM;
    a.row_tiles = (a.m.rows + kWsM - 1) / kWsM;
    const long long grid = std::max(1LL, std::min(tiles_hint, (long long)qmoe::sm_count()));
    rvq_ws_kernel<<<(unsigned)grid, kWsThreads, kWsSmem, st>>>(a);
    return qmoe::launch_check("rvq_ws_kernel");
}

// ---------------------------------------------------------------- decode (test)
__global__ void rvq_decode_kernel(RvqDev m, float* __restrict__ out) {
    const size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    const size_t nv = (size_t)m.rows * (m.cols / 8);
    if (v >= nv) return;
    const int r = (int)(v / (m.cols / 8));
    const int S = stages_of(m, 0);
    const uint8_t* ip = codes_of(m, 0) + v * S;
    const uint4* cb = (const uint4*)m.cb;
    float w[8];
    if (m.e8p) {
        const uint32_t code = ((const uint16_t*)codes_of(m, 0))[v];
        e8p_float8(e8p_bytes(__ldg((const uint32_t*)m.cb + (code & 255u))), code, w);
    } else if (S == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = 0.0f;
    } else if (S == 1) {
        const uint32_t code[1] = {ip[0]};
        decode_vec<1>(cb, code, w);
    } else if (S == 2) {
        const uint32_t code[2] = {ip[0], ip[1]};
        decode_vec<2>(cb, code, w);
    } else {
        const uint32_t code[3] = {ip[0], ip[1], ip[2]};
        decode_vec<3>(cb, code, w);
    }
    const float s = f16_to_f32(m.scale[r]);
    float* o = out + v * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __fmul_rn(s, w[j]);
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// jobs_hint: an upper bound on the launch's jobs; the row tiles shrink (down to 16 rows) until there
// are about two tiles per SM.
int launch_rvq_gemm(RvqGemmArgs a, cudaStream_t st, long long jobs_hint) {
    const int sms = qmoe::sm_count();
    const size_t tab = a.m.e8p ? (size_t)256 * kE8pRepGemm * 8 : (size_t)a.m.n_st * 256 * 16;
    const size_t smem = tab + (size_t)a.m.cols * a.nt_max * 4;
    int rc = qmoe::smem_attr((const void*)rvq_gemm_kernel, (int)smem, "rvq attr");
    if (rc) return rc;
    int rpt = std::min(a.m.rows, 128);
    while (rpt > 16 && std::max(1LL, jobs_hint) * ((a.m.rows + rpt - 1) / rpt) < 2LL * sms) rpt >>= 1;
    a.rows_per_tile = rpt;
    a.row_tiles = (a.m.rows + a.rows_per_tile - 1) / a.rows_per_tile;
    rvq_gemm_kernel<<<sms * 2, kRvqThreads, smem, st>>>(a);
    return qmoe::launch_check("rvq_gemm_kernel");
}

int nt_for(int cols) {
    // staged activations: cols * nt * 4 bytes, at most 64 KB
    return cols * 8 * 4 <= 65536 ? 8 : cols * 4 * 4 <= 65536 ? 4 : 1;
}

// Tensor-core path: a launch with at least kTcMinTokens activation rows, K a multiple of the
// 128-wide chunk.  An M128 x K16 MMA costs about 83 cycles whatever N <= 64 is, so the tensor
// path's cost is per weight (one MMA per stage and K16 step), not per token.
constexpr int kTcMinTokens = 16;
bool use_tc(long long rows_of_x, int cols) { return rows_of_x >= kTcMinTokens && cols % kTcK == 0; }

float inv_sqrt(int n) { return (float)(1.0 / std::sqrt((double)n)); }

int fwht_threads(int n) { return std::min(512, std::max(32, n / 2)); }

// Output transform of T tokens with k slots each (slot outputs yp [T*k][n]).
int launch_out_transform(const float* yp, const int32_t* expert_of, const int8_t* so, const float* gates, int T,
                         int k, int n, void* y, int y_is_f32, cudaStream_t st) {
    if (k >= 2 && k <= 8) {
        // one block per slot, the slots of a token in one cluster
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(T * k));
        cfg.blockDim = dim3((unsigned)fwht_threads(n));
        cfg.dynamicSmemBytes = (size_t)n * sizeof(float);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)k;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int rc = qmoe::cuda_check(cudaLaunchKernelEx(&cfg, out_transform_cluster_kernel, yp, expert_of, so, gates, k,
                                                     n, inv_sqrt(n), y, y_is_f32),
                                  "out transform (cluster) launch");
        if (rc) return rc;
        return qmoe::launch_check("out_transform_cluster_kernel");
    }
    const int kg = std::max(1, std::min(k, 98304 / (4 * n) - 1));
    const size_t smem = (size_t)(kg + 1) * n * sizeof(float);
    int rc = qmoe::smem_attr((const void*)out_transform_kernel, (int)smem, "out transform attr");
    if (rc) return rc;
    const int threads = std::min(1024, std::max(32, kg * n / 2));
    out_transform_kernel<<<T, threads, smem, st>>>(yp, expert_of, so, gates, k, kg, n, inv_sqrt(n), y, y_is_f32);
    return qmoe::launch_check("out_transform_kernel");
}

}  // namespace

namespace qmoe {
int rvq_take_error() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_rvq_error, sizeof(int)) != cudaSuccess) return QMOE_ECUDA;
    const int z = 0;
    if (cudaMemcpyToSymbol(g_rvq_error, &z, sizeof(int)) != cudaSuccess) return QMOE_ECUDA;
    return v;
}
}  // namespace qmoe

using qmoe::fail;

extern "C" int rvq_decode_dense(const rvq_matrix_set* mat, float* w_out, void* stream) {
    qmoe::clear_error();
    if (!valid_set(mat) || mat->count != 1 || !w_out) return fail(QMOE_EINVAL, "rvq_decode_dense: bad arguments");
    const size_t nv = (size_t)mat->rows * (mat->cols / 8);
    rvq_decode_kernel<<<(unsigned)((nv + 255) / 256), 256, 0, (cudaStream_t)stream>>>(to_dev(mat), w_out);
    return qmoe::launch_check("rvq_decode_dense");
}

extern "C" int rvq_expert_matmul_ws_size(int rows, int cols, int T, size_t* bytes) {
    qmoe::clear_error();
    if (!bytes || !pow2(rows) || !pow2(cols) || T < 0) return fail(QMOE_EINVAL, "rvq_expert_matmul_ws_size: bad sizes");
    *bytes = align256(sizeof(float) * (size_t)T * cols) + align256(sizeof(float) * (size_t)T * rows) +
             align256(sizeof(float) * (size_t)T);
    return QMOE_OK;
}

extern "C" int rvq_expert_matmul(const rvq_matrix_set* mat, const void* x_bf16, int T, void* y, int y_is_f32,
                                 void* workspace, size_t ws_bytes, void* stream) {
    qmoe::clear_error();
    if (!valid_set(mat) || mat->count != 1) return fail(QMOE_EINVAL, "rvq_expert_matmul: bad matrix (count must be 1)");
    if (T < 0) return fail(QMOE_EINVAL, "rvq_expert_matmul: T < 0");
    if (T == 0) return QMOE_OK;
    if (!x_bf16 || !y || !workspace) return fail(QMOE_EINVAL, "rvq_expert_matmul: NULL pointer");
    size_t need = 0;
    rvq_expert_matmul_ws_size(mat->rows, mat->cols, T, &need);
    if (ws_bytes < need) return fail(QMOE_ECAPACITY, "rvq_expert_matmul: workspace too small");
    cudaStream_t st = (cudaStream_t)stream;
    float* xr = (float*)workspace;
    float* yr = (float*)((char*)workspace + align256(sizeof(float) * (size_t)T * mat->cols));
    float* xs = (float*)((char*)yr + align256(sizeof(float) * (size_t)T * mat->rows));
    const int rows = mat->rows, cols = mat->cols;
    in_transform_kernel<<<T, fwht_threads(cols), 2 * cols * sizeof(float), st>>>(
        (const uint16_t*)x_bf16, 1, nullptr, 1, mat->sign_in, nullptr, cols, inv_sqrt(cols), xr, nullptr, xs,
        nullptr);
    int rc = qmoe::launch_check("in_transform_kernel");
    if (rc) return rc;
    RvqGemmArgs a{};
    a.m = to_dev(mat);
    a.xr = xr;
    a.xs = xs;
    a.jobs = nullptr;
    a.slots = nullptr;
    a.T_implicit = T;
    a.nt_max = nt_for(cols);
    a.out = yr;
    if (use_tc(T, cols)) rc = launch_rvq_tc(a, st, (long long)((T + kTcN - 1) / kTcN) * ((rows + kTcM - 1) / kTcM));
    else rc = launch_rvq_gemm(a, st, (T + a.nt_max - 1) / a.nt_max);
    if (rc) return rc;
    return launch_out_transform(yr, nullptr, mat->sign_out, nullptr, T, 1, rows, y, y_is_f32 ? 1 : 0, st);
}

namespace {
struct RvqMoeWs {
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    Job* jobs_a;
    Job* jobs_b;
    int* n_jobs;
    int32_t* expert_of;
    float* xg;
    float* xu;
    float* gp;
    float* up;
    float* hr;
    float* dp;
    float* xg_s;      // per-slot staging scales of xg, xu and hr (tensor-core kernel)
    float* xu_s;
    float* hr_s;
    size_t bytes;
};

RvqMoeWs rvq_moe_layout(void* base, int E, int d_model, int d_ff, int T, int k) {
    RvqMoeWs w{};
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
    w.n_jobs = (int*)take(sizeof(int) * 4);
    w.expert_of = nullptr;
    w.xg = (float*)take(sizeof(float) * slots * d_model);
    w.xu = (float*)take(sizeof(float) * slots * d_model);
    w.gp = (float*)take(sizeof(float) * slots * d_ff);
    w.up = (float*)take(sizeof(float) * slots * d_ff);
    w.hr = (float*)take(sizeof(float) * slots * d_ff);
    w.dp = (float*)take(sizeof(float) * slots * d_model);
    w.xg_s = (float*)take(sizeof(float) * std::max<size_t>(slots, 1));
    w.xu_s = (float*)take(sizeof(float) * std::max<size_t>(slots, 1));
    w.hr_s = (float*)take(sizeof(float) * std::max<size_t>(slots, 1));
    w.bytes = off;
    return w;
}
}  // namespace

extern "C" int rvq_moe_layer_ws_size(int E, int d_model, int d_ff, int T, int k, size_t* bytes) {
    qmoe::clear_error();
    if (!bytes || E < 1 || E > qmoe::kPlanMaxE || !pow2(d_model) || !pow2(d_ff) || T < 0 || k < 1 || k > E)
        return fail(QMOE_EINVAL, "rvq_moe_layer_ws_size: bad sizes");
    *bytes = rvq_moe_layout(nullptr, E, d_model, d_ff, T, k).bytes;
    return QMOE_OK;
}

extern "C" int rvq_moe_layer(const rvq_matrix_set* gate, const rvq_matrix_set* up, const rvq_matrix_set* down,
                             const void* x_bf16, int T, int k, const int32_t* ids, const float* gates, void* y,
                             int y_is_f32, void* workspace, size_t ws_bytes, void* stream) {
    qmoe::clear_error();
    if (!valid_set(gate) || !valid_set(up) || !valid_set(down)) return fail(QMOE_EINVAL, "rvq_moe_layer: bad matrix sets");
    const int E = gate->count, d_model = gate->cols, d_ff = gate->rows;
    if (up->count != E || up->rows != d_ff || up->cols != d_model || down->count != E || down->rows != d_model ||
        down->cols != d_ff)
        return fail(QMOE_EINVAL, "rvq_moe_layer: gate/up must be d_ff x d_model and down d_model x d_ff");
    if (E > qmoe::kPlanMaxE || T < 0 || k < 1 || k > E) return fail(QMOE_EINVAL, "rvq_moe_layer: bad E, T or k");
    if (T == 0) return QMOE_OK;
    if (!x_bf16 || !ids || !gates || !y || !workspace) return fail(QMOE_EINVAL, "rvq_moe_layer: NULL pointer");
    RvqMoeWs w = rvq_moe_layout(workspace, E, d_model, d_ff, T, k);
    if (ws_bytes < w.bytes) return fail(QMOE_ECAPACITY, "rvq_moe_layer: workspace too small");
    cudaStream_t st = (cudaStream_t)stream;
    const int slots = T * k;
    // with at least kTcMinTokens slots every expert takes the tensor-core kernel (jobs of kTcN
    // tokens): its cost is per weight, whatever the expert's token count; fewer slots take the
    // CUDA-core kernel
    const bool tc = use_tc(slots, d_model) && use_tc(slots, d_ff);
    const int nt_a = tc ? kTcN : nt_for(d_model), nt_b = tc ? kTcN : nt_for(d_ff);
    auto gemm = [&](RvqGemmArgs& ga, int rows) {
        return tc ? launch_rvq_tc(ga, st, (long long)slots * ((rows + kTcM - 1) / kTcM)) : launch_rvq_gemm(ga, st, slots);
    };
    qmoe::phase_event(0, st);
    int rc = qmoe::launch_plan(ids, slots, E, nt_a, nt_b, w.counts, w.offsets, w.perm, w.jobs_a, w.jobs_b, w.n_jobs, st);
    if (rc) return rc;
    // ids is [T][k] = expert of each flat slot
    in_transform_kernel<<<slots, fwht_threads(d_model), 2 * d_model * sizeof(float), st>>>(
        (const uint16_t*)x_bf16, k, ids, k, gate->sign_in, up->sign_in, d_model, inv_sqrt(d_model), w.xg, w.xu,
        w.xg_s, w.xu_s);
    if ((rc = qmoe::launch_check("in_transform_kernel"))) return rc;
    qmoe::phase_event(1, st);
    RvqGemmArgs a{};
    a.jobs = w.jobs_a;
    a.n_jobs_dev = w.n_jobs;
    a.slots = w.perm;
    a.nt_max = nt_a;
    a.m = to_dev(gate);
    a.xr = w.xg;
    a.xs = w.xg_s;
    a.out = w.gp;
    if ((rc = gemm(a, d_ff))) return rc;
    a.m = to_dev(up);
    a.xr = w.xu;
    a.xs = w.xu_s;
    a.out = w.up;
    if ((rc = gemm(a, d_ff))) return rc;
    qmoe::phase_event(2, st);
    swiglu_transform_kernel<<<slots, fwht_threads(d_ff), 2 * d_ff * sizeof(float), st>>>(
        w.gp, w.up, ids, gate->sign_out, up->sign_out, down->sign_in, d_ff, inv_sqrt(d_ff), w.hr, w.hr_s);
    if ((rc = qmoe::launch_check("swiglu_transform_kernel"))) return rc;
    qmoe::phase_event(3, st);
    a.jobs = w.jobs_b;
    a.n_jobs_dev = w.n_jobs + 1;
    a.nt_max = nt_b;
    a.m = to_dev(down);
    a.xr = w.hr;
    a.xs = w.hr_s;
    a.out = w.dp;
    if ((rc = gemm(a, d_model))) return rc;
    qmoe::phase_event(4, st);
    rc = launch_out_transform(w.dp, ids, down->sign_out, gates, T, k, d_model, y, y_is_f32 ? 1 : 0, st);
    qmoe::phase_event(5, st);
    return rc;
}
