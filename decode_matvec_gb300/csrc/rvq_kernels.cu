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
// memory butterflies (O(n log n)), one block per activation row.

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
};

RvqDev to_dev(const rvq_matrix_set* s) {
    return RvqDev{s->idx, s->codebooks, s->scale_f16, s->sign_out, s->sign_in, s->count, s->rows, s->cols};
}

bool pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

bool valid_set(const rvq_matrix_set* s) {
    return s && s->idx && s->codebooks && s->scale_f16 && s->sign_out && s->sign_in && s->count >= 1 &&
           pow2(s->rows) && pow2(s->cols) && s->cols >= 8 && s->rows <= 8192 && s->cols <= 8192;
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

// x'[row] = H (D_in x[src]) for one or two sign vectors (gate and up share the input).
__global__ void in_transform_kernel(const uint16_t* __restrict__ x, int x_div, const int32_t* __restrict__ expert_of,
                                    int k_of, const int8_t* __restrict__ si0, const int8_t* __restrict__ si1, int n,
                                    float norm, float* __restrict__ out0, float* __restrict__ out1) {
    extern __shared__ float sm[];
    const int row = blockIdx.x;
    const int e = expert_of ? expert_of[row] : 0;
    const uint16_t* src = x + (size_t)(row / x_div) * n;
    float* s0 = sm;
    float* s1 = sm + n;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float v = bf16_to_f32(src[i]);
        s0[i] = v * (float)si0[(size_t)e * n + i];
        if (si1) s1[i] = v * (float)si1[(size_t)e * n + i];
    }
    __syncthreads();
    fwht_smem(s0, n, norm);
    if (si1) fwht_smem(s1, n, norm);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        out0[(size_t)row * n + i] = s0[i];
        if (si1) out1[(size_t)row * n + i] = s1[i];
    }
    (void)k_of;
}

// h = bf16(silu(g) * u) with g = D_out,g H g', u = D_out,u H u'; then the down
// matrix's input transform h' = H (D_in,down h).
__global__ void swiglu_transform_kernel(const float* __restrict__ gp, const float* __restrict__ up,
                                        const int32_t* __restrict__ expert_of, const int8_t* __restrict__ so_g,
                                        const int8_t* __restrict__ so_u, const int8_t* __restrict__ si_d, int n,
                                        float norm, float* __restrict__ out) {
    extern __shared__ float sm[];
    const int row = blockIdx.x;
    const int e = expert_of[row];
    float* sg = sm;
    float* su = sm + n;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        sg[i] = gp[(size_t)row * n + i];
        su[i] = up[(size_t)row * n + i];
    }
    __syncthreads();
    fwht_smem(sg, n, norm);
    fwht_smem(su, n, norm);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float g = sg[i] * (float)so_g[(size_t)e * n + i];
        const float u = su[i] * (float)so_u[(size_t)e * n + i];
        const float silu = g / (1.0f + expf(-g));
        const float h = bf16_to_f32(f32_to_bf16(silu * u));
        sg[i] = h * (float)si_d[(size_t)e * n + i];
    }
    __syncthreads();
    fwht_smem(sg, n, norm);
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[(size_t)row * n + i] = sg[i];
}

// y[t] = sum_j gate[t][j] * D_out H y'[t*k + j]  (k == 1 and gates == NULL: plain output transform)
__global__ void out_transform_kernel(const float* __restrict__ yp, const int32_t* __restrict__ expert_of,
                                     const int8_t* __restrict__ so, const float* __restrict__ gates, int k, int n,
                                     float norm, void* __restrict__ y, int y_is_f32) {
    extern __shared__ float sm[];
    const int t = blockIdx.x;
    float* s = sm;
    float* acc = sm + n;
    for (int i = threadIdx.x; i < n; i += blockDim.x) acc[i] = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int slot = t * k + j;
        const int e = expert_of ? expert_of[slot] : 0;
        const float g = gates ? gates[slot] : 1.0f;
        for (int i = threadIdx.x; i < n; i += blockDim.x) s[i] = yp[(size_t)slot * n + i];
        __syncthreads();
        fwht_smem(s, n, norm);
        for (int i = threadIdx.x; i < n; i += blockDim.x) acc[i] = fmaf(g, s[i] * (float)so[(size_t)e * n + i], acc[i]);
        __syncthreads();
    }
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (y_is_f32) ((float*)y)[(size_t)t * n + i] = acc[i];
        else ((uint16_t*)y)[(size_t)t * n + i] = f32_to_bf16(acc[i]);
    }
}

// ---------------------------------------------------------------- decode-multiply (CUDA cores)
struct RvqGemmArgs {
    RvqDev m;
    const float* xr;      // rotated activations, fp32 [slot][cols]
    const Job* jobs;
    const int* n_jobs_dev;
    const int* slots;
    int T_implicit;
    int nt_max;
    int rows_per_tile;
    int row_tiles;
    float* out;           // rotated outputs, fp32 [slot][rows]
};

__device__ __forceinline__ void decode8(uint4 c1, uint4 c2, float (&w)[8]) {
    const uint32_t a[4] = {c1.x, c1.y, c1.z, c1.w};
    const uint32_t b[4] = {c2.x, c2.y, c2.z, c2.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a[q]));
        const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b[q]));
        w[2 * q] = fa.x + fb.x;
        w[2 * q + 1] = fa.y + fb.y;
    }
}

template <int NT>
__device__ void rvq_tile_rows(const RvqGemmArgs& a, const uint4* scb, const float* xs, const Job& job, int r0,
                              int warp, int nwarps, int lane) {
    const RvqDev& m = a.m;
    const int nv = m.cols / 8;
    const int r1 = min(m.rows, r0 + a.rows_per_tile);
    for (int r = r0 + warp; r < r1; r += nwarps) {
        const uint16_t* ip = (const uint16_t*)(m.idx + ((size_t)job.matrix * m.rows + r) * nv * 2);
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
        for (int v = lane; v < nv; v += 32) {
            const uint32_t pr = __ldg(ip + v);
            float w[8];
            decode8(scb[pr & 255u], scb[256 + (pr >> 8)], w);
            if constexpr (NT == 1) {
                const float4 x0 = ((const float4*)xs)[2 * v], x1 = ((const float4*)xs)[2 * v + 1];
                acc[0] = fmaf(w[0], x0.x, acc[0]);
                acc[0] = fmaf(w[1], x0.y, acc[0]);
                acc[0] = fmaf(w[2], x0.z, acc[0]);
                acc[0] = fmaf(w[3], x0.w, acc[0]);
                acc[0] = fmaf(w[4], x1.x, acc[0]);
                acc[0] = fmaf(w[5], x1.y, acc[0]);
                acc[0] = fmaf(w[6], x1.z, acc[0]);
                acc[0] = fmaf(w[7], x1.w, acc[0]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float* xc = xs + (size_t)(8 * v + j) * NT;
#pragma unroll
                    for (int t = 0; t < NT; t += 4) {
                        const float4 xv = *(const float4*)(xc + t);
                        acc[t] = fmaf(w[j], xv.x, acc[t]);
                        if (t + 1 < NT) acc[t + 1] = fmaf(w[j], xv.y, acc[t + 1]);
                        if (t + 2 < NT) acc[t + 2] = fmaf(w[j], xv.z, acc[t + 2]);
                        if (t + 3 < NT) acc[t + 3] = fmaf(w[j], xv.w, acc[t + 3]);
                    }
                }
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

template <int NT>
__device__ void rvq_stage(const RvqGemmArgs& a, const Job& job, float* xs) {
    const int cols = a.m.cols;
    for (int t = 0; t < NT; ++t) {
        if (t < job.n_tok) {
            const int slot = a.slots ? a.slots[job.slot_begin + t] : job.slot_begin + t;
            const float* src = a.xr + (size_t)slot * cols;
            for (int c = threadIdx.x; c < cols; c += blockDim.x) xs[(size_t)c * NT + t] = src[c];
        } else {
            for (int c = threadIdx.x; c < cols; c += blockDim.x) xs[(size_t)c * NT + t] = 0.0f;
        }
    }
}

__global__ void __launch_bounds__(kRvqThreads) rvq_gemm_kernel(const RvqGemmArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint4* scb = (uint4*)smem;                  // [2][256] x 8 fp16
    float* xs = (float*)(smem + 2 * 256 * 16);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    for (int i = tid; i < 2 * 256; i += blockDim.x) scb[i] = __ldg((const uint4*)a.m.cb + i);
    __syncthreads();
    const int n_jobs = a.jobs ? *a.n_jobs_dev : (a.T_implicit + a.nt_max - 1) / a.nt_max;
    const int n_tiles = n_jobs * a.row_tiles;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
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
        if (nt == 1) rvq_stage<1>(a, job, xs);
        else if (nt == 4) rvq_stage<4>(a, job, xs);
        else rvq_stage<8>(a, job, xs);
        __syncthreads();
        if (nt == 1) rvq_tile_rows<1>(a, scb, xs, job, r0, warp, nwarps, lane);
        else if (nt == 4) rvq_tile_rows<4>(a, scb, xs, job, r0, warp, nwarps, lane);
        else rvq_tile_rows<8>(a, scb, xs, job, r0, warp, nwarps, lane);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- decode (test)
__global__ void rvq_decode_kernel(RvqDev m, float* __restrict__ out) {
    const size_t v = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    const size_t nv = (size_t)m.rows * (m.cols / 8);
    if (v >= nv) return;
    const int r = (int)(v / (m.cols / 8));
    const uint32_t i1 = m.idx[2 * v], i2 = m.idx[2 * v + 1];
    const uint4 c1 = __ldg((const uint4*)m.cb + i1);
    const uint4 c2 = __ldg((const uint4*)m.cb + 256 + i2);
    float w[8];
    decode8(c1, c2, w);
    const float s = f16_to_f32(m.scale[r]);
    float* o = out + v * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __fmul_rn(s, w[j]);
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

int launch_rvq_gemm(RvqGemmArgs a, cudaStream_t st) {
    const int sms = qmoe::sm_count();
    const size_t smem = 2 * 256 * 16 + (size_t)a.m.cols * a.nt_max * 4;
    int rc = qmoe::cuda_check(
        cudaFuncSetAttribute(rvq_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem), "rvq attr");
    if (rc) return rc;
    a.rows_per_tile = 16;
    a.row_tiles = (a.m.rows + 15) / 16;
    rvq_gemm_kernel<<<sms * 2, kRvqThreads, smem, st>>>(a);
    return qmoe::launch_check("rvq_gemm_kernel");
}

int nt_for(int cols) {
    // staged activations: cols * nt * 4 bytes, at most 64 KB
    return cols * 8 * 4 <= 65536 ? 8 : cols * 4 * 4 <= 65536 ? 4 : 1;
}

float inv_sqrt(int n) { return (float)(1.0 / std::sqrt((double)n)); }

int fwht_threads(int n) { return std::min(512, std::max(32, n / 2)); }

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
    *bytes = align256(sizeof(float) * (size_t)T * cols) + align256(sizeof(float) * (size_t)T * rows);
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
    const int rows = mat->rows, cols = mat->cols;
    in_transform_kernel<<<T, fwht_threads(cols), 2 * cols * sizeof(float), st>>>(
        (const uint16_t*)x_bf16, 1, nullptr, 1, mat->sign_in, nullptr, cols, inv_sqrt(cols), xr, nullptr);
    int rc = qmoe::launch_check("in_transform_kernel");
    if (rc) return rc;
    RvqGemmArgs a{};
    a.m = to_dev(mat);
    a.xr = xr;
    a.jobs = nullptr;
    a.slots = nullptr;
    a.T_implicit = T;
    a.nt_max = nt_for(cols);
    a.out = yr;
    rc = launch_rvq_gemm(a, st);
    if (rc) return rc;
    out_transform_kernel<<<T, fwht_threads(rows), 2 * rows * sizeof(float), st>>>(
        yr, nullptr, mat->sign_out, nullptr, 1, rows, inv_sqrt(rows), y, y_is_f32 ? 1 : 0);
    return qmoe::launch_check("out_transform_kernel");
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
    w.n_jobs = (int*)take(sizeof(int) * 2);
    w.expert_of = nullptr;
    w.xg = (float*)take(sizeof(float) * slots * d_model);
    w.xu = (float*)take(sizeof(float) * slots * d_model);
    w.gp = (float*)take(sizeof(float) * slots * d_ff);
    w.up = (float*)take(sizeof(float) * slots * d_ff);
    w.hr = (float*)take(sizeof(float) * slots * d_ff);
    w.dp = (float*)take(sizeof(float) * slots * d_model);
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
    const int nt_a = nt_for(d_model), nt_b = nt_for(d_ff);
    qmoe::phase_event(0, st);
    int rc = qmoe::launch_plan(ids, slots, E, nt_a, nt_b, w.counts, w.offsets, w.perm, w.jobs_a, w.jobs_b, w.n_jobs, st);
    if (rc) return rc;
    // ids is [T][k] = expert of each flat slot
    in_transform_kernel<<<slots, fwht_threads(d_model), 2 * d_model * sizeof(float), st>>>(
        (const uint16_t*)x_bf16, k, ids, k, gate->sign_in, up->sign_in, d_model, inv_sqrt(d_model), w.xg, w.xu);
    if ((rc = qmoe::launch_check("in_transform_kernel"))) return rc;
    qmoe::phase_event(1, st);
    RvqGemmArgs a{};
    a.jobs = w.jobs_a;
    a.n_jobs_dev = w.n_jobs;
    a.slots = w.perm;
    a.nt_max = nt_a;
    a.m = to_dev(gate);
    a.xr = w.xg;
    a.out = w.gp;
    if ((rc = launch_rvq_gemm(a, st))) return rc;
    a.m = to_dev(up);
    a.xr = w.xu;
    a.out = w.up;
    if ((rc = launch_rvq_gemm(a, st))) return rc;
    qmoe::phase_event(2, st);
    swiglu_transform_kernel<<<slots, fwht_threads(d_ff), 2 * d_ff * sizeof(float), st>>>(
        w.gp, w.up, ids, gate->sign_out, up->sign_out, down->sign_in, d_ff, inv_sqrt(d_ff), w.hr);
    if ((rc = qmoe::launch_check("swiglu_transform_kernel"))) return rc;
    qmoe::phase_event(3, st);
    a.jobs = w.jobs_b;
    a.n_jobs_dev = w.n_jobs + 1;
    a.nt_max = nt_b;
    a.m = to_dev(down);
    a.xr = w.hr;
    a.out = w.dp;
    if ((rc = launch_rvq_gemm(a, st))) return rc;
    qmoe::phase_event(4, st);
    out_transform_kernel<<<T, fwht_threads(d_model), 2 * d_model * sizeof(float), st>>>(
        w.dp, ids, down->sign_out, gates, k, d_model, inv_sqrt(d_model), y, y_is_f32 ? 1 : 0);
    rc = qmoe::launch_check("out_transform_kernel");
    qmoe::phase_event(5, st);
    return rc;
}
