// Device-side helpers shared by the kernels of the library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "host_common.h"
#include "qmoe.h"

#define QMOE_FULL_MASK 0xFFFFFFFFu

namespace qmoe {

// Number of SMs of the current device (cached per device).
int sm_count();

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The limit is a per-kernel, per-device setting, so the call
// reaches the runtime once per (kernel, device, larger size); later launches
// only look it up.
int smem_attr(const void* kernel, int bytes, const char* where);

// The calling thread's current CUDA context (the driver's handle), or NULL
// when it cannot be read.  Per-device caches key on it as well, so that a
// device reset or a caller-created context never reuses a stale entry.
void* current_context();

// Records a CUDA failure (if any) and returns QMOE_ECUDA, else QMOE_OK.
inline int cuda_check(cudaError_t e, const char* where) {
    if (e == cudaSuccess) return QMOE_OK;
    return fail(QMOE_ECUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

// After a launch: picks up launch-configuration errors.
inline int launch_check(const char* where) { return cuda_check(cudaGetLastError(), where); }

// Each translation unit owns one device error word and exposes a host accessor
// that reads and clears it (synchronously, after the caller synchronised).
int dict_take_error();
int rvq_take_error();
int pack_take_error();

// Unit of work of the expert kernels: one expert matrix applied to up to
// `n_tok` tokens whose slots are slots[slot_begin .. slot_begin + n_tok).
struct Job {
    int matrix;
    int slot_begin;
    int n_tok;
    int pad;
};

// Enqueues the single-block planner: per-expert counts, exclusive offsets,
// the stable slot permutation and, when jobs_a/jobs_b are given, job tables
// that cut each expert's slots into chunks of nt_a / nt_b tokens
// (n_jobs[0], n_jobs[1] receive the job counts).  With tc_min > 0 and a
// jobs_tc table, experts with at least tc_min tokens are left out of the
// first two tables and cut into chunks of nt_tc tokens in jobs_tc
// (count in n_jobs[2]).
int launch_plan(const int32_t* ids, int n_slots, int E, int nt_a, int nt_b, int32_t* counts,
                int32_t* offsets, int32_t* perm, Job* jobs_a, Job* jobs_b, int* n_jobs,
                cudaStream_t st, int tc_min = 0, int nt_tc = 1, Job* jobs_tc = nullptr);
constexpr int kPlanMaxE = 8192;

// Records phase event i on st when the measurement hook is set.
void phase_event(int i, cudaStream_t st);

}  // namespace qmoe

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// float -> bf16 bits, round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float f16_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(QMOE_FULL_MASK, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(QMOE_FULL_MASK, v, d);
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(QMOE_FULL_MASK, v, d);
    return v;
}
