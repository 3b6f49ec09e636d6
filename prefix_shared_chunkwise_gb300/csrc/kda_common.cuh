// Shared device-side definitions for the packed-tree KDA kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "plan_internal.h"

namespace harts {

// Device error codes written into PlanDev::err[0] (first error wins).
enum : int32_t {
    kDevErrNone = 0,
    kDevErrDecayRange = 1,   // a chunk's decay too large for the reference-scaled factorisation
    kDevErrBadIndex = 2,     // a plan index out of range
    kDevErrTimeout = 3,      // a bounded wait ran out
};

// Floats per replay-gradient row: dk, dv, dg (D each) and dbeta, padded to 16 bytes so that
// rows can be written with 16-byte stores.
__host__ __device__ constexpr int rep_width(int D) { return 3 * D + 4; }

// Largest |exponent| the reference-scaled factorisation may form (exp(85) < FLT_MAX).
constexpr float kMaxExpArg = 85.f;

struct FwdParams {
    const void *q, *k, *v, *g, *beta;
    void *o;
    float *states, *final_state;
    const float *h0;
    void *chunk_states;
    int32_t H, D;            // dk == dv == D
    float scale;
};

struct BwdParams {
    FwdParams f;
    const void *d_o;
    const float *d_final;
    void *dq, *dk, *dv, *dg, *dbeta;
    float *dh0;
    float *ds_init;          // [n_seq, H, D, D] gradient w.r.t. each sequence's initial state
    float *rep_grad;         // [R, H, rep_width(D)]: dk, dv, dg, dbeta of every replay occurrence
    void *dchunk;            // [n_chunks, H, D, D] bf16: dL/dS^T at every chunk end (tensor-core path)
};

__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_out(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

__device__ __forceinline__ void dev_error(const PlanDev &pd, int32_t code, int32_t a, int32_t b) {
    if (atomicCAS(pd.err, 0, code) == 0) { pd.err[1] = a; pd.err[2] = b; }
}

// Compact row of local position r of sequence `seq` (replay rows first), or -1 past its end.
__device__ __forceinline__ int64_t local_row(const PlanDev &pd, int32_t seq, int32_t rho,
                                             int32_t L, int32_t r) {
    if (r >= L) return -1;
    if (r < rho) return pd.replay_idx[pd.seq_rptr[seq] + r];
    return static_cast<int64_t>(pd.seq_row0[seq]) + (r - rho);
}

}  // namespace harts
