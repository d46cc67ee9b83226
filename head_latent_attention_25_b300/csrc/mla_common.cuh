// Shared device/host helpers of the MLA decode library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr double kTwoPi = 6.283185307179586476925286766559;

// ---- element access -------------------------------------------------------------
__device__ __forceinline__ float ld(const float* p) { return *p; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st(float* p, float v) { *p = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// ---- rotary angle -----------------------------------------------------------------
// cos/sin of pos * theta_k, theta_k = base^(-2k/d_r).  The product is formed and
// reduced into [-pi, pi] in fp64 so that positions up to 2^31 keep full fp32
// accuracy after the final single-precision sincos.
__device__ __forceinline__ void rope_cos_sin(int64_t pos, int k, int d_r, float base,
                                             float* c, float* s) {
    double theta = pow((double)base, -2.0 * (double)k / (double)d_r);
    double ang = (double)pos * theta;
    double red = ang - kTwoPi * rint(ang / kTwoPi);
    sincosf((float)red, s, c);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- decode schedule ----------------------------------------------------------------
// The flattened context of all sequences (sequence 0's rows, then sequence 1's, ...)
// is cut into `workers` equal contiguous ranges.  A worker walks the sequences its
// range touches; a sequence it covers entirely is finished in place, a sequence cut
// by a range boundary leaves one partial result per piece.  A worker holds at most
// two cut pieces (its first and its last sequence), so partial slots are 2*worker
// and 2*worker+1.
struct Schedule {
    int64_t total;      // sum of max(seq_len, 0)
    int64_t per;        // rows per worker range (>= 1)
    int32_t workers;
    int32_t batch;
};

// Layout of the decode workspace (offsets in bytes, each 256-aligned).
struct DecodeWorkspace {
    size_t q_off, q_bytes;          // folded query Q' [batch, n_h, d_c + d_r]
    size_t cum_off, cum_bytes;      // int64 prefix sums of sequence lengths [batch + 1]
    size_t sched_off, sched_bytes;  // Schedule
    size_t po_off, po_bytes;        // partial o_lat [2*workers, n_h, d_c] fp32
    size_t pl_off, pl_bytes;        // partial log2-sum-exp [2*workers, n_h] fp32
    size_t total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace mla
