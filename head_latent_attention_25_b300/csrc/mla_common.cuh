// Shared device/host helpers of the MLA decode library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
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
// theta_k = base^(-2k/d_r) = r^k with r = base^(-2/d_r).  The host forms r once per
// call in fp64 (rope_ratio); the kernels raise it to the integer power k by binary
// powering (at most 2*log2(k) fp64 products, relative error below 1e-14), form
// pos * theta_k and reduce it into [-pi, pi] in fp64, so positions up to 2^31 keep
// full fp32 accuracy after the final single-precision sincos.  No fp64
// transcendental runs on the device (fp64 throughput on this part is low).
inline double rope_ratio(float base, int d_r) { return pow((double)base, -2.0 / (double)d_r); }

__device__ __forceinline__ double rope_theta(double r, int k) {
    double t = 1.0, p = r;
    for (; k; k >>= 1) {
        if (k & 1) t *= p;
        p *= p;
    }
    return t;
}

__device__ __forceinline__ void rope_cos_sin(int64_t pos, int k, double r, float* c, float* s) {
    const double ang = (double)pos * rope_theta(r, k);
    const double red = fma(-kTwoPi, rint(ang * (1.0 / kTwoPi)), ang);
    sincosf((float)red, s, c);
}

// ---- paired element access (rotary pairs, vectorised epilogues) --------------------
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st2(float* p, float a, float b) {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
}
__device__ __forceinline__ void st2(__nv_bfloat16* p, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
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
    int32_t whole;      // 1: worker g takes sequence g whole (no sequence is cut)
};

// Rows [*begin, *end) of the flattened context that worker g covers: an equal share
// (the last one shorter), or sequence g whole.
__host__ __device__ __forceinline__ void worker_range(const Schedule& S, const int64_t* cum, int g,
                                                      int64_t* begin, int64_t* end) {
    if (S.whole) {
        *begin = g < S.batch ? cum[g] : 0;
        *end = g < S.batch ? cum[g + 1] : 0;
    } else {
        *begin = (int64_t)g * S.per;
        *end = *begin + S.per < S.total ? *begin + S.per : S.total;
    }
}

// Where worker g starts, written by the schedule kernel so that a decode kernel reaches its
// first tile through one dependent load: the worker's range, its first sequence b (the
// last one whose rows start at or before the range start), that sequence's span in the
// flattened context and its first cache row.
struct __align__(16) WorkerStart {
    int64_t begin, end;     // rows [begin, end) of the flattened context (worker_range)
    int64_t seq0, seq1;     // cum[b], cum[b + 1]
    int64_t row0;           // row_off[b] for a contiguous cache, else 0
    int32_t b;
    int32_t pad;
};
static_assert(sizeof(WorkerStart) == 48, "three 16-byte loads");

// Where the latent rows of the cache live (the tensor-core path): the latent part in kv,
// the rotary part in pe (or packed after the latent in kv), and the row of position t of
// sequence b either row_off[b] + t (contiguous) or from a block table (paged).
// Bytes of one row of the fp8 cache layout: E4M3 codes of the latent, one fp32 scale per
// 128 latent columns, the rotary part in bf16 (MLA_FP8_ROW_BYTES in the public header).
__host__ __device__ constexpr int kFp8RowBytes(int d_c, int d_r) { return d_c + 4 * (d_c / 128) + 2 * d_r; }

struct CacheView {
    const void* kv;
    const void* pe;                 // null: packed, the rotary part at column d_c of kv
    int64_t kv_stride, pe_stride;   // elements between rows
    int64_t rows;
    const int32_t* block_table;     // null: contiguous
    int32_t block_size, max_blocks;
};

// Row of position pos of sequence b (contiguous: row_off[b] + pos).
__device__ __forceinline__ int64_t cache_row(const CacheView& c, const int64_t* row_off, int b, int64_t pos) {
    if (!c.block_table) return row_off[b] + pos;
    return (int64_t)c.block_table[(int64_t)b * c.max_blocks + pos / c.block_size] * c.block_size +
           pos % c.block_size;
}

// Layout of the decode workspace (offsets in bytes, each 256-aligned).
struct DecodeWorkspace {
    size_t q_off, q_bytes;          // folded query Q' [batch, n_h, d_c + d_r]
    size_t cum_off, cum_bytes;      // int64 prefix sums of sequence lengths [batch + 1]
    size_t sched_off, sched_bytes;  // Schedule
    size_t ws_off, ws_bytes;        // int32 first sequence of each worker's range [workers]
    size_t po_off, po_bytes;        // partial o_lat [2*workers, n_h, d_c] fp32
    size_t pl_off, pl_bytes;        // partial log2-sum-exp [2*workers, n_h] fp32
    size_t total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- programmatic dependent launch --------------------------------------------------
// A kernel launched with pdl = true may start while the previous kernel of its stream
// (always one of this library's, enqueued by the same call) is still running.  It must
// call pdl_wait() before it touches memory that kernel writes or reads; pdl_wait()
// returns once that kernel has completed and its writes are visible (and at once for a
// kernel launched without the attribute).  pdl_trigger() lets the next such kernel be
// scheduled before this one ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? at : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace mla
