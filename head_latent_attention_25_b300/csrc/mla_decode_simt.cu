// Split-K decode over the latent cache, CUDA-core (SIMT) variant, plus the pieces
// every decode variant shares: the work schedule and the merge of cut sequences.
//
// Scores are taken against the folded query Q' = alpha * [W_UK^T q_C ; RoPE(q_R)]
// with alpha = softmax_scale * log2(e), so exp2 of a score difference is the
// softmax ratio.  Each (worker, head) keeps a running maximum m, running sum l and
// an unnormalised latent accumulator, rescaled whenever m grows (online softmax).
#include <math.h>

#include <cuda_fp8.h>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "mla_schedule.cuh"

namespace mla {

namespace {

// ------------------------------------------------------------------ schedule
__global__ void __launch_bounds__(1024) schedule_kernel(ScheduleArgs a) { build_schedule(a); }

// ------------------------------------------------------------------ multi-query index
__global__ void __launch_bounds__(256) expand_queries_kernel(const int64_t* __restrict__ row_off,
                                                             const int32_t* __restrict__ seq_len, int batch,
                                                             int n_q, int64_t* __restrict__ row_off_v,
                                                             int32_t* __restrict__ seq_len_v) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)batch * n_q) return;
    const int64_t b = i / n_q, j = i % n_q;
    row_off_v[i] = row_off[b];
    // a length below 1 marks the query as empty (flagged and zero-filled by the decode)
    const int64_t len = (int64_t)seq_len[b] - n_q + j + 1;
    seq_len_v[i] = (int32_t)(len < 0 ? 0 : len);
}

// ------------------------------------------------------------------ SIMT split
constexpr int kWarps = 8, kTileRows = 32, kMaxColsPerLane = 16;

struct SplitArgs {
    const float* qp; const void* cache; const int64_t* row_off; const int64_t* cum;
    const WorkerStart* wstart; void* o_lat; float* lse; float* part_o; float* part_l;
    int n_h, d_c, d_r, batch;
};

// Element k of a row of the fp8 cache layout: a latent code times its group's scale, or
// the bf16 rotary value.
__device__ __forceinline__ float ld_fp8_row(const uint8_t* row, int k, int d_c) {
    if (k < d_c) {
        __nv_fp8_e4m3 q;
        q.__x = row[k];
        return float(q) * *reinterpret_cast<const float*>(row + d_c + 4 * (k >> 7));
    }
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(row + d_c + 4 * (d_c >> 7) + 2 * (k - d_c)));
}

// Tc: the cache element type (float or bf16 rows of d_c + d_r elements; the output o_lat
// has the same type).  kFp8: the cache holds rows of the fp8 layout instead, o_lat is bf16.
template <typename Tc, bool kFp8 = false>
__global__ void __launch_bounds__(kWarps * 32) split_simt_kernel(SplitArgs a) {
    extern __shared__ float smem[];
    const int dq = a.d_c + a.d_r;
    const int ts = dq + 1;                      // odd stride: lane j reading row j is conflict-free
    float* tile = smem;                         // [kTileRows][ts]
    float* qs = smem + kTileRows * ts;          // [kWarps][dq]
    const int g = blockIdx.x;
    const WorkerStart W = a.wstart[g];
    const int64_t begin = W.begin, end = W.end;
    if (begin >= end) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y * kWarps + warp;
    const bool active = h < a.n_h;
    const Tc* cache = (const Tc*)a.cache;

    int b = W.b;                                // last sequence whose rows start at or before begin
    int64_t cur = begin;
    bool first = true;
    while (cur < end) {
        while (a.cum[b + 1] <= cur) ++b;
        const int64_t seq0 = a.cum[b];
        const int64_t len = a.cum[b + 1] - seq0;
        const int64_t r_lo = cur - seq0;
        const int64_t r_hi = min(len, end - seq0);
        __syncthreads();                        // previous segment done with qs / tile
        if (active)
            for (int k = lane; k < dq; k += 32)
                qs[warp * dq + k] = a.qp[((int64_t)b * a.n_h + h) * dq + k];
        float m = -INFINITY, l = 0.f;
        float acc[kMaxColsPerLane];
#pragma unroll
        for (int t = 0; t < kMaxColsPerLane; ++t) acc[t] = 0.f;
        const Tc* rows = cache + a.row_off[b] * dq;
        const int rb = kFp8RowBytes(a.d_c, a.d_r);
        const uint8_t* rows8 = (const uint8_t*)a.cache + a.row_off[b] * (int64_t)rb;
        for (int64_t r0 = r_lo; r0 < r_hi; r0 += kTileRows) {
            const int nr = (int)min((int64_t)kTileRows, r_hi - r0);
            __syncthreads();
            for (int e = tid; e < nr * dq; e += kWarps * 32) {
                const int j = e / dq, k = e - j * dq;
                if constexpr (kFp8) tile[j * ts + k] = ld_fp8_row(rows8 + (r0 + j) * (int64_t)rb, k, a.d_c);
                else tile[j * ts + k] = ld(rows + (r0 + j) * dq + k);
            }
            __syncthreads();
            if (!active) continue;
            float s = -INFINITY;
            if (lane < nr) {
                const float* row = tile + lane * ts;
                const float* q = qs + warp * dq;
                float acc_s = 0.f;
                for (int k = 0; k < dq; ++k) acc_s = fmaf(q[k], row[k], acc_s);
                s = acc_s;
            }
            const float mn = fmaxf(m, warp_max(s));
            const float alpha = exp2f(m - mn);
            const float p = (lane < nr) ? exp2f(s - mn) : 0.f;
            l = l * alpha + warp_sum(p);
#pragma unroll
            for (int t = 0; t < kMaxColsPerLane; ++t) acc[t] *= alpha;
            for (int j = 0; j < nr; ++j) {
                const float pj = __shfl_sync(0xffffffffu, p, j);
                const float* row = tile + j * ts;
#pragma unroll
                for (int t = 0; t < kMaxColsPerLane; ++t) {
                    const int c = lane + 32 * t;
                    if (c < a.d_c) acc[t] = fmaf(pj, row[c], acc[t]);
                }
            }
            m = mn;
        }
        if (active) {
            const float inv = 1.f / l;
            const float lse2 = m + log2f(l);
            if (r_lo == 0 && r_hi == len) {     // whole sequence here: final output
                const int64_t o = ((int64_t)b * a.n_h + h) * a.d_c;
                if (a.lse && lane == 0) a.lse[(int64_t)b * a.n_h + h] = lse2 * kLn2;
#pragma unroll
                for (int t = 0; t < kMaxColsPerLane; ++t) {
                    const int c = lane + 32 * t;
                    if (c < a.d_c) {
                        if (sizeof(Tc) == 2) st((__nv_bfloat16*)a.o_lat + o + c, acc[t] * inv);
                        else st((float*)a.o_lat + o + c, acc[t] * inv);
                    }
                }
            } else {
                const int64_t slot = 2 * (int64_t)g + (first ? 0 : 1);
                const int64_t o = (slot * a.n_h + h) * a.d_c;
                if (lane == 0) a.part_l[slot * a.n_h + h] = lse2;
#pragma unroll
                for (int t = 0; t < kMaxColsPerLane; ++t) {
                    const int c = lane + 32 * t;
                    if (c < a.d_c) a.part_o[o + c] = acc[t] * inv;
                }
            }
        }
        cur = seq0 + r_hi;
        first = false;
    }
}

// ------------------------------------------------------------------ merge
// Grid (batch, head groups of 8, column chunks): warp w of a block merges head
// 8*blockIdx.y + w of a sequence that was cut across workers.  Lane j keeps the
// log2-sum-exps of pieces j, j+32, ... in registers (one load round), the warp reduces
// their maximum and sum with shuffles, and each piece's weight is broadcast from its
// lane while every lane adds its kCols columns of that piece (float4 loads, 64 / kCols
// pieces in flight).  Large batches take 16 columns a lane and one chunk (a warp reads
// 2 KB of a piece contiguously); small batches, whose few sequences are cut into many
// pieces, take 4 columns a lane and spread the column rounds over blockIdx.z, so that
// enough blocks stream the partial results.
constexpr int kMergeHeads = 8;
constexpr int kMergeRegs = 4;                   // pieces held per lane before the slow path

__device__ __forceinline__ int64_t piece_slot(int64_t w, int64_t seq_begin, int64_t per) {
    // the worker's first segment (slot 2w) unless the sequence starts inside its range
    return 2 * w + (seq_begin <= w * per ? 0 : 1);
}

// Wide column chunks (kCols = 16, the many-sequence grids) hold 8 float4 loads a lane in
// flight and at most 85 registers, so three blocks fit on an SM (the grid's blocks start in
// fewer waves once the split kernel frees the SMs); narrow chunks (kCols = 4, a few long
// sequences cut in many pieces) keep 16 loads a lane in flight and two blocks an SM.
template <typename Tout, int kCols>
__global__ void __launch_bounds__(32 * kMergeHeads, kCols == 16 ? 3 : 2) merge_kernel(const int64_t* __restrict__ cum,
                                                                 const Schedule* __restrict__ sched,
                                                                 const float* __restrict__ part_o,
                                                                 const float* __restrict__ part_l,
                                                                 Tout* __restrict__ o_lat,
                                                                 float* __restrict__ lse, int n_h, int d_c) {
    // The kernel behind this one may set up at once: it can then overlap only this kernel
    // and the split kernel of the same call (which triggered after its own wait, so all
    // before it is complete).
    pdl_trigger();
    pdl_wait();                                 // launched behind the split kernel
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.y * kMergeHeads + (threadIdx.x >> 5);
    if (h >= n_h) return;
    const int64_t seq0 = cum[b], seq1 = cum[b + 1];
    const int64_t per = sched->per;
    Tout* out = o_lat + ((int64_t)b * n_h + h) * d_c;
    if (seq1 == seq0) {                         // empty or rejected by the schedule
        if (blockIdx.z != 0) return;
        for (int c = 2 * lane; c < d_c; c += 64) st2(out + c, 0.f, 0.f);
        if (lane == 0 && lse) lse[(int64_t)b * n_h + h] = -INFINITY;
        return;
    }
    if (sched->whole) return;                   // every sequence was finished by its worker
    const int64_t first_w = seq0 / per, last_w = (seq1 - 1) / per;
    if (first_w == last_w) return;              // finished in place by its only worker
    const int64_t np = last_w - first_w + 1;
    // pass 1: maximum and sum of the pieces' log2-sum-exps
    float lr[kMergeRegs];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kMergeRegs; ++k) {
        const int64_t p = lane + 32 * k;
        lr[k] = p < np ? part_l[piece_slot(first_w + p, seq0, per) * n_h + h] : -INFINITY;
        mx = fmaxf(mx, lr[k]);
    }
    for (int64_t p = lane + 32 * kMergeRegs; p < np; p += 32)
        mx = fmaxf(mx, part_l[piece_slot(first_w + p, seq0, per) * n_h + h]);
    mx = warp_max(mx);
    float L = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeRegs; ++k) L += exp2f(lr[k] - mx);
    for (int64_t p = lane + 32 * kMergeRegs; p < np; p += 32)
        L += exp2f(part_l[piece_slot(first_w + p, seq0, per) * n_h + h] - mx);
    L = warp_sum(L);
    const float inv = 1.f / L;
    if (lane == 0 && lse && blockIdx.z == 0) lse[(int64_t)b * n_h + h] = (mx + log2f(L)) * kLn2;
    // pass 2: in round rd a lane owns columns [kCols lane, kCols lane + kCols) + 32 kCols rd
    constexpr int kIn = (kCols == 16 ? 32 : 64) / kCols;   // pieces in flight
    const bool vec = (d_c % kCols) == 0;        // float4 loads stay aligned
    const int rounds = (d_c + 32 * kCols - 1) / (32 * kCols);
    for (int rd = blockIdx.z; rd < rounds; rd += gridDim.z) {
        // every lane runs the loop the same number of times (the shuffles need all 32)
        const int c0 = kCols * lane + 32 * kCols * rd;
        float acc[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
        const int nc = max(0, min(kCols, d_c - c0));
        auto add_piece = [&](int64_t p, float lp) {
            const float wp = exp2f(lp - mx) * inv;
            const float* src = part_o + (piece_slot(first_w + p, seq0, per) * n_h + h) * d_c + c0;
            if (vec && nc == kCols) {
#pragma unroll
                for (int q = 0; q < kCols / 4; ++q) {
                    const float4 v = *reinterpret_cast<const float4*>(src + 4 * q);
                    acc[4 * q] = fmaf(wp, v.x, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(wp, v.y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(wp, v.z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(wp, v.w, acc[4 * q + 3]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < kCols; ++e)
                    if (e < nc) acc[e] = fmaf(wp, src[e], acc[e]);
            }
        };
        if (vec) {
            // kIn pieces per round: sixteen 16-byte loads of a lane in flight together.  The
            // branch is warp-uniform (the shuffles need all 32 lanes); with vec a lane's
            // chunk is either whole (nc == kCols) or past the end (nc == 0, no loads).
#pragma unroll
            for (int k = 0; k < kMergeRegs; ++k) {
                if (32 * k >= np) break;
                const int nj = (int)min((int64_t)32, np - 32 * k);
                for (int j0 = 0; j0 < nj; j0 += kIn) {
                    float4 v[kIn][kCols / 4];
                    float wp[kIn];
#pragma unroll
                    for (int u = 0; u < kIn; ++u) {
                        const int j = j0 + u < nj ? j0 + u : j0;
                        wp[u] = j0 + u < nj ? exp2f(__shfl_sync(0xffffffffu, lr[k], j) - mx) * inv : 0.f;
                        const float4* src = reinterpret_cast<const float4*>(
                            part_o + (piece_slot(first_w + 32 * k + j, seq0, per) * n_h + h) * d_c + c0);
#pragma unroll
                        for (int q = 0; q < kCols / 4; ++q) v[u][q] = nc ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < kIn; ++u)
#pragma unroll
                        for (int q = 0; q < kCols / 4; ++q) {
                            acc[4 * q] = fmaf(wp[u], v[u][q].x, acc[4 * q]);
                            acc[4 * q + 1] = fmaf(wp[u], v[u][q].y, acc[4 * q + 1]);
                            acc[4 * q + 2] = fmaf(wp[u], v[u][q].z, acc[4 * q + 2]);
                            acc[4 * q + 3] = fmaf(wp[u], v[u][q].w, acc[4 * q + 3]);
                        }
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < kMergeRegs; ++k) {
                if (32 * k >= np) break;
                const int nj = (int)min((int64_t)32, np - 32 * k);
                for (int j = 0; j < nj; ++j) add_piece(32 * k + j, __shfl_sync(0xffffffffu, lr[k], j));
            }
        }
        for (int64_t p = 32 * kMergeRegs; p < np; ++p)
            add_piece(p, part_l[piece_slot(first_w + p, seq0, per) * n_h + h]);
#pragma unroll
        for (int e = 0; e < kCols; e += 2)
            if (e < nc) st2(out + c0 + e, acc[e], acc[e + 1]);
    }
}

}  // namespace

cudaError_t launch_expand_queries(const int64_t* row_off, const int32_t* seq_len, int batch, int n_q,
                                  int64_t* row_off_v, int32_t* seq_len_v, cudaStream_t s) {
    const int64_t n = (int64_t)batch * n_q;
    expand_queries_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(row_off, seq_len, batch, n_q, row_off_v,
                                                                      seq_len_v);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s) {
    schedule_kernel<<<1, 1024, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

int simt_workers(int batch, int n_heads, int64_t max_total_rows, int sm_count) {
    const int groups = (n_heads + kWarps - 1) / kWarps;
    int64_t w = (2LL * sm_count + groups - 1) / groups;
    const int64_t by_rows = (max_total_rows + kTileRows - 1) / kTileRows;
    if (w > by_rows) w = by_rows;
    if (w < 1) w = 1;
    (void)batch;
    return (int)w;
}

cudaError_t launch_split_simt(const mla_dims& d, bool bf16, int batch, int workers, const float* qp,
                              const void* cache, const int64_t* row_off, const int64_t* cum,
                              const void* sched, const WorkerStart* wstart, void* o_lat, float* lse,
                              float* part_o, float* part_l, cudaStream_t s, bool fp8) {
    (void)sched;                                // the kernel reads the start records instead
    SplitArgs a{qp, cache, row_off, cum, wstart, o_lat, lse, part_o, part_l, d.n_heads, d.d_c, d.d_r, batch};
    const int dq = d.d_c + d.d_r;
    const size_t smem = (size_t)(kTileRows * (dq + 1) + kWarps * dq) * sizeof(float);
    dim3 grid(workers, (d.n_heads + kWarps - 1) / kWarps);
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(split_simt_kernel<__nv_bfloat16, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        profile_before_split(s);
        split_simt_kernel<__nv_bfloat16, true><<<grid, kWarps * 32, smem, s>>>(a);
    } else if (bf16) {
        e = cudaFuncSetAttribute(split_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        profile_before_split(s);
        split_simt_kernel<__nv_bfloat16><<<grid, kWarps * 32, smem, s>>>(a);
    } else {
        e = cudaFuncSetAttribute(split_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        profile_before_split(s);
        split_simt_kernel<float><<<grid, kWarps * 32, smem, s>>>(a);
    }
    profile_after_split(s);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_merge(const mla_dims& d, bool bf16, int batch, const int64_t* cum,
                         const void* sched, const float* part_o, const float* part_l, void* o_lat,
                         float* lse, cudaStream_t s, bool pdl) {
    const int groups = (d.n_heads + kMergeHeads - 1) / kMergeHeads;
    // fewer (sequence, head group) blocks than two per SM: narrow column chunks over blockIdx.z
    const bool narrow = (int64_t)batch * groups < 2 * 148;
    const int chunks = narrow ? (d.d_c + 127) / 128 : 1;
    const dim3 grid(batch, groups, chunks);
    const dim3 block(32 * kMergeHeads);
    cudaError_t e;
    if (bf16)
        e = narrow ? launch_ex(merge_kernel<__nv_bfloat16, 4>, grid, block, 0, s, pdl, cum, (const Schedule*)sched,
                               part_o, part_l, (__nv_bfloat16*)o_lat, lse, d.n_heads, d.d_c)
                   : launch_ex(merge_kernel<__nv_bfloat16, 16>, grid, block, 0, s, pdl, cum, (const Schedule*)sched,
                               part_o, part_l, (__nv_bfloat16*)o_lat, lse, d.n_heads, d.d_c);
    else
        e = narrow ? launch_ex(merge_kernel<float, 4>, grid, block, 0, s, pdl, cum, (const Schedule*)sched,
                               part_o, part_l, (float*)o_lat, lse, d.n_heads, d.d_c)
                   : launch_ex(merge_kernel<float, 16>, grid, block, 0, s, pdl, cum, (const Schedule*)sched,
                               part_o, part_l, (float*)o_lat, lse, d.n_heads, d.d_c);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
