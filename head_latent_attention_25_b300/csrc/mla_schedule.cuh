// The split schedule of the decode: prefix sums of the sequence lengths over the
// flattened context, the equal share of rows per worker, and each worker's first
// sequence.  Built by one thread block of any size (a multiple of 32, at most 1024).
#pragma once

#include "mla_common.cuh"

namespace mla {

struct ScheduleArgs {
    const int32_t* seq_len;
    const int64_t* row_off;
    int64_t cache_rows;
    int batch;
    int workers;
    int64_t* cum;           // [batch + 1]
    Schedule* sched;
    WorkerStart* wstart;    // [workers]
    int32_t* dev_status;
    int align;              // sequences flattened in multiples of this many rows (1, or a tile for paged caches)
    int64_t paged_cap;      // > 0: paged cache, a sequence is usable when 1 <= seq_len <= paged_cap (row_off unused)
};

// A sequence takes part with its length when 1 <= seq_len and its rows lie inside the
// cache buffer (paged: its length is covered by its block-table entries); otherwise it
// counts as empty and MLA_DEV_BAD_LENGTH is raised.  With align > 1 every sequence spans
// its length rounded up to a multiple of align in the flattened context.
__device__ __forceinline__ void build_schedule(const ScheduleArgs& a) {
    __shared__ long long warp_tot[32];
    __shared__ long long carry;
    __shared__ unsigned long long longest;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x;
    if (tid == 0) { carry = 0; longest = 0; }
    __syncthreads();
    for (int base = 0; base < a.batch; base += nt) {
        const int i = base + tid;
        long long x = 0;
        if (i < a.batch) {
            const long long n = a.seq_len[i];
            const bool usable = a.paged_cap > 0 ? (n >= 1 && n <= a.paged_cap)
                                                : (n >= 1 && a.row_off[i] >= 0 && a.row_off[i] + n <= a.cache_rows);
            if (usable) x = (n + a.align - 1) / a.align * a.align;
            else atomicOr(a.dev_status, MLA_DEV_BAD_LENGTH);
            atomicMax(&longest, (unsigned long long)x);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            long long t = lane < nt / 32 ? warp_tot[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                long long y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const long long incl = carry + (warp ? warp_tot[warp - 1] : 0) + x;
        if (i < a.batch) a.cum[i + 1] = incl;
        __syncthreads();
        if (tid == nt - 1) carry = incl;
        __syncthreads();
    }
    const long long total = carry;
    int64_t per = total > 0 ? (total + a.workers - 1) / a.workers : 1;
    per = (per + a.align - 1) / a.align * a.align;          // range boundaries on whole tiles
    // Whole sequences per worker when there are no more sequences than workers and the
    // longest is within a quarter of the equal share: a little more time on the busiest
    // worker buys no cut sequence (no partial results, no merge, no mid-range reload of
    // the folded query).
    const bool whole = a.batch <= a.workers && (long long)longest <= per + per / 4;
    Schedule s;
    s.total = total;
    s.workers = a.workers;
    s.batch = a.batch;
    s.per = per;
    s.whole = whole ? 1 : 0;
    if (tid == 0) {
        a.cum[0] = 0;
        *a.sched = s;
    }
    __syncthreads();                            // cum complete and visible to the block
    // each worker's start: its range, and its first sequence, the last one whose rows start
    // at or before the range start (saves every role of the split kernels a binary search
    // and the loads of a walk to its first tile)
    for (int g = tid; g < a.workers; g += nt) {
        WorkerStart w;
        worker_range(s, a.cum, g, &w.begin, &w.end);
        int b;
        if (whole) {
            b = g < a.batch ? g : a.batch - 1;
        } else {
            int lo = 0, hi = a.batch - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.cum[mid] <= w.begin) lo = mid; else hi = mid - 1;
            }
            b = lo;
        }
        w.b = b;
        w.pad = 0;
        w.seq0 = a.cum[b];
        w.seq1 = a.cum[b + 1];
        w.row0 = (a.paged_cap > 0 || a.row_off == nullptr) ? 0 : a.row_off[b];
        a.wstart[g] = w;
    }
}

}  // namespace mla
