// C-ABI entry points: argument checks, workspace planning and kernel dispatch.
#include <math.h>

#include <atomic>
#include <climits>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "mla_schedule.cuh"

using namespace mla;

namespace {

std::atomic<unsigned long long> g_launches{0};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
thread_local cudaEvent_t t_ev_start = nullptr;
thread_local cudaEvent_t t_ev_stop = nullptr;

}  // namespace

namespace mla {

void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

void profile_before_split(cudaStream_t s) {
    if (t_ev_start) cudaEventRecord(t_ev_start, s);
}

void profile_after_split(cudaStream_t s) {
    if (t_ev_stop) cudaEventRecord(t_ev_stop, s);
}

}  // namespace mla

namespace {

bool dims_ok(const mla_dims* d) {
    if (!d) return false;
    if (d->n_heads < 1 || d->d_h < 1 || d->d_c < 2 || d->d_r < 2 || d->hidden < 1) return false;
    if ((d->d_c & 1) || (d->d_r & 1)) return false;
    if (!(d->rope_base > 0.f) || !isfinite(d->rope_base)) return false;
    if (!(d->softmax_scale >= 0.f) || !isfinite(d->softmax_scale)) return false;
    if ((int64_t)d->n_heads * d->d_h > (1 << 24) || d->d_c > 65536 || d->d_r > 65536) return false;
    return true;
}

bool dtype_ok(mla_dtype t) { return t == MLA_F32 || t == MLA_BF16; }
size_t elt(mla_dtype t) { return t == MLA_BF16 ? 2 : 4; }
bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

float scale_of(const mla_dims* d) {
    return d->softmax_scale > 0.f ? d->softmax_scale : 1.f / sqrtf((float)(d->d_h + d->d_r));
}

// Largest latent width the SIMT decode keeps in registers (16 columns per lane).
constexpr int kSimtMaxDc = 512;

bool simt_supported(const mla_dims* d) {
    return d->d_c <= kSimtMaxDc && (d->d_c + d->d_r) <= 1024;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// The tcgen05 kernel is written for the DeepSeek latent shape: 512 latent + 64 rotary
// columns, at most 128 heads (one MMA M tile) and a cache of at least one 32-row tile.
bool tc_shape(const mla_dims* d, mla_dtype t) {
    return t == MLA_BF16 && d->d_c == 512 && d->d_r == 64 && d->n_heads <= 128;
}

struct DecodePlan {
    bool tc;
    int workers;
    int64_t q_rows;                  // rows of the folded-query buffer
    DecodeWorkspace ws;
};

bool plan_decode(const mla_dims* d, mla_dtype t, int batch, int max_seq_len, int num_splits,
                 bool tc, DecodePlan* p) {
    if (!dims_ok(d) || !dtype_ok(t) || batch < 1 || max_seq_len < 0 || num_splits < 0) return false;
    if (!tc && !simt_supported(d)) return false;
    const int64_t rows_bound = (int64_t)batch * (max_seq_len > 0 ? max_seq_len : 1);
    int w = num_splits;
    if (w == 0) {
        const int sms = sm_count();
        if (sms <= 0) return false;
        w = tc ? tc_workers(rows_bound, sms) : simt_workers(batch, d->n_heads, rows_bound, sms);
    }
    if (w > (1 << 20)) return false;
    p->tc = tc;
    p->workers = w;
    DecodeWorkspace& ws = p->ws;
    const size_t A = 256;
    const int dq = d->d_c + d->d_r;
    p->q_rows = (int64_t)batch * d->n_heads;
    if (tc && p->q_rows < 128) p->q_rows = 128;      // one full 128-row TMA box always fits
    size_t off = 0;
    ws.q_off = off;
    ws.q_bytes = (size_t)p->q_rows * dq * (tc ? 2 : sizeof(float));
    off = align_up(off + ws.q_bytes, A);
    ws.cum_off = off;   ws.cum_bytes = (size_t)(batch + 1) * sizeof(int64_t);
    off = align_up(off + ws.cum_bytes, A);
    ws.sched_off = off; ws.sched_bytes = sizeof(Schedule);
    off = align_up(off + ws.sched_bytes, A);
    ws.ws_off = off;    ws.ws_bytes = (size_t)w * sizeof(WorkerStart);
    off = align_up(off + ws.ws_bytes, A);
    ws.po_off = off;    ws.po_bytes = (size_t)2 * w * d->n_heads * d->d_c * sizeof(float);
    off = align_up(off + ws.po_bytes, A);
    ws.pl_off = off;    ws.pl_bytes = (size_t)2 * w * d->n_heads * sizeof(float);
    off = align_up(off + ws.pl_bytes, A);
    ws.total = off;
    return true;
}

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace

extern "C" {

const char* mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported dims/dtype";
        case MLA_ERR_WORKSPACE: return "workspace missing or too small";
        case MLA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

uint64_t mla_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t mla_set_wait_limit_ns(uint64_t ns) {
    return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

mla_status mla_profile_events(void* start, void* stop) {
    if ((start == nullptr) != (stop == nullptr)) return MLA_ERR_INVALID_ARG;
    t_ev_start = (cudaEvent_t)start;
    t_ev_stop = (cudaEvent_t)stop;
    return MLA_OK;
}

size_t mla_append_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_new) {
    if (!dims_ok(dims) || !dtype_ok(dtype) || batch < 1 || n_new < 1) return 0;
    if (dtype != MLA_BF16 || !gemm_tc_shapes_ok(*dims)) return 0;
    return append_tc_workspace(*dims, batch * n_new, nullptr, sm_count());
}

mla_status mla_cache_append(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_new,
                            const void* h, const void* w_dkv, const void* w_kr,
                            const int64_t* row_off, const int32_t* cap, const int32_t* pos0,
                            void* cache, int64_t cache_rows, void* workspace, size_t workspace_bytes,
                            int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || n_new < 1 || (int64_t)batch * n_new > (1LL << 30) || cache_rows < 1)
        return MLA_ERR_INVALID_ARG;
    if (!h || !w_dkv || !w_kr || !row_off || !cap || !pos0 || !cache || !dev_status)
        return MLA_ERR_INVALID_ARG;
    const size_t row_bytes = (size_t)(dims->d_c + dims->d_r) * elt(dtype);
    if (!aligned(cache, 16) || row_bytes % 16) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == MLA_BF16 && gemm_tc_shapes_ok(*dims)) {
        const int sms = sm_count();
        const size_t need = append_tc_workspace(*dims, batch * n_new, nullptr, sms);
        if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
        if (!aligned(h, 16) || !aligned(w_dkv, 16) || !aligned(w_kr, 16)) return MLA_ERR_INVALID_ARG;
        const CacheView cv{cache, nullptr, dims->d_c + dims->d_r, 0, cache_rows, nullptr, 0, 0};
        return cuda_status(launch_append_tc(*dims, batch, n_new, h, w_dkv, w_kr, row_off, cap, pos0,
                                            cv, workspace, dev_status, sms, s));
    }
    return cuda_status(launch_append(*dims, dtype == MLA_BF16, batch, n_new, h, w_dkv, w_kr,
                                     row_off, cap, pos0, cache, cache_rows, dev_status, s));
}

mla_status mla_project_query(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t d_in,
                             const void* x, const void* w_uq, const void* w_qr, void* q_c,
                             void* q_r, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || d_in < 1) return MLA_ERR_INVALID_ARG;
    if (!x || !w_uq || !w_qr || !q_c || !q_r || !dev_status) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t m1 = (int64_t)dims->n_heads * dims->d_h, m2 = (int64_t)dims->n_heads * dims->d_r;
    if (dtype == MLA_BF16 && m1 % 128 == 0 && m2 % 8 == 0 && m1 + m2 <= (1 << 24) && d_in % 64 == 0 &&
        aligned(x, 16) && aligned(w_uq, 16) && aligned(w_qr, 16) && aligned(q_c, 16) && aligned(q_r, 16))
        return cuda_status(launch_project_query_tc(*dims, batch, d_in, x, w_uq, w_qr, q_c, q_r, dev_status, s));
    return cuda_status(launch_project_query(*dims, dtype == MLA_BF16, batch, d_in, x, w_uq, w_qr,
                                            q_c, q_r, s));
}

// The output projection after the decode runs on tensor cores only: bf16 with d_h, d_c
// and hidden multiples of 128.
static bool output_tc(const mla_dims* d, mla_dtype t) {
    return t == MLA_BF16 && d->d_h % 128 == 0 && d->d_c % 128 == 0 && d->hidden % 128 == 0 &&
           (int64_t)d->n_heads * d->d_c <= (1 << 24);
}

size_t mla_output_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t merged) {
    if (!dims_ok(dims) || !dtype_ok(dtype) || batch < 1 || !output_tc(dims, dtype)) return 0;
    const int k_in = dims->n_heads * (merged ? dims->d_c : dims->d_h);
    return output_tc_workspace(dims->hidden, k_in, batch, sm_count());
}

static mla_status output_common(const mla_dims* dims, mla_dtype dtype, int32_t batch, const void* x,
                                const void* w, void* workspace, size_t workspace_bytes, void* u,
                                int32_t* dev_status, bool merged) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || !x || !w || !u || !dev_status) return MLA_ERR_INVALID_ARG;
    if (!output_tc(dims, dtype)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(u, 4)) return MLA_ERR_INVALID_ARG;
    const size_t need = mla_output_workspace_size(dims, dtype, batch, merged ? 1 : 0);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
    return MLA_OK;
}

mla_status mla_project_output(const mla_dims* dims, mla_dtype dtype, int32_t batch, const void* o,
                              const void* w_o, void* workspace, size_t workspace_bytes, void* u,
                              int32_t* dev_status, void* stream) {
    const mla_status st = output_common(dims, dtype, batch, o, w_o, workspace, workspace_bytes, u, dev_status, false);
    if (st != MLA_OK) return st;
    return cuda_status(launch_output_tc(*dims, batch, o, w_o, workspace, u, dev_status, sm_count(),
                                        (cudaStream_t)stream));
}

mla_status mla_project_output_merged(const mla_dims* dims, mla_dtype dtype, int32_t batch, const void* o_lat,
                                     const void* w_ov, void* workspace, size_t workspace_bytes, void* u,
                                     int32_t* dev_status, void* stream) {
    const mla_status st = output_common(dims, dtype, batch, o_lat, w_ov, workspace, workspace_bytes, u, dev_status,
                                        true);
    if (st != MLA_OK) return st;
    return cuda_status(launch_output_merged_tc(*dims, batch, o_lat, w_ov, workspace, u, dev_status, sm_count(),
                                               (cudaStream_t)stream));
}

mla_status mla_merge_output_weights(const mla_dims* dims, mla_dtype dtype, const void* w_o, const void* w_uv,
                                    void* w_ov, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (!w_o || !w_uv || !w_ov || !dev_status) return MLA_ERR_INVALID_ARG;
    if (!output_tc(dims, dtype)) return MLA_ERR_UNSUPPORTED;
    if (!aligned(w_o, 16) || !aligned(w_uv, 16) || !aligned(w_ov, 16)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_merge_output_weights_tc(*dims, w_o, w_uv, w_ov, dev_status, (cudaStream_t)stream));
}

static bool query_latent_tc(const mla_dims* d, mla_dtype t, int32_t d_q) {
    return t == MLA_BF16 && d_q % 128 == 0 && d->hidden % 64 == 0;
}

size_t mla_query_latent_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t d_q) {
    if (!dims_ok(dims) || !dtype_ok(dtype) || batch < 1 || d_q < 1) return 0;
    if (!query_latent_tc(dims, dtype, d_q)) return 0;
    return query_latent_tc_workspace(dims->hidden, d_q, batch, nullptr, sm_count());
}

mla_status mla_project_query_latent(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t d_q,
                                    const void* h, const void* w_dq, void* workspace, size_t workspace_bytes,
                                    void* c_q, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || d_q < 1 || (int64_t)batch * d_q > (1LL << 30)) return MLA_ERR_INVALID_ARG;
    if (!h || !w_dq || !c_q || !dev_status) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (query_latent_tc(dims, dtype, d_q)) {
        const int sms = sm_count();
        const size_t need = query_latent_tc_workspace(dims->hidden, d_q, batch, nullptr, sms);
        if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
        if (!aligned(h, 16) || !aligned(w_dq, 16) || !aligned(c_q, 4)) return MLA_ERR_INVALID_ARG;
        return cuda_status(launch_query_latent_tc(dims->hidden, d_q, batch, h, w_dq, workspace, c_q,
                                                  dev_status, sms, s));
    }
    return cuda_status(launch_query_latent(*dims, dtype == MLA_BF16, batch, d_q, h, w_dq, c_q, s));
}

size_t mla_decode_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                 int32_t max_seq_len, int32_t num_splits) {
    // bf16 latent-shape calls use the tensor-core kernel unless the cache is smaller
    // than one tile, so size for whichever of the two kernels needs more.
    DecodePlan p;
    size_t need = 0;
    if (plan_decode(dims, dtype, batch, max_seq_len, num_splits, false, &p)) need = p.ws.total;
    if (dims_ok(dims) && dtype_ok(dtype) && tc_shape(dims, dtype) &&
        plan_decode(dims, dtype, batch, max_seq_len, num_splits, true, &p) && p.ws.total > need)
        need = p.ws.total;
    return need;
}

}  // extern "C"

namespace {

enum : int { kPrepare = 1, kAttend = 2, kBeside = 4 };

// The decode in two phases: kPrepare (fold W_UK^T into the queries, rotate q_R, build the
// schedule; reads no cache row) and kAttend (split-K attention over the cache, merge).
// `layout` (null: the packed contiguous cache `cache`) selects where the rows live; a
// layout other than packed contiguous runs on the tensor-core kernel only.
mla_status decode_phases(int phases, const mla_dims* dims, mla_dtype dtype, int32_t batch,
                         const void* q_c, const void* q_r, const void* w_uk,
                         const void* cache, int64_t cache_rows, const int64_t* row_off,
                         const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                         void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                         int32_t* dev_status, void* stream, const CacheView* layout = nullptr,
                         bool fp8 = false) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (fp8 && (dtype != MLA_BF16 || layout || dims->d_c % 128)) return MLA_ERR_UNSUPPORTED;
    if (batch < 1 || max_seq_len < 0 || num_splits < 0 || cache_rows < 1) return MLA_ERR_INVALID_ARG;
    if (!q_c || !q_r || !w_uk || !cache || (!row_off && !(layout && layout->block_table)) || !seq_len ||
        !o_lat || !dev_status)
        return MLA_ERR_INVALID_ARG;
    const size_t row_bytes = fp8 ? (size_t)kFp8RowBytes(dims->d_c, dims->d_r)
                                 : (size_t)(dims->d_c + dims->d_r) * elt(dtype);
    if (!aligned(cache, 16) || row_bytes % 16) return MLA_ERR_INVALID_ARG;
    // the fp8 layout runs on the tensor-core kernel for its shapes, on CUDA cores otherwise
    const bool tc = tc_shape(dims, dtype) && cache_rows >= 32 && cache_rows <= INT32_MAX;
    if (!tc && !simt_supported(dims)) return MLA_ERR_UNSUPPORTED;
    if (layout && !tc) return MLA_ERR_UNSUPPORTED;
    CacheView cv{cache, nullptr, dims->d_c + dims->d_r, 0, cache_rows, nullptr, 0, 0};
    if (layout) cv = *layout;
    DecodePlan p;
    if (!plan_decode(dims, dtype, batch, max_seq_len, num_splits, tc, &p)) return MLA_ERR_CUDA;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < p.ws.total)
        return MLA_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    void* qp = ws + p.ws.q_off;
    int64_t* cum = (int64_t*)(ws + p.ws.cum_off);
    void* sched = ws + p.ws.sched_off;
    WorkerStart* wstart = (WorkerStart*)(ws + p.ws.ws_off);
    float* part_o = (float*)(ws + p.ws.po_off);
    float* part_l = (float*)(ws + p.ws.pl_off);
    const bool bf16 = dtype == MLA_BF16;
    const float alpha = scale_of(dims) * kLog2e;
    cudaError_t e = cudaSuccess;
    // a paged cache flattens the context in whole tiles, so no tile crosses a block
    const ScheduleArgs sa{seq_len, row_off, cache_rows, batch, p.workers, cum, (Schedule*)sched, wstart,
                          dev_status, cv.block_table ? 64 : 1,
                          cv.block_table ? (int64_t)cv.max_blocks * cv.block_size : 0};
    if (phases & kPrepare) {
        if (tc && gemm_tc_shapes_ok(*dims) && aligned(q_c, 16) && aligned(w_uk, 16)) {
            // fold GEMM, then q_R rotation and the schedule in one launch
            // the rotation and schedule kernel runs beside the fold GEMM (programmatic
            // dependent launch; it waits for the GEMM only at its end)
            e = launch_fold_tc(*dims, batch, q_c, w_uk, alpha, qp, dev_status, s, (phases & kBeside) != 0);
            if (e == cudaSuccess)
                e = launch_fold_rope(*dims, true, true, batch, q_r, seq_len, alpha, qp, s, &sa, true);
        } else {
            e = launch_fold(*dims, bf16, tc, batch, q_c, q_r, w_uk, seq_len, alpha, qp, s);
            if (e == cudaSuccess) e = launch_schedule(sa, s);
        }
    }
    if (e == cudaSuccess && (phases & kAttend)) {
        if (tc) {
            // the attention kernel may start (set-up only) before the kernel before it on the
            // stream ends: it waits for that kernel before it reads anything
            e = launch_split_tc(*dims, batch, p.workers, qp, p.q_rows, cv, seq_len, row_off, cum,
                                sched, wstart, o_lat, lse, part_o, part_l, dev_status, s, true, fp8);
        } else {
            e = launch_split_simt(*dims, bf16, batch, p.workers, (const float*)qp, cache, row_off, cum,
                                  sched, wstart, o_lat, lse, part_o, part_l, s, fp8);
        }
        // the merge kernel follows the attention kernel of this same call (programmatic
        // dependent launch: it is scheduled early and waits for it)
        if (e == cudaSuccess)
            e = launch_merge(*dims, bf16, batch, cum, sched, part_o, part_l, o_lat, lse, s, true);
    }
    return cuda_status(e);
}

}  // namespace

extern "C" {

mla_status mla_decode_absorbed(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                               const void* q_c, const void* q_r, const void* w_uk,
                               const void* cache, int64_t cache_rows, const int64_t* row_off,
                               const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                               void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                               int32_t* dev_status, void* stream) {
    return decode_phases(kPrepare | kAttend, dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off,
                         seq_len, max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                         stream);
}

// Several causal queries per sequence: query j of sequence b sits at position
// seq_len[b] - n_q + j and attends over rows 0 .. that position.  Each query becomes a
// sequence of its own for the decode (same cache rows, its own length), so the same
// kernels run on batch * n_q sequences; the expanded row offsets and lengths sit at the
// start of the workspace, the decode's own workspace after them.
static size_t multi_index_bytes(int64_t n) {
    return align_up((size_t)n * sizeof(int64_t), 256) + align_up((size_t)n * sizeof(int32_t), 256);
}

size_t mla_decode_multi_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_q,
                                       int32_t max_seq_len, int32_t num_splits) {
    if (batch < 1 || n_q < 1 || (int64_t)batch * n_q > (1 << 30)) return 0;
    const size_t dec = mla_decode_workspace_size(dims, dtype, batch * n_q, max_seq_len, num_splits);
    return dec ? multi_index_bytes((int64_t)batch * n_q) + dec : 0;
}

mla_status mla_decode_absorbed_multi(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_q,
                                     const void* q_c, const void* q_r, const void* w_uk,
                                     const void* cache, int64_t cache_rows, const int64_t* row_off,
                                     const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                                     void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                                     int32_t* dev_status, void* stream) {
    if (batch < 1 || n_q < 1 || (int64_t)batch * n_q > (1 << 30)) return MLA_ERR_INVALID_ARG;
    if (!row_off || !seq_len || !dev_status) return MLA_ERR_INVALID_ARG;
    const int64_t nv = (int64_t)batch * n_q;
    const size_t idx = multi_index_bytes(nv);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < idx) return MLA_ERR_WORKSPACE;
    int64_t* row_off_v = (int64_t*)workspace;
    int32_t* seq_len_v = (int32_t*)((char*)workspace + align_up((size_t)nv * sizeof(int64_t), 256));
    // host checks of the decode first (nothing is enqueued when they fail)
    DecodePlan p;
    if (!dims_ok(dims) || !dtype_ok(dtype) || max_seq_len < 0 || num_splits < 0) return MLA_ERR_INVALID_ARG;
    if (!plan_decode(dims, dtype, (int)nv, max_seq_len, num_splits,
                     tc_shape(dims, dtype) && cache_rows >= 32 && cache_rows <= INT32_MAX, &p))
        return tc_shape(dims, dtype) || simt_supported(dims) ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED;
    if (workspace_bytes - idx < p.ws.total) return MLA_ERR_WORKSPACE;
    cudaError_t e = launch_expand_queries(row_off, seq_len, batch, n_q, row_off_v, seq_len_v, (cudaStream_t)stream);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return decode_phases(kPrepare | kAttend, dims, dtype, (int32_t)nv, q_c, q_r, w_uk, cache, cache_rows, row_off_v,
                         seq_len_v, max_seq_len, num_splits, (char*)workspace + idx, workspace_bytes - idx, o_lat,
                         lse, dev_status, stream);
}

// Checks a caller's cache layout for the tensor-core shapes (d_c = 512, d_r = 64) and
// turns it into the internal view.
static mla_status view_of(const mla_dims* d, const mla_cache_layout* c, CacheView* v) {
    if (!c || !c->kv || c->rows < 32 || c->rows > INT32_MAX) return MLA_ERR_INVALID_ARG;
    const int64_t kv_need = c->pe ? d->d_c : d->d_c + d->d_r;
    if (c->kv_stride < kv_need || c->kv_stride % 8 || !aligned(c->kv, 16)) return MLA_ERR_INVALID_ARG;
    if (c->pe && (c->pe_stride < d->d_r || c->pe_stride % 8 || !aligned(c->pe, 16))) return MLA_ERR_INVALID_ARG;
    if (c->block_table && (c->block_size < 64 || c->block_size % 64 || c->max_blocks < 1))
        return MLA_ERR_INVALID_ARG;
    *v = CacheView{c->kv, c->pe, c->kv_stride, c->pe ? c->pe_stride : 0, c->rows, c->block_table,
                   c->block_table ? c->block_size : 0, c->block_table ? c->max_blocks : 0};
    return MLA_OK;
}

mla_status mla_cache_append_ex(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_new,
                               const void* h, const void* w_dkv, const void* w_kr, const mla_cache_layout* cache,
                               const int64_t* row_off, const int32_t* cap, const int32_t* pos0, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || n_new < 1 || (int64_t)batch * n_new > (1LL << 30)) return MLA_ERR_INVALID_ARG;
    if (!h || !w_dkv || !w_kr || !cap || !pos0 || !dev_status) return MLA_ERR_INVALID_ARG;
    if (!tc_shape(dims, dtype) || !gemm_tc_shapes_ok(*dims)) return MLA_ERR_UNSUPPORTED;
    CacheView cv;
    const mla_status st = view_of(dims, cache, &cv);
    if (st != MLA_OK) return st;
    if (!cv.block_table && !row_off) return MLA_ERR_INVALID_ARG;
    const int sms = sm_count();
    const size_t need = append_tc_workspace(*dims, batch * n_new, nullptr, sms);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
    if (!aligned(h, 16) || !aligned(w_dkv, 16) || !aligned(w_kr, 16)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_append_tc(*dims, batch, n_new, h, w_dkv, w_kr, row_off, cap, pos0, cv, workspace,
                                        dev_status, sms, (cudaStream_t)stream));
}

mla_status mla_decode_absorbed_ex(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                  const void* q_c, const void* q_r, const void* w_uk, const mla_cache_layout* cache,
                                  const int64_t* row_off, const int32_t* seq_len, int32_t max_seq_len,
                                  int32_t num_splits, void* workspace, size_t workspace_bytes, void* o_lat,
                                  float* lse, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (!tc_shape(dims, dtype)) return MLA_ERR_UNSUPPORTED;
    CacheView cv;
    const mla_status st = view_of(dims, cache, &cv);
    if (st != MLA_OK) return st;
    return decode_phases(kPrepare | kAttend, dims, dtype, batch, q_c, q_r, w_uk, cv.kv, cv.rows, row_off, seq_len,
                         max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status, stream, &cv);
}

mla_status mla_cache_append_fp8(const mla_dims* dims, int32_t batch, int32_t n_new, const void* h,
                                const void* w_dkv, const void* w_kr, const int64_t* row_off, const int32_t* cap,
                                const int32_t* pos0, void* cache, int64_t cache_rows, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || n_new < 1 || (int64_t)batch * n_new > (1LL << 30) || cache_rows < 1) return MLA_ERR_INVALID_ARG;
    if (!h || !w_dkv || !w_kr || !row_off || !cap || !pos0 || !cache || !dev_status) return MLA_ERR_INVALID_ARG;
    if (!tc_shape(dims, MLA_BF16) || !gemm_tc_shapes_ok(*dims) || dims->d_c % 128) return MLA_ERR_UNSUPPORTED;
    if (!aligned(cache, 16) || kFp8RowBytes(dims->d_c, dims->d_r) % 16) return MLA_ERR_INVALID_ARG;
    const int sms = sm_count();
    const size_t need = append_tc_workspace(*dims, batch * n_new, nullptr, sms);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
    if (!aligned(h, 16) || !aligned(w_dkv, 16) || !aligned(w_kr, 16)) return MLA_ERR_INVALID_ARG;
    return cuda_status(launch_append_fp8_tc(*dims, batch, n_new, h, w_dkv, w_kr, row_off, cap, pos0, cache,
                                            cache_rows, workspace, dev_status, sms, (cudaStream_t)stream));
}

mla_status mla_decode_absorbed_fp8(const mla_dims* dims, int32_t batch, const void* q_c, const void* q_r,
                                   const void* w_uk, const void* cache, int64_t cache_rows, const int64_t* row_off,
                                   const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits, void* workspace,
                                   size_t workspace_bytes, void* o_lat, float* lse, int32_t* dev_status,
                                   void* stream) {
    return decode_phases(kPrepare | kAttend, dims, MLA_BF16, batch, q_c, q_r, w_uk, cache, cache_rows, row_off,
                         seq_len, max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status, stream,
                         nullptr, true);
}

mla_status mla_decode_prepare(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                              const void* q_c, const void* q_r, const void* w_uk,
                              const void* cache, int64_t cache_rows, const int64_t* row_off,
                              const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                              void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                              int32_t* dev_status, void* stream) {
    return decode_phases(kPrepare, dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off,
                         seq_len, max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                         stream);
}

mla_status mla_decode_prepare_beside(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                     const void* q_c, const void* q_r, const void* w_uk,
                                     const void* cache, int64_t cache_rows, const int64_t* row_off,
                                     const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                                     void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                                     int32_t* dev_status, void* stream) {
    return decode_phases(kPrepare | kBeside, dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off,
                         seq_len, max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                         stream);
}

mla_status mla_decode_attend(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                             const void* q_c, const void* q_r, const void* w_uk,
                             const void* cache, int64_t cache_rows, const int64_t* row_off,
                             const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                             void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                             int32_t* dev_status, void* stream) {
    return decode_phases(kAttend, dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off,
                         seq_len, max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                         stream);
}


mla_status mla_project_out(const mla_dims* dims, mla_dtype dtype, int32_t batch, const void* o_lat,
                           const void* w_uv, void* out, int32_t* dev_status, void* stream) {
    if (!dims_ok(dims) || !dtype_ok(dtype)) return MLA_ERR_INVALID_ARG;
    if (batch < 1 || !o_lat || !w_uv || !out || !dev_status) return MLA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == MLA_BF16 && gemm_tc_shapes_ok(*dims) && aligned(o_lat, 16) && aligned(w_uv, 16))
        return cuda_status(launch_project_out_tc(*dims, batch, o_lat, w_uv, out, dev_status, s));
    return cuda_status(launch_project_out(*dims, dtype == MLA_BF16, batch, o_lat, w_uv, out, s));
}

}  // extern "C"
