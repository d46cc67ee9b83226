// Projection kernels around the attention core: cache append (W_DKV, W_KR + RoPE),
// query projection (W_UQ, W_QR), the key-side fold (W_UK^T) and the value-side
// up-projection (W_UV).  All four are batched products Y = X W^T with fp32
// accumulation; they differ only in strides and in what the epilogue does.
#include "mla_common.cuh"
#include "mla_internal.h"
#include "mla_schedule.cuh"

namespace mla {

namespace {

constexpr int BM = 32, BN = 64, BK = 32, NT = 256;

enum EpilogueMode : int { kPlain = 0, kAppend = 1 };

struct GemmArgs {
    const void* x; int64_t x_g, x_m;             // X[g,m,k] = x[g*x_g + m*x_m + k]
    const void* w; const void* w2; int32_t n_split;  // W[g,n,k]: rows n >= n_split from w2
    int64_t w_g, w_n, w_k;                       //   = w[g*w_g + n*w_n + k*w_k]
    void* y; int64_t y_g, y_m;                   // Y[g,m,n] = y[g*y_g + m*y_m + n]
    int32_t G, M, N, K;
    float alpha;
    int32_t mode;
    // append epilogue
    int32_t n_new, d_c, d_r;
    double rope_r;
    const int64_t* row_off; const int32_t* cap; const int32_t* pos0; int32_t* dev_status;
    int64_t cache_rows;
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(NT) gemm_xwt_kernel(GemmArgs a) {
    __shared__ float xs[BK][BM + 1];
    __shared__ float ws[BK][BN + 2];
    const int g = blockIdx.z;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    const Tin* X = (const Tin*)a.x + (int64_t)g * a.x_g;
    const Tin* W1 = (const Tin*)a.w + (int64_t)g * a.w_g;
    const Tin* W2 = a.w2 ? (const Tin*)a.w2 + (int64_t)g * a.w_g : nullptr;
    float acc[4][2] = {};
    for (int k0 = 0; k0 < a.K; k0 += BK) {
        for (int e = tid; e < BM * BK; e += NT) {
            int mm = e / BK, kk = e % BK;
            int m = m0 + mm, k = k0 + kk;
            xs[kk][mm] = (m < a.M && k < a.K) ? ld(X + (int64_t)m * a.x_m + k) : 0.f;
        }
        for (int e = tid; e < BN * BK; e += NT) {
            int nn, kk;
            if (a.w_k == 1) { nn = e / BK; kk = e % BK; } else { kk = e / BN; nn = e % BN; }
            int n = n0 + nn, k = k0 + kk;
            float v = 0.f;
            if (n < a.N && k < a.K) {
                const Tin* Wr = (n < a.n_split) ? W1 + (int64_t)n * a.w_n
                                                : W2 + (int64_t)(n - a.n_split) * a.w_n;
                v = ld(Wr + (int64_t)k * a.w_k);
            }
            ws[kk][nn] = v;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            float xv[4], wv[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = xs[kk][ty * 4 + i];
            wv[0] = ws[kk][tx * 2];
            wv[1] = ws[kk][tx * 2 + 1];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[i][0] = fmaf(xv[i], wv[0], acc[i][0]);
                acc[i][1] = fmaf(xv[i], wv[1], acc[i][1]);
            }
        }
        __syncthreads();
    }
    const int n = n0 + tx * 2;           // even: a rotary pair never straddles threads
    if (n >= a.N) return;
    const bool two = n + 1 < a.N;
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= a.M) break;
        float v0 = acc[i][0] * a.alpha, v1 = acc[i][1] * a.alpha;
        if (a.mode == kPlain) {
            Tout* Y = (Tout*)a.y + (int64_t)g * a.y_g + (int64_t)m * a.y_m + n;
            st(Y, v0);
            if (two) st(Y + 1, v1);
        } else {
            const int b = m / a.n_new, t = m % a.n_new;
            const int p0 = a.pos0[b];
            const int64_t off = a.row_off[b], cap = a.cap[b];
            if (p0 < 0 || (int64_t)p0 + a.n_new > cap || off < 0 || off + cap > a.cache_rows) {
                if (t == 0 && n == 0) atomicOr(a.dev_status, MLA_DEV_BAD_POSITION);
                continue;
            }
            const int64_t pos = (int64_t)p0 + t;
            const int row_elems = a.d_c + a.d_r;
            Tout* Y = (Tout*)a.y + (off + pos) * row_elems + n;
            if (n >= a.d_c) {            // k_R = RoPE(W_KR h, pos) on the pair (2k, 2k+1)
                float c, s;
                rope_cos_sin(pos, (n - a.d_c) >> 1, a.rope_r, &c, &s);
                float r0 = v0 * c - v1 * s, r1 = v0 * s + v1 * c;
                v0 = r0; v1 = r1;
            }
            st(Y, v0);
            if (two) st(Y + 1, v1);
        }
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
    dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, a.G);
    gemm_xwt_kernel<Tin, Tout><<<grid, NT, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_gemm_in(const GemmArgs& a, bool out_bf16, cudaStream_t s) {
    return out_bf16 ? launch_gemm<Tin, __nv_bfloat16>(a, s) : launch_gemm<Tin, float>(a, s);
}

cudaError_t dispatch(const GemmArgs& a, bool in_bf16, bool out_bf16, cudaStream_t s) {
    return in_bf16 ? launch_gemm_in<__nv_bfloat16>(a, out_bf16, s)
                   : launch_gemm_in<float>(a, out_bf16, s);
}

GemmArgs blank() {
    GemmArgs a{};
    a.n_split = 0x7fffffff;
    a.alpha = 1.f;
    a.mode = kPlain;
    return a;
}

// Q'[b, i, d_c + 2k .. 2k+1] = alpha * RoPE(q_R[b, i, :], seq_len[b] - 1) pair k.
// Grid (batch, head groups of kRopeHeads): the d_r/2 angles of a sequence are formed
// once per block in shared memory and shared by its heads; every thread then turns
// independent pairs (paired loads and stores, no dependence between iterations).
constexpr int kMaxRopePairs = 512;
constexpr int kRopeHeads = 16;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256) fold_rope_kernel(const Tin* __restrict__ q_r,
                                                        const int32_t* __restrict__ seq_len,
                                                        Tout* __restrict__ qp, int n_h, int d_c,
                                                        int d_r, double rope_r, float alpha,
                                                        ScheduleArgs sch) {
    __shared__ float cs[kMaxRopePairs], sn[kMaxRopePairs];
    // Launched right behind the fold GEMM (programmatic dependent launch), this kernel
    // touches nothing that GEMM reads or writes (the GEMM fills Q' columns [0, d_c), this
    // kernel columns [d_c, d_c + d_r) and the schedule), so it runs beside it and only
    // waits for it at the end: its own completion then implies the GEMM's, which is what
    // the attention kernel behind it waits for.
    pdl_trigger();
    const int b = blockIdx.x;
    if (b == gridDim.x - 1 && sch.cum) {
        // one extra column of blocks: its first block builds the split schedule, which
        // saves the decode a launch (it depends only on seq_len and row_off)
        if (blockIdx.y == 0) build_schedule(sch);
        pdl_wait();
        return;
    }
    const int h0 = blockIdx.y * kRopeHeads;
    const int half = d_r / 2;
    const int n_heads = min(kRopeHeads, n_h - h0);
    const int len = seq_len[b];
    const int64_t pos = len > 0 ? (int64_t)len - 1 : 0;
    for (int k = threadIdx.x; k < half; k += blockDim.x) rope_cos_sin(pos, k, rope_r, &cs[k], &sn[k]);
    __syncthreads();
    const int items = n_heads * half;
#pragma unroll 4
    for (int e = threadIdx.x; e < items; e += blockDim.x) {
        const int i = h0 + e / half, k = e % half;
        const float2 x = ld2(q_r + ((int64_t)b * n_h + i) * d_r + 2 * k);
        st2(qp + ((int64_t)b * n_h + i) * (d_c + d_r) + d_c + 2 * k,
            alpha * (x.x * cs[k] - x.y * sn[k]), alpha * (x.x * sn[k] + x.y * cs[k]));
    }
    pdl_wait();
}

}  // namespace

cudaError_t launch_append(const mla_dims& d, bool bf16, int batch, int n_new, const void* h,
                          const void* w_dkv, const void* w_kr, const int64_t* row_off,
                          const int32_t* cap, const int32_t* pos0, void* cache, int64_t cache_rows,
                          int32_t* dev_status, cudaStream_t s) {
    GemmArgs a = blank();
    a.cache_rows = cache_rows;
    a.x = h; a.x_g = 0; a.x_m = d.hidden;
    a.w = w_dkv; a.w2 = w_kr; a.n_split = d.d_c;
    a.w_g = 0; a.w_n = d.hidden; a.w_k = 1;
    a.y = cache;
    a.G = 1; a.M = batch * n_new; a.N = d.d_c + d.d_r; a.K = d.hidden;
    a.mode = kAppend; a.n_new = n_new; a.d_c = d.d_c; a.d_r = d.d_r; a.rope_r = rope_ratio(d.rope_base, d.d_r);
    a.row_off = row_off; a.cap = cap; a.pos0 = pos0; a.dev_status = dev_status;
    return dispatch(a, bf16, bf16, s);
}

cudaError_t launch_project_query(const mla_dims& d, bool bf16, int batch, int d_in, const void* x,
                                 const void* w_uq, const void* w_qr, void* q_c, void* q_r,
                                 cudaStream_t s) {
    GemmArgs a = blank();
    a.x = x; a.x_m = d_in;
    a.w = w_uq; a.w_n = d_in; a.w_k = 1;
    a.y = q_c; a.y_m = (int64_t)d.n_heads * d.d_h;
    a.G = 1; a.M = batch; a.N = d.n_heads * d.d_h; a.K = d_in;
    cudaError_t e = dispatch(a, bf16, bf16, s);
    if (e != cudaSuccess) return e;
    a.w = w_qr; a.y = q_r; a.y_m = (int64_t)d.n_heads * d.d_r; a.N = d.n_heads * d.d_r;
    return dispatch(a, bf16, bf16, s);
}

cudaError_t launch_query_latent(const mla_dims& d, bool bf16, int batch, int d_q, const void* h,
                                const void* w_dq, void* c_q, cudaStream_t s) {
    GemmArgs a = blank();
    a.x = h; a.x_m = d.hidden;
    a.w = w_dq; a.w_n = d.hidden; a.w_k = 1;
    a.y = c_q; a.y_m = d_q;
    a.G = 1; a.M = batch; a.N = d_q; a.K = d.hidden;
    return dispatch(a, bf16, bf16, s);
}

cudaError_t launch_fold(const mla_dims& d, bool in_bf16, bool out_bf16, int batch, const void* q_c,
                        const void* q_r, const void* w_uk, const int32_t* seq_len, float alpha,
                        void* qp, cudaStream_t s) {
    const int dq = d.d_c + d.d_r;
    GemmArgs a = blank();
    a.x = q_c; a.x_g = d.d_h; a.x_m = (int64_t)d.n_heads * d.d_h;
    a.w = w_uk; a.w_g = (int64_t)d.d_h * d.d_c; a.w_n = 1; a.w_k = d.d_c;
    a.y = qp; a.y_g = dq; a.y_m = (int64_t)d.n_heads * dq;
    a.G = d.n_heads; a.M = batch; a.N = d.d_c; a.K = d.d_h;
    a.alpha = alpha;
    cudaError_t e = dispatch(a, in_bf16, out_bf16, s);
    if (e != cudaSuccess) return e;
    return launch_fold_rope(d, in_bf16, out_bf16, batch, q_r, seq_len, alpha, qp, s, nullptr, false);
}

cudaError_t launch_fold_rope(const mla_dims& d, bool in_bf16, bool out_bf16, int batch, const void* q_r,
                             const int32_t* seq_len, float alpha, void* qp, cudaStream_t s,
                             const ScheduleArgs* sched_args, bool pdl) {
    if (d.d_r / 2 > kMaxRopePairs) return cudaErrorInvalidValue;
    ScheduleArgs sch{};
    if (sched_args) sch = *sched_args;
    const dim3 grid(batch + (sched_args ? 1 : 0), (d.n_heads + kRopeHeads - 1) / kRopeHeads);
    const double r = rope_ratio(d.rope_base, d.d_r);
    cudaError_t e;
    if (in_bf16) {
        if (out_bf16)
            e = launch_ex(fold_rope_kernel<__nv_bfloat16, __nv_bfloat16>, grid, dim3(256), 0, s, pdl,
                          (const __nv_bfloat16*)q_r, seq_len, (__nv_bfloat16*)qp, d.n_heads, d.d_c, d.d_r, r,
                          alpha, sch);
        else
            e = launch_ex(fold_rope_kernel<__nv_bfloat16, float>, grid, dim3(256), 0, s, pdl,
                          (const __nv_bfloat16*)q_r, seq_len, (float*)qp, d.n_heads, d.d_c, d.d_r, r, alpha, sch);
    } else {
        e = launch_ex(fold_rope_kernel<float, float>, grid, dim3(256), 0, s, pdl, (const float*)q_r, seq_len,
                      (float*)qp, d.n_heads, d.d_c, d.d_r, r, alpha, sch);
    }
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_project_out(const mla_dims& d, bool bf16, int batch, const void* o_lat,
                               const void* w_uv, void* out, cudaStream_t s) {
    GemmArgs a = blank();
    a.x = o_lat; a.x_g = d.d_c; a.x_m = (int64_t)d.n_heads * d.d_c;
    a.w = w_uv; a.w_g = (int64_t)d.d_h * d.d_c; a.w_n = d.d_c; a.w_k = 1;
    a.y = out; a.y_g = d.d_h; a.y_m = (int64_t)d.n_heads * d.d_h;
    a.G = d.n_heads; a.M = batch; a.N = d.d_h; a.K = d.d_c;
    return dispatch(a, bf16, bf16, s);
}

}  // namespace mla
