// Launch helpers shared between the kernel files and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

struct DecodeWorkspace;

cudaError_t launch_append(const mla_dims& d, bool bf16, int batch, int n_new, const void* h,
                          const void* w_dkv, const void* w_kr, const int64_t* row_off,
                          const int32_t* cap, const int32_t* pos0, void* cache, int64_t cache_rows,
                          int32_t* dev_status, cudaStream_t s);

cudaError_t launch_project_query(const mla_dims& d, bool bf16, int batch, int d_in, const void* x,
                                 const void* w_uq, const void* w_qr, void* q_c, void* q_r,
                                 cudaStream_t s);

// c_q = W_DQ h on CUDA cores (any shape)
cudaError_t launch_query_latent(const mla_dims& d, bool bf16, int batch, int d_q, const void* h,
                                const void* w_dq, void* c_q, cudaStream_t s);

// Q'[b, i, :] = alpha * [W_UK^(i)T q_C[b,i] ; RoPE(q_R[b,i], seq_len[b]-1)]
cudaError_t launch_fold(const mla_dims& d, bool in_bf16, bool out_bf16, int batch, const void* q_c,
                        const void* q_r, const void* w_uk, const int32_t* seq_len, float alpha,
                        void* qp, cudaStream_t s);

cudaError_t launch_project_out(const mla_dims& d, bool bf16, int batch, const void* o_lat,
                               const void* w_uv, void* out, cudaStream_t s);

// The rotary part of Q' alone (the content part comes from a GEMM).
struct ScheduleArgs;
struct WorkerStart;
// q_R rotation into Q'; with sched_args it also builds the split schedule (one extra
// block column), otherwise launch_schedule does.
cudaError_t launch_fold_rope(const mla_dims& d, bool in_bf16, bool out_bf16, int batch, const void* q_r,
                             const int32_t* seq_len, float alpha, void* qp, cudaStream_t s,
                             const ScheduleArgs* sched_args, bool pdl);

// tcgen05 projections (bf16; shapes accepted by gemm_tc_shapes_ok)
bool gemm_tc_shapes_ok(const mla_dims& d);
size_t append_tc_workspace(const mla_dims& d, int n_tok, int* k_splits_out, int sm_count);
struct CacheView;
// the append into the fp8 cache layout (contiguous rows of kFp8RowBytes bytes)
cudaError_t launch_append_fp8_tc(const mla_dims& d, int batch, int n_new, const void* h, const void* w_dkv,
                                 const void* w_kr, const int64_t* row_off, const int32_t* cap,
                                 const int32_t* pos0, void* cache, int64_t cache_rows, void* workspace,
                                 int32_t* dev_status, int sm_count, cudaStream_t s);
cudaError_t launch_append_tc(const mla_dims& d, int batch, int n_new, const void* h, const void* w_dkv,
                             const void* w_kr, const int64_t* row_off, const int32_t* cap,
                             const int32_t* pos0, const CacheView& cv, void* workspace,
                             int32_t* dev_status, int sm_count, cudaStream_t s);
size_t query_latent_tc_workspace(int hidden, int d_q, int n_tok, int* k_splits_out, int sm_count);
// c_q = W_DQ h on tensor cores (split-K GEMM, then a fixed-order reduction to bf16)
cudaError_t launch_query_latent_tc(int hidden, int d_q, int batch, const void* h, const void* w_dq,
                                   void* workspace, void* c_q, int32_t* dev_status, int sm_count,
                                   cudaStream_t s);
// [q_C ; q_R] = [W_UQ ; W_QR] x on tensor cores (one launch, two weight maps, two outputs)
cudaError_t launch_project_query_tc(const mla_dims& d, int batch, int d_in, const void* x, const void* w_uq,
                                    const void* w_qr, void* q_c, void* q_r, int32_t* dev_status,
                                    cudaStream_t s);
// Output projection after the decode (tensor cores, bf16): u = W_O o, the merged form
// u = W_OV o_lat, and the merge of the weights W_OV^(i) = W_O^(i) W_UV^(i).
size_t output_tc_workspace(int hidden, int k_in, int n_tok, int sm_count);
cudaError_t launch_output_tc(const mla_dims& d, int batch, const void* o, const void* w_o, void* workspace,
                             void* u, int32_t* dev_status, int sm_count, cudaStream_t s);
cudaError_t launch_output_merged_tc(const mla_dims& d, int batch, const void* o_lat, const void* w_ov,
                                    void* workspace, void* u, int32_t* dev_status, int sm_count, cudaStream_t s);
cudaError_t launch_merge_output_weights_tc(const mla_dims& d, const void* w_o, const void* w_uv, void* w_ov,
                                           int32_t* dev_status, cudaStream_t s);
// beside: the fold may run beside the kernel before it on the stream (that kernel writes
// nothing it reads); it waits for that kernel only at its end
cudaError_t launch_fold_tc(const mla_dims& d, int batch, const void* q_c, const void* w_uk, float alpha,
                           void* qp, int32_t* dev_status, cudaStream_t s, bool beside = false);
cudaError_t launch_project_out_tc(const mla_dims& d, int batch, const void* o_lat, const void* w_uv,
                                  void* out, int32_t* dev_status, cudaStream_t s);

// Work split of the flattened context: prefix sums of the usable sequence lengths and
// the Schedule, written into the workspace; flags unusable sequences.
cudaError_t launch_schedule(const ScheduleArgs& a, cudaStream_t s);

// One decode sequence per query of a multi-query call: query j of sequence b becomes
// sequence b*n_q + j with row offset row_off[b] and length seq_len[b] - n_q + j + 1.
cudaError_t launch_expand_queries(const int64_t* row_off, const int32_t* seq_len, int batch, int n_q,
                                  int64_t* row_off_v, int32_t* seq_len_v, cudaStream_t s);

// fp32-Q' SIMT split kernel (any supported dims, fp32 or bf16 cache).
cudaError_t launch_split_simt(const mla_dims& d, bool bf16, int batch, int workers, const float* qp,
                              const void* cache, const int64_t* row_off, const int64_t* cum,
                              const void* sched, const WorkerStart* wstart, void* o_lat, float* lse,
                              float* part_o, float* part_l, cudaStream_t s, bool fp8 = false);

// bf16 tcgen05 split kernel for d_c = 512, d_r = 64, n_heads <= 128 (2-CTA clusters).
cudaError_t launch_split_tc(const mla_dims& d, int batch, int workers, const void* qp,
                            int64_t q_rows, const CacheView& cv, const int32_t* seq_len,
                            const int64_t* row_off, const int64_t* cum, const void* sched,
                            const WorkerStart* wstart, void* o_lat, float* lse, float* part_o,
                            float* part_l, int32_t* dev_status, cudaStream_t s, bool pdl, bool fp8 = false);

// Combines the partial results of sequences cut across workers; zero-fills empty ones.
cudaError_t launch_merge(const mla_dims& d, bool bf16, int batch, const int64_t* cum,
                         const void* sched, const float* part_o, const float* part_l, void* o_lat,
                         float* lse, cudaStream_t s, bool pdl);

// Launch accounting and the optional per-thread timing hook around the split kernel.
void note_launch(int n = 1);
// Limit of the bounded waits of the pipelined kernels (mla_set_wait_limit_ns).
uint64_t wait_limit_ns();
void profile_before_split(cudaStream_t s);
void profile_after_split(cudaStream_t s);

int simt_workers(int batch, int n_heads, int64_t max_total_rows, int sm_count);
int tc_workers(int64_t max_total_rows, int sm_count);

}  // namespace mla
