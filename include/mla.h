/*
 * mla.h -- C ABI of the absorbed Multi-Head Latent Attention (MLA) decode library
 * for NVIDIA B300 (sm_103a).
 *
 * The operations follow the column-vector equations of "Grouped-query and latent
 * attention" (sections "Multi-head latent attention", "The absorption trick" and
 * "Why a separate rotary key"):
 *
 *   c     = W_DKV h                      latent, d_c numbers, cached
 *   k_R   = RoPE(W_KR h, pos)            rotary key, d_r numbers, cached, shared by heads
 *   q'_i  = W_UK^(i)T q_C,i              query folded through the key up-projection
 *   s_ij  = (q'_i . c_j + RoPE(q_R,i, p) . k_R,j) / sqrt(d_h + d_r)
 *   o_lat_i = sum_j softmax_j(s_ij) c_j  latent weighted sum
 *   o_i   = W_UV^(i) o_lat_i             value up-projection
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer (cudaMalloc'd or equivalent) except
 *   `dims`, which points to host memory.  The caller owns all memory; the library
 *   allocates nothing, frees nothing and never synchronises.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   Every call only enqueues work on that stream and returns.
 * - Element type: `dtype` selects the storage type of weights, activations, the
 *   latent cache and the outputs (fp32 or bf16).  Accumulation is always fp32.
 *   `lse` is always fp32.
 * - All arrays are dense row-major with the shapes given in brackets.  Weights use
 *   the column convention y = W x, so W is [out, in]; the per-head blocks
 *   W_UK^(i), W_UV^(i) (rows i*d_h .. (i+1)*d_h-1 of a (n_h*d_h) x d_c matrix)
 *   are stored as [n_h, d_h, d_c].
 * - Latent cache: one buffer of rows of (d_c + d_r) elements, each row laid out as
 *   [c ; k_R] ("MLA storage", section "Storing a positional key separately").
 *   Sequence b owns rows row_off[b] .. row_off[b] + cap[b] - 1; the token at
 *   position t of sequence b is row row_off[b] + t.  The cache base pointer and
 *   every row must be 16-byte aligned (row bytes a multiple of 16).
 * - Errors the host can detect (null pointers, bad sizes, unsupported shapes, a
 *   small workspace) are returned before anything is enqueued.  A failed launch
 *   returns MLA_ERR_CUDA.  Conditions only the device can see are OR-ed into
 *   *dev_status (MLA_DEV_* bits) and the affected outputs are left as documented;
 *   read it after synchronising.  No kernel traps, asserts or waits without bound.
 * - Rotary embedding pairs dimensions (2k, 2k+1) and turns them by pos*theta_k,
 *   theta_k = rope_base^(-2k/d_r).  The query of a sequence holding n rows sits at
 *   position n-1.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misaligned buffer */
    MLA_ERR_UNSUPPORTED = 2,  /* no kernel for this dims/dtype combination */
    MLA_ERR_WORKSPACE = 3,    /* workspace pointer null or smaller than required */
    MLA_ERR_CUDA = 4          /* a CUDA runtime call or a kernel launch failed */
} mla_status;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype;

/* Bits OR-ed into *dev_status by kernels. */
#define MLA_DEV_BAD_LENGTH   0x1  /* decode: seq_len[b] < 1; that sequence's outputs are zero, lse -inf */
#define MLA_DEV_BAD_POSITION 0x2  /* append: pos0[b] < 0 or pos0[b] + n_new > cap[b]; rows of b not written */
#define MLA_DEV_TIMEOUT      0x4  /* a bounded wait inside a kernel gave up; outputs undefined */
#define MLA_DEV_SMEM_ALIGN   0x8  /* the attention kernel's dynamic shared memory did not start on a
                                     1024-byte boundary (its swizzled tiles need one); it returned
                                     without work, outputs undefined */

typedef struct {
    int32_t n_heads;      /* n_h: attention heads */
    int32_t d_h;          /* per-head content key / value width */
    int32_t d_c;          /* latent width (cached) */
    int32_t d_r;          /* decoupled rotary key width (cached once per token), even */
    int32_t hidden;       /* width of the token input h */
    float rope_base;      /* rotary base, > 0 */
    float softmax_scale;  /* 0 selects 1/sqrt(d_h + d_r) */
} mla_dims;

/*
 * Where the latent cache lives, for mla_cache_append_ex and mla_decode_absorbed_ex (the
 * other calls take one packed contiguous buffer).  Two choices, freely combined:
 * - packed rows [c ; k_R] in kv (pe NULL), or the latents in kv and the rotary keys in a
 *   buffer of their own, pe, row for row ("DeepSeek MLA: 4 Attention Methods Compared",
 *   section "Why DeepSeek reconstruction does not erase the MLA benefit": separate
 *   kv_cache and pe_cache);
 * - contiguous sequences (block_table NULL: position t of sequence b is row row_off[b] + t)
 *   or a paged cache ("The Journey to Multi-Head Latent Attention", section "Why the KV
 *   cache explodes": paged attention): position t of sequence b is row
 *   block_table[b * max_blocks + t / block_size] * block_size + t % block_size.
 * Rows are bf16, 16-byte aligned, in DeepSeek's shape (d_c = 512, d_r = 64).
 */
typedef struct {
    void* kv;                   /* latent rows (d_c elements each), or packed rows when pe is NULL */
    void* pe;                   /* rotary-key rows (d_r elements each), or NULL */
    int64_t kv_stride;          /* elements from one kv row to the next: >= d_c (>= d_c + d_r packed), multiple of 8 */
    int64_t pe_stride;          /* elements from one pe row to the next: >= d_r, multiple of 8 */
    int64_t rows;               /* rows in kv (and in pe), at least 32 */
    const int32_t* block_table; /* device [batch, max_blocks] physical block of each logical block, or NULL */
    int32_t block_size;         /* rows per block, a positive multiple of 64 (paged only) */
    int32_t max_blocks;         /* block-table entries per sequence (paged only) */
} mla_cache_layout;

/*
 * mla_cache_append -- write the latent rows of new tokens into the cache.
 * Defines c = W_DKV h and k_R = RoPE(W_KR h, pos) ("Grouped-query and latent
 * attention", sections "Multi-head latent attention" and "Why a separate rotary
 * key"; "MLA storage", section "Storing a positional key separately").
 *
 *   h        [batch, n_new, hidden]   inputs of the new tokens
 *   w_dkv    [d_c, hidden]            down-projection
 *   w_kr     [d_r, hidden]            rotary key projection
 *   row_off  [batch] int64            first cache row of each sequence
 *   cap      [batch] int32            rows reserved for each sequence
 *   pos0     [batch] int32            position of the first new token of each sequence
 *   cache    rows of d_c + d_r        token t of sequence b goes to row
 *                                     row_off[b] + pos0[b] + t, rotated at position pos0[b] + t
 *   cache_rows                        rows in the cache buffer (host value, >= 1)
 *   workspace  device scratch of at least mla_append_workspace_size(dims, dtype, batch, n_new)
 *              bytes, 256-byte aligned (may be NULL when that size is 0); contents ignored
 *   dev_status int32 (device)         MLA_DEV_BAD_POSITION is OR-ed in for a sequence whose
 *                                     new rows would leave [0, cap[b]) or the buffer
 *                                     (row_off[b] < 0 or row_off[b] + cap[b] > cache_rows);
 *                                     its rows are skipped
 * Row values are rounded once from the fp32 accumulator to `dtype`.
 */
MLA_API mla_status mla_cache_append(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_new,
                            const void* h, const void* w_dkv, const void* w_kr,
                            const int64_t* row_off, const int32_t* cap, const int32_t* pos0,
                            void* cache, int64_t cache_rows, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * mla_cache_append_ex -- mla_cache_append into a cache described by `cache` (see
 * mla_cache_layout).  row_off is read only for a contiguous layout (may be NULL when
 * paged); cap[b] bounds the positions of sequence b as before, and a paged sequence also
 * needs cap[b] <= max_blocks * block_size and every written row inside the buffer
 * (MLA_DEV_BAD_POSITION otherwise, that row skipped).  Runs on tensor cores only: bf16,
 * d_c = 512, d_r = 64, d_h and hidden multiples of 128 and 64; MLA_ERR_UNSUPPORTED
 * otherwise.  Same workspace as mla_cache_append.
 */
MLA_API mla_status mla_cache_append_ex(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_new,
                               const void* h, const void* w_dkv, const void* w_kr,
                               const mla_cache_layout* cache, const int64_t* row_off, const int32_t* cap,
                               const int32_t* pos0, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/*
 * mla_append_workspace_size -- bytes of device workspace mla_cache_append needs (bf16
 * with tensor-core shapes splits the long hidden reduction across CTAs and keeps
 * fp32 partial sums there); 0 when no workspace is needed or the arguments are bad.
 */
MLA_API size_t mla_append_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                         int32_t n_new);

/*
 * mla_project_query_latent -- the query's own latent, c_q = W_DQ h ("Grouped-query and
 * latent attention", section "Multi-head latent attention": the query is compressed
 * like the keys and values, with a query latent of d_q = 1536 in DeepSeek-V3).
 *
 *   h      [batch, hidden]      the token inputs (one per sequence)
 *   w_dq   [d_q, hidden]        query down-projection
 *   workspace  device scratch of at least mla_query_latent_workspace_size(dims, dtype, batch,
 *              d_q) bytes, 256-byte aligned (may be NULL when that size is 0); contents ignored
 *   c_q    [batch, d_q]         out, rounded once from the fp32 accumulator to `dtype`
 *   dev_status                  MLA_DEV_TIMEOUT if a bounded wait expired
 * bf16 with d_q a multiple of 128 and hidden a multiple of 64 runs on tensor cores (the
 * long hidden reduction split across CTAs, partial sums added in a fixed order).
 */
MLA_API mla_status mla_project_query_latent(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t d_q,
                                    const void* h, const void* w_dq, void* workspace,
                                    size_t workspace_bytes, void* c_q, int32_t* dev_status,
                                    void* stream);

/* Bytes of workspace mla_project_query_latent needs (0: none, or bad arguments). */
MLA_API size_t mla_query_latent_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                               int32_t d_q);

/*
 * mla_project_query -- per-head query parts from a query input x (the query latent
 * c_q, or h itself when the model has no query down-projection): q_C = W_UQ x and
 * q_R = W_QR x, the latter NOT yet rotated (decode rotates it at the query's
 * position).  ("Grouped-query and latent attention", sections "Multi-head latent
 * attention" and "Why a separate rotary key".)
 *
 *   x     [batch, d_in]
 *   w_uq  [n_h*d_h, d_in]       w_qr [n_h*d_r, d_in]
 *   q_c   [batch, n_h, d_h]     q_r  [batch, n_h, d_r]
 *   dev_status                  MLA_DEV_TIMEOUT if a bounded wait expired
 * bf16 with n_h*d_h a multiple of 128, d_in a multiple of 64 and 16-byte aligned
 * buffers runs both products in one tensor-core launch; other shapes on CUDA cores.
 */
MLA_API mla_status mla_project_query(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t d_in,
                             const void* x, const void* w_uq, const void* w_qr,
                             void* q_c, void* q_r, int32_t* dev_status, void* stream);

/*
 * mla_decode_workspace_size -- bytes of device workspace mla_decode_absorbed needs
 * for these arguments (the same batch, max_seq_len and num_splits must be passed to
 * the decode call).  Returns 0 for arguments the decode would reject.
 */
MLA_API size_t mla_decode_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                 int32_t max_seq_len, int32_t num_splits);

/*
 * mla_decode_absorbed -- one decode query per sequence over that sequence's cached
 * rows, with the key-side and value-side absorption ("Grouped-query and latent
 * attention", section "The absorption trick"; scale from section "Why a separate
 * rotary key").  Full per-head keys and values are never formed.
 *
 *   q_c      [batch, n_h, d_h]     content query
 *   q_r      [batch, n_h, d_r]     rotary query, not yet rotated
 *   w_uk     [n_h, d_h, d_c]       key up-projection
 *   cache, cache_rows, row_off     as for mla_cache_append
 *   seq_len  [batch] int32         rows of each sequence (new token included); the query
 *                                  sits at position seq_len[b]-1 and attends over rows
 *                                  0 .. seq_len[b]-1
 *   max_seq_len  host int           upper bound used only to size the split grid
 *   num_splits   host int           number of context pieces the work is cut into
 *                                  (0 = choose from the GPU's SM count); results do not
 *                                  depend on it beyond fp32 rounding order
 *   workspace    device buffer of at least mla_decode_workspace_size(...) bytes, 256-byte
 *                aligned; contents on entry are ignored
 *   o_lat    [batch, n_h, d_c]     out: sum_j a_ij c_j, in `dtype`
 *   lse      [batch, n_h] fp32     out (may be NULL): natural log of sum_j exp(s_ij)
 *   dev_status                     MLA_DEV_BAD_LENGTH for seq_len[b] < 1 or rows outside
 *                                  the buffer (row_off[b] < 0 or row_off[b] + seq_len[b] >
 *                                  cache_rows): outputs of b zero, lse -inf;
 *                                  MLA_DEV_TIMEOUT if a bounded wait expired
 * bf16 with d_c = 512, d_r = 64, n_heads <= 128 and cache_rows >= 32 runs on the tcgen05
 * tensor-core kernel; every other supported shape runs on CUDA cores.
 */
MLA_API mla_status mla_decode_absorbed(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                               const void* q_c, const void* q_r, const void* w_uk,
                               const void* cache, int64_t cache_rows, const int64_t* row_off,
                               const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                               void* workspace, size_t workspace_bytes,
                               void* o_lat, float* lse, int32_t* dev_status, void* stream);

/*
 * mla_decode_absorbed_ex -- mla_decode_absorbed over a cache described by `cache` (see
 * mla_cache_layout); row_off is read only for a contiguous layout.  A paged sequence is
 * usable when 1 <= seq_len[b] <= max_blocks * block_size (MLA_DEV_BAD_LENGTH otherwise);
 * block-table entries are not checked: a block outside the buffer reads as zeros.  Runs
 * on the tensor-core kernel only (bf16, d_c = 512, d_r = 64, n_heads <= 128);
 * MLA_ERR_UNSUPPORTED otherwise.  Same workspace as mla_decode_absorbed.
 */
MLA_API mla_status mla_decode_absorbed_ex(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                  const void* q_c, const void* q_r, const void* w_uk,
                                  const mla_cache_layout* cache, const int64_t* row_off,
                                  const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                                  void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                                  int32_t* dev_status, void* stream);

/*
 * mla_decode_absorbed_multi -- n_q causal queries per sequence (several new tokens decoded
 * at once, as in a verification step of speculative decoding or a short chunk of prefill):
 * query j of sequence b sits at position seq_len[b] - n_q + j and attends over rows
 * 0 .. that position, with the absorption of mla_decode_absorbed ("Grouped-query and
 * latent attention", section "The absorption trick"; the causal rule of "The Journey to
 * Multi-Head Latent Attention", section "The KV cache": a token attends to itself and
 * every earlier token).
 *
 *   q_c  [batch, n_q, n_h, d_h]    q_r [batch, n_q, n_h, d_r] (not yet rotated)
 *   o_lat [batch, n_q, n_h, d_c]   lse [batch, n_q, n_h] (may be NULL)
 *   workspace  at least mla_decode_multi_workspace_size(dims, dtype, batch, n_q, max_seq_len,
 *              num_splits) bytes, 256-byte aligned
 * Every other argument is as for mla_decode_absorbed.  Each query is decoded as a sequence
 * of its own over the shared cache rows (the rows a chunk of queries shares are read once
 * per query).  A query whose position would be negative (seq_len[b] < n_q) counts as an
 * empty sequence: MLA_DEV_BAD_LENGTH, zero outputs, lse -inf.
 */
MLA_API mla_status mla_decode_absorbed_multi(const mla_dims* dims, mla_dtype dtype, int32_t batch, int32_t n_q,
                                     const void* q_c, const void* q_r, const void* w_uk,
                                     const void* cache, int64_t cache_rows, const int64_t* row_off,
                                     const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                                     void* workspace, size_t workspace_bytes,
                                     void* o_lat, float* lse, int32_t* dev_status, void* stream);

/* Bytes of workspace mla_decode_absorbed_multi needs (0 for arguments it would reject). */
MLA_API size_t mla_decode_multi_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                               int32_t n_q, int32_t max_seq_len, int32_t num_splits);

/*
 * fp8 latent cache.  The pages name quantization among the things a cache layout may add
 * ("DeepSeek MLA: 4 Attention Methods Compared", section "Memory savings do not
 * automatically equal latency savings") without fixing a format; this library's reading:
 * one contiguous row of MLA_FP8_ROW_BYTES(d_c, d_r) bytes per token,
 *   bytes [0, d_c)                      FP8 E4M3 codes of the latent c, in groups of 128
 *                                       columns
 *   bytes [d_c, d_c + 4 d_c/128)        one scale per group, stored as fp32: the smallest
 *                                       power of two 2^k with the group's largest |c| /
 *                                       2^k <= 448 (1 for a group of zeros); c = code * scale
 *   bytes [d_c + 4 d_c/128, + 2 d_r)    the rotary part k_R in bf16
 * (DeepSeek-V3 shapes: 512 + 16 + 128 = 656 bytes, against 1,152 for a bf16 row).  Rows
 * are addressed like the packed contiguous cache: token t of sequence b is row
 * row_off[b] + t.  Requires d_c % 128 == 0 and a row size that is a multiple of 16.
 *
 * mla_cache_append_fp8 -- mla_cache_append (bf16 h and weights, tensor-core shapes) that
 *   writes fp8 rows: the fp32 row is formed exactly as for a bf16 cache, then each group's
 *   scale is found in fp32 and its codes are x / scale rounded to nearest even.
 *   workspace: mla_append_workspace_size(dims, MLA_BF16, batch, n_new) bytes.
 * mla_decode_absorbed_fp8 -- mla_decode_absorbed over an fp8 cache (bf16 queries, weights
 *   and o_lat).  For DeepSeek-V3 shapes (d_c = 512, d_r = 64, up to 128 heads, at least 32
 *   cache rows) the attention runs on tensor cores: each landed tile's codes are turned into
 *   bf16 (code * scale, exact since the scale is a power of two) in shared memory; otherwise
 *   on CUDA cores.  workspace: mla_decode_workspace_size(dims, MLA_BF16, ...) bytes.
 * Arguments, errors and dev_status flags otherwise as for the bf16 calls; MLA_ERR_UNSUPPORTED
 * for shapes outside the above.
 */
#define MLA_FP8_ROW_BYTES(d_c, d_r) ((d_c) + 4 * ((d_c) / 128) + 2 * (d_r))
MLA_API mla_status mla_cache_append_fp8(const mla_dims* dims, int32_t batch, int32_t n_new, const void* h,
                                        const void* w_dkv, const void* w_kr, const int64_t* row_off,
                                        const int32_t* cap, const int32_t* pos0, void* cache, int64_t cache_rows,
                                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                        void* stream);
MLA_API mla_status mla_decode_absorbed_fp8(const mla_dims* dims, int32_t batch, const void* q_c,
                                           const void* q_r, const void* w_uk, const void* cache,
                                           int64_t cache_rows, const int64_t* row_off, const int32_t* seq_len,
                                           int32_t max_seq_len, int32_t num_splits, void* workspace,
                                           size_t workspace_bytes, void* o_lat, float* lse, int32_t* dev_status,
                                           void* stream);

/*
 * mla_decode_prepare, mla_decode_attend -- mla_decode_absorbed in two calls, so that the
 * query-side work can run beside the cache append of the same step (the fold reads no
 * cache row).  Both take exactly the arguments of mla_decode_absorbed, and the two calls
 * together have exactly its effect:
 *   mla_decode_prepare  folds W_UK^T into the queries, rotates q_r and builds the split
 *                       schedule, all into `workspace`; it reads q_c, q_r, w_uk, row_off and
 *                       seq_len but no cache row, and writes neither o_lat nor lse;
 *   mla_decode_attend   runs the split-K attention over the cache and the merge, reading
 *                       what mla_decode_prepare left in `workspace`; it must follow that
 *                       call in stream order, with identical arguments and an untouched
 *                       workspace, and after every cache row it attends over is written.
 * Errors and dev_status flags are those of mla_decode_absorbed.
 */
MLA_API mla_status mla_decode_prepare(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                              const void* q_c, const void* q_r, const void* w_uk,
                              const void* cache, int64_t cache_rows, const int64_t* row_off,
                              const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                              void* workspace, size_t workspace_bytes,
                              void* o_lat, float* lse, int32_t* dev_status, void* stream);
/*
 * mla_decode_prepare_beside -- mla_decode_prepare whose kernels may start while the
 * kernels of the library call enqueued just before it on `stream` are still running (for
 * instance the cache append of the same step), so that the two run side by side on one
 * stream.  The caller guarantees that that call writes none of what this call reads
 * (q_c, q_r, w_uk, row_off, seq_len) and does not use `workspace`.  Work enqueued before
 * that call is complete when a kernel of this call starts (the library's kernels that wait
 * for the kernel before them let the next one start only after that wait), and every
 * kernel of this call ends only after that call's kernels have ended, so work enqueued
 * behind it (such as mla_decode_attend) still sees everything before it complete.  Same arguments, errors
 * and effect as mla_decode_prepare.  Launch scheduling of the library, no step of the
 * method.
 */
MLA_API mla_status mla_decode_prepare_beside(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                              const void* q_c, const void* q_r, const void* w_uk,
                              const void* cache, int64_t cache_rows, const int64_t* row_off,
                              const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                              void* workspace, size_t workspace_bytes,
                              void* o_lat, float* lse, int32_t* dev_status, void* stream);
MLA_API mla_status mla_decode_attend(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                             const void* q_c, const void* q_r, const void* w_uk,
                             const void* cache, int64_t cache_rows, const int64_t* row_off,
                             const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                             void* workspace, size_t workspace_bytes,
                             void* o_lat, float* lse, int32_t* dev_status, void* stream);

/*
 * mla_project_out -- o_i = W_UV^(i) o_lat_i for every head ("Grouped-query and
 * latent attention", section "The absorption trick", value side).
 *
 *   o_lat [batch, n_h, d_c]    w_uv [n_h, d_h, d_c]    out [batch, n_h, d_h]
 *   dev_status                 MLA_DEV_TIMEOUT if a bounded wait expired
 */
MLA_API mla_status mla_project_out(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                           const void* o_lat, const void* w_uv, void* out, int32_t* dev_status,
                           void* stream);

/*
 * mla_project_output -- the attention layer's output u = W_O [o_1 ; ... ; o_n_h] after the
 * per-head value up-projection (mla_project_out), the two-step form of "Grouped-query and
 * latent attention", section "The absorption trick" (value side).
 *
 *   o     [batch, n_h, d_h]       per-head outputs (from mla_project_out)
 *   w_o   [hidden, n_h*d_h]       output projection
 *   u     [batch, hidden]         out, rounded once from the fp32 sums
 *   workspace  at least mla_output_workspace_size(dims, dtype, batch, 0) bytes, 256-byte aligned
 *   dev_status                    MLA_DEV_TIMEOUT if a bounded wait expired
 * bf16 with d_h, d_c and hidden multiples of 128 (tensor cores); MLA_ERR_UNSUPPORTED otherwise.
 */
MLA_API mla_status mla_project_output(const mla_dims* dims, mla_dtype dtype, int32_t batch, const void* o,
                              const void* w_o, void* workspace, size_t workspace_bytes, void* u,
                              int32_t* dev_status, void* stream);

/*
 * mla_merge_output_weights -- W_UV merged into W_O ("Grouped-query and latent attention",
 * section "The absorption trick": the value up-projection can be merged into the output
 * matrix; "The Journey to Multi-Head Latent Attention", section "The absorption trick"):
 * W_OV^(i) = W_O^(i) W_UV^(i), with W_O^(i) the columns i*d_h .. (i+1)*d_h - 1 of W_O.
 * A one-time preparation of the weights.
 *
 *   w_o   [hidden, n_h*d_h]    w_uv [n_h, d_h, d_c]
 *   w_ov  [n_h, d_c, hidden]   out: element (i, c, m) = sum_k W_O[m, i*d_h + k] W_UV[i, k, c]
 * Same shape rule as mla_project_output.
 */
MLA_API mla_status mla_merge_output_weights(const mla_dims* dims, mla_dtype dtype, const void* w_o,
                                    const void* w_uv, void* w_ov, int32_t* dev_status, void* stream);

/*
 * mla_project_output_merged -- u = sum_i W_OV^(i) o_lat_i straight from the decode's latent
 * output (no per-head o), with the merged weights of mla_merge_output_weights.  It reads
 * n_h*d_c*hidden weights instead of n_h*d_h*(d_c + hidden): for DeepSeek-V3 shapes
 * (128 heads, d_h 128, d_c 512, hidden 7168) 939 MB against 252 MB in bf16, so the
 * two-step form moves fewer bytes per decode step.
 *
 *   o_lat [batch, n_h, d_c]    w_ov [n_h, d_c, hidden]    u [batch, hidden]
 *   workspace  at least mla_output_workspace_size(dims, dtype, batch, 1) bytes, 256-byte aligned
 */
MLA_API mla_status mla_project_output_merged(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                     const void* o_lat, const void* w_ov, void* workspace,
                                     size_t workspace_bytes, void* u, int32_t* dev_status, void* stream);

/* Bytes of workspace the output projection needs (merged != 0: the merged form). */
MLA_API size_t mla_output_workspace_size(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                         int32_t merged);

/*
 * mla_decode_absorbed_noalloc -- mla_decode_absorbed for callers that cannot allocate
 * device memory (code running where cudaMalloc is unavailable or not allowed, such as
 * inside an allocator's own callbacks or in hosts that hand out all device memory).
 * This entry point is an addition of this library; the pages describe no counterpart.
 *
 * Same arguments and results as mla_decode_absorbed, minus the workspace: the scratch
 * is a fixed 32 MiB array compiled into the library, which every GPU that loads the
 * library keeps until the process exits.  Nothing is allocated or freed by the call.
 * - Returns MLA_ERR_WORKSPACE, before any kernel launch or device memory access, when
 *   mla_decode_workspace_size(dims, dtype, batch, max_seq_len, num_splits) exceeds
 *   32 MiB (lower num_splits, batch or max_seq_len, or use mla_decode_absorbed).
 * - Every call looks up the current device's address of the array
 *   (cudaGetSymbolAddress); the first call on a device may load the library's GPU code
 *   there, so make that first call before any stream capture.
 * - All calls on a device share the one array and it keeps the last call's contents
 *   (nothing in it needs clearing: the decode overwrites whatever it reads).  Calls
 *   whose work overlaps on the GPU (different streams, or host threads without
 *   ordering) race on it and must be serialised by the caller.
 */
MLA_API mla_status mla_decode_absorbed_noalloc(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                       const void* q_c, const void* q_r, const void* w_uk,
                                       const void* cache, int64_t cache_rows, const int64_t* row_off,
                                       const int32_t* seq_len, int32_t max_seq_len,
                                       int32_t num_splits, void* o_lat, float* lse,
                                       int32_t* dev_status, void* stream);

/*
 * mla_set_wait_limit_ns -- time limit, in nanoseconds, of every bounded wait inside the
 * pipelined tensor-core kernels (attention, projections) enqueued after this call by any
 * host thread; 0 restores the default of 2 s.  Returns the previous limit.  A wait that
 * runs out sets MLA_DEV_TIMEOUT in *dev_status; the kernel then stops issuing work, waits
 * for its own copies and MMAs already in flight (those waits keep the 2 s bound), frees its
 * tensor memory and returns, and the outputs of that call are undefined.  The default is
 * far above the longest wait of a healthy launch; lowering it serves tests of the
 * time-out path.  The library's own protocol, not a page of the method, defines it.
 */
MLA_API uint64_t mla_set_wait_limit_ns(uint64_t ns);

/*
 * mla_copy_from_host -- copy `bytes` from page-locked host memory to device memory with a
 * kernel that loads the host buffer directly over the bus (zero-copy reads), enqueued on
 * `stream` (cudaStream_t as void*; NULL = the legacy default stream).  For staging a
 * step's inputs in a serving loop: on hosts where a copy-engine transfer of a few MB pays
 * a large fixed cost per call, this streams close to the link rate.  Transport plumbing
 * of the library; the pages of the method have no counterpart.
 *   dst    device memory (cudaMalloc or managed), `bytes` long, owned by the caller
 *   src    host memory from cudaHostAlloc / cudaMallocHost / cudaHostRegister (page-locked
 *          and mapped into the device's address space), owned by the caller; it must stay
 *          valid and unchanged until the copy has run on `stream`
 *   bytes  any size (16-byte aligned addresses and size take the wide path); 0 is a no-op
 * Returns MLA_ERR_INVALID_ARG for a NULL pointer, a src that is not page-locked mapped host
 * memory or a dst that is not device memory (checked with cudaPointerGetAttributes before
 * any launch), MLA_ERR_CUDA if the launch fails.
 */
MLA_API mla_status mla_copy_from_host(void* dst, const void* src, size_t bytes, void* stream);

/* Static description of a status code (never NULL). */
MLA_API const char* mla_status_string(mla_status status);

/*
 * mla_launch_count -- number of kernels this library has enqueued in this process
 * (all host threads, all devices), for accounting of what ran on the GPU.
 */
MLA_API uint64_t mla_launch_count(void);

/*
 * mla_profile_events -- optional timing hook.  While set, every mla_decode_absorbed
 * call made from the CALLING HOST THREAD records `start` on its stream just before
 * the attention (split) kernel and `stop` just after it, so the caller can read that
 * kernel's own duration with cudaEventElapsedTime.  Both are cudaEvent_t handles
 * passed as void*, created by the caller; (NULL, NULL) turns the hook off.  Returns
 * MLA_ERR_INVALID_ARG when exactly one of them is NULL.
 */
MLA_API mla_status mla_profile_events(void* start, void* stop);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
