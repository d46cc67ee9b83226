// Weight-stationary tcgen05 GEMM for the projections around the attention core.
//
//   D[m, t] = sum_k W_g[m, k] X_g[t, k]      m: output feature, t: token, g: head
//
// The weights are the A operand (M = 128 output features per tile, TMA-loaded, K-major
// or MN-major), the tokens are the B operand (N <= 128 per tile), the accumulator
// lives in TMEM, and K is cut into 64-wide chunks streamed through a ring whose depth
// is chosen per launch (all of a CTA's chunks in flight when shared memory allows).
// For the cache append the long K (hidden = 7168) is also split across CTAs, which
// write fp32 partial sums; a finalize kernel adds them in a fixed order, rotates the
// k_R pairs and stores the bf16 cache rows.
#include <mutex>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>
#include <cuda_fp8.h>

namespace mla {
namespace {

using namespace tc;

constexpr int kGM = 128;              // output features per tile (MMA M)
constexpr int kGK = 64;               // K chunk (one 128-byte swizzle row of bf16)
constexpr int kGNMax = 128;           // tokens per tile (MMA N)
constexpr int kGMaxStages = 8;        // ring depth is chosen per launch (stages <= this)
constexpr int kGThreads = 128;
constexpr uint32_t kATile = kGM * kGK * 2;      // 16 KB
constexpr uint64_t kGTimeoutNs = 2000000000ull;  // bound of the drain waits after an abort

// Shared memory per token-tile width: the ring of stages x (A tile + B tile), reused by
// the epilogue as a staging tile, then the barriers (offset chosen per launch).
template <int NT>
struct GemmSmem {
    static constexpr uint32_t kBTile = NT * kGK * 2;
    static constexpr uint32_t kStage = kATile + kBTile;
};

enum GemmMode : int { kOutBf16 = 0, kOutPartial = 1 };

struct GemmTcArgs {
    int M;                // output features (all tiles)
    int N;                // tokens
    int k_chunks;         // ceil(K / 64)
    int chunks_per_split; // K chunks per CTA
    int k_splits;
    int a_mn;             // weights stored with the output feature contiguous (MN-major A)
    int b_mn;             // B stored with the token index contiguous (MN-major B, NT >= 64)
    int m_split_tile;     // M tiles >= this read the second weight map (rows - tile offset)
    int a2_rows;          // rows loaded from the second weight map (<= 128)
    int mode;
    int stages;           // ring depth (1 .. kGMaxStages)
    int staged;           // bf16 output goes through a shared-memory tile (16-byte stores)
    uint32_t off_bar;     // byte offset of the barriers: after the ring and the staging tile
    float alpha;
    void* y; int64_t y_g, y_tok;      // bf16 output: y[g*y_g + t*y_tok + m]
    void* y2; int64_t y2_tok;         // bf16 output of the second map's rows (when set):
                                      //   y2[t*y2_tok + m - m_split_tile*128]
    float* part; int part_ld;         // fp32 partial: part[(split*N + t)*part_ld + m]
    int32_t* dev_status;
    uint64_t wait_ns;     // limit of every wait of the pipeline
    int defer_wait;       // wait for the kernel before this one only at the end (it writes
                          // nothing this one reads): the two run side by side
};

__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* st,
                                      uint64_t limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    // plain try_wait (no suspend-time hint): a thread suspended with a long hint was seen
    // to wake late after the phase completed, which cost the short GEMMs of a step ~1 us
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort = 1;
            if (st) atomicOr(st, MLA_DEV_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void gdrain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kGTimeoutNs) return;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            int32_t z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}

template <int NT>
__global__ void __launch_bounds__(kGThreads)
gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a2,
               const __grid_constant__ CUtensorMap map_b, GemmTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t base = smem_addr(sm);
    using L = GemmSmem<NT>;
    const uint32_t off_bar = a.off_bar;
    uint64_t* bars = (uint64_t*)(sm + off_bar);
    uint32_t* tslot = (uint32_t*)(sm + off_bar + 8 * (2 * kGMaxStages + 1));
    volatile int* abort_flag = (volatile int*)(sm + off_bar + 8 * (2 * kGMaxStages + 1) + 4);
    // barriers: [0, stages) full, [kGMaxStages, kGMaxStages + stages) empty, 2*kGMaxStages done
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    constexpr int E = kGMaxStages, DONE = 2 * kGMaxStages;
    const uint32_t NS = (uint32_t)a.stages;
    constexpr uint32_t kBTile = L::kBTile;
    constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m_tile = blockIdx.x, n_tile = blockIdx.y;
    const int g = blockIdx.z / a.k_splits, ks = blockIdx.z % a.k_splits;
    const int kc0 = ks * a.chunks_per_split;
    const int kc1 = min(kc0 + a.chunks_per_split, a.k_chunks);
    const bool second = m_tile >= a.m_split_tile;
    const uint32_t a_bytes = second ? (uint32_t)a.a2_rows * kGK * 2 : kATile;

    if (tid == 0) {
        for (uint32_t i = 0; i < NS; ++i) { mbar_init(bar(i), 1); mbar_init(bar(E + i), 1); }
        mbar_init(bar(DONE), 1);
        *abort_flag = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 2) {
        tmem_alloc(smem_addr(tslot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // The kernel behind this one may be scheduled once this one has waited for the kernel
    // before it (a kernel launched beside this one reads its inputs before it waits, so
    // everything before this kernel must be complete when it starts); beside the kernel
    // before it (defer_wait), this one lets it in at once.
    if (!a.defer_wait) pdl_wait();
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        // producer
        uint32_t i = 0;
        for (int kc = kc0; kc < kc1; ++kc, ++i) {
            const uint32_t st = i % NS;
            if (!gwait(bar(E + st), ((i / NS) & 1) ^ 1, abort_flag, a.dev_status, a.wait_ns)) break;
            const uint32_t sa = base + st * L::kStage, sb = sa + kATile;
            mbar_expect_tx(bar(st), a_bytes + kBTile);
            if (second) {
                tma_load_3d(sa, &map_a2, kc * kGK, (m_tile - a.m_split_tile) * kGM, g, bar(st));
            } else if (a.a_mn) {
                tma_load_3d(sa, &map_a, m_tile * kGM, kc * kGK, g, bar(st));
                tma_load_3d(sa + kATile / 2, &map_a, m_tile * kGM + 64, kc * kGK, g, bar(st));
            } else {
                tma_load_3d(sa, &map_a, kc * kGK, m_tile * kGM, g, bar(st));
            }
            if (a.b_mn) {
                // 64-token halves of the tile, 64 K rows each (one 128-byte swizzle atom wide)
                for (int j = 0; j < NT / 64; ++j)
                    tma_load_3d(sb + j * (kGK * 128), &map_b, n_tile * NT + 64 * j, kc * kGK, g, bar(st));
            } else {
                tma_load_3d(sb, &map_b, kc * kGK, g, n_tile * NT, bar(st));
            }
        }
        for (uint32_t k = 0; k < NS && k < i; ++k) {
            const uint32_t j = i - 1 - k;
            gdrain(bar(j % NS), (j / NS) & 1);
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        const uint32_t idesc = idesc_bf16_f32(kGM, NT, a.a_mn && !second ? 1u : 0u, a.b_mn ? 1u : 0u);
        uint32_t i = 0;
        for (int kc = kc0; kc < kc1; ++kc, ++i) {
            const uint32_t st = i % NS;
            if (!gwait(bar(st), (i / NS) & 1, abort_flag, a.dev_status, a.wait_ns)) break;
            tc_fence_after();
            const uint32_t sa = base + st * L::kStage, sb = sa + kATile;
            for (int k = 0; k < kGK / 16; ++k) {
                const uint64_t da = (a.a_mn && !second)
                    ? smem_desc(sa + 2048 * k, kATile / 2, 1024, kSwizzle128B)   // MN-major: 64-wide atoms 8 KB apart
                    : smem_desc(sa + 32 * k, 16, 1024, kSwizzle128B);
                const uint64_t db = a.b_mn
                    ? smem_desc(sb + 2048 * k, kGK * 128, 1024, kSwizzle128B)    // MN-major: 64-token atoms 8 KB apart
                    : smem_desc(sb + 32 * k, 16, 1024, kSwizzle128B);
                mma_bf16(tmem, da, db, idesc, (i > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(bar(E + st));
        }
        mma_commit(bar(DONE));
    }
    // epilogue: thread <-> output feature (TMEM lane), 32 tokens per TMEM load
    __syncwarp();
    const bool ok = gwait(bar(DONE), 0, abort_flag, a.dev_status, a.wait_ns);
    tc_fence_after();
    const int m = m_tile * kGM + warp * 32 + lane;
    const bool m_ok = m < a.M;
    const bool all_ok = __all_sync(0xffffffffu, ok);
    constexpr int kChunks = NT < 32 ? 1 : NT / 32;
    constexpr int kCols = NT < 32 ? NT : 32;
    // bf16 output through shared memory: the stage ring is idle once the MMAs are done,
    // and whole 128-feature rows (256 B) of a token go out as 16-byte stores
    const bool staged = a.staged != 0;
    constexpr int kLd = kGM + 4;                // fp32 row pitch of the staging tile
    float* tile = reinterpret_cast<float*>(sm);
    if (all_ok) {
        for (int c = 0; c < kChunks; ++c) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32 * c, v);
            tmem_wait_ld();
            if (staged) {
#pragma unroll
                for (int j = 0; j < kCols; ++j) tile[(32 * c + j) * kLd + warp * 32 + lane] = a.alpha * v[j];
                continue;
            }
            if (!m_ok) continue;
            for (int j = 0; j < kCols; ++j) {
                const int t = n_tile * NT + 32 * c + j;
                if (t >= a.N) break;
                if (a.mode == kOutBf16 && second && a.y2)
                    ((__nv_bfloat16*)a.y2)[(int64_t)t * a.y2_tok + m - a.m_split_tile * kGM] =
                        __float2bfloat16_rn(a.alpha * v[j]);
                else if (a.mode == kOutBf16)
                    ((__nv_bfloat16*)a.y)[(int64_t)g * a.y_g + (int64_t)t * a.y_tok + m] =
                        __float2bfloat16_rn(a.alpha * v[j]);
                else
                    a.part[((int64_t)ks * a.N + t) * a.part_ld + m] = v[j];
            }
        }
    }
    if (staged) {
        __syncthreads();                        // every warp's columns are in the tile
        if (all_ok) {
            for (int e = tid; e < NT * (kGM / 8); e += kGThreads) {
                const int j = e / (kGM / 8), f8 = e % (kGM / 8);
                const int t = n_tile * NT + j;
                if (t >= a.N) continue;
                const float* src = tile + j * kLd + 8 * f8;
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * q], src[2 * q + 1]);
                    w[q] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                __nv_bfloat16* dst = (second && a.y2)
                    ? (__nv_bfloat16*)a.y2 + (int64_t)t * a.y2_tok + (m_tile - a.m_split_tile) * kGM + 8 * f8
                    : (__nv_bfloat16*)a.y + (int64_t)g * a.y_g + (int64_t)t * a.y_tok + m_tile * kGM + 8 * f8;
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    // after an abort the epilogue did not wait for the MMAs: every MMA (the issuer's
    // DONE commit follows its last one in both paths) completes before TMEM is freed
    if (!all_ok && warp == 2) gdrain(bar(DONE), 0);
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // beside the kernel before it: this kernel's end implies that one's, for the kernels
    // behind this one that wait for it
    if (a.defer_wait) pdl_wait();
}

// cache row = [sum of partials for c ; RoPE(sum of partials for k_R, pos)] in bf16.
// Grid (token, pair groups of kFinPairs): thread (x, y) of a block adds splits
// y, y + kFinGroups, ... of pair x; the kFinGroups partial sums are then added in a
// fixed order through shared memory (so the result does not depend on timing), and
// the y = 0 threads rotate the k_R pairs and store the row.  A rotary pair stays in
// one thread.
constexpr int kFinPairs = 32;
constexpr int kFinGroups = 8;

__global__ void __launch_bounds__(kFinPairs * kFinGroups)
append_finalize_kernel(const float* __restrict__ part, int k_splits, int n_tok, int n_new, int d_c,
                       int d_r, double rope_r, const int64_t* __restrict__ row_off,
                       const int32_t* __restrict__ cap, const int32_t* __restrict__ pos0,
                       CacheView cv, int32_t* dev_status) {
    __shared__ float2 red[kFinGroups][kFinPairs];
    // The kernel behind this one (the decode's query fold, beside the append) may start at
    // once: the append GEMM let this kernel in only after its own wait, so all work before
    // the append call is complete.
    pdl_trigger();
    pdl_wait();                 // launched behind the append GEMM: its partial sums are complete
    const int t = blockIdx.x;
    const int width = d_c + d_r;
    const int x = threadIdx.x % kFinPairs, y = threadIdx.x / kFinPairs;
    const int e = 2 * (blockIdx.y * kFinPairs + x);
    const int b = t / n_new, j = t % n_new;
    const int p0 = pos0[b];
    const int64_t cp = cap[b];
    // contiguous: the sequence's rows must lie in the buffer; paged: its positions must be
    // covered by its block-table entries, and this token's block must lie in the buffer
    bool bad = p0 < 0 || (int64_t)p0 + n_new > cp;
    int64_t row = -1;
    if (!bad) {
        if (!cv.block_table) {
            const int64_t off = row_off[b];
            bad = off < 0 || off + cp > cv.rows;
        } else {
            bad = cp > (int64_t)cv.max_blocks * cv.block_size;
        }
        if (!bad) {
            row = cache_row(cv, row_off, b, (int64_t)p0 + j);
            bad = row < 0 || row >= cv.rows;
        }
    }
    if (bad) {
        if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(dev_status, MLA_DEV_BAD_POSITION);
        return;
    }
    float2 acc = make_float2(0.f, 0.f);
    if (e < width) {
        const float* p = part + (int64_t)t * width + e;
        const int64_t split_stride = (int64_t)n_tok * width;
        for (int s0 = y; s0 < k_splits; s0 += 4 * kFinGroups) {
            float2 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int sp = s0 + q * kFinGroups;
                v[q] = sp < k_splits ? *reinterpret_cast<const float2*>(p + sp * split_stride) : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) { acc.x += v[q].x; acc.y += v[q].y; }
        }
    }
    red[y][x] = acc;
    __syncthreads();
    if (y != 0 || e >= width) return;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int q = 0; q < kFinGroups; ++q) { v0 += red[q][x].x; v1 += red[q][x].y; }
    const int64_t pos = (int64_t)p0 + j;
    if (e >= d_c) {
        float c, sn;
        rope_cos_sin(pos, (e - d_c) >> 1, rope_r, &c, &sn);
        const float r0 = v0 * c - v1 * sn, r1 = v0 * sn + v1 * c;
        v0 = r0;
        v1 = r1;
    }
    __nv_bfloat16* dst = (cv.pe && e >= d_c) ? (__nv_bfloat16*)cv.pe + row * cv.pe_stride + (e - d_c)
                                             : (__nv_bfloat16*)cv.kv + row * cv.kv_stride + e;
    *(__nv_bfloat162*)dst = __floats2bfloat162_rn(v0, v1);
}

// The same row written in the fp8 layout (contiguous cache of rows of kFp8RowBytes(d_c, d_r)
// bytes): the latent as E4M3 codes in 128-column groups with one scale each, the smallest
// power of two 2^k with (largest magnitude of the group) / 2^k <= 448 (1 for a zero
// group), stored as fp32; the rotary part rotated and kept in bf16.  Grid (token, 128-column groups, the rotary part last): thread (x, y) of a block
// adds splits y, y + kF8Groups, ... of pair x; the groups' sums are added in a fixed order,
// and the y = 0 threads (two warps) find the group's largest magnitude and store the codes.
constexpr int kF8Pairs = 64;
constexpr int kF8Groups = 4;

__global__ void __launch_bounds__(kF8Pairs * kF8Groups)
append_finalize_fp8_kernel(const float* __restrict__ part, int k_splits, int n_tok, int n_new, int d_c,
                           int d_r, double rope_r, const int64_t* __restrict__ row_off,
                           const int32_t* __restrict__ cap, const int32_t* __restrict__ pos0,
                           uint8_t* __restrict__ cache, int64_t cache_rows, int32_t* dev_status) {
    __shared__ float2 red[kF8Groups][kF8Pairs];
    __shared__ float wmax[2];
    // The kernel behind this one (the decode's query fold, beside the append) may start at
    // once: the append GEMM let this kernel in only after its own wait, so all work before
    // the append call is complete.
    pdl_trigger();
    pdl_wait();                 // launched behind the append GEMM: its partial sums are complete
    const int t = blockIdx.x;
    const int width = d_c + d_r;
    const int x = threadIdx.x % kF8Pairs, y = threadIdx.x / kF8Pairs;
    const int e = 2 * (blockIdx.y * kF8Pairs + x);
    const int b = t / n_new, j = t % n_new;
    const int p0 = pos0[b];
    const int64_t cp = cap[b];
    const int64_t off = row_off[b];
    const bool bad = p0 < 0 || (int64_t)p0 + n_new > cp || off < 0 || off + cp > cache_rows;
    if (bad) {
        if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(dev_status, MLA_DEV_BAD_POSITION);
        return;
    }
    const int64_t row = off + p0 + j;
    uint8_t* dst = cache + row * (int64_t)kFp8RowBytes(d_c, d_r);
    float2 acc = make_float2(0.f, 0.f);
    if (e < width) {
        const float* p = part + (int64_t)t * width + e;
        const int64_t split_stride = (int64_t)n_tok * width;
        for (int sp = y; sp < k_splits; sp += kF8Groups) {
            const float2 v = *reinterpret_cast<const float2*>(p + sp * split_stride);
            acc.x += v.x;
            acc.y += v.y;
        }
    }
    red[y][x] = acc;
    __syncthreads();
    if (y != 0) return;                         // warps 0 and 1 go on (x = lane + 32 * warp)
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int q = 0; q < kF8Groups; ++q) { v0 += red[q][x].x; v1 += red[q][x].y; }
    if (e >= d_c) {                             // the rotary block: rotate, store bf16
        if (e >= width) return;
        float c, sn;
        rope_cos_sin((int64_t)p0 + j, (e - d_c) >> 1, rope_r, &c, &sn);
        const float r0 = v0 * c - v1 * sn, r1 = v0 * sn + v1 * c;
        *(__nv_bfloat162*)(dst + d_c + 4 * (d_c / 128) + 2 * (e - d_c)) = __floats2bfloat162_rn(r0, r1);
        return;
    }
    // a latent group of 128 columns: every one of the 64 threads holds a pair
    float m = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    asm volatile("bar.sync 1, 64;" ::: "memory");    // the two warps of this group only
    const float amax = fmaxf(wmax[0], wmax[1]);
    // q = amax / 448 (fp32 division); 2^k is the smallest power of two >= q, read off q's
    // binary exponent (q = m 2^e with m in [0.5, 1): k = e, or e - 1 when m = 0.5)
    float scale = 1.f;
    if (amax > 0.f) {
        int e;
        const float m = frexpf(amax / 448.f, &e);
        scale = ldexpf(1.f, m == 0.5f ? e - 1 : e);
    }
    const __nv_fp8x2_storage_t q2 = __nv_cvt_float2_to_fp8x2(make_float2(v0 / scale, v1 / scale), __NV_SATFINITE,
                                                              __NV_E4M3);
    *reinterpret_cast<__nv_fp8x2_storage_t*>(dst + e) = q2;
    if (x == 0) *reinterpret_cast<float*>(dst + d_c + 4 * blockIdx.y) = scale;
}

// y[t, e] = bf16(sum over splits of part[split, t, e]) for a split-K GEMM, summed in a
// fixed order (8 thread groups per column pair, then a shared-memory reduction), so the
// result does not depend on timing.  Grid (token, column-pair groups of kFinPairs).
__global__ void __launch_bounds__(kFinPairs * kFinGroups)
splitk_reduce_kernel(const float* __restrict__ part, int k_splits, int n_tok, int width,
                     __nv_bfloat16* __restrict__ y, int64_t y_tok) {
    __shared__ float2 red[kFinGroups][kFinPairs];
    pdl_wait();                 // launched behind the split-K GEMM: its partial sums are complete
    const int t = blockIdx.x;
    const int x = threadIdx.x % kFinPairs, g = threadIdx.x / kFinPairs;
    const int e = 2 * (blockIdx.y * kFinPairs + x);
    float2 acc = make_float2(0.f, 0.f);
    if (e < width) {
        const float* p = part + (int64_t)t * width + e;
        const int64_t split_stride = (int64_t)n_tok * width;
        for (int s0 = g; s0 < k_splits; s0 += kFinGroups) {
            const float2 v = *reinterpret_cast<const float2*>(p + s0 * split_stride);
            acc.x += v.x;
            acc.y += v.y;
        }
    }
    red[g][x] = acc;
    __syncthreads();
    if (g != 0 || e >= width) return;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int q = 0; q < kFinGroups; ++q) { v0 += red[q][x].x; v1 += red[q][x].y; }
    *(__nv_bfloat162*)(y + (int64_t)t * y_tok + e) = __floats2bfloat162_rn(v0, v1);
}

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

bool encoder() {
    std::call_once(g_enc_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_enc = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    });
    return g_enc != nullptr;
}

// 3-D bf16 map: dims (inner..outer) d0, d1, d2 with byte strides s1, s2; box b0 x b1 x b2.
bool map3(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
          uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    return g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pick_nt(int n) {
    if (n <= 16) return 16;
    if (n <= 32) return 32;
    if (n <= 64) return 64;
    return 128;
}

cudaError_t run_gemm(const CUtensorMap& ma, const CUtensorMap& ma2, const CUtensorMap& mb, GemmTcArgs a,
                     int G, int nt, cudaStream_t s) {
    const int m_tiles = (a.M + kGM - 1) / kGM;
    const int n_tiles = (a.N + nt - 1) / nt;
    dim3 grid(m_tiles, n_tiles, G * a.k_splits);
    // ring depth: every K chunk of a CTA in flight at once when it fits, else as deep as
    // shared memory allows
    const uint32_t stage_bytes = kATile + (uint32_t)nt * kGK * 2;
    int stages = min(a.chunks_per_split, kGMaxStages);
    while (stages > 1 && (uint32_t)stages * stage_bytes + 256 + 1024 > 232448u) --stages;
    a.stages = max(stages, 1);
    a.staged = a.mode == kOutBf16 && a.M % kGM == 0 && (a.y_tok % 8) == 0 && (a.y_g % 8) == 0 &&
               ((uintptr_t)a.y % 16) == 0 && (!a.y2 || ((a.y2_tok % 8) == 0 && ((uintptr_t)a.y2 % 16) == 0));
    const uint32_t tile_bytes = (uint32_t)nt * (kGM + 4) * 4;
    uint32_t ring = (uint32_t)a.stages * stage_bytes;
    if (a.staged && tile_bytes > ring) ring = (tile_bytes + 1023) / 1024 * 1024;
    a.off_bar = ring;
    const uint32_t smem = ring + 256 + 1024;
    // Launched as a programmatic dependent of the kernel before it on the stream: the set-up
    // (barriers, tensor memory) overlaps that kernel's tail, and the kernel waits for it
    // (griddepcontrol.wait) before it reads any input.
    cudaError_t e;
#define MLA_GEMM_CASE(NTV)                                                                         \
    case NTV: {                                                                                    \
        e = cudaFuncSetAttribute(gemm_tc_kernel<NTV>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 (int)smem);                                                      \
        if (e != cudaSuccess) return e;                                                           \
        e = launch_ex(gemm_tc_kernel<NTV>, grid, dim3(kGThreads), smem, s, true, ma, ma2, mb, a);  \
        if (e != cudaSuccess) return e;                                                           \
        break;                                                                                    \
    }
    switch (nt) {
        MLA_GEMM_CASE(16)
        MLA_GEMM_CASE(32)
        MLA_GEMM_CASE(64)
        MLA_GEMM_CASE(128)
        default: return cudaErrorInvalidValue;
    }
#undef MLA_GEMM_CASE
    note_launch();
    return cudaGetLastError();
}

GemmTcArgs gblank() {
    GemmTcArgs a{};
    a.k_splits = 1;
    a.stages = 1;
    a.m_split_tile = 1 << 30;
    a.alpha = 1.f;
    a.mode = kOutBf16;
    a.wait_ns = wait_limit_ns();
    return a;
}

}  // namespace

bool gemm_tc_shapes_ok(const mla_dims& d) {
    return d.d_c % 128 == 0 && d.d_h % 128 == 0 && d.d_r % 16 == 0 && d.d_r <= 128 &&
           d.hidden % 64 == 0;
}

// Splits of a long reduction (K) across CTAs so that the M x N tiles times the splits
// fill the GPU about once; at least two 64-wide chunks per split.
int k_splits_for(int K, int M, int n_tok, int sm_count) {
    const int k_chunks = (K + kGK - 1) / kGK;
    const int m_tiles = (M + kGM - 1) / kGM;
    const int n_tiles = (n_tok + kGNMax - 1) / kGNMax;
    int want = (sm_count > 0 ? sm_count : 148) / (m_tiles * n_tiles);
    if (want < 1) want = 1;
    int per = (k_chunks + want - 1) / want;
    if (per < 2) per = 2;
    return (k_chunks + per - 1) / per;
}

size_t append_tc_workspace(const mla_dims& d, int n_tok, int* k_splits_out, int sm_count) {
    const int splits = k_splits_for(d.hidden, d.d_c + d.d_r, n_tok, sm_count);
    if (k_splits_out) *k_splits_out = splits;
    return align_up((size_t)splits * n_tok * (d.d_c + d.d_r) * sizeof(float), 256);
}

size_t query_latent_tc_workspace(int hidden, int d_q, int n_tok, int* k_splits_out, int sm_count) {
    const int splits = k_splits_for(hidden, d_q, n_tok, sm_count);
    if (k_splits_out) *k_splits_out = splits;
    return align_up((size_t)splits * n_tok * d_q * sizeof(float), 256);
}

cudaError_t launch_query_latent_tc(int hidden, int d_q, int batch, const void* h, const void* w_dq,
                                   void* workspace, void* c_q, int32_t* dev_status, int sm_count,
                                   cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    int splits = 1;
    query_latent_tc_workspace(hidden, d_q, batch, &splits, sm_count);
    const int nt = pick_nt(batch);
    const uint64_t H = hidden;
    CUtensorMap ma, mb;
    // W_DQ [d_q, hidden] (K-major), h [batch, hidden]
    if (!map3(&ma, w_dq, H, d_q, 1, H * 2, H * 2 * d_q, kGK, kGM, 1) ||
        !map3(&mb, h, H, 1, batch, H * 2, H * 2, kGK, 1, nt))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = d_q;
    a.N = batch;
    a.k_chunks = (hidden + kGK - 1) / kGK;
    a.k_splits = splits;
    a.chunks_per_split = (a.k_chunks + splits - 1) / splits;
    a.mode = kOutPartial;
    a.part = (float*)workspace;
    a.part_ld = d_q;
    a.dev_status = dev_status;
    cudaError_t e = run_gemm(ma, ma, mb, a, 1, nt, s);
    if (e != cudaSuccess) return e;
    const dim3 grid(batch, (d_q / 2 + kFinPairs - 1) / kFinPairs);
    e = launch_ex(splitk_reduce_kernel, grid, dim3(kFinPairs * kFinGroups), 0, s, true, (const float*)workspace,
                  splits, batch, d_q, (__nv_bfloat16*)c_q, (int64_t)d_q);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Split-K product u[t, m] = sum_k A[m, k] x[t, k] for a long K, then the fixed-order
// reduction of the partial sums to bf16 u[t*u_tok + m].  ma: the A map (K-major, or
// MN-major when a_mn), mb: x as [batch, K].
cudaError_t splitk_linear(const CUtensorMap& ma, const CUtensorMap& mb, int a_mn, int M, int K, int batch,
                          void* workspace, void* u, int64_t u_tok, int32_t* dev_status, int sm_count,
                          cudaStream_t s) {
    const int splits = k_splits_for(K, M, batch, sm_count);
    GemmTcArgs a = gblank();
    a.M = M;
    a.N = batch;
    a.k_chunks = (K + kGK - 1) / kGK;
    a.k_splits = splits;
    a.chunks_per_split = (a.k_chunks + splits - 1) / splits;
    a.a_mn = a_mn;
    a.mode = kOutPartial;
    a.part = (float*)workspace;
    a.part_ld = M;
    a.dev_status = dev_status;
    cudaError_t e = run_gemm(ma, ma, mb, a, 1, pick_nt(batch), s);
    if (e != cudaSuccess) return e;
    const dim3 grid(batch, (M / 2 + kFinPairs - 1) / kFinPairs);
    e = launch_ex(splitk_reduce_kernel, grid, dim3(kFinPairs * kFinGroups), 0, s, true, (const float*)workspace,
                  splits, batch, M, (__nv_bfloat16*)u, u_tok);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

size_t output_tc_workspace(int hidden, int k_in, int n_tok, int sm_count) {
    return align_up((size_t)k_splits_for(k_in, hidden, n_tok, sm_count) * n_tok * hidden * sizeof(float), 256);
}

cudaError_t launch_output_tc(const mla_dims& d, int batch, const void* o, const void* w_o, void* workspace,
                             void* u, int32_t* dev_status, int sm_count, cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const uint64_t K = (uint64_t)d.n_heads * d.d_h, H = d.hidden;
    CUtensorMap ma, mb;
    // W_O [hidden, n_h*d_h] (K-major), o [batch, n_h*d_h]
    if (!map3(&ma, w_o, K, H, 1, K * 2, K * 2 * H, kGK, kGM, 1) ||
        !map3(&mb, o, K, 1, batch, K * 2, K * 2, kGK, 1, pick_nt(batch)))
        return cudaErrorInvalidValue;
    return splitk_linear(ma, mb, 0, d.hidden, (int)K, batch, workspace, u, d.hidden, dev_status, sm_count, s);
}

cudaError_t launch_output_merged_tc(const mla_dims& d, int batch, const void* o_lat, const void* w_ov,
                                    void* workspace, void* u, int32_t* dev_status, int sm_count, cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const uint64_t K = (uint64_t)d.n_heads * d.d_c, H = d.hidden;
    CUtensorMap ma, mb;
    // W_OV stored [n_h * d_c, hidden]: the output feature contiguous (MN-major A), o_lat [batch, n_h*d_c]
    if (!map3(&ma, w_ov, H, K, 1, H * 2, H * 2 * K, 64, kGK, 1) ||
        !map3(&mb, o_lat, K, 1, batch, K * 2, K * 2, kGK, 1, pick_nt(batch)))
        return cudaErrorInvalidValue;
    return splitk_linear(ma, mb, 1, d.hidden, (int)K, batch, workspace, u, d.hidden, dev_status, sm_count, s);
}

cudaError_t launch_merge_output_weights_tc(const mla_dims& d, const void* w_o, const void* w_uv, void* w_ov,
                                           int32_t* dev_status, cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const uint64_t H = d.hidden, nh = d.n_heads, dh = d.d_h, dc = d.d_c;
    CUtensorMap ma, mb;
    // A = W_O^(i): rows m of W_O, columns i*d_h .. i*d_h + d_h - 1 (K-major, head = 3rd dim);
    // B = W_UV^(i) read as [d_c tokens x d_h] with the token index contiguous (MN-major)
    if (!map3(&ma, w_o, dh, H, nh, nh * dh * 2, dh * 2, kGK, kGM, 1) ||
        !map3(&mb, w_uv, dc, dh, nh, dc * 2, dh * dc * 2, 64, kGK, 1))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = d.hidden;
    a.N = d.d_c;
    a.k_chunks = (d.d_h + kGK - 1) / kGK;
    a.chunks_per_split = a.k_chunks;
    a.b_mn = 1;
    a.y = w_ov;                        // W_OV^(i)[c][m] at i*d_c*hidden + c*hidden + m
    a.y_g = (int64_t)d.d_c * d.hidden;
    a.y_tok = d.hidden;
    a.dev_status = dev_status;
    return run_gemm(ma, ma, mb, a, d.n_heads, kGNMax, s);
}

cudaError_t launch_project_query_tc(const mla_dims& d, int batch, int d_in, const void* x, const void* w_uq,
                                    const void* w_qr, void* q_c, void* q_r, int32_t* dev_status,
                                    cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const int nt = pick_nt(batch);
    const uint64_t K = d_in;
    const int m1 = d.n_heads * d.d_h, m2 = d.n_heads * d.d_r;
    CUtensorMap ma, ma2, mb;
    // [W_UQ ; W_QR] as one M range: tiles below m1/128 read W_UQ, the rest W_QR
    if (!map3(&ma, w_uq, K, m1, 1, K * 2, K * 2 * m1, kGK, kGM, 1) ||
        !map3(&ma2, w_qr, K, m2, 1, K * 2, K * 2 * m2, kGK, kGM, 1) ||
        !map3(&mb, x, K, 1, batch, K * 2, K * 2, kGK, 1, nt))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = m1 + m2;
    a.N = batch;
    a.k_chunks = (d_in + kGK - 1) / kGK;
    a.chunks_per_split = a.k_chunks;
    a.m_split_tile = m1 / kGM;
    a.a2_rows = kGM;
    a.y = q_c;
    a.y_tok = m1;
    a.y2 = q_r;
    a.y2_tok = m2;
    a.dev_status = dev_status;
    return run_gemm(ma, ma2, mb, a, 1, nt, s);
}

cudaError_t launch_append_tc(const mla_dims& d, int batch, int n_new, const void* h, const void* w_dkv,
                             const void* w_kr, const int64_t* row_off, const int32_t* cap,
                             const int32_t* pos0, const CacheView& cv, void* workspace,
                             int32_t* dev_status, int sm_count, cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const int n_tok = batch * n_new;
    int splits = 1;
    append_tc_workspace(d, n_tok, &splits, sm_count);
    const int width = d.d_c + d.d_r;
    const int k_chunks = (d.hidden + kGK - 1) / kGK;
    const int nt = pick_nt(n_tok);
    CUtensorMap ma, ma2, mb;
    const uint64_t H = d.hidden;
    if (!map3(&ma, w_dkv, H, d.d_c, 1, H * 2, H * 2 * d.d_c, kGK, kGM, 1) ||
        !map3(&ma2, w_kr, H, d.d_r, 1, H * 2, H * 2 * d.d_r, kGK, d.d_r, 1) ||
        !map3(&mb, h, H, 1, n_tok, H * 2, H * 2, kGK, 1, nt))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = width;
    a.N = n_tok;
    a.k_chunks = k_chunks;
    a.k_splits = splits;
    a.chunks_per_split = (k_chunks + splits - 1) / splits;
    a.m_split_tile = d.d_c / kGM;
    a.a2_rows = d.d_r;
    a.mode = kOutPartial;
    a.part = (float*)workspace;
    a.part_ld = width;
    a.dev_status = dev_status;
    cudaError_t e = run_gemm(ma, ma2, mb, a, 1, nt, s);
    if (e != cudaSuccess) return e;
    const dim3 fin_grid(n_tok, (width / 2 + kFinPairs - 1) / kFinPairs);
    e = launch_ex(append_finalize_kernel, fin_grid, dim3(kFinPairs * kFinGroups), 0, s, true,
                  (const float*)workspace, splits, n_tok, n_new, d.d_c, d.d_r, rope_ratio(d.rope_base, d.d_r),
                  row_off, cap, pos0, cv, dev_status);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_append_fp8_tc(const mla_dims& d, int batch, int n_new, const void* h, const void* w_dkv,
                                 const void* w_kr, const int64_t* row_off, const int32_t* cap,
                                 const int32_t* pos0, void* cache, int64_t cache_rows, void* workspace,
                                 int32_t* dev_status, int sm_count, cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const int n_tok = batch * n_new;
    int splits = 1;
    append_tc_workspace(d, n_tok, &splits, sm_count);
    const int width = d.d_c + d.d_r;
    const int k_chunks = (d.hidden + kGK - 1) / kGK;
    const int nt = pick_nt(n_tok);
    CUtensorMap ma, ma2, mb;
    const uint64_t H = d.hidden;
    if (!map3(&ma, w_dkv, H, d.d_c, 1, H * 2, H * 2 * d.d_c, kGK, kGM, 1) ||
        !map3(&ma2, w_kr, H, d.d_r, 1, H * 2, H * 2 * d.d_r, kGK, d.d_r, 1) ||
        !map3(&mb, h, H, 1, n_tok, H * 2, H * 2, kGK, 1, nt))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = width;
    a.N = n_tok;
    a.k_chunks = k_chunks;
    a.k_splits = splits;
    a.chunks_per_split = (k_chunks + splits - 1) / splits;
    a.m_split_tile = d.d_c / kGM;
    a.a2_rows = d.d_r;
    a.mode = kOutPartial;
    a.part = (float*)workspace;
    a.part_ld = width;
    a.dev_status = dev_status;
    cudaError_t e = run_gemm(ma, ma2, mb, a, 1, nt, s);
    if (e != cudaSuccess) return e;
    // one block per 128 latent columns, and one for the rotary part
    const dim3 fin_grid(n_tok, d.d_c / 128 + (d.d_r / 2 + kF8Pairs - 1) / kF8Pairs);
    e = launch_ex(append_finalize_fp8_kernel, fin_grid, dim3(kF8Pairs * kF8Groups), 0, s, true,
                  (const float*)workspace, splits, n_tok, n_new, d.d_c, d.d_r, rope_ratio(d.rope_base, d.d_r),
                  row_off, cap, pos0, (uint8_t*)cache, cache_rows, dev_status);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_fold_tc(const mla_dims& d, int batch, const void* q_c, const void* w_uk, float alpha,
                           void* qp, int32_t* dev_status, cudaStream_t s, bool beside) {
    if (!encoder()) return cudaErrorNotSupported;
    const int nt = pick_nt(batch);
    const uint64_t dc = d.d_c, dh = d.d_h, nh = d.n_heads;
    CUtensorMap ma, mb;
    // W_UK [n_h, d_h, d_c]: the output feature c is contiguous (MN-major A), K = d_h
    if (!map3(&ma, w_uk, dc, dh, nh, dc * 2, dc * dh * 2, 64, kGK, 1) ||
        !map3(&mb, q_c, dh, nh, batch, dh * 2, dh * nh * 2, kGK, 1, nt))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = d.d_c;
    a.N = batch;
    a.k_chunks = (d.d_h + kGK - 1) / kGK;
    a.chunks_per_split = a.k_chunks;
    a.a_mn = 1;
    a.alpha = alpha;
    a.y = qp;
    a.y_g = d.d_c + d.d_r;
    a.y_tok = (int64_t)d.n_heads * (d.d_c + d.d_r);
    a.dev_status = dev_status;
    a.defer_wait = beside ? 1 : 0;
    return run_gemm(ma, ma, mb, a, d.n_heads, nt, s);
}

cudaError_t launch_project_out_tc(const mla_dims& d, int batch, const void* o_lat, const void* w_uv,
                                  void* out, int32_t* dev_status, cudaStream_t s) {
    if (!encoder()) return cudaErrorNotSupported;
    const int nt = pick_nt(batch);
    const uint64_t dc = d.d_c, dh = d.d_h, nh = d.n_heads;
    CUtensorMap ma, mb;
    // W_UV [n_h, d_h, d_c]: rows are output features d, K = d_c contiguous (K-major A)
    if (!map3(&ma, w_uv, dc, dh, nh, dc * 2, dc * dh * 2, kGK, kGM, 1) ||
        !map3(&mb, o_lat, dc, nh, batch, dc * 2, dc * nh * 2, kGK, 1, nt))
        return cudaErrorInvalidValue;
    GemmTcArgs a = gblank();
    a.M = d.d_h;
    a.N = batch;
    a.k_chunks = (d.d_c + kGK - 1) / kGK;
    a.chunks_per_split = a.k_chunks;
    a.y = out;
    a.y_g = d.d_h;
    a.y_tok = (int64_t)d.n_heads * d.d_h;
    a.dev_status = dev_status;
    return run_gemm(ma, ma, mb, a, d.n_heads, nt, s);
}

}  // namespace mla
