// Split-K absorbed decode on tcgen05 tensor cores (sm_103a), bf16 latent cache with
// d_c = 512, d_r = 64 and up to 128 heads.
//
// Work unit: a 2-CTA cluster walks one contiguous range of the flattened context
// (same schedule as the CUDA-core kernel).  CTA r of the pair owns latent columns
// [256r, 256r+256) and rotary columns [512+32r, 512+32r+32) of every cache row, so
// the pair streams each row from HBM exactly once.  Per tile of 64 rows:
//
//   S_r = Q'_r C_r^T         tcgen05, M=128 heads, N=64 rows, K=288; Q'_r is the A
//                            operand (latent columns 0-127 in tensor memory, columns
//                            128-255 and the rotary part in shared memory); the cache
//                            tile is the B operand
//   S   = S_0 + S_1          each CTA sends its partial to the peer (DSMEM), as an
//                            fp32 offset per head plus fp16 differences
//   P   = exp2(S - m)        online softmax (identical in both CTAs; lazy max update)
//   O_r += P C_r[:, :256]    tcgen05, M=128, N=256, K=64; P (bf16) from tensor memory,
//                            the cache tile read again as an MN-major B operand
//
// Tensor memory (512 columns): O_r 128 x 256 fp32, latent columns 0-127 of Q'_r
// (64 columns), P[2] 2 x 128 x 64 bf16 and S[2] 2 x 128 x 64 fp32 (one of each per tile
// parity).  Shared memory: a 4-stage ring of cache tiles (about 147 KB in flight; one
// TMA copy for a tile's latent half and one for its rotary half), two exchange buffers,
// the rest of Q'_r, per-piece statistics.
//
// Warp roles: warp 0 TMA producer, warps 1 and 3 issue the score
// MMAs of the even and odd tiles, warp 2 owns the tensor memory and issues the value
// MMAs, warps 4-7 and 8-11 two softmax/exchange groups that take alternate tiles
// (thread i <-> head i <-> TMEM lane i), warps 12-15 load Q' of each piece and write
// each piece's output.  Each group has its own exchange buffer, laid out [16-byte
// chunk][head], so the 32 lanes of a warp write 512 contiguous bytes into the peer
// (whole 32-byte sectors on the cluster interconnect); the peer's mbarrier counts the
// bytes, and each warp that has read its rows returns a credit.  Every wait is
// bounded in time; on expiry the CTA raises MLA_DEV_TIMEOUT, drains its own in-flight
// copies and MMAs, frees TMEM and returns.
#include <mutex>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "tc_ptx.cuh"

#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

namespace mla {
namespace {

using namespace tc;

constexpr int kTok = 64;              // cache rows per tile (score MMA N, value MMA K)
constexpr int kStages = 4;            // TMA ring depth
constexpr int kThreads = 512;
constexpr int kHeads = 128;           // MMA M (heads beyond n_heads are computed and dropped)
constexpr int kLatHalf = 256;         // latent columns per CTA
constexpr int kRopeHalf = 32;         // rotary columns per CTA
constexpr int kRowElems = 576;        // d_c + d_r
constexpr uint64_t kTimeoutNs = 2000000000ull;   // bound of the drain waits after an abort

// shared memory layout (byte offsets from a 1024-aligned base)
constexpr uint32_t kTBox = kTok * 128;                   // 64 rows x 64 bf16, 128B swizzle
constexpr uint32_t kTRope = kTok * 64;                   // 64 rows x 32 bf16, 64B swizzle
constexpr uint32_t kStageBytes = 4 * kTBox + kTRope;     // 36864
// the peer's partial scores of one tile: per head an fp32 offset (the partial of the
// tile's first row) and 64 fp16 differences from it
constexpr uint32_t kXResBytes = kHeads * kTok * 2;
constexpr uint32_t kXBytes = kXResBytes + kHeads * 4;
constexpr uint32_t kOffStage = 0;
constexpr uint32_t kOffX = kOffStage + kStages * kStageBytes;
// latent chunks 2 and 3 (columns 128..255 of this CTA's half) of Q'_r: the A operand of
// half of the latent score MMAs, 2 x (128 heads x 64 bf16), K-major, 128B swizzle
constexpr uint32_t kOffQL = kOffX + 2 * kXBytes;
constexpr uint32_t kQLChunk = kHeads * 128;
constexpr uint32_t kOffQR = kOffQL + 2 * kQLChunk;       // rotary part of Q'_r: 128 x 32 bf16, 64B swizzle
constexpr uint32_t kOffStats = kOffQR + kHeads * 64;      // [piece % 4][group][m, l][head] fp32
constexpr uint32_t kOffMh = kOffStats + 4 * 2 * 2 * kHeads * 4;   // [tile parity][head] running max
constexpr uint32_t kOffBar = kOffMh + 2 * kHeads * 4;
constexpr uint32_t kBarBytes = 320;                      // mbarriers, then the TMEM slot and abort flag
// No alignment slack: dynamic shared memory starts on a 1024-byte boundary (it follows the
// 1 KB reserved at the bottom of a CTA's window, and the kernel has no static shared
// memory); the kernel checks this and returns MLA_DEV_SMEM_ALIGN otherwise.
constexpr uint32_t kSmemBytes = kOffBar + kBarBytes + 16;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffQL % 1024 == 0 && kQLChunk % 1024 == 0, "swizzled operands need 1024-byte alignment");

// barrier indices
enum : int {
    B_FULL = 0, B_EMPTY = B_FULL + kStages, B_QFULL = B_EMPTY + kStages, B_QEMPTY, B_SFULL,
    B_SEMPTY = B_SFULL + 2, B_PFULL = B_SEMPTY + 2, B_VDONE = B_PFULL + 2, B_OFREE = B_VDONE + 2, B_XFULL,
    B_XEMPTY = B_XFULL + 2, B_MH = B_XEMPTY + 2, B_STATS = B_MH + 2, B_FIN = B_STATS + 4,
    B_CONV = B_FIN + 1, B_CREAD = B_CONV + kStages, B_COUNT = B_CREAD + 1
};
static_assert(B_COUNT * 8 <= kBarBytes, "barrier area");

// fp8 cache rows (kFp8): a stage receives the tile's E4M3 latent half (64 rows x 256 bytes)
// in the upper half of its latent area, the rows' four fp32 group scales just below, and
// the bf16 rotary half in its usual place; the epilogue warps then write the bf16 latent
// chunks over the whole latent area (in place: every code and scale is read first).
constexpr uint32_t kF8Codes = 16384;                     // stage offset of the codes
constexpr uint32_t kF8Scales = 15360;                    // stage offset of the scales (16 B per row)
constexpr uint32_t kF8StageTx = 64 * 256 + 64 * 16 + kTRope;
constexpr uint32_t kOffTslot = kOffBar + kBarBytes;
constexpr uint32_t kOffAbort = kOffTslot + 4;

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;          // O_r: 256 fp32 columns
constexpr uint32_t kColQ = 256;        // latent chunks 0, 1 of Q'_r: 128 bf16 = 64 columns
constexpr uint32_t kColP = 320;        // P[2] (by tile parity): 128 heads x 64 rows bf16 = 2 x 32 columns,
                                       // the A operand of the value MMA
constexpr uint32_t kColS = 384;        // S[2] (by tile parity): 2 x 64 fp32 columns

struct TcArgs {
    const __nv_bfloat16* qp;           // folded queries [batch * n_h, 576]
    const int64_t* row_off;
    const int32_t* seq_len;            // real lengths when the schedule pads sequences to whole tiles, else null
    const int32_t* block_table;        // paged cache (null: contiguous, row_off)
    int32_t block_size, max_blocks;
    int32_t rope_x0;                   // column of the rotary part in its tensor map (512 packed, 0 split)
    const int64_t* cum;
    const WorkerStart* wstart;         // where each worker starts
    __nv_bfloat16* o_lat;
    float* lse;
    float* part_o;
    float* part_l;
    int32_t* dev_status;
    uint64_t wait_ns;                  // limit of every wait of the pipeline
    int n_h;
    int batch;
};

struct Seg {
    int b;
    int64_t lo, hi, len;
    bool complete;
    int64_t slot;
};

// Walks the sequences that a worker's range of the flattened context touches
// (identical in every role of both CTAs).
// kTiled: the context is flattened in whole tiles (a paged cache), so a sequence spans
// its length rounded up to a tile and its real length comes from real_len; the rows past
// its length are never visited (range boundaries are tile-aligned).  A separate
// instantiation keeps the contiguous walk free of that work.
// kKeep: the walk keeps the current sequence's span (its first one from the start record),
// so its first piece needs no load of cum; the roles on the way to the first tile (the TMA
// producer, the loaders of Q') use it, the others re-read cum and hold fewer registers.
template <bool kTiled, bool kKeep = false>
struct SegWalk {
    const int64_t* cum;
    const int32_t* real_len;
    int64_t cur, end;
    int64_t seq0, seq1;                // cum[b], cum[b + 1]
    int b, g;
    bool first;
    // w: the worker's start record, written by the schedule kernel
    __device__ void init(const int64_t* c, const int32_t* rl, const WorkerStart& w, int gi) {
        cum = c;
        real_len = rl;
        g = gi;
        cur = w.begin;
        end = w.end;
        b = w.b;
        if (kKeep) {
            seq0 = w.seq0;
            seq1 = w.seq1;
        }
        first = true;
    }
    __device__ bool next(Seg& s) {
        if (cur >= end) return false;
        if (kKeep) {
            while (seq1 <= cur) {
                ++b;
                seq0 = seq1;
                seq1 = cum[b + 1];
            }
        } else {
            while (cum[b + 1] <= cur) ++b;
            seq0 = cum[b];
            seq1 = cum[b + 1];
        }
        const int64_t span = seq1 - seq0;
        s.b = b;
        s.len = kTiled ? min(span, (int64_t)real_len[b]) : span;
        s.lo = cur - seq0;
        s.hi = min(s.len, end - seq0);
        s.complete = (s.lo == 0 && s.hi == s.len);
        s.slot = 2 * (int64_t)g + (first ? 0 : 1);
        cur = (kTiled && s.hi == s.len) ? seq0 + span : seq0 + s.hi;
        first = false;
        return true;
    }
};

__device__ __forceinline__ int tiles_of(const Seg& s) { return (int)((s.hi - s.lo + kTok - 1) / kTok); }

// The worker's tiles in order: global tile index T, piece index si, tile t of ntiles.
template <bool kTiled, bool kKeep = false>
struct TileIt {
    SegWalk<kTiled, kKeep> walk;
    Seg seg;
    int t = -1, ntiles = 0;
    uint32_t T = 0xffffffffu, si = 0xffffffffu;
    __device__ bool next() {
        if (t + 1 < ntiles) { ++t; ++T; return true; }
        if (!walk.next(seg)) return false;
        ++si;
        ++T;
        t = 0;
        ntiles = tiles_of(seg);
        return true;
    }
    __device__ bool first_tile() const { return t == 0; }
    __device__ bool last_tile() const { return t == ntiles - 1; }
    __device__ int valid_rows() const {
        return (int)min((int64_t)kTok, seg.hi - seg.lo - (int64_t)t * kTok);
    }
};

struct Ctl {
    volatile int* abort;
    int32_t* dev_status;
    uint64_t limit_ns;
};

// Bounded wait: true when the phase completed; false on abort or time-out (which
// also raises the abort flag and MLA_DEV_TIMEOUT).
template <bool kCluster>
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, const Ctl& c) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*c.abort) return false;
        if (globaltimer_ns() - t0 > c.limit_ns) {
            *c.abort = 1;
            atomicOr(c.dev_status, MLA_DEV_TIMEOUT);
            return false;
        }
    }
}

// Warp-uniform form for warps that issue tcgen05.ld/st (all 32 lanes on one path).
template <bool kCluster>
__device__ __forceinline__ bool wwait(uint32_t bar, uint32_t parity, const Ctl& c) {
    const bool ok = wait<kCluster>(bar, parity, c);
    return __all_sync(0xffffffffu, ok);
}

// Wait used while draining after an abort: ignores the abort flag, bounded in time.
__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kTimeoutNs) return;
}

__device__ __forceinline__ uint64_t kdesc128(uint32_t a) { return smem_desc(a, 16, 1024, kSwizzle128B); }

// One TMA copy of a 3-D box (x, y, z): here a tile's four 64-column latent chunks, which land as
// four consecutive 64-row x 128-byte swizzled boxes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            int32_t z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}

// Row i of Q'_r's latent chunks 2 and 3 into shared memory: two 128-head x 64-column bf16
// chunks, K-major with the 128B swizzle (16-byte unit c of row i stored at unit c ^ (i & 7)).
// src: the row's 16 uint4 (chunk 2 then chunk 3), or null for a zero row.
__device__ __forceinline__ void store_ql_row(uint8_t* ql, int i, const uint4* src) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = src ? src[8 * h + c] : zero;
#pragma unroll
        for (int c = 0; c < 8; ++c) *(uint4*)(ql + h * kQLChunk + i * 128 + ((c ^ (i & 7)) << 4)) = v[c];
    }
}
__device__ __forceinline__ uint64_t kdesc64(uint32_t a) { return smem_desc(a, 16, 512, kSwizzle64B); }
// MN-major 128B-swizzled B: 64-column atoms one TMA box (kTBox bytes) apart, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t mndesc128(uint32_t a) { return smem_desc(a, kTBox, 1024, kSwizzle128B); }

// 2^x with the special-function unit (relative error about 2^-22; the result is
// rounded to bf16 right after, and exp2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// kTiled: paged cache (block table).  kFp8: rows of the fp8 layout (contiguous); map_c128
// then covers the rows as bytes (box 256 x 64 rows), map_c64 the rotary bytes (64 x 64, 64B
// swizzle) and map_sc the group scales (16 x 64); for bf16 rows map_sc is unused.
template <bool kTiled, bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
split_tc_kernel(const __grid_constant__ CUtensorMap map_c128, const __grid_constant__ CUtensorMap map_c64,
                const __grid_constant__ CUtensorMap map_sc, TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw;
    if (smem_addr(sm) & 1023u) {        // the same in every CTA of the launch: all return here
        if (threadIdx.x == 0) atomicOr(a.dev_status, MLA_DEV_SMEM_ALIGN);
        return;
    }
    const uint32_t base = smem_addr(sm);
    const uint32_t sStage = base + kOffStage, sX = base + kOffX;
    uint64_t* bars = (uint64_t*)(sm + kOffBar);
    uint32_t* tslot = (uint32_t*)(sm + kOffTslot);
    float* stats = (float*)(sm + kOffStats);
    volatile int* abort_flag = (volatile int*)(sm + kOffAbort);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    Ctl ctl{abort_flag, a.dev_status, a.wait_ns};

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
            mbar_init(bar(B_CONV + i), 128);          // fp8: the epilogue warps converted stage i
        }
        mbar_init(bar(B_CREAD), 128);                 // fp8: every converter has read its codes
        // Q' of a piece is in place: the first piece's is loaded by the softmax groups (latent
        // part) and the epilogue warps (rotary part), later ones by the epilogue warps alone,
        // which then arrive three times each
        mbar_init(bar(B_QFULL), 384);
        mbar_init(bar(B_QEMPTY), 2);                  // one commit per score issuer
        // score and value barriers per tile parity: each phase of one is waited for in
        // order by the issuer or group that owns (or follows) those tiles
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_SEMPTY + i), 128);
            mbar_init(bar(B_VDONE + i), 1);
            mbar_init(bar(B_PFULL + i), 128);       // the group that owns the tile parity
        }
        mbar_init(bar(B_OFREE), 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_XFULL + i), 1);
            mbar_init(bar(B_XEMPTY + i), 4);            // one credit from each warp of the peer's group
            mbar_init(bar(B_MH + i), 128);
        }
        for (int i = 0; i < 4; ++i) mbar_init(bar(B_STATS + i), 256);
        mbar_init(bar(B_FIN), 3);                     // one commit per MMA issuer
        *abort_flag = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 2) {
        tmem_alloc(smem_addr(tslot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&map_c128);
        prefetch_tmap(&map_c64);
    }
    tc_fence_before();
    cluster_sync();                 // barriers of both CTAs initialised before any remote signal
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // Everything above touches only this CTA's shared and tensor memory.  Everything below
    // reads what the kernels before this one wrote: launched behind them (programmatic
    // dependent launch), the kernel waits here, so its set-up overlaps their tail.
    pdl_wait();
    pdl_trigger();                  // the merge kernel behind this one may be scheduled
    const int g = blockIdx.x >> 1;
    const WorkerStart W = a.wstart[g];                 // one load: range, first sequence and row
    const bool active = W.begin < W.end;               // the same for both CTAs of the pair

    // Registers: 128 per thread at launch; each role re-sizes its warpgroup's share
    // first thing in its own branch (80 + 168 + 168 + 96 = 4 x 128).
    if (active) {
        if (warp < 4) reg_alloc_dec<80>();
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producer
            // One thread loads the cache tiles into the ring: one copy for a tile's latent
            // half and one for its rotary half.  (It paces the kernel; the exchange credits
            // are sent by the softmax warps themselves.)
            if (lane == 0) {
                TileIt<kTiled, true> ip;                            // next tile to load
                ip.walk.init(a.cum, a.seq_len, W, g);
                bool mp = ip.next();
                // cache row of the next tile to load, fetched one tile ahead (a block-table
                // entry is a global load; its latency hides behind the wait for a free stage)
                auto tile_row = [&](const TileIt<kTiled, true>& t) -> int {
                    const int64_t pos = t.seg.lo + (int64_t)t.t * kTok;
                    if (!kTiled)                                              // contiguous
                        return (int)((t.seg.b == W.b ? W.row0 : a.row_off[t.seg.b]) + pos);
                    return a.block_table[(int64_t)t.seg.b * a.max_blocks + pos / a.block_size] * a.block_size +
                           (int)(pos % a.block_size);
                };
                int next_y = mp ? tile_row(ip) : 0;
                uint32_t issued = 0;
                uint64_t t_prog = globaltimer_ns();
                while (mp) {
                    bool prog = false;
                    {
                        const uint32_t T = ip.T, st = T % kStages;
                        if (mbar_test_wait(bar(B_EMPTY + st), ((T / kStages) & 1) ^ 1)) {
                            const uint32_t dst = sStage + st * kStageBytes;
                            const int y = next_y;
                            if constexpr (kFp8) {
                                // codes of this CTA's latent half, the row's group scales, the
                                // rotary half (bf16, 64B swizzle), all as bytes of the row
                                mbar_expect_tx(bar(B_FULL + st), kF8StageTx);
                                tma_load_2d(dst + kF8Codes, &map_c128, (int)rank * 256, y, bar(B_FULL + st));
                                tma_load_2d(dst + kF8Scales, &map_sc, 512, y, bar(B_FULL + st));
                                tma_load_2d(dst + 4 * kTBox, &map_c64, 528 + (int)rank * 64, y, bar(B_FULL + st));
                            } else {
                                mbar_expect_tx(bar(B_FULL + st), kStageBytes);
                                tma_load_3d(dst, &map_c128, 0, y, (int)rank * 4, bar(B_FULL + st));
                                tma_load_2d(dst + 4 * kTBox, &map_c64, a.rope_x0 + rank * kRopeHalf, y, bar(B_FULL + st));
                            }
                            issued = T + 1;
                            mp = ip.next();
                            if (mp) next_y = tile_row(ip);
                            prog = true;
                        }
                    }
                    if (prog) {
                        // (the clock read of an idle round also spaces the polls of the barriers,
                        // which the arriving threads and the copy engine share)
                        t_prog = globaltimer_ns();
                    } else {
                        if (*abort_flag) break;
                        if (globaltimer_ns() - t_prog > a.wait_ns) {
                            *abort_flag = 1;
                            atomicOr(a.dev_status, MLA_DEV_TIMEOUT);
                            break;
                        }
                    }
                }
                // drain: every copy this thread issued has landed before the CTA may exit
                for (uint32_t k = 0; k < kStages && k < issued; ++k) {
                    const uint32_t Tk = issued - 1 - k;
                    drain(bar(B_FULL + Tk % kStages), (Tk / kStages) & 1);
                }
            }
        } else if (warp == 1 || warp == 3) {
            // ------------------------------------------------------------ score MMA issuers
            // Warp 1 issues the score MMAs of the even tiles into S[0], warp 3 those of the odd
            // tiles into S[1]: two issue streams, so a score never waits for the previous
            // tile's scores to be read.  With an even ring depth each stage, and so each
            // FULL barrier, belongs to one issuer.  Both wait for every piece's Q' and both
            // release it (QEMPTY counts two commits).
            if (lane == 0) {
                const uint32_t par = warp == 1 ? 0u : 1u;
                const uint32_t id_s = idesc_bf16_f32(kHeads, kTok, 0, 0);
                const uint32_t sQL = base + kOffQL, sQR = base + kOffQR;
                TileIt<kTiled> it;
                it.walk.init(a.cum, a.seq_len, W, g);
                bool ok = true;
                while (ok && it.next()) {
                    const uint32_t T = it.T;
                    if (it.first_tile() && !(ok = wait<false>(bar(B_QFULL), it.si & 1, ctl))) break;
                    if ((T & 1u) == par) {
                        const uint32_t st = T % kStages;
                        if (!(ok = wait<false>(bar((kFp8 ? B_CONV : B_FULL) + st), (T / kStages) & 1, ctl))) break;
                        if (T >= 2 && !(ok = wait<false>(bar(B_SEMPTY + par), ((T >> 1) - 1) & 1, ctl))) break;
                        tc_fence_after();
                        const uint32_t stage = sStage + st * kStageBytes;
                        const uint32_t d = tmem + kColS + 64 * par;
                        // latent chunks 0, 1: A (Q') from tensor memory; chunks 2, 3 and the
                        // rotary part: A from shared memory
                        for (int kk = 0; kk < 8; ++kk)
                            mma_bf16_ts(d, tmem + kColQ + 8 * kk, kdesc128(stage + (kk >> 2) * kTBox + 32 * (kk & 3)),
                                        id_s, kk ? 1u : 0u);
                        for (int kk = 8; kk < 16; ++kk)
                            mma_bf16(d, kdesc128(sQL + ((kk >> 2) - 2) * kQLChunk + 32 * (kk & 3)),
                                     kdesc128(stage + (kk >> 2) * kTBox + 32 * (kk & 3)), id_s, 1u);
                        for (int kk = 0; kk < 2; ++kk)
                            mma_bf16(d, kdesc64(sQR + 32 * kk), kdesc64(stage + 4 * kTBox + 32 * kk), id_s, 1u);
                        mma_commit(bar(B_SFULL + par));
                    }
                    if (it.last_tile()) mma_commit(bar(B_QEMPTY));
                }
                mma_commit(bar(B_FIN));
                drain(bar(B_FIN), 0);
            }
        } else if (warp == 2) {
            // ------------------------------------------------------------ value MMA issuer
            // O_r += P C_r: P (bf16, 128 heads x 64 rows) from tensor memory, the tile's
            // latent half as an MN-major B operand.  A stage is released here: the value MMA
            // of a tile always completes after its score MMA (the softmax in between needs it).
            if (lane == 0) {
                const uint32_t id_o = idesc_bf16_f32(kHeads, kLatHalf, 0, 1);
                TileIt<kTiled> it;
                it.walk.init(a.cum, a.seq_len, W, g);
                bool ok = true;
                while (ok && it.next()) {
                    const uint32_t T = it.T, st = T % kStages;
                    if (!(ok = wait<false>(bar(B_PFULL + (T & 1)), (T >> 1) & 1, ctl))) break;
                    if (it.first_tile() && it.si > 0 && !(ok = wait<false>(bar(B_OFREE), (it.si - 1) & 1, ctl))) break;
                    tc_fence_after();
                    const uint32_t stage = sStage + st * kStageBytes;
                    for (int k = 0; k < kTok / 16; ++k)
                        mma_bf16_ts(tmem + kColO, tmem + kColP + 32 * (T & 1) + 8 * k, mndesc128(stage + 2048 * k), id_o,
                                 (it.first_tile() && k == 0) ? 0u : 1u);
                    mma_commit(bar(B_EMPTY + st));
                    mma_commit(bar(B_VDONE + (T & 1)));
                }
                // every MMA this thread issued has completed before the CTA may tear down
                mma_commit(bar(B_FIN));
                drain(bar(B_FIN), 0);
            }
        } else if (warp >= 4 && warp < 12) {
            // ------------------------------------------------------------ softmax / exchange
            reg_alloc_inc<168>();
            // Two groups of four warps take alternate tiles (group grp owns the tiles T with
            // T % 2 == grp), so one group's exchange overlaps the other's exponentials.  The
            // running maximum is handed from the owner of tile T-1 to the owner of tile T
            // through shared memory; each group keeps its own sum relative to the maximum it
            // last saw, and the epilogue combines the two.
            const int grp = (warp - 4) >> 2;
            const int i = (tid - 128) & (kHeads - 1);      // head row == TMEM lane
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t xb = (uint32_t)grp;              // this group's exchange buffer
            const uint32_t peer_x = mapa(sX + xb * kXBytes, peer);
            const uint32_t peer_xfull = mapa(bar(B_XFULL + xb), peer);
                float* mshare = (float*)(sm + kOffMh);
            {
                // the first piece's Q' (latent part): group grp loads the 64-column chunks
                // 2 grp and 2 grp + 1 of this CTA's half (group 0 into tensor memory, group 1
                // into shared memory), one round of loads, while the epilogue warps load the
                // rotary part (at the start of a launch the three warpgroups together cut the
                // wait for Q')
                SegWalk<kTiled, true> w0;
                w0.init(a.cum, a.seq_len, W, g);
                Seg s0;
                if (w0.next(s0)) {
                    const bool row_ok = i < a.n_h;
                    const uint4* src = reinterpret_cast<const uint4*>(
                        a.qp + ((int64_t)s0.b * a.n_h + (row_ok ? i : 0)) * kRowElems) + rank * 32 + 16 * grp;
                    if (grp == 0) {                 // chunks 0, 1: tensor memory
                        const uint4 zero = make_uint4(0, 0, 0, 0);
                        uint32_t r0[32], r1[32];
    #pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint4 v = row_ok ? src[c] : zero;
                            const uint4 w = row_ok ? src[8 + c] : zero;
                            r0[4 * c] = v.x; r0[4 * c + 1] = v.y; r0[4 * c + 2] = v.z; r0[4 * c + 3] = v.w;
                            r1[4 * c] = w.x; r1[4 * c + 1] = w.y; r1[4 * c + 2] = w.z; r1[4 * c + 3] = w.w;
                        }
                        tmem_st32u(tmem + lane_base + kColQ, r0);
                        tmem_st32u(tmem + lane_base + kColQ + 32, r1);
                        tmem_wait_st();
                    } else {                        // chunks 2, 3: shared memory
                        store_ql_row(sm + kOffQL, i, row_ok ? src : nullptr);
                        fence_proxy_async_smem();
                    }
                    tc_fence_before();
                    mbar_arrive(bar(B_QFULL));
                }
            }
            TileIt<kTiled> co;
            co.walk.init(a.cum, a.seq_len, W, g);
            bool ok = true;
            float m_g = -INFINITY, l_g = 0.f;
            while (ok && co.next()) {
                const uint32_t T = co.T;
                if (co.first_tile()) { m_g = -INFINITY; l_g = 0.f; }
                if ((T & 1u) == xb) {
                    const uint32_t st = T % kStages;
                    // this CTA's partial scores: out of TMEM, then to the peer
                    float s[kTok];
                    if (!(ok = wwait<false>(bar(B_SFULL + xb), (T >> 1) & 1, ctl))) break;
                    tc_fence_after();
                    tmem_ld32(tmem + lane_base + kColS + 64 * xb, *reinterpret_cast<float(*)[32]>(&s[0]));
                    tmem_ld32(tmem + lane_base + kColS + 64 * xb + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(B_SEMPTY + xb));
                    // the peer has finished reading what this group sent for tile T - 2
                    if (T >= 2 && !(ok = wwait<true>(bar(B_XEMPTY + xb), ((T >> 1) - 1) & 1, ctl))) break;
                    if (i == 0) mbar_expect_tx(bar(B_XFULL + xb), kXBytes);      // the peer's copy of tile T
                    {
                        // block-scaled fp16: s = off + r with off the partial of the tile's first
                        // row (always a row of the piece), so each r is rounded relative to the
                        // spread of the partial within the tile, not to its magnitude
                        // (|error| <= 2^-11 |s - off|); a difference beyond the fp16 range
                        // saturates at +-65504 instead of becoming infinite
                        const float off = s[0];
    #pragma unroll
                        for (int c = 0; c < kTok / 8; ++c) {
                            uint32_t w[4];
    #pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack_half2_satfinite(s[8 * c + 2 * e] - off, s[8 * c + 2 * e + 1] - off);
                            st_async_v4u(peer_x + (uint32_t)(c * kHeads + i) * 16, w[0], w[1], w[2], w[3], peer_xfull);
                        }
                        st_async_f32(peer_x + kXResBytes + (uint32_t)i * 4, off, peer_xfull);
                    }
                    // add the peer's partial scores of tile T
                    if (!(ok = wwait<true>(bar(B_XFULL + xb), (T >> 1) & 1, ctl))) break;
                    {
                        const uint8_t* xbase = sm + kOffX + xb * kXBytes;
                        const uint4* xr = reinterpret_cast<const uint4*>(xbase) + i;
                        const float off = reinterpret_cast<const float*>(xbase + kXResBytes)[i];
    #pragma unroll
                        for (int c = 0; c < kTok / 8; ++c) {
                            const uint4 v = xr[c * kHeads];
                            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                                s[8 * c + 2 * e] += f.x + off;
                                s[8 * c + 2 * e + 1] += f.y + off;
                            }
                        }
                    }
                    // this warp has read its rows of X: pass the credit to the peer (relaxed, no
                    // data is published; the loads above have returned)
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote_relaxed(mapa(bar(B_XEMPTY + xb), peer));
                    // rows past the end of this piece do not count (only the last tile of a
                    // piece is partial)
                    const int valid = co.valid_rows();
                    if (valid < kTok) {
    #pragma unroll
                        for (int j = 0; j < kTok; ++j)
                            if (j >= valid) s[j] = -INFINITY;
                    }
                    // tile maximum: eight running maxima, then a tree (short dependency chains)
                    float m8[8];
    #pragma unroll
                    for (int j = 0; j < 8; ++j)
                        m8[j] = fmaxf(fmaxf(fmaxf(s[j], s[j + 8]), fmaxf(s[j + 16], s[j + 24])),
                                      fmaxf(fmaxf(s[j + 32], s[j + 40]), fmaxf(s[j + 48], s[j + 56])));
    #pragma unroll
                    for (int w = 4; w >= 1; w >>= 1)
    #pragma unroll
                        for (int j = 0; j < w; ++j) m8[j] = fmaxf(m8[j], m8[j + w]);
                    const float mt = m8[0];
                    // the running maximum after tile T - 1 (decided by the other group)
                    if (T > 0) {
                        if (!(ok = wwait<false>(bar(B_MH + ((T - 1) & 1)), ((T - 1) >> 1) & 1, ctl))) break;
                        const float mp = mshare[((T - 1) & 1) * kHeads + i];
                        if (!co.first_tile() && mp != m_g) { l_g *= fast_exp2(m_g - mp); m_g = mp; }
                    }
                    // lazy maximum: move it (and rescale) only when a score exceeds it by 2^8
                    const bool need = mt > m_g + 8.f;
                    float alpha = 1.f;
                    if (need) {
                        alpha = fast_exp2(m_g - mt);
                        m_g = mt;
                        l_g *= alpha;
                    }
                    mshare[(T & 1) * kHeads + i] = m_g;
                    mbar_arrive(bar(B_MH + (T & 1)));
                    // P tile (bf16) for the value MMA; the sum uses the rounded values
                    uint32_t packed[kTok / 2];
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};     // four partial sums (short chains)
    #pragma unroll
                    for (int j = 0; j < kTok / 2; ++j) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(fast_exp2(s[2 * j] - m_g),
                                                                        fast_exp2(s[2 * j + 1] - m_g));
                        ls[j & 3] += __low2float(h2) + __high2float(h2);
                        packed[j] = *reinterpret_cast<const uint32_t*>(&h2);
                    }
                    l_g += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    // P[T % 2] is free once the value MMA of tile T - 2 has finished
                    if (T >= 2) {
                        if (!(ok = wwait<false>(bar(B_VDONE + (T & 1)), ((T - 2) >> 1) & 1, ctl))) break;
                        tc_fence_after();
                    }
                    if (!co.first_tile() && __any_sync(0xffffffffu, need)) {
                        // a moved maximum rescales O: after the value MMA of tile T - 1 (whose P
                        // is on the old scale), before that of tile T (held back by PFULL)
                        if (!(ok = wwait<false>(bar(B_VDONE + ((T - 1) & 1)), ((T - 1) >> 1) & 1, ctl))) break;
                        tc_fence_after();
                        for (int c = 0; c < kLatHalf / 16; ++c) {
                            float o[16];
                            tmem_ld16(tmem + lane_base + kColO + 16 * c, o);
                            tmem_wait_ld();
                            uint32_t u[16];
    #pragma unroll
                            for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(o[j] * alpha);
                            tmem_st16(tmem + lane_base + kColO + 16 * c, u);
                        }
                    }
                    // row i of P into tensor memory (lane i, two bf16 per column, the lower row
                    // in the low half: the A operand layout of the value MMA)
                    tmem_st32u(tmem + lane_base + kColP + 32 * xb, packed);
                    if (valid < kTok) {
                        // the value MMA must not see rows of the tile beyond the piece (they may
                        // hold anything): zero them in this CTA's latent half of the stage
                        uint8_t* stage = sm + kOffStage + st * kStageBytes;
                        for (int e = i; e < (kTok - valid) * 4 * 8; e += 128) {
                            const int r = valid + e / 32, box = (e / 8) & 3, ch = e & 7;
                            *(uint4*)(stage + box * kTBox + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();               // the zeroed rows to the tensor core
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar(B_PFULL + xb));
                }
                if (co.last_tile()) {
                    // this group's share of the piece's statistics
                    float* sp = stats + ((co.si & 3) * 2 + grp) * 2 * kHeads;
                    sp[i] = m_g;
                    sp[kHeads + i] = l_g;
                    mbar_arrive(bar(B_STATS + (co.si & 3)));
                }
            }
        } else if (warp >= 12) {
            // ------------------------------------------------------------ Q' loader / epilogue
            reg_alloc_dec<96>();
            const int i = tid - 384;                        // head row == TMEM lane
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            SegWalk<kTiled, !kFp8> walk;              // (fp8: measured faster without the kept span)
            walk.init(a.cum, a.seq_len, W, g);
            Seg cur, nxt;
            bool have = walk.next(cur);
            uint32_t si = 0, t_end = 0;                     // piece index, global index past its last tile
            // Q' of one piece (zero rows for heads >= n_h): latent chunks 0, 1 into tensor
            // memory, latent chunks 2, 3 and the rotary part into shared memory.  first: the
            // softmax groups load the latent part (the first piece of a launch), this
            // warpgroup only the rotary part.
            auto load_q = [&](const Seg& sg, bool first) {
                const bool row_ok = i < a.n_h;
                const uint4* src = reinterpret_cast<const uint4*>(a.qp + ((int64_t)sg.b * a.n_h + (row_ok ? i : 0)) * kRowElems);
                const uint4 zero = make_uint4(0, 0, 0, 0);
                {   // rotary columns [512 + 32r, 512 + 32r + 32): the A operand of the rotary
                    // score MMAs (row i: 64 bytes, 16-byte chunk c stored at chunk
                    // c ^ ((i >> 1) & 3), the 64B swizzle)
                    uint8_t* qrow = sm + kOffQR + i * 64;
    #pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *(uint4*)(qrow + ((c ^ ((i >> 1) & 3)) << 4)) = row_ok ? src[64 + rank * 4 + c] : zero;
                    fence_proxy_async_smem();
                }
                if (first) {
                    tc_fence_before();
                    mbar_arrive(bar(B_QFULL));
                    return;
                }
                {   // latent chunks 0, 1 (columns [256r, 256r + 128)) into tensor memory
                    uint32_t r0[32], r1[32];
    #pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint4 v = row_ok ? src[rank * 32 + c] : zero;
                        const uint4 w = row_ok ? src[rank * 32 + 8 + c] : zero;
                        r0[4 * c] = v.x; r0[4 * c + 1] = v.y; r0[4 * c + 2] = v.z; r0[4 * c + 3] = v.w;
                        r1[4 * c] = w.x; r1[4 * c + 1] = w.y; r1[4 * c + 2] = w.z; r1[4 * c + 3] = w.w;
                    }
                    tmem_st32u(tmem + lane_base + kColQ, r0);
                    tmem_st32u(tmem + lane_base + kColQ + 32, r1);
                }
                // latent chunks 2, 3 (columns [256r + 128, 256r + 256)) into shared memory
                store_ql_row(sm + kOffQL, i, row_ok ? src + rank * 32 + 16 : nullptr);
                fence_proxy_async_smem();
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive_cnt(bar(B_QFULL), 3);
            };
            // fp8 rows: turn the landed codes of tile T into the bf16 latent chunks the MMAs read.
            // Thread i takes row i / 2, columns [128 (i % 2), +128) of this CTA's half (one
            // group, one scale); all 128 read before any writes (CREAD), since the output
            // covers the bytes the codes and scales landed in.
            auto convert_tile = [&](uint32_t T) -> bool {
                const uint32_t st = T % kStages;
                if (!wwait<false>(bar(B_FULL + st), (T / kStages) & 1, ctl)) return false;
                uint8_t* stage = sm + kOffStage + st * kStageBytes;
                const int r = i >> 1, hh = i & 1;
                const uint4* src = reinterpret_cast<const uint4*>(stage + kF8Codes + r * 256 + 128 * hh);
                uint4 v[8];
    #pragma unroll
                for (int c = 0; c < 8; ++c) v[c] = src[c];
                const float scale = reinterpret_cast<const float*>(stage + kF8Scales + r * 16)[2 * rank + hh];
                mbar_arrive(bar(B_CREAD));
                if (!wwait<false>(bar(B_CREAD), T & 1, ctl)) return false;
                // code * scale is exact in bf16: the scale is a power of two (an integer-only
                // form that adds the exponent to the code's bits measured slower than these
                // conversions)
    #pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    // one code vector a round, the next ones moved down (a rolled loop keeps
                    // the conversion's code small)
                    const uint4 vc = v[0];
    #pragma unroll
                    for (int q = 0; q < 7; ++q) v[q] = v[q + 1];
                    const uint32_t w[4] = {vc.x, vc.y, vc.z, vc.w};   // 16 codes, lowest column first
                    uint32_t o[8];
    #pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(w[e >> 1] >> (16 * (e & 1)));
                        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
                        const float2 f = __half22float2(__half2(hr));
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * scale, f.y * scale);
                        o[e] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    // columns 16c .. 16c + 15 of the thread's 128: chunk j, 16-byte units u, u + 1
                    // (K-major, 128B swizzle: unit u of row r stored at unit u ^ (r & 7))
                    const int col = 128 * hh + 16 * c;
                    const int j = col >> 6, u = (col & 63) >> 3;
                    uint8_t* rowp = stage + j * kTBox + r * 128;
                    *(uint4*)(rowp + ((u ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    *(uint4*)(rowp + (((u + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(B_CONV + st));
                return true;
            };
            bool ok = true;
            if (have) load_q(cur, true);
            while (ok && have) {
                const uint32_t t_begin = t_end;
                t_end += (uint32_t)tiles_of(cur);
                if constexpr (kFp8) {
                    // this piece's tiles first: its scores (and so the next piece's Q') wait for them
                    for (uint32_t T = t_begin; ok && T < t_end; ++T) ok = convert_tile(T);
                    if (!ok) break;
                }
                const bool more = walk.next(nxt);
                if (more) {
                    // the score MMAs of this piece are done with Q'
                    if (!(ok = wwait<false>(bar(B_QEMPTY), si & 1, ctl))) break;
                    tc_fence_after();
                    load_q(nxt, false);
                }
                // epilogue of this piece: O_r / l, log2-sum-exp
                if (!(ok = wwait<false>(bar(B_STATS + (si & 3)), (si >> 2) & 1, ctl))) break;
                const float* sp = stats + (si & 3) * 4 * kHeads;
                const float m0 = sp[i], l0 = sp[kHeads + i], m1 = sp[2 * kHeads + i], l1 = sp[3 * kHeads + i];
                const float m_fin = fmaxf(m0, m1);
                const float l_fin = l0 * exp2f(m0 - m_fin) + l1 * exp2f(m1 - m_fin);
                if (!(ok = wwait<false>(bar(B_VDONE + ((t_end - 1) & 1)), ((t_end - 1) >> 1) & 1, ctl))) break;
                tc_fence_after();
                const float inv = 1.f / l_fin;
                const float lse2 = m_fin + log2f(l_fin);
                const bool row_ok = i < a.n_h;
                for (int c = 0; c < kLatHalf / 32; ++c) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + kColO + 32 * c, o);
                    tmem_wait_ld();
                    if (!row_ok) continue;
                    const int col = (int)rank * kLatHalf + 32 * c;
                    if (cur.complete) {
                        __nv_bfloat16* dst = a.o_lat + ((int64_t)cur.b * a.n_h + i) * 512 + col;
    #pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
    #pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[8 * q + 2 * e] * inv, o[8 * q + 2 * e + 1] * inv);
                                w[e] = *reinterpret_cast<const uint32_t*>(&h2);
                            }
                            *(uint4*)(dst + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        float* dst = a.part_o + (cur.slot * a.n_h + i) * 512 + col;
    #pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *(float4*)(dst + 4 * q) = make_float4(o[4 * q] * inv, o[4 * q + 1] * inv,
                                                                  o[4 * q + 2] * inv, o[4 * q + 3] * inv);
                    }
                }
                if (row_ok && rank == 0) {
                    if (cur.complete) { if (a.lse) a.lse[(int64_t)cur.b * a.n_h + i] = lse2 * kLn2; }
                    else a.part_l[cur.slot * a.n_h + i] = lse2;
                }
                tc_fence_before();
                mbar_arrive(bar(B_OFREE));
                cur = nxt;
                have = more;
                ++si;
            }
        }
    }
    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    cluster_sync();                 // the peer no longer writes into this CTA's shared memory
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    });
    return g_encode != nullptr;
}

// The latent columns as a 3-D tensor (64 columns, rows, 64-column chunks): one box of
// 64 columns x kTok rows x 4 chunks is a tile's latent half.
bool encode_latent_3d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t stride) {
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {stride * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kTok, 4};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of bytes (the fp8 layout): cols bytes per row, rows rows of `stride` bytes, box bx x by.
bool encode_u8(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t stride, uint32_t bx,
               uint32_t by, CUtensorMapSwizzle sw) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {stride};
    cuuint32_t box[2] = {bx, by};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t stride, uint32_t bx,
               uint32_t by, CUtensorMapSwizzle sw) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {stride * 2};
    cuuint32_t box[2] = {bx, by};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// How many 2-CTA clusters of the attention kernel can be resident at once on the
// current device (a cluster must sit inside one GPC, so this can be below sm_count/2);
// 0 when the query is not available.
int resident_pairs() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaFuncSetAttribute(split_tc_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) ==
            cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * 256);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = kSmemBytes;
            if (cudaOccupancyMaxActiveClusters(&n, split_tc_kernel<false, false>, &cfg) != cudaSuccess) n = 0;
        }
        (void)cudaGetLastError();
        cache[dev] = n > 0 ? n : -1;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

int tc_workers(int64_t max_total_rows, int sm_count) {
    int64_t w = sm_count / 2;                           // one 2-CTA cluster per SM pair
    const int resident = resident_pairs();              // all workers in one wave
    if (resident > 0 && w > resident) w = resident;
    const int64_t by_rows = (max_total_rows + kTok - 1) / kTok;
    if (w > by_rows) w = by_rows;
    if (w < 1) w = 1;
    return (int)w;
}

cudaError_t launch_split_tc(const mla_dims& d, int batch, int workers, const void* qp,
                            int64_t q_rows, const CacheView& cv, const int32_t* seq_len,
                            const int64_t* row_off, const int64_t* cum, const void* sched,
                            const WorkerStart* wstart, void* o_lat, float* lse, float* part_o,
                            float* part_l, int32_t* dev_status, cudaStream_t s, bool pdl, bool fp8) {
    (void)q_rows;
    (void)sched;                                    // the kernel reads the start records instead
    if (!get_encoder()) return cudaErrorNotSupported;
    CUtensorMap mc128, mc64, msc;
    if (fp8) {
        // rows of the fp8 layout as bytes: this CTA's 256 codes, the 16 bytes of group scales,
        // its 64 rotary bytes (64B swizzle, as the rotary score MMAs expect)
        if (cv.block_table || cv.pe) return cudaErrorInvalidValue;
        const uint64_t rb = (uint64_t)kFp8RowBytes(512, 64);
        if (!encode_u8(&mc128, cv.kv, rb, (uint64_t)cv.rows, rb, 256, kTok, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_u8(&msc, cv.kv, rb, (uint64_t)cv.rows, rb, 16, kTok, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_u8(&mc64, cv.kv, rb, (uint64_t)cv.rows, rb, 64, kTok, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        // latent boxes from kv; the rotary box from pe, or from kv after the latent when packed
        const uint64_t kv_cols = cv.pe ? 512 : (uint64_t)kRowElems;
        if (!encode_latent_3d(&mc128, cv.kv, kv_cols, (uint64_t)cv.rows, (uint64_t)cv.kv_stride) ||
            !encode_2d(&mc64, cv.pe ? cv.pe : cv.kv, cv.pe ? 64 : (uint64_t)kRowElems, (uint64_t)cv.rows,
                       (uint64_t)(cv.pe ? cv.pe_stride : cv.kv_stride), 32, kTok, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
        msc = mc64;                                     // unused by the bf16 kernels
    }
    TcArgs a{(const __nv_bfloat16*)qp, row_off, cv.block_table ? seq_len : nullptr, cv.block_table,
             cv.block_size, cv.max_blocks, cv.pe ? 0 : 512, cum, wstart, (__nv_bfloat16*)o_lat,
             lse, part_o, part_l, dev_status, wait_limit_ns(), d.n_heads, batch};
    auto kernel = fp8 ? split_tc_kernel<false, true>
                      : cv.block_table ? split_tc_kernel<true, false> : split_tc_kernel<false, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    profile_before_split(s);
    e = launch_ex(kernel, dim3(2 * workers), dim3(kThreads), kSmemBytes, s, pdl, mc128, mc64, msc, a);
    profile_after_split(s);
    note_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mla
