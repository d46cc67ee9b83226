// Host-to-device staging by a kernel that reads page-locked host memory directly.
//
// A serving loop moves every step's new tokens (and queries) from host memory into the
// device buffers the decode reads.  A copy-engine transfer (cudaMemcpyAsync) of a few MB
// pays a large fixed cost per call on some hosts; a kernel that loads the mapped host
// buffer over the bus with many 16-byte loads in flight streams it at close to the link
// rate instead.  This is transport plumbing of the library, not a step of the method.
#include <algorithm>

#include "mla_common.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;               // 16-byte loads in flight per thread
constexpr int kCopyMaxBlocks = 64;

// dst[i] = src[i] for 16-byte words: each thread keeps kCopyUnroll loads in flight
// (the loads cross the host link, so latency, not the device, sets the pace).
__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(const uint4* __restrict__ src,
                                                              uint4* __restrict__ dst, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads * kCopyUnroll;
    for (int64_t base = (int64_t)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x; base < n;
         base += stride) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + (int64_t)u * kCopyThreads;
            if (i < n) v[u] = src[i];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = base + (int64_t)u * kCopyThreads;
            if (i < n) dst[i] = v[u];
        }
    }
}

// Byte copy for buffers whose addresses or size are not 16-byte multiples.
__global__ void __launch_bounds__(kCopyThreads) copy8_kernel(const uint8_t* __restrict__ src,
                                                             uint8_t* __restrict__ dst, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * kCopyThreads)
        dst[i] = src[i];
}

}  // namespace
}  // namespace mla

extern "C" {

mla_status mla_copy_from_host(void* dst, const void* src, size_t bytes, void* stream) {
    if (bytes == 0) return MLA_OK;
    if (!dst || !src) return MLA_ERR_INVALID_ARG;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, src) != cudaSuccess) {
        (void)cudaGetLastError();
        return MLA_ERR_INVALID_ARG;
    }
    // page-locked host memory the device can address (mapped; with unified addressing
    // every page-locked allocation is)
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return MLA_ERR_INVALID_ARG;
    cudaPointerAttributes ad{};
    if (cudaPointerGetAttributes(&ad, dst) != cudaSuccess) {
        (void)cudaGetLastError();
        return MLA_ERR_INVALID_ARG;
    }
    if (ad.type != cudaMemoryTypeDevice && ad.type != cudaMemoryTypeManaged) return MLA_ERR_INVALID_ARG;
    const void* s_dev = at.devicePointer;
    cudaStream_t s = (cudaStream_t)stream;
    const bool vec = (((uintptr_t)s_dev | (uintptr_t)dst | bytes) & 15u) == 0;
    if (vec) {
        const int64_t n = (int64_t)(bytes / 16);
        const int64_t per_block = (int64_t)mla::kCopyThreads * mla::kCopyUnroll;
        const int blocks = (int)std::min<int64_t>(mla::kCopyMaxBlocks, (n + per_block - 1) / per_block);
        mla::copy16_kernel<<<blocks, mla::kCopyThreads, 0, s>>>((const uint4*)s_dev, (uint4*)dst, n);
    } else {
        const int64_t n = (int64_t)bytes;
        const int blocks = (int)std::min<int64_t>(mla::kCopyMaxBlocks, (n + mla::kCopyThreads - 1) / mla::kCopyThreads);
        mla::copy8_kernel<<<blocks, mla::kCopyThreads, 0, s>>>((const uint8_t*)s_dev, (uint8_t*)dst, n);
    }
    mla::note_launch();
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
