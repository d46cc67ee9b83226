// Allocation-free form of the absorbed decode.
//
// Some callers cannot call cudaMalloc at all: code that runs where the allocator is
// unavailable or forbidden (for instance inside a custom allocator's own callbacks,
// in plugin hosts that own all device memory, or in hot paths whose rules forbid any
// allocation).  For them the library carries its decode scratch as a file-scope
// __device__ array of fixed size, which every GPU that loads this library holds
// until the process exits.
//
// In host code `g_decode_scratch` names a host-side stand-in, not device memory, so
// it is never passed to a kernel directly: every call looks the device address up with
// cudaGetSymbolAddress on the current device (no cached address can outlive a reset of
// the device's context).

#include "mla_common.cuh"
#include "mla_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;     // 32 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device.
mla_status scratch_of_current_device(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    *out = p;
    return MLA_OK;
}

}  // namespace

extern "C" {

mla_status mla_decode_absorbed_noalloc(const mla_dims* dims, mla_dtype dtype, int32_t batch,
                                       const void* q_c, const void* q_r, const void* w_uk,
                                       const void* cache, int64_t cache_rows, const int64_t* row_off,
                                       const int32_t* seq_len, int32_t max_seq_len, int32_t num_splits,
                                       void* o_lat, float* lse, int32_t* dev_status, void* stream) {
    // Size check first: a problem whose scratch does not fit is refused before any
    // CUDA call.  A zero size means the arguments are bad; the regular entry point
    // below then returns the precise error.
    const size_t need = mla_decode_workspace_size(dims, dtype, batch, max_seq_len, num_splits);
    if (need > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
    void* scratch = nullptr;
    const mla_status st = scratch_of_current_device(&scratch);
    if (st != MLA_OK) return st;
    // The decode writes every scratch byte it later reads within the same call (folded
    // queries, prefix sums, schedule, split partials), so nothing has to be cleared.
    return mla_decode_absorbed(dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len,
                               max_seq_len, num_splits, scratch, kStaticScratchBytes, o_lat, lse,
                               dev_status, stream);
}

}  // extern "C"
