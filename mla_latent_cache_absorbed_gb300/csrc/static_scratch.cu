// mla_decode_paged_static: the paged decode with its split scratch in a
// library-owned, statically sized device array instead of a caller buffer.
//
// Some callers cannot allocate device memory at the time they decode: code
// running inside a captured or replayed CUDA graph, custom allocators that
// forbid cudaMalloc on the serving path, plugin hosts that hand out only the
// input and output buffers, or embedded runtimes with a fixed memory budget.
// For them this entry point uses a file-scope __device__ array that the CUDA
// module reserves once per GPU when the library's kernels are loaded there;
// it is held until the process exits. The caller still passes inputs and
// outputs; nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is shared by every call on a device and keeps the last call's
// contents. The decode writes every scratch slot it later reads, so nothing
// needs clearing between calls. Calls whose work overlaps on the GPU (two
// streams, or two host threads without ordering) race on the array: order
// them, e.g. by issuing them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[MLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device. The first call
// on a device resolves it (cudaGetSymbolAddress also loads the module there
// if it is not loaded yet); later calls reuse the cached address. The address
// belongs to the device's context: after a cudaDeviceReset the module loads
// again in a new context, possibly elsewhere, so the entry point is not for
// use on a device that has been reset (its header says so).
mla_status scratch_address(void** out) {
    int dev = -1;
    MLA_CUDA_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        mla::set_error("device ordinal %d is beyond the %d this entry point tracks", dev,
                       kMaxDevices);
        return MLA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        MLA_CUDA_TRY(cudaGetSymbolAddress(&p, g_decode_scratch),
                     "cudaGetSymbolAddress(static decode scratch)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_paged_static(void* out, float* lse, const void* q_abs,
                                              const void* kv_cache,
                                              const int32_t* block_table,
                                              const int32_t* seq_lens, int32_t batch,
                                              int32_t max_blocks, int32_t num_blocks,
                                              const mla_dims* dims, float scale,
                                              int32_t* dev_err, void* stream) {
    size_t need = 0;
    if (mla_status st = mla_decode_workspace_size(batch, max_blocks, dims, &need)) return st;
    if (need > (size_t)MLA_STATIC_SCRATCH_BYTES) {
        mla::set_error("mla_decode_paged_static: this batch needs %zu bytes of decode scratch "
                       "but the static scratch holds %zu; decode it in smaller batches or "
                       "call mla_decode_paged with a caller-provided workspace",
                       need, (size_t)MLA_STATIC_SCRATCH_BYTES);
        return MLA_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    if (batch > 0) {
        if (mla_status st = scratch_address(&scratch)) return st;
    }
    return mla_decode_paged(out, lse, q_abs, kv_cache, block_table, seq_lens, batch,
                            max_blocks, num_blocks, dims, scale, scratch,
                            (size_t)MLA_STATIC_SCRATCH_BYTES, dev_err, stream);
}
