// Tensor-core (tcgen05 / TMEM / TMA) kernels of the bf16 path.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

// True when the bf16 tensor-core decode serves this geometry.
bool tc_decode_supported(const mla_dims& d);
cudaError_t tc_decode_workspace(int32_t batch, int32_t max_blocks, const mla_dims& d,
                                size_t* bytes);
cudaError_t launch_decode_tc(void* out, float* lse, const void* q_abs, const void* kv_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             int32_t batch, int32_t max_blocks, int32_t num_blocks,
                             const mla_dims& d, float scale, void* workspace,
                             int32_t* dev_err, cudaStream_t s);

// True when the bf16 tensor-core absorb (absorb = true) or decompress GEMM
// serves this geometry and row count.
bool tc_gemm_supported(const mla_dims& d, int32_t rows, bool absorb);
cudaError_t launch_absorb_tc(void* q_abs, const void* q_nope, const void* q_pe,
                             const void* w_uk, int32_t rows, const mla_dims& d,
                             cudaStream_t s);
cudaError_t launch_decompress_tc(void* out, const void* o_lat, const void* w_uv, int32_t rows,
                                 const mla_dims& d, cudaStream_t s);

}  // namespace mla
