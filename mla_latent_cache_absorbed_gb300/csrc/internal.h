// Internal declarations shared by the translation units of libmla_gb300.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

// Sets the thread-local message returned by mla_last_error().
void set_error(const char* fmt, ...);

// CUDA failures become MLA_ERR_CUDA with the runtime's message.
mla_status cuda_status(cudaError_t e, const char* what);

#define MLA_CUDA_TRY(expr, what)                                  \
    do {                                                          \
        cudaError_t _e = (expr);                                  \
        if (_e != cudaSuccess) return ::mla::cuda_status(_e, what); \
    } while (0)

// Split-KV plan of the SIMT decode: one CTA per (query row, split).
struct SimtDecodePlan {
    int32_t nsplit;   // splits per query row
    int32_t chunk;    // keys per split (multiple of the block size)
    int64_t rows;     // batch * t_q * n_head query rows
    size_t bytes;     // workspace bytes
};
SimtDecodePlan simt_decode_plan(int32_t batch, int32_t max_blocks, const mla_dims& d);

// Launchers (SIMT kernels; any geometry within the documented limits).
cudaError_t launch_cache_append(void* cache, const void* kv_c, const void* k_pe,
                                const int64_t* slots, int32_t n_tokens, int32_t num_blocks,
                                int32_t src_dtype, const mla_dims& d, int32_t* dev_err,
                                cudaStream_t s);
cudaError_t launch_cache_append_rmsnorm_rope(void* cache, const void* kv_c, const void* k_pe,
                                             const void* gamma, const int64_t* positions,
                                             const int64_t* slots, int32_t n_tokens,
                                             int32_t num_blocks, int32_t src_dtype, float eps,
                                             float theta_scale, const mla_dims& d,
                                             int32_t* dev_err, cudaStream_t s);
// positions: null copies q_pe into the rope tail; otherwise the tail is the
// NEOX rope of q_pe at positions[r] (theta_j = pos * theta_scale^j)
cudaError_t launch_absorb_simt(void* q_abs, const void* q_nope, const void* q_pe,
                               const void* w_uk, int32_t rows, const mla_dims& d,
                               cudaStream_t s, const int64_t* positions = nullptr,
                               float theta_scale = 1.f);
// The query half of the prolog (tc_prolog.cu): the tensor-core kernel when
// tc_prolog_supported, else the SIMT form.
bool tc_prolog_supported(const mla_dims& d, int32_t q_rank);
cudaError_t launch_prolog_q(void* q_abs, const void* c_q, const void* gamma_q, const void* w_uq,
                            const void* w_qr, const void* w_uk, const int64_t* positions,
                            int32_t rows, int32_t q_rank, float eps, float theta_scale,
                            const mla_dims& d, int32_t* dev_err, cudaStream_t s);
cudaError_t launch_decompress_simt(void* out, const void* o_lat, const void* w_uv,
                                   int32_t rows, const mla_dims& d, cudaStream_t s);
cudaError_t launch_decode_simt(void* out, float* lse, const void* q_abs,
                               const void* kv_cache, const int32_t* block_table,
                               const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                               int32_t num_blocks, const mla_dims& d, float scale,
                               void* workspace, int32_t* dev_err, cudaStream_t s);

}  // namespace mla
