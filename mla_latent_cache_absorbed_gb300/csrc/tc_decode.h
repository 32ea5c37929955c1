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
// early: the previous kernel on the stream writes none of kv_cache,
// block_table, seq_lens (only q_abs), so they may be read before it
// completes. combine: merge split rows into out with the combine kernel (else
// the caller merges them from the workspace, see tc_decode_split_info).
cudaError_t launch_decode_tc(void* out, float* lse, const void* q_abs, const void* kv_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             int32_t batch, int32_t max_blocks, int32_t num_blocks,
                             const mla_dims& d, float scale, void* workspace,
                             int32_t* dev_err, cudaStream_t s, bool early, bool combine);

// The timeout-path test switch (mla_debug_decode_wait_test): the bounded
// waits' limit for later decode launches (0: the default, 2 s) and whether
// their score MMA warp first waits on a barrier nothing arrives on.
struct DecodeWaitTest {
    unsigned long long limit_ns;
    int stall;
};
DecodeWaitTest decode_wait_test();
void set_decode_wait_test(unsigned long long limit_ns, int stall);

// Where the decode keeps its split partial rows in `workspace`, and the split
// parameters tc_split.cuh needs (pairs of the grid, fewest units per pair).
struct DecodeSplitInfo {
    int NP, min_units;
    void* ws_o;     // bf16 partial rows [2 NP][128][512]
    float* ws_lse;  // [2 NP][128]
};
cudaError_t tc_decode_split_info(const mla_dims& d, void* workspace, DecodeSplitInfo* info);
// Workspace bytes per CTA pair of the decode's grid: two partial slots of
// 128 rows x 512 bf16 and their 128 f32 LSEs (tc_decode_workspace is the
// pairs times this).
constexpr size_t kTcDecodeBytesPerPair = 2 * (128 * 512 * 2 + 128 * 4);

// True when the bf16 tensor-core absorb (absorb = true) or decompress GEMM
// serves this geometry and row count.
bool tc_gemm_supported(const mla_dims& d, int32_t rows, bool absorb);
// early: the weights may be read before the previous kernel completes (it
// does not write them).
// positions: as for launch_absorb_simt (null: q_pe copied unchanged).
cudaError_t launch_absorb_tc(void* q_abs, const void* q_nope, const void* q_pe,
                             const void* w_uk, int32_t rows, const mla_dims& d,
                             cudaStream_t s, bool early, const int64_t* positions = nullptr,
                             float theta_scale = 1.f);
cudaError_t launch_decompress_tc(void* out, const void* o_lat, const void* w_uv, int32_t rows,
                                 const mla_dims& d, cudaStream_t s, bool early);

// The decompress of the fused path: merges the decode's split rows (the
// decode ran with combine = false on the same stream just before) while it
// streams the weights. lse: the merged rows' LSEs, or null.
bool tc_merge_supported(const mla_dims& d, int32_t rows, int np);
cudaError_t launch_decompress_merge_tc(void* out, float* lse, const void* o_lat,
                                       const void* w_uv, const int32_t* seq_lens,
                                       int32_t batch, int32_t max_blocks, const mla_dims& d,
                                       const DecodeSplitInfo& info, int32_t* dev_err,
                                       cudaStream_t s);

}  // namespace mla
