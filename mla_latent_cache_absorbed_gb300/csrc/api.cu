// C ABI of libmla_gb300 (declared in include/mla.h): argument validation,
// status codes, workspace sizing and dispatch to the kernels.
#include <math.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <vector>

#include "internal.h"
#include "tc_decode.h"

namespace mla {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
}

mla_status cuda_status(cudaError_t e, const char* what) {
    set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    return MLA_ERR_CUDA;
}

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

mla_status check_dims(const mla_dims* d) {
    if (!d) {
        set_error("dims is NULL");
        return MLA_ERR_INVALID_ARG;
    }
    if (d->n_head <= 0 || d->d_nope <= 0 || d->d_rope < 0 || d->d_v <= 0 ||
        d->kv_rank <= 0 || d->t_q <= 0) {
        set_error("dims: n_head, d_nope, d_v, kv_rank, t_q must be > 0 and d_rope >= 0 "
                  "(got %d %d %d %d %d %d)", d->n_head, d->d_nope, d->d_rope, d->d_v,
                  d->kv_rank, d->t_q);
        return MLA_ERR_INVALID_ARG;
    }
    if (d->block_size != 16) {
        set_error("dims: block_size must be 16 (got %d)", d->block_size);
        return MLA_ERR_INVALID_ARG;
    }
    if (d->dtype != MLA_F32 && d->dtype != MLA_BF16 && d->dtype != MLA_F16) {
        set_error("dims: dtype must be MLA_F32, MLA_BF16 or MLA_F16 (got %d)", d->dtype);
        return MLA_ERR_INVALID_ARG;
    }
    if (d->kv_rank > 1024 || d->kv_rank + d->d_rope > 1152 || d->d_nope > 1024 ||
        d->d_v > 4096) {
        set_error("dims: kv_rank <= 1024, kv_rank + d_rope <= 1152, d_nope <= 1024 and "
                  "d_v <= 4096 are supported");
        return MLA_ERR_UNSUPPORTED;
    }
    // every row of every operand must start on a 16-byte boundary
    const int esz = d->dtype == MLA_F32 ? 4 : 2;
    const int per16 = 16 / esz;
    if (d->kv_rank % per16 || d->d_rope % per16 || d->d_nope % per16 || d->d_v % per16) {
        set_error("dims: kv_rank, d_rope, d_nope and d_v must be multiples of %d for this "
                  "dtype (16-byte rows)", per16);
        return MLA_ERR_INVALID_ARG;
    }
    return MLA_OK;
}

#define REQUIRE(cond, ...)               \
    do {                                 \
        if (!(cond)) {                   \
            set_error(__VA_ARGS__);      \
            return MLA_ERR_INVALID_ARG;  \
        }                                \
    } while (0)

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_str(mla_status s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: unsupported geometry";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA runtime error";
        case MLA_ERR_DEVICE_BOUNDS: return "MLA_ERR_DEVICE_BOUNDS: invalid device data";
        case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a device wait gave up";
    }
    return "unknown mla_status";
}

const char* mla_last_error(void) { return g_last_error; }

mla_status mla_debug_decode_wait_test(uint64_t limit_ns, int32_t stall) {
    mla::set_decode_wait_test(limit_ns, stall);
    return MLA_OK;
}

mla_status mla_absorb_q(void* q_abs, const void* q_nope, const void* q_pe, const void* w_uk,
                        int32_t rows, const mla_dims* dims, void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(rows >= 0, "rows must be >= 0 (got %d)", rows);
    if (rows == 0) return MLA_OK;
    REQUIRE(q_abs && q_nope && w_uk, "q_abs, q_nope and w_uk must be non-NULL");
    REQUIRE(q_pe || dims->d_rope == 0, "q_pe may be NULL only when d_rope == 0");
    REQUIRE(aligned16(q_abs) && aligned16(q_nope) && aligned16(w_uk) &&
                (!q_pe || aligned16(q_pe)),
            "device buffers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (dims->dtype != MLA_F32 && tc_gemm_supported(*dims, rows, /*absorb=*/true)) {
        MLA_CUDA_TRY(launch_absorb_tc(q_abs, q_nope, q_pe, w_uk, rows, *dims, s, /*early=*/false),
                     "absorb (tensor cores)");
        return MLA_OK;
    }
    MLA_CUDA_TRY(launch_absorb_simt(q_abs, q_nope, q_pe, w_uk, rows, *dims, s), "absorb");
    return MLA_OK;
}

mla_status mla_absorb_q_rope(void* q_abs, const void* q_nope, const void* q_pe,
                             const void* w_uk, const int64_t* positions, int32_t rows,
                             float rope_base, const mla_dims* dims, void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(rows >= 0, "rows must be >= 0 (got %d)", rows);
    const int P = dims->d_rope;
    REQUIRE(P == 0 || (std::isfinite(rope_base) && rope_base > 0.f),
            "rope_base must be finite and > 0");
    if (rows == 0) return MLA_OK;
    REQUIRE(q_abs && q_nope && w_uk, "q_abs, q_nope and w_uk must be non-NULL");
    REQUIRE(P == 0 || (q_pe && positions), "q_pe and positions may be NULL only when d_rope == 0");
    REQUIRE(aligned16(q_abs) && aligned16(q_nope) && aligned16(w_uk) &&
                (!q_pe || aligned16(q_pe)) && ((uintptr_t)positions & 7u) == 0,
            "device buffers must be 16-byte aligned, positions 8-byte aligned");
    if (P == 0) return mla_absorb_q(q_abs, q_nope, q_pe, w_uk, rows, dims, stream);
    // the rope's per-pair frequency ratio, once, in f32 as the rope is computed
    // (the same ratio the fused cache append uses for the keys)
    const float theta_scale = powf(rope_base, -2.0f / (float)P);
    cudaStream_t s = (cudaStream_t)stream;
    if (dims->dtype != MLA_F32 && tc_gemm_supported(*dims, rows, /*absorb=*/true)) {
        MLA_CUDA_TRY(launch_absorb_tc(q_abs, q_nope, q_pe, w_uk, rows, *dims, s, /*early=*/false,
                                      positions, theta_scale),
                     "absorb with rope (tensor cores)");
        return MLA_OK;
    }
    MLA_CUDA_TRY(launch_absorb_simt(q_abs, q_nope, q_pe, w_uk, rows, *dims, s, positions,
                                    theta_scale),
                 "absorb with rope");
    return MLA_OK;
}

mla_status mla_prolog_q(void* q_abs, const void* c_q, const void* gamma_q, const void* w_uq,
                        const void* w_qr, const void* w_uk, const int64_t* positions,
                        int32_t rows, int32_t q_rank, float eps, float rope_base,
                        const mla_dims* dims, int32_t* dev_err, void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(rows >= 0, "rows must be >= 0 (got %d)", rows);
    REQUIRE(q_rank > 0 && q_rank % 8 == 0 && q_rank <= 16384,
            "q_rank must be a positive multiple of 8, at most 16384 (got %d)", q_rank);
    const int P = dims->d_rope;
    REQUIRE(std::isfinite(eps) && eps >= 0.f, "eps must be finite and >= 0");
    REQUIRE(P == 0 || (std::isfinite(rope_base) && rope_base > 0.f),
            "rope_base must be finite and > 0");
    REQUIRE((P & 1) == 0, "d_rope must be even");
    if (rows == 0) return MLA_OK;
    REQUIRE(q_abs && c_q && gamma_q && w_uq && w_uk, "q_abs, c_q, gamma_q, w_uq and w_uk must be non-NULL");
    REQUIRE(P == 0 || (w_qr && positions), "w_qr and positions may be NULL only when d_rope == 0");
    REQUIRE(aligned16(q_abs) && aligned16(c_q) && aligned16(gamma_q) && aligned16(w_uq) &&
                aligned16(w_uk) && (!w_qr || aligned16(w_qr)) && ((uintptr_t)positions & 7u) == 0,
            "device buffers must be 16-byte aligned, positions 8-byte aligned");
    const float theta_scale = P > 0 ? powf(rope_base, -2.0f / (float)P) : 1.f;
    MLA_CUDA_TRY(launch_prolog_q(q_abs, c_q, gamma_q, w_uq, w_qr, w_uk, positions, rows, q_rank,
                                 eps, theta_scale, *dims, dev_err, (cudaStream_t)stream),
                 "query prolog");
    return MLA_OK;
}

mla_status mla_cache_append(void* kv_cache, const void* kv_c, const void* k_pe,
                            const int64_t* slot_mapping, int32_t n_tokens, int32_t num_blocks,
                            int32_t src_dtype, const mla_dims* dims, int32_t* dev_err,
                            void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(n_tokens >= 0 && num_blocks >= 0, "n_tokens and num_blocks must be >= 0");
    REQUIRE(src_dtype == MLA_F32 || src_dtype == MLA_BF16, "src_dtype must be MLA_F32 or MLA_BF16");
    if (dims->dtype == MLA_F16) {
        set_error("cache append: f16 caches are not supported (f32 or bf16)");
        return MLA_ERR_UNSUPPORTED;
    }
    if (n_tokens == 0) return MLA_OK;
    REQUIRE(kv_cache && kv_c && slot_mapping, "kv_cache, kv_c and slot_mapping must be non-NULL");
    REQUIRE(dims->d_rope == 0 || k_pe, "k_pe may be NULL only when d_rope == 0");
    REQUIRE(aligned16(kv_cache) && aligned16(kv_c) && (!k_pe || aligned16(k_pe)) &&
                ((uintptr_t)slot_mapping & 7u) == 0,
            "kv_cache, kv_c and k_pe must be 16-byte aligned, slot_mapping 8-byte aligned");
    // one 16-byte piece of a cache row never straddles kv_c and k_pe
    const int piece = dims->dtype == MLA_BF16 ? 8 : 4;
    if (dims->kv_rank % piece || dims->d_rope % piece) {
        set_error("cache append: kv_rank and d_rope must be multiples of %d", piece);
        return MLA_ERR_UNSUPPORTED;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MLA_CUDA_TRY(launch_cache_append(kv_cache, kv_c, k_pe, slot_mapping, n_tokens, num_blocks,
                                     src_dtype, *dims, dev_err, s),
                 "cache append");
    return MLA_OK;
}

mla_status mla_cache_append_rmsnorm_rope(void* kv_cache, const void* kv_c, const void* k_pe,
                                         const void* gamma, const int64_t* positions,
                                         const int64_t* slot_mapping, int32_t n_tokens,
                                         int32_t num_blocks, int32_t src_dtype, float eps,
                                         float rope_base, const mla_dims* dims, int32_t* dev_err,
                                         void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(n_tokens >= 0 && num_blocks >= 0, "n_tokens and num_blocks must be >= 0");
    REQUIRE(src_dtype == MLA_F32 || src_dtype == MLA_BF16, "src_dtype must be MLA_F32 or MLA_BF16");
    if (dims->dtype == MLA_F16) {
        set_error("cache append: f16 caches are not supported (f32 or bf16)");
        return MLA_ERR_UNSUPPORTED;
    }
    REQUIRE(std::isfinite(eps) && eps >= 0.f, "eps must be finite and >= 0");
    const int P = dims->d_rope;
    REQUIRE(P == 0 || (std::isfinite(rope_base) && rope_base > 0.f),
            "rope_base must be finite and > 0");
    if (n_tokens == 0) return MLA_OK;
    REQUIRE(kv_cache && kv_c && gamma && slot_mapping,
            "kv_cache, kv_c, gamma and slot_mapping must be non-NULL");
    REQUIRE(P == 0 || (k_pe && positions), "k_pe and positions may be NULL only when d_rope == 0");
    REQUIRE(aligned16(kv_cache) && aligned16(kv_c) && aligned16(gamma) &&
                ((uintptr_t)slot_mapping & 7u) == 0 && ((uintptr_t)positions & 7u) == 0 &&
                ((uintptr_t)k_pe & (src_dtype == MLA_BF16 ? 1u : 3u)) == 0,
            "kv_cache, kv_c and gamma must be 16-byte aligned, slot_mapping and positions "
            "8-byte aligned, k_pe element aligned");
    const int piece = dims->dtype == MLA_BF16 ? 8 : 4;
    if (dims->kv_rank % piece || P % piece) {
        set_error("cache append: kv_rank and d_rope must be multiples of %d", piece);
        return MLA_ERR_UNSUPPORTED;
    }
    // the rope's per-pair frequency ratio, once, in f32 as the rope is computed
    const float theta_scale = P > 0 ? powf(rope_base, -2.0f / (float)P) : 1.f;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MLA_CUDA_TRY(launch_cache_append_rmsnorm_rope(kv_cache, kv_c, k_pe, gamma, positions,
                                                  slot_mapping, n_tokens, num_blocks, src_dtype,
                                                  eps, theta_scale, *dims, dev_err, s),
                 "cache append (rmsnorm, rope)");
    return MLA_OK;
}

mla_status mla_decompress_out(void* out, const void* o_lat, const void* w_uv, int32_t rows,
                              const mla_dims* dims, void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(rows >= 0, "rows must be >= 0 (got %d)", rows);
    if (rows == 0) return MLA_OK;
    REQUIRE(out && o_lat && w_uv, "out, o_lat and w_uv must be non-NULL");
    REQUIRE(aligned16(out) && aligned16(o_lat) && aligned16(w_uv),
            "device buffers must be 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    if (dims->dtype != MLA_F32 && tc_gemm_supported(*dims, rows, /*absorb=*/false)) {
        MLA_CUDA_TRY(launch_decompress_tc(out, o_lat, w_uv, rows, *dims, s, /*early=*/false),
                     "decompress (tensor cores)");
        return MLA_OK;
    }
    MLA_CUDA_TRY(launch_decompress_simt(out, o_lat, w_uv, rows, *dims, s), "decompress");
    return MLA_OK;
}

namespace {
// Index limits of the decode kernels: query rows (batch * t_q * n_head),
// cache positions (max_blocks * 16) and the work split's units (64-token
// tiles, at most ceil(max_blocks / 4) a request, summed over the batch) are
// 32-bit counts.
mla_status check_decode_shape(int32_t batch, int32_t max_blocks, const mla_dims& d) {
    if ((long long)batch * d.t_q * d.n_head > INT32_MAX || max_blocks >= (1 << 27)) {
        set_error("decode: batch * t_q * n_head = %lld query rows (at most 2^31 - 1) and "
                  "max_blocks = %d (below 2^27) are supported",
                  (long long)batch * d.t_q * d.n_head, max_blocks);
        return MLA_ERR_UNSUPPORTED;
    }
    const long long tiles = (long long)batch * ((max_blocks + 3) / 4);
    if (tiles > INT32_MAX) {
        set_error("decode: batch * ceil(max_blocks / 4) = %lld cache tiles of 64 tokens "
                  "(at most 2^31 - 1) are supported", tiles);
        return MLA_ERR_UNSUPPORTED;
    }
    return MLA_OK;
}

// The 16-bit types take the tensor-core decode. It gives each row group of a
// request (128 of its t_q * n_head query rows) a set of CTA pairs of its own;
// when the row groups do not divide the grid's pairs, or outnumber them (a
// long prefill chunk), all row groups' tiles are pooled and shared out
// evenly, a pair walking on from one row group into the next.
bool use_tc_decode(const mla_dims& d) {
    if (d.dtype == MLA_F32 || !tc_decode_supported(d)) return false;
    size_t bytes = 0;
    return tc_decode_workspace(1, 1, d, &bytes) == cudaSuccess;
}
}  // namespace

mla_status mla_decode_workspace_size(int32_t batch, int32_t max_blocks, const mla_dims* dims,
                                     size_t* bytes) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(bytes, "bytes must be non-NULL");
    REQUIRE(batch >= 0 && max_blocks >= 1, "batch >= 0 and max_blocks >= 1 required");
    if (mla_status st = check_decode_shape(batch, max_blocks, *dims)) return st;
    if (use_tc_decode(*dims)) {
        size_t b = 0;
        MLA_CUDA_TRY(tc_decode_workspace(batch, max_blocks, *dims, &b), "decode workspace");
        *bytes = b;
        return MLA_OK;
    }
    *bytes = simt_decode_plan(batch, max_blocks, *dims).bytes;
    return MLA_OK;
}

mla_status mla_decode_paged(void* out, float* lse, const void* q_abs, const void* kv_cache,
                            const int32_t* block_table, const int32_t* seq_lens,
                            int32_t batch, int32_t max_blocks, int32_t num_blocks,
                            const mla_dims* dims, float scale, void* workspace,
                            size_t workspace_bytes, int32_t* dev_err, void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(batch >= 0 && max_blocks >= 1 && num_blocks >= 1,
            "batch >= 0, max_blocks >= 1 and num_blocks >= 1 required");
    if (batch == 0) return MLA_OK;
    REQUIRE(out && q_abs && kv_cache && block_table && seq_lens && workspace,
            "out, q_abs, kv_cache, block_table, seq_lens and workspace must be non-NULL");
    REQUIRE(aligned16(out) && aligned16(q_abs) && aligned16(kv_cache) &&
                aligned16(block_table) && aligned16(seq_lens) && (!lse || aligned16(lse)),
            "device buffers must be 16-byte aligned");
    REQUIRE(((uintptr_t)workspace & 255u) == 0, "workspace must be 256-byte aligned");
    REQUIRE(scale == scale, "scale is NaN");
    size_t need = 0;
    if (mla_status st = mla_decode_workspace_size(batch, max_blocks, dims, &need)) return st;
    REQUIRE(workspace_bytes >= need, "workspace too small: %zu bytes given, %zu needed",
            workspace_bytes, need);
    cudaStream_t s = (cudaStream_t)stream;
    if (use_tc_decode(*dims)) {
        MLA_CUDA_TRY(launch_decode_tc(out, lse, q_abs, kv_cache, block_table, seq_lens, batch,
                                      max_blocks, num_blocks, *dims, scale, workspace, dev_err,
                                      s, /*early=*/false, /*combine=*/true),
                     "decode (tensor cores)");
        return MLA_OK;
    }
    MLA_CUDA_TRY(launch_decode_simt(out, lse, q_abs, kv_cache, block_table, seq_lens, batch,
                                    max_blocks, num_blocks, *dims, scale, workspace, dev_err,
                                    s),
                 "decode");
    return MLA_OK;
}

namespace {
size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }
}  // namespace

mla_status mla_attend_workspace_size(int32_t batch, int32_t max_blocks, const mla_dims* dims,
                                     size_t* bytes) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(bytes, "bytes must be non-NULL");
    REQUIRE(batch >= 0 && max_blocks >= 1, "batch >= 0 and max_blocks >= 1 required");
    size_t dws = 0;
    if (mla_status st = mla_decode_workspace_size(batch, max_blocks, dims, &dws)) return st;
    const size_t esz = dims->dtype == MLA_F32 ? 4 : 2;
    const size_t qrows = (size_t)batch * dims->t_q * dims->n_head;
    *bytes = round256(qrows * (dims->kv_rank + dims->d_rope) * esz) +
             round256(qrows * dims->kv_rank * esz) + dws;
    return MLA_OK;
}

mla_status mla_attend_absorbed(void* out, float* lse, const void* q_nope, const void* q_pe,
                               const void* w_uk, const void* w_uv, const void* kv_cache,
                               const int32_t* block_table, const int32_t* seq_lens,
                               int32_t batch, int32_t max_blocks, int32_t num_blocks,
                               const mla_dims* dims, float scale, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err, void* stream) {
    g_last_error[0] = 0;
    if (mla_status st = check_dims(dims)) return st;
    REQUIRE(batch >= 0 && max_blocks >= 1 && num_blocks >= 1,
            "batch >= 0, max_blocks >= 1 and num_blocks >= 1 required");
    if (batch == 0) return MLA_OK;
    REQUIRE(out && q_nope && w_uk && w_uv && kv_cache && block_table && seq_lens && workspace,
            "out, q_nope, w_uk, w_uv, kv_cache, block_table, seq_lens and workspace must be "
            "non-NULL");
    REQUIRE(q_pe || dims->d_rope == 0, "q_pe may be NULL only when d_rope == 0");
    REQUIRE(aligned16(out) && aligned16(q_nope) && (!q_pe || aligned16(q_pe)) &&
                aligned16(w_uk) && aligned16(w_uv) && aligned16(kv_cache) &&
                aligned16(block_table) && aligned16(seq_lens) && (!lse || aligned16(lse)),
            "device buffers must be 16-byte aligned");
    REQUIRE(((uintptr_t)workspace & 255u) == 0, "workspace must be 256-byte aligned");
    REQUIRE(scale == scale, "scale is NaN");
    size_t need = 0;
    if (mla_status st = mla_attend_workspace_size(batch, max_blocks, dims, &need)) return st;
    REQUIRE(workspace_bytes >= need, "workspace too small: %zu bytes given, %zu needed",
            workspace_bytes, need);
    const size_t esz = dims->dtype == MLA_F32 ? 4 : 2;
    const size_t qrows = (size_t)batch * dims->t_q * dims->n_head;
    const int32_t rows = batch * dims->t_q;
    char* ws = static_cast<char*>(workspace);
    void* q_abs = ws;
    void* o_lat = ws + round256(qrows * (dims->kv_rank + dims->d_rope) * esz);
    void* dws = static_cast<char*>(o_lat) + round256(qrows * dims->kv_rank * esz);
    const size_t dws_bytes = workspace_bytes - (size_t)(static_cast<char*>(dws) - ws);
    cudaStream_t s = (cudaStream_t)stream;
    DecodeSplitInfo info = {};
    // The merging decompress finds each of its rows' split parts through the
    // row group the row belongs to; the 128 rows of one of its CTAs (128
    // query positions of one head) fall in up to 128 row groups of the
    // decode, and with many row groups per request those lookups outweigh
    // the combine they replace (a 128-query chunk of 64 heads: 619 us fused
    // against 374 us for the three stages). Up to two row groups of queries
    // per request take the fused chain, larger query blocks the three calls.
    const bool few_row_groups = (long long)dims->t_q * dims->n_head <= 256;
    if (few_row_groups && use_tc_decode(*dims) &&
        tc_gemm_supported(*dims, rows, /*absorb=*/true) &&
        tc_decode_split_info(*dims, dws, &info) == cudaSuccess &&
        tc_merge_supported(*dims, rows, info.NP)) {
        // the library's own chain: the absorb waits for the caller's previous
        // kernel before reading anything; the decode may read the cache before
        // the absorb completes (the absorb writes only q_abs); the decompress
        // merges the decode's split rows and streams its weights meanwhile
        MLA_CUDA_TRY(launch_absorb_tc(q_abs, q_nope, q_pe, w_uk, rows, *dims, s, /*early=*/false),
                     "attend: absorb (tensor cores)");
        MLA_CUDA_TRY(launch_decode_tc(o_lat, lse, q_abs, kv_cache, block_table, seq_lens, batch,
                                      max_blocks, num_blocks, *dims, scale, dws, dev_err, s,
                                      /*early=*/true, /*combine=*/false),
                     "attend: decode (tensor cores)");
        MLA_CUDA_TRY(launch_decompress_merge_tc(out, lse, o_lat, w_uv, seq_lens, batch, max_blocks,
                                                *dims, info, dev_err, s),
                     "attend: merge + decompress (tensor cores)");
        return MLA_OK;
    }
    if (mla_status st = mla_absorb_q(q_abs, q_nope, q_pe, w_uk, rows, dims, stream)) return st;
    if (mla_status st = mla_decode_paged(o_lat, lse, q_abs, kv_cache, block_table, seq_lens,
                                         batch, max_blocks, num_blocks, dims, scale, dws,
                                         dws_bytes, dev_err, stream))
        return st;
    return mla_decompress_out(out, o_lat, w_uv, rows, dims, stream);
}

mla_status mla_rope_norm_to_neox_perm(int32_t n_dims, int32_t* perm_out) {
    g_last_error[0] = 0;
    REQUIRE(n_dims >= 0 && n_dims % 2 == 0, "n_dims must be even and >= 0 (got %d)", n_dims);
    REQUIRE(perm_out || n_dims == 0, "perm_out must be non-NULL");
    const int32_t half = n_dims / 2;
    for (int32_t j = 0; j < half; ++j) {
        perm_out[2 * j] = j;
        perm_out[2 * j + 1] = j + half;
    }
    return MLA_OK;
}

mla_status mla_permute_rope_cols(void* x, int32_t elem_bytes, int64_t rows, int64_t row_stride,
                                 int32_t col0, int32_t n_dims) {
    g_last_error[0] = 0;
    REQUIRE(elem_bytes == 2 || elem_bytes == 4, "elem_bytes must be 2 or 4");
    REQUIRE(rows >= 0 && col0 >= 0 && n_dims >= 0 && n_dims % 2 == 0,
            "rows >= 0, col0 >= 0 and an even n_dims >= 0 required");
    REQUIRE(row_stride >= (int64_t)col0 + n_dims, "row_stride must cover col0 + n_dims");
    if (rows == 0 || n_dims == 0) return MLA_OK;
    REQUIRE(x, "x must be non-NULL");
    std::vector<int32_t> perm(n_dims);
    mla_rope_norm_to_neox_perm(n_dims, perm.data());
    std::vector<unsigned char> tmp((size_t)n_dims * elem_bytes);
    unsigned char* base = (unsigned char*)x;
    for (int64_t r = 0; r < rows; ++r) {
        unsigned char* span = base + (r * row_stride + col0) * elem_bytes;
        for (int32_t i = 0; i < n_dims; ++i)
            memcpy(&tmp[(size_t)perm[i] * elem_bytes], span + (size_t)i * elem_bytes, elem_bytes);
        memcpy(span, tmp.data(), tmp.size());
    }
    return MLA_OK;
}

mla_status mla_permute_rope_rows(void* w, int32_t elem_bytes, int64_t row_len, int32_t row0,
                                 int32_t n_dims) {
    g_last_error[0] = 0;
    REQUIRE(elem_bytes == 2 || elem_bytes == 4, "elem_bytes must be 2 or 4");
    REQUIRE(row_len >= 0 && row0 >= 0 && n_dims >= 0 && n_dims % 2 == 0,
            "row_len >= 0, row0 >= 0 and an even n_dims >= 0 required");
    if (row_len == 0 || n_dims == 0) return MLA_OK;
    REQUIRE(w, "w must be non-NULL");
    std::vector<int32_t> perm(n_dims);
    mla_rope_norm_to_neox_perm(n_dims, perm.data());
    const size_t rb = (size_t)row_len * elem_bytes;
    std::vector<unsigned char> tmp(rb * n_dims);
    unsigned char* base = (unsigned char*)w + (size_t)row0 * rb;
    for (int32_t i = 0; i < n_dims; ++i) memcpy(&tmp[(size_t)perm[i] * rb], base + i * rb, rb);
    memcpy(base, tmp.data(), tmp.size());
    return MLA_OK;
}

}  // extern "C"
