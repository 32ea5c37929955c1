/*
 * mla.h — C ABI of libmla_gb300: absorbed multi-head latent attention (MLA)
 * decode over a paged latent KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The path (each entry point cites the passage that defines its operation):
 *   mla_absorb_q        fold the query through W_UK into rank space
 *   mla_decode_paged    all heads attend MQA-style to the shared cache rows
 *                       [c_kv | k_pe], split over the keys, merged by LSE
 *   mla_decompress_out  decompress the latent output once through W_UV
 *   mla_attend_absorbed the three above as one call (absorb, decode, merge
 *                       and decompress), the form a decode step uses
 *   mla_cache_append    write new tokens' latent rows into the paged cache
 *   mla_cache_append_rmsnorm_rope  the same, with the RmsNorm of the latent
 *                       and the rope of k_pe computed on the way in
 *   mla_rope_norm_to_neox_perm / mla_permute_rope_cols / mla_permute_rope_rows
 *                       the host-side load-time rope permutation
 *
 * Conventions shared by every entry point:
 *   - Device buffers are caller-owned, dense, row-major and 16-byte aligned.
 *     The library allocates no device memory; decode scratch is passed in
 *     (sized by mla_decode_workspace_size).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Device work is enqueued asynchronously; no call synchronises.
 *   - Host-side validation failures return immediately and enqueue nothing;
 *     mla_last_error() then describes the failure (thread-local).
 *   - The GPU device current on the calling thread must be the one that owns
 *     the buffers.
 *   - Element types: MLA_F32, MLA_BF16 or MLA_F16 for q, cache, weights and
 *     outputs (one type per call, dims->dtype); f16 is one of the types the
 *     "vllm.v1.attention.backends.mla.cpu_mla" page lists for CPUMLABackend.
 *     The LSE is always f32. Accumulation is always f32. The cache appends
 *     write f32 or bf16 caches only.
 *   - Results are deterministic: the same inputs on the same device give the
 *     same bits (every reduction has a fixed order).
 *   - Kernels launch as programmatic dependents of the kernel before them on
 *     the stream: their set-up overlaps its end, but they read no input and
 *     write nothing before it has completed. (Inside mla_attend_absorbed the
 *     library's own later kernels read the inputs its earlier ones do not
 *     write, the cache and the weights, early.)
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mla_status {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or geometry */
    MLA_ERR_UNSUPPORTED = 2,   /* valid but not built (e.g. an unusual width) */
    MLA_ERR_CUDA = 3,          /* a CUDA runtime call failed (see mla_last_error) */
    MLA_ERR_DEVICE_BOUNDS = 4, /* reserved for callers mapping dev_err bits */
    MLA_ERR_TIMEOUT = 5        /* reserved for callers mapping dev_err bits */
} mla_status;

typedef enum mla_dtype { MLA_F32 = 0, MLA_BF16 = 1, MLA_F16 = 2 } mla_dtype;

/*
 * Head geometry ("memra_engine/mla.rs source", struct MlaDims) plus the decode
 * query count and cache block size.
 *   n_head      attention heads H
 *   d_nope      qk no-position head dim (Dn)
 *   d_rope      decoupled rope dim (P); 0 for the NoPE geometry
 *   d_v         per-head decompressed V width (Dv)
 *   kv_rank     latent rank R; a cache row is W = R + P wide
 *   t_q         queries per request (1 for plain decode); the queries are the
 *               last t_q positions of the request
 *   block_size  cache rows per block; must be 16 ("vllm.v1...cpu_mla",
 *               CPUMLABackend.get_supported_kernel_block_sizes)
 *   dtype       mla_dtype of q, cache, weights and outputs
 */
typedef struct mla_dims {
    int32_t n_head, d_nope, d_rope, d_v, kv_rank, t_q, block_size;
    int32_t dtype;
} mla_dims;

/* Bits OR-ed into the optional device error word by mla_decode_paged. The
 * affected query rows get a zero output row and LSE = -inf. */
#define MLA_DEVERR_BAD_BLOCK 1u     /* a block id outside [0, num_blocks) */
#define MLA_DEVERR_SEQ_TOO_LONG 2u  /* seq_len > max_blocks * block_size */
#define MLA_DEVERR_SEQ_SHORT 4u     /* 0 < seq_len < t_q, or seq_len < 0 */
#define MLA_DEVERR_TIMEOUT 8u       /* a bounded wait inside a kernel gave up */
#define MLA_DEVERR_BAD_SLOT 16u     /* mla_cache_append: a slot past the cache */

/*
 * Absorb ("memra_engine/mla.rs source", fn mla_attend_absorbed, absorb step;
 * "vllm.v1.attention.backends.mla.cpu_mla", CPUMLAImpl.forward_mqa, the
 * concatenation of the absorbed query with q_pe):
 *   q_abs[r][h][l]     = sum_p q_nope[r][h][p] * w_uk[h][p][l]   (l < R)
 *   q_abs[r][h][R + j] = q_pe[r][h][j]                           (j < P)
 * q_abs  [rows][H][R+P]   out, dims->dtype
 * q_nope [rows][H][Dn]    in
 * q_pe   [rows][H][P]     in; may be NULL only when P == 0
 * w_uk   [H][Dn][R]       in
 * rows = batch * t_q query rows. rows == 0 is a no-op.
 */
mla_status mla_absorb_q(void* q_abs, const void* q_nope, const void* q_pe,
                        const void* w_uk, int32_t rows, const mla_dims* dims,
                        void* stream);

/*
 * The absorb with the query's rope ("aclnnMlaProlog", computation formulas
 * of the query: q^N = q^C W^UK and q^R = ROPE(c^Q W^QR)), for callers that
 * hold the query's rope part before its rotation:
 *   q_abs[r][h] = [ sum_p q_nope[r][h][p] * w_uk[h][p][:]  |  rope(q_pe[r][h]) ]
 * where rope turns the NEOX pair (j, j + P/2) by theta_j = positions[r] *
 * base^(-2j/P), the ratio base^(-2/P) applied j times in f32 ("memra_engine/
 * mla.rs source", fn rope_neox; the rope columns of W^QR carry the load-time
 * permutation, so q_pe arrives in NEOX order). This is the rotation
 * mla_cache_append_rmsnorm_rope gives the keys, so q^R . k^R depends only on
 * the distance of the two positions.
 * q_abs      [rows][H][R+P]  out, dims->dtype
 * q_nope     [rows][H][Dn], q_pe [rows][H][P] (before the rope), w_uk [H][Dn][R]
 * positions  [rows] int64, device, 8-byte aligned: each query row's position
 *            (for the decode, query t of request b sits at seq_len - t_q + t)
 * rope_base  rotary base (> 0); unused when P == 0, where this is mla_absorb_q
 */
mla_status mla_absorb_q_rope(void* q_abs, const void* q_nope, const void* q_pe,
                             const void* w_uk, const int64_t* positions, int32_t rows,
                             float rope_base, const mla_dims* dims, void* stream);

/*
 * The query half of the MLA prolog in one call ("aclnnMlaProlog", computation
 * formulas of the query), from each query row's x W^DQ (the down-projected
 * query before its norm) to the decode's query row:
 *   c^Q = RmsNorm(c_q[r]):  gamma_q[i] c_q[r][i] / sqrt(sum_k c_q[r][k]^2 / q_rank + eps)
 *   q^C = c^Q W^UQ (head h: columns h Dn .. h Dn + Dn - 1), q^N = q^C W^UK[h]
 *   q^R = ROPE(c^Q W^QR) (head h: columns h P .. h P + P - 1), the NEOX rope of
 *         mla_absorb_q_rope at positions[r] (the rope columns of W^QR carry
 *         the load-time permutation)
 *   q_abs[r][h] = [ q^N | q^R ]
 * Arithmetic: f32 sums; on the 16-bit paths c^Q and q^C are rounded to the
 * path's type before they enter their products (they are tensor-core
 * operands), q^R is turned in f32 and rounded once.
 * q_abs     [rows][H][R+P]   out, dims->dtype
 * c_q       [rows][q_rank]   in, dims->dtype
 * gamma_q   [q_rank]         in, dims->dtype
 * w_uq      [q_rank][H*Dn]   in, dims->dtype (the page's (k, n) layout)
 * w_qr      [q_rank][H*P]    in, dims->dtype; may be NULL only when P == 0
 * w_uk      [H][Dn][R]       in, dims->dtype
 * positions [rows] int64     in, device, 8-byte aligned; may be NULL only when P == 0
 * q_rank    > 0; a multiple of 8 (of 64 on the tensor-core path: bf16/f16,
 *           kv_rank 512, d_nope and d_rope multiples of 64, d_nope + d_rope <= 256)
 * eps       >= 0, finite; rope_base > 0 (unused when P == 0)
 * dev_err   optional device int32: MLA_DEVERR_TIMEOUT if a bounded wait of the
 *           tensor-core kernel gave up (its output is then undefined)
 * rows == 0 is a no-op. Buffers 16-byte aligned. Stream-ordered, no sync.
 */
mla_status mla_prolog_q(void* q_abs, const void* c_q, const void* gamma_q, const void* w_uq,
                        const void* w_qr, const void* w_uk, const int64_t* positions,
                        int32_t rows, int32_t q_rank, float eps, float rope_base,
                        const mla_dims* dims, int32_t* dev_err, void* stream);

/*
 * Scratch bytes mla_decode_paged needs for this batch shape on the current
 * device (split-KV partial outputs and LSEs). The contents need no
 * initialisation and are dead after the call's work completes on the stream.
 */
mla_status mla_decode_workspace_size(int32_t batch, int32_t max_blocks,
                                     const mla_dims* dims, size_t* bytes);

/*
 * Paged decode ("vllm.cpp src/vt/cpu/cpu_mla_attn.cpp",
 * MlaDecodeAttentionKernel; causal horizon from "memra_engine/mla.rs source",
 * struct MlaInputs). For request b, query t < t_q and head h, with
 * S = seq_lens[b] and horizon = S - t_q + t + 1:
 *   row_j  = kv_cache[block_table[b][j / 16]][j % 16][0 : R+P]
 *   s_j    = scale * (q_abs[b][t][h] . row_j)               j < horizon
 *   out    = sum_j softmax(s)_j * row_j[0 : R]   (V = leading R of the row)
 *   lse    = ln sum_j exp(s_j)                   (natural log, scaled scores)
 * S == 0 gives a zero row and lse = -inf. The work is split over the keys and
 * the partial results merged by their LSE (the split + combine pair named in
 * the header of cpu_mla_attn.cpp).
 *
 * out         [B][t_q][H][R]         out, dims->dtype
 * lse         [B][t_q][H] f32        out; may be NULL
 * q_abs       [B][t_q][H][R+P]       in, dims->dtype
 * kv_cache    [num_blocks][16][R+P]  in, dims->dtype
 * block_table [B][max_blocks] int32  in; entries past ceil(S/16) are not read
 * seq_lens    [B] int32              in
 * scale       softmax scale; normally 1/sqrt(d_nope + d_rope)
 *             ("memra_engine/mla.rs source", MlaDims::scale)
 * workspace   >= mla_decode_workspace_size(batch, max_blocks, dims) bytes,
 *             256-byte aligned, not shared with a concurrent call
 * dev_err     optional device int32: MLA_DEVERR_* bits are OR-ed in when the
 *             device data is invalid (the row is then zero / -inf); the
 *             library never clears it
 * Supported: R+P in {576, 512} with R == 512 for bf16 and f16 (the tensor-core
 * path, for query blocks t_q * H of any size: the 128-row groups' tiles are
 * shared out over the grid's CTA pairs);
 * any R <= 1024, R+P <= 1152 for f32 (the SIMT kernels).
 * batch * t_q * H must stay below 2^31, max_blocks below 2^27 and the cache
 * tiles batch * ceil(max_blocks / 4) (64 tokens each) below 2^31
 * (MLA_ERR_UNSUPPORTED otherwise, also from mla_decode_workspace_size).
 */
mla_status mla_decode_paged(void* out, float* lse, const void* q_abs,
                            const void* kv_cache, const int32_t* block_table,
                            const int32_t* seq_lens, int32_t batch,
                            int32_t max_blocks, int32_t num_blocks,
                            const mla_dims* dims, float scale, void* workspace,
                            size_t workspace_bytes, int32_t* dev_err,
                            void* stream);

/*
 * Bytes of the library-owned decode scratch used by mla_decode_paged_static.
 * Every GPU on which the library's kernels are loaded reserves this much
 * device memory for the life of the process.
 */
#define MLA_STATIC_SCRATCH_BYTES (64u << 20)

/*
 * mla_decode_paged without a caller workspace. The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory when
 * they decode (work recorded into CUDA graphs, serving loops whose allocator
 * forbids cudaMalloc, plugin hosts that hand over only inputs and outputs).
 * It computes exactly what mla_decode_paged computes, with the same arguments
 * minus workspace / workspace_bytes; the split scratch lives in a static
 * device array of MLA_STATIC_SCRATCH_BYTES. It allocates nothing.
 *   - Returns MLA_ERR_INVALID_ARG (with mla_last_error() saying so) when the
 *     batch needs more scratch than MLA_STATIC_SCRATCH_BYTES
 *     (mla_decode_workspace_size tells the need); nothing is enqueued then.
 *   - The first call on a device looks up the array's device address (and
 *     loads the library's module there if needed) and keeps it for the life
 *     of the process; make that first call before any stream capture on that
 *     device. A cudaDeviceReset destroys the context that address belongs to:
 *     do not call this entry point on a device after resetting it.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents (nothing in it needs clearing between calls). Calls whose GPU
 *     work overlaps race on it: issue them on one stream or order them.
 */
mla_status mla_decode_paged_static(void* out, float* lse, const void* q_abs,
                                   const void* kv_cache, const int32_t* block_table,
                                   const int32_t* seq_lens, int32_t batch,
                                   int32_t max_blocks, int32_t num_blocks,
                                   const mla_dims* dims, float scale,
                                   int32_t* dev_err, void* stream);

/*
 * Decompress ("memra_engine/mla.rs source", fn mla_attend_absorbed,
 * decompress step):
 *   out[r][h][j] = sum_l w_uv[h][j][l] * o_lat[r][h][l]
 * out   [rows][H][Dv]  out, dims->dtype
 * o_lat [rows][H][R]   in, dims->dtype
 * w_uv  [H][Dv][R]     in
 */
mla_status mla_decompress_out(void* out, const void* o_lat, const void* w_uv,
                              int32_t rows, const mla_dims* dims, void* stream);

/*
 * Bytes of scratch mla_attend_absorbed needs: the absorbed queries, the
 * latent output and the decode's split scratch.
 */
mla_status mla_attend_workspace_size(int32_t batch, int32_t max_blocks,
                                     const mla_dims* dims, size_t* bytes);

/*
 * The absorbed attention of one decode step ("memra_engine/mla.rs source",
 * fn mla_attend_absorbed): absorb, paged decode, decompress, as
 *   q_abs = mla_absorb_q(q_nope, q_pe, w_uk)          rows = batch * t_q
 *   o_lat, lse = mla_decode_paged(q_abs, kv_cache, ...)
 *   out = mla_decompress_out(o_lat, w_uv)
 * with the same results (the same bits) as those three calls. On the bf16
 * tensor-core path, for up to 256 query rows per request (t_q * n_head), the
 * decompress also merges the decode's split rows (the combine) while it
 * streams W_UV, and the decode starts its cache stream while the absorb
 * finishes; larger query blocks (prefill chunks) run the three calls.
 * out         [B][t_q][H][Dv]  out, dims->dtype
 * lse         [B][t_q][H] f32  out; may be NULL
 * q_nope      [B][t_q][H][Dn], q_pe [B][t_q][H][P] (NULL when P == 0)
 * w_uk        [H][Dn][R], w_uv [H][Dv][R]
 * kv_cache, block_table, seq_lens, batch, max_blocks, num_blocks, scale,
 * dev_err     as for mla_decode_paged
 * workspace   >= mla_attend_workspace_size(batch, max_blocks, dims) bytes,
 *             256-byte aligned, not shared with a concurrent call
 */
mla_status mla_attend_absorbed(void* out, float* lse, const void* q_nope,
                               const void* q_pe, const void* w_uk, const void* w_uv,
                               const void* kv_cache, const int32_t* block_table,
                               const int32_t* seq_lens, int32_t batch,
                               int32_t max_blocks, int32_t num_blocks,
                               const mla_dims* dims, float scale, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err,
                               void* stream);

/*
 * Cache append ("vllm.v1.attention.backends.mla.cpu_mla",
 * CPUMLAImpl.do_kv_cache_update): the step before decode on every token.
 * With flat = kv_cache viewed as [num_blocks * 16][R + P], for every token n
 * whose slot_mapping[n] >= 0:
 *   flat[slot_mapping[n]] = [kv_c[n][0:R] | k_pe[n][0:P]]   cast to dims->dtype
 * kv_cache     [num_blocks][16][R+P]  in/out, dims->dtype
 * kv_c         [n_tokens][R]          in, src_dtype (MLA_F32 or MLA_BF16); the
 *                                     latent rows, already RMS-normed
 * k_pe         [n_tokens][P]          in, src_dtype, already roped; may be NULL
 *                                     only when P == 0
 * slot_mapping [n_tokens] int64       in; a negative slot is padding and is
 *                                     skipped (the page's valid mask)
 * A slot >= num_blocks * 16 is skipped and MLA_DEVERR_BAD_SLOT is OR-ed into
 * the optional device word dev_err. The cast to bf16 rounds to nearest, ties
 * to even; a NaN stays a NaN. Slots should be unique: when two tokens name
 * one slot, the row that lands there is one of theirs, unspecified which.
 * Buffers 16-byte aligned; n_tokens == 0 is a no-op. Stream-ordered, no sync.
 */
mla_status mla_cache_append(void* kv_cache, const void* kv_c, const void* k_pe,
                            const int64_t* slot_mapping, int32_t n_tokens, int32_t num_blocks,
                            int32_t src_dtype, const mla_dims* dims, int32_t* dev_err,
                            void* stream);

/*
 * Cache append with the key half of the MLA prolog fused in ("aclnnMlaProlog",
 * computation formulas of the key: c^KV = RmsNorm(x W^DKV) and
 * k^R = ROPE(x W^KR), both stored in the cache). Takes the projections x W^DKV
 * and x W^KR and writes, for every token n whose slot_mapping[n] >= 0,
 *   flat[slot_mapping[n]] = [ gamma * kv_c[n] / RMS(kv_c[n]) |
 *                             rope_neox(k_pe[n], positions[n]) ]   cast to dims->dtype
 * with RMS(x) = sqrt(mean_i x_i^2 + eps) over the R latent elements, and the
 * NEOX rope of the "memra_engine/mla.rs source" (fn rope_neox): pair
 * (j, j + P/2) rotated by theta_j = pos * s^j, s = rope_base^(-2/P), theta
 * stepped from pos by s in f32. The rope features are in NEOX order: the
 * load-time permutation (below) has been applied to W^KR's rope rows.
 * kv_cache, slot_mapping, num_blocks, dev_err: as mla_cache_append.
 * kv_c      [n_tokens][R]   in, src_dtype; the latent before the norm
 * k_pe      [n_tokens][P]   in, src_dtype; before the rope. NULL only if P == 0
 * gamma     [R]             in, src_dtype; the norm's weight
 * positions [n_tokens] int64 in; each token's position (theta uses it as an
 *                           f32, exact below 2^24). NULL only if P == 0
 * eps       >= 0, finite; rope_base > 0, finite (unused when P == 0)
 * Arithmetic in f32 (sum of squares, scale, rotation); the cast to bf16
 * rounds to nearest even. kv_c, gamma, kv_cache 16-byte aligned; slot_mapping
 * and positions 8-byte aligned. n_tokens == 0 is a no-op. Stream-ordered.
 */
mla_status mla_cache_append_rmsnorm_rope(void* kv_cache, const void* kv_c, const void* k_pe,
                                         const void* gamma, const int64_t* positions,
                                         const int64_t* slot_mapping, int32_t n_tokens,
                                         int32_t num_blocks, int32_t src_dtype, float eps,
                                         float rope_base, const mla_dims* dims, int32_t* dev_err,
                                         void* stream);

/*
 * Load-time rope permutation ("memra_engine/mla.rs source", fn
 * norm_to_neox_perm): perm_out[src] = NEOX index of interleaved index src,
 * pi(2j) = j, pi(2j+1) = j + n_dims/2. Host only. n_dims must be even, >= 0.
 */
mla_status mla_rope_norm_to_neox_perm(int32_t n_dims, int32_t* perm_out);

/*
 * Apply the permutation in place to the column span [col0, col0 + n_dims) of
 * each of `rows` rows of a host matrix (row stride in elements):
 * new[col0 + pi(i)] = old[col0 + i]. elem_bytes is 2 (bf16/f16) or 4 (f32).
 * Used on activations whose rope features are laid out interleaved.
 */
mla_status mla_permute_rope_cols(void* x, int32_t elem_bytes, int64_t rows,
                                 int64_t row_stride, int32_t col0,
                                 int32_t n_dims);

/*
 * Apply the permutation in place to the rows [row0, row0 + n_dims) of a host
 * row-major matrix whose rows are row_len elements long: new row row0 + pi(i)
 * = old row row0 + i. This is the "rope rows of the projection weights at
 * load" form of the same permutation.
 */
mla_status mla_permute_rope_rows(void* w, int32_t elem_bytes, int64_t row_len,
                                 int32_t row0, int32_t n_dims);

/*
 * Test hook for the decode's timeout path; the pages have no counterpart (the
 * CPU kernel of "vllm.cpp cpu_mla_attn.cpp" aborts the process on bad input,
 * which a GPU kernel cannot do; this library's kernels give every wait a time
 * limit instead, and report a wait that gave up in dev_err).
 *   limit_ns  the limit of every bounded wait of the tensor-core decode
 *             launches issued after this call, in nanoseconds; 0 restores the
 *             default (2 s)
 *   stall     nonzero: in those launches the score MMA warp of every CTA pair
 *             first waits on a barrier that nothing arrives on. That wait gives
 *             up after limit_ns, so does every wait that depended on it; the
 *             kernel then drains the copies it issued, frees its tensor memory,
 *             ORs MLA_DEVERR_TIMEOUT into dev_err and returns. Its outputs are
 *             undefined; the stream and the context stay usable.
 * Process-wide and read at launch time; for tests only. Set it back with
 * (0, 0) before decoding for real. Always returns MLA_OK.
 */
mla_status mla_debug_decode_wait_test(uint64_t limit_ns, int32_t stall);

/* Static description of a status code. */
const char* mla_status_str(mla_status status);

/* Message of the last failing call on this thread ("" if none). */
const char* mla_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
