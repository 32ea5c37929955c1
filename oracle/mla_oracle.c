/*
 * Plain CPU oracle for absorbed multi-head latent attention (MLA) decode over a
 * paged latent cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header or constant with the CUDA library.
 *
 * Precision: f32 storage and f32 accumulation, one sequential summation per
 * dot product, as the pages fix it (the "memra_engine/mla.rs" module docs
 * describe their oracle as f32 code on the CPU; the header comment of
 * "vllm.cpp cpu_mla_attn.cpp" has every sum in f32). Built with
 * -ffp-contract=off so that no multiply-add is fused and x86 and Arm builds
 * sum identically.
 *
 * Every function is a direct restatement of one passage:
 *   oracle_absorb_q        mla.rs, fn mla_attend_absorbed, absorb step
 *                          (q_lat[l] = sum_p q_nope[p] * w_uk[h][p][l]), and
 *                          the vLLM CPU MLA page, CPUMLAImpl.forward_mqa
 *                          (the decode query is concat(q_lat, q_pe)).
 *   oracle_decode_range    cpu_mla_attn.cpp, MlaDecodeAttentionKernel: block
 *                          table walk, single-pass online softmax with the
 *                          "rescale 0 while the max is -inf" rule, V = leading
 *                          kv_rank slice of the same cache row, LSE = m + ln l,
 *                          zero row and -inf LSE when no key is visible.
 *                          Causal horizon for query t of t_q: mla.rs, struct
 *                          MlaInputs doc (rows 0 ..= t_kv - t_q + t).
 *   oracle_combine         the split+combine schedule named in the header of
 *                          cpu_mla_attn.cpp (merge of partial softmaxes by
 *                          their LSE, lse = max + ln(sum)).
 *   oracle_decompress      mla.rs, fn mla_attend_absorbed, decompress step
 *                          (out[j] = sum_l w_uv[h][j][l] * o_lat[l]).
 *   oracle_attend_naive    mla.rs, fn mla_attend_naive (per-head decompression
 *                          of the whole cache, ordinary two-pass softmax).
 *   oracle_attend_absorbed mla.rs, fn mla_attend_absorbed (contiguous cache,
 *                          two-pass softmax).
 *   oracle_rope_interleaved / oracle_rope_neox / oracle_norm_to_neox_perm
 *                          mla.rs, fns rope_interleaved, rope_neox,
 *                          norm_to_neox_perm.
 *   oracle_cache_append    the vLLM CPU MLA page, CPUMLAImpl.do_kv_cache_update
 *                          (scatter of [kv_c | k_pe] rows by slot mapping,
 *                          padding slots -1 skipped, cast to the cache type).
 *   oracle_absorb_q_rope   the "aclnnMlaProlog" page, computation formulas of
 *                          the query (q^N = q^C W^UK; q^R = ROPE(c^Q W^QR)):
 *                          the absorb above with the mla.rs NEOX rope of the
 *                          query's rope part at the row's position.
 *   oracle_kv_prolog_row / oracle_cache_append_rmsnorm_rope
 *                          the "aclnnMlaProlog" page, computation formulas of
 *                          the key (RmsNorm of the latent, rope of k^R, both
 *                          stored in the cache), with the mla.rs NEOX rope and
 *                          the scatter of do_kv_cache_update. The RmsNorm is
 *                          taken in f64 (the page fixes no precision).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_BLOCK (-2)
#define ORACLE_SEQ_TOO_LONG (-3)
#define ORACLE_SEQ_SHORTER_THAN_TQ (-4)

/* element types accepted for the query and cache buffers of the decode */
#define ORACLE_F32 0
#define ORACLE_BF16 1 /* raw bf16 bit patterns (uint16) */

/* bf16 -> f32 is exact: the bf16 pattern is the upper half of the f32 one. */
static float load_elem(const void* base, int dtype, int64_t i) {
    if (dtype == ORACLE_F32) return ((const float*)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------- */
/* absorb: q_abs[r][h][0:R] = w_uk[h]^T q_nope[r][h]; q_abs[r][h][R:R+P] = q_pe */
/* ------------------------------------------------------------------------- */
int oracle_absorb_q(float* q_abs, const float* q_nope, const float* q_pe,
                    const float* w_uk, int rows, int n_head, int d_nope,
                    int d_rope, int kv_rank) {
    if (rows < 0 || n_head <= 0 || d_nope <= 0 || d_rope < 0 || kv_rank <= 0)
        return ORACLE_BAD_ARG;
    const int W = kv_rank + d_rope;
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < n_head; ++h) {
            const float* qn = q_nope + ((int64_t)r * n_head + h) * d_nope;
            const float* wuk = w_uk + (int64_t)h * d_nope * kv_rank;
            float* dst = q_abs + ((int64_t)r * n_head + h) * W;
            for (int l = 0; l < kv_rank; ++l) dst[l] = 0.0f;
            for (int p = 0; p < d_nope; ++p) {
                const float qv = qn[p];
                const float* wrow = wuk + (int64_t)p * kv_rank;
                for (int l = 0; l < kv_rank; ++l) dst[l] += qv * wrow[l];
            }
            const float* qp = q_pe + ((int64_t)r * n_head + h) * d_rope;
            for (int j = 0; j < d_rope; ++j) dst[kv_rank + j] = qp[j];
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* decode of one query row over the visible keys j in [j_begin, j_end)        */
/* ------------------------------------------------------------------------- */
/*
 * q_row     : W = kv_rank + d_rope values (dtype q_dtype)
 * kv_cache  : [num_blocks][block_size][W] (dtype kv_dtype)
 * bt_row    : the request's block-table row, max_blocks entries
 * seq_len   : keys in the request's cache; the query is number t of t_q and
 *             sees keys 0 .. seq_len - t_q + t
 * [j_begin, j_end) restricts the walk to a slice of the visible keys (a split);
 *             pass 0 and seq_len for the whole request.
 * o_out     : kv_rank values = acc / l (zeros when nothing was visible)
 * lse_out   : m + ln l, or -inf when nothing was visible
 */
int oracle_decode_range(float* o_out, float* lse_out, const void* q_row,
                        int q_dtype, const void* kv_cache, int kv_dtype,
                        const int32_t* bt_row, int seq_len, int t_q, int t,
                        int kv_rank, int d_rope, int block_size,
                        int max_blocks, int num_blocks, float scale,
                        int j_begin, int j_end, float* acc /* kv_rank scratch */,
                        float* q_f /* W scratch */) {
    const int W = kv_rank + d_rope;
    if (seq_len < 0 || t_q <= 0 || t < 0 || t >= t_q || block_size <= 0)
        return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
    int horizon = 0; /* number of keys this query may see */
    if (seq_len > 0) {
        if (seq_len < t_q) {
            status = ORACLE_SEQ_SHORTER_THAN_TQ;
        } else if (seq_len > max_blocks * block_size) {
            status = ORACLE_SEQ_TOO_LONG;
        } else {
            horizon = seq_len - t_q + t + 1;
        }
    }
    if (j_begin < 0) j_begin = 0;
    if (j_end > horizon) j_end = horizon;

    for (int d = 0; d < W; ++d) q_f[d] = load_elem(q_row, q_dtype, d);

    float m = -INFINITY;
    float l = 0.0f;
    for (int d = 0; d < kv_rank; ++d) acc[d] = 0.0f;

    for (int j = j_begin; j < j_end && status == ORACLE_OK; ++j) {
        const int slot = j / block_size;
        const int32_t blk = bt_row[slot];
        if (blk < 0 || blk >= num_blocks) {
            status = ORACLE_BAD_BLOCK;
            break;
        }
        const int64_t entry = ((int64_t)blk * block_size + (j % block_size)) * W;
        float qk = 0.0f;
        for (int d = 0; d < W; ++d)
            qk += q_f[d] * load_elem(kv_cache, kv_dtype, entry + d);
        qk *= scale;
        const float m_new = m > qk ? m : qk;
        const float rescale = isinf(m) ? 0.0f : expf(m - m_new);
        const float p = expf(qk - m_new);
        for (int d = 0; d < kv_rank; ++d)
            acc[d] = acc[d] * rescale + p * load_elem(kv_cache, kv_dtype, entry + d);
        l = l * rescale + p;
        m = m_new;
    }
    if (status != ORACLE_OK) { /* an invalid request yields the empty result */
        m = -INFINITY;
        l = 0.0f;
    }
    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
    for (int d = 0; d < kv_rank; ++d) o_out[d] = l > 0.0f ? acc[d] * inv : 0.0f;
    *lse_out = l > 0.0f ? m + logf(l) : -INFINITY;
    return status;
}

/*
 * Decode of selected query rows. Row id = (b * t_q + t) * n_head + h, the
 * flattened [batch][t_q][n_head] index. o_out is [n_rows][kv_rank], lse_out is
 * [n_rows]. Returns the first error met (rows with errors hold the empty
 * result) or ORACLE_OK.
 */
int oracle_decode_rows(float* o_out, float* lse_out, const void* q_abs,
                       int q_dtype, const void* kv_cache, int kv_dtype,
                       const int32_t* block_table, const int32_t* seq_lens,
                       int batch, int t_q, int n_head, int kv_rank, int d_rope,
                       int block_size, int max_blocks, int num_blocks,
                       float scale, const int64_t* row_ids, int64_t n_rows,
                       float* scratch /* kv_rank + kv_rank + d_rope floats */) {
    if (batch < 0 || t_q <= 0 || n_head <= 0 || kv_rank <= 0 || d_rope < 0)
        return ORACLE_BAD_ARG;
    const int W = kv_rank + d_rope;
    const int elem = q_dtype == ORACLE_F32 ? 4 : 2;
    int first_err = ORACLE_OK;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = row_ids[i];
        if (r < 0 || r >= (int64_t)batch * t_q * n_head) return ORACLE_BAD_ARG;
        const int64_t bt_idx = r / n_head; /* b * t_q + t */
        const int b = (int)(bt_idx / t_q);
        const int t = (int)(bt_idx % t_q);
        const char* q_row = (const char*)q_abs + r * W * elem;
        int st = oracle_decode_range(
            o_out + i * kv_rank, lse_out + i, q_row, q_dtype, kv_cache, kv_dtype,
            block_table + (int64_t)b * max_blocks, seq_lens[b], t_q, t, kv_rank,
            d_rope, block_size, max_blocks, num_blocks, scale, 0, seq_lens[b],
            scratch, scratch + kv_rank);
        if (st != ORACLE_OK && first_err == ORACLE_OK) first_err = st;
    }
    return first_err;
}

/* All rows, in order: o_out is [batch][t_q][n_head][kv_rank]. */
int oracle_decode_paged(float* o_out, float* lse_out, const void* q_abs,
                        int q_dtype, const void* kv_cache, int kv_dtype,
                        const int32_t* block_table, const int32_t* seq_lens,
                        int batch, int t_q, int n_head, int kv_rank, int d_rope,
                        int block_size, int max_blocks, int num_blocks,
                        float scale, float* scratch) {
    int first_err = ORACLE_OK;
    const int64_t n = (int64_t)batch * t_q * n_head;
    for (int64_t r = 0; r < n; ++r) {
        int st = oracle_decode_rows(o_out + r * kv_rank, lse_out + r, q_abs,
                                    q_dtype, kv_cache, kv_dtype, block_table,
                                    seq_lens, batch, t_q, n_head, kv_rank,
                                    d_rope, block_size, max_blocks, num_blocks,
                                    scale, &r, 1, scratch);
        if (st != ORACLE_OK && first_err == ORACLE_OK) first_err = st;
    }
    return first_err;
}

/* ------------------------------------------------------------------------- */
/* merge of partial softmax results by their LSE                              */
/* ------------------------------------------------------------------------- */
/*
 * o_parts [n_parts][kv_rank] are normalised partial outputs, lse_parts their
 * LSEs (-inf for an empty part). M = max lse_s, w_s = exp(lse_s - M),
 * out = sum w_s o_s / sum w_s, lse = M + ln sum w_s. All parts empty gives
 * zeros and -inf.
 */
int oracle_combine(float* o_out, float* lse_out, const float* o_parts,
                   const float* lse_parts, int n_parts, int kv_rank) {
    if (n_parts < 0 || kv_rank <= 0) return ORACLE_BAD_ARG;
    float M = -INFINITY;
    for (int s = 0; s < n_parts; ++s)
        if (lse_parts[s] > M) M = lse_parts[s];
    for (int d = 0; d < kv_rank; ++d) o_out[d] = 0.0f;
    if (isinf(M) && M < 0) {
        *lse_out = -INFINITY;
        return ORACLE_OK;
    }
    float wsum = 0.0f;
    for (int s = 0; s < n_parts; ++s) {
        if (isinf(lse_parts[s])) continue; /* an empty part has weight 0 */
        const float w = expf(lse_parts[s] - M);
        wsum += w;
        for (int d = 0; d < kv_rank; ++d) o_out[d] += w * o_parts[(int64_t)s * kv_rank + d];
    }
    for (int d = 0; d < kv_rank; ++d) o_out[d] /= wsum;
    *lse_out = M + logf(wsum);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* decompress: out[r][h][j] = sum_l w_uv[h][j][l] * o_lat[r][h][l]            */
/* ------------------------------------------------------------------------- */
int oracle_decompress(float* out, const float* o_lat, const float* w_uv,
                      int rows, int n_head, int d_v, int kv_rank) {
    if (rows < 0 || n_head <= 0 || d_v <= 0 || kv_rank <= 0) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < n_head; ++h) {
            const float* o = o_lat + ((int64_t)r * n_head + h) * kv_rank;
            const float* wuv = w_uv + (int64_t)h * d_v * kv_rank;
            float* dst = out + ((int64_t)r * n_head + h) * d_v;
            for (int j = 0; j < d_v; ++j) {
                const float* wrow = wuv + (int64_t)j * kv_rank;
                float acc = 0.0f;
                for (int l = 0; l < kv_rank; ++l) acc += wrow[l] * o[l];
                dst[j] = acc;
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* the two forms over a contiguous cache (mla.rs)                              */
/* ------------------------------------------------------------------------- */
/* max-subtracted softmax over s[0..n) in place */
static void softmax_inplace(float* s, int n) {
    float m = -INFINITY;
    for (int i = 0; i < n; ++i) m = s[i] > m ? s[i] : m;
    float sum = 0.0f;
    for (int i = 0; i < n; ++i) {
        s[i] = expf(s[i] - m);
        sum += s[i];
    }
    const float inv = 1.0f / sum;
    for (int i = 0; i < n; ++i) s[i] *= inv;
}

/*
 * Layouts (row-major): q_nope [t_q][H][Dn], q_pe [t_q][H][P], c_kv [t_kv][R],
 * k_pe [t_kv][P], w_uk [H][Dn][R], w_uv [H][Dv][R]; out [t_q][H][Dv].
 * Scratch: k_nope t_kv*Dn, v t_kv*Dv, scores t_kv floats.
 */
int oracle_attend_naive(float* out, const float* q_nope, const float* q_pe,
                        const float* c_kv, const float* k_pe, const float* w_uk,
                        const float* w_uv, int t_q, int t_kv, int n_head,
                        int d_nope, int d_rope, int d_v, int kv_rank,
                        float scale, float* k_nope, float* v, float* scores) {
    if (t_q <= 0 || t_q > t_kv) return ORACLE_BAD_ARG;
    const int nh = n_head, dn = d_nope, dr = d_rope, dv = d_v, r = kv_rank;
    for (int64_t i = 0; i < (int64_t)t_q * nh * dv; ++i) out[i] = 0.0f;
    for (int h = 0; h < nh; ++h) {
        const float* wuk = w_uk + (int64_t)h * dn * r;
        const float* wuv = w_uv + (int64_t)h * dv * r;
        for (int t = 0; t < t_kv; ++t) {
            const float* c = c_kv + (int64_t)t * r;
            for (int p = 0; p < dn; ++p) {
                float acc = 0.0f;
                for (int l = 0; l < r; ++l) acc += wuk[(int64_t)p * r + l] * c[l];
                k_nope[(int64_t)t * dn + p] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                float acc = 0.0f;
                for (int l = 0; l < r; ++l) acc += wuv[(int64_t)j * r + l] * c[l];
                v[(int64_t)t * dv + j] = acc;
            }
        }
        for (int i = 0; i < t_q; ++i) {
            const int visible = t_kv - t_q + i + 1;
            const float* qn = q_nope + ((int64_t)i * nh + h) * dn;
            const float* qp = q_pe + ((int64_t)i * nh + h) * dr;
            for (int t = 0; t < visible; ++t) {
                float s = 0.0f;
                for (int p = 0; p < dn; ++p) s += qn[p] * k_nope[(int64_t)t * dn + p];
                for (int p = 0; p < dr; ++p) s += qp[p] * k_pe[(int64_t)t * dr + p];
                scores[t] = s * scale;
            }
            softmax_inplace(scores, visible);
            float* o = out + ((int64_t)i * nh + h) * dv;
            for (int t = 0; t < visible; ++t)
                for (int j = 0; j < dv; ++j) o[j] += scores[t] * v[(int64_t)t * dv + j];
        }
    }
    return ORACLE_OK;
}

/* Scratch: q_lat R, o_lat R, scores t_kv floats. */
int oracle_attend_absorbed(float* out, const float* q_nope, const float* q_pe,
                           const float* c_kv, const float* k_pe,
                           const float* w_uk, const float* w_uv, int t_q,
                           int t_kv, int n_head, int d_nope, int d_rope,
                           int d_v, int kv_rank, float scale, float* q_lat,
                           float* o_lat, float* scores) {
    if (t_q <= 0 || t_q > t_kv) return ORACLE_BAD_ARG;
    const int nh = n_head, dn = d_nope, dr = d_rope, dv = d_v, r = kv_rank;
    for (int h = 0; h < nh; ++h) {
        const float* wuk = w_uk + (int64_t)h * dn * r;
        const float* wuv = w_uv + (int64_t)h * dv * r;
        for (int i = 0; i < t_q; ++i) {
            const int visible = t_kv - t_q + i + 1;
            const float* qn = q_nope + ((int64_t)i * nh + h) * dn;
            const float* qp = q_pe + ((int64_t)i * nh + h) * dr;
            for (int l = 0; l < r; ++l) q_lat[l] = 0.0f;
            for (int p = 0; p < dn; ++p)
                for (int l = 0; l < r; ++l) q_lat[l] += qn[p] * wuk[(int64_t)p * r + l];
            for (int t = 0; t < visible; ++t) {
                const float* c = c_kv + (int64_t)t * r;
                float s = 0.0f;
                for (int l = 0; l < r; ++l) s += q_lat[l] * c[l];
                for (int p = 0; p < dr; ++p) s += qp[p] * k_pe[(int64_t)t * dr + p];
                scores[t] = s * scale;
            }
            softmax_inplace(scores, visible);
            for (int l = 0; l < r; ++l) o_lat[l] = 0.0f;
            for (int t = 0; t < visible; ++t)
                for (int l = 0; l < r; ++l) o_lat[l] += scores[t] * c_kv[(int64_t)t * r + l];
            float* o = out + ((int64_t)i * nh + h) * dv;
            for (int j = 0; j < dv; ++j) {
                float acc = 0.0f;
                for (int l = 0; l < r; ++l) acc += wuv[(int64_t)j * r + l] * o_lat[l];
                o[j] = acc;
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* rope pairings and the load-time permutation (mla.rs, rope section)          */
/* ------------------------------------------------------------------------- */
/* pair (x[2j], x[2j+1]) rotated by theta_j = pos * base^(-2j/n), theta stepped
 * by the factor base^(-2/n) as the page does */
void oracle_rope_interleaved(float* x, int n_dims, float pos, float base) {
    const int half = n_dims / 2;
    const float theta_scale = powf(base, -2.0f / (float)n_dims);
    float theta = pos;
    for (int j = 0; j < half; ++j) {
        const float s = sinf(theta), c = cosf(theta);
        const float a = x[2 * j], b = x[2 * j + 1];
        x[2 * j] = a * c - b * s;
        x[2 * j + 1] = a * s + b * c;
        theta *= theta_scale;
    }
}

/* pair (x[j], x[j+n/2]) rotated by the same theta_j sequence */
void oracle_rope_neox(float* x, int n_dims, float pos, float base) {
    const int half = n_dims / 2;
    const float theta_scale = powf(base, -2.0f / (float)n_dims);
    float theta = pos;
    for (int j = 0; j < half; ++j) {
        const float s = sinf(theta), c = cosf(theta);
        const float a = x[j], b = x[j + half];
        x[j] = a * c - b * s;
        x[j + half] = a * s + b * c;
        theta *= theta_scale;
    }
}

/* ------------------------------------------------------------------------- */
/* cache append (vLLM CPU MLA page, CPUMLAImpl.do_kv_cache_update)            */
/* ------------------------------------------------------------------------- */
/* f32 -> bf16 bits, round to nearest with ties to even (the rounding of a
 * "to(bfloat16)" cast); NaN stays a quiet NaN of the same sign */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

/* Write token n's latent row [kv_c[n] | k_pe[n]] into cache row slot[n] of the
 * flat cache [num_slots][R + P], cast to the cache's element type; a negative
 * slot is padding and is skipped (the page's valid mask). A slot at or past
 * num_slots is an invalid request: skipped and reported (status BAD_BLOCK).
 * src_dtype / cache_dtype: ORACLE_F32 or ORACLE_BF16 (bf16 as uint16 bits). */
int oracle_cache_append(void* cache, int cache_dtype, const void* kv_c, const void* k_pe,
                        int src_dtype, const int64_t* slots, int n_tokens, int64_t num_slots,
                        int kv_rank, int d_rope) {
    if (n_tokens < 0 || kv_rank <= 0 || d_rope < 0) return ORACLE_BAD_ARG;
    const int W = kv_rank + d_rope;
    int status = ORACLE_OK;
    for (int n = 0; n < n_tokens; ++n) {
        const int64_t s = slots[n];
        if (s < 0) continue;
        if (s >= num_slots) {
            status = ORACLE_BAD_BLOCK;
            continue;
        }
        for (int j = 0; j < W; ++j) {
            const float v = j < kv_rank ? load_elem(kv_c, src_dtype, (int64_t)n * kv_rank + j)
                                        : load_elem(k_pe, src_dtype, (int64_t)n * d_rope + (j - kv_rank));
            if (cache_dtype == ORACLE_BF16)
                ((uint16_t*)cache)[s * W + j] = f32_to_bf16_rne(v);
            else
                ((float*)cache)[s * W + j] = v;
        }
    }
    return status;
}

/* source (interleaved) index -> NEOX index: pi(2j) = j, pi(2j+1) = j + n/2 */
int oracle_norm_to_neox_perm(int n_dims, int32_t* perm) {
    if (n_dims < 0 || (n_dims & 1)) return ORACLE_BAD_ARG;
    const int half = n_dims / 2;
    for (int j = 0; j < half; ++j) {
        perm[2 * j] = j;
        perm[2 * j + 1] = j + half;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* Query half of the MLA prolog, as the decode consumes it ("aclnnMlaProlog"  */
/* page, computation formulas of the query)                                   */
/* ------------------------------------------------------------------------- */
/* q_abs[r][h] = [q^N | q^R] for query row r and head h:
 *   q^N = q_nope[r][h] W^UK[h]  (q_nope is q^C = c^Q W^UQ, one head's slice;
 *                                the absorb of oracle_absorb_q)
 *   q^R = the mla.rs NEOX rope of q_pe[r][h] (= c^Q W^QR before the rope,
 *         whose columns carry the load-time permutation) at positions[r], in
 *         f32 as that page computes it: the same rope as the key half's, so
 *         that q^R . k^R depends only on the distance of the two positions. */
int oracle_absorb_q_rope(float* q_abs, const float* q_nope, const float* q_pe,
                         const float* w_uk, const int64_t* positions, int rows, int n_head,
                         int d_nope, int d_rope, int kv_rank, float rope_base) {
    if ((d_rope & 1) || (d_rope > 0 && !(rope_base > 0.0f))) return ORACLE_BAD_ARG;
    const int st = oracle_absorb_q(q_abs, q_nope, q_pe, w_uk, rows, n_head, d_nope, d_rope,
                                   kv_rank);
    if (st != ORACLE_OK || d_rope == 0) return st;
    const int W = kv_rank + d_rope;
    for (int r = 0; r < rows; ++r)
        for (int h = 0; h < n_head; ++h)
            oracle_rope_neox(q_abs + ((int64_t)r * n_head + h) * W + kv_rank, d_rope,
                             (float)positions[r], rope_base);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* KV half of the MLA prolog ("aclnnMlaProlog" page, computation formulas of  */
/* the key: c^KV = RmsNorm(x W^DKV) to the cache, k^R = Cache(ROPE(x W^KR))),  */
/* written by slot mapping as the vLLM CPU MLA page's do_kv_cache_update does  */
/* ------------------------------------------------------------------------- */
/* One token's cache row before the cast, in f64:
 *   row[i]     = gamma_i * x_i / RMS(x),  RMS(x) = sqrt(sum_k x_k^2 / R + eps)
 *                over the R = kv_rank latent elements x = kv_c[n] (the page's
 *                RmsNorm formula; it fixes no precision, so this is f64);
 *   row[R + j] = the mla.rs NEOX rope of k_pe[n] at the token's position, in
 *                f32 as that page computes it (the rope features are in NEOX
 *                order: the load-time permutation was applied to W^KR).
 * gamma has kv_rank elements of src_dtype. */
int oracle_kv_prolog_row(double* row, const void* kv_c, const void* k_pe, const void* gamma,
                         int src_dtype, int64_t n, int64_t position, int kv_rank, int d_rope,
                         double eps, float rope_base) {
    if (kv_rank <= 0 || d_rope < 0 || (d_rope & 1) || d_rope > 4096 || !(eps >= 0.0))
        return ORACLE_BAD_ARG;
    double ss = 0.0;
    for (int k = 0; k < kv_rank; ++k) {
        const double x = load_elem(kv_c, src_dtype, n * kv_rank + k);
        ss += x * x;
    }
    const double rms = sqrt(ss / (double)kv_rank + eps);
    for (int i = 0; i < kv_rank; ++i) {
        const double x = load_elem(kv_c, src_dtype, n * kv_rank + i);
        const double g = load_elem(gamma, src_dtype, i);
        row[i] = g * x / rms;
    }
    if (d_rope > 0) {
        float pe[4096];
        for (int j = 0; j < d_rope; ++j) pe[j] = load_elem(k_pe, src_dtype, n * d_rope + j);
        oracle_rope_neox(pe, d_rope, (float)position, rope_base);
        for (int j = 0; j < d_rope; ++j) row[kv_rank + j] = pe[j];
    }
    return ORACLE_OK;
}

/* For every token n with slot s = slots[n] >= 0: flat cache row s = the row
 * above, rounded to f32 and then cast to the cache type (the kernel rounds
 * from f32 too, so both sides take the bf16 rounding from the same f32
 * value). Padding slots (< 0) are skipped; a slot at or past num_slots is
 * skipped and reported (status BAD_BLOCK), as in oracle_cache_append. */
int oracle_cache_append_rmsnorm_rope(void* cache, int cache_dtype, const void* kv_c,
                                     const void* k_pe, const void* gamma, int src_dtype,
                                     const int64_t* positions, const int64_t* slots, int n_tokens,
                                     int64_t num_slots, int kv_rank, int d_rope, double eps,
                                     float rope_base) {
    if (n_tokens < 0 || kv_rank <= 0 || d_rope < 0 || kv_rank + d_rope > 8192) return ORACLE_BAD_ARG;
    const int W = kv_rank + d_rope;
    double row[8192];
    int status = ORACLE_OK;
    for (int n = 0; n < n_tokens; ++n) {
        const int64_t s = slots[n];
        if (s < 0) continue;
        if (s >= num_slots) {
            status = ORACLE_BAD_BLOCK;
            continue;
        }
        const int st = oracle_kv_prolog_row(row, kv_c, k_pe, gamma, src_dtype, n,
                                            d_rope > 0 ? positions[n] : 0, kv_rank, d_rope, eps,
                                            rope_base);
        if (st != ORACLE_OK) return st;
        for (int j = 0; j < W; ++j) {
            const float v = (float)row[j];
            if (cache_dtype == ORACLE_BF16)
                ((uint16_t*)cache)[s * W + j] = f32_to_bf16_rne(v);
            else
                ((float*)cache)[s * W + j] = v;
        }
    }
    return status;
}
