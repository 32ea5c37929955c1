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
 *   oracle_rmsnorm_rows / oracle_project
 *                          the "aclnnMlaProlog" page, computation formulas of
 *                          the query before the absorb: c^Q = RmsNorm(x W^DQ)
 *                          (its RmsNorm formula, in f64) and the projections
 *                          q^C = c^Q W^UQ, c^Q W^QR (plain f32 sums).
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

/* sum_k x[k sx] y[k sy] for k = 0 .. n-1, added in index order onto `start`,
 * each product rounded before it is added. Every f32 dot product of this
 * file is this one summation. */
static float dot_from(float start, const float* x, int64_t sx, const float* y, int64_t sy,
                      int n) {
    float s = start;
    for (int k = 0; k < n; ++k) s += x[k * sx] * y[k * sy];
    return s;
}

/* the same over a row of a typed buffer: sum_d q[d] * base[off + d] */
static float dot_elem(const float* q, const void* base, int dtype, int64_t off, int n) {
    float s = 0.0f;
    for (int d = 0; d < n; ++d) s += q[d] * load_elem(base, dtype, off + d);
    return s;
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
    /* one (row, head) pair at a time, row-major like the buffers */
    for (int64_t rh = 0; rh < (int64_t)rows * n_head; ++rh) {
        const int h = (int)(rh % n_head);
        const float* w_h = w_uk + (int64_t)h * d_nope * kv_rank; /* [d_nope][kv_rank] */
        const float* q = q_nope + rh * d_nope;
        float* dst = q_abs + rh * W;
        /* q_lat[l]: the query against column l of w_uk[h] */
        for (int l = 0; l < kv_rank; ++l) dst[l] = dot_from(0.0f, q, 1, w_h + l, kv_rank, d_nope);
        /* the rope part rides along as it is */
        memcpy(dst + kv_rank, q_pe + rh * d_rope, (size_t)d_rope * sizeof(float));
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
/* Single-pass softmax state (cpu_mla_attn.cpp, MlaDecodeAttentionKernel):
 * the largest scaled score taken so far, the sum of exp(score - largest), and
 * the matching weighted sum of value rows. */
typedef struct {
    float top;   /* running maximum; -inf before the first key */
    float mass;  /* sum of exp(score - top) */
    float* acc;  /* sum of exp(score - top) * value row, n entries */
    int n;
} run_softmax;

/* Take one key: its scaled score s and its value row, n entries of `base`
 * from element `off`. When the maximum grows, everything summed so far is
 * scaled by exp(old top - new top); while nothing has been summed (old top
 * -inf) that factor is 0, never exp(-inf + inf). */
static void run_softmax_take(run_softmax* st, float s, const void* base, int dtype,
                             int64_t off) {
    const float top = st->top > s ? st->top : s;
    const float carry = isinf(st->top) ? 0.0f : expf(st->top - top);
    const float w = expf(s - top);
    for (int d = 0; d < st->n; ++d)
        st->acc[d] = st->acc[d] * carry + w * load_elem(base, dtype, off + d);
    st->mass = st->mass * carry + w;
    st->top = top;
}

/* o = acc / mass and lse = top + ln mass; zeros and -inf when no key was
 * taken */
static void run_softmax_result(const run_softmax* st, float* o, float* lse) {
    const int any = st->mass > 0.0f;
    const float inv = any ? 1.0f / st->mass : 0.0f;
    for (int d = 0; d < st->n; ++d) o[d] = any ? st->acc[d] * inv : 0.0f;
    *lse = any ? st->top + logf(st->mass) : -INFINITY;
}

/* Element offset of key j's row in the paged cache: the block the request's
 * table names for j / block_size, row j % block_size in it; -1 when that
 * block is outside the pool. */
static int64_t paged_row(const int32_t* bt_row, int j, int block_size, int num_blocks, int W) {
    const int32_t blk = bt_row[j / block_size];
    if (blk < 0 || blk >= num_blocks) return -1;
    return ((int64_t)blk * block_size + j % block_size) * W;
}

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
    /* keys the query sees: the t_q queries are the request's last positions
       (mla.rs, struct MlaInputs), so query t sees keys 0 .. seq_len - t_q + t */
    int status = ORACLE_OK;
    int horizon = 0;
    if (seq_len > 0) {
        if (seq_len < t_q)
            status = ORACLE_SEQ_SHORTER_THAN_TQ;
        else if (seq_len > max_blocks * block_size)
            status = ORACLE_SEQ_TOO_LONG;
        else
            horizon = seq_len - t_q + t + 1;
    }
    const int j0 = j_begin > 0 ? j_begin : 0;
    const int j1 = j_end < horizon ? j_end : horizon;

    for (int d = 0; d < W; ++d) q_f[d] = load_elem(q_row, q_dtype, d);
    for (int d = 0; d < kv_rank; ++d) acc[d] = 0.0f;
    run_softmax st = {-INFINITY, 0.0f, acc, kv_rank};
    for (int j = j0; j < j1 && status == ORACLE_OK; ++j) {
        const int64_t off = paged_row(bt_row, j, block_size, num_blocks, W);
        if (off < 0) {
            status = ORACLE_BAD_BLOCK;
            break;
        }
        /* the score spans the whole row [c_kv | k_pe]; the value is its
           leading kv_rank entries */
        const float s = dot_elem(q_f, kv_cache, kv_dtype, off, W) * scale;
        run_softmax_take(&st, s, kv_cache, kv_dtype, off);
    }
    if (status != ORACLE_OK) { /* an invalid request yields the empty result */
        st.top = -INFINITY;
        st.mass = 0.0f;
    }
    run_softmax_result(&st, o_out, lse_out);
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
    for (int64_t rh = 0; rh < (int64_t)rows * n_head; ++rh) {
        const float* w_h = w_uv + (rh % n_head) * d_v * kv_rank; /* [d_v][kv_rank] */
        const float* o = o_lat + rh * kv_rank;
        for (int j = 0; j < d_v; ++j)
            out[rh * d_v + j] = dot_from(0.0f, w_h + (int64_t)j * kv_rank, 1, o, 1, kv_rank);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* the two forms over a contiguous cache (mla.rs)                              */
/* ------------------------------------------------------------------------- */
/* softmax over s[0..n) in place: exp(s - max) / sum, two passes */
static void to_probabilities(float* s, int n) {
    float top = -INFINITY;
    for (int k = 0; k < n; ++k)
        if (s[k] > top) top = s[k];
    float total = 0.0f;
    for (int k = 0; k < n; ++k) total += (s[k] = expf(s[k] - top));
    const float inv = 1.0f / total;
    for (int k = 0; k < n; ++k) s[k] = s[k] * inv;
}

/* One head's keys and values, decompressed from every latent row:
 * k_nope[t][p] = w_uk[h][p] . c_kv[t] and v[t][j] = w_uv[h][j] . c_kv[t]. */
static void expand_head(float* k_nope, float* v, const float* c_kv, const float* wk,
                        const float* wv, int t_kv, int dn, int dv, int r) {
    for (int t = 0; t < t_kv; ++t) {
        const float* c = c_kv + (int64_t)t * r;
        for (int p = 0; p < dn; ++p)
            k_nope[(int64_t)t * dn + p] = dot_from(0.0f, wk + (int64_t)p * r, 1, c, 1, r);
        for (int j = 0; j < dv; ++j)
            v[(int64_t)t * dv + j] = dot_from(0.0f, wv + (int64_t)j * r, 1, c, 1, r);
    }
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
    const int dn = d_nope, dr = d_rope, dv = d_v, r = kv_rank;
    for (int h = 0; h < n_head; ++h) {
        /* every key and value of this head, in full */
        expand_head(k_nope, v, c_kv, w_uk + (int64_t)h * dn * r, w_uv + (int64_t)h * dv * r,
                    t_kv, dn, dv, r);
        for (int i = 0; i < t_q; ++i) {
            const int64_t qrow = (int64_t)i * n_head + h;
            const int n_vis = t_kv - t_q + i + 1; /* causal: keys 0 .. t_kv - t_q + i */
            /* ordinary attention with a d_nope + d_rope wide query and key */
            for (int t = 0; t < n_vis; ++t) {
                const float nope = dot_from(0.0f, q_nope + qrow * dn, 1,
                                            k_nope + (int64_t)t * dn, 1, dn);
                scores[t] = dot_from(nope, q_pe + qrow * dr, 1, k_pe + (int64_t)t * dr, 1, dr) *
                            scale;
            }
            to_probabilities(scores, n_vis);
            for (int j = 0; j < dv; ++j)
                out[qrow * dv + j] = dot_from(0.0f, scores, 1, v + j, dv, n_vis);
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
    const int dn = d_nope, dr = d_rope, dv = d_v, r = kv_rank;
    for (int h = 0; h < n_head; ++h) {
        const float* wk = w_uk + (int64_t)h * dn * r;
        const float* wv = w_uv + (int64_t)h * dv * r;
        for (int i = 0; i < t_q; ++i) {
            const int64_t qrow = (int64_t)i * n_head + h;
            const int n_vis = t_kv - t_q + i + 1;
            /* fold the query into rank space: q_lat[l] = q_nope . column l of w_uk[h] */
            for (int l = 0; l < r; ++l) q_lat[l] = dot_from(0.0f, q_nope + qrow * dn, 1, wk + l, r, dn);
            /* MQA scores against the raw rows [c_kv | k_pe] */
            for (int t = 0; t < n_vis; ++t) {
                const float lat = dot_from(0.0f, q_lat, 1, c_kv + (int64_t)t * r, 1, r);
                scores[t] = dot_from(lat, q_pe + qrow * dr, 1, k_pe + (int64_t)t * dr, 1, dr) *
                            scale;
            }
            to_probabilities(scores, n_vis);
            /* the output in latent space, then decompressed once */
            for (int l = 0; l < r; ++l) o_lat[l] = dot_from(0.0f, scores, 1, c_kv + l, r, n_vis);
            for (int j = 0; j < dv; ++j)
                out[qrow * dv + j] = dot_from(0.0f, wv + (int64_t)j * r, 1, o_lat, 1, r);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* rope pairings and the load-time permutation (mla.rs, rope section)          */
/* ------------------------------------------------------------------------- */
/* Turn the plane of entries u and v of x by the angle a:
 * x[u] <- x[u] cos a - x[v] sin a,  x[v] <- x[u] sin a + x[v] cos a,
 * each product rounded before the sum. */
static void turn_plane(float* x, int u, int v, float a) {
    const float sn = sinf(a), cs = cosf(a);
    const float xu = x[u], xv = x[v];
    x[u] = xu * cs - xv * sn;
    x[v] = xu * sn + xv * cs;
}

/* The rope of the mla.rs rope functions turns n_dims / 2 planes of x. Plane k
 * turns by pos * base^(-2k/n_dims), reached as those functions reach it: the
 * angle of plane 0 is pos, and each next plane's is the previous one times
 * base^(-2/n_dims), rounded to f32 at every step. The two layouts differ only
 * in which entries form plane k. */

/* interleaved ("NORM") layout: plane k is entries 2k and 2k + 1 */
void oracle_rope_interleaved(float* x, int n_dims, float pos, float base) {
    const float step = powf(base, -2.0f / (float)n_dims);
    float angle = pos;
    for (int k = 0; k < n_dims / 2; ++k, angle *= step) turn_plane(x, 2 * k, 2 * k + 1, angle);
}

/* NEOX layout: plane k is entries k and k + n_dims / 2 */
void oracle_rope_neox(float* x, int n_dims, float pos, float base) {
    const float step = powf(base, -2.0f / (float)n_dims);
    const int half = n_dims / 2;
    float angle = pos;
    for (int k = 0; k < half; ++k, angle *= step) turn_plane(x, k, k + half, angle);
}

/* The load-time permutation (mla.rs, norm_to_neox_perm), as an index map
 * from the interleaved layout to the NEOX one: entry i is plane i / 2, its
 * first member when i is even (-> i / 2) and its second when odd
 * (-> i / 2 + n_dims / 2). */
int oracle_norm_to_neox_perm(int n_dims, int32_t* perm) {
    if (n_dims < 0 || (n_dims & 1)) return ORACLE_BAD_ARG;
    for (int i = 0; i < n_dims; ++i) perm[i] = (i & 1) ? (i >> 1) + n_dims / 2 : (i >> 1);
    return ORACLE_OK;
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

/* c^Q = RmsNorm(x W^DQ), one query row r at a time: out[r][i] = gamma_i x_i /
 * RMS(x) with RMS(x) = sqrt(sum_k x_k^2 / n + eps) over the row's n elements
 * x = xin[r] (the page's RmsNorm formula; f64 arithmetic, the result stored as
 * f32). xin and gamma are of src_dtype (f32, or bf16 bit patterns). */
int oracle_rmsnorm_rows(float* out, const void* xin, const void* gamma, int src_dtype, int rows,
                        int n, double eps) {
    if (rows < 0 || n <= 0 || !(eps >= 0.0)) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int k = 0; k < n; ++k) {
            const double x = load_elem(xin, src_dtype, (int64_t)r * n + k);
            ss += x * x;
        }
        const double rms = sqrt(ss / (double)n + eps);
        for (int i = 0; i < n; ++i) {
            const double x = load_elem(xin, src_dtype, (int64_t)r * n + i);
            const double g = load_elem(gamma, src_dtype, i);
            out[(int64_t)r * n + i] = (float)(g * x / rms);
        }
    }
    return ORACLE_OK;
}

/* A projection of the prolog (q^C = c^Q W^UQ, or c^Q W^QR): y[r][j] =
 * sum_k x[r][k] w[k][j], the weight stored (k, n) as the page lays out its
 * projection weights; one f32 sum per output in k order. */
int oracle_project(float* y, const float* x, const float* w, int rows, int k, int n) {
    if (rows < 0 || k <= 0 || n <= 0) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r)
        for (int j = 0; j < n; ++j)
            y[(int64_t)r * n + j] = dot_from(0.0f, x + (int64_t)r * k, 1, w + j, n, k);
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
