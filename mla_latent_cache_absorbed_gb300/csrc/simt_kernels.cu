// SIMT (CUDA-core FFMA) kernels of the absorbed MLA decode path.
//
// These serve every geometry and both element types with f32 accumulation.
// The f32 path stays on them: tf32 tensor cores cannot hold the 1e-4 absolute
// error budget of f32 inputs.
//
//   absorb_simt      q_abs = [w_uk[h]^T q_nope | q_pe]   ("memra_engine/mla.rs
//                    source", fn mla_attend_absorbed, absorb step)
//   decode_split     one CTA per (query row, key split): block-table walk and
//                    single-pass online softmax ("vllm.cpp cpu_mla_attn.cpp",
//                    MlaDecodeAttentionKernel), writing a normalised partial
//                    output and its LSE
//   decode_combine   LSE merge of the splits (the split + combine pair of the
//                    same page's header); empty or invalid rows get 0 / -inf
//   decompress_simt  out = w_uv[h] o_lat (mla.rs, decompress step)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "internal.h"

namespace mla {
namespace {

template <typename T>
__device__ __forceinline__ float ld(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}

template <>
__device__ __forceinline__ float ld<__half>(const __half* p, int64_t i) {
    return __half2float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st(T* p, int64_t i, float v);
template <>
__device__ __forceinline__ void st<__half>(__half* p, int64_t i, float v) {
    p[i] = __float2half_rn(v);
}
template <>
__device__ __forceinline__ void st<float>(float* p, int64_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int kRowTile = 16;  // query rows per CTA in the absorb / decompress kernels

// ---------------------------------------------------------------------------
// absorb: grid (H, ceil(R/256), ceil(rows/16)), 256 threads; thread = one l.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) absorb_simt(T* __restrict__ q_abs,
                                                   const T* __restrict__ q_nope,
                                                   const T* __restrict__ q_pe,
                                                   const T* __restrict__ w_uk, int rows,
                                                   int H, int Dn, int P, int R,
                                                   const int64_t* __restrict__ positions,
                                                   float theta_scale) {
    extern __shared__ float sq[];  // [kRowTile][Dn]
    const int h = blockIdx.x;
    const int r0 = blockIdx.z * kRowTile;
    const int nr = min(kRowTile, rows - r0);
    const int W = R + P;
    for (int i = threadIdx.x; i < kRowTile * Dn; i += blockDim.x) {
        const int r = i / Dn, p = i % Dn;
        sq[i] = r < nr ? ld(q_nope, ((int64_t)(r0 + r) * H + h) * Dn + p) : 0.f;
    }
    __syncthreads();
    const int l = blockIdx.y * blockDim.x + threadIdx.x;
    if (l < R) {
        float acc[kRowTile];
#pragma unroll
        for (int r = 0; r < kRowTile; ++r) acc[r] = 0.f;
        const T* w = w_uk + (int64_t)h * Dn * R + l;
        for (int p = 0; p < Dn; ++p) {
            const float wv = ld(w, (int64_t)p * R);
#pragma unroll
            for (int r = 0; r < kRowTile; ++r) acc[r] = fmaf(sq[r * Dn + p], wv, acc[r]);
        }
        for (int r = 0; r < nr; ++r) st(q_abs, ((int64_t)(r0 + r) * H + h) * W + l, acc[r]);
    }
    if (blockIdx.y == 0 && !positions) {
        for (int i = threadIdx.x; i < nr * P; i += blockDim.x) {
            const int r = i / P, j = i % P;
            const int64_t row = (int64_t)(r0 + r) * H + h;
            st(q_abs, row * W + R + j, ld(q_pe, row * P + j));
        }
    } else if (blockIdx.y == 0) {
        // the query's rope at its row's position: NEOX pair (j, j + P/2)
        // turned by theta_j = pos * theta_scale^j, the ratio applied j times
        const int half = P / 2;
        for (int i = threadIdx.x; i < nr * half; i += blockDim.x) {
            const int r = i / half, j = i % half;
            const int64_t row = (int64_t)(r0 + r) * H + h;
            float theta = (float)positions[r0 + r];
            for (int k = 0; k < j; ++k) theta = __fmul_rn(theta, theta_scale);
            float sn, cs;
            sincosf(theta, &sn, &cs);
            const float a = ld(q_pe, row * P + j), b = ld(q_pe, row * P + j + half);
            st(q_abs, row * W + R + j, __fsub_rn(__fmul_rn(a, cs), __fmul_rn(b, sn)));
            st(q_abs, row * W + R + j + half, __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cs)));
        }
    }
}

// ---------------------------------------------------------------------------
// decompress: grid (H, ceil(Dv/8), ceil(rows/16)), 256 threads; warp = one j.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) decompress_simt(T* __restrict__ out,
                                                       const T* __restrict__ o_lat,
                                                       const T* __restrict__ w_uv, int rows,
                                                       int H, int Dv, int R) {
    extern __shared__ float so[];  // [kRowTile][R]
    const int h = blockIdx.x;
    const int r0 = blockIdx.z * kRowTile;
    const int nr = min(kRowTile, rows - r0);
    for (int i = threadIdx.x; i < kRowTile * R; i += blockDim.x) {
        const int r = i / R, l = i % R;
        so[i] = r < nr ? ld(o_lat, ((int64_t)(r0 + r) * H + h) * R + l) : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.y * 8 + warp;
    if (j >= Dv) return;
    float acc[kRowTile];
#pragma unroll
    for (int r = 0; r < kRowTile; ++r) acc[r] = 0.f;
    const T* w = w_uv + ((int64_t)h * Dv + j) * R;
    for (int l = lane; l < R; l += 32) {
        const float wv = ld(w, l);
#pragma unroll
        for (int r = 0; r < kRowTile; ++r) acc[r] = fmaf(wv, so[r * R + l], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < kRowTile; ++r) acc[r] = warp_sum(acc[r]);
    if (lane < nr) {
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < kRowTile; ++r) v = (r == lane) ? acc[r] : v;
        st(out, ((int64_t)(r0 + lane) * H + h) * Dv + j, v);
    }
}

// ---------------------------------------------------------------------------
// decode split: grid (rows, nsplit), 256 threads (8 warps = 8 keys per step).
// Workspace per (row, split): o[R] f32, then (after all o) lse f32, status i32.
// ---------------------------------------------------------------------------
constexpr int kDecWarps = 8;
constexpr int kMaxColsPerThread = 4;  // R <= 1024

template <typename T>
__global__ void __launch_bounds__(kDecWarps * 32) decode_split(
    const T* __restrict__ q_abs, const T* __restrict__ kv, const int32_t* __restrict__ bt,
    const int32_t* __restrict__ seq_lens, int T_q, int H, int R, int P, int max_blocks,
    int num_blocks, float scale, int nsplit, int chunk, float* __restrict__ part_o,
    float* __restrict__ part_lse, int32_t* __restrict__ part_status,
    int32_t* __restrict__ dev_err) {
    extern __shared__ float smem[];
    const int W = R + P;
    float* sq = smem;               // [W]
    float* ss = smem + W;           // [kDecWarps] scores of this step
    __shared__ int s_bad;
    const int64_t row = blockIdx.x;
    const int split = blockIdx.y;
    const int b = (int)(row / ((int64_t)T_q * H));
    const int t = (int)((row / H) % T_q);
    const int S = seq_lens[b];
    int status = 0;
    if (S < 0 || (S > 0 && S < T_q)) status = MLA_DEVERR_SEQ_SHORT;
    else if (S > max_blocks * 16) status = MLA_DEVERR_SEQ_TOO_LONG;
    const int horizon = (status == 0 && S > 0) ? S - T_q + t + 1 : 0;
    const int j0 = split * chunk;
    const int j1 = min(j0 + chunk, horizon);
    if (threadIdx.x == 0) {
        s_bad = 0;
        if (status && split == 0 && dev_err) atomicOr(dev_err, status);
    }
    for (int d = threadIdx.x; d < W; d += blockDim.x) sq[d] = ld(q_abs, row * W + d);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float acc[kMaxColsPerThread];
#pragma unroll
    for (int k = 0; k < kMaxColsPerThread; ++k) acc[k] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int32_t* bt_row = bt + (int64_t)b * max_blocks;

    for (int jb = j0; jb < j1; jb += kDecWarps) {
        // scores: warp w handles key jb + w
        const int j = jb + warp;
        float s = -INFINITY;
        if (j < j1) {
            const int32_t blk = bt_row[j >> 4];
            if (blk < 0 || blk >= num_blocks) {
                if (lane == 0) s_bad = 1;
            } else {
                const T* rowp = kv + ((int64_t)blk * 16 + (j & 15)) * W;
                float d = 0.f;
                for (int c = lane; c < W; c += 32) d = fmaf(sq[c], ld(rowp, c), d);
                s = warp_sum(d) * scale;
            }
        }
        if (lane == 0) ss[warp] = s;
        __syncthreads();
        if (s_bad) break;
        float mx = m;
#pragma unroll
        for (int i = 0; i < kDecWarps; ++i) mx = fmaxf(mx, ss[i]);
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - mx);
        float p[kDecWarps];
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < kDecWarps; ++i) {
            p[i] = (ss[i] == -INFINITY) ? 0.f : expf(ss[i] - mx);
            psum += p[i];
        }
#pragma unroll
        for (int k = 0; k < kMaxColsPerThread; ++k) {
            const int c = threadIdx.x + k * blockDim.x;
            if (c < R) {
                float a = acc[k] * alpha;
#pragma unroll
                for (int i = 0; i < kDecWarps; ++i) {
                    const int jj = jb + i;
                    if (jj < j1) {
                        const int32_t blk = bt_row[jj >> 4];
                        a = fmaf(p[i], ld(kv, ((int64_t)blk * 16 + (jj & 15)) * W + c), a);
                    }
                }
                acc[k] = a;
            }
        }
        l = l * alpha + psum;
        m = mx;
        __syncthreads();
    }
    if (s_bad) {
        status = MLA_DEVERR_BAD_BLOCK;
        if (threadIdx.x == 0 && dev_err) atomicOr(dev_err, status);
        l = 0.f;
    }
    const int64_t slot = row * nsplit + split;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int k = 0; k < kMaxColsPerThread; ++k) {
        const int c = threadIdx.x + k * blockDim.x;
        if (c < R) part_o[slot * R + c] = acc[k] * inv;
    }
    if (threadIdx.x == 0) {
        part_lse[slot] = l > 0.f ? m + logf(l) : -INFINITY;
        part_status[slot] = status;
    }
}

// ---------------------------------------------------------------------------
// combine: grid (rows), 256 threads.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) decode_combine(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      const int32_t* __restrict__ part_status,
                                                      int nsplit, int R, T* __restrict__ out,
                                                      float* __restrict__ lse_out) {
    __shared__ float sw[64];
    __shared__ float s_wsum, s_M;
    __shared__ int s_bad;
    const int64_t row = blockIdx.x;
    if (threadIdx.x == 0) {
        int bad = 0;
        float M = -INFINITY;
        for (int s = 0; s < nsplit; ++s) {
            bad |= part_status[row * nsplit + s];
            M = fmaxf(M, part_lse[row * nsplit + s]);
        }
        float wsum = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float ls = part_lse[row * nsplit + s];
            const float w = (bad || ls == -INFINITY) ? 0.f : expf(ls - M);
            sw[s] = w;
            wsum += w;
        }
        s_bad = bad || M == -INFINITY;
        s_wsum = wsum;
        s_M = M;
    }
    __syncthreads();
    const float inv = s_bad ? 0.f : 1.f / s_wsum;
    for (int c = threadIdx.x; c < R; c += blockDim.x) {
        float a = 0.f;
        if (!s_bad)
            for (int s = 0; s < nsplit; ++s)
                if (sw[s] != 0.f) a = fmaf(sw[s], part_o[(row * nsplit + s) * R + c], a);
        st(out, row * R + c, a * inv);
    }
    if (threadIdx.x == 0 && lse_out) lse_out[row] = s_bad ? -INFINITY : s_M + logf(s_wsum);
}

}  // namespace

SimtDecodePlan simt_decode_plan(int32_t batch, int32_t max_blocks, const mla_dims& d) {
    SimtDecodePlan p;
    const int64_t cap = (int64_t)max_blocks * d.block_size;
    p.nsplit = (int32_t)((cap + 255) / 256);
    if (p.nsplit > 32) p.nsplit = 32;
    if (p.nsplit < 1) p.nsplit = 1;
    int64_t chunk = (cap + p.nsplit - 1) / p.nsplit;
    chunk = (chunk + 15) / 16 * 16;
    p.chunk = (int32_t)(chunk > 0 ? chunk : 16);
    p.rows = (int64_t)batch * d.t_q * d.n_head;
    const int64_t slots = p.rows * p.nsplit;
    size_t o_bytes = (size_t)slots * d.kv_rank * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    size_t l_bytes = ((size_t)slots * sizeof(float) + 255) / 256 * 256;
    p.bytes = o_bytes + l_bytes + (size_t)slots * sizeof(int32_t);
    return p;
}

// the element type of a dtype: f32, bf16 or f16
template <class F>
cudaError_t by_dtype(int32_t dt, F&& f) {
    if (dt == MLA_F32) return f(float{});
    if (dt == MLA_F16) return f(__half{});
    return f(__nv_bfloat16{});
}

cudaError_t launch_absorb_simt(void* q_abs, const void* q_nope, const void* q_pe,
                               const void* w_uk, int32_t rows, const mla_dims& d,
                               cudaStream_t s, const int64_t* positions, float theta_scale) {
    if (rows == 0) return cudaSuccess;
    dim3 grid(d.n_head, (d.kv_rank + 255) / 256, (rows + kRowTile - 1) / kRowTile);
    const size_t smem = (size_t)kRowTile * d.d_nope * sizeof(float);
    return by_dtype(d.dtype, [&](auto t) {
        using T = decltype(t);
        absorb_simt<T><<<grid, 256, smem, s>>>((T*)q_abs, (const T*)q_nope, (const T*)q_pe,
                                                (const T*)w_uk, rows, d.n_head, d.d_nope,
                                                d.d_rope, d.kv_rank, positions, theta_scale);
        return cudaGetLastError();
    });
}

cudaError_t launch_decompress_simt(void* out, const void* o_lat, const void* w_uv,
                                   int32_t rows, const mla_dims& d, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    dim3 grid(d.n_head, (d.d_v + 7) / 8, (rows + kRowTile - 1) / kRowTile);
    const size_t smem = (size_t)kRowTile * d.kv_rank * sizeof(float);
    return by_dtype(d.dtype, [&](auto t) {
        using T = decltype(t);
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(decompress_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        decompress_simt<T><<<grid, 256, smem, s>>>((T*)out, (const T*)o_lat, (const T*)w_uv,
                                                   rows, d.n_head, d.d_v, d.kv_rank);
        return cudaGetLastError();
    });
}

cudaError_t launch_decode_simt(void* out, float* lse, const void* q_abs,
                               const void* kv_cache, const int32_t* block_table,
                               const int32_t* seq_lens, int32_t batch, int32_t max_blocks,
                               int32_t num_blocks, const mla_dims& d, float scale,
                               void* workspace, int32_t* dev_err, cudaStream_t s) {
    const SimtDecodePlan p = simt_decode_plan(batch, max_blocks, d);
    if (p.rows == 0) return cudaSuccess;
    char* ws = (char*)workspace;
    const int64_t slots = p.rows * p.nsplit;
    size_t o_bytes = ((size_t)slots * d.kv_rank * sizeof(float) + 255) / 256 * 256;
    size_t l_bytes = ((size_t)slots * sizeof(float) + 255) / 256 * 256;
    float* part_o = (float*)ws;
    float* part_lse = (float*)(ws + o_bytes);
    int32_t* part_status = (int32_t*)(ws + o_bytes + l_bytes);
    const int W = d.kv_rank + d.d_rope;
    dim3 grid((unsigned)p.rows, p.nsplit);
    const size_t smem = (size_t)(W + kDecWarps) * sizeof(float);
    return by_dtype(d.dtype, [&](auto t) {
        using T = decltype(t);
        decode_split<T><<<grid, kDecWarps * 32, smem, s>>>(
            (const T*)q_abs, (const T*)kv_cache, block_table, seq_lens, d.t_q, d.n_head,
            d.kv_rank, d.d_rope, max_blocks, num_blocks, scale, p.nsplit, p.chunk, part_o,
            part_lse, part_status, dev_err);
        if (cudaError_t e = cudaGetLastError()) return e;
        decode_combine<T><<<(unsigned)p.rows, 256, 0, s>>>(part_o, part_lse, part_status,
                                                           p.nsplit, d.kv_rank, (T*)out, lse);
        return cudaGetLastError();
    });
}

}  // namespace mla
