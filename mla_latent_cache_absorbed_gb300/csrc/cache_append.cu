// Cache append (the vLLM CPU MLA page, CPUMLAImpl.do_kv_cache_update): each
// token's latent row [kv_c | k_pe] is written to its slot of the paged cache,
// cast to the cache's element type; padding slots (< 0) are skipped.
//
// One warp per token: lane 0 reads the slot, the warp copies the row in
// 16-byte pieces (eight bf16 or four f32 elements of the cache row), reading
// the matching source elements and converting them (f32 -> bf16 rounds to
// nearest, ties to even). The work is pure data movement: 2 W e_src bytes in
// and W e_cache bytes out per token.
//
// The fused variant also computes the rows it writes: the key formulas of the
// "aclnnMlaProlog" page, c^KV = RmsNorm(latent) and k^R = ROPE(k_pe), both
// stored in the cache. Same warp per token: the latent row and gamma (from
// L1/L2, shared by all tokens) are held in registers across the warp's sum of
// squares, and lane j rotates the rope pair (j, j + P/2) by theta_j = pos *
// s^j, stepped in f32 from the token's position by the factor s = base^(-2/P)
// as the mla.rs page's rope_neox steps it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace mla {
namespace {

constexpr int kAppendWarps = 8;

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// source element e (e < R: kv_c, else k_pe) of token n, as f32
template <bool kSrcBf16>
__device__ __forceinline__ const void* src_row(const void* kv_c, const void* k_pe, int64_t n, int R,
                                               int P, int e, int* off) {
    if (e < R) {
        *off = e;
        return static_cast<const char*>(kv_c) + n * R * (kSrcBf16 ? 2 : 4);
    }
    *off = e - R;
    return static_cast<const char*>(k_pe) + n * P * (kSrcBf16 ? 2 : 4);
}

// kPer (4 or 8) consecutive source elements from element off of a row, as f32
template <bool kSrcBf16, int kPer>
__device__ __forceinline__ void load_piece(const void* row, int off, float* v) {
    if (kSrcBf16) {
        const uint32_t* s = static_cast<const uint32_t*>(row) + off / 2;
        if (kPer == 8) {
            const uint4 x = *reinterpret_cast<const uint4*>(s);
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[2 * k] = bf16_lo(w4[k]);
                v[2 * k + 1] = bf16_hi(w4[k]);
            }
        } else {
            const uint2 x = *reinterpret_cast<const uint2*>(s);
            v[0] = bf16_lo(x.x);
            v[1] = bf16_hi(x.x);
            v[2] = bf16_lo(x.y);
            v[3] = bf16_hi(x.y);
        }
    } else {
        const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(row) + off);
        const float4 a = s[0];
        v[0] = a.x;
        v[1] = a.y;
        v[2] = a.z;
        v[3] = a.w;
        if (kPer == 8) {
            const float4 b = s[1];
            v[4] = b.x;
            v[5] = b.y;
            v[6] = b.z;
            v[7] = b.w;
        }
    }
}

// one 16-byte piece of a cache row (eight bf16 or four f32 elements)
template <bool kDstBf16>
__device__ __forceinline__ void store_piece(char* dst, const float* v) {
    if (kDstBf16)
        *reinterpret_cast<uint4*>(dst) = make_uint4(pack2_bf16(v[0], v[1]), pack2_bf16(v[2], v[3]),
                                                    pack2_bf16(v[4], v[5]), pack2_bf16(v[6], v[7]));
    else
        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

template <bool kSrcBf16>
__device__ __forceinline__ float load_one(const void* row, int i) {
    if (kSrcBf16) return __uint_as_float((uint32_t)static_cast<const uint16_t*>(row)[i] << 16);
    return static_cast<const float*>(row)[i];
}
template <bool kDstBf16>
__device__ __forceinline__ void store_one(char* row, int i, float v) {
    if (kDstBf16)
        reinterpret_cast<__nv_bfloat16*>(row)[i] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(row)[i] = v;
}

// the token's slot, or -1 when it writes nothing (padding, or a slot past the
// cache, which is reported)
__device__ __forceinline__ int64_t token_slot(const int64_t* slots, int64_t n, long long num_slots,
                                              int lane, int32_t* dev_err) {
    const int64_t slot = slots[n];
    if (slot < 0) return -1;  // padding
    if (slot >= num_slots) {
        if (lane == 0 && dev_err) atomicOr(dev_err, (int32_t)MLA_DEVERR_BAD_SLOT);
        return -1;
    }
    return slot;
}

template <bool kSrcBf16, bool kDstBf16>
__global__ void __launch_bounds__(kAppendWarps * 32)
    cache_append_kernel(void* cache, const void* kv_c, const void* k_pe, const int64_t* slots,
                        int n_tokens, long long num_slots, int R, int P, int32_t* dev_err) {
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (n >= n_tokens) return;
    const int64_t slot = token_slot(slots, n, num_slots, lane, dev_err);
    if (slot < 0) return;
    const int W = R + P;
    constexpr int kPer = kDstBf16 ? 8 : 4;  // cache elements per 16-byte piece
    char* dst_row = static_cast<char*>(cache) + slot * W * (kDstBf16 ? 2 : 4);
    for (int e = lane * kPer; e < W; e += 32 * kPer) {
        int off;
        const void* src = src_row<kSrcBf16>(kv_c, k_pe, n, R, P, e, &off);
        float v[kPer];
        load_piece<kSrcBf16, kPer>(src, off, v);
        store_piece<kDstBf16>(dst_row + e * (kDstBf16 ? 2 : 4), v);
    }
}

// Fused: row = [gamma * kv_c / RMS(kv_c) | NEOX rope of k_pe at positions[n]].
// kPieces 16-byte pieces of the latent row per lane (R <= 32 kPer kPieces):
// every input of the token is loaded before any arithmetic, the latent row and
// gamma stay in registers, and only the stores wait for the slot.
template <bool kSrcBf16, bool kDstBf16, int kPieces>
__global__ void __launch_bounds__(kAppendWarps * 32)
    cache_append_rmsnorm_rope_kernel(void* cache, const void* kv_c, const void* k_pe,
                                     const void* gamma, const int64_t* positions,
                                     const int64_t* slots, int n_tokens, long long num_slots,
                                     int R, int P, float eps, float theta_scale,
                                     int32_t* dev_err) {
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (n >= n_tokens) return;
    constexpr int kPer = kDstBf16 ? 8 : 4;
    constexpr int kSrcB = kSrcBf16 ? 2 : 4, kDstB = kDstBf16 ? 2 : 4;
    const char* x_row = static_cast<const char*>(kv_c) + n * R * kSrcB;
    const char* pe_row = static_cast<const char*>(k_pe) + n * P * kSrcB;
    const int half = P / 2;

    const int64_t slot_in = slots[n];
    const int64_t pos_in = P > 0 ? positions[n] : 0;
    float x[kPieces][kPer], g[kPieces][kPer];
#pragma unroll
    for (int k = 0; k < kPieces; ++k) {
        const int e = (k * 32 + lane) * kPer;
        if (e < R) {
            load_piece<kSrcBf16, kPer>(x_row, e, x[k]);
            load_piece<kSrcBf16, kPer>(gamma, e, g[k]);
        }
    }
    float a0 = 0.f, b0 = 0.f;  // the lane's first rope pair
    if (lane < half) {
        a0 = load_one<kSrcBf16>(pe_row, lane);
        b0 = load_one<kSrcBf16>(pe_row, lane + half);
    }

    // RMS(x) = sqrt(mean(x^2) + eps): lane partial sums, then the warp's butterfly
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < kPieces; ++k)
        if ((k * 32 + lane) * kPer < R) {
#pragma unroll
            for (int i = 0; i < kPer; ++i) ss = fmaf(x[k][i], x[k][i], ss);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv_rms = 1.0f / sqrtf(ss / (float)R + eps);

    if (slot_in < 0) return;  // padding
    if (slot_in >= num_slots) {
        if (lane == 0 && dev_err) atomicOr(dev_err, (int32_t)MLA_DEVERR_BAD_SLOT);
        return;
    }
    char* dst_row = static_cast<char*>(cache) + slot_in * (R + P) * kDstB;
#pragma unroll
    for (int k = 0; k < kPieces; ++k) {
        const int e = (k * 32 + lane) * kPer;
        if (e < R) {
            float v[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) v[i] = g[k][i] * (x[k][i] * inv_rms);
            store_piece<kDstBf16>(dst_row + e * kDstB, v);
        }
    }

    const float pos = (float)pos_in;
    char* dst_pe = dst_row + R * kDstB;
    for (int j = lane; j < half; j += 32) {
        float theta = pos;
        for (int k = 0; k < j; ++k) theta = __fmul_rn(theta, theta_scale);
        float sn, cs;
        sincosf(theta, &sn, &cs);
        const float a = j == lane ? a0 : load_one<kSrcBf16>(pe_row, j);
        const float b = j == lane ? b0 : load_one<kSrcBf16>(pe_row, j + half);
        // products rounded before the sum, as the rotation is written
        store_one<kDstBf16>(dst_pe, j, __fsub_rn(__fmul_rn(a, cs), __fmul_rn(b, sn)));
        store_one<kDstBf16>(dst_pe, j + half, __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cs)));
    }
}

}  // namespace

cudaError_t launch_cache_append(void* cache, const void* kv_c, const void* k_pe,
                                const int64_t* slots, int32_t n_tokens, int32_t num_blocks,
                                int32_t src_dtype, const mla_dims& d, int32_t* dev_err,
                                cudaStream_t s) {
    const long long num_slots = (long long)num_blocks * d.block_size;
    const unsigned grid = (unsigned)((n_tokens + kAppendWarps - 1) / kAppendWarps);
    const bool sb = src_dtype == MLA_BF16, db = d.dtype == MLA_BF16;
    const int R = d.kv_rank, P = d.d_rope;
    if (sb && db)
        cache_append_kernel<true, true><<<grid, kAppendWarps * 32, 0, s>>>(cache, kv_c, k_pe, slots, n_tokens, num_slots, R, P, dev_err);
    else if (sb)
        cache_append_kernel<true, false><<<grid, kAppendWarps * 32, 0, s>>>(cache, kv_c, k_pe, slots, n_tokens, num_slots, R, P, dev_err);
    else if (db)
        cache_append_kernel<false, true><<<grid, kAppendWarps * 32, 0, s>>>(cache, kv_c, k_pe, slots, n_tokens, num_slots, R, P, dev_err);
    else
        cache_append_kernel<false, false><<<grid, kAppendWarps * 32, 0, s>>>(cache, kv_c, k_pe, slots, n_tokens, num_slots, R, P, dev_err);
    return cudaGetLastError();
}

cudaError_t launch_cache_append_rmsnorm_rope(void* cache, const void* kv_c, const void* k_pe,
                                             const void* gamma, const int64_t* positions,
                                             const int64_t* slots, int32_t n_tokens,
                                             int32_t num_blocks, int32_t src_dtype, float eps,
                                             float theta_scale, const mla_dims& d,
                                             int32_t* dev_err, cudaStream_t s) {
    const long long num_slots = (long long)num_blocks * d.block_size;
    const unsigned grid = (unsigned)((n_tokens + kAppendWarps - 1) / kAppendWarps);
    const bool sb = src_dtype == MLA_BF16, db = d.dtype == MLA_BF16;
    const int R = d.kv_rank, P = d.d_rope;
    // pieces per lane: R <= 1024 (the geometry limit) fits 4 bf16 or 8 f32 pieces
    const int per_lane = (R + 32 * (db ? 8 : 4) - 1) / (32 * (db ? 8 : 4));
#define MLA_APPEND_FUSED(SB, DB, NP)                                                             \
    cache_append_rmsnorm_rope_kernel<SB, DB, NP><<<grid, kAppendWarps * 32, 0, s>>>(             \
        cache, kv_c, k_pe, gamma, positions, slots, n_tokens, num_slots, R, P, eps, theta_scale, \
        dev_err)
    if (per_lane > (db ? 4 : 8)) return cudaErrorInvalidValue;
    if (sb && db) {
        if (per_lane <= 2) MLA_APPEND_FUSED(true, true, 2);
        else MLA_APPEND_FUSED(true, true, 4);
    } else if (db) {
        if (per_lane <= 2) MLA_APPEND_FUSED(false, true, 2);
        else MLA_APPEND_FUSED(false, true, 4);
    } else if (sb) {
        if (per_lane <= 4) MLA_APPEND_FUSED(true, false, 4);
        else MLA_APPEND_FUSED(true, false, 8);
    } else {
        if (per_lane <= 4) MLA_APPEND_FUSED(false, false, 4);
        else MLA_APPEND_FUSED(false, false, 8);
    }
#undef MLA_APPEND_FUSED
    return cudaGetLastError();
}

}  // namespace mla
