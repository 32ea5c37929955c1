// Cache append (the vLLM CPU MLA page, CPUMLAImpl.do_kv_cache_update): each
// token's latent row [kv_c | k_pe] is written to its slot of the paged cache,
// cast to the cache's element type; padding slots (< 0) are skipped.
//
// One warp per token: lane 0 reads the slot, the warp copies the row in
// 16-byte pieces (eight bf16 or four f32 elements of the cache row), reading
// the matching source elements and converting them (f32 -> bf16 rounds to
// nearest, ties to even). The work is pure data movement: 2 W e_src bytes in
// and W e_cache bytes out per token.
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

template <bool kSrcBf16, bool kDstBf16>
__global__ void __launch_bounds__(kAppendWarps * 32)
    cache_append_kernel(void* cache, const void* kv_c, const void* k_pe, const int64_t* slots,
                        int n_tokens, long long num_slots, int R, int P, int32_t* dev_err) {
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
    if (n >= n_tokens) return;
    const int64_t slot = slots[n];
    if (slot < 0) return;  // padding
    if (slot >= num_slots) {
        if (lane == 0 && dev_err) atomicOr(dev_err, (int32_t)MLA_DEVERR_BAD_SLOT);
        return;
    }
    const int W = R + P;
    constexpr int kPer = kDstBf16 ? 8 : 4;  // cache elements per 16-byte piece
    char* dst_row = static_cast<char*>(cache) + slot * W * (kDstBf16 ? 2 : 4);
    for (int e = lane * kPer; e < W; e += 32 * kPer) {
        int off;
        const char* src = static_cast<const char*>(src_row<kSrcBf16>(kv_c, k_pe, n, R, P, e, &off));
        float v[kPer];
        if (kSrcBf16) {
            const uint32_t* s = reinterpret_cast<const uint32_t*>(src) + off / 2;
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
            const float4* s = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) + off);
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
        if (kDstBf16) {
            *reinterpret_cast<uint4*>(dst_row + e * 2) =
                make_uint4(pack2_bf16(v[0], v[1]), pack2_bf16(v[2], v[3]), pack2_bf16(v[4], v[5]),
                           pack2_bf16(v[6], v[7]));
        } else {
            *reinterpret_cast<float4*>(dst_row + e * 4) = make_float4(v[0], v[1], v[2], v[3]);
        }
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

}  // namespace mla
