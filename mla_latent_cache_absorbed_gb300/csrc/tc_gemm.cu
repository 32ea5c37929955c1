// Tensor-core (tcgen05) batched GEMMs of the bf16 path: the W_UK absorb and
// the W_UV decompress ("memra_engine/mla.rs source", fn mla_attend_absorbed,
// absorb and decompress steps). Both are one small GEMM per head,
//   absorb      q_lat[r, n]  = sum_k q_nope[r, h, k] * w_uk[h, k, n]   (K = d_nope)
//   decompress  out[r, j]    = sum_l o_lat[r, h, l]  * w_uv[h, j, l]   (K = kv_rank)
// with few query rows (M = batch * t_q), so they stream the weights: each CTA
// owns one (head, N tile, M tile of 128 rows), brings A and the weight slice
// in 64-wide K chunks through a TMA ring, accumulates in TMEM (M = 128; only
// the tile's real rows are loaded and stored) and converts to bf16 in the
// epilogue. The absorb epilogue also copies q_pe into the rope tail of each
// q_abs row.
//
// Both launch as programmatic dependents of the kernel before them on the
// stream: the weight chunks that fit the ring are requested before waiting
// for that kernel (they depend on nothing it writes); A and every write come
// after the wait.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sm100.cuh"
#include "tc_decode.h"

namespace mla {
namespace {

using namespace sm100;

constexpr int kGThreads = 192;   // warp 0 TMA, 1 MMA, 2-5 epilogue
constexpr int kGStages = 4;
constexpr int kAChunk = 128 * 128;           // A: 128 rows x 64 K (bf16)
constexpr uint64_t kGWaitNs = 2000000000ull;

struct GemmParams {
    __nv_bfloat16* out;          // absorb: q_abs; decompress: out
    const __nv_bfloat16* q_pe;   // absorb only
    int rows, H, K, N;           // N = full output width per head (R or Dv)
    int n_tile;                  // output columns per CTA (<= 256)
    int out_stride;              // elements between consecutive (r, h) rows: W or Dv
    int P;                       // absorb: rope width copied from q_pe
    int a_rows;                  // rows of the A box (the M tile's real rows, multiple of 8)
    int32_t* dev_err;            // optional: timeout bit
};

template <bool kBMnMajor>
__global__ void __launch_bounds__(kGThreads, 1)
    tc_bgemm_kernel(const __grid_constant__ CUtensorMap amap,
                    const __grid_constant__ CUtensorMap bmap, const GemmParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x;
    const int n0 = blockIdx.y * p.n_tile;
    const int m0 = blockIdx.z * 128;
    const int nk = p.K / 64;
    const int bchunk = p.n_tile * 128;  // bytes of one B chunk (n_tile x 64 K)
    const int stage_bytes = kAChunk + bchunk;
    const uint32_t a_bytes = (uint32_t)p.a_rows * 128;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGStages * stage_bytes);
    uint64_t* empty = full + kGStages;
    uint64_t* done = empty + kGStages;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    grid_dependents_launch();  // the next kernel may start its own prologue
    if ((smem_u32(smem) & 1023) != 0) return;
    if (tid == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(done), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (warp == 0) {
        if (elect_one()) {
            tma_prefetch_desc(&amap);
            tma_prefetch_desc(&bmap);
            // weight chunks first (inputs of no earlier kernel), the first ring's
            // worth before waiting for the previous kernel; A after the wait
            auto load_b = [&](int kc) {
                const int s = kc % kGStages;
                unsigned char* st = smem + s * stage_bytes;
                if (kBMnMajor) {
                    // weight [K][N] (N contiguous): n_tile/64 boxes of [64 K rows][64 N]
                    for (int j = 0; j < p.n_tile / 64; ++j)
                        tma_load_3d(smem_u32(st + kAChunk + j * 8192), &bmap,
                                    smem_u32(&full[s]), n0 + j * 64, kc * 64, h);
                } else {
                    // weight [N][K] (K contiguous): one box of [n_tile rows][64 K]
                    tma_load_3d(smem_u32(st + kAChunk), &bmap, smem_u32(&full[s]), kc * 64,
                                n0, h);
                }
            };
            const int early = nk < kGStages ? nk : kGStages;
            for (int kc = 0; kc < early; ++kc) {
                mbar_arrive_expect_tx(smem_u32(&full[kc]), (uint32_t)bchunk + a_bytes);
                load_b(kc);
            }
            grid_dependency_wait();
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kGStages;
                if (kc >= early) {
                    if (!mbar_wait(smem_u32(&empty[s]), ((kc / kGStages) & 1) ^ 1, kGWaitNs)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(smem_u32(&full[s]), (uint32_t)bchunk + a_bytes);
                    load_b(kc);
                }
                // A: the tile's rows m0.. of head h, K columns kc*64..
                tma_load_3d(smem_u32(smem + s * stage_bytes), &amap, smem_u32(&full[s]), kc * 64, h,
                            m0);
            }
        }
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t idesc = idesc_bf16_f32(128, p.n_tile, 0, kBMnMajor ? 1 : 0);
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % kGStages;
                if (!mbar_wait(smem_u32(&full[s]), (kc / kGStages) & 1, kGWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_u32(smem + s * stage_bytes);
                const uint32_t b = a + kAChunk;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd = kBMnMajor ? sdesc_sw128(b + kk * 2048, 8192, 1024)
                                                  : sdesc_sw128(b + kk * 32, 16, 1024);
                    mma_ss(tbase, sdesc_sw128(a + kk * 32, 16, 1024), bd, idesc,
                           (kc | kk) != 0);
                }
                mma_commit(smem_u32(&empty[s]));
            }
            mma_commit(smem_u32(done));
        }
    } else {
        // epilogue: one output row per thread
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int row = m0 + r;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        grid_dependency_wait();  // (writes follow the previous kernel)
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(done), 0, kGWaitNs));
        tc_fence_after();
        if (ok) {
            __nv_bfloat16* dst = p.out + ((long long)row * p.H + h) * p.out_stride + n0;
            for (int cc = 0; cc < p.n_tile; cc += 32) {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + cc, v);
                tmem_wait_ld();
                if (row < p.rows) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        d4[j] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]),
                                                       __uint_as_float(v[8 * j + 1])),
                                           pack_bf16x2(__uint_as_float(v[8 * j + 2]),
                                                       __uint_as_float(v[8 * j + 3])),
                                           pack_bf16x2(__uint_as_float(v[8 * j + 4]),
                                                       __uint_as_float(v[8 * j + 5])),
                                           pack_bf16x2(__uint_as_float(v[8 * j + 6]),
                                                       __uint_as_float(v[8 * j + 7])));
                }
            }
            if (p.P > 0 && blockIdx.y == 0 && row < p.rows) {
                // rope tail of the absorbed query: q_abs[r, h, N:N+P] = q_pe[r, h, :]
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.q_pe + ((long long)row * p.H + h) * p.P);
                uint4* d = reinterpret_cast<uint4*>(
                    p.out + ((long long)row * p.H + h) * p.out_stride + p.N);
                for (int j = 0; j < p.P / 8; ++j) d[j] = src[j];
            }
        }
    }
    if (!ok && tid % 32 == 0 && p.dev_err) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

// 3-D bf16 tensor map with 128-byte swizzle; dims/strides innermost first
cudaError_t make_map(CUtensorMap* m, const void* base, cuuint64_t d0, cuuint64_t d1,
                     cuuint64_t d2, cuuint64_t s1_bytes, cuuint64_t s2_bytes, cuuint32_t b0,
                     cuuint32_t b1, cuuint32_t b2) {
    auto enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

int smem_for(int n_tile) { return kGStages * (kAChunk + n_tile * 128) + 256; }

template <bool kBMnMajor>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                   cudaStream_t s) {
    const int smem = smem_for(p.n_tile);
    static std::once_flag once[2];
    static cudaError_t attr_err[2] = {cudaSuccess, cudaSuccess};
    std::call_once(once[kBMnMajor ? 1 : 0], [&] {
        attr_err[kBMnMajor ? 1 : 0] = cudaFuncSetAttribute(
            tc_bgemm_kernel<kBMnMajor>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            smem_for(256));
    });
    if (attr_err[kBMnMajor ? 1 : 0] != cudaSuccess) return attr_err[kBMnMajor ? 1 : 0];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(p.H, p.N / p.n_tile, (p.rows + 127) / 128);
    cfg.blockDim = dim3(kGThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_bgemm_kernel<kBMnMajor>, a, b, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool tc_gemm_supported(const mla_dims& d, int32_t rows, bool absorb) {
    if (d.dtype != MLA_BF16 || rows <= 0 || d.n_head > 65535) return false;
    if (absorb)
        return d.d_nope % 64 == 0 && d.kv_rank % 256 == 0 && d.d_rope % 8 == 0;
    return d.kv_rank % 64 == 0 && (d.d_v == 128 || d.d_v % 256 == 0);
}

cudaError_t launch_absorb_tc(void* q_abs, const void* q_nope, const void* q_pe,
                             const void* w_uk, int32_t rows, const mla_dims& d,
                             cudaStream_t s) {
    const int H = d.n_head, Dn = d.d_nope, R = d.kv_rank, P = d.d_rope;
    CUtensorMap a, b;
    // A: q_nope viewed as {Dn, H, rows}; box {64, 1, a_rows}
    const int a_rows = rows >= 128 ? 128 : (rows + 7) / 8 * 8;
    cudaError_t e = make_map(&a, q_nope, Dn, H, rows, (cuuint64_t)Dn * 2, (cuuint64_t)H * Dn * 2,
                             64, 1, (cuuint32_t)a_rows);
    if (e != cudaSuccess) return e;
    // B: w_uk viewed as {R, Dn, H} (N contiguous); box {64 N, 64 K, 1}
    e = make_map(&b, w_uk, R, Dn, H, (cuuint64_t)R * 2, (cuuint64_t)Dn * R * 2, 64, 64, 1);
    if (e != cudaSuccess) return e;
    GemmParams p;
    p.out = (__nv_bfloat16*)q_abs;
    p.q_pe = (const __nv_bfloat16*)q_pe;
    p.rows = rows;
    p.H = H;
    p.K = Dn;
    p.N = R;
    p.n_tile = 256;
    p.out_stride = R + P;
    p.P = P;
    p.a_rows = a_rows;
    p.dev_err = nullptr;
    return launch<true>(a, b, p, s);
}

cudaError_t launch_decompress_tc(void* out, const void* o_lat, const void* w_uv, int32_t rows,
                                 const mla_dims& d, cudaStream_t s) {
    const int H = d.n_head, R = d.kv_rank, Dv = d.d_v;
    const int n_tile = Dv == 128 ? 128 : (Dv >= 256 && Dv % 256 == 0 ? 128 : 128);
    CUtensorMap a, b;
    // A: o_lat viewed as {R, H, rows}; box {64, 1, a_rows}
    const int a_rows = rows >= 128 ? 128 : (rows + 7) / 8 * 8;
    cudaError_t e = make_map(&a, o_lat, R, H, rows, (cuuint64_t)R * 2, (cuuint64_t)H * R * 2, 64,
                             1, (cuuint32_t)a_rows);
    if (e != cudaSuccess) return e;
    // B: w_uv viewed as {R, Dv, H} (K contiguous); box {64 K, n_tile N, 1}
    e = make_map(&b, w_uv, R, Dv, H, (cuuint64_t)R * 2, (cuuint64_t)Dv * R * 2, 64,
                 (cuuint32_t)n_tile, 1);
    if (e != cudaSuccess) return e;
    GemmParams p;
    p.out = (__nv_bfloat16*)out;
    p.q_pe = nullptr;
    p.rows = rows;
    p.H = H;
    p.K = R;
    p.N = Dv;
    p.n_tile = n_tile;
    p.out_stride = Dv;
    p.P = 0;
    p.a_rows = a_rows;
    p.dev_err = nullptr;
    return launch<false>(a, b, p, s);
}

}  // namespace mla
