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
#include "tc_split.cuh"

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
    int P;                       // absorb: rope width copied (or roped) from q_pe
    const int64_t* positions;    // absorb: null, or each query row's rope position
    float theta_scale;           // absorb with positions: base^(-2/P)
    int a_rows;                  // rows of the A box (the M tile's real rows, multiple of 8)
    int early;                   // weights may be read before the previous kernel completes
    int ns;                      // ring stages in use: min(kGStages, K / 64), so that a short
                                 // K (the absorb's d_nope) leaves room for 2 CTAs per SM
    int32_t* dev_err;            // optional: timeout bit
};

template <bool kBMnMajor, bool kF16>
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
    const int ns = p.ns;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + ns * stage_bytes);
    uint64_t* empty = full + kGStages;
    uint64_t* done = empty + kGStages;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    grid_dependents_launch();  // the next kernel may start its own prologue
    if ((smem_u32(smem) & 1023) != 0) return;
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
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
            // weight chunks first: in the library's own chain (early) the first
            // ring's worth before waiting for the previous kernel, which does
            // not write them; otherwise only L2 prefetches of them before the
            // wait. A after the wait.
            if (!p.early) {
                for (int kc = 0; kc < nk; ++kc) {
                    if (kBMnMajor) {
                        for (int j = 0; j < p.n_tile / 64; ++j)
                            tma_prefetch_l2_3d(&bmap, n0 + j * 64, kc * 64, h);
                    } else {
                        tma_prefetch_l2_3d(&bmap, kc * 64, n0, h);
                    }
                }
                grid_dependency_wait();
            }
            auto load_b = [&](int kc) {
                const int s = kc % ns;
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
            const int early = nk < ns ? nk : ns;
            for (int kc = 0; kc < early; ++kc) {
                mbar_arrive_expect_tx(smem_u32(&full[kc]), (uint32_t)bchunk + a_bytes);
                load_b(kc);
            }
            grid_dependency_wait();
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % ns;
                if (kc >= early) {
                    if (!mbar_wait(smem_u32(&empty[s]), ((kc / ns) & 1) ^ 1, kGWaitNs)) {
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
            const uint32_t idesc = idesc_f32acc<kF16>(128, p.n_tile, 0, kBMnMajor ? 1 : 0);
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % ns;
                if (!mbar_wait(smem_u32(&full[s]), (kc / ns) & 1, kGWaitNs)) {
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
                        d4[j] = make_uint4(pack2<kF16>(__uint_as_float(v[8 * j]),
                                                       __uint_as_float(v[8 * j + 1])),
                                           pack2<kF16>(__uint_as_float(v[8 * j + 2]),
                                                       __uint_as_float(v[8 * j + 3])),
                                           pack2<kF16>(__uint_as_float(v[8 * j + 4]),
                                                       __uint_as_float(v[8 * j + 5])),
                                           pack2<kF16>(__uint_as_float(v[8 * j + 6]),
                                                       __uint_as_float(v[8 * j + 7])));
                }
            }
            if (p.P > 0 && blockIdx.y == 0 && row < p.rows && !p.positions) {
                // rope tail of the absorbed query: q_abs[r, h, N:N+P] = q_pe[r, h, :]
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.q_pe + ((long long)row * p.H + h) * p.P);
                uint4* d = reinterpret_cast<uint4*>(
                    p.out + ((long long)row * p.H + h) * p.out_stride + p.N);
                for (int j = 0; j < p.P / 8; ++j) d[j] = src[j];
            } else if (p.P > 0 && blockIdx.y == 0 && row < p.rows) {
                // the query's rope at its row's position: NEOX pair (j, j + P/2)
                // turned by theta_j = pos * theta_scale^j (the ratio applied j
                // times, in f32); products rounded before the sum
                // (16-bit elements of the path's type, f16 or bf16)
                const uint16_t* src = reinterpret_cast<const uint16_t*>(p.q_pe) +
                                      ((long long)row * p.H + h) * p.P;
                uint16_t* d = reinterpret_cast<uint16_t*>(p.out) +
                              ((long long)row * p.H + h) * p.out_stride + p.N;
                const int half = p.P / 2;
                float theta = (float)p.positions[row];
                for (int j = 0; j < half; ++j) {
                    float sn, cs;
                    sincosf(theta, &sn, &cs);
                    const float a = elem_lo<kF16>(src[j]), b = elem_lo<kF16>(src[j + half]);
                    const uint32_t pr = pack2<kF16>(__fsub_rn(__fmul_rn(a, cs), __fmul_rn(b, sn)),
                                                    __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cs)));
                    d[j] = (uint16_t)(pr & 0xffffu);
                    d[j + half] = (uint16_t)(pr >> 16);
                    theta = __fmul_rn(theta, p.theta_scale);
                }
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

// 3-D tensor map of 16-bit elements (f16 or bf16) with 128-byte swizzle;
// dims/strides innermost first
cudaError_t make_map(CUtensorMap* m, const void* base, cuuint64_t d0, cuuint64_t d1,
                     cuuint64_t d2, cuuint64_t s1_bytes, cuuint64_t s2_bytes, cuuint32_t b0,
                     cuuint32_t b1, cuuint32_t b2, bool f16) {
    auto enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", (int)r);
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

int smem_for(int n_tile, int ns) { return ns * (kAChunk + n_tile * 128) + 256; }

template <bool kBMnMajor, bool kF16>
cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                   cudaStream_t s) {
    const int smem = smem_for(p.n_tile, p.ns);
    constexpr int kInst = (kBMnMajor ? 1 : 0) + (kF16 ? 2 : 0);
    static std::once_flag once[4];
    static cudaError_t attr_err[4] = {cudaSuccess, cudaSuccess, cudaSuccess, cudaSuccess};
    std::call_once(once[kInst], [&] {
        attr_err[kInst] = cudaFuncSetAttribute(
            tc_bgemm_kernel<kBMnMajor, kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            smem_for(256, kGStages));
    });
    if (attr_err[kInst] != cudaSuccess) return attr_err[kInst];
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, tc_bgemm_kernel<kBMnMajor, kF16>, a, b, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Decompress that merges the split decode's partial rows itself (the fused
// path, mla_attend_absorbed). Same GEMM as the decompress above, but the A
// operand (the latent output rows of head h, K = 512) is built in shared
// memory by the CTA: a row held whole by one pair is copied from o_lat, a row
// of a request split across pairs is merged from the pairs' partial rows with
// the combine's LSE weights (out = sum_k exp(lse_k - lse) o_k), and a row of
// an empty or invalid request is zero. No combine kernel runs in between, and
// the merge overlaps the weight stream.
//
// The CTAs of one head (its d_v / n_tile column tiles, 1 to 4) form a
// cluster and share the merge: each merges every csize-th row and writes it into all of
// their A operands (its own by st.shared, the others' by st.async, counted
// on their A barriers).
//
// Roles: warp 0 streams the weight chunks (3-stage ring), warp 1 issues the
// MMAs once A is complete, warps 2..11 build A, warps 2..5 then run the
// epilogue. Launched as a programmatic dependent of the decode kernel: the
// split shape and the weight stream start before it completes; the partial
// rows, o_lat and every write wait for it.
constexpr int kMThreads = 384;
constexpr int kMStages = 3;
constexpr int kMergeWarps = 10;
constexpr int kMergeLanes = kMergeWarps * 32 / 64;  // rows a merge step covers
constexpr int kMChunks = 8;                 // K = 512 in 64-column chunks

struct MergeParams {
    // the decode's split (fields read by tc_split.cuh)
    const int32_t* seq_lens;
    int B, T, H, max_blocks, NP, min_units;
    const __nv_bfloat16* ws_o;   // partial rows [2 NP][128][512]
    const float* ws_lse;         // [2 NP][128] (NaN: the part met an invalid block id)
    const __nv_bfloat16* o_lat;  // [rows][H][512], rows held whole by one pair
    __nv_bfloat16* out;          // [rows][H][Dv]
    float* lse;                  // [rows][H] or null
    int32_t* dev_err;
    int rows, Dv, n_tile;
};

__device__ __forceinline__ void named_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// One merge step of a thread: piece pc (16 bytes, K chunk pc / 8) of the G
// rows r_g = r0 + step * g (g < G, r_g < mrows), whose parts are loaded KP at
// a time (G * KP loads in flight). Per row, np: 0 empty (zeros), 1 copied from
// o_lat (weight 1), more: the parts' partial rows with the weights in sh_w.
template <int G, int KP, bool kF16>
__device__ __forceinline__ void merge_rows(const MergeParams& p, int h, int m0, int mrows, int r0,
                                           int step, int pc, int np_max, const int* sh_pf,
                                           const int* sh_np, const int* sh_s0, const int* sh_rr,
                                           const float* sh_w, unsigned char* a_smem, int csize,
                                           uint32_t rank, uint32_t aready) {
    // per row: its piece in part k's slot is at base + 2 k * kSlot (k > 0) and
    // base + s0 * kSlot (k = 0); a copied row reads o_lat at base
    constexpr long long kSlot = 128 * 64;  // uint4 per slot
    const uint4* base[G];
    int np[G], s0[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int r = r0 + step * g;
        np[g] = r < mrows ? sh_np[r] : 0;
        s0[g] = r < mrows ? sh_s0[r] : 0;
        base[g] = np[g] == 1
                      ? reinterpret_cast<const uint4*>(p.o_lat + ((long long)(m0 + r) * p.H + h) * 512) + pc
                      : reinterpret_cast<const uint4*>(p.ws_o) +
                            (r < mrows ? (2LL * sh_pf[r] * kSlot + sh_rr[r] * 64) : 0) + pc;
    }
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    for (int k0 = 0; k0 < np_max; k0 += KP) {
        uint4 v[G][KP];
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int kk = 0; kk < KP; ++kk) {
                const int k = k0 + kk;
                if (k < np[g])
                    v[g][kk] = base[g][np[g] == 1 ? 0 : (k == 0 ? s0[g] : 2 * k) * kSlot];
            }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int r = r0 + step * g;
#pragma unroll
            for (int kk = 0; kk < KP; ++kk) {
                const int k = k0 + kk;
                if (k < np[g]) {
                    const float wk = np[g] == 1 ? 1.f : sh_w[r * p.NP + k];
                    const uint32_t x[4] = {v[g][kk].x, v[g][kk].y, v[g][kk].z, v[g][kk].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[g][2 * e] += wk * elem_lo<kF16>(x[e]);
                        acc[g][2 * e + 1] += wk * elem_hi<kF16>(x[e]);
                    }
                }
            }
        }
    }
    const int kc = pc >> 3, u = pc & 7;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int r = r0 + step * g;
        if (r < mrows) {
            const uint32_t x0 = pack2<kF16>(acc[g][0], acc[g][1]), x1 = pack2<kF16>(acc[g][2], acc[g][3]);
            const uint32_t x2 = pack2<kF16>(acc[g][4], acc[g][5]), x3 = pack2<kF16>(acc[g][6], acc[g][7]);
            const uint32_t at = smem_u32(a_smem + kc * 16384 + r * 128 + ((u ^ (r & 7)) << 4));
            st_shared_v4(at, x0, x1, x2, x3);
            // the same A row in the other CTAs of the cluster
            for (int c = 1; c < csize; ++c) {
                const uint32_t dst = (rank + c) % csize;
                st_async_v4(mapa(at, dst), x0, x1, x2, x3, mapa(aready, dst));
            }
        }
    }
}

template <bool kF16>
__global__ void __launch_bounds__(kMThreads, 1)
    tc_decompress_merge_kernel(const __grid_constant__ CUtensorMap bmap, const MergeParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x;
    const int n0 = blockIdx.y * p.n_tile;
    const int m0 = blockIdx.z * 128;
    const int mrows = min(128, p.rows - m0);          // the tile's valid rows
    const int bstage = p.n_tile * 128;                 // one weight chunk [n_tile][64 K]
    unsigned char* a_smem = smem;                      // [8 chunks][128 rows][128 B]
    unsigned char* b_smem = smem + kMChunks * 16384;
    // per row of the tile: its parts (first pair, count, slot offset), its row
    // within the group's partial slots, the LSE-load prefix, the merged LSE,
    // and the parts' weights [128][NP]
    uint64_t* full = reinterpret_cast<uint64_t*>(b_smem + kMStages * bstage);
    int* sh_pf = reinterpret_cast<int*>(full + 2 * kMStages + 2 + 1);
    int* sh_np = sh_pf + 128;     // parts per row: 0 empty, 1 copied from o_lat, >1 merged
    int* sh_s0 = sh_np + 128;
    int* sh_rr = sh_s0 + 128;
    int* sh_off = sh_rr + 128;    // 132 entries: the LSE-load prefix, the largest part count, the others' rows, prefetch
    float* sh_lse = reinterpret_cast<float*>(sh_off + 132);
    float* sh_w = sh_lse + 128;
    uint64_t* empty = full + kMStages;
    uint64_t* aready = empty + kMStages;
    uint64_t* done = aready + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 1);
    grid_dependents_launch();
    if ((smem_u32(smem) & 1023) != 0) return;
    if (tid == 0) {
        for (int s = 0; s < kMStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(aready), 1);
        mbar_init(smem_u32(done), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), 128);
        tmem_relinquish();
    }
    // the cluster's CTAs share one head: each merges every csize-th row and
    // writes it into every CTA's A (barriers initialised cluster-wide first)
    const int csize = (int)(gridDim.y);
    const uint32_t rank = cluster_ctarank();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (warp == 0) {
        // weight chunks [n_tile rows][64 K]: inputs of no kernel of the chain
        if (elect_one()) {
            tma_prefetch_desc(&bmap);
            for (int kc = 0; kc < kMChunks; ++kc) {
                const int s = kc % kMStages;
                if (kc >= kMStages &&
                    !mbar_wait_sleep(smem_u32(&empty[s]), ((kc / kMStages) & 1) ^ 1, kGWaitNs)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&full[s]), (uint32_t)bstage);
                tma_load_3d(smem_u32(b_smem + s * bstage), &bmap, smem_u32(&full[s]), kc * 64, n0, h);
            }
        }
    } else if (warp == 1) {
        if (elect_one()) {
            const uint32_t idesc = idesc_f32acc<kF16>(128, p.n_tile, 0, 0);
            ok = mbar_wait_sleep(smem_u32(aready), 0, kGWaitNs);
            for (int kc = 0; kc < kMChunks && ok; ++kc) {
                const int s = kc % kMStages;
                if (!mbar_wait_sleep(smem_u32(&full[s]), (kc / kMStages) & 1, kGWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_u32(a_smem + kc * 16384);
                const uint32_t b = smem_u32(b_smem + s * bstage);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tbase, sdesc_sw128(a + kk * 32, 16, 1024), sdesc_sw128(b + kk * 32, 16, 1024),
                           idesc, (kc | kk) != 0);
                mma_commit(smem_u32(&empty[s]));
            }
            mma_commit(smem_u32(done));
        }
    } else {
        const int mt = tid - 64;  // the merge threads
        constexpr int kMT = kMergeWarps * 32;
        // 1. the split's shape, and each row's parts (before the decode ends:
        //    seq_lens is an input of the chain, not a result)
        if (warp == 2) {
            const split::SplitShape sh = split::split_shape(p, lane);
            // lane l of a chunk is request b = b0 + l; its rows in the tile are
            // those with grow / T == b (t = grow - b T, query row t H + h)
            int base = 0;
            for (int b0 = 0; b0 < p.B; b0 += 32) {
                const split::ChunkScan c = split::scan_chunk(p, b0, lane);
                const long long b = b0 + lane;
                const int r_lo = (int)max(0LL, b * p.T - m0);
                const int r_hi = (int)min((long long)mrows, (b + 1) * p.T - m0);
                if (b < p.B) {
                    for (int r = r_lo; r < r_hi; ++r) {
                        const int t = (int)(m0 + r - b * p.T);
                        const int qi = t * p.H + h;
                        sh_rr[r] = qi & 127;
                        if (c.v == 0) {
                            sh_np[r] = 0;
                            // invalid requests: reported once (head 0, first N tile, t == 0)
                            if (t == 0 && h == 0 && blockIdx.y == 0 && p.dev_err) {
                                if (c.S < 0 || (c.S > 0 && c.S < p.T))
                                    atomicOr(p.dev_err, (int32_t)MLA_DEVERR_SEQ_SHORT);
                                else if (c.S > p.max_blocks * 16)
                                    atomicOr(p.dev_err, (int32_t)MLA_DEVERR_SEQ_TOO_LONG);
                            }
                        } else {
                            const split::Parts q = split::parts_of(sh, base + c.incl - c.v, c.v, qi >> 7);
                            sh_np[r] = q.nparts;
                            sh_pf[r] = q.pf;
                            sh_s0[r] = q.slot0_off;
                        }
                    }
                }
                base += c.total;
            }
            __syncwarp();
            // prefix of the LSE loads (rows with more than one part)
            if (lane == 0) {
                // over this CTA's own rows (r % csize == rank): the LSE-load
                // prefix and the largest part count; and the rows the other
                // CTAs write into this one's A
                int o = 0, npm = 0, others = 0;
                for (int r = 0; r < mrows; ++r) {
                    sh_off[r] = o;
                    if (r % csize == (int)rank) {
                        o += sh_np[r] > 1 ? sh_np[r] : 0;
                        npm = max(npm, sh_np[r]);
                    } else {
                        ++others;
                    }
                }
                sh_off[mrows] = o;
                sh_off[mrows + 1] = npm;
                sh_off[mrows + 2] = others;
                // a long decode (pairs past 32 tiles) wrote its first partial rows
                // long before it ends: they are prefetched back into L2 below
                sh_off[mrows + 3] = (sh.pooled ? (long long)sh.G * sh.U >
                                                     (long long)split::kAlignedMaxShare * sh.np_all
                                               : sh.U > split::kAlignedMaxShare * sh.np_g)
                                        ? 1
                                        : 0;
            }
        }
        named_sync(1, kMT);
        // the rows this CTA will read (partial rows, copied o_lat rows) into L2
        // while the decode finishes: L2 is the coherence point, so rows the
        // decode writes after their prefetch still read back as written. Only
        // after a long decode: a short one's rows are still in L2, and the
        // prefetches would only delay the merge.
        if (sh_off[mrows + 3]) {
            const int nl0 = sh_off[mrows];
            for (int i = mt; i < nl0; i += kMT) {
                int r = 0;
                while (sh_off[r + 1] <= i) ++r;
                const int k = i - sh_off[r];
                split::Parts q;
                q.pf = sh_pf[r];
                q.slot0_off = sh_s0[r];
                prefetch_l2_bulk(p.ws_o + (split::part_slot(q, k) * 128 + sh_rr[r]) * 512, 1024);
            }
            for (int r = mt; r < mrows; r += kMT)
                if (sh_np[r] == 1 && r % csize == (int)rank)
                    prefetch_l2_bulk(p.o_lat + ((long long)(m0 + r) * p.H + h) * 512, 1024);
        }
        // 2. the decode's results are read from here on
        grid_dependency_wait();
        // 3. the parts' LSEs of the merged rows, all at once, then the weights
        const int nl = sh_off[mrows];
        for (int i = mt; i < nl; i += kMT) {
            int r = 0;
            while (sh_off[r + 1] <= i) ++r;
            const int k = i - sh_off[r];
            split::Parts q;
            q.pf = sh_pf[r];
            q.slot0_off = sh_s0[r];
            sh_w[r * p.NP + k] = p.ws_lse[split::part_slot(q, k) * 128 + sh_rr[r]];
        }
        named_sync(1, kMT);
        // weights: one thread per row (the parts' LSEs are in sh_w); NaN marks a
        // part that met an invalid block id (the row is voided)
        {
            // 8 lanes per row (split::row_weights, as the combine), in
            // warp-uniform rounds of kMT / 8 rows
            constexpr int kGroups = kMT / split::kWeightLanes;
            const int grp = mt / split::kWeightLanes, gl = mt % split::kWeightLanes;
            for (int i0 = 0; i0 * csize < mrows; i0 += kGroups) {
                const int r = (int)rank + csize * (i0 + grp);  // this CTA's rows
                const int np = r < mrows ? sh_np[r] : 0;
                const float l = split::row_weights(sh_w + (r < mrows ? r : 0) * p.NP, np > 1 ? np : 0, gl);
                if (r < mrows && gl == 0) sh_lse[r] = np > 1 ? l : (np == 0 ? -INFINITY : 0.f);
            }
        }
        named_sync(1, kMT);
        // 4. A: thread mt takes the 16-byte piece pc = mt % 64 of rows
        //    mt / 64 + kMergeLanes j, G rows at a time with their parts KP at
        //    a time (G * KP = 16 loads in flight); the CTA picks (G, KP) from
        //    its largest part count
        {
            // this CTA's rows rank + csize (rl + kMergeLanes j)
            const int pc = mt & 63, rl = mt >> 6;
            const int npm = sh_off[mrows + 1];
            const int r0 = (int)rank + csize * rl, step = csize * kMergeLanes;
            const int nsteps = r0 < mrows ? (mrows - r0 + step - 1) / step : 0;
            const uint32_t ab = smem_u32(aready);
            if (npm <= 4) {
                for (int j = 0; j < nsteps; j += 4)
                    merge_rows<4, 4, kF16>(p, h, m0, mrows, r0 + step * j, step, pc, npm, sh_pf, sh_np,
                                     sh_s0, sh_rr, sh_w, a_smem, csize, rank, ab);
            } else if (npm <= 8) {
                for (int j = 0; j < nsteps; j += 2)
                    merge_rows<2, 8, kF16>(p, h, m0, mrows, r0 + step * j, step, pc, npm, sh_pf, sh_np,
                                     sh_s0, sh_rr, sh_w, a_smem, csize, rank, ab);
            } else {
                for (int j = 0; j < nsteps; ++j)
                    merge_rows<1, 16, kF16>(p, h, m0, mrows, r0 + step * j, step, pc, npm, sh_pf, sh_np,
                                      sh_s0, sh_rr, sh_w, a_smem, csize, rank, ab);
            }
        }
        // the merged rows' LSEs (the rows held whole have theirs from the decode)
        if (p.lse)
            for (int r = mt; r < mrows; r += kMT)
                if (sh_np[r] != 1 && r % csize == (int)rank)
                    p.lse[(long long)(m0 + r) * p.H + h] = sh_lse[r];
        fence_proxy_async_smem();  // A is read by the MMA (async proxy)
        named_sync(1, kMT);
        // A is complete once this CTA's rows are written (the arrival below)
        // and the other CTAs' rows have landed (their st.async bytes)
        if (mt == 0) mbar_arrive_expect_tx(smem_u32(aready), (uint32_t)sh_off[mrows + 2] * 1024u);
        // 5. epilogue (warps 2..5): one output row per thread
        if (warp < 6) {
            const int q = warp & 3;
            const int r = q * 32 + lane;
            const int row = m0 + r;
            const uint32_t lane_off = (uint32_t)(q * 32) << 16;
            ok = __all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(done), 0, kGWaitNs));
            tc_fence_after();
            if (ok) {
                __nv_bfloat16* dst = p.out + ((long long)row * p.H + h) * p.Dv + n0;
                for (int cc = 0; cc < p.n_tile; cc += 32) {
                    uint32_t v[32];
                    tmem_ld32(tbase + lane_off + cc, v);
                    tmem_wait_ld();
                    if (row < p.rows) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d4[j] = make_uint4(pack2<kF16>(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                                               pack2<kF16>(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                                               pack2<kF16>(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                                               pack2<kF16>(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
                    }
                }
            }
        }
    }
    if (!ok && tid % 32 == 0 && p.dev_err) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_TIMEOUT);
    tc_fence_before();
    cluster_sync();  // no CTA leaves while another may still write its A
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, 128);
}

size_t merge_smem_bytes(int n_tile, int np) {
    return (size_t)kMChunks * 16384 + (size_t)kMStages * n_tile * 128 +
           (size_t)(2 * kMStages + 3) * 8 + (size_t)(4 * 128 + 132) * 4 + 128 * 4 +
           (size_t)128 * np * 4;
}

}  // namespace

bool tc_gemm_supported(const mla_dims& d, int32_t rows, bool absorb) {
    if ((d.dtype != MLA_BF16 && d.dtype != MLA_F16) || rows <= 0 || d.n_head > 65535)
        return false;
    if (absorb)
        return d.d_nope % 64 == 0 && d.kv_rank % 256 == 0 && d.d_rope % 8 == 0;
    return d.kv_rank % 64 == 0 && (d.d_v == 128 || d.d_v % 256 == 0);
}

cudaError_t launch_absorb_tc(void* q_abs, const void* q_nope, const void* q_pe,
                             const void* w_uk, int32_t rows, const mla_dims& d,
                             cudaStream_t s, bool early, const int64_t* positions,
                             float theta_scale) {
    const int H = d.n_head, Dn = d.d_nope, R = d.kv_rank, P = d.d_rope;
    const bool f16 = d.dtype == MLA_F16;
    CUtensorMap a, b;
    // A: q_nope viewed as {Dn, H, rows}; box {64, 1, a_rows}
    const int a_rows = rows >= 128 ? 128 : (rows + 7) / 8 * 8;
    cudaError_t e = make_map(&a, q_nope, Dn, H, rows, (cuuint64_t)Dn * 2, (cuuint64_t)H * Dn * 2,
                             64, 1, (cuuint32_t)a_rows, f16);
    if (e != cudaSuccess) return e;
    // B: w_uk viewed as {R, Dn, H} (N contiguous); box {64 N, 64 K, 1}
    e = make_map(&b, w_uk, R, Dn, H, (cuuint64_t)R * 2, (cuuint64_t)Dn * R * 2, 64, 64, 1, f16);
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
    p.positions = positions;
    p.theta_scale = theta_scale;
    p.a_rows = a_rows;
    p.early = early ? 1 : 0;
    p.ns = Dn / 64 < kGStages ? Dn / 64 : kGStages;
    p.dev_err = nullptr;
    return f16 ? launch<true, true>(a, b, p, s) : launch<true, false>(a, b, p, s);
}

cudaError_t launch_decompress_tc(void* out, const void* o_lat, const void* w_uv, int32_t rows,
                                 const mla_dims& d, cudaStream_t s, bool early) {
    const int H = d.n_head, R = d.kv_rank, Dv = d.d_v;
    const int n_tile = Dv == 128 ? 128 : (Dv >= 256 && Dv % 256 == 0 ? 128 : 128);
    CUtensorMap a, b;
    // A: o_lat viewed as {R, H, rows}; box {64, 1, a_rows}
    const int a_rows = rows >= 128 ? 128 : (rows + 7) / 8 * 8;
    const bool f16 = d.dtype == MLA_F16;
    cudaError_t e = make_map(&a, o_lat, R, H, rows, (cuuint64_t)R * 2, (cuuint64_t)H * R * 2, 64,
                             1, (cuuint32_t)a_rows, f16);
    if (e != cudaSuccess) return e;
    // B: w_uv viewed as {R, Dv, H} (K contiguous); box {64 K, n_tile N, 1}
    e = make_map(&b, w_uv, R, Dv, H, (cuuint64_t)R * 2, (cuuint64_t)Dv * R * 2, 64,
                 (cuuint32_t)n_tile, 1, f16);
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
    p.positions = nullptr;
    p.theta_scale = 1.f;
    p.a_rows = a_rows;
    p.early = early ? 1 : 0;
    p.ns = R / 64 < kGStages ? R / 64 : kGStages;
    p.dev_err = nullptr;
    return f16 ? launch<false, true>(a, b, p, s) : launch<false, false>(a, b, p, s);
}

// Output columns per CTA of the merging decompress. The CTAs of one head
// (d_v / n_tile of them) form a cluster that shares the merge. A d_v of 128
// is split in two 64-column tiles only while the grid stays one wave (one
// CTA per SM): a second wave costs more than the shared merge saves.
int merge_n_tile(const mla_dims& d, int32_t rows) {
    if (d.d_v != 128) return 128;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 128;
    const long long ctas = 2LL * d.n_head * ((rows + 127) / 128);
    return ctas <= sms ? 64 : 128;
}

bool tc_merge_supported(const mla_dims& d, int32_t rows, int np) {
    return tc_gemm_supported(d, rows, /*absorb=*/false) && d.kv_rank == 512 && d.d_v % 128 == 0 &&
           d.d_v <= 512 && np > 0 && merge_smem_bytes(128, np) + 1024 <= 232448;
}

cudaError_t launch_decompress_merge_tc(void* out, float* lse, const void* o_lat,
                                       const void* w_uv, const int32_t* seq_lens,
                                       int32_t batch, int32_t max_blocks, const mla_dims& d,
                                       const DecodeSplitInfo& info, int32_t* dev_err,
                                       cudaStream_t s) {
    const int H = d.n_head, R = d.kv_rank, Dv = d.d_v;
    const int rows = batch * d.t_q;
    const int n_tile = merge_n_tile(d, rows);
    const bool f16 = d.dtype == MLA_F16;
    CUtensorMap b;
    // B: w_uv viewed as {R, Dv, H} (K contiguous); box {64 K, n_tile N, 1}
    cudaError_t e = make_map(&b, w_uv, R, Dv, H, (cuuint64_t)R * 2, (cuuint64_t)Dv * R * 2, 64,
                             (cuuint32_t)n_tile, 1, f16);
    if (e != cudaSuccess) return e;
    MergeParams p;
    p.seq_lens = seq_lens;
    p.B = batch;
    p.T = d.t_q;
    p.H = H;
    p.max_blocks = max_blocks;
    p.NP = info.NP;
    p.min_units = info.min_units;
    p.ws_o = (const __nv_bfloat16*)info.ws_o;
    p.ws_lse = info.ws_lse;
    p.o_lat = (const __nv_bfloat16*)o_lat;
    p.out = (__nv_bfloat16*)out;
    p.lse = lse;
    p.dev_err = dev_err;
    p.rows = rows;
    p.Dv = Dv;
    p.n_tile = n_tile;
    const size_t smem = merge_smem_bytes(n_tile, info.NP) + 1024;  // + alignment slack
    static std::once_flag once[2];
    static cudaError_t attr_err[2] = {cudaSuccess, cudaSuccess};
    std::call_once(once[f16 ? 1 : 0], [&] {
        attr_err[f16 ? 1 : 0] = f16 ? cudaFuncSetAttribute(tc_decompress_merge_kernel<true>,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           232448)
                                    : cudaFuncSetAttribute(tc_decompress_merge_kernel<false>,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           232448);
    });
    if (attr_err[f16 ? 1 : 0] != cudaSuccess) return attr_err[f16 ? 1 : 0];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;  // the CTAs of one head
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = (unsigned)(Dv / n_tile);
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(H, Dv / n_tile, (rows + 127) / 128);
    cfg.blockDim = dim3(kMThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = f16 ? cudaLaunchKernelEx(&cfg, tc_decompress_merge_kernel<true>, b, p)
            : cudaLaunchKernelEx(&cfg, tc_decompress_merge_kernel<false>, b, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mla
