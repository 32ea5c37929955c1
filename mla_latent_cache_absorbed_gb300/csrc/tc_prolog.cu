// Query half of the MLA prolog in one kernel ("aclnnMlaProlog", computation
// formulas of the query), from the query's row after the W^DQ down-projection:
//   c^Q = RmsNorm(x W^DQ)            gamma_i x_i / sqrt(mean(x^2) + eps)
//   q^C = c^Q W^UQ                   one head's d_nope columns
//   q^N = q^C W^UK                   the absorb ("memra_engine/mla.rs source",
//                                    fn mla_attend_absorbed, absorb step)
//   q^R = ROPE(c^Q W^QR)             the NEOX rope of mla.rs (rope_neox), at the
//                                    row's position; W^QR's rope columns carry
//                                    the load-time permutation
// and writes the decode's query row q_abs[r][h] = [q^N | q^R].
//
// Tensor-core kernel (bf16 / f16): one CTA per (head, 128 query rows).
//   warp 0      TMA through a 3-stage ring: first the tile's rows of c_q
//               (64 columns a stage) for the norm's sums; then, for the first
//               GEMM, the same rows again with the head's [W^UQ | W^QR]
//               columns; then W^UK[h] for the second GEMM
//   warps 2..5  one query row per thread: the row's sum of squares over the
//               first sweep, then gamma x / RMS(x) in place in each stage of
//               the second (the A operand of the first GEMM, rounded to the
//               path's type); after it, the epilogues
//   warp 1      tcgen05 MMAs (TMEM accumulators) and the TMEM allocation
// GEMM 1: D1 [128 x (Dn + P)] = c^Q [128 x q_rank] . [W^UQ_h | W^QR_h].
// Epilogue 1: q^C (Dn columns of D1) is rounded to the path's type into shared
// memory as the A operand of GEMM 2; the P columns are turned by the rope in
// f32 and stored as the rope tail of q_abs.
// GEMM 2: D2 [128 x 512] = q^C . W^UK[h] in all 512 TMEM columns (D1 is read
// out by then); epilogue 2 stores it as the latent part of q_abs.
// While heads and row tiles leave half the SMs idle, a head is split over a
// CTA pair (a cluster of 2): GEMM 1's 64-column blocks (W^UQ's, then W^QR's)
// go half to each CTA, all rope columns to CTA 1; each CTA writes its q^C
// columns into both CTAs' GEMM 2 operand (st.async into the partner's), and
// computes one 256-column half of the latent part.
//
// A SIMT kernel serves f32 and the geometries the tensor-core kernel does not
// (one CTA per (head, query row)), rounding at the same points.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kPThreads = 192;
// Shared memory (worked out at launch from the tile's rows, rounded to 8):
//   ns ring stages, each [A: the tile's rows x 64 columns | B: 32 KB]
//   q^C, GEMM 2's A: Dn / 64 chunks of the tile's rows x 64 columns
//   barriers, then gamma
// A tile of fewer than 128 rows keeps only its rows; the MMAs (M = 128) then
// read the memory after them as the rows past the tile, whose results are
// never used, and the ring gets more stages: more weight bytes in flight.
constexpr int kPAFull = 128 * 128;           // A of a full tile: 128 rows x 64 columns, 16-bit
constexpr int kPBChunk = 256 * 128;          // B: up to 256 output columns x 64 K
constexpr int kPMaxStages = 6;
constexpr int kPMaxDn = 256;
constexpr int kPMaxQRank = 8192;
constexpr int kPSmemMax = 232448 - 1024;     // with the alignment slack
constexpr int kPBarBytes = 1024;             // barriers and the TMEM slot, then 1/RMS of 128 rows
constexpr int kPInvOff = 512;
static_assert((5 * kPMaxStages + 3) * 8 + 4 <= kPInvOff && kPInvOff + 128 * 4 <= kPBarBytes,
              "barrier area");
constexpr uint64_t kPWaitNs = 2000000000ull;

struct PrologParams {
    const uint16_t* cq;         // [rows][q_rank], 16-bit elements
    const uint16_t* gamma;      // [q_rank]
    uint16_t* q_abs;            // [rows][H][R + P]
    const int64_t* positions;   // [rows] (P > 0)
    int rows, q_rank, H, Dn, P, R;
    int a_rows;                 // rows of the c_q box: the tile's rows, rounded up to 8
    int ns, stage, areg;        // ring stages, bytes per stage, bytes of its A part
    int a2, a2s, bar, gam;      // offsets of q^C, its chunk stride, barriers, gamma
    int split;                  // a head split over a CTA pair (cluster of 2)
    int ab1;                    // split: the first of GEMM 1's 64-column blocks CTA 1 takes
    float eps, theta_scale;
    int32_t* dev_err;
};

template <bool kF16>
__device__ __forceinline__ float to_f32(uint32_t bits16) {
    return elem_lo<kF16>(bits16);
}

template <bool kF16>
__global__ void __launch_bounds__(kPThreads, 1)
    tc_prolog_q_kernel(const __grid_constant__ CUtensorMap cqmap,
                       const __grid_constant__ CUtensorMap uqmap,
                       const __grid_constant__ CUtensorMap qrmap,
                       const __grid_constant__ CUtensorMap ukmap, const PrologParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled operands need a 1 KB-aligned base
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int ns = p.ns;
    uint64_t* fullA = reinterpret_cast<uint64_t*>(smem + p.bar);  // row threads (128)
    uint64_t* fullB = fullA + kPMaxStages;                        // TMA bytes (1): c_q + weights
    uint64_t* empty = fullB + kPMaxStages;                        // MMA commit (1)
    uint64_t* d1done = empty + ns;
    uint64_t* a2ready = d1done + 1;
    uint64_t* d2done = a2ready + 1;
    uint64_t* ssfull = d2done + 1;          // first sweep: c_q chunk landed (TMA bytes)
    uint64_t* ssfree = ssfull + kPMaxStages;  // first sweep: chunk read (row threads, 128)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(ssfree + kPMaxStages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = p.split ? cluster_ctarank() : 0u;
    const int h = p.split ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int m0 = blockIdx.y * 128;
    const int nuq = p.Dn / 64;           // GEMM 1's 64-column blocks of W^UQ; W^QR's follow
    const int nat = (p.Dn + p.P) / 64;
    const int ab = crank == 0 ? 0 : p.ab1;                    // this CTA's blocks [ab, ae)
    const int ae = (p.split && crank == 0) ? p.ab1 : nat;
    const int N1 = 64 * (ae - ab);       // GEMM 1 output columns of this CTA
    const int qc0 = 64 * ab, qc1 = 64 * min(ae, nuq);          // its q^C columns
    const bool rope_here = p.P > 0 && ae == nat;
    const int nk1 = p.q_rank / 64;       // GEMM 1 K chunks
    const int nk2 = p.Dn / 64;           // GEMM 2 K chunks
    const int nhalf = p.split ? 1 : 2;   // GEMM 2's 256-column halves of this CTA
    const int half0 = p.split ? (int)crank : 0;
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(smem_u32(&fullA[s]), 128);
            mbar_init(smem_u32(&fullB[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(d1done), 1);
        // the row threads' q^C writes, and on a split the partner's (bytes)
        mbar_init(smem_u32(a2ready), p.split ? 129 : 128);
        mbar_init(smem_u32(d2done), 1);
        for (int s = 0; s < ns; ++s) {
            mbar_init(smem_u32(&ssfull[s]), 1);
            mbar_init(smem_u32(&ssfree[s]), 128);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync();  // (a CTA alone is a cluster of one) the partner's barriers are set up
    tc_fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;
    if (p.split && tid == 0) {
        // the partner's q^C columns, a_rows rows of them
        const int pab = crank == 0 ? p.ab1 : 0, pae = crank == 0 ? nat : p.ab1;
        const int pcols = 64 * (min(pae, nuq) - min(pab, nuq));
        mbar_arrive_expect_tx(smem_u32(a2ready), (uint32_t)(p.a_rows * pcols * 2));
    }

    if (warp == 0) {
        // ---------------- weights: GEMM 1 chunks, then GEMM 2 chunks, one ring
        if (elect_one()) {
            tma_prefetch_desc(&cqmap);
            tma_prefetch_desc(&uqmap);
            if (p.P) tma_prefetch_desc(&qrmap);
            tma_prefetch_desc(&ukmap);
            // first sweep: c_q chunks for the norm's sums
            for (int j = 0; j < nk1 && ok; ++j) {
                const int s = j % ns;
                if (j >= ns &&
                    !mbar_wait_sleep(smem_u32(&ssfree[s]), ((j / ns) - 1) & 1, kPWaitNs)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(&ssfull[s]), (uint32_t)(p.a_rows * 128));
                tma_load_2d(smem_u32(smem + s * p.stage), &cqmap, smem_u32(&ssfull[s]), j * 64, m0);
            }
            // each stage's last use in the first sweep must be read before the
            // second sweep refills it
            for (int s = 0; s < ns && s < nk1 && ok; ++s) {
                const int jl = s + ((nk1 - 1 - s) / ns) * ns;  // last chunk in stage s
                if (!mbar_wait_sleep(smem_u32(&ssfree[s]), (jl / ns) & 1, kPWaitNs)) ok = false;
            }
            const int nload = nk1 + nhalf * nk2;
            for (int j = 0; j < nload && ok; ++j) {
                const int s = j % ns;
                if (!mbar_wait_sleep(smem_u32(&empty[s]), ((j / ns) & 1) ^ 1, kPWaitNs)) {
                    ok = false;
                    break;
                }
                unsigned char* b = smem + s * p.stage + p.areg;
                if (j < nk1) {
                    // the tile's rows of c_q, columns 64 j .. +63 (rows past the
                    // batch read as zeros), then [64 K rows][64 N] boxes: W^UQ's Dn
                    // columns of head h and W^QR's P
                    mbar_arrive_expect_tx(smem_u32(&fullB[s]), (uint32_t)(p.a_rows * 128 + N1 * 128));
                    tma_load_2d(smem_u32(smem + s * p.stage), &cqmap, smem_u32(&fullB[s]), j * 64, m0);
                    for (int a = ab; a < ae; ++a) {
                        if (a < nuq)
                            tma_load_2d(smem_u32(b + (a - ab) * 8192), &uqmap, smem_u32(&fullB[s]),
                                        h * p.Dn + a * 64, j * 64);
                        else
                            tma_load_2d(smem_u32(b + (a - ab) * 8192), &qrmap, smem_u32(&fullB[s]),
                                        h * p.P + (a - nuq) * 64, j * 64);
                    }
                } else {
                    // W^UK[h] rows 64 kc .. +63, columns 256 half .. +255
                    const int t = j - nk1;
                    const int kc = nhalf == 2 ? t >> 1 : t, half = nhalf == 2 ? t & 1 : half0;
                    mbar_arrive_expect_tx(smem_u32(&fullB[s]), 256u * 128u);
                    for (int c = 0; c < 4; ++c)
                        tma_load_3d(smem_u32(b + c * 8192), &ukmap, smem_u32(&fullB[s]),
                                    half * 256 + c * 64, kc * 64, h);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMAs
        if (elect_one()) {
            const uint32_t idesc1 = idesc_f32acc<kF16>(128, N1, 0, 1);
            constexpr uint32_t idesc2 = idesc_f32acc<kF16>(128, 256, 0, 1);
            for (int j = 0; j < nk1; ++j) {
                const int s = j % ns;
                const uint32_t par = (j / ns) & 1;
                if (!mbar_wait(smem_u32(&fullB[s]), par, kPWaitNs) ||
                    !mbar_wait(smem_u32(&fullA[s]), par, kPWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_u32(smem + s * p.stage);
                const uint32_t b = a + p.areg;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tbase, sdesc_sw128(a + kk * 32, 16, 1024),
                           sdesc_sw128(b + kk * 2048, 8192, 1024), idesc1, (j | kk) != 0);
                mma_commit(smem_u32(&empty[s]));
            }
            mma_commit(smem_u32(d1done));
            // GEMM 2 once epilogue 1 has read D1 and written q^C
            if (ok && mbar_wait_sleep(smem_u32(a2ready), 0, kPWaitNs)) {
                fence_proxy_async_smem();  // the partner's q^C columns came by st.async
                tc_fence_after();
                for (int t = 0; t < nhalf * nk2; ++t) {
                    const int j = nk1 + t, s = j % ns;
                    const int kc = nhalf == 2 ? t >> 1 : t, half = nhalf == 2 ? t & 1 : 0;
                    if (!mbar_wait(smem_u32(&fullB[s]), (j / ns) & 1, kPWaitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(smem + p.a2 + kc * p.a2s);
                    const uint32_t b = smem_u32(smem + s * p.stage + p.areg);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(tbase + half * 256, sdesc_sw128(a + kk * 32, 16, 1024),
                               sdesc_sw128(b + kk * 2048, 8192, 1024), idesc2, (kc | kk) != 0);
                    mma_commit(smem_u32(&empty[s]));
                }
            } else {
                ok = false;
            }
            mma_commit(smem_u32(d2done));
        }
    } else {
        // ---------------- row threads: row r = 32 (warp % 4) + lane of the tile
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int row = m0 + r;
        const bool valid = row < p.rows;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        // gamma into shared memory once (the 128 row threads; read back after
        // the first sweep)
        const uint32_t gsm = smem_u32(smem + p.gam);
        const bool in_box = r < p.a_rows;  // the row has its place in the stages and in q^C
        for (int i = q * 32 + lane; i < p.q_rank / 8; i += 128) {
            const uint4 g = reinterpret_cast<const uint4*>(p.gamma)[i];
            st_shared_v4(gsm + i * 16, g.x, g.y, g.z, g.w);
        }
        // The sweeps take the stage's 16-byte pieces as work items: thread rt
        // of the 128 handles piece rt % 8 of rows rt / 8 + 16 k, so that every
        // row's eight pieces sit in eight lanes of one warp and a tile of few
        // rows still spreads over many threads; each thread issues all its
        // loads of a stage before it uses them.
        const int rt = (warp - 2) * 32 + lane;
        const int pc = rt & 7, g16 = rt >> 3;
        float* inv_sh = reinterpret_cast<float*>(smem + p.bar + kPInvOff);
        // 1. each row's sum of squares over the first sweep (f32; the row's
        //    pieces summed in order of their columns, then across the pieces)
        float ssk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ssk[k] = 0.f;
        for (int j = 0; j < nk1; ++j) {
            const int s = j % ns;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&ssfull[s]), (j / ns) & 1, kPWaitNs))) {
                ok = false;
                break;
            }
            const uint32_t st = smem_u32(smem + s * p.stage);
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = g16 + 16 * k;
                v[k] = rr < p.a_rows ? ld_shared_v4(st + rr * 128 + ((pc ^ (rr & 7)) << 4))
                                     : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = elem_lo<kF16>(u[e]), b = elem_hi<kF16>(u[e]);
                    ssk[k] = fmaf(a, a, ssk[k]);
                    ssk[k] = fmaf(b, b, ssk[k]);
                }
            }
            mbar_arrive(smem_u32(&ssfree[s]));
        }
        // each row's norm factor 1 / RMS (zero for rows past the batch)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float t = ssk[k];
            t += __shfl_xor_sync(0xffffffffu, t, 1);
            t += __shfl_xor_sync(0xffffffffu, t, 2);
            t += __shfl_xor_sync(0xffffffffu, t, 4);
            const int rr = g16 + 16 * k;
            if (pc == 0) inv_sh[rr] = (m0 + rr < p.rows) ? 1.0f / sqrtf(t / (float)p.q_rank + p.eps) : 0.f;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");  // gamma and 1/RMS are in shared memory
        float invk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) invk[k] = inv_sh[g16 + 16 * k];
        // 2. the A operand of GEMM 1, gamma x / RMS, in place in each stage of
        //    the second sweep as it lands (rows past the box are not touched:
        //    the MMA reads whatever follows them, and those rows are never stored)
        for (int j = 0; j < nk1 && ok; ++j) {
            const int s = j % ns;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(smem_u32(&fullB[s]), (j / ns) & 1, kPWaitNs))) {
                ok = false;
                break;
            }
            const uint32_t st = smem_u32(smem + s * p.stage);
            const uint4 gv = ld_shared_v4(gsm + (j * 8 + pc) * 16);
            const uint32_t gu[4] = {gv.x, gv.y, gv.z, gv.w};
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = g16 + 16 * k;
                v[k] = rr < p.a_rows ? ld_shared_v4(st + rr * 128 + ((pc ^ (rr & 7)) << 4))
                                     : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = g16 + 16 * k;
                if (rr < p.a_rows) {
                    const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = pack2<kF16>(elem_lo<kF16>(gu[e]) * elem_lo<kF16>(u[e]) * invk[k],
                                           elem_hi<kF16>(gu[e]) * elem_hi<kF16>(u[e]) * invk[k]);
                    st_shared_v4(st + rr * 128 + ((pc ^ (rr & 7)) << 4), o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&fullA[s]));
        }
        // 3. epilogue 1: q^C -> GEMM 2's A; the P columns -> rope -> q_abs tail
        ok = __all_sync(0xffffffffu, ok && mbar_wait_sleep(smem_u32(d1done), 0, kPWaitNs));
        tc_fence_after();
        uint16_t* qrow = p.q_abs + ((long long)(valid ? row : 0) * p.H + h) * (p.R + p.P);
        if (ok) {
            const uint32_t peer_bar = p.split ? mapa(smem_u32(a2ready), crank ^ 1u) : 0u;
            for (int cb = qc0; cb < qc1; cb += 32) {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + (cb - qc0), v);
                tmem_wait_ld();
                const uint32_t chunk = smem_u32(smem + p.a2 + (cb >> 6) * p.a2s) + r * 128;
                if (!in_box) continue;  // (the TMEM load above is warp-wide)
                float f[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]);  // q^C
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c = ((cb & 63) >> 3) + u;  // 16-byte piece within the 128-byte row
                    const uint32_t a = chunk + ((c ^ (r & 7)) << 4);
                    const uint32_t w0 = pack2<kF16>(f[8 * u], f[8 * u + 1]);
                    const uint32_t w1 = pack2<kF16>(f[8 * u + 2], f[8 * u + 3]);
                    const uint32_t w2 = pack2<kF16>(f[8 * u + 4], f[8 * u + 5]);
                    const uint32_t w3 = pack2<kF16>(f[8 * u + 6], f[8 * u + 7]);
                    st_shared_v4(a, w0, w1, w2, w3);
                    if (p.split) st_async_v4(mapa(a, crank ^ 1u), w0, w1, w2, w3, peer_bar);
                }
            }
            if (rope_here) {
                // NEOX pairs (j, j + P/2), theta_j = pos * theta_scale^j (the ratio
                // applied j times in f32), products rounded before the sum
                const int half = p.P / 2;
                float theta = valid ? (float)p.positions[row] : 0.f;
                for (int j0 = 0; j0 < half; j0 += 32) {
                    uint32_t a[32], b[32];
                    tmem_ld32(tbase + lane_off + (p.Dn - qc0) + j0, a);
                    tmem_ld32(tbase + lane_off + (p.Dn - qc0) + half + j0, b);
                    tmem_wait_ld();
                    const int n = min(32, half - j0);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        if (jj >= n) break;
                        float sn, cs;
                        sincosf(theta, &sn, &cs);
                        const float x = __uint_as_float(a[jj]), y = __uint_as_float(b[jj]);
                        const uint32_t pr = pack2<kF16>(__fsub_rn(__fmul_rn(x, cs), __fmul_rn(y, sn)),
                                                        __fadd_rn(__fmul_rn(x, sn), __fmul_rn(y, cs)));
                        if (valid) {
                            qrow[p.R + j0 + jj] = (uint16_t)(pr & 0xffffu);
                            qrow[p.R + half + j0 + jj] = (uint16_t)(pr >> 16);
                        }
                        theta = __fmul_rn(theta, p.theta_scale);
                    }
                }
            }
        }
        fence_proxy_async_smem();  // q^C is read by the MMA (async proxy)
        tc_fence_before();
        mbar_arrive(smem_u32(a2ready));
        // 4. epilogue 2: the latent part
        ok = __all_sync(0xffffffffu, ok && mbar_wait_sleep(smem_u32(d2done), 0, kPWaitNs));
        tc_fence_after();
        if (ok) {
            uint4* dst = reinterpret_cast<uint4*>(qrow) + half0 * 32;  // latent column 256 half0
            for (int cb = 0; cb < 256 * nhalf; cb += 32) {
                uint32_t v[32];
                tmem_ld32(tbase + lane_off + cb, v);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[(cb >> 3) + u] =
                            make_uint4(pack2<kF16>(__uint_as_float(v[8 * u]), __uint_as_float(v[8 * u + 1])),
                                       pack2<kF16>(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                                       pack2<kF16>(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                                       pack2<kF16>(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
                }
            }
        }
    }
    if (!ok && lane == 0 && p.dev_err) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_TIMEOUT);
    tc_fence_before();
    cluster_sync();  // neither CTA of a pair leaves while the other may still write into it
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// SIMT form: one CTA per (head, query row); the same formulas and rounding
// points (c^Q and q^C rounded to T before their products; f32 sums).
template <typename T>
__device__ __forceinline__ float ldx(const T* p, long long i);
template <>
__device__ __forceinline__ float ldx<float>(const float* p, long long i) { return p[i]; }
template <>
__device__ __forceinline__ float ldx<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
    return __bfloat162float(p[i]);
}
template <>
__device__ __forceinline__ float ldx<__half>(const __half* p, long long i) {
    return __half2float(p[i]);
}
template <typename T>
__device__ __forceinline__ T cvt(float v);
template <>
__device__ __forceinline__ float cvt<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }
template <>
__device__ __forceinline__ __half cvt<__half>(float v) { return __float2half_rn(v); }
template <typename T>
__device__ __forceinline__ float round_to(float v) {
    const T t = cvt<T>(v);
    return ldx<T>(&t, 0);
}

template <typename T>
__global__ void __launch_bounds__(256) prolog_q_simt(T* __restrict__ q_abs, const T* __restrict__ cq,
                                                     const T* __restrict__ gamma,
                                                     const T* __restrict__ w_uq,
                                                     const T* __restrict__ w_qr,
                                                     const T* __restrict__ w_uk,
                                                     const int64_t* __restrict__ positions,
                                                     int q_rank, int H, int Dn, int P, int R,
                                                     float eps, float theta_scale) {
    extern __shared__ float sh[];  // c^Q [q_rank], q^C [Dn], q_pe [P], partial sums [8]
    float* cn = sh;
    float* qc = cn + q_rank;
    float* qp = qc + Dn;
    float* red = qp + P;
    const int h = blockIdx.x;
    const long long row = blockIdx.y;
    const int tid = threadIdx.x;
    // RMS of the row
    float ss = 0.f;
    for (int k = tid; k < q_rank; k += blockDim.x) {
        const float x = ldx(cq, row * q_rank + k);
        ss = fmaf(x, x, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        red[0] = 1.0f / sqrtf(t / (float)q_rank + eps);
    }
    __syncthreads();
    const float inv = red[0];
    for (int k = tid; k < q_rank; k += blockDim.x)
        cn[k] = round_to<T>(ldx(gamma, k) * ldx(cq, row * q_rank + k) * inv);
    __syncthreads();
    // q^C and the rope part before the rope: one output column per thread
    for (int d = tid; d < Dn + P; d += blockDim.x) {
        float acc = 0.f;
        if (d < Dn) {
            for (int k = 0; k < q_rank; ++k) acc = fmaf(cn[k], ldx(w_uq, (long long)k * H * Dn + h * Dn + d), acc);
            qc[d] = round_to<T>(acc);
        } else {
            const int j = d - Dn;
            for (int k = 0; k < q_rank; ++k) acc = fmaf(cn[k], ldx(w_qr, (long long)k * H * P + h * P + j), acc);
            qp[j] = acc;
        }
    }
    __syncthreads();
    T* dst = q_abs + (row * H + h) * (R + P);
    for (int l = tid; l < R; l += blockDim.x) {
        float acc = 0.f;
        for (int d = 0; d < Dn; ++d) acc = fmaf(qc[d], ldx(w_uk, ((long long)h * Dn + d) * R + l), acc);
        dst[l] = cvt<T>(acc);
    }
    if (tid == 0 && P > 0) {
        const int half = P / 2;
        float theta = (float)positions[row];
        for (int j = 0; j < half; ++j) {
            float sn, cs;
            sincosf(theta, &sn, &cs);
            const float x = qp[j], y = qp[j + half];
            dst[R + j] = cvt<T>(__fsub_rn(__fmul_rn(x, cs), __fmul_rn(y, sn)));
            dst[R + half + j] = cvt<T>(__fadd_rn(__fmul_rn(x, sn), __fmul_rn(y, cs)));
            theta = __fmul_rn(theta, theta_scale);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 prolog_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

// tensor map of 16-bit elements, 128-byte swizzle, boxes {64, 64(, 1)}
cudaError_t prolog_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, bool f16) {
    auto enc = prolog_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     rank, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (prolog weights) failed (%d)", (int)r);
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

}  // namespace

bool tc_prolog_supported(const mla_dims& d, int32_t q_rank) {
    return d.dtype != MLA_F32 && d.kv_rank == 512 && d.d_nope % 64 == 0 && d.d_rope % 64 == 0 &&
           d.d_nope + d.d_rope <= 256 && d.d_nope <= kPMaxDn && q_rank % 64 == 0 && q_rank > 0 &&
           q_rank <= kPMaxQRank &&
           d.n_head <= 65535;
}

cudaError_t launch_prolog_q(void* q_abs, const void* c_q, const void* gamma_q, const void* w_uq,
                            const void* w_qr, const void* w_uk, const int64_t* positions,
                            int32_t rows, int32_t q_rank, float eps, float theta_scale,
                            const mla_dims& d, int32_t* dev_err, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    const int H = d.n_head, Dn = d.d_nope, P = d.d_rope, R = d.kv_rank;
    if (tc_prolog_supported(d, q_rank)) {
        const bool f16 = d.dtype == MLA_F16;
        CUtensorMap cqm, uq, qr, uk;
        {
            // c_q [rows][q_rank]: {q_rank, rows}, boxes of 64 columns x 128 rows
            cuuint64_t dims[2] = {(cuuint64_t)q_rank, (cuuint64_t)rows};
            cuuint64_t str[1] = {(cuuint64_t)q_rank * 2};
            cuuint32_t box[2] = {64, (cuuint32_t)(rows >= 128 ? 128 : (rows + 7) / 8 * 8)};
            if (cudaError_t e = prolog_map(&cqm, c_q, 2, dims, str, box, f16)) return e;
        }
        {
            // W^UQ [q_rank][H * Dn]: {H * Dn, q_rank}, boxes of 64 columns x 64 rows
            cuuint64_t dims[2] = {(cuuint64_t)H * Dn, (cuuint64_t)q_rank};
            cuuint64_t str[1] = {(cuuint64_t)H * Dn * 2};
            cuuint32_t box[2] = {64, 64};
            if (cudaError_t e = prolog_map(&uq, w_uq, 2, dims, str, box, f16)) return e;
        }
        if (P > 0) {
            cuuint64_t dims[2] = {(cuuint64_t)H * P, (cuuint64_t)q_rank};
            cuuint64_t str[1] = {(cuuint64_t)H * P * 2};
            cuuint32_t box[2] = {64, 64};
            if (cudaError_t e = prolog_map(&qr, w_qr, 2, dims, str, box, f16)) return e;
        } else {
            qr = uq;  // unused
        }
        {
            // W^UK [H][Dn][R]: {R, Dn, H}
            cuuint64_t dims[3] = {(cuuint64_t)R, (cuuint64_t)Dn, (cuuint64_t)H};
            cuuint64_t str[2] = {(cuuint64_t)R * 2, (cuuint64_t)Dn * R * 2};
            cuuint32_t box[3] = {64, 64, 1};
            if (cudaError_t e = prolog_map(&uk, w_uk, 3, dims, str, box, f16)) return e;
        }
        PrologParams p;
        p.cq = (const uint16_t*)c_q;
        p.gamma = (const uint16_t*)gamma_q;
        p.q_abs = (uint16_t*)q_abs;
        p.positions = positions;
        p.rows = rows;
        p.q_rank = q_rank;
        p.H = H;
        p.Dn = Dn;
        p.P = P;
        p.R = R;
        p.a_rows = rows >= 128 ? 128 : (rows + 7) / 8 * 8;
        {
            // the layout above: A parts and q^C chunks of the tile's rows
            // (whole 8-row groups), the ring as deep as the rest allows
            const int areg = (p.a_rows * 128 + 1023) / 1024 * 1024;
            p.areg = areg;
            p.stage = areg + kPBChunk;
            const int nk2 = Dn / 64;
            const int a2_bytes = nk2 * areg + (kPAFull - areg);  // the last chunk's MMA reads 16 KB
            const int tail = a2_bytes + kPBarBytes + q_rank * 2;
            int ns = (kPSmemMax - tail) / p.stage;
            ns = ns > kPMaxStages ? kPMaxStages : ns;
            if (ns < 2) {
                set_error("mla_prolog_q: shared memory for the ring does not fit");
                return cudaErrorInvalidValue;
            }
            p.ns = ns;
            p.a2 = ns * p.stage;
            p.a2s = areg;
            p.bar = p.a2 + a2_bytes;
            p.gam = p.bar + kPBarBytes;
        }
        p.eps = eps;
        p.theta_scale = theta_scale;
        p.dev_err = dev_err;
        // a head over a CTA pair while the pairs of all heads and row tiles fit
        // the SMs in one wave: GEMM 1's blocks halved (rounded up to CTA 0), all
        // of W^QR's with CTA 1
        const int tiles = (rows + 127) / 128;
        {
            int dev = 0, sms = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                sms = 0;
            const int nuq = Dn / 64, nat = (Dn + P) / 64;
            int ab1 = (nat + 1) / 2;
            if (ab1 > nuq) ab1 = nuq;
            p.split = (nat >= 2 && ab1 >= 1 && (long long)H * tiles * 2 <= sms) ? 1 : 0;
            p.ab1 = ab1;
        }
        const int smem = p.gam + q_rank * 2 + 1024;  // + alignment slack
        static std::once_flag once[2];
        static cudaError_t attr_err[2] = {cudaSuccess, cudaSuccess};
        std::call_once(once[f16 ? 1 : 0], [&] {
            attr_err[f16 ? 1 : 0] =
                f16 ? cudaFuncSetAttribute(tc_prolog_q_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kPSmemMax + 1024)
                    : cudaFuncSetAttribute(tc_prolog_q_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kPSmemMax + 1024);
        });
        if (attr_err[f16 ? 1 : 0] != cudaSuccess) return attr_err[f16 ? 1 : 0];
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = p.split ? 2 : 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(H * (p.split ? 2 : 1)), (unsigned)tiles, 1);
        cfg.blockDim = dim3(kPThreads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)smem;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = f16 ? cudaLaunchKernelEx(&cfg, tc_prolog_q_kernel<true>, cqm, uq, qr, uk, p)
                                  : cudaLaunchKernelEx(&cfg, tc_prolog_q_kernel<false>, cqm, uq, qr, uk, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const size_t smem = (size_t)(q_rank + Dn + P + 8) * sizeof(float);
    if (smem > 227 * 1024) {
        set_error("mla_prolog_q: q_rank %d is too large for the SIMT form", q_rank);
        return cudaErrorInvalidValue;
    }
    const dim3 grid((unsigned)H, (unsigned)rows, 1);
    auto run = [&](auto t) {
        using T = decltype(t);
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(prolog_q_simt<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        prolog_q_simt<T><<<grid, 256, smem, s>>>((T*)q_abs, (const T*)c_q, (const T*)gamma_q,
                                                 (const T*)w_uq, (const T*)w_qr, (const T*)w_uk,
                                                 positions, q_rank, H, Dn, P, R, eps, theta_scale);
        return cudaGetLastError();
    };
    if (d.dtype == MLA_F32) return run(float{});
    if (d.dtype == MLA_F16) return run(__half{});
    return run(__nv_bfloat16{});
}

}  // namespace mla
