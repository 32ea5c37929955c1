// Tensor-core paged decode for bf16 (sm_103a): tcgen05 MMAs with TMEM
// accumulators, TMA-gathered cache blocks, a two-CTA cluster per work unit.
//
// What it computes is the paged single-pass decode of "vllm.cpp
// cpu_mla_attn.cpp" (MlaDecodeAttentionKernel): per query row, softmax over
// scale * (q_abs . row_j) for the visible keys and the latent output
// sum_j p_j row_j[0:512] with its LSE; the split + combine pair named in that
// page's header merges the partial results of a request split across CTAs.
//
// Layout of the work. The query rows of one request (t_q * n_head of them)
// form row groups of 128 (the MMA M dimension); all rows share the same
// cache rows, so heads are the M dimension and cache tokens the N (scores)
// or K (P*V) dimension. A unit of work is (request, row group, 64-token
// tile). A persistent grid of CTA pairs splits the unit sequence as
// tc_split.cuh describes (evenly, or aligned to requests when pairs get few
// tiles, or pooled over the row groups when they do not divide the pairs).
// In each pair:
//   CTA 0 ("S-CTA") holds the 128 query rows in TMEM (A operand) and computes
//     S = Q K^T for each tile (M=128, N=64, K=576 or 512) into TMEM, runs the
//     online softmax (two threads per query row, lazy rescaling) and stages
//     the bf16 probabilities P [128 x 64] in TMEM; four sender warps copy
//     them into CTA 1's shared memory, so the SM-to-SM transfer (tens of
//     GB/s) overlaps the next tile's softmax instead of stalling it.
//   CTA 1 ("O-CTA") holds O [128 x 512] f32 in all 512 TMEM columns and
//     computes O += P V (M=128, N=2x256, K=64) with V the leading 512 columns
//     of the same tile, which it loads itself (mostly L2 hits: the S-CTA
//     loaded the tile shortly before).
// The O accumulator alone fills a TMEM, so splitting the roles keeps both the
// QK^T and the P*V contractions at M=128 with no repeated work; the only
// exchange is P (16 KB per 64-token tile) plus per-row rescale factors.
//
// Every wait is bounded; on timeout the kernel records MLA_DEVERR_TIMEOUT,
// drains its outstanding copies, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "sm100.cuh"
#include "tc_decode.h"
#include "tc_split.cuh"

namespace mla {
namespace {

using namespace sm100;
using split::ntiles_of;
using split::ChunkScan;
using split::scan_chunk;
using split::aligned_tried;
using split::aligned_first_pair;
using split::aligned_check;
using split::aligned_decide;
using split::pairs_per_set;

constexpr int kTok = 64;                      // cache tokens per tile
constexpr int kNS = 3;                        // S-CTA pipeline stages (K of a tile)
constexpr int kNV = 2;                        // O-CTA pipeline stages (V of a tile)
constexpr int kNP = 5;                        // O-CTA P slots
constexpr int kChunk = 64 * 128;              // 64 tokens x 64 columns of bf16
constexpr int kStage = 8 * kChunk;            // O-CTA: V (latent 512 columns) of a tile
constexpr int kSideOff = kNV * kStage;        // O-CTA: P slots
constexpr int kPBytes = 128 * 128;            // P [128 rows x 64 tokens] bf16
constexpr int kPSlot = kPBytes + 1024;        // a P slot: P, then its AlphaMsg (1 KB aligned)
constexpr int kQChunk = 128 * 128;            // 128 query rows x 64 columns of bf16
constexpr int kVBlock = 8 * 2048;             // O-CTA: one block's V as [8 chunks][16 rows][128 B]
// S-CTA stage of a tile: its 4 cache blocks, each landed by one 5-D box as
// [2 halves][nkc chunks][8 rows][128 B] (nkc = W / 64). The 8-row group of
// tokens 8g..8g+7 of the tile (block g / 2, half g % 2) of chunk kc then sits
// at g * nkc * 1 KB + kc * 1 KB: a uniform group stride the score MMA's
// K-major operand takes as its SBO.
__host__ __device__ constexpr int s_stage_bytes(int nkc) { return nkc * kChunk; }
// the first segment's queries sit in stages 1-2 (chunk cc at 16 KB * cc);
// tile 0 uses stage 0 meanwhile
__host__ __device__ constexpr int q_chunk_off(int nkc, int cc) {
    return s_stage_bytes(nkc) + cc * kQChunk;
}
static_assert(9 * kQChunk <= 2 * s_stage_bytes(9) && 8 * kQChunk <= 2 * s_stage_bytes(8),
              "queries fit stages 1-2");
// S-CTA: above its stages, 2 KB per sender warp to regroup P rows (16 rows of
// 128 B) so that each store to the O-CTA writes 512 contiguous bytes
__host__ __device__ constexpr int p_regroup_off(int nkc) { return kNS * s_stage_bytes(nkc); }
constexpr int kCtrlOff = p_regroup_off(9) + 8 * 1024;  // both CTAs: the control block
static_assert(kSideOff + kNP * kPSlot <= kCtrlOff, "O-CTA V stages and P slots below the control block");
constexpr int kThreads = 448;                 // see the role map in the kernel
constexpr int kSmxWarps = 8;                  // S-CTA softmax warps: two threads per query row
constexpr int kSenders = 4;                   // S-CTA P senders: one per TMEM lane quadrant
constexpr uint64_t kWaitLimit = 2000000000ull;  // ns before a wait gives up (default)
constexpr uint32_t kSuspendHintNs = 1000;     // longest suspension of one wait poll
constexpr float kRescaleThreshold = 8.0f;     // lazy rescale, log2 units

// per-tile rescale message from the S-CTA's softmax to the O-CTA (st.async)
struct __align__(16) AlphaMsg {
    float alpha[128];           // per-row rescale factors of the P slot
    int32_t flags[kSenders];    // per sender warp (32 rows), some row needs a rescale
};

struct Ctrl {
    uint64_t full[kNS];     // both: this CTA's part of the tile landed (complete_tx)
    uint64_t pdone[kNP];    // O: the P*V reading P slot k finished (MMA commit); the
                            //    relay warp passes it on to the S-CTA's pempty
    uint64_t empty[kNS];    // both: stage free (own QK / P*V commit)
    uint64_t sfull[2];      // S: scores ready (QK commit)
    uint64_t sfree[2];      // S: scores read (the 256 softmax threads)
    uint64_t pempty[kNP];   // S: O-CTA P slot k consumed (its relay, 1 remote arrival)
    uint64_t pstaged[2];    // S: P + alpha of a tile in its TMEM slot (256 softmax threads)
    uint64_t pfree[2];      // S: that TMEM slot read by the senders (128 threads)
    uint64_t qready;        // S: Q stored in TMEM (256 softmax threads)
    uint64_t qland;         // S: first segment's queries landed in shared memory (TMA)
    uint64_t qfree;         // S: those queries are in TMEM; stages 1-2 reusable (256)
    uint64_t statack;       // S: O-CTA has read the segment statistics (1 remote)
    uint64_t pfull[kNP];    // O: P slot k written: P, alpha, flags (st.async bytes)
    uint64_t vready[kNS];   // O: tile tail zeroed (fix warp)
    uint64_t odone;         // O: all issued P*V complete (MMA commit)
    uint64_t evt;           // O: MMA warp -> row warps event
    uint64_t evtdone;       // O: row warps -> MMA warp (256)
    uint64_t statfull;      // O: segment statistics written (1 remote)
    uint64_t rowbar;        // both: barrier among the 256 row threads
    uint64_t never;         // S: arrived on by nothing (the timeout-path test waits on it)
    uint32_t tmem_base;
    int32_t abort;
    int32_t evt_type;       // 1 = rescale slot evt_slot, 2 = segment epilogue
    int32_t evt_slot;
    int32_t bad;            // O: the segment met an invalid block id
    int32_t badw[kSmxWarps];  // S: per softmax warp, the segment met an invalid block id
    float mstat[128];       // O: segment max (log2 units) per row
    float lstat[128];       // O: segment sum per row
    long long walk_u, walk_ue, walk_pe;  // both: the pair's unit range (see walk_init)
    int32_t walk_b, walk_g, walk_tile, walk_S, walk_nt, walk_ok;  // and its first unit
    int32_t walk_U, walk_b0, walk_S0, walk_nt0;                  // and its passes
};
constexpr int kSmemBytes = kCtrlOff + (int)sizeof(Ctrl);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Params {
    const __nv_bfloat16* q_abs;   // [B][T][H][W]
    const __nv_bfloat16* kv;      // [num_blocks][16][W]
    const int32_t* block_table;   // [B][max_blocks]
    const int32_t* seq_lens;      // [B]
    __nv_bfloat16* out;           // [B][T][H][512]
    float* lse;                   // [B][T][H] or null
    __nv_bfloat16* ws_o;          // partial rows: [2*NP slots][128 rows][512]
    float* ws_lse;                // [2*NP][128]
    int32_t* dev_err;
    int B, T, H, W, max_blocks, num_blocks;
    int NP, min_units;
    int combine_rpt;              // combine: query rows per thread (1, 2, 4 or 8)
    int early;                    // read cache, table and seq_lens before the previous
                                  // kernel completes (it writes none of them)
    float scale_log2;
    unsigned long long wait_ns;   // a bounded wait gives up after this long
    int stall;                    // test of the timeout path: the score MMA warp first
                                  // waits on a barrier nothing arrives on
};

// ------------------------------------------------------------------ schedule
// The work split is the one tc_split.cuh defines (even or request-aligned
// within each set, or pooled over the sets). With G > 1 row groups and one
// set of pairs per row group, the G sets read the same cache tiles at about
// the same time: one HBM read, the rest from L2. One warp per CTA works out
// the pair's walk; every warp of both CTAs then follows it.
static_assert(kTok == split::kTok, "unit size");
struct Walk {
    int b, g, tile, ntiles, S;
    long long u, u_end;
    // pooled split: the walk goes on from one set into the next (U units
    // each); pass_end is where the current set's units end, and a new set
    // starts again at (b0, S0, nt0), the first request with tiles
    long long pass_end;
    int U, b0, S0, nt0;
};

// This pair's set and unit range; warp-cooperative, at most two passes over
// seq_lens (one load when the batch fits a chunk). Returns false when the
// pair has no work.
__device__ bool walk_init(const Params& p, int pair, Walk& w) {
    const int lane = threadIdx.x & 31;
    const int Mq = p.T * p.H;
    const int G = (Mq + 127) / 128;
    ChunkScan c0 = scan_chunk(p, 0, lane);
    int U = c0.total;
    for (int b0 = 32; b0 < p.B; b0 += 32) U += scan_chunk(p, b0, lane).total;
    if (U == 0) return false;
    if (split::pooled_split(p, G)) {
        // this pair's share of the pooled units, from set g's unit ui
        const int np = split::pooled_pairs(p, G, U);
        if (pair >= np) return false;
        const long long T = (long long)G * U;
        const long long ub = T * pair / np, ue = T * (pair + 1) / np;
        if (ub >= ue) return false;
        const int g = (int)(ub / U);
        const int ui = (int)(ub - (long long)g * U);
        int base = 0, fb = -1, first = 0, S = 0, b0r = -1, S0 = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const ChunkScan c = b0 == 0 ? c0 : scan_chunk(p, b0, lane);
            const int excl = base + c.incl - c.v, incl = base + c.incl;
            const unsigned hit = __ballot_sync(0xffffffffu, incl > ui && c.v > 0);
            if (fb < 0 && hit) {
                const int l = __ffs(hit) - 1;
                fb = b0 + l;
                first = __shfl_sync(0xffffffffu, excl, l);
                S = __shfl_sync(0xffffffffu, c.S, l);
            }
            const unsigned any = __ballot_sync(0xffffffffu, c.v > 0);
            if (b0r < 0 && any) {
                const int l = __ffs(any) - 1;
                b0r = b0 + l;
                S0 = __shfl_sync(0xffffffffu, c.S, l);
            }
            base += c.total;
        }
        if (fb < 0 || b0r < 0) return false;
        w.b = fb;
        w.g = g;
        w.S = S;
        w.ntiles = ntiles_of(S, p.T, p.max_blocks);
        w.tile = ui - first;
        w.u = ub;
        w.u_end = ue;
        w.pass_end = (long long)(g + 1) * U;
        w.U = U;
        w.b0 = b0r;
        w.S0 = S0;
        w.nt0 = ntiles_of(S0, p.T, p.max_blocks);
        return true;
    }
    const int np_g = pairs_per_set(p, G, U);
    const int g = pair / np_g, k = pair % np_g;
    if (g >= G) return false;
    const bool tried = aligned_tried(U, np_g);
    const int ub_even = (int)((long long)U * k / np_g), ue_even = (int)((long long)U * (k + 1) / np_g);
    // one pass: the even split's first request, the aligned split's request
    // for pair k, and whether the aligned split is used
    int base = 0, worst = 0, bad = 0;
    int ev_b = -1, ev_first = 0, ev_S = 0;
    int al_b = -1, al_first = 0, al_S = 0, al_v = 0, al_p0 = 0, al_n = 1;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const ChunkScan c = b0 == 0 ? c0 : scan_chunk(p, b0, lane);
        const int excl = base + c.incl - c.v, incl = base + c.incl;
        const unsigned hit = __ballot_sync(0xffffffffu, incl > ub_even && c.v > 0);
        if (ev_b < 0 && hit) {
            const int l = __ffs(hit) - 1;
            ev_b = b0 + l;
            ev_first = __shfl_sync(0xffffffffu, excl, l);
            ev_S = __shfl_sync(0xffffffffu, c.S, l);
        }
        if (tried) {
            aligned_check(c, base, U, np_g, bad, worst);
            const int pb = aligned_first_pair(excl, U, np_g), pe = aligned_first_pair(incl, U, np_g);
            const unsigned ah = __ballot_sync(0xffffffffu, c.v > 0 && pb <= k && k < pe);
            if (al_b < 0 && ah) {
                const int l = __ffs(ah) - 1;
                al_b = b0 + l;
                al_first = __shfl_sync(0xffffffffu, excl, l);
                al_S = __shfl_sync(0xffffffffu, c.S, l);
                al_v = __shfl_sync(0xffffffffu, c.v, l);
                al_p0 = __shfl_sync(0xffffffffu, pb, l);
                al_n = __shfl_sync(0xffffffffu, pe - pb, l);
            }
        }
        base += c.total;
    }
    const bool aligned = tried && aligned_decide(bad, worst, U, np_g);
    int ub, ue, fb, first, S;
    if (aligned) {
        if (al_b < 0) return false;
        ub = al_first + (int)((uint32_t)al_v * (uint32_t)(k - al_p0) / (uint32_t)al_n);
        ue = al_first + (int)((uint32_t)al_v * (uint32_t)(k - al_p0 + 1) / (uint32_t)al_n);
        fb = al_b;
        first = al_first;
        S = al_S;
    } else {
        if (ev_b < 0) return false;
        ub = ub_even;
        ue = ue_even;
        fb = ev_b;
        first = ev_first;
        S = ev_S;
    }
    if (ub >= ue) return false;
    w.b = fb;
    w.g = g;
    w.S = S;
    w.ntiles = ntiles_of(S, p.T, p.max_blocks);
    w.tile = ub - first;
    w.u = ub;
    w.u_end = ue;
    w.pass_end = ue;  // (one set: no next one)
    w.U = U;
    w.b0 = fb;
    w.S0 = S;
    w.nt0 = w.ntiles;
    return true;
}

// advance to the next unit (caller checks u < u_end first)
__device__ __forceinline__ void walk_next(const Params& p, Walk& w) {
    ++w.u;
    if (w.u >= w.u_end) return;
    if (w.u == w.pass_end) {
        // the next row group (pooled split): the same requests and tiles again
        w.pass_end += w.U;
        w.g += 1;
        w.b = w.b0;
        w.S = w.S0;
        w.ntiles = w.nt0;
        w.tile = 0;
        return;
    }
    if (++w.tile < w.ntiles) return;
    w.tile = 0;
    do {
        ++w.b;
        w.S = p.seq_lens[w.b];
        w.ntiles = ntiles_of(w.S, p.T, p.max_blocks);
    } while (w.ntiles == 0);
}

__device__ __forceinline__ bool seg_first(const Walk& w, long long ub) {
    return w.u == ub || w.tile == 0;
}
__device__ __forceinline__ bool seg_last(const Walk& w) {
    return w.u + 1 == w.u_end || w.tile + 1 == w.ntiles;
}

// ------------------------------------------------------------------ helpers
struct Waiter {
    volatile int32_t* abort;
    int32_t* dev_err;
    uint64_t limit;  // ns
    __device__ bool wait(uint32_t bar, uint32_t parity) {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 1;; ++i) {
            if (mbar_try_wait_hint(bar, parity, kSuspendHintNs)) return true;
            if ((i & 255) == 0) {
                if (*abort) return false;
                if (globaltimer_ns() - t0 > limit) break;
            }
        }
        *abort = 1;
        if (dev_err) atomicOr(dev_err, (int32_t)MLA_DEVERR_TIMEOUT);
        return false;
    }
    // every lane of the warp waits; the result is the same in all lanes, so a
    // timeout in one lane takes the whole warp out of the loop together
    __device__ bool wait_warp(uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, wait(bar, parity));
    }
    // the same without suspension hints: for short waits on the critical
    // path (a barrier among the row warps)
    __device__ bool spin_warp(uint32_t bar, uint32_t parity) {
        bool ok = mbar_try_wait(bar, parity);
        if (!ok) {
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t i = 1;; ++i) {
                if (mbar_try_wait(bar, parity)) { ok = true; break; }
                if ((i & 255) == 0) {
                    if (*abort) break;
                    if (globaltimer_ns() - t0 > limit) {
                        *abort = 1;
                        if (dev_err) atomicOr(dev_err, (int32_t)MLA_DEVERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
        return __all_sync(0xffffffffu, ok);
    }
};

// Bounded barrier among the 256 row threads (warps 5..12) of one CTA; `phase`
// counts the caller's uses. Returns false on timeout.
__device__ __forceinline__ bool rows_sync(Waiter& wt, uint32_t bar, uint32_t& phase) {
    mbar_arrive(bar);
    return wt.spin_warp(bar, (phase++) & 1);
}

__device__ __forceinline__ int valid_blocks(const Walk& w) {
    const int rem = w.S - w.tile * kTok;
    const int nb = (rem + 15) / 16;
    return nb < 4 ? nb : 4;
}

// ------------------------------------------------------------------ kernel
// Role map (14 warps per CTA):
//   S-CTA  warps 0-3  P senders: warp q reads the staged P rows of TMEM lanes
//                     32q..32q+31 and writes them (and their rescale factors)
//                     into the O-CTA's P slot by st.async
//          warp 4     S = Q K^T MMA issuer; owns the TMEM allocation
//          warps 5-12 softmax, two threads per query row (32 score columns
//                     each); P and alpha go to a TMEM slot
//          warp 13    K loader: one 5-D box per cache block of each tile
//   O-CTA  warp 0     V loader: one 4-D box per cache block
//          warp 1     V landing: zeroes the rows of a partial last block past
//                     the request, releases the stage
//          warp 2     idle after working out the walk (an L2 prefetcher of the
//                     coming cache blocks here cost 6% of the causal t_q = 4
//                     decode: its requests competed with the loads)
//          warp 4     O += P V MMA issuer; owns the TMEM allocation
//          warps 5-12 rescale and epilogue: warp w takes the TMEM lanes of
//                     its quadrant (w % 4) and half the 512 columns
//          warp 3     relay: passes each P*V completion (its own barrier) on to
//                     the S-CTA's P-slot barrier by a remote mbarrier arrive
//          warp 13    idle
// In both CTAs warp 2 first works out the pair's unit range (walk_init) while
// the barriers and TMEM are set up; every warp then follows that walk.
template <int W, bool kF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                       const __grid_constant__ CUtensorMap wmap, const Params p) {
    constexpr int NKC = W / 64;  // 64-column chunks in a cache row (9 or 8)
    extern __shared__ __align__(1024) unsigned char smem[];
    Ctrl& c = *reinterpret_cast<Ctrl*>(smem + kCtrlOff);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1;
    Waiter wt{&c.abort, p.dev_err, p.wait_ns};

    grid_dependents_launch();  // the combine kernel may be scheduled (it waits for this grid)
    if ((smem_u32(smem) & 1023) != 0) {  // swizzled operands need 1 KB alignment
        if (tid == 0 && p.dev_err) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_TIMEOUT);
        return;  // both CTAs take this path together (same layout)
    }
    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(smem_u32(&c.full[s]), 1);
            mbar_init(smem_u32(&c.empty[s]), 1);
            mbar_init(smem_u32(&c.vready[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&c.sfull[i]), 1);
            mbar_init(smem_u32(&c.sfree[i]), kSmxWarps * 32);
            mbar_init(smem_u32(&c.pstaged[i]), kSmxWarps * 32);
            mbar_init(smem_u32(&c.pfree[i]), kSenders * 32);
        }
        for (int k = 0; k < kNP; ++k) {
            mbar_init(smem_u32(&c.pempty[k]), 1);
            mbar_init(smem_u32(&c.pfull[k]), 1);
            mbar_init(smem_u32(&c.pdone[k]), 1);
        }
        mbar_init(smem_u32(&c.qready), 256);
        mbar_init(smem_u32(&c.qland), 1);
        mbar_init(smem_u32(&c.qfree), 256);
        mbar_init(smem_u32(&c.statack), 1);
        mbar_init(smem_u32(&c.odone), 1);
        mbar_init(smem_u32(&c.evt), 1);
        mbar_init(smem_u32(&c.evtdone), 256);
        mbar_init(smem_u32(&c.statfull), 1);
        mbar_init(smem_u32(&c.rowbar), 256);
        mbar_init(smem_u32(&c.never), 1);
        c.abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_u32(&c.tmem_base), 512);
        tmem_relinquish();
    }
    if (rank == 1 && warp != 2) {
        // O-CTA: clear the V stages once, so a block past a request's end that
        // the P*V MMA reads (under P = 0) never holds a NaN
        for (int i = tid - (warp > 2 ? 32 : 0); i < kNV * kStage / 16; i += kThreads - 32)
            reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (warp == 2) {
        // the pair's unit range, worked out once per CTA while the barriers and
        // TMEM are set up; every warp starts its walk from it
        if (!p.early) grid_dependency_wait();
        Walk w0;
        const bool ok = walk_init(p, pair, w0);
        if (lane == 0) {
            c.walk_ok = ok ? 1 : 0;
            if (ok) {
                c.walk_u = w0.u;
                c.walk_ue = w0.u_end;
                c.walk_b = w0.b;
                c.walk_g = w0.g;
                c.walk_tile = w0.tile;
                c.walk_S = w0.S;
                c.walk_nt = w0.ntiles;
                c.walk_pe = w0.pass_end;
                c.walk_U = w0.U;
                c.walk_b0 = w0.b0;
                c.walk_S0 = w0.S0;
                c.walk_nt0 = w0.nt0;
            }
        }
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tbase = c.tmem_base;
    // a call outside the library's own chain: the previous kernel may have
    // written any input, so nothing is read before it completes
    if (!p.early) grid_dependency_wait();

    Walk w;
    const bool has_work = c.walk_ok != 0;
    if (has_work) {
        w.b = c.walk_b;
        w.g = c.walk_g;
        w.tile = c.walk_tile;
        w.S = c.walk_S;
        w.ntiles = c.walk_nt;
        w.u = c.walk_u;
        w.u_end = c.walk_ue;
        w.pass_end = c.walk_pe;
        w.U = c.walk_U;
        w.b0 = c.walk_b0;
        w.S0 = c.walk_S0;
        w.nt0 = c.walk_nt0;
    }
    const long long ub = has_work ? w.u : 0;
    const int Mq = p.T * p.H;

    if (has_work && rank == 0) {
        // =============================== S-CTA ===============================
        const uint32_t tq = tbase;              // Q: columns [0, W/2)
        const uint32_t ts0 = tbase + W / 2;     // S buffers: 2 x 64 columns
        const uint32_t tp0 = ts0 + 2 * kTok;    // P slots: 2 x 32 columns (bf16 pairs)
        const uint32_t ta0 = tp0 + 64;          // alpha: 2 x 2 columns
        static_assert(W / 2 + 2 * kTok + 64 + 4 <= 512, "S-CTA TMEM columns");
        if (warp < 4) {
            // ---------------- P senders: warp q ships the P rows of TMEM lanes
            // 32q..32q+31 and their rescale factors to the O-CTA's P slot
            const int q = warp;
            const uint32_t lane_q = (uint32_t)(q * 32) << 16;
            const int row = q * 32 + lane;
            const uint32_t pslot_remote = mapa(smem_u32(smem + kSideOff), 1);
            const uint32_t pfull_remote = mapa(smem_u32(&c.pfull[0]), 1);
            const uint32_t regroup = smem_u32(smem + p_regroup_off(NKC)) + (uint32_t)q * 2048;
            long long i = 0;
            for (; w.u < w.u_end; walk_next(p, w), ++i) {
                const int buf = (int)(i & 1);
                if (!wt.wait_warp(smem_u32(&c.pstaged[buf]), (uint32_t)((i >> 1) & 1))) break;
                tc_fence_after();
                uint32_t v[32], av;
                tmem_ld32(tp0 + buf * 32 + lane_q, v);  // this row's 32 bf16 pairs
                tmem_ld1(ta0 + buf * 2 + lane_q, av);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(smem_u32(&c.pfree[buf]));
                // the O-CTA's P slot free? (its P*V kNP tiles back)
                const int slot = (int)(i % kNP);
                if (!wt.wait_warp(smem_u32(&c.pempty[slot]), (uint32_t)((i / kNP) & 1) ^ 1)) break;
                const uint32_t pbar = pfull_remote + slot * 8;
                const uint32_t dst = pslot_remote + slot * kPSlot;
                const int grows = min(128, Mq - w.g * 128);
                // The rows go out 16 at a time: the 16 threads holding them write
                // them into the warp's 2 KB in the P slot's swizzled layout, then
                // every lane ships four 16-byte pieces, so that each store covers 4
                // whole rows (512 contiguous bytes). Rows past the group are never
                // read back and are not sent.
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    if ((lane >> 4) == a) {
                        const int rr = lane & 15;  // row 32q + 16a + rr: its swizzle phase is rr & 7
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            st_shared_v4(regroup + rr * 128 + ((u ^ (rr & 7)) << 4), v[4 * u], v[4 * u + 1],
                                         v[4 * u + 2], v[4 * u + 3]);
                    }
                    __syncwarp();
                    uint4 d[4];
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2)
                        d[h2] = ld_shared_v4(regroup + (4 * h2 + (lane >> 3)) * 128 + ((lane & 7) << 4));
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        const int r = q * 32 + 16 * a + 4 * h2 + (lane >> 3);
                        if (r < grows)
                            st_async_v4(dst + r * 128 + ((lane & 7) << 4), d[h2].x, d[h2].y, d[h2].z, d[h2].w,
                                        pbar);
                    }
                    __syncwarp();  // the next round overwrites the warp's 2 KB
                }
                // alpha is 1 on a segment's first tile (no running max yet), so a
                // factor other than 1 is a rescale of the rows' earlier P*V
                if (row < grows) st_async_b32(dst + kPBytes + row * 4, av, pbar);
                const unsigned any = __ballot_sync(0xffffffffu, row < grows && __uint_as_float(av) != 1.f);
                if (lane == 0)
                    st_async_b32(dst + kPBytes + (uint32_t)offsetof(AlphaMsg, flags) + q * 4, any ? 1u : 0u,
                                 pbar);
            }
        } else if (warp == 13) {
            // ---------------- K loader: the tile's cache blocks, one box each
            if (elect_one()) {
                tma_prefetch_desc(&tmap);
                tma_prefetch_desc(&qmap);
                // the first segment's queries: TMA into stages 1 and 2 (free until
                // the rows move them to TMEM), while tile 0 goes to stage 0.
                // They come from the previous kernel (programmatic launch).
                // (a request's rows past t_q * n_head are outside the map)
                grid_dependency_wait();
                {
                    const int qrows = Mq < 128 ? Mq : 128;
                    mbar_arrive_expect_tx(smem_u32(&c.qland), (uint32_t)(NKC * qrows * 128));
                    for (int cc = 0; cc < NKC; ++cc)
                        tma_load_3d(smem_u32(smem + q_chunk_off(NKC, cc)), &qmap, smem_u32(&c.qland),
                                    cc * 64, w.g * 128, w.b);
                }
                long long i = 0;
                long long last_issue[kNS];
                for (int s = 0; s < kNS; ++s) last_issue[s] = -1;
                for (; w.u < w.u_end; walk_next(p, w), ++i) {
                    const int s = (int)(i % kNS);
                    if (!wt.wait(smem_u32(&c.empty[s]), (uint32_t)((i / kNS) & 1) ^ 1)) break;
                    if (i == 1 || i == 2)  // first use of a stage that held the queries
                        if (!wt.wait(smem_u32(&c.qfree), 0)) break;
                    if (i > 0 && w.tile == 0) {
                        // a later segment: warm L2 with its queries for the row threads
                        const int rows = min(128, Mq - w.g * 128);
                        prefetch_l2_bulk(p.q_abs + ((long long)w.b * Mq + w.g * 128) * W,
                                         (uint32_t)(rows * W * 2));
                    }
                    const int nb = valid_blocks(w);
                    const int32_t* bt = p.block_table + (long long)w.b * p.max_blocks + w.tile * 4;
                    int32_t blk[4];
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) blk[kb] = kb < nb ? bt[kb] : 0;
                    mbar_arrive_expect_tx(smem_u32(&c.full[s]), (uint32_t)(nb * NKC * 2048));
                    last_issue[s] = i;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb) {
                        if (kb >= nb) break;
                        int32_t b = blk[kb];
                        if (b < 0 || b >= p.num_blocks) {
                            // load a valid stand-in; the row threads void the segment
                            if (p.dev_err) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_BAD_BLOCK);
                            b = 0;
                        }
                        // the whole block (all NKC chunks, both 8-row halves) in one box
                        tma_load_5d(smem_u32(smem + s * s_stage_bytes(NKC) + kb * NKC * 2048), &tmap,
                                    smem_u32(&c.full[s]), 0, 0, 0, 0, b);
                    }
                }
                // drain: the copies issued into each stage must have landed
                mbar_wait(smem_u32(&c.qland), 0, p.wait_ns);
                for (int s = 0; s < kNS; ++s)
                    if (last_issue[s] >= 0)
                        mbar_wait(smem_u32(&c.full[s]), (uint32_t)((last_issue[s] / kNS) & 1),
                                  p.wait_ns);
            }
        } else if (warp == 4) {
            // ---------------- MMA issuer: S = Q K^T
            if (elect_one()) {
                constexpr uint32_t idesc = idesc_f32acc<kF16>(128, kTok, 0, 0);
                long long i = 0;
                int seg = 0;
                // the timeout-path test: this wait gives up (recording the
                // timeout and raising the abort flag) and no MMA is issued
                if (p.stall && !wt.wait(smem_u32(&c.never), 0)) w.u = w.u_end;
                for (; w.u < w.u_end; walk_next(p, w), ++i) {
                    const int s = (int)(i % kNS);
                    const int buf = (int)(i & 1);
                    if (seg_first(w, ub)) {
                        if (!wt.wait(smem_u32(&c.qready), (uint32_t)(seg & 1))) break;
                        ++seg;
                    }
                    if (!wt.wait(smem_u32(&c.full[s]), (uint32_t)((i / kNS) & 1))) break;
                    if (!wt.wait(smem_u32(&c.sfree[buf]), (uint32_t)((i >> 1) & 1) ^ 1)) break;
                    tc_fence_after();
                    const uint32_t d = ts0 + buf * kTok;
#pragma unroll 1
                    for (int kc = 0; kc < NKC; ++kc) {
                        // chunk kc: 8 groups of 8 tokens at a stride of NKC KB
                        const uint32_t base = smem_u32(smem + s * s_stage_bytes(NKC) + kc * 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(d, tq + kc * 32 + kk * 8,
                                   sdesc_sw128(base + kk * 32, 16, NKC * 1024), idesc,
                                   (kc | kk) != 0);
                    }
                    mma_commit(smem_u32(&c.sfull[buf]));
                    mma_commit(smem_u32(&c.empty[s]));
                }
            }
        } else if (warp >= 5 && warp <= 12) {
            // ---------------- softmax (warps 5..12): warp w reads the 16 TMEM lanes
            // 32 (w % 4) + 16 h (h = 0 for warps 5..8, 1 for 9..12) with the 16x64b
            // shape; the two threads of a query row hold its even and odd score
            // columns, share the row max by one shuffle and trade columns so each
            // holds the bf16 pairs it stores back in the same layout
            const int q = warp & 3;
            const int h = warp >= 9 ? 1 : 0;
            const int sw = warp - 5;                                  // 0..7
            const int R = q * 32 + h * 16 + (lane >> 2) + 8 * (lane & 1);  // query row
            const int par = (lane >> 1) & 1;                          // odd columns
            const uint32_t lane_base16 = (uint32_t)(q * 32 + h * 16) << 16;
            const uint32_t lane_off = (uint32_t)(q * 32) << 16;      // Q moves
            const int rq = q * 32 + lane;                             // their row
            const uint32_t mstat_remote = mapa(smem_u32(&c.mstat[0]), 1);
            const uint32_t lstat_remote = mapa(smem_u32(&c.lstat[0]), 1);
            const uint32_t bad_remote = mapa(smem_u32(&c.bad), 1);
            const uint32_t statfull_remote = mapa(smem_u32(&c.statfull), 1);
            const float sl2 = p.scale_log2;
            grid_dependency_wait();  // later segments read their queries from global memory
            long long i = 0;
            int seg = 0;
            uint32_t rphase = 0;
            float m_used = -INFINITY, l = 0.f;
            int horizon = 0, bad = 0;
            bool row_ok = false;
            for (; w.u < w.u_end; walk_next(p, w), ++i) {
                const int buf = (int)(i & 1);
                const bool first_tile = seg_first(w, ub);
                if (first_tile) {
                    const int grow = w.g * 128 + R;
                    row_ok = grow < Mq;
                    const int t = row_ok ? grow / p.H : 0;
                    horizon = row_ok ? w.S - p.T + t + 1 : 0;
                    m_used = -INFINITY;
                    l = 0.f;
                    bad = 0;
                    {
                        // all eight warps move the segment's queries into TMEM, a row
                        // per thread: warps 5..8 chunks [0, kQSplit), warps 9..12 the rest
                        constexpr int kQSplit = (NKC + 1) / 2;
                        const int c0 = h ? kQSplit : 0, c1 = h ? NKC : kQSplit;
                        const int growq = w.g * 128 + rq;
                        const bool rq_ok = growq < Mq;
                        if (seg == 0) {
                            // landed in shared memory by TMA
                            if (!wt.wait_warp(smem_u32(&c.qland), 0)) break;
#pragma unroll 1
                            for (int cc = c0; cc < c1; ++cc) {
                                const uint32_t rowa = smem_u32(smem + q_chunk_off(NKC, cc)) + rq * 128;
                                uint32_t v[32];
#pragma unroll
                                for (int u = 0; u < 8; ++u) {
                                    const uint4 x = ld_shared_v4(rowa + ((u ^ (rq & 7)) << 4));
                                    v[4 * u] = rq_ok ? x.x : 0u;
                                    v[4 * u + 1] = rq_ok ? x.y : 0u;
                                    v[4 * u + 2] = rq_ok ? x.z : 0u;
                                    v[4 * u + 3] = rq_ok ? x.w : 0u;
                                }
                                tmem_st32(tq + lane_off + cc * 32, v);
                            }
                            tmem_wait_st();
                            mbar_arrive(smem_u32(&c.qfree));  // stages 1 and 2 may be refilled
                        } else {
                            // later segments: from global memory (warmed in L2 by the
                            // loader), two chunks per round trip
                            const uint4* src = reinterpret_cast<const uint4*>(
                                p.q_abs + ((long long)w.b * Mq + (rq_ok ? growq : 0)) * W);
#pragma unroll 1
                            for (int cc = c0; cc < c1; cc += 2) {
                                const bool two = cc + 1 < c1;
                                uint4 x[16];
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    x[j] = (rq_ok && (j < 8 || two)) ? src[cc * 8 + j] : make_uint4(0, 0, 0, 0);
#pragma unroll
                                for (int k = 0; k < 2; ++k) {
                                    if (k == 1 && !two) break;
                                    uint32_t v[32];
#pragma unroll
                                    for (int j = 0; j < 8; ++j) {
                                        v[4 * j] = x[8 * k + j].x;
                                        v[4 * j + 1] = x[8 * k + j].y;
                                        v[4 * j + 2] = x[8 * k + j].z;
                                        v[4 * j + 3] = x[8 * k + j].w;
                                    }
                                    tmem_st32(tq + lane_off + (cc + k) * 32, v);
                                }
                            }
                            tmem_wait_st();
                        }
                        tc_fence_before();
                        mbar_arrive(smem_u32(&c.qready));
                    }
                    // invalid block ids anywhere in the segment void it (the loader
                    // loaded a stand-in block): the softmax warps scan its table
                    // slice now, while the first QK runs; the segment's end reads it
                    {
                        const long long left = w.u_end - 1 - w.u;
                        const int last_tile = (int)min((long long)w.ntiles - 1, (long long)w.tile + left);
                        const int blk0 = w.tile * 4;
                        const int blk1 = min(last_tile * 4 + 4, (w.S + 15) / 16);
                        const int32_t* bt = p.block_table + (long long)w.b * p.max_blocks;
                        int b_any = 0;
                        for (int k = blk0 + sw * 32 + lane; k < blk1; k += kSmxWarps * 32) {
                            const int32_t blk = bt[k];
                            b_any |= (blk < 0 || blk >= p.num_blocks);
                        }
                        b_any = __any_sync(0xffffffffu, b_any);
                        if (lane == 0) c.badw[sw] = b_any;
                    }
                }
                if (!wt.wait_warp(smem_u32(&c.sfull[buf]), (uint32_t)((i >> 1) & 1))) break;
                tc_fence_after();
                float x[32];  // columns 2 j + par
                {
                    uint32_t v[32];
                    tmem_ld16x64(ts0 + buf * kTok + lane_base16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 2)
                        mul2(x[j], x[j + 1], __uint_as_float(v[j]), __uint_as_float(v[j + 1]), sl2);
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&c.sfree[buf]));
                // keys past this row's horizon (only near the request's end)
                const int j0 = w.tile * kTok + par;
                if (w.tile * kTok + kTok > horizon) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j0 + 2 * j >= horizon) x[j] = -INFINITY;
                }
                float mx0 = x[0], mx1 = x[1];
#pragma unroll
                for (int j = 2; j < 32; j += 2) {
                    mx0 = fmaxf(mx0, x[j]);
                    mx1 = fmaxf(mx1, x[j + 1]);
                }
                float mx = fmaxf(mx0, mx1);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                float alpha = 1.f;
                if (mx > m_used + kRescaleThreshold || (m_used == -INFINITY && mx > -INFINITY)) {
                    alpha = (m_used == -INFINITY) ? 1.f : ex2_approx(m_used - mx);
                    m_used = mx;
                }
                const float mref = (m_used == -INFINITY) ? 0.f : m_used;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    sub2(x[j], x[j + 1], mref);
                    x[j] = ex2_approx(x[j]);  // 2^-inf = +0
                    x[j + 1] = ex2_approx(x[j + 1]);
                    add2(ps0, ps1, x[j], x[j + 1]);
                }
                l = l * alpha + (ps0 + ps1);  // this thread's columns; the pair adds at the end
                // P into the TMEM slot, in the 16x64b layout the scores came in:
                // register k of thread `par` is bf16 pair 2k + par of its row (pair
                // c = columns 2c, 2c + 1), so the two threads trade one value per pair
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float got = __shfl_xor_sync(0xffffffffu, par ? x[2 * k] : x[2 * k + 1], 2);
                    pk[k] = par ? pack2<kF16>(got, x[2 * k + 1]) : pack2<kF16>(x[2 * k], got);
                }
                // the slot free? (its senders have read tile i - 2)
                if (!wt.wait_warp(smem_u32(&c.pfree[buf]), (uint32_t)((i >> 1) & 1) ^ 1)) break;
                tc_fence_after();
                tmem_st16x64_x16(tp0 + buf * 32 + lane_base16, pk);
                tmem_st16x64_x1(ta0 + buf * 2 + lane_base16, __float_as_uint(alpha));  // both columns
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&c.pstaged[buf]));
                if (seg_last(w)) {
                    const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 2);
                    if (!rows_sync(wt, smem_u32(&c.rowbar), rphase)) break;
                    bad = 0;
#pragma unroll
                    for (int k = 0; k < kSmxWarps; ++k) bad |= c.badw[k];
                    // hand the row statistics to the O-CTA
                    if (seg > 0 && !wt.wait_warp(smem_u32(&c.statack), (uint32_t)((seg - 1) & 1))) break;
                    if (par == 0) {
                        st_cluster_f32(mstat_remote + R * 4, row_ok ? m_used : -INFINITY);
                        st_cluster_f32(lstat_remote + R * 4, row_ok ? l_row : 0.f);
                    }
                    if (sw == 0 && lane == 0)
                        asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(bad_remote), "r"(bad)
                                     : "memory");
                    if (!rows_sync(wt, smem_u32(&c.rowbar), rphase)) break;
                    if (sw == 0 && lane == 0) mbar_arrive_remote(statfull_remote);
                    ++seg;
                }
            }
        }
    } else if (has_work) {
        // =============================== O-CTA ===============================
        if (warp == 0) {
            // ---------------- V loader: one 4-D box [8 chunks][16 rows][64 cols] per block
            if (elect_one()) {
                tma_prefetch_desc(&vmap);
                long long i = 0;
                long long last_issue[kNV];
                for (int s = 0; s < kNV; ++s) last_issue[s] = -1;
                for (; w.u < w.u_end; walk_next(p, w), ++i) {
                    const int s = (int)(i % kNV);
                    if (!wt.wait(smem_u32(&c.empty[s]), (uint32_t)((i / kNV) & 1) ^ 1)) break;
                    const int nb = valid_blocks(w);
                    const int32_t* bt = p.block_table + (long long)w.b * p.max_blocks + w.tile * 4;
                    mbar_arrive_expect_tx(smem_u32(&c.full[s]), (uint32_t)(nb * kVBlock));
                    last_issue[s] = i;
                    for (int k = 0; k < nb; ++k) {
                        int32_t blk = bt[k];
                        if (blk < 0 || blk >= p.num_blocks) blk = 0;  // voided by the S-CTA rows
                        tma_load_4d(smem_u32(smem + s * kStage + k * kVBlock), &vmap,
                                    smem_u32(&c.full[s]), 0, 0, 0, blk);
                    }
                }
                for (int s = 0; s < kNV; ++s)
                    if (last_issue[s] >= 0)
                        mbar_wait(smem_u32(&c.full[s]), (uint32_t)((last_issue[s] / kNV) & 1),
                                  p.wait_ns);
            }
        } else if (warp == 1) {
            // ---------------- V landing: the rows of the tile's last cache block
            // past the request are zeroed (P there is 0, but 0 * NaN would still
            // poison the accumulator). Blocks past the request are not loaded;
            // their rows are zeros (the stages are cleared at start) or rows of
            // an earlier tile, all finite.
            long long i = 0;
            for (; w.u < w.u_end; walk_next(p, w), ++i) {
                const int s = (int)(i % kNV);
                if (!wt.wait_warp(smem_u32(&c.full[s]), (uint32_t)((i / kNV) & 1))) break;
                const int nvalid = min(kTok, w.S - w.tile * kTok);
                const int r0 = nvalid & 15;  // first row past the request in its block
                if (r0 != 0) {
                    // [8 chunks][16 - r0 rows][8 pieces of 16 bytes] of block nvalid / 16
                    const int nr = 16 - r0;
                    unsigned char* blk = smem + s * kStage + (nvalid >> 4) * kVBlock + r0 * 128;
                    for (int e = lane; e < 8 * 8 * nr; e += 32) {
                        const int ch = e >> 3 & 7, u = e & 7, rr = e >> 6;
                        *reinterpret_cast<uint4*>(blk + ch * 2048 + rr * 128 + u * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&c.vready[s]));
            }
        } else if (warp == 3) {
            // ---------------- relay: once the P*V that read P slot i % kNP has
            // finished (this CTA's pdone), the S-CTA may refill the slot: one
            // remote arrival on its pempty per tile
            if (elect_one()) {
                const uint32_t pempty_remote = mapa(smem_u32(&c.pempty[0]), 0);
                long long i = 0;
                for (; w.u < w.u_end; walk_next(p, w), ++i) {
                    const int slot = (int)(i % kNP);
                    if (!wt.wait(smem_u32(&c.pdone[slot]), (uint32_t)((i / kNP) & 1))) break;
                    mbar_arrive_remote(pempty_remote + slot * 8);
                }
            }
        } else if (warp == 4) {
            // ---------------- MMA issuer: O += P V
            if (elect_one()) {
                constexpr uint32_t idesc = idesc_f32acc<kF16>(128, 256, 0, 1);
                long long i = 0;
                int nevt = 0, ndone = 0;
                for (; w.u < w.u_end; walk_next(p, w), ++i) {
                    const int s = (int)(i % kNV);
                    const int slot = (int)(i % kNP);
                    // this tile's P rows, rescale factors and flags arrive by st.async
                    {
                        const int grows = min(128, Mq - w.g * 128);
                        mbar_arrive_expect_tx(smem_u32(&c.pfull[slot]),
                                              (uint32_t)(grows * (128 + 4) + kSenders * 4));
                    }
                    if (!wt.wait(smem_u32(&c.vready[s]), (uint32_t)((i / kNV) & 1))) break;
                    if (!wt.wait(smem_u32(&c.pfull[slot]), (uint32_t)((i / kNP) & 1))) break;
                    const bool first = seg_first(w, ub);
                    const volatile int32_t* fl =
                        reinterpret_cast<const AlphaMsg*>(smem + kSideOff + slot * kPSlot + kPBytes)->flags;
                    int any_flag = 0;
#pragma unroll
                    for (int k = 0; k < kSenders; ++k) any_flag |= fl[k];
                    if (!first && any_flag) {
                        // rows whose max moved: rescale O once the issued P*V is done
                        mma_commit(smem_u32(&c.odone));
                        if (!wt.wait(smem_u32(&c.odone), (uint32_t)(ndone & 1))) break;
                        ++ndone;
                        c.evt_type = 1;
                        c.evt_slot = slot;
                        mbar_arrive(smem_u32(&c.evt));
                        if (!wt.wait(smem_u32(&c.evtdone), (uint32_t)(nevt & 1))) break;
                        ++nevt;
                    }
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const uint32_t pa = smem_u32(smem + kSideOff + slot * kPSlot);
                    const uint32_t va = smem_u32(smem + s * kStage);
                    // V: K-step kk is cache block kk of the tile; its latent columns
                    // sit in 8 chunks of [16 rows][128 B] at a 2 KB stride. A block
                    // past the request holds zeros or an earlier tile's rows (finite),
                    // under P columns that are 0.
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tbase + half * 256, sdesc_sw128(pa + kk * 32, 16, 1024),
                                   sdesc_sw128(va + kk * kVBlock + half * 4 * 2048, 2048, 1024),
                                   idesc, !(first && kk == 0));
                    const bool last = seg_last(w);
                    // the last tile of a segment keeps its stage: the epilogue stages
                    // the output there, then releases it
                    if (!last) mma_commit(smem_u32(&c.empty[s]));
                    mma_commit(smem_u32(&c.pdone[slot]));  // the relay tells the S-CTA
                    if (last) {
                        mma_commit(smem_u32(&c.odone));
                        if (!wt.wait(smem_u32(&c.odone), (uint32_t)(ndone & 1))) break;
                        ++ndone;
                        c.evt_type = 2;
                        c.evt_slot = s;
                        mbar_arrive(smem_u32(&c.evt));
                        if (!wt.wait(smem_u32(&c.evtdone), (uint32_t)(nevt & 1))) break;
                        ++nevt;
                        mbar_arrive(smem_u32(&c.empty[s]));
                    }
                }
            }
        } else if (warp >= 5 && warp <= 12) {
            // ---------------- row warps: rescale and epilogue. Warps 5..8 take
            // columns 0..255 of their 32 rows, warps 9..12 columns 256..511.
            const int q = warp & 3;
            const int hc = warp >= 9 ? 1 : 0;
            const int c_lo = hc * 256;
            const int r = q * 32 + lane;
            const bool lead = hc == 0;               // writes the per-row values once
            const uint32_t lane_off = (uint32_t)(q * 32) << 16;
            const uint32_t statack_remote = mapa(smem_u32(&c.statack), 0);
            grid_dependency_wait();  // their writes follow the previous kernel's
            int nevt = 0, seg = 0;
            uint32_t rphase = 0;
            int seg_tile0 = w.tile;
            bool done = false;
            while (!done) {
                if (!wt.wait_warp(smem_u32(&c.evt), (uint32_t)(nevt & 1))) break;
                ++nevt;
                tc_fence_after();
                const int type = *(volatile int32_t*)&c.evt_type;
                if (type == 1) {
                    const int slot = *(volatile int32_t*)&c.evt_slot;
                    const float a =
                        reinterpret_cast<const AlphaMsg*>(smem + kSideOff + slot * kPSlot + kPBytes)->alpha[r];
                    if (a != 1.f) {
#pragma unroll 1
                        for (int cc = c_lo; cc < c_lo + 256; cc += 32) {
                            uint32_t v[32];
                            tmem_ld32(tbase + lane_off + cc, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __float_as_uint(__uint_as_float(v[j]) * a);
                            tmem_st32(tbase + lane_off + cc, v);
                        }
                        tmem_wait_st();
                    }
                    tc_fence_before();
                    mbar_arrive(smem_u32(&c.evtdone));
                    continue;
                }
                // segment epilogue: locate the segment (advance the walk to its end)
                while (!seg_last(w)) walk_next(p, w);
                const int stage = *(volatile int32_t*)&c.evt_slot;
                if (!wt.wait_warp(smem_u32(&c.statfull), (uint32_t)(seg & 1))) break;
                const float m = c.mstat[r];
                const float lsum = c.lstat[r];
                const int seg_bad = *(volatile int32_t*)&c.bad;
                // statistics consumed: the S-CTA may send the next segment's
                if (!rows_sync(wt, smem_u32(&c.rowbar), rphase)) break;
                if (lead && r == 0) mbar_arrive_remote(statack_remote);
                const int grow = w.g * 128 + r;
                const bool row_ok = grow < Mq;
                const bool full_seg = (seg_tile0 == 0) && (w.tile + 1 == w.ntiles);
                const bool empty = seg_bad || !(lsum > 0.f);
                const float inv = empty ? 0.f : 1.f / lsum;
                const float lse_v = empty ? -INFINITY : (m + log2f(lsum)) * 0.69314718055994531f;
                // bf16 rows: each warp takes its 32 rows and its half of the
                // columns, 64 at a time, into one of two private 4 KB scratch
                // buffers in the freed V stage, and one lane stores the
                // [32 rows x 64 columns] box by TMA; the next block's TMEM load
                // runs while that store reads its buffer. A full segment writes
                // the output rows (rows past the request's fall outside the
                // output map), a partial one its workspace slot, which the
                // combine or the merging decompress reads.
                const int slot = pair * 2 + (seg == 0 ? 0 : 1);
                const int row_lim = min(128, Mq - w.g * 128) - q * 32;  // this warp's valid rows
                if (row_lim > 0) {
                    const uint32_t scr0 = smem_u32(smem + stage * kStage) + (uint32_t)(warp - 5) * 8192;
#pragma unroll 1
                    for (int cb = c_lo, nb = 0; cb < c_lo + 256; cb += 64, ++nb) {
                        const uint32_t scr = scr0 + (uint32_t)(nb & 1) * 4096;
                        if (nb >= 2) {
                            if (lane == 0) bulk_wait_read_1();  // the store of block nb - 2 has read it
                            __syncwarp();
                        }
                        uint32_t v0[32], v1[32];
                        tmem_ld32(tbase + lane_off + cb, v0);
                        tmem_ld32(tbase + lane_off + cb + 32, v1);
                        tmem_wait_ld();
                        const uint32_t rowa = scr + lane * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const uint32_t* x = u < 4 ? &v0[8 * u] : &v1[8 * (u - 4)];
                            st_shared_v4(rowa + ((u ^ (lane & 7)) << 4),
                                         pack2<kF16>(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                                         pack2<kF16>(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                                         pack2<kF16>(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                                         pack2<kF16>(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (full_seg)
                                tma_store_3d(&omap, scr, cb, w.g * 128 + q * 32, w.b);
                            else
                                tma_store_3d(&wmap, scr, cb, q * 32, slot);
                            bulk_commit();
                        }
                    }
                    if (lane == 0) bulk_wait_read_all();  // the stage may be refilled after this
                    __syncwarp();
                }
                if (lead && row_ok) {
                    if (full_seg) {
                        if (p.lse) p.lse[(long long)w.b * Mq + grow] = lse_v;
                    } else {
                        p.ws_lse[(long long)slot * 128 + r] =
                            seg_bad ? __int_as_float(0x7fc00000) : lse_v;  // NaN marks bad
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&c.evtdone));
                ++seg;
                if (w.u + 1 >= w.u_end) {
                    done = true;
                } else {
                    walk_next(p, w);
                    seg_tile0 = w.tile;
                }
            }
            if (lane == 0) bulk_wait_all();  // the epilogue's stores are complete
            __syncwarp();
        }
    }

    tc_fence_before();
    __syncwarp();
    cluster_sync();
    tc_fence_after();
    if (warp == 4) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ combine
// Merges the partial segments of row groups that were split across pairs
// (LSE-weighted: out = sum_k exp(lse_k - lse) o_k with lse = log sum_k
// exp(lse_k)) and writes the rows of empty or invalid requests. One CTA per
// (request, row group, 4 * rpt query rows), rpt = 1, 2, 4 or 8 picked by the
// host so that the CTAs holding rows fit in one wave. Thread t takes the eight columns 8 (t % 64) .. + 7
// of rows t / 64 + 4 j (j < rpt), so a warp reads 512 contiguous bytes of one
// partial row. Its (row, part) items are walked row by row, kCombineBatch
// loads in flight at a time, so a request split into a few parts costs one
// memory round trip for all the thread's rows. The parts' LSEs of all the
// CTA's rows are loaded together while the first loads are in flight; eight
// lanes per row then work out its weights.
//
// Launched as a programmatic dependent of the decode kernel: everything up to
// the partials' first read overlaps the decode kernel's tail.
constexpr int kCombineThreads = 256;
constexpr int kCombineBatch = 16;     // loads in flight per thread
constexpr int kCombineMaxRpt = 8;     // rows per thread
constexpr int kCombineMaxParts = 256; // parts per row group (pairs of a set)

__device__ __forceinline__ uint4 load_part(const Params& p, long long slot, int r, int c8) {
    return reinterpret_cast<const uint4*>(p.ws_o + (slot * 128 + r) * 512)[c8];
}

template <bool kF16>
__global__ void __launch_bounds__(kCombineThreads, 2) combine_kernel(const Params p) {
    __shared__ int sh_parts[3];  // first pair, part count, first part's slot offset
    __shared__ float sh_w[4 * kCombineMaxRpt][kCombineMaxParts];
    __shared__ float sh_lse[4 * kCombineMaxRpt];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Mq = p.T * p.H;
    const int G = (Mq + 127) / 128;
    const int rpt = p.combine_rpt;
    const int cr = 4 * rpt;                 // rows per CTA
    const int nq = 128 / cr;                // CTAs per row group
    const int quad = (int)(blockIdx.x % nq);
    const long long bg = blockIdx.x / nq;
    if (bg >= (long long)p.B * G) return;
    const int b = (int)(bg / G), g = (int)(bg % G);
    const int rows = min(128, Mq - g * 128);
    const int row0 = quad * cr;             // the CTA's first row within the group
    if (row0 >= rows) return;               // rows past the group: nothing to do
    const int rr = tid >> 6;                // the thread's rows: row0 + rr + 4 j
    const int c8 = tid & 63;                // eight-column group
    const int S = p.seq_lens[b];
    const int nt = ntiles_of(S, p.T, p.max_blocks);
    const long long orow0 = (long long)b * Mq + g * 128;
    // which pairs hold this row group, from seq_lens alone (as the decode
    // kernel partitions the units); one warp works it out for the CTA
    if (warp == 0 && nt > 0) {
        const split::Parts q = split::request_parts(p, b, g, lane);
        if (lane == 0) {
            sh_parts[0] = q.pf;
            sh_parts[1] = q.nparts;
            sh_parts[2] = q.slot0_off;
        }
    }
    // from here on the decode kernel's results (and the output rows it may
    // also write) are touched: wait for it to complete
    grid_dependency_wait();
    if (nt == 0) {
        if (quad == 0 && g == 0 && tid == 0 && p.dev_err) {
            if (S < 0 || (S > 0 && S < p.T)) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_SEQ_SHORT);
            else if (S > p.max_blocks * 16) atomicOr(p.dev_err, (int32_t)MLA_DEVERR_SEQ_TOO_LONG);
        }
        for (int j = 0; j < rpt; ++j) {
            const int r = row0 + rr + 4 * j;
            if (r < rows) {
                reinterpret_cast<uint4*>(p.out + (orow0 + r) * 512)[c8] = make_uint4(0u, 0u, 0u, 0u);
                if (c8 == 0 && p.lse) p.lse[orow0 + r] = -INFINITY;
            }
        }
        return;
    }
    __syncthreads();
    const int pf = sh_parts[0], nparts = sh_parts[1], slot0_off = sh_parts[2];
    if (nparts <= 1) return;  // one pair held the whole row group and wrote it
    auto slot_of = [&](int k) -> long long {
        return (long long)(pf + k) * 2 + (k == 0 ? slot0_off : 0);
    };
    // the thread's items (row j, part k), f = j * nparts + k; rows past the
    // group are skipped. The first batch is in flight while the weights are
    // worked out.
    const int nitems = rpt * nparts;
    uint4 v[kCombineBatch];
    {
        int j = 0, k = 0;
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) {
            const int r = row0 + rr + 4 * j;
            if (q < nitems && r < rows) v[q] = load_part(p, slot_of(k), r, c8);
            if (++k == nparts) { k = 0; ++j; }
        }
    }
    // the parts' LSEs of the CTA's rows, all at once
    for (int idx = tid; idx < cr * nparts; idx += kCombineThreads) {
        const int cw = idx / nparts, k = idx - cw * nparts;
        const int r = row0 + cw;
        if (r < rows) sh_w[cw][k] = p.ws_lse[slot_of(k) * 128 + r];
    }
    __syncthreads();
    // weights: 8 lanes per row (split::row_weights; the merging decompress of
    // the fused path computes them the same way, bit for bit)
    {
        // a group of 8 lanes per row (rows of a CTA <= 32 = its groups)
        const int grp = tid / split::kWeightLanes, gl = tid % split::kWeightLanes;
        const int r = row0 + grp;
        const bool mine = grp < cr && r < rows;
        const float l = split::row_weights(sh_w[mine ? grp : 0], mine ? nparts : 0, gl);
        if (mine && gl == 0) sh_lse[grp] = l;
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    int j = 0, k = 0;  // the item after the last accumulated one
    for (int f0 = 0; f0 < nitems; f0 += kCombineBatch) {
        if (f0 > 0) {
            int jj = j, kk = k;
#pragma unroll
            for (int q = 0; q < kCombineBatch; ++q) {
                const int r = row0 + rr + 4 * jj;
                if (f0 + q < nitems && r < rows) v[q] = load_part(p, slot_of(kk), r, c8);
                if (++kk == nparts) { kk = 0; ++jj; }
            }
        }
#pragma unroll
        for (int q = 0; q < kCombineBatch; ++q) {
            if (f0 + q < nitems) {
                const int cw = rr + 4 * j;
                const int r = row0 + cw;
                if (r < rows) {
                    const float wk = sh_w[cw][k];
                    const uint32_t u[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] += wk * elem_lo<kF16>(u[e]);
                        acc[2 * e + 1] += wk * elem_hi<kF16>(u[e]);
                    }
                }
                if (++k == nparts) {  // row done: write it
                    if (r < rows) {
                        reinterpret_cast<uint4*>(p.out + (orow0 + r) * 512)[c8] =
                            make_uint4(pack2<kF16>(acc[0], acc[1]), pack2<kF16>(acc[2], acc[3]),
                                       pack2<kF16>(acc[4], acc[5]), pack2<kF16>(acc[6], acc[7]));
                        if (c8 == 0 && p.lse) p.lse[orow0 + r] = sh_lse[cw];
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
                    k = 0;
                    ++j;
                }
            }
        }
    }
}

// ------------------------------------------------------------------ host
struct DeviceInfo {
    int max_pairs = 0;
};
std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !f) return cudaErrorNotSupported;
        g_encode = (PFN_cuTensorMapEncodeTiled_v12000)f;
    }
    *fn = g_encode;
    return cudaSuccess;
}

template <int W, bool kF16>
cudaError_t setup_kernel(int dev, int* max_pairs) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& di = g_dev[dev & 63];
    static bool attr_set[4][64] = {};
    const int wi = (W == 576 ? 0 : 1) + (kF16 ? 2 : 0);
    if (!attr_set[wi][dev & 63]) {
        cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<W, kF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[wi][dev & 63] = true;
    }
    if (di.max_pairs == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel<W, kF16>, &cfg);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorNotSupported;
        di.max_pairs = n < kCombineMaxParts ? n : kCombineMaxParts;
    }
    *max_pairs = di.max_pairs;
    return cudaSuccess;
}

int max_pairs_for(const mla_dims& d, cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return 0;
    int n = 0;
    // the f16 and bf16 instances share one layout, so one occupancy answer
    // serves both; each still gets its shared-memory attribute set
    const bool f16 = d.dtype == MLA_F16;
    if (d.kv_rank + d.d_rope == 576)
        *err = f16 ? setup_kernel<576, true>(dev, &n) : setup_kernel<576, false>(dev, &n);
    else
        *err = f16 ? setup_kernel<512, true>(dev, &n) : setup_kernel<512, false>(dev, &n);
    return n;
}

std::atomic<unsigned long long> g_wait_limit_ns{0};
std::atomic<int> g_stall{0};

}  // namespace

DecodeWaitTest decode_wait_test() {
    return DecodeWaitTest{g_wait_limit_ns.load(), g_stall.load()};
}

void set_decode_wait_test(unsigned long long limit_ns, int stall) {
    g_wait_limit_ns.store(limit_ns);
    g_stall.store(stall ? 1 : 0);
}

bool tc_decode_supported(const mla_dims& d) {
    const int W = d.kv_rank + d.d_rope;
    return (d.dtype == MLA_BF16 || d.dtype == MLA_F16) && d.kv_rank == 512 &&
           (W == 576 || W == 512) &&
           d.block_size == 16 && d.t_q * d.n_head <= 1 << 20;
}

cudaError_t tc_decode_split_info(const mla_dims& d, void* workspace, DecodeSplitInfo* info) {
    cudaError_t e;
    const int np = max_pairs_for(d, &e);
    if (e != cudaSuccess) return e;
    info->NP = np;
    info->min_units = 2;
    info->ws_o = workspace;
    info->ws_lse = (float*)((char*)workspace + (size_t)2 * np * 128 * 512 * sizeof(__nv_bfloat16));
    return cudaSuccess;
}

cudaError_t tc_decode_workspace(int32_t batch, int32_t max_blocks, const mla_dims& d,
                                size_t* bytes) {
    (void)batch;
    (void)max_blocks;
    cudaError_t e;
    const int np = max_pairs_for(d, &e);
    if (e != cudaSuccess) return e;
    const size_t o = (size_t)2 * np * 128 * 512 * sizeof(__nv_bfloat16);
    const size_t l = (size_t)2 * np * 128 * sizeof(float);
    *bytes = o + l;
    return cudaSuccess;
}

cudaError_t launch_decode_tc(void* out, float* lse, const void* q_abs, const void* kv_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             int32_t batch, int32_t max_blocks, int32_t num_blocks,
                             const mla_dims& d, float scale, void* workspace,
                             int32_t* dev_err, cudaStream_t s, bool early, bool combine) {
    const int W = d.kv_rank + d.d_rope;
    if ((long long)batch * max_blocks > (1LL << 33)) {  // unit counts are 32-bit
        set_error("batch * max_blocks = %lld exceeds 2^33", (long long)batch * max_blocks);
        return cudaErrorInvalidValue;
    }
    cudaError_t e;
    const int np = max_pairs_for(d, &e);
    if (e != cudaSuccess) return e;
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    if ((e = get_encode(&enc)) != cudaSuccess) return e;
    const bool f16 = d.dtype == MLA_F16;
    const CUtensorMapDataType tdt = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // the S-CTA's view of the cache: {64 columns, 8 rows, W/64 column chunks,
    // 2 halves of a block, blocks}; one box is a whole block, landing as
    // [half][chunk][8 rows][128 B]
    CUtensorMap tmap;
    const int nkc = W / 64;
    cuuint64_t dims[5] = {64, 8, (cuuint64_t)nkc, 2, (cuuint64_t)num_blocks};
    cuuint64_t strides[4] = {(cuuint64_t)W * 2, 128, (cuuint64_t)8 * W * 2,
                             (cuuint64_t)16 * W * 2};
    cuuint32_t box[5] = {64, 8, (cuuint32_t)nkc, 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult cr = enc(&tmap, tdt, 5, const_cast<void*>(kv_cache),
                      dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (%d)", (int)cr);
        return cudaErrorInvalidValue;
    }
    CUtensorMap qmap;
    {
        // queries as {W columns, t_q * n_head rows, batch}: a 128-row box of one
        // request never reads the next request's rows
        const int Mq = d.t_q * d.n_head;
        cuuint64_t qdims[3] = {(cuuint64_t)W, (cuuint64_t)Mq, (cuuint64_t)batch};
        cuuint64_t qstrides[2] = {(cuuint64_t)W * 2, (cuuint64_t)Mq * W * 2};
        cuuint32_t qbox[3] = {64, (cuuint32_t)(Mq < 128 ? Mq : 128), 1};
        cuuint32_t qes[3] = {1, 1, 1};
        cr = enc(&qmap, tdt, 3, const_cast<void*>(q_abs), qdims,
                 qstrides, qbox, qes, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) {
            set_error("cuTensorMapEncodeTiled (queries) failed (%d)", (int)cr);
            return cudaErrorInvalidValue;
        }
    }
    CUtensorMap vmap;
    {
        // 4-D view of the cache: {64 columns, 16 rows, 8 column chunks, blocks}
        cuuint64_t vdims[4] = {64, 16, 8, (cuuint64_t)num_blocks};
        cuuint64_t vstrides[3] = {(cuuint64_t)W * 2, 128, (cuuint64_t)16 * W * 2};
        cuuint32_t vbox[4] = {64, 16, 8, 1};
        cuuint32_t ves[4] = {1, 1, 1, 1};
        cr = enc(&vmap, tdt, 4, const_cast<void*>(kv_cache), vdims,
                 vstrides, vbox, ves, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) {
            set_error("cuTensorMapEncodeTiled (values) failed (%d)", (int)cr);
            return cudaErrorInvalidValue;
        }
    }
    // epilogue stores: [32 rows x 64 columns] boxes of output rows
    // {512, t_q * n_head, batch} (rows past a request's fall outside) and of
    // the workspace's partial rows {512, 128, 2 * pairs}
    CUtensorMap omap, wmap;
    {
        const int Mq = d.t_q * d.n_head;
        cuuint64_t odims[3] = {512, (cuuint64_t)Mq, (cuuint64_t)batch};
        cuuint64_t ostrides[2] = {512 * 2, (cuuint64_t)Mq * 512 * 2};
        cuuint64_t wdims[3] = {512, 128, (cuuint64_t)2 * np};
        cuuint64_t wstrides[2] = {512 * 2, 128 * 512 * 2};
        cuuint32_t box[3] = {64, 32, 1};
        cuuint32_t es3[3] = {1, 1, 1};
        cr = enc(&omap, tdt, 3, out, odims, ostrides, box, es3,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr == CUDA_SUCCESS)
            cr = enc(&wmap, tdt, 3, workspace, wdims, wstrides, box,
                     es3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) {
            set_error("cuTensorMapEncodeTiled (epilogue stores) failed (%d)", (int)cr);
            return cudaErrorInvalidValue;
        }
    }
    Params p;
    p.q_abs = (const __nv_bfloat16*)q_abs;
    p.kv = (const __nv_bfloat16*)kv_cache;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = (__nv_bfloat16*)out;
    p.lse = lse;
    p.ws_o = (__nv_bfloat16*)workspace;
    p.ws_lse = (float*)((char*)workspace + (size_t)2 * np * 128 * 512 * sizeof(__nv_bfloat16));
    p.dev_err = dev_err;
    p.B = batch;
    p.T = d.t_q;
    p.H = d.n_head;
    p.W = W;
    p.max_blocks = max_blocks;
    p.num_blocks = num_blocks;
    p.NP = np;
    p.min_units = 2;  // as tc_decode_split_info reports
    p.combine_rpt = 1;
    p.early = early ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    {
        const DecodeWaitTest t = decode_wait_test();
        p.wait_ns = t.limit_ns ? t.limit_ns : kWaitLimit;
        p.stall = t.stall;
    }

    // a programmatic dependent of the kernel before it: the cache pipeline
    // starts while that kernel finishes; the queries, and every write, wait
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * np, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (W == 576)
        e = f16 ? cudaLaunchKernelEx(&cfg, decode_pair_kernel<576, true>, tmap, qmap, vmap, omap,
                                     wmap, p)
                : cudaLaunchKernelEx(&cfg, decode_pair_kernel<576, false>, tmap, qmap, vmap, omap,
                                     wmap, p);
    else
        e = f16 ? cudaLaunchKernelEx(&cfg, decode_pair_kernel<512, true>, tmap, qmap, vmap, omap,
                                     wmap, p)
                : cudaLaunchKernelEx(&cfg, decode_pair_kernel<512, false>, tmap, qmap, vmap, omap,
                                     wmap, p);
    if (e != cudaSuccess) return e;
    if (!combine) return cudaGetLastError();
    const long long G = (d.t_q * d.n_head + 127) / 128;
    cudaLaunchConfig_t ccfg = {};
    cudaLaunchAttribute cattr[1];
    cattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    cattr[0].val.programmaticStreamSerializationAllowed = 1;
    // rows per combine thread: one while a single wave of CTAs (two per SM,
    // four rows each) covers every row, more for larger batches
    {
        const int rows = d.t_q * d.n_head < 128 ? d.t_q * d.n_head : 128;
        const long long wave = 2LL * 2 * np;  // two CTAs per SM, two SMs per pair
        int rpt = 1;
        while (rpt < kCombineMaxRpt &&
               (long long)batch * G * ((rows + 4 * rpt - 1) / (4 * rpt)) > wave)
            rpt *= 2;
        p.combine_rpt = rpt;
    }
    ccfg.gridDim = dim3((unsigned)((long long)batch * G * (128 / (4 * p.combine_rpt))), 1, 1);
    ccfg.blockDim = dim3(kCombineThreads, 1, 1);
    ccfg.dynamicSmemBytes = 0;
    ccfg.stream = s;
    ccfg.attrs = cattr;
    ccfg.numAttrs = 1;
    e = f16 ? cudaLaunchKernelEx(&ccfg, combine_kernel<true>, p)
            : cudaLaunchKernelEx(&ccfg, combine_kernel<false>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mla
