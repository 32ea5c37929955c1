// Work split of the tensor-core decode, shared by the kernels that need to
// know it: the decode itself (which pair takes which cache tiles), the
// combine and the decompress that merges the split partial results (which
// pairs hold the parts of a request).
//
// Units are (request, 64-token tile) pairs. When a request has G > 1 row
// groups (t_q * n_head > 128), the pairs form G sets of np_g: set g handles
// row group g of every request, and pair k of each set covers the same
// (request, tile) range. Within a set the unit sequence is request b, then
// tile, U units in all. Two splits of that sequence exist:
//   even     pair k takes units [U k / np_g, U (k + 1) / np_g);
//   aligned  request b (tiles_b units, prefix_b before it) gets the pairs
//            [P_b, P_{b+1}), P_b = round(np_g prefix_b / U), and its units
//            evenly among them, so no pair holds two segments.
// The aligned split is used when every non-empty request gets a pair and no
// pair gets more than two tiles above the even split's ceil(U / np_g) (a
// pair holding two partial segments costs more than that: an extra epilogue
// and a query reload); it is only tried while a pair's share is small and
// the arithmetic fits 32 bits.
//
// A pair writes at most two partial segments, into workspace slots
// 2 pair + 0 (its first segment) and 2 pair + 1 (its last one).
//
// Every function taking a params object reads its fields seq_lens, B, T, H,
// max_blocks, NP (pairs of the grid) and min_units (fewest units a pair of a
// small problem gets).
#pragma once

#include <math.h>
#include <stdint.h>

namespace mla {
namespace split {

constexpr int kTok = 64;               // cache tokens per unit
constexpr int kAlignedMaxShare = 32;   // tiles per pair up to which the aligned split is tried

// tiles of a request with S cached tokens; 0 for an empty or invalid request
__device__ __forceinline__ int ntiles_of(int S, int T, int max_blocks) {
    if (S <= 0 || S < T || S > max_blocks * 16) return 0;
    return (S + kTok - 1) / kTok;
}

// pairs per set (np_g) and the set size cap
// Pooled split: when the G sets would share the pairs unevenly (G does not
// divide the pairs, or exceeds them), the sets' units are numbered one after
// the other (set g's unit i is g U + i) and pair k takes the even share
// [G U k / np, G U (k + 1) / np) of all of them, walking on into the next set.
// A set ends with a request's last tile, so a pair still holds at most two
// partial segments: its first and its last.
template <class P>
__device__ __forceinline__ bool pooled_split(const P& p, int G) {
    return G > 1 && (G > p.NP || p.NP % G != 0);
}
template <class P>
__device__ __forceinline__ int pooled_pairs(const P& p, int G, long long U) {
    const long long cap = ((long long)G * U + p.min_units - 1) / p.min_units;
    return (int)(cap < p.NP ? cap : p.NP);
}

template <class P>
__device__ __forceinline__ int pairs_per_set(const P& p, int G, long long U) {
    int np_g = p.NP / G;
    if (np_g < 1) np_g = 1;
    const long long cap = (U + p.min_units - 1) / p.min_units;
    if (cap < np_g) np_g = (int)(cap > 0 ? cap : 1);
    return np_g;
}

// One chunk of 32 requests, warp-cooperative: lane l holds request b0 + l's
// units v (0 past the batch), its seq_len S, and the inclusive prefix of v
// within the chunk; total is the chunk's sum. Unit counts fit 32 bits (the
// host requires batch * ceil(max_blocks / 4) < 2^31).
struct ChunkScan {
    int v, S, incl, total;
};
template <class P>
__device__ __forceinline__ ChunkScan scan_chunk(const P& p, int b0, int lane) {
    const int b = b0 + lane;
    ChunkScan c;
    c.S = b < p.B ? p.seq_lens[b] : 0;
    c.v = b < p.B ? ntiles_of(c.S, p.T, p.max_blocks) : 0;
    c.incl = c.v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, c.incl, o);
        if (lane >= o) c.incl += t;
    }
    c.total = __shfl_sync(0xffffffffu, c.incl, 31);
    return c;
}

__device__ __forceinline__ bool aligned_tried(long long U, int np_g) {
    return U <= (long long)kAlignedMaxShare * np_g && 2 * (long long)np_g * U + U < (1LL << 31);
}
// P_b for the units before a request
__device__ __forceinline__ int aligned_first_pair(long long prefix, long long U, int np_g) {
    return (int)((2u * (uint32_t)np_g * (uint32_t)prefix + (uint32_t)U) / (2u * (uint32_t)U));
}
// per chunk: lanes whose request gets no pair (bad) and the largest share
__device__ __forceinline__ void aligned_check(const ChunkScan& c, int base, long long U, int np_g,
                                              int& bad, int& worst) {
    const int n = aligned_first_pair(base + c.incl, U, np_g) -
                  aligned_first_pair(base + c.incl - c.v, U, np_g);
    if (c.v > 0) {
        if (n <= 0) bad = 1;
        else worst = max(worst, (int)(((uint32_t)c.v + (uint32_t)n - 1u) / (uint32_t)n));
    }
}
__device__ __forceinline__ bool aligned_decide(int bad, int worst, long long U, int np_g) {
    bad = __any_sync(0xffffffffu, bad);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) worst = max(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    return !bad && worst <= (U + np_g - 1) / np_g + 2;
}

// The parts of one row group: pairs pf .. pf + nparts - 1 (global indices)
// hold its partial segments; part 0 sits in its pair's slot 2 pf + slot0_off,
// every later part k in slot 2 (pf + k). nt is the request's unit count. With
// nparts == 1 the pair wrote the rows themselves, not a partial segment.
struct Parts {
    int pf, nparts, slot0_off, nt;
};
__device__ __forceinline__ long long part_slot(const Parts& q, int k) {
    return (long long)(q.pf + k) * 2 + (k == 0 ? q.slot0_off : 0);
}

// The parts of a request with nt > 0 units, `before` units ahead of it in its
// set, given the set's total U, its pairs np_g and the split in use.
__device__ __forceinline__ Parts parts_from(int before, int nt, int U, int np_g, bool aligned,
                                            int g) {
    Parts q;
    q.nt = nt;
    if (aligned) {
        // the request's own pairs, each holding one segment of it
        const int pb = aligned_first_pair(before, U, np_g);
        const int pe = aligned_first_pair(before + nt, U, np_g);
        q.pf = g * np_g + pb;
        q.nparts = pe - pb;
        q.slot0_off = 0;
    } else {
        const long long u0 = before, u1 = u0 + nt;  // within row group g's set
        auto owner = [&](long long u) {  // pair of the set whose range holds unit u
            long long pp = (u * np_g) / U;
            while (pp + 1 < np_g && (long long)U * (pp + 1) / np_g <= u) ++pp;
            while (pp > 0 && (long long)U * pp / np_g > u) --pp;
            return (int)pp;
        };
        const int kf = owner(u0), kl = owner(u1 - 1);
        q.pf = g * np_g + kf;
        q.nparts = kl - kf + 1;
        // part 0 is pair kf's first segment when its range starts at u0, else
        // its last one; every later part is that pair's first segment
        q.slot0_off = ((long long)U * kf / np_g) >= u0 ? 0 : 1;
    }
    return q;
}

// The parts of a request under the pooled split: its units are g U + before
// .. + nt - 1 of the G U pooled units, shared by np pairs as evenly as the
// even split shares a set's.
__device__ __forceinline__ Parts parts_pooled(int before, int nt, int U, int G, int np, int g) {
    Parts q;
    q.nt = nt;
    const long long T = (long long)G * U;
    const long long u0 = (long long)g * U + before, u1 = u0 + nt;
    auto owner = [&](long long u) {
        long long pp = (u * np) / T;
        while (pp + 1 < np && T * (pp + 1) / np <= u) ++pp;
        while (pp > 0 && T * pp / np > u) --pp;
        return (int)pp;
    };
    const int kf = owner(u0), kl = owner(u1 - 1);
    q.pf = kf;
    q.nparts = kl - kf + 1;
    q.slot0_off = (T * kf / np) >= u0 ? 0 : 1;
    return q;
}

// Warp-cooperative: the set's unit total U, its pairs np_g and whether the
// aligned split is in use (every lane gets the same answer).
struct SplitShape {
    int U, np_g;
    bool aligned;
    bool pooled;   // pooled split over np_all pairs
    int G, np_all;
};
template <class P>
__device__ SplitShape split_shape(const P& p, int lane) {
    const int G = (p.T * p.H + 127) / 128;
    SplitShape sh;
    sh.U = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) sh.U += scan_chunk(p, b0, lane).total;
    sh.np_g = sh.U > 0 ? pairs_per_set(p, G, sh.U) : 1;
    sh.aligned = false;
    sh.G = G;
    sh.pooled = pooled_split(p, G);
    sh.np_all = sh.U > 0 ? pooled_pairs(p, G, sh.U) : 1;
    if (sh.pooled) return sh;
    if (sh.U > 0 && aligned_tried(sh.U, sh.np_g)) {
        int base = 0, worst = 0, bad = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const ChunkScan c = scan_chunk(p, b0, lane);
            aligned_check(c, base, sh.U, sh.np_g, bad, worst);
            base += c.total;
        }
        sh.aligned = aligned_decide(bad, worst, sh.U, sh.np_g);
    }
    return sh;
}

// Warp-cooperative: the parts of request b's row group g (every lane gets
// the same answer). nparts is 0 for an empty or invalid request.
// the parts of a request of row group g under the split in use
__device__ __forceinline__ Parts parts_of(const SplitShape& sh, int before, int nt, int g) {
    return sh.pooled ? parts_pooled(before, nt, sh.U, sh.G, sh.np_all, g)
                     : parts_from(before, nt, sh.U, sh.np_g, sh.aligned, g);
}

template <class P>
__device__ Parts request_parts(const P& p, int b, int g, int lane) {
    Parts q;
    q.pf = 0;
    q.nparts = 0;
    q.slot0_off = 0;
    q.nt = 0;
    int U = 0, before = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const ChunkScan c = scan_chunk(p, b0, lane);
        if (b >= b0 && b < b0 + 32) {
            const int l = b - b0;
            q.nt = __shfl_sync(0xffffffffu, c.v, l);
            before = U + __shfl_sync(0xffffffffu, c.incl - c.v, l);
        }
        U += c.total;
    }
    if (q.nt == 0) return q;
    const SplitShape sh = split_shape(p, lane);
    return parts_of(sh, before, q.nt, g);
}

// The merge weights of one row, by a group of 8 adjacent lanes: w holds the
// parts' LSEs (natural log; NaN marks a part that met an invalid block id)
// and gets w_k = exp(lse_k - max) / sum; the row's LSE is returned in every
// lane of the group (-inf for an empty or voided row, whose weights are 0).
// Lane j of the group takes parts j, j + 8, ... and sums them in that order;
// the group then adds its lanes' sums by an xor butterfly (4, 2, 1). The
// combine and the merging decompress both call this with the same grouping,
// so they agree bit for bit. Every lane of the warp must call it (the
// shuffles span the warp); a group with nothing to do passes np = 0.
constexpr int kWeightLanes = 8;
__device__ __forceinline__ float row_weights(float* w, int np, int gl) {
    float m = -INFINITY;
    int bad = 0;
    for (int k = gl; k < np; k += kWeightLanes) {
        const float l = w[k];
        bad |= (l != l);
        m = fmaxf(m, l);
    }
#pragma unroll
    for (int o = kWeightLanes / 2; o > 0; o >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o, kWeightLanes));
        bad |= __shfl_xor_sync(0xffffffffu, bad, o, kWeightLanes);
    }
    float sum = 0.f;
    for (int k = gl; k < np; k += kWeightLanes) {
        const float l = w[k];
        const float e = (l == -INFINITY || m == -INFINITY) ? 0.f : expf(l - m);
        w[k] = e;
        sum += e;
    }
#pragma unroll
    for (int o = kWeightLanes / 2; o > 0; o >>= 1)
        sum += __shfl_xor_sync(0xffffffffu, sum, o, kWeightLanes);
    const bool empty = bad || !(sum > 0.f);
    const float inv = empty ? 0.f : 1.f / sum;
    for (int k = gl; k < np; k += kWeightLanes) w[k] *= inv;
    return empty ? -INFINITY : m + logf(sum);
}

}  // namespace split
}  // namespace mla
