// Host build of the tensor-core decode's work-split arithmetic, for the CPU
// tests (tests/test_split_host.py). It compiles csrc/tc_split.cuh with the
// CUDA qualifiers defined away and exports the header's scalar functions
// through plain C entry points. The warp-cooperative functions of the header
// (shuffles, votes) are declared here but never defined: the shim is linked
// with --no-undefined, so a scalar function that reached one would fail to
// link instead of running on a made-up warp.
#include <algorithm>
#include <stdint.h>

#define __device__
#define __forceinline__ inline

using std::max;
int __shfl_up_sync(unsigned, int, int);
int __shfl_sync(unsigned, int, int);
int __any_sync(unsigned, int);
int __shfl_xor_sync(unsigned, int, int, int = 32);
float __shfl_xor_sync(unsigned, float, int, int = 32);

#include "tc_split.cuh"

namespace {
struct Shape {
    int NP, min_units;
};
void put(const mla::split::Parts& q, int* out) {
    out[0] = q.pf;
    out[1] = q.nparts;
    out[2] = q.slot0_off;
    out[3] = q.nt;
}
}  // namespace

extern "C" {

int shim_ntiles_of(int S, int T, int max_blocks) {
    return mla::split::ntiles_of(S, T, max_blocks);
}
int shim_pooled_split(int NP, int min_units, int G) {
    return mla::split::pooled_split(Shape{NP, min_units}, G) ? 1 : 0;
}
int shim_pooled_pairs(int NP, int min_units, int G, long long U) {
    return mla::split::pooled_pairs(Shape{NP, min_units}, G, U);
}
int shim_pairs_per_set(int NP, int min_units, int G, long long U) {
    return mla::split::pairs_per_set(Shape{NP, min_units}, G, U);
}
int shim_aligned_tried(long long U, int np_g) {
    return mla::split::aligned_tried(U, np_g) ? 1 : 0;
}
int shim_aligned_first_pair(long long prefix, long long U, int np_g) {
    return mla::split::aligned_first_pair(prefix, U, np_g);
}
void shim_parts_from(int before, int nt, int U, int np_g, int aligned, int g, int* out) {
    put(mla::split::parts_from(before, nt, U, np_g, aligned != 0, g), out);
}
void shim_parts_pooled(int before, int nt, int U, int G, int np, int g, int* out) {
    put(mla::split::parts_pooled(before, nt, U, G, np, g), out);
}
long long shim_part_slot(int pf, int nparts, int slot0_off, int nt, int k) {
    mla::split::Parts q;
    q.pf = pf;
    q.nparts = nparts;
    q.slot0_off = slot0_off;
    q.nt = nt;
    return mla::split::part_slot(q, k);
}

}  // extern "C"
