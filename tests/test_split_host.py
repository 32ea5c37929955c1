"""The tensor-core decode's work split, on the CPU.

The split (csrc/tc_split.cuh) decides which CTA pair of the decode takes which
(request, 64-token tile) units, and from it the combine and the merging
decompress find the partial segments of each request's rows. Its scalar
functions are compiled here for the host (tests/split_shim.cpp) and checked
against a brute-force reading of the split as the header states it:

  units       (request b, tile) pairs, ntiles = ceil(S / 64) for a valid
              request (T <= S <= max_blocks * 16), else none; U per set;
  sets        G = ceil(t_q * n_head / 128) row groups; with G == 1, or G
              dividing the pairs, set g takes np_g = min(NP / G,
              ceil(U / min_units)) pairs (at least 1), pairs g np_g .. ;
  even        pair k of a set takes units [U k / np_g, U (k + 1) / np_g);
  aligned     request b gets pairs [P_b, P_b+1), P_b = round(np_g prefix_b
              / U), its units split evenly over them; used when it is tried
              (U <= 32 np_g, 32-bit arithmetic), every non-empty request
              gets a pair and no pair gets more than ceil(U / np_g) + 2;
  pooled      otherwise (G > 1 not dividing the pairs, or G > NP): all G U
              units numbered set after set, np = min(NP, ceil(G U /
              min_units)) pairs, pair k taking [G U k / np, G U (k+1) / np);
  slots       a pair writes its first partial segment to workspace slot
              2 pair and its last to 2 pair + 1; a request held by one pair
              is written as rows, not as a partial segment.

The brute force walks every pair's units, cuts them into (set, request)
segments and derives each request's parts and slots from that walk; the
header's parts functions must give the same answer. The stated invariants are
checked on the way: a pair holds at most two partial segments (its first and
last), no two segments share a slot, and no pair index reaches NP.
"""
import bisect
import ctypes
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mla_latent_cache_absorbed_gb300", "csrc")

TOK = 64
ALIGNED_MAX_SHARE = 32


@pytest.fixture(scope="module")
def shim(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    so = str(tmp_path_factory.mktemp("split") / "split_shim.so")
    subprocess.run([cxx, "-O1", "-std=c++17", "-shared", "-fPIC", "-Wl,--no-undefined",
                    "-Wno-unknown-pragmas", "-I", CSRC, os.path.join(HERE, "split_shim.cpp"),
                    "-o", so], check=True)
    lib = ctypes.CDLL(so)
    I, LL, P = ctypes.c_int, ctypes.c_longlong, ctypes.POINTER(ctypes.c_int)
    for name, args, res in [
            ("shim_ntiles_of", [I, I, I], I),
            ("shim_pooled_split", [I, I, I], I),
            ("shim_pooled_pairs", [I, I, I, LL], I),
            ("shim_pairs_per_set", [I, I, I, LL], I),
            ("shim_aligned_tried", [LL, I], I),
            ("shim_aligned_first_pair", [LL, LL, I], I),
            ("shim_parts_from", [I, I, I, I, I, I, P], None),
            ("shim_parts_pooled", [I, I, I, I, I, I, P], None),
            ("shim_part_slot", [I, I, I, I, I], LL)]:
        f = getattr(lib, name)
        f.argtypes, f.restype = args, res
    return lib


def parts_of(lib, pooled, before, nt, U, G, n, aligned, g):
    out = (ctypes.c_int * 4)()
    if pooled:
        lib.shim_parts_pooled(before, nt, U, G, n, g, out)
    else:
        lib.shim_parts_from(before, nt, U, n, 1 if aligned else 0, g, out)
    pf, nparts, slot0_off, ntq = out
    assert ntq == nt
    slots = [lib.shim_part_slot(pf, nparts, slot0_off, nt, k) for k in range(nparts)]
    return pf, nparts, slots


# ---------------------------------------------------------------- brute force

def ntiles(S, T, max_blocks):
    if S <= 0 or S < T or S > max_blocks * 16:
        return 0
    return -(-S // TOK)


def split_plan(seq_lens, T, H, NP, min_units, max_blocks, force=None, variant=None):
    """The split as stated: per pair, its list of (set, unit range within the
    set) pieces, plus the shape (pooled, G, pairs, aligned). force picks the
    within-set split ("even" or "aligned") instead of the stated decision;
    variant plants a mistake in this statement (for the test of the checks)."""
    nt = [ntiles(S, T, max_blocks) for S in seq_lens]
    U = sum(nt)
    G = -(-(T * H) // 128)
    prefix = [0]
    for v in nt:
        prefix.append(prefix[-1] + v)
    shape = dict(nt=nt, U=U, G=G, prefix=prefix)
    if U == 0:
        return shape, {}
    pooled = G > 1 and (G > NP or NP % G != 0)
    shape["pooled"] = pooled
    ranges = {}   # global pair -> list of (g, unit_begin, unit_end) within set g
    if pooled:
        n = NP if variant == "pooled_no_cap" else min(NP, -(-(G * U) // min_units))
        shape["n"] = n
        shape["aligned"] = False
        for k in range(n):
            a, e = G * U * k // n, G * U * (k + 1) // n
            if variant == "pooled_ceil":
                a, e = -(-(G * U * k) // n), -(-(G * U * (k + 1)) // n)
            pieces = []
            while a < e:
                g = a // U
                end = min(e, (g + 1) * U)
                pieces.append((g, a - g * U, end - g * U))
                a = end
            if pieces:
                ranges[k] = pieces
        return shape, ranges
    np_g = max(1, min(NP // G, -(-U // min_units)))
    shape["n"] = np_g
    # aligned: P_b = round half up (np_g prefix_b / U), exactly
    if variant == "aligned_floor":
        P = [np_g * pr // U for pr in prefix]
    else:
        P = [(2 * np_g * pr + U) // (2 * U) for pr in prefix]
    tried = U <= ALIGNED_MAX_SHARE * np_g and 2 * np_g * U + U < 2 ** 31
    bad = any(v > 0 and P[b + 1] - P[b] <= 0 for b, v in enumerate(nt))
    worst = max((-(-v // (P[b + 1] - P[b])) for b, v in enumerate(nt)
                 if v > 0 and P[b + 1] > P[b]), default=0)
    aligned = tried and not bad and worst <= -(-U // np_g) + 2
    if force == "even":
        aligned = False
    elif force == "aligned":
        if bad:
            return None, None
        aligned = True
    shape["aligned"] = aligned
    shape["P"] = P
    for g in range(G):
        if aligned:
            for b, v in enumerate(nt):
                npairs = P[b + 1] - P[b]
                for j in range(npairs):
                    a = prefix[b] + v * j // npairs
                    e = prefix[b] + v * (j + 1) // npairs
                    if a < e:
                        ranges.setdefault(g * np_g + P[b] + j, []).append((g, a, e))
        else:
            for k in range(np_g):
                a, e = U * k // np_g, U * (k + 1) // np_g
                if variant == "even_ceil":
                    a, e = -(-(U * k) // np_g), -(-(U * (k + 1)) // np_g)
                if a < e:
                    ranges[g * np_g + k] = [(g, a, e)]
    return shape, ranges


def segments(shape, ranges, variant=None):
    """Walk every pair's units in order and cut them into (set, request)
    segments. Returns, for each (set, request), the pairs holding it in walk
    order and the slot each writes (None for a request held whole)."""
    nt, prefix = shape["nt"], shape["prefix"]
    holders = {}   # (g, b) -> [(pair, slot or None)]
    for pair in sorted(ranges):
        segs = []
        for g, a, e in ranges[pair]:
            b = bisect.bisect_right(prefix, a) - 1
            while a < e:
                while nt[b] == 0:
                    b += 1
                end = min(e, prefix[b + 1])
                whole = a == prefix[b] and end == prefix[b + 1]
                segs.append((g, b, whole))
                a = end
                b += 1
        for i, (g, b, whole) in enumerate(segs):
            slot = None
            if not whole:
                # a partial segment is the pair's first or its last, no other
                assert i == 0 or i == len(segs) - 1, (pair, segs)
                first = (i == 0) != (variant == "slots_swapped")
                slot = 2 * pair + (0 if first else 1)
            holders.setdefault((g, b), []).append((pair, slot))
    return holders


def check_case(lib, seq_lens, T, H, NP, min_units, max_blocks, force=None, variant=None,
               stats=None):
    """Compare the header's split functions with the brute force on one
    batch; returns the number of (set, request) parts compared."""
    shape, ranges = split_plan(seq_lens, T, H, NP, min_units, max_blocks, force, variant)
    if shape is None:
        return 0
    nt, U, G, prefix = shape["nt"], shape["U"], shape["G"], shape["prefix"]
    for S, v in zip(seq_lens, nt):
        assert lib.shim_ntiles_of(int(S), T, max_blocks) == v
    if U == 0:
        return 0
    pooled = shape["pooled"]
    assert lib.shim_pooled_split(NP, min_units, G) == int(pooled)
    if pooled:
        assert lib.shim_pooled_pairs(NP, min_units, G, U) == shape["n"]
    else:
        assert lib.shim_pairs_per_set(NP, min_units, G, U) == shape["n"]
        assert G * shape["n"] <= NP
        assert lib.shim_aligned_tried(U, shape["n"]) == int(
            U <= ALIGNED_MAX_SHARE * shape["n"] and 2 * shape["n"] * U + U < 2 ** 31)
        for pr, want in zip(prefix, shape["P"]):
            assert lib.shim_aligned_first_pair(pr, U, shape["n"]) == want
    assert all(0 <= p < NP for p in ranges)
    # every unit of every set is taken exactly once
    count = np.zeros((G, U), np.int32)
    for pieces in ranges.values():
        for g, a, e in pieces:
            count[g, a:e] += 1
    assert (count == 1).all()
    holders = segments(shape, ranges, variant)
    slots_seen = set()
    checked = 0
    for g in range(G):
        for b, v in enumerate(nt):
            if v == 0:
                continue
            pf, nparts, slots = parts_of(lib, pooled, prefix[b], v, U, G, shape["n"],
                                         shape["aligned"], g)
            held = holders[(g, b)]
            pairs = [p for p, _ in held]
            assert pairs == list(range(pf, pf + nparts)), (g, b, pf, nparts, pairs)
            if nparts > 1:
                assert slots == [s for _, s in held], (g, b, slots, held)
                for s in slots:
                    assert s not in slots_seen and s < 2 * NP
                    slots_seen.add(s)
            else:
                assert held[0][1] is None
            if stats is not None:
                stats["pooled"] += pooled
                stats["aligned"] += shape["aligned"]
                stats["even"] += not pooled and not shape["aligned"]
                stats["split3"] += nparts >= 3
                stats["slot1"] += nparts > 1 and slots[0] % 2 == 1
                stats["cross_set"] += pooled and any(len(ranges[p]) > 1 for p in pairs)
            checked += 1
    return checked


# ---------------------------------------------------------------- cases

def lens_mix(rng, B, T, max_blocks):
    """Ragged seq_lens: mostly valid, with empty, too-short (S < t_q) and
    over-long (past the block table) requests mixed in."""
    cap = max_blocks * 16
    S = rng.integers(min(max(T, 1), cap), cap + 1, size=B)
    r = rng.random(B)
    S[r < 0.08] = 0
    if T > 1:
        S[(r >= 0.08) & (r < 0.12)] = T - 1
    S[(r >= 0.12) & (r < 0.15)] = cap + 1
    return [int(x) for x in S]


GEOMS = [  # (t_q, n_head): G = 1, 2, 4, 5, 10, 40, 80, 160, 128 row groups
    (1, 64), (1, 128), (4, 64), (8, 64), (10, 64), (20, 64), (80, 64), (160, 64), (320, 64),
    (5, 128), (128, 128)]


def random_cases(seed, n, geoms=GEOMS, nps=(76, 75, 74, 64, 17, 3, 2, 1)):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        T, H = geoms[int(rng.integers(len(geoms)))]
        G = -(-(T * H) // 128)
        NP = int(rng.choice(nps))
        B = int(rng.choice([1, 2, 5, 8, 33, 64, 130]))
        max_blocks = int(rng.choice([1, 4, 16, 64, 256]))
        # keep G * U (units over all sets) small enough for the brute force
        while max_blocks > 1 and B * max_blocks * 16 // TOK * G > 200_000:
            max_blocks //= 2
        yield lens_mix(rng, B, T, max_blocks), T, H, NP, 2, max_blocks


def test_split_matches_its_statement(shim):
    stats = dict.fromkeys(["pooled", "aligned", "even", "split3", "slot1", "cross_set"], 0)
    total = 0
    for case in random_cases(1234, 400):
        total += check_case(shim, *case, stats=stats)
    assert total > 1000
    # the cases reach every branch of the split
    assert all(v > 0 for v in stats.values()), stats


@pytest.mark.parametrize("force", ["even", "aligned"])
def test_both_within_set_splits(shim, force):
    """parts_from under either within-set split, whichever the decision
    would pick (the aligned one wherever every request gets a pair)."""
    total = 0
    for case in random_cases(7 if force == "even" else 8, 300,
                             geoms=[(1, 64), (1, 128), (4, 64), (2, 64)],
                             nps=(76, 38, 19, 8, 4)):
        total += check_case(shim, *case, force=force)
    assert total > 0


def test_degenerate_shapes(shim):
    """One tile in all, one request, every request empty, min_units above the
    total, one pair, a single long request over every pair."""
    cases = [
        ([1], 1, 64, 76, 2, 1),
        ([64], 1, 64, 76, 2, 4),
        ([65], 1, 64, 76, 2, 8),
        ([0, 0, 0], 1, 64, 76, 2, 4),
        ([3, 0, 5], 4, 64, 76, 2, 4),      # the first request too short for t_q
        ([16 * 4096], 1, 64, 76, 2, 4096),  # one request over all pairs
        ([16 * 4096], 4, 64, 76, 2, 4096),
        ([16 * 4096], 320, 64, 76, 2, 4096),
        ([100, 200, 300], 1, 64, 1, 2, 32),
        ([100, 200, 300], 80, 64, 1, 2, 32),
        ([1000] * 7, 1, 64, 76, 50, 64),
        ([1000] * 7, 10, 64, 76, 3, 64),
    ]
    for seq_lens, T, H, NP, min_units, max_blocks in cases:
        check_case(shim, seq_lens, T, H, NP, min_units, max_blocks)
        check_case(shim, seq_lens, T, H, NP, min_units, max_blocks, force="even")


@pytest.mark.parametrize("variant", ["even_ceil", "aligned_floor", "pooled_no_cap",
                                     "pooled_ceil", "slots_swapped"])
def test_checks_catch_a_misstated_split(shim, variant):
    """The comparison has teeth: the brute force with one plausible mistake
    planted in its statement of the split (ranges rounded up, P_b rounded
    down, the pooled pairs not capped by min_units, first and last slots
    swapped) disagrees with the header on some of the random cases."""
    caught = 0
    for case in random_cases(99, 60):
        try:
            check_case(shim, *case, variant=variant)
        except AssertionError:
            caught += 1
    assert caught > 0
