"""The index and bit arithmetic the score and selection kernels rely on,
restated in Python from the kernels' algorithms and checked against plain
definitions (the GPU parity tests check the kernels themselves):

- keep test: order_key(x) >= t_lo is one unsigned compare on the raw FP32
  bits, (u - lo) <= span, for every threshold that can occur (the start of
  any of the 4096 top-12-bit bins);
- float keep test (prefill selection): for the same thresholds and every
  finite score x, order_key(x) >= t_lo exactly when x >= key_floor(t_lo) as
  an IEEE compare (so -0 and +0 agree), key_floor giving -inf below the key
  of -FLT_MAX;
- unit search: a warp probing 32 tile prefixes per round trip finds the same
  (token, tile) as a scalar binary search;
- look-ahead: 32 consecutive tiles' tokens found from one load of the next
  32 token boundaries and a shuffle search, with the batch-to-batch hand-off
  the producer uses, including tokens with no tiles.
"""
import random

import numpy as np

M32 = 0xFFFFFFFF


def order_key(u):
    """Order-preserving key of the FP32 bit pattern u (-0 as +0)."""
    u = np.asarray(u, dtype=np.uint64)
    u = np.where((u << np.uint64(1)) & np.uint64(M32) == 0, np.uint64(0), u)
    neg = (u & np.uint64(0x80000000)) != 0
    return np.where(neg, (~u) & np.uint64(M32), u | np.uint64(0x80000000))


def keep_range(t_lo):
    if t_lo >= 0x80000000:
        lo = t_lo - 0x80000000
        span = 0x80000000 if lo == 0 else 0x7FFFFFFF - lo
    else:
        lo, span = 0, (~t_lo) & M32
    return lo, span


def test_keep_range_equals_the_key_compare():
    rng = np.random.default_rng(0)
    u = np.concatenate([rng.integers(0, 1 << 32, 200000, dtype=np.uint64),
                        np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFFFFFFF,
                                  1, 0x80000001, 0x7FFFFFFF], dtype=np.uint64)])
    k = order_key(u)
    for b in range(4096):
        t_lo = b << 20
        lo, span = keep_range(t_lo)
        fast = ((u - np.uint64(lo)) & np.uint64(M32)) <= np.uint64(span)
        assert np.array_equal(fast, k >= np.uint64(t_lo)), b


def key_floor(key):
    """The smallest score of key >= `key` on a bin boundary: the inverse of
    order_key, -inf below the key of -FLT_MAX."""
    if key < 0x00800000:
        return np.float32(-np.inf)
    bits = (key & 0x7FFFFFFF) if key & 0x80000000 else (~key) & M32
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def test_float_compare_equals_the_key_compare():
    rng = np.random.default_rng(1)
    u = np.concatenate([rng.integers(0, 1 << 32, 200000, dtype=np.uint64),
                        np.array([0, 0x80000000, 0x7F7FFFFF, 0xFF7FFFFF, 1, 0x80000001,
                                  0x00800000, 0x80800000, 0x7F800000, 0xFF800000], dtype=np.uint64)])
    x = u.astype(np.uint32).view(np.float32)
    finite = ~np.isnan(x)
    u, x = u[finite], x[finite]
    k = order_key(u)
    for b in range(4096):
        t_lo = b << 20
        f_p = key_floor(t_lo)      # NaN above the key of +inf: nothing passes
        assert np.array_equal(x >= f_p, k >= np.uint64(t_lo)), b


def scalar_search(us, T, u):
    lo, hi = 0, T - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if us[mid] <= u:
            lo = mid
        else:
            hi = mid - 1
    return lo, u - us[lo]


def warp_search(us, T, u):
    lo, hi = 0, T
    while hi - lo > 1:
        step = (hi - lo + 31) >> 5
        n = sum(1 for lane in range(32)
                if lo + (lane + 1) * step < hi and us[lo + (lane + 1) * step] <= u)
        lo += n * step
        hi = min(hi, lo + step)
    return lo, u - us[lo]


def shuffle_count(nb, uj):
    n = 0
    for w in (16, 8, 4, 2, 1):
        if nb[n + w - 1] <= uj:
            n += w
    if nb[n] <= uj:
        n += 1
    return n


def layouts(seed, count):
    rng = random.Random(seed)
    for _ in range(count):
        T = rng.randint(1, 700)
        tiles = [rng.randint(0, 5) if rng.random() < 0.5 else rng.randint(0, 300) for _ in range(T)]
        if rng.random() < 0.3:
            tiles = [t if rng.random() < 0.5 else 0 for t in tiles]
        if sum(tiles) == 0:
            tiles[rng.randrange(T)] = 1
        us = [0]
        for t in tiles:
            us.append(us[-1] + t)
        yield T, us, rng.randint(1, 160)


def test_warp_search_equals_scalar_search():
    for T, us, G in layouts(1, 300):
        U = us[T]
        for g in range(G):
            u0 = U * g // G
            if u0 < U:
                assert warp_search(us, T, u0) == scalar_search(us, T, u0)


def test_look_ahead_places_every_tile():
    for T, us, G in layouts(2, 300):
        U = us[T]
        for g in range(G):
            u0, u1 = U * g // G, U * (g + 1) // G
            nk = u1 - u0
            if nk <= 0:
                continue
            ct, ctile = warp_search(us, T, u0)
            for k in range(0, nk, 32):
                nb = [us[ct + 1 + l] if ct + 1 + l <= T else 0x7FFFFFFF for l in range(32)]
                got = []
                for lane in range(32):
                    uj = u0 + k + lane
                    cnt = shuffle_count(nb, uj)
                    if k + lane >= nk:
                        got.append((ct, 0))
                    elif cnt < 32:
                        below = nb[cnt - 1] if cnt > 0 else u0 + k - ctile
                        got.append((ct + cnt, uj - below))
                    else:
                        got.append(scalar_search(us, T, uj))
                for lane in range(min(32, nk - k)):
                    assert got[lane] == scalar_search(us, T, u0 + k + lane)
                ct, ctile = got[31][0], got[31][1] + 1


def packed_offsets(keep):
    """compact_short's placement: keep[t][c] is thread t's 4-bit keep mask in
    chunk c (1024 threads, 8 chunks). Per-chunk counts travel as 8-bit fields
    (chunks 0-3 and 4-7 in two words) through a warp inclusive scan, and as
    16-bit fields (widened from each warp's total) through a scan across the
    32 warps; a kept entry's output index is (entries of earlier chunks) +
    (chunk c in earlier warps) + (chunk c in earlier lanes) + (earlier bits)."""
    T, C = len(keep), len(keep[0])
    mine = [[0, 0] for _ in range(T)]
    for t in range(T):
        for c in range(C):
            mine[t][c >> 2] |= bin(keep[t][c]).count("1") << (8 * (c & 3))
    incl = [[0, 0] for _ in range(T)]
    for w in range(T // 32):
        acc = [0, 0]
        for l in range(32):
            t = 32 * w + l
            for h in range(2):
                acc[h] = (acc[h] + mine[t][h]) & M32
                assert all(((acc[h] >> (8 * f)) & 0xFF) <= 128 for f in range(4))
                incl[t][h] = acc[h]
    nw = T // 32
    wide = []
    for w in range(nw):
        lo, hi = incl[32 * w + 31]
        wide.append([(lo & 0xFF) | (((lo >> 8) & 0xFF) << 16), ((lo >> 16) & 0xFF) | ((lo >> 24) << 16),
                     (hi & 0xFF) | (((hi >> 8) & 0xFF) << 16), ((hi >> 16) & 0xFF) | ((hi >> 24) << 16)])
    wincl, acc = [], [0, 0, 0, 0]
    for w in range(nw):
        acc = [(acc[h] + wide[w][h]) & M32 for h in range(4)]
        assert all(((acc[h] >> (16 * f)) & 0xFFFF) <= 4096 for h in range(4) for f in range(2))
        wincl.append(list(acc))
    out = {}
    for t in range(T):
        w = t // 32
        total = 0
        for c in range(C):
            shift = 16 * (c & 1)
            tot_c = (wincl[nw - 1][c >> 1] >> shift) & 0xFFFF
            bw = ((wincl[w][c >> 1] - wide[w][c >> 1]) >> shift) & 0xFFFF
            bt = ((incl[t][c >> 2] - mine[t][c >> 2]) >> (8 * (c & 3))) & 0xFF
            at = total + bw + bt
            total += tot_c
            for j in range(4):
                if keep[t][c] >> j & 1:
                    out[(c, t, j)] = at
                    at += 1
    return out


def test_packed_scans_place_entries_in_row_order():
    rng = random.Random(5)
    for trial in range(12):
        dens = rng.choice([0.0, 0.02, 0.1, 0.5, 1.0])
        keep = [[sum(1 << j for j in range(4) if rng.random() < dens) for _ in range(8)]
                for _ in range(1024)]
        got = packed_offsets(keep)
        # row order: chunk c covers entries c*4096 + 4t + j
        order = sorted(got, key=lambda e: e[0] * 4096 + 4 * e[1] + e[2])
        assert [got[e] for e in order] == list(range(len(order)))
