"""Pins for the CPU oracle: each test ties it to something other than itself.

* IEEE binary16 facts and exact rational arithmetic pin the FP16 steps;
* a per-position statement of the causal rule pins the visible count;
* a dense numpy recomputation from the logical (unpaged) K rows, with numpy's
  own float16 arithmetic and a full lexsort, pins scoring, paging and the
  orderings on tiny inputs;
* closed forms (K >= V, C >= blocks), a textbook reduction (N = 1, unit
  weights and scales: TopK of an integer matrix product), and invariants from
  the guide "DeepSeek V4.1 QLI V2 与候选集成" (sections 数据流 and 当前 A3 契约)
  pin the selection rules.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_qli_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- FP16 ----

def f16_rne(x: Fraction):
    """Exact IEEE binary16 round-to-nearest-even of a rational (inf on overflow)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)                       # subnormals share the 2^-24 spacing
    ulp = Fraction(2) ** (e - 10)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * ulp
    if v > 65504:
        return sign * math.inf
    return sign * v


def f16_bits_value(bits: int) -> Fraction:
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    m = bits & 0x3FF
    assert e != 31
    if e == 0:
        return s * Fraction(m, 1 << 24)
    return s * (1 + Fraction(m, 1024)) * Fraction(2) ** (e - 15)


KNOWN_F16 = [
    (1.0, 0x3C00), (-2.0, 0xC000), (1.0 / 3.0, 0x3555), (65504.0, 0x7BFF),
    (65520.0, 0x7C00),            # halfway to 2^16 rounds to even -> overflow
    (65519.0, 0x7BFF), (2049.0, 0x6800), (2051.0, 0x6802),   # ties to even
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (3 * 2.0 ** -25, 0x0002),
    (2.0 ** -14, 0x0400), (-0.0, 0x8000), (0.1, 0x2E66),
]


@pytest.mark.parametrize("x,bits", KNOWN_F16)
def test_f16_known_bit_patterns(x, bits):
    assert oracle.f32_to_f16_bits(x) == bits


def test_f16_rounding_matches_exact_rationals():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.uniform(-3000, 3000, 400), rng.uniform(-1e-4, 1e-4, 300),
        (rng.integers(-2 ** 14, 2 ** 14, 300) + 0.5) / 1024.0,   # halfway cases
    ]).astype(np.float32)
    for v in vals:
        got = oracle.f32_to_f16_bits(float(v))
        want = f16_rne(Fraction(float(v)))
        assert f16_bits_value(got) == want, (float(v), hex(got))


def test_f16_matches_numpy_conversion():
    rng = np.random.default_rng(12)
    vals = rng.normal(0, 50, 2000).astype(np.float32)
    want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def _term_exact(s, wb, qb):
    x = f16_rne(Fraction(s, 1024))
    r = x if x > 0 else Fraction(0)
    wq = f16_rne(f16_bits_value(wb) * f16_bits_value(qb))
    return f16_rne(r * wq)


def test_head_term_closed_forms():
    one = 0x3C00
    assert oracle.head_term(1024, one, one) == 1.0
    assert oracle.head_term(-5, one, one) == 0.0          # ReLU
    assert oracle.head_term(0, one, one) == 0.0
    assert oracle.head_term(1025, one, one) == 1.0 + 2.0 ** -10   # representable
    assert oracle.head_term(2049, one, one) == 2.0         # 2049/1024 ties to even
    assert oracle.head_term(2051, one, one) == 2.0 + 2.0 ** -8
    assert oracle.head_term(3, one, one) == 3 * 2.0 ** -10
    half = 0x3800
    assert oracle.head_term(2048, half, half) == 0.5      # 2 * (0.5*0.5)
    neg = 0xBC00
    assert oracle.head_term(4096, neg, one) == -4.0        # negative weights pass


def test_head_term_matches_exact_rationals():
    rng = np.random.default_rng(13)
    w = rng.normal(0, 0.1, 300).astype(np.float16).view(np.uint16)
    qs = rng.uniform(0.005, 0.02, 300).astype(np.float16).view(np.uint16)
    s = rng.integers(-2_064_512, 2_064_513, 300)
    for a, b, c in zip(s, w, qs):
        got = Fraction(oracle.head_term(int(a), int(b), int(c)))
        assert got == _term_exact(int(a), int(b), int(c))


# ----------------------------------------------------------- visibility ----

def test_visible_count_hand_values():
    # ratio 2, S = 10 raw tokens (5 compressed, residual 0), 4 queries at raw
    # positions 6..9: 7, 8, 9, 10 raw tokens seen -> 3, 4, 4, 5 complete pairs
    assert [oracle.visible_count(5, 0, 2, 4, i) for i in range(4)] == [3, 4, 4, 5]
    # ratio 2, S = 11 (residual 1): a decode query at raw position 10 sees 5
    assert oracle.visible_count(5, 1, 2, 1, 0) == 5
    # ratio 1 is plain bottom-right causal: query i of 3 over S = 7 sees 5, 6, 7
    assert [oracle.visible_count(7, 0, 1, 3, i) for i in range(3)] == [5, 6, 7]
    # more queries than raw tokens before them: nothing visible
    assert oracle.visible_count(2, 0, 2, 8, 0) == 0
    assert oracle.visible_count(0, 0, 1, 1, 0) == 0


def test_visible_count_per_position_rule():
    # compressed j covers raw [j*r, j*r + r - 1]; it is visible once the query's
    # raw position has reached its last raw token
    rng = np.random.default_rng(14)
    for _ in range(300):
        r = int(rng.integers(1, 3))
        S = int(rng.integers(0, 200))
        q_len = int(rng.integers(1, S + 2))
        i = int(rng.integers(0, q_len))
        Lk, res = S // r, S % r
        pos = S - q_len + i
        want = sum(1 for j in range(Lk) if j * r + r - 1 <= pos)
        assert oracle.visible_count(Lk, res, r, q_len, i) == want


# ---------------------------------------------------- dense brute force ----

def dense(case, cand_in="from_case"):
    """Independent recomputation on the logical K rows (no paging), numpy
    float16 arithmetic, per-position visibility, full lexsort."""
    cin = case.cand_in if isinstance(cand_in, str) else cand_in
    T, N, D = case.q.shape
    K, C, r = case.topk, case.cand_blocks, case.ratio
    idx = np.full((T, K), -1, np.int32)
    cand = np.full((T, C), -1, np.int32) if case.cand_mode == "source" else None
    scores = {}
    for b in range(case.B):
        Kb = case.k_rows_of(b).astype(np.int64)
        ks = case.k_scale_of(b).view(np.float16).astype(np.float32)
        Lk = Kb.shape[0]
        S = int(case.raw_lens[b])
        c0, c1 = int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1])
        for t in range(c0, c1):
            pos = S - (c1 - c0) + (t - c0)
            j = np.arange(Lk)
            vis = j * r + r - 1 <= pos
            V = int(vis.sum())
            s = case.q[t].astype(np.int64) @ Kb.T                       # [N, Lk]
            x = (s / 1024.0).astype(np.float16)
            rl = np.maximum(x, np.float16(0))
            wq = case.head_weights[t].view(np.float16) * case.q_scale[t].view(np.float16)
            p = rl * wq[:, None]
            acc = np.zeros(Lk, np.float32)
            for h in range(N):
                acc = (acc + p[h].astype(np.float32)).astype(np.float32)
            sc = (acc * ks).astype(np.float32)[:V]
            scores[t] = sc
            elig = np.ones(V, bool)
            if case.cand_mode == "consumer":
                ids = {int(c) for c in cin[t, 0] if c >= 0}
                elig = np.array([(jj // 8) in ids for jj in range(V)], bool)
            jj = np.nonzero(elig)[0]
            order = jj[np.lexsort((jj, -sc[jj]))]
            sel = np.sort(order[:K])
            idx[t, :sel.size] = sel
            if case.cand_mode == "source":
                nb = (V + 7) // 8
                if nb <= C:
                    cand[t, :nb] = np.arange(nb)
                else:
                    bs = np.array([sc[8 * k:8 * k + 8].max() for k in range(nb - 1)], np.float32)
                    ids = np.arange(nb - 1)
                    top = ids[np.lexsort((ids, -bs))][:C - 1]
                    cand[t] = np.sort(np.concatenate([top, [nb - 1]]))
    return idx, cand, scores


TINY = [
    # (seed, raw_lens, q_lens, N, ratio, topk, mode, C, R)
    (0, [300], [1], 1, 1, 16, "none", 0, 64),
    (1, [301, 9], [3, 2], 2, 2, 7, "none", 0, 64),
    (2, [290, 41, 0], [4, 1, 1], 32, 1, 24, "none", 0, 16),
    (3, [600, 17], [2, 3], 2, 2, 5, "source", 64, 64),
    (4, [1200], [2], 1, 2, 40, "source", 64, 128),
    (5, [523, 260], [3, 2], 32, 2, 9, "consumer", 64, 64),
    (6, [250, 250], [1, 4], 2, 1, 300, "consumer", 64, 64),
]


def _case(p, **kw):
    seed, raw, ql, N, r, K, mode, C, R = p
    return synth.make_case(seed, raw, ql, N=N, ratio=r, topk=K, cand_mode=mode,
                           cand_blocks=C, rows_per_page=R, **kw)


@pytest.mark.parametrize("p", TINY)
@pytest.mark.parametrize("compact", [True, False])
def test_oracle_matches_dense_brute_force(p, compact):
    case = _case(p, cand_policy="messy")
    out = oracle.run(oracle.prepare(case, compact=compact), want_scores=True)
    idx, cand, scores = dense(case)
    assert np.array_equal(out["indices"], idx)
    if cand is not None:
        assert np.array_equal(out["cand"], cand)
    for t, sc in scores.items():
        V = sc.size
        assert out["visible"][t] == V
        assert np.array_equal(out["scores"][t, :V], sc)   # -0 == +0, else bit-equal


def test_textbook_reduction_integer_topk():
    # N = 1 with unit weight, Q scale and K scale, and dots that are multiples
    # of 1024: each score is relu(s / 1024) exactly, so the position TopK is the
    # top-k of an integer matrix product.
    rng = np.random.default_rng(21)
    vals = rng.permutation(np.arange(-120, 121))[:200]
    case = synth.make_case(22, [200], [1], N=1, ratio=1, topk=37)
    case.q[0, 0, :] = 0
    case.q[0, 0, :64] = 16                     # dot = 16 * 64 * v = 1024 v
    case.k_rows[:] = 0
    case.k_rows[:, :64] = vals[:, None].astype(np.int8)
    one = np.float16(1).view(np.uint16)
    case.head_weights[:] = one
    case.q_scale[:] = one
    case.k_scale[:] = one
    out = oracle.run(oracle.prepare(case))
    dots = (case.q[0, 0].astype(np.int64) @ case.k_rows.astype(np.int64).T) // 1024
    relu = np.maximum(dots, 0)
    assert (relu > 0).sum() > 37               # distinct positive values decide all
    top = np.argpartition(-relu, 36)[:37]
    assert np.array_equal(out["indices"][0], np.sort(top))


def test_closed_forms_small_context():
    # K >= V: every visible position in order; C >= blocks: every block in order
    case = synth.make_case(31, [130, 61], [3, 1], N=2, ratio=2, topk=80,
                           cand_mode="source", cand_blocks=64)
    out = oracle.run(oracle.prepare(case))
    for r in range(case.T):
        V = int(out["visible"][r])
        assert V <= 80
        want = np.full(80, -1)
        want[:V] = np.arange(V)
        assert np.array_equal(out["indices"][r], want)
        nb = (V + 7) // 8
        wc = np.full(64, -1)
        wc[:nb] = np.arange(nb)
        assert np.array_equal(out["cand"][r], wc)


def test_invariants_source_mode():
    case = synth.make_case(41, [3000, 5, 1401], [3, 1, 2], N=32, ratio=2, topk=64,
                           cand_mode="source", cand_blocks=64)
    out = oracle.run(oracle.prepare(case))
    for r in range(case.T):
        V = int(out["visible"][r])
        ids = out["indices"][r]
        valid = ids[ids >= 0]
        assert np.all(valid < V)                                 # no future positions
        assert np.all(np.diff(valid) > 0)                        # chronological
        assert np.all(ids[valid.size:] == -1)                    # -1 at the end
        assert valid.size == min(64, V)
        nb = (V + 7) // 8
        c = out["cand"][r]
        cv = c[c >= 0]
        if nb:
            assert nb - 1 in cv                                  # last block pinned
        assert cv.size == min(64, nb)
        assert np.all(np.diff(cv) > 0) and np.all(cv < max(nb, 1))


def test_empty_context():
    case = synth.make_case(42, [0, 1, 40], [1, 3, 1], N=2, ratio=2, topk=10,
                           cand_mode="source", cand_blocks=64)
    out = oracle.run(oracle.prepare(case))
    # request 0 (S = 0) and the first queries of request 1 (S = 1, ratio 2) see nothing
    for r in range(4):
        assert out["visible"][r] == 0
        assert np.all(out["indices"][r] == -1)
        assert np.all(out["cand"][r] == -1)


def test_errors():
    case = synth.make_case(43, [100], [1], N=2, ratio=2, topk=4, cand_mode="consumer",
                           cand_blocks=64)
    with pytest.raises(oracle.OracleError, match="consumer without source"):
        oracle.run(oracle.prepare(case, cand_in=None))
    case1 = synth.make_case(44, [100], [1], N=2, ratio=1, topk=4)
    with pytest.raises(oracle.OracleError, match="residual with ratio 1"):
        oracle.run(oracle.prepare(case1, residual=np.zeros(1, np.int32)))


def test_consumer_with_all_blocks_equals_none():
    case = synth.make_case(51, [777, 300], [2, 2], N=32, ratio=2, topk=33,
                           cand_mode="consumer", cand_blocks=128)
    C = 128
    full = np.full((case.T, 1, C), -1, np.int32)
    rng = np.random.default_rng(5)
    for t in range(case.T):
        b = 0 if t < 2 else 1
        nb = (int(case.k_lens[b]) + 7) // 8
        ids = np.concatenate([np.arange(nb), rng.integers(0, nb, 5)])   # duplicates too
        rng.shuffle(ids)
        full[t, 0, :ids.size] = ids
    cons = oracle.run(oracle.prepare(case, cand_in=full))
    none = oracle.run(oracle.prepare(case, cand_mode="none"))
    assert np.array_equal(cons["indices"], none["indices"])


def test_source_topk_lies_in_candidate_blocks():
    case = synth.make_case(52, [4000, 2500], [2, 1], N=64, ratio=2, topk=63,
                           cand_mode="source", cand_blocks=64)
    out = oracle.run(oracle.prepare(case), want_scores=True)
    for r in range(case.T):
        V = int(out["visible"][r])
        sc = out["scores"][r, :V]
        assert np.unique(sc).size == V          # distinct scores: containment holds
        blocks = set(out["cand"][r][out["cand"][r] >= 0].tolist())
        for j in out["indices"][r]:
            if j >= 0:
                assert j // 8 in blocks


def test_paging_invariance():
    case = synth.make_case(53, [900, 333], [2, 1], N=32, ratio=2, topk=20,
                           cand_mode="source", cand_blocks=64)
    a = oracle.run(oracle.prepare(case, compact=False))
    # move every page to a new slot and rewrite the block table to match
    perm = np.random.default_rng(9).permutation(case.num_pages)
    pages = case.pack_pages_numpy()
    moved = np.empty_like(pages)
    moved[perm] = pages
    case.block_table = perm[case.block_table].astype(np.int32)
    b = oracle.run(oracle.prepare(case, pages=moved))
    assert np.array_equal(a["indices"], b["indices"])
    assert np.array_equal(a["cand"], b["cand"])


def test_batch_independence():
    raws, qls = [700, 95, 1500], [2, 1, 3]
    mixed = synth.make_case(54, raws, qls, N=32, ratio=2, topk=16, cand_mode="source",
                            cand_blocks=64)
    out = oracle.run(oracle.prepare(mixed))
    for b in range(3):
        c0, c1 = int(mixed.cu_seqlens_q[b]), int(mixed.cu_seqlens_q[b + 1])
        alone = synth.make_case(54, [raws[b]], [qls[b]], N=32, ratio=2, topk=16,
                                cand_mode="source", cand_blocks=64)
        alone.q = mixed.q[c0:c1].copy()
        alone.head_weights = mixed.head_weights[c0:c1].copy()
        alone.q_scale = mixed.q_scale[c0:c1].copy()
        alone.k_rows = mixed.k_rows_of(b).copy()
        alone.k_scale = mixed.k_scale_of(b).copy()
        o = oracle.run(oracle.prepare(alone))
        assert np.array_equal(o["indices"], out["indices"][c0:c1])
        assert np.array_equal(o["cand"], out["cand"][c0:c1])


def test_k_scale_doubling_preserves_selection():
    # doubling every K scale (exact in FP16 here) doubles every score exactly
    case = synth.make_case(55, [1200], [2], N=32, ratio=2, topk=30, cand_mode="source",
                           cand_blocks=64)
    a = oracle.run(oracle.prepare(case), want_scores=True)
    case.k_scale = (case.k_scale.view(np.float16) * np.float16(2)).view(np.uint16)
    b = oracle.run(oracle.prepare(case), want_scores=True)
    assert np.array_equal(a["indices"], b["indices"])
    assert np.array_equal(a["cand"], b["cand"])
    V = int(a["visible"][0])
    assert np.array_equal(a["scores"][0, :V] * 2, b["scores"][0, :V])


def test_contract_geometry_matches_pages():
    with open(os.path.join(HERE, "golden", "contract.json")) as f:
        g = json.load(f)["page_geometry"]
    assert synth.GEOMETRY[2] == (g["ratio2"]["rows_per_page"], g["ratio2"]["page_stride"])
    assert synth.GEOMETRY[1] == (g["ratio1"]["rows_per_page"], g["ratio1"]["page_stride"])
    # index K rows and scales fit after the KV inside each page
    for r in (1, 2):
        R, stride = synth.GEOMETRY[r]
        k_off, s_off = synth.page_offsets(R)
        assert s_off + 2 * R <= stride
    assert synth.page_offsets(128)[1] + 2 * 128 == 147712
