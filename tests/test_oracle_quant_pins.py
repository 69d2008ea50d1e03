"""Pins of the query quantiser and index-K writer oracle (qli_quant_oracle.c)
against what the pages and arithmetic fix, independent of the oracle's code:

- BF16 decoding against PyTorch's own BF16 type;
- rows on a power-of-two grid round-trip exactly (closed form);
- the scale is amax/127 to FP16 precision and the largest code is +-127;
- every code is the integer nearest x/s, checked in exact rational
  arithmetic (Fraction), away from the rare FP32 ties;
- sign symmetry and power-of-two scaling;
- degenerate rows: zero, below the FP16 range, above it, non-finite;
- the writer puts each row exactly where the indexer's page packing puts it
  and touches no other byte; padding and out-of-range slots.

Guide "DeepSeek V4.1 QLI V2 与候选集成", section 数据流: queries quantised per
head to INT8 with a scale representable in FP16; index K and FP16 scales
packed after the KV inside the page.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_qli_gb300 import synth

D = 128


def f16(b):
    return oracle.f16_bits_to_f32(int(b))


def bf16_of(values):
    """BF16 bit patterns of values that BF16 holds exactly (checked)."""
    import torch
    t = torch.tensor(np.asarray(values, dtype=np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "value not exact in BF16"
    return b.view(torch.int16).numpy().view(np.uint16)


def bf16_decode(bits):
    import torch
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy()) \
        .view(torch.bfloat16).float().numpy()


def test_bf16_decode_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bf16_decode(bits)
    got = np.array([oracle.bf16_bits_to_f32(int(b)) for b in bits[::7]], dtype=np.float32)
    w = want[::7]
    nan = np.isnan(w)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), w[~nan].view(np.uint32))


@pytest.mark.parametrize("e", [-24, -20, -14, -8, -1, 0, 3, 8, 15])
def test_power_of_two_grid_round_trips(e):
    rng = np.random.default_rng(100 + e)
    c = rng.integers(-127, 128, size=(6, D))
    c[np.arange(6), rng.integers(0, D, size=6)] = np.where(rng.random(6) < 0.5, 127, -127)
    s = 2.0 ** e
    x = bf16_of(c * s)
    q, sc = oracle.quantize_rows(x)
    assert np.array_equal(q.astype(np.int64), c)
    assert all(f16(b) == s for b in sc)


def _rows(seed, n, sigmas):
    out = []
    for i in range(n):
        out.append(synth.bf16_rows(seed + i, (D,), sigma=sigmas[i % len(sigmas)]))
    return np.stack(out)


SIGMAS = [1e-4, 3e-3, 0.07, 1.0, 13.0, 450.0, 9000.0]


def test_scale_is_amax_over_127_to_fp16_precision():
    x = _rows(7, 70, SIGMAS)
    q, sc = oracle.quantize_rows(x)
    xv = bf16_decode(x).astype(np.float64)
    for r in range(x.shape[0]):
        amax = np.abs(xv[r]).max()
        s = f16(sc[r])
        # half an FP16 ulp: relative 2^-11 for normal scales, 2^-25 below 2^-14
        assert abs(s - amax / 127) <= max(2.0 ** -11 * amax / 127, 2.0 ** -25), (r, s, amax)
        if s >= 2.0 ** -14:
            assert np.abs(q[r].astype(np.int64)).max() == 127


def _nearest_even(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def test_codes_are_nearest_integers_in_exact_arithmetic():
    x = _rows(11, 28, SIGMAS)
    q, sc = oracle.quantize_rows(x)
    xv = bf16_decode(x)
    checked = 0
    for r in range(x.shape[0]):
        s = Fraction(f16(sc[r]))
        for d in range(D):
            exact = Fraction(float(xv[r, d])) / s
            frac = exact - (exact.numerator // exact.denominator)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 2 ** 16):
                continue          # FP32 rounding of the quotient may decide this tie
            want = max(-127, min(127, _nearest_even(exact)))
            assert int(q[r, d]) == want, (r, d, float(exact))
            checked += 1
    assert checked > 0.99 * x.size


def test_sign_symmetry_and_power_of_two_scaling():
    x = _rows(21, 14, [0.05, 1.0, 40.0])
    q, sc = oracle.quantize_rows(x)
    qn, scn = oracle.quantize_rows(x ^ np.uint16(0x8000))        # -x
    assert np.array_equal(qn.astype(np.int64), -q.astype(np.int64))
    assert np.array_equal(scn, sc)
    x4 = bf16_of(bf16_decode(x) * 4.0)
    q4, sc4 = oracle.quantize_rows(x4)
    assert np.array_equal(q4, q)
    assert all(f16(a) == 4 * f16(b) for a, b in zip(sc4, sc))


def test_degenerate_rows():
    zero = np.zeros((1, D), dtype=np.uint16)
    q, sc = oracle.quantize_rows(zero)
    assert not q.any() and sc[0] == 0
    # amax/127 below half the smallest FP16 subnormal: scale 0, codes 0
    tiny = bf16_of(np.full((1, D), 2.0 ** -40))
    q, sc = oracle.quantize_rows(tiny)
    assert not q.any() and sc[0] == 0
    # subnormal FP16 scale: 127 * 2^-20 -> s = 2^-20 exactly
    sub = bf16_of(np.full((1, D), 127 * 2.0 ** -20))
    q, sc = oracle.quantize_rows(sub)
    assert f16(sc[0]) == 2.0 ** -20 and np.all(q == 127)
    # amax/127 past the FP16 range: the scale saturates at 65504, codes at +-127
    big = bf16_of(np.where(np.arange(D) % 2 == 0, 2.0 ** 127, -2.0 ** 125)[None])
    q, sc = oracle.quantize_rows(big)
    assert sc[0] == 0x7BFF
    assert np.all(q[0, ::2] == 127) and np.all(q[0, 1::2] == -127)


@pytest.mark.parametrize("bits", [0x7F80, 0xFF80, 0x7FC0])
def test_non_finite_rows_are_rejected(bits):
    x = np.zeros((2, D), dtype=np.uint16)
    x[1, 5] = bits
    with pytest.raises(oracle.OracleError):
        oracle.quantize_rows(x)


def test_quantised_dot_approximates_the_real_dot():
    # the INT8 product, rescaled, stays within the quantisation error bound
    xq = _rows(31, 8, [1.0])
    xk = _rows(41, 8, [0.3])
    cq, sq = oracle.quantize_rows(xq)
    ck, sk = oracle.quantize_rows(xk)
    a, b = bf16_decode(xq).astype(np.float64), bf16_decode(xk).astype(np.float64)
    for i in range(8):
        s1, s2 = f16(sq[i]), f16(sk[i])
        approx = s1 * s2 * float(np.dot(cq[i].astype(np.int64), ck[i].astype(np.int64)))
        bound = (0.5 * s1 * np.abs(b[i]).sum() + 0.5 * s2 * np.abs(a[i]).sum()
                 + 0.25 * s1 * s2 * D)
        assert abs(approx - float(np.dot(a[i], b[i]))) <= bound


# ---- index-K writer -------------------------------------------------------

def _writer_case(seed, ratio):
    case = synth.make_case(seed, [700, 130, 1], [1, 1, 1], N=32, ratio=ratio, topk=16)
    n = int(case.k_lens.sum())
    kb = synth.bf16_rows(seed, (n, D), sigma=2.0)
    codes, scales = oracle.quantize_rows(kb)
    case.k_rows = codes
    case.k_scale = scales
    slots = np.concatenate([synth.slots_of(case, b, np.arange(int(case.k_lens[b])))
                            for b in range(case.B)])
    return case, kb, slots


@pytest.mark.parametrize("ratio", [1, 2])
def test_writer_places_rows_where_the_indexer_reads_them(ratio):
    case, kb, slots = _writer_case(50 + ratio, ratio)
    want = case.pack_pages_numpy()              # the case's real page geometry
    pages = want.copy()
    R = case.rows_per_page
    rng = np.random.default_rng(3)
    for m in slots:                              # scribble over every target slot
        p, r = divmod(int(m), R)
        pages[p, case.k_offset + r * D:case.k_offset + (r + 1) * D] = rng.integers(0, 256, D)
        pages[p, case.scale_offset + 2 * r:case.scale_offset + 2 * r + 2] = rng.integers(0, 256, 2)
    perm = rng.permutation(len(slots))           # the order of the rows does not matter
    rc = oracle.write_index_k(kb[perm], slots[perm], pages, R, case.k_offset, case.scale_offset)
    assert rc == 0
    assert np.array_equal(pages, want)


def test_writer_padding_and_out_of_range_slots():
    case, kb, slots = _writer_case(60, 2)
    R = case.rows_per_page
    pages = case.pack_pages_numpy()
    before = pages.copy()
    sl = slots[:5].copy()
    sl[1] = -1                                   # padding: nothing written
    sl[3] = case.num_pages * R                   # past the pool: error, nothing written
    rc = oracle.write_index_k(kb[:5], sl, pages, R, case.k_offset, case.scale_offset)
    assert rc == -5
    codes, scales = oracle.quantize_rows(kb[:5])
    changed = np.zeros(pages.shape, dtype=bool)
    for i in (0, 2, 4):
        p, r = divmod(int(sl[i]), R)
        row = pages[p, case.k_offset + r * D:case.k_offset + (r + 1) * D]
        assert np.array_equal(row.view(np.int8), codes[i])
        assert pages[p, case.scale_offset + 2 * r:case.scale_offset + 2 * r + 2].view(np.uint16)[0] \
            == scales[i]
        changed[p, case.k_offset + r * D:case.k_offset + (r + 1) * D] = True
        changed[p, case.scale_offset + 2 * r:case.scale_offset + 2 * r + 2] = True
    assert np.array_equal(pages[~changed], before[~changed])
