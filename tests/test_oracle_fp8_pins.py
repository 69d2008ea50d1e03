"""Pins of the oracle's FP8 variant (quant mode 1: E4M3 codes) against what
fixes it independently of the oracle's code:

- E4M3 decoding of all 256 codes, and encoding (round to nearest even,
  every halfway point included), against PyTorch's float8_e4m3fn type;
  saturation past 448 by definition;
- the dot product: the exact rational sum of the decoded products, rounded
  once to FP32 (exact in double first: the sum is a multiple of 2^-18 below
  2^43);
- pair scores and TopK against a numpy brute force of the chain with
  np.float16 steps (the A3 chain from the division by 1024 on);
- the E4M3 quantiser: scale FP16(amax / 448), codes E4M3(x / s), degenerate
  rows.

The pages name FP8 as quant mode 1 of the A5 build (guide "DeepSeek V4.1 QLI
V2 与候选集成", section 编译范围) but print no FP8 golden; the oracle's
reading (same layout, same FP16 scales, the A3 chain on the exact dot) is
stated in its header.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_qli_gb300 import synth

torch = pytest.importorskip("torch")
if not hasattr(torch, "float8_e4m3fn"):
    pytest.skip("torch without float8_e4m3fn", allow_module_level=True)

FINITE = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy()).view(
        torch.float8_e4m3fn).float().numpy().astype(np.float64)


def torch_encode(values):
    return torch.from_numpy(np.asarray(values, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    want = torch_decode(codes)
    got = np.array([oracle.e4m3_to_f64(c) for c in codes])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_encode_matches_torch_including_every_tie():
    pos = np.sort(torch_decode(FINITE[FINITE < 0x80]))
    mids = (pos[:-1] + pos[1:]) / 2                    # exact in FP32: ties to even
    rng = np.random.default_rng(3)
    v = np.concatenate([pos, mids, -mids, rng.uniform(-448, 448, 20000),
                        rng.normal(0, 0.02, 5000)]).astype(np.float32)
    got = np.array([oracle.f32_to_e4m3(x) for x in v], dtype=np.uint8)
    assert np.array_equal(got, torch_encode(v))
    # ties go to the even code (mantissa LSB clear)
    tie_codes = got[len(pos):len(pos) + len(mids)]
    assert np.all(tie_codes & 1 == 0)


@pytest.mark.parametrize("x,code", [(448.0, 0x7E), (463.9, 0x7E), (1e6, 0x7E), (3.0e38, 0x7E),
                                    (-500.0, 0xFE), (0.0, 0x00), (-0.0, 0x80),
                                    (2.0 ** -10, 0x00), (3 * 2.0 ** -11, 0x01)])
def test_encode_saturates_and_rounds_at_the_edges(x, code):
    assert oracle.f32_to_e4m3(x) == code


def test_dot_is_the_exact_sum_rounded_once():
    rng = np.random.default_rng(5)
    for trial in range(200):
        q = rng.choice(FINITE, 128)
        k = rng.choice(FINITE, 128)
        exact = sum((Fraction(oracle.e4m3_to_f64(a)) * Fraction(oracle.e4m3_to_f64(b))
                     for a, b in zip(q, k)), Fraction(0))
        assert (exact * 2 ** 18).denominator == 1 and abs(exact) < 2 ** 25
        want = np.float32(float(exact))                # float(exact) is exact: one rounding
        assert np.float32(oracle.dot_e4m3(q, k)) == want


def fp8_case(seed, raw, ql, N, ratio, topk, mode="none", C=0):
    case = synth.make_case(seed, raw, ql, N=N, ratio=ratio, topk=topk, cand_mode=mode,
                           cand_blocks=C)
    rng = np.random.default_rng(seed + 1000)
    case.q = rng.choice(FINITE, case.q.shape).astype(np.uint8)
    case.k_rows = rng.choice(FINITE, case.k_rows.shape).astype(np.uint8)
    case.quant_mode = 1
    return case


def brute_scores(case):
    """Dense numpy restatement: exact dot -> FP32 -> /1024 -> FP16, ReLU,
    x FP16(w * qs) in FP16, FP32 sum over heads in order, x K scale."""
    dec = torch_decode(np.arange(256, dtype=np.uint8))
    out = {}
    for t in range(case.T):
        b = int(np.searchsorted(case.cu_seqlens_q, t, side="right") - 1)
        ql = int(case.cu_seqlens_q[b + 1] - case.cu_seqlens_q[b])
        res = 0 if case.residual is None else int(case.residual[b])
        V = oracle.visible_count(int(case.k_lens[b]), res, case.ratio, ql, t - int(case.cu_seqlens_q[b]))
        rows = case.k_rows[case.k_row_start[b]:case.k_row_start[b] + V]
        ks = case.k_scale[case.k_row_start[b]:case.k_row_start[b] + V].view(np.float16).astype(np.float32)
        kd = dec[rows]                                  # [V, D] exact values
        sc = np.zeros(V, dtype=np.float32)
        for h in range(case.N):
            qd = dec[case.q[t, h]]
            s = (kd @ qd).astype(np.float32)            # float64 sums are exact here
            x = (s / np.float32(1024)).astype(np.float16)
            r = np.maximum(x, np.float16(0))
            w = case.head_weights[t, h:h + 1].view(np.float16).astype(np.float32)
            qs = case.q_scale[t, h:h + 1].view(np.float16).astype(np.float32)
            wq = (w * qs).astype(np.float16)
            p = (r.astype(np.float32) * wq.astype(np.float32)).astype(np.float16)
            sc = (sc + p.astype(np.float32)).astype(np.float32)
        out[t] = sc * ks
    return out


@pytest.mark.parametrize("ratio,N", [(2, 32), (1, 64)])
def test_scores_and_topk_match_the_brute_force(ratio, N):
    case = fp8_case(40 + ratio, [700, 130, 1], [2, 1, 1], N=N, ratio=ratio, topk=50)
    prep = oracle.prepare(case)
    res = oracle.run(prep, want_scores=True)
    want = brute_scores(case)
    for t in range(case.T):
        V = int(res["visible"][t])
        got = res["scores"][t, :V]
        assert np.array_equal(got, want[t]), t          # float compare: -0 == +0, else exact
        # TopK: (score desc, position asc), -0 == +0, ascending output
        s = want[t] + np.float32(0)
        order = np.lexsort((np.arange(V), -s.astype(np.float64)))
        top = np.sort(order[:min(case.topk, V)])
        idx = res["indices"][t]
        assert np.array_equal(idx[:top.size], top) and np.all(idx[top.size:] == -1)


def test_fp8_scores_differ_from_int8_on_the_same_bytes():
    # the mode switch reaches the dot: the same bytes read as INT8 give other scores
    case = fp8_case(9, [300], [1], N=32, ratio=2, topk=10)
    prep = oracle.prepare(case)
    s8 = oracle.run(prep, want_scores=True)["scores"]
    case.quant_mode = 2
    case.q = case.q.view(np.int8)
    case.k_rows = case.k_rows.view(np.int8)
    s2 = oracle.run(oracle.prepare(case), want_scores=True)["scores"]
    V = 150
    assert not np.array_equal(s8[0, :V], s2[0, :V])


def test_unknown_quant_mode_is_rejected():
    case = fp8_case(10, [200], [1], N=32, ratio=2, topk=10)
    case.quant_mode = 3
    with pytest.raises(oracle.OracleError):
        oracle.run(oracle.prepare(case))


def bf16(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_quantiser_scale_and_codes():
    rng = np.random.default_rng(12)
    x = np.stack([synth.bf16_rows(60 + i, (128,), sigma=s)
                  for i, s in enumerate([1e-3, 0.1, 1.0, 37.0, 5000.0] * 4)])
    c, sc = oracle.quantize_rows_e4m3(x)
    xv = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    for r in range(x.shape[0]):
        amax = float(np.abs(xv[r]).max())
        s = oracle.f16_bits_to_f32(int(sc[r]))
        assert abs(s - amax / 448) <= max(2.0 ** -11 * amax / 448, 2.0 ** -25)
        q = (xv[r] / np.float32(s)).astype(np.float32)       # the FP32 quotient
        assert np.array_equal(c[r], torch_encode(np.clip(q, -448, 448)))
        assert np.abs(torch_decode(c[r])).max() <= 448


def test_quantiser_degenerate_rows():
    c, sc = oracle.quantize_rows_e4m3(np.zeros((1, 128), np.uint16))
    assert not c.any() and sc[0] == 0
    c, sc = oracle.quantize_rows_e4m3(bf16(np.full((1, 128), 2.0 ** -40)))
    assert not c.any() and sc[0] == 0
    big = bf16(np.where(np.arange(128) % 2 == 0, 2.0 ** 127, -2.0 ** 126)[None])
    c, sc = oracle.quantize_rows_e4m3(big)
    assert sc[0] == 0x7BFF and np.all(c[0, ::2] == 0x7E) and np.all(c[0, 1::2] == 0xFE)
    with pytest.raises(oracle.OracleError):
        oracle.quantize_rows_e4m3(np.full((1, 128), 0x7F80, np.uint16))


@pytest.mark.parametrize("ratio", [1, 2])
def test_fp8_writer_places_rows_where_the_indexer_reads_them(ratio):
    # the E4M3 writer fills the same bytes the indexer's page packing puts
    # the E4M3 codes and scales in (synth's packing, not the writer's code)
    case = synth.make_case(70 + ratio, [700, 130, 1], [1, 1, 1], N=32, ratio=ratio, topk=16)
    n = int(case.k_lens.sum())
    kb = synth.bf16_rows(70 + ratio, (n, 128), sigma=2.0)
    codes, scales = oracle.quantize_rows_e4m3(kb)
    case.k_rows = codes.view(np.int8)
    case.k_scale = scales
    slots = np.concatenate([synth.slots_of(case, b, np.arange(int(case.k_lens[b])))
                            for b in range(case.B)])
    want = case.pack_pages_numpy()
    pages = want.copy()
    R = case.rows_per_page
    rng = np.random.default_rng(4)
    for m in slots:                              # scribble over every target slot
        p, r = divmod(int(m), R)
        pages[p, case.k_offset + r * 128:case.k_offset + (r + 1) * 128] = rng.integers(0, 256, 128)
        pages[p, case.scale_offset + 2 * r:case.scale_offset + 2 * r + 2] = rng.integers(0, 256, 2)
    perm = rng.permutation(len(slots))
    rc = oracle.write_index_k(kb[perm], slots[perm], pages, R, case.k_offset, case.scale_offset,
                              fp8=True)
    assert rc == 0
    assert np.array_equal(pages, want)
    # and the INT8 writer touches exactly the same bytes
    other = want.copy()
    oracle.write_index_k(kb, slots, other, R, case.k_offset, case.scale_offset)
    int8_codes, int8_scales = oracle.quantize_rows(kb)
    assert not np.array_equal(other, want)
    case.k_rows, case.k_scale = int8_codes, int8_scales
    assert np.array_equal(other, case.pack_pages_numpy())
