"""GPU parity of the query quantiser and the index-K cache writer (through the
C ABI) against the oracle (qli_quant_oracle.c): codes and FP16 scale bits
must be identical (the quantisation decides integers, and both sides take
those decisions in FP32 with the same rounding), and the writer must leave
the page pool byte-identical to the oracle's write. Guide "DeepSeek V4.1 QLI
V2 与候选集成", section 数据流."""
import numpy as np
import pytest

import oracle
from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    qli.lib()


def _to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _mixed_rows(seed, n):
    """BF16 rows across magnitudes, plus the degenerate rows of the contract."""
    sig = [1e-4, 3e-3, 0.07, 1.0, 13.0, 450.0, 9000.0]
    rows = [synth.bf16_rows(seed + i, (D,), sigma=sig[i % len(sig)]) for i in range(n)]
    x = np.stack(rows) if rows else np.zeros((0, D), np.uint16)
    if n >= 6:
        x[0] = 0                                           # zero row
        x[1] = 0x2A80                                      # 2^-42: scale underflows to 0
        x[2] = 0x3A80                                      # 2^-10: subnormal FP16 scale
        x[3, ::2], x[3, 1::2] = 0x7F00, 0xFE00             # 2^127 / -2^125: scale saturates
        x[4] = x[4] ^ np.uint16(0x8000)                    # negated row
        x[5, :] = 0x8000                                   # -0 everywhere
    return x


@pytest.mark.parametrize("n", [1, 2, 3, 6, 257, 4099])
def test_quantize_q_matches_oracle(n):
    import torch
    x = _mixed_rows(300 + n, n)
    want_q, want_s = oracle.quantize_rows(x)
    q, s = qli.quantize_q(_to_dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), want_s)


def test_quantize_q_prefill_queries_full_size():
    # the prefill workload's queries: 4096 tokens x 64 heads
    import torch
    x = synth.bf16_rows(17, (4096, 64, D), sigma=1.0)
    want_q, want_s = oracle.quantize_rows(x)
    q, s = qli.quantize_q(_to_dev(x))
    torch.cuda.synchronize()
    assert q.shape == (4096, 64, D) and s.shape == (4096, 64)
    assert np.array_equal(q.cpu().numpy(), want_q)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), want_s)


def _writer_setup(seed, ratio, raw_lens):
    case = synth.make_case(seed, raw_lens, [1] * len(raw_lens), N=32, ratio=ratio, topk=16)
    n = int(case.k_lens.sum())
    kb = synth.bf16_rows(seed, (n, D), sigma=2.0)
    slots = np.concatenate([synth.slots_of(case, b, np.arange(int(case.k_lens[b])))
                            for b in range(case.B)]) if n else np.zeros(0, np.int64)
    return case, kb, slots


@pytest.mark.parametrize("ratio,raw_lens", [(1, [700, 130, 1]), (2, [5000, 64, 3, 0]),
                                             (2, [131072])])
def test_write_index_k_matches_oracle(ratio, raw_lens):
    import torch
    case, kb, slots = _writer_setup(80 + ratio + len(raw_lens), ratio, raw_lens)
    rng = np.random.default_rng(5)
    perm = rng.permutation(len(slots))
    kb, slots = kb[perm], slots[perm]
    slots = slots.copy()
    if len(slots) > 4:
        slots[1] = -1                                       # padding rows
        slots[3] = -7
    pages = case.pack_pages_numpy()                         # filler everywhere else
    want = pages.copy()
    rc = oracle.write_index_k(kb, slots, want, case.rows_per_page, case.k_offset,
                              case.scale_offset)
    assert rc == 0
    dev = torch.from_numpy(pages).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qli.write_index_k(_to_dev(kb), torch.from_numpy(slots).cuda(), dev,
                      rows_per_page=case.rows_per_page, page_stride=case.page_stride,
                      k_offset=case.k_offset, scale_offset=case.scale_offset, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(dev.cpu().numpy(), want)


def test_write_index_k_flags_slots_past_the_pool():
    import torch
    case, kb, slots = _writer_setup(90, 2, [300])
    slots = slots[:8].copy()
    slots[2] = case.num_pages * case.rows_per_page           # one past the pool
    slots[5] = 1 << 40
    pages = case.pack_pages_numpy()
    want = pages.copy()
    assert oracle.write_index_k(kb[:8], slots, want, case.rows_per_page, case.k_offset,
                                case.scale_offset) == -5
    dev = torch.from_numpy(pages).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qli.write_index_k(_to_dev(kb[:8]), torch.from_numpy(slots).cuda(), dev,
                      rows_per_page=case.rows_per_page, page_stride=case.page_stride,
                      k_offset=case.k_offset, scale_offset=case.scale_offset, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 8                               # QLI_DEVERR_PAGE
    assert np.array_equal(dev.cpu().numpy(), want)


def test_written_cache_and_quantised_queries_feed_the_indexer():
    """BF16 queries and index K quantised on the GPU, K written into the page
    pool on the GPU, then the indexer: equal to the oracle indexer run on the
    oracle's quantisation of the same BF16 inputs."""
    import torch
    case, kb, slots = _writer_setup(95, 2, [9000, 2500])
    codes, scales = oracle.quantize_rows(kb)
    case.k_rows, case.k_scale = codes, scales
    qb = synth.bf16_rows(96, case.q.shape, sigma=1.0)
    case.q, case.q_scale = oracle.quantize_rows(qb)
    prep = oracle.prepare(case)
    want = oracle.run(prep)["indices"]

    kw = synth.upload(case, "cuda")
    cache = kw["cache"]
    R = case.rows_per_page
    for m in slots:                                   # scramble the index-K rows first
        p, r = divmod(int(m), R)
        cache[p, case.k_offset + r * D:case.k_offset + (r + 1) * D] = 0x5A
    qli.write_index_k(_to_dev(kb), torch.from_numpy(slots).cuda(), cache, rows_per_page=R,
                      page_stride=case.page_stride, k_offset=case.k_offset,
                      scale_offset=case.scale_offset)
    q, s = qli.quantize_q(_to_dev(qb))
    kw["q"].copy_(q)
    kw["q_scale"].view(torch.int16).copy_(s)
    call = qli.Call(**kw)
    idx, _ = call.run(call.alloc_workspace())
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy()[:, 0, :], want)


def test_division_matches_ieee_on_every_bf16_value_and_fp16_scale():
    # the kernels' reciprocal-and-correction quotient against IEEE FP32
    # division, exhaustively over every (x, scale) pair a row can produce
    counts = qli.check_quant_rounding()
    assert counts == (0, 0)


# ---- FP8 (E4M3) variant ---------------------------------------------------

@pytest.mark.parametrize("n", [1, 6, 257, 4099])
def test_quantize_q_fp8_matches_oracle(n):
    import torch
    x = _mixed_rows(400 + n, n)
    want_c, want_s = oracle.quantize_rows_e4m3(x)
    c, s = qli.quantize_q(_to_dev(x), quant_mode=qli.QUANT_FP8)
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy().view(np.uint8), want_c)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), want_s)


@pytest.mark.parametrize("ratio,raw_lens", [(1, [700, 130, 1]), (2, [5000, 64, 3, 0])])
def test_write_index_k_fp8_matches_oracle(ratio, raw_lens):
    import torch
    case, kb, slots = _writer_setup(180 + ratio + len(raw_lens), ratio, raw_lens)
    slots = slots.copy()
    if len(slots) > 4:
        slots[2] = -1                                       # padding row
    pages = case.pack_pages_numpy()
    want = pages.copy()
    assert oracle.write_index_k(kb, slots, want, case.rows_per_page, case.k_offset,
                                case.scale_offset, fp8=True) == 0
    dev = torch.from_numpy(pages).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qli.write_index_k(_to_dev(kb), torch.from_numpy(slots).cuda(), dev,
                      rows_per_page=case.rows_per_page, page_stride=case.page_stride,
                      k_offset=case.k_offset, scale_offset=case.scale_offset, err_word=err,
                      quant_mode=qli.QUANT_FP8)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(dev.cpu().numpy(), want)


def test_fp8_quantised_inputs_feed_the_indexer():
    """BF16 queries and index K quantised to E4M3 on the GPU (bit-equal to the
    oracle's quantisation), K written into the pages on the GPU, then the
    indexer in quant mode 1: the FP8 parity rule against the oracle."""
    import torch
    from test_fp8_gpu import check as check_fp8
    case, kb, slots = _writer_setup(97, 2, [9000, 2500])
    case.quant_mode = qli.QUANT_FP8
    codes, scales = oracle.quantize_rows_e4m3(kb)
    case.k_rows, case.k_scale = codes.view(np.int8), scales
    qb = synth.bf16_rows(98, case.q.shape, sigma=1.0)
    qc, qs = oracle.quantize_rows_e4m3(qb)
    case.q, case.q_scale = qc.view(np.int8), qs
    kw = synth.upload(case, "cuda")
    cache = kw["cache"]
    want = cache.cpu().numpy()
    assert oracle.write_index_k(kb, slots, want, case.rows_per_page, case.k_offset,
                                case.scale_offset, fp8=True) == 0
    R = case.rows_per_page
    for m in slots:                                   # scramble the index-K rows first
        p, r = divmod(int(m), R)
        cache[p, case.k_offset + r * D:case.k_offset + (r + 1) * D] = 0x5A
    qli.write_index_k(_to_dev(kb), torch.from_numpy(slots).cuda(), cache,
                      rows_per_page=R, page_stride=case.page_stride,
                      k_offset=case.k_offset, scale_offset=case.scale_offset,
                      quant_mode=qli.QUANT_FP8)
    q, s = qli.quantize_q(_to_dev(qb), quant_mode=qli.QUANT_FP8)
    torch.cuda.synchronize()
    assert np.array_equal(cache.cpu().numpy(), want)
    assert np.array_equal(q.cpu().numpy(), case.q)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), case.q_scale)
    check_fp8(case)
