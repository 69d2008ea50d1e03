"""GPU parity of the sparse attention over the selected positions
(qli_sparse_attention, through the C ABI) against the float64 oracle
(oracle/csa.py).

Tolerance, derived from the arithmetic: the BF16 products are exact; the
FP32 sums of 512 of them move a score s by at most ~5e-4 (after the 1/sqrt(512)
scale, for values of unit size); the weights are rounded to BF16 for the value
product (relative 2^-9) while the normaliser sums them unrounded (2^-9); the
output is rounded to BF16 (2^-9 of |o|). Together
    |o_gpu - o| <= 2^-7 * max_j |kv_j| + 2^-7 * |o|
elementwise (about twice the bound), and |lse_gpu - lse| <= 2e-3 + 1e-5 |lse|.
"""
import zlib

import numpy as np
import pytest

from oracle import csa
from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(512.0)
ATOL_REL_KV = 2.0 ** -7
RTOL = 2.0 ** -7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    qli.lib()


def run_gpu(case, scale=SCALE, err=None):
    import torch
    dev = "cuda"
    cache = case.pack_pages_torch(dev)
    q = torch.from_numpy(case.q_attn.view(np.int16)).to(dev).view(torch.bfloat16)
    cu = torch.from_numpy(case.cu_seqlens_q).to(dev)
    bt = torch.from_numpy(case.block_table).to(dev)
    idx = torch.from_numpy(case.attn_indices).to(dev)
    out, lse = qli.sparse_attention(q, cu, cache, bt, idx, rows_per_page=case.rows_per_page,
                                    page_stride=case.page_stride, scale=scale, err_word=err)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy().astype(np.float64)
    return o, lse.cpu().numpy().astype(np.float64)


def check(case, tokens=None, scale=SCALE):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_g, lse_g = run_gpu(case, scale, err)
    assert int(err.item()) == 0
    tokens = list(range(case.T)) if tokens is None else list(tokens)
    o_r, lse_r = csa.attention(case, scale, tokens=tokens, rows=csa.rows_from_logical(case))
    for r, t in enumerate(tokens):
        b = csa.request_of(case.cu_seqlens_q, t)
        js = case.attn_indices[t, 0]
        js = js[js >= 0]
        if js.size == 0:
            assert np.all(o_g[t] == 0.0) and np.all(np.isneginf(lse_g[t])), t
            continue
        kvmax = np.abs(csa.bf16_to_f64(case.kv_of(b)[js])).max()
        tol = ATOL_REL_KV * kvmax + RTOL * np.abs(o_r[r])
        bad = np.abs(o_g[t] - o_r[r]) > tol
        assert not bad.any(), (t, np.argwhere(bad)[:4], o_g[t][bad][:4], o_r[r][bad][:4])
        assert np.all(np.abs(lse_g[t] - lse_r[r]) <= 2e-3 + 1e-5 * np.abs(lse_r[r])), t


SMALL = [
    # name, raw_lens, q_lens, ratio, H, K, count
    ("r2-h32-k256", [3000, 900], [2, 1], 2, 32, 256, None),
    ("r1-h64-k300", [2600, 1111, 4000], [1, 2, 1], 1, 64, 300, None),
    ("r2-h64-k2048", [9000, 5000], [1, 1], 2, 64, 2048, None),
    ("r1-h32-k1", [500, 40], [1, 1], 1, 32, 1, None),
    ("r2-h128-k129", [3000], [2], 2, 128, 129, None),
    ("r1-h64-short-lists", [3000, 2000], [2, 2], 1, 64, 512, (0, 200)),
    ("r2-h96-k100", [1000, 1000], [1, 1], 2, 96, 100, None),
]


@pytest.mark.parametrize("p", SMALL, ids=[p[0] for p in SMALL])
def test_attention_parity_small(p):
    name, raw, ql, r, H, K, count = p
    seed = zlib.crc32(name.encode()) % 1000
    case = synth.make_case(seed, raw, ql, N=64, ratio=r, topk=16, name=name)
    synth.add_attention(case, H=H, topk=K, count=count)
    check(case)


def test_attention_holes_duplicates_and_empty_rows():
    case = synth.make_case(12, [2000, 700, 300], [2, 1, 1], N=64, ratio=2, topk=16)
    synth.add_attention(case, H=64, topk=384)
    rng = np.random.default_rng(3)
    row = case.attn_indices[0, 0]
    row[rng.choice(384, 100, replace=False)] = -1          # holes anywhere
    case.attn_indices[1, 0, 10:20] = case.attn_indices[1, 0, 0]   # a position listed 11 times
    case.attn_indices[2] = -1                              # nothing listed
    check(case)


def test_attention_dominant_scores():
    # a large scale: each head's weights concentrate on one or two rows
    case = synth.make_case(13, [4000, 2500], [1, 1], N=64, ratio=1, topk=16)
    synth.add_attention(case, H=64, topk=1024)
    check(case, scale=0.5)


def test_attention_flags_positions_past_the_block_table():
    import torch
    case = synth.make_case(14, [1000], [1], N=64, ratio=2, topk=16)
    synth.add_attention(case, H=32, topk=64)
    cap = case.bt_stride * case.rows_per_page
    case.attn_indices[0, 0, 5] = cap + 3                   # past the table: skipped, flagged
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_g, lse_g = run_gpu(case, err=err)
    assert int(err.item()) & 8                             # QLI_DEVERR_PAGE
    case.attn_indices[0, 0, 5] = -1
    o_r, lse_r = csa.attention(case, SCALE, rows=csa.rows_from_logical(case))
    assert np.allclose(o_g[0], o_r[0], atol=ATOL_REL_KV * 4, rtol=RTOL)


def test_attention_after_the_indexer():
    """The two stages chained: the indexer's TopK indices of a decode batch
    feed the attention directly on the device."""
    import torch
    case = synth.make_case(15, [6000, 3000, 9000], [1, 1, 1], N=64, ratio=1, topk=512)
    synth.add_attention(case, H=64, topk=512)
    kw = synth.upload(case, "cuda")
    call = qli.Call(**kw)
    ws = call.alloc_workspace()
    idx, _ = call.run(ws)
    q = torch.from_numpy(case.q_attn.view(np.int16)).cuda().view(torch.bfloat16)
    out, lse = qli.sparse_attention(q, kw["cu_seqlens_q"], kw["cache"], kw["block_table"], idx,
                                    rows_per_page=case.rows_per_page,
                                    page_stride=case.page_stride, scale=SCALE)
    torch.cuda.synchronize()
    case.attn_indices = idx.cpu().numpy()
    o_r, lse_r = csa.attention(case, SCALE, rows=csa.rows_from_logical(case))
    o_g = out.float().cpu().numpy()
    for t in range(case.T):
        js = case.attn_indices[t, 0]
        b = csa.request_of(case.cu_seqlens_q, t)
        kvmax = np.abs(csa.bf16_to_f64(case.kv_of(b)[js[js >= 0]])).max()
        assert np.all(np.abs(o_g[t] - o_r[t]) <= ATOL_REL_KV * kvmax + RTOL * np.abs(o_r[t]))


def test_attention_full_size_workload():
    """The bench workload (64 decode tokens of the ratio-1 batch, 64 heads,
    2048 listed positions each), every token checked against the oracle."""
    check(synth.attention_workload(seed=21))


def _fuzz_cases(n=16, seed=20261205):
    """A seeded sweep of small attention calls: ratio (page geometry), 32 to
    128 heads, one to three requests up to 6000 raw tokens with one to four
    tokens each, 1 to 2048 listed entries, list lengths drawn below that
    (some rows listing nothing), and a softmax scale from 1/sqrt(512) up."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        ratio = int(rng.integers(1, 3))
        H = int(rng.choice([32, 64, 96, 128]))
        raw = rng.integers(1, 6001, size=B)
        ql = rng.integers(1, 5, size=B)
        K = int(rng.choice([1, 40, 129, 512, 2048]))
        lo = int(rng.integers(0, K + 1))
        scale = float(SCALE * rng.choice([1.0, 1.0, 4.0, 16.0]))
        out.append(("attnfuzz%02d-r%d-h%d-k%d" % (i, ratio, H, K), int(rng.integers(0, 1 << 30)),
                    raw.tolist(), ql.tolist(), ratio, H, K, (lo, K), scale))
    return out


FUZZ = _fuzz_cases()


@pytest.mark.parametrize("p", FUZZ, ids=[p[0] for p in FUZZ])
def test_attention_parity_seeded_sweep(p):
    name, seed, raw, ql, ratio, H, K, count, scale = p
    case = synth.make_case(seed, raw, ql, N=64, ratio=ratio, topk=16, name=name)
    synth.add_attention(case, H=H, topk=K, count=count)
    check(case, scale=scale)
