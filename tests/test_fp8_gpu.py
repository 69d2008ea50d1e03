"""GPU parity of the FP8 variant (quant mode 1: E4M3 codes in q and the index
K) against the oracle's FP8 reading (guide "DeepSeek V4.1 QLI V2 与候选集成",
section 编译范围 names FP8 as quant mode 1; the oracle's header states the
reading: the dot of the decoded codes rounded once to FP32, then the A3 chain
from the division by 1024 on).

The kernels widen the codes to FP16 exactly and sum on the tensor cores in
FP32, which is not the exactly rounded dot: a head's dot / 1024 can land on
the other side of an FP16 rounding boundary, changing that head's term by
about one FP16 ulp of x (2^-10 relative) and its FP16 product by one more
ulp. Tolerance per score, from that arithmetic with a factor two to spare:
    |s_gpu - s| <= 2^-8 * sum_h |x_h| * |wq_h| * k_scale + 2^-24 * k_scale,
with x_h = dot_h / 1024 computed exactly here. Selections may differ only
where the differing elements tie the boundary within 1e-3 relative (the rule
of every parity test here); most scores are bit-identical.
"""
import zlib

import numpy as np
import pytest

import oracle
from parity_rules import assert_selection
from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    qli.lib()


def decode_table():
    codes = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def score_bounds(case, t, V):
    """2^-8 * sum_h |dot_h / 1024| * |fp16(w * qs)| * ks + 2^-24 * ks for
    positions 0..V-1 of token t."""
    dec = decode_table()
    b = int(np.searchsorted(case.cu_seqlens_q, t, side="right") - 1)
    rows = case.k_rows[case.k_row_start[b]:case.k_row_start[b] + V]
    ks = np.abs(case.k_scale[case.k_row_start[b]:case.k_row_start[b] + V].view(np.float16)
                .astype(np.float64))
    dots = dec[rows] @ dec[case.q[t]].T                       # [V, N], exact in float64
    w = case.head_weights[t].view(np.float16).astype(np.float32)
    qs = case.q_scale[t].view(np.float16).astype(np.float32)
    wq = np.abs((w * qs).astype(np.float16).astype(np.float64))
    return (2.0 ** -8 * (np.abs(dots / 1024.0) @ wq) + 2.0 ** -24) * ks


def check(case, rows=None):
    kw = synth.upload(case, "cuda")
    call = qli.Call(**kw)
    ws = call.alloc_workspace()
    idx, cand = call.run(ws)
    torch.cuda.synchronize()
    assert call.device_error(ws) == 0
    g_idx = idx.cpu().numpy()[:, 0, :]
    g_cand = None if cand is None else cand.cpu().numpy()[:, 0, :]
    gs = call.scores(ws)
    rows = np.arange(case.T) if rows is None else np.asarray(rows)
    ora = oracle.run(oracle.prepare(case), rows=rows, want_scores=True,
                     score_stride=max(1, int(case.k_lens.max(initial=1))))
    exact = total = 0
    for r, t in enumerate(rows):
        t = int(t)
        V = int(ora["visible"][r])
        osc = ora["scores"][r]
        nb = (V + 7) // 8
        in_set = None
        if case.cand_mode == "consumer":
            ids = np.unique(case.cand_in[t, 0])
            in_set = set(ids[(ids >= 0) & (ids < nb)].tolist())

        def eligible(j):
            return 0 <= j < V and (in_set is None or j // 8 in in_set)

        assert_selection(g_idx[t], ora["indices"][r], lambda j: float(osc[j]), eligible,
                         ("indices", t))
        if case.cand_mode == "source":
            assert_selection(g_cand[t], ora["cand"][r],
                             lambda k: float(osc[8 * k:min(8 * k + 8, V)].max()),
                             lambda k: 0 <= k < nb, ("cand", t),
                             pinned=nb - 1 if nb > case.cand_blocks else None)
        if V == 0:
            continue
        if case.cand_mode == "consumer":
            blocks = np.array(sorted(in_set), dtype=np.int64)
            pos = (blocks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
            keep = pos < V
            got = gs[t, :pos.size].cpu().numpy()[keep].astype(np.float64)
            pos = pos[keep]
        else:
            got = gs[t, :V].cpu().numpy().astype(np.float64)
            pos = np.arange(V)
        want = osc[pos].astype(np.float64)
        bound = score_bounds(case, t, V)[pos]
        bad = np.abs(got - want) > bound
        assert not bad.any(), (t, np.flatnonzero(bad)[:4], got[bad][:4], want[bad][:4])
        exact += int((got == want).sum())
        total += got.size
    # the bound above is the contract; as a sanity check most scores are
    # bit-identical (about 98.5% on these inputs, whose codes span the whole
    # E4M3 range, so that FP32 sums round often)
    assert exact >= 0.95 * total, (exact, total)


SMALL = [
    ("decode-r1-n64", [1000, 129, 5000], [1, 1, 1], 64, 1, 300, "none", 0, {}),
    ("decode-r2-n32", [4097, 2, 3000], [1, 1, 1], 32, 2, 128, "none", 0, {}),
    ("prefill-r2-n64", [1500, 600, 2100], [5, 3, 9], 64, 2, 77, "none", 0, {}),
    ("source-r1-n32", [2600, 1111], [7, 1], 32, 1, 64, "source", 128, {}),
    ("source-r2-n64", [30000, 5000], [1, 2], 64, 2, 512, "source", 2048, {}),
    ("consumer-r2-n32-messy", [5000, 2111, 700], [1, 3, 2], 32, 2, 200, "consumer", 128,
     dict(cand_policy="messy")),
]


@pytest.mark.parametrize("p", SMALL, ids=[p[0] for p in SMALL])
def test_fp8_parity_small(p):
    name, raw, ql, N, r, K, mode, C, extra = p
    case = synth.make_case(zlib.crc32(name.encode()) % 1000, raw, ql, N=N, ratio=r, topk=K,
                           cand_mode=mode, cand_blocks=C, name=name, **extra)
    check(synth.to_fp8(case))


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_fp8_parity_workloads(idx):
    """The five workloads with E4M3 codes in place of the INT8 values: every
    row, except 256 rows (the requests' first and last tokens among them) of
    the 4096-token prefill workload."""
    case = synth.to_fp8(synth.config(idx))
    rows = None
    if idx == 3:
        rng = np.random.default_rng(33)
        edge = [0, 2047, 2048, 4095]
        rows = sorted(set(edge) | set(rng.choice(case.T, 252, replace=False).tolist()))
    check(case, rows=rows)


def test_fp8_and_int8_bytes_give_different_scores():
    # the mode reaches the kernels: the same bytes read as INT8 score otherwise
    case = synth.to_fp8(synth.make_case(3, [3000], [1], N=64, ratio=2, topk=64))
    kw = synth.upload(case, "cuda")
    a = qli.Call(**kw)
    ws = a.alloc_workspace()
    a.run(ws)
    s8 = a.scores(ws)[0, :1500].clone()
    kw["quant_mode"] = qli.QUANT_INT8
    b = qli.Call(**kw)
    b.run(ws)
    torch.cuda.synchronize()
    assert not torch.equal(s8, b.scores(ws)[0, :1500])


def _fuzz_cases(n=16, seed=20261204):
    """A seeded sweep of small E4M3 batches: ratio, head count, candidate
    mode, one to three requests up to 6000 raw tokens, decode- or
    prefill-shaped, TopK and candidate counts drawn at random."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 4))
        ratio = int(rng.integers(1, 3))
        N = int(rng.choice([32, 64]))
        mode = str(rng.choice(["none", "source", "consumer"]))
        raw = rng.integers(0, 6001, size=B)
        ql = np.ones(B, dtype=np.int64) if rng.random() < 0.5 else rng.integers(1, 17, size=B)
        topk = int(rng.choice([1, 33, 256, 2048]))
        C = int(rng.integers(1, 9)) * 64 if mode != "none" else 0
        out.append(("fp8fuzz%02d-%s-r%d-n%d" % (i, mode, ratio, N), int(rng.integers(0, 1 << 30)),
                    raw.tolist(), ql.tolist(), N, ratio, topk, mode, C))
    return out


FUZZ = _fuzz_cases()


@pytest.mark.parametrize("p", FUZZ, ids=[p[0] for p in FUZZ])
def test_fp8_parity_seeded_sweep(p):
    name, seed, raw, ql, N, ratio, topk, mode, C = p
    case = synth.make_case(seed, raw, ql, N=N, ratio=ratio, topk=topk, cand_mode=mode,
                           cand_blocks=C, name=name)
    check(synth.to_fp8(case))
