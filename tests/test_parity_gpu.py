"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Indices and candidate IDs must be equal, with one allowance: an element may
differ when its oracle score ties the selection boundary within 1e-3
relative (REL_TIE_TOL). The FP32 scores the SCORE stage leaves in the
workspace must equal the oracle's bit for bit (-0 and +0 compare equal): the
INT32 dots are exact and the epilogue follows the golden's operation order.
"""
import zlib

import numpy as np
import pytest

import oracle
from parity_rules import REL_TIE_TOL, assert_selection  # noqa: F401
from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    qli.lib()


def run_gpu(case, cache=None):
    import torch
    kw = synth.upload(case, "cuda", cache=cache)
    call = qli.Call(**kw)
    ws = call.alloc_workspace()
    idx, cand = call.run(ws)
    torch.cuda.synchronize()
    out = {
        "indices": idx.cpu().numpy()[:, 0, :],
        "cand": None if cand is None else cand.cpu().numpy()[:, 0, :],
        "scores": call.scores(ws),
        "err": call.device_error(ws),
    }
    return out


def consumer_slots(case, t, V):
    """Sorted distinct candidate blocks of token t that hold a visible position."""
    nb = (V + 7) // 8
    ids = np.unique(case.cand_in[t, 0])
    return ids[(ids >= 0) & (ids < nb)]


def cand_width(case):
    return case.cand_blocks


def check(case, rows=None, scores=True):
    import torch
    gpu = run_gpu(case)
    assert gpu["err"] == 0, gpu["err"]
    prep = oracle.prepare(case)
    rows = np.arange(case.T) if rows is None else np.asarray(rows)
    ora = oracle.run(prep, rows=rows, want_scores=True, score_stride=max(1, int(case.k_lens.max(initial=1))))
    gs = gpu["scores"]
    for r, t in enumerate(rows):
        V = int(ora["visible"][r])
        osc = ora["scores"][r]

        nb = (V + 7) // 8
        if case.cand_mode == "consumer":
            in_set = set(consumer_slots(case, t, V).tolist())
        else:
            in_set = None

        def score_of(j):
            return float(osc[j])

        def eligible(j):
            return 0 <= j < V and (in_set is None or j // 8 in in_set)

        assert_selection(gpu["indices"][t], ora["indices"][r], score_of, eligible,
                         ("indices", int(t)))
        if case.cand_mode == "source":
            def bscore(k):
                return float(osc[8 * k:min(8 * k + 8, V)].max())

            def block_eligible(k):
                return 0 <= k < nb

            assert_selection(gpu["cand"][t], ora["cand"][r], bscore, block_eligible,
                             ("cand", int(t)), pinned=nb - 1 if nb > cand_width(case) else None)
            if nb:
                assert nb - 1 in gpu["cand"][t]
        if not scores or V == 0:
            continue
        if case.cand_mode == "consumer":
            blocks = consumer_slots(case, t, V)
            pos = (blocks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
            slot = np.arange(pos.size)
            keep = pos < V
            got = gs[int(t), :pos.size].cpu().numpy()[keep]
            want = osc[pos[keep]]
        else:
            got = gs[int(t), :V].cpu().numpy()
            want = osc[:V]
        assert np.array_equal(got, want), ("scores", int(t), np.flatnonzero(got != want)[:5])
    torch.cuda.synchronize()


SMALL = [
    # name, raw_lens, q_lens, N, ratio, topk, mode, C, extra
    ("decode-r1-n64", [1000, 129, 128, 1, 0, 5000], [1] * 6, 64, 1, 300, "none", 0, {}),
    ("decode-r2-n32", [4097, 2, 257, 3000], [1] * 4, 32, 2, 128, "none", 0, {}),
    ("prefill-r2-n64", [1500, 600, 2100], [5, 3, 9], 64, 2, 77, "none", 0, {}),
    ("prefill-r1-n32", [700, 260], [13, 2], 32, 1, 50, "none", 0, {}),
    ("source-r2-n64", [3000, 1301, 90], [1, 6, 1], 64, 2, 100, "source", 64, {}),
    ("source-r1-n32", [2600, 1111], [7, 1], 32, 1, 64, "source", 128, {}),
    ("consumer-r2-n32-messy", [5000, 2111, 700], [1, 3, 2], 32, 2, 200, "consumer", 128,
     dict(cand_policy="messy")),
    ("consumer-r1-n64", [3000, 1800], [2, 1], 64, 1, 256, "consumer", 64, {}),
    ("topk1", [2000, 777], [1, 2], 64, 2, 1, "source", 64, {}),
    ("topk2048-short", [3000, 600], [1, 1], 64, 2, 2048, "none", 0, {}),
    ("topk2048-long", [9000, 4100], [1, 1], 64, 1, 2048, "none", 0, {}),
    ("cand2048", [30000, 5000], [1, 2], 64, 2, 512, "source", 2048, {}),
    ("empty", [0, 0, 1], [1, 2, 1], 64, 2, 16, "source", 64, {}),
    ("tile-exact", [256, 128, 512], [1, 1, 1], 64, 1, 64, "none", 0, {}),
]


@pytest.mark.parametrize("p", SMALL, ids=[p[0] for p in SMALL])
def test_parity_small(p):
    name, raw, ql, N, r, K, mode, C, extra = p
    case = synth.make_case(zlib.crc32(name.encode()) % 1000, raw, ql, N=N, ratio=r, topk=K, cand_mode=mode,
                           cand_blocks=C, name=name, **extra)
    check(case)


def test_consumer_all_blocks_equals_none_on_gpu():
    case = synth.make_case(7, [1900, 800], [2, 1], N=64, ratio=2, topk=150,
                           cand_mode="consumer", cand_blocks=256)
    for t in range(case.T):
        b = 0 if t < 2 else 1
        nb = (int(case.k_lens[b]) + 7) // 8
        row = np.full(256, -1, np.int32)
        ids = np.random.default_rng(t).permutation(nb)
        row[:nb] = ids
        case.cand_in[t, 0] = row
    g_cons = run_gpu(case)
    case.cand_mode = "none"
    case.cand_blocks = 0
    g_none = run_gpu(case)
    assert np.array_equal(g_cons["indices"], g_none["indices"])


def test_consumer_beyond_the_bitmap_takes_the_sorting_path():
    # a block table wide enough that a request could hold more blocks than
    # the candidate kernel's shared-memory bitmap covers (66000 x 64
    # positions > 16384 x 32 x 8): the candidates are sorted by the bitonic
    # fallback, which also looks up their pages and scales
    case = synth.make_case(11, [3000, 1700], [2, 1], N=32, ratio=2, topk=100,
                           cand_mode="consumer", cand_blocks=128, bt_stride=66000,
                           cand_policy="messy", name="consumer-wide-table")
    assert case.bt_stride * case.rows_per_page > 16384 * 32 * 8
    check(case)


@pytest.mark.parametrize("geom", ["compact", "scales-first"])
@pytest.mark.parametrize("ratio", [1, 2])
def test_stream_path_page_geometries(geom, ratio):
    """Page geometries other than the pages' own: the FP16 scales right after
    the index-K rows in a compact page (stride R*130), and the scales placed
    before the rows. The stream kernel takes k_offset and scale_offset as
    given and matches the oracle in both, for source and consumer calls."""
    import dataclasses
    for mode, C in (("source", 64), ("consumer", 128)):
        case = synth.make_case(90 + ratio, [9000, 1300, 260], [1, 1, 1], N=64, ratio=ratio,
                               topk=200, cand_mode=mode, cand_blocks=C,
                               name=f"geometry-{geom}-r{ratio}-{mode}")
        R = case.rows_per_page
        assert case.bt_stride * R > 4096        # not the single-launch path
        if geom == "compact":
            stride, ko, so = R * 130, 0, R * 128
        else:
            so, ko = 0, 2 * R + 16
            stride = ko + R * 128 + 16
        check(dataclasses.replace(case, page_stride=stride, k_offset=ko, scale_offset=so))


def test_device_checks_flag_bad_metadata():
    import torch
    case = synth.make_case(8, [500, 300], [1, 1], N=64, ratio=2, topk=16)
    kw = synth.upload(case, "cuda")
    kw["k_lens"] = torch.tensor([500, 10 ** 6], dtype=torch.int32, device="cuda")  # > capacity
    call = qli.Call(**kw)
    ws = call.alloc_workspace()
    call.run(ws)
    err = call.device_error(ws)
    assert err & 2                                     # k_lens clamped and flagged
    idx = call.indices.cpu().numpy()[:, 0, :]
    assert np.all(idx[idx >= 0] < case.bt_stride * case.rows_per_page)


def test_repeat_calls_reuse_workspace():
    case = synth.make_case(9, [2500, 1200], [3, 1], N=64, ratio=2, topk=64, cand_mode="source",
                           cand_blocks=64)
    import torch
    kw = synth.upload(case, "cuda")
    call = qli.Call(**kw)
    ws = call.alloc_workspace()
    ws.fill_(0xFF)                        # garbage in the workspace must not matter
    a, ca = [x.clone() for x in call.run(ws)]
    b, cb = call.run(ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(ca, cb)


@pytest.mark.parametrize("mode", ["none", "source", "consumer"])
def test_stages_and_graph_replay_equal_one_call(mode):
    """PLAN, SCORE and SELECT queued one by one, and a CUDA graph of the whole
    call (whose kernels start early and wait on their predecessors on the
    device), give what one plain call gives, over a dirty workspace."""
    import torch
    case = synth.make_case(31, [100000, 2500, 9000], [1, 2, 1], N=64, ratio=2, topk=512,
                           cand_mode=mode, cand_blocks=256 if mode != "none" else 0,
                           cand_policy="messy" if mode == "consumer" else "valid")
    call = qli.Call(**synth.upload(case, "cuda"))
    ws = call.alloc_workspace()
    idx, cand = call.run(ws)
    torch.cuda.synchronize()
    want = (idx.clone(), None if cand is None else cand.clone())

    def same():
        torch.cuda.synchronize()
        assert torch.equal(call.indices, want[0])
        if want[1] is not None:
            assert torch.equal(call.cand, want[1])

    for rep in range(2):                       # the second pass starts from a used workspace
        call.indices.fill_(-7)
        for stage in (qli.STAGE_PLAN, qli.STAGE_SCORE, qli.STAGE_SELECT):
            call.run_stage(stage, ws)
        same()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            call.run(ws)
    torch.cuda.current_stream().wait_stream(s)
    for rep in range(3):
        call.indices.fill_(-7)
        g.replay()
        same()
    assert call.device_error(ws) == 0


@pytest.mark.parametrize("idx", [2, 5])
def test_back_to_back_graph_replays_never_time_out(idx):
    """Hundreds of back-to-back replays of a CUDA graph of the whole call on a
    full-size workload. Each kernel overlaps its neighbours (programmatic
    launch) and every on-chip wait must complete: a wait that gave up would
    cost 200 ms and set the timeout bit in the device error word, which the
    plan kernel resets at each call, so the word is read every ten calls."""
    import time

    import torch
    case = synth.config(idx)
    call = qli.Call(**synth.upload(case, "cuda"))
    ws = call.alloc_workspace()
    idx_out, _ = call.run(ws)
    torch.cuda.synchronize()
    want = idx_out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            call.run(ws)
    torch.cuda.current_stream().wait_stream(s)
    t0 = time.perf_counter()
    for rep in range(300):
        g.replay()
        if rep % 10 == 9:
            assert call.device_error(ws) == 0, rep
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 2.0
    assert torch.equal(call.indices, want)


def test_parity_long_rows():
    """Rows longer than one CTA's shared memory take the multi-CTA selection
    (statistics, histogram, compaction, exact ranking of the candidates)."""
    case = synth.make_case(81, [140000, 30001, 101], [1, 1, 1], N=64, ratio=2, topk=2048,
                           cand_mode="source", cand_blocks=1024, name="long-rows")
    check(case)


def test_parity_long_rows_all_equal_scores():
    """Every score of a long row equal: ties everywhere, the candidate buffer
    overflows and the row is ranked from L2; TopK = the first K positions."""
    case = synth.make_case(82, [120000, 5000], [1, 1], N=32, ratio=2, topk=1000,
                           name="long-rows-ties")
    case.k_rows[:] = 7
    case.k_scale[:] = np.float16(0.01).view(np.uint16)
    check(case)


def test_parity_long_rows_heavy_ties():
    """Long rows whose scores take few distinct values: the threshold key is
    shared by many positions and the lowest positions must win."""
    case = synth.make_case(83, [130000], [1], N=64, ratio=2, topk=1500, cand_mode="source",
                           cand_blocks=512, name="long-rows-few-values")
    rng = np.random.default_rng(5)
    base = rng.integers(-127, 128, size=(16, 128), dtype=np.int8)
    case.k_rows[:] = base[rng.integers(0, 16, size=case.k_rows.shape[0])]
    case.k_scale[:] = np.float16(0.01).view(np.uint16)
    check(case)


@pytest.mark.parametrize("idx", [1, 2, 3, 4, 5])
def test_parity_workloads_full_size(idx):
    """The five workloads at full size, every row checked against the oracle
    (the prefill workload's 4096 rows take the oracle about a minute)."""
    check(synth.config(idx))


def test_prefill_rows_with_heavy_ties_take_the_general_selection():
    """Prefill-shaped calls (many tokens per request): rows whose scores take
    a few distinct values put more entries at the threshold than the
    many-rows-per-SM selection keeps, so they are listed for the general
    selection; rows of equal scores do too. Both give the oracle's rows
    (equal scores rank by lower position)."""
    case = synth.make_case(84, [24000, 9000], [6, 3], N=64, ratio=2, topk=1500,
                           cand_mode="source", cand_blocks=512, name="prefill-ties")
    rng = np.random.default_rng(7)
    base = rng.integers(-127, 128, size=(6, 128), dtype=np.int8)
    case.k_rows[:] = base[rng.integers(0, 6, size=case.k_rows.shape[0])]
    case.k_scale[:] = np.float16(0.01).view(np.uint16)
    assert case.T > 2 * case.B                      # the prefill (group) path
    check(case)
    case.k_rows[:] = 5
    check(case)


def test_prefill_rows_longer_than_the_candidate_space_sample_a_threshold():
    """Prefill rows of 5K-12K positions (more than the 4608 candidates one
    CTA keeps): a sampled provisional threshold, one pass, exact select."""
    case = synth.make_case(85, [24000, 10000, 9500], [5, 3, 4], N=64, ratio=2, topk=2048,
                           cand_mode="source", cand_blocks=1024, name="prefill-sampled")
    assert case.T > 2 * case.B
    check(case)


def _sample_runs(n):
    """Entries of a row of n the many-rows-per-SM selection samples: 16
    evenly spread runs of 64 (each start rounded down to a multiple of 4)."""
    tid = np.arange(256)
    s0 = (((n * (tid >> 4)) // 16) & ~3) + 4 * (tid & 15)
    idx = (s0[:, None] + np.arange(4)[None, :]).reshape(-1)
    return idx[idx < n]


def _threshold_attempts(sc, want, cap=4608, sample=1024):
    """What the sampled pass keeps, attempt by attempt: the threshold is the
    floor of the 12-bit key bin holding the sample's rank-th best (rank 10%
    past the want-th best's expected sample rank, plus 24); a count outside
    [want, cap] scales the rank once by (want + cap) / 2 over the count."""
    def keys(f):
        u = np.asarray(f, dtype=np.float32).view(np.uint32).copy()
        u[(u << np.uint32(1)) == 0] = 0
        return np.where(u >> np.uint32(31) == 1, ~u, u | np.uint32(0x80000000)).astype(np.uint32)
    n = sc.size
    hist = np.bincount(keys(sc[_sample_runs(n)]) >> np.uint32(20), minlength=4096)
    k = keys(sc)
    rank = (want * sample * 11) // (10 * n) + 24
    got = []
    for attempt in range(2):
        b = 4095 - int(np.argmax(np.cumsum(hist[::-1]) >= rank))
        got.append(int(np.count_nonzero(k >= np.uint32(b << 20))))
        if want <= got[-1] <= cap:
            break
        rank = min(max(rank * ((want + cap) // 2) // got[-1] if got[-1] else 2 * rank + 32, 1),
                   sample - 64)
    return got


def test_prefill_rows_whose_sample_misjudges_the_threshold():
    """K scales raised by half at the entries the selection samples make the
    sample overrate its row: the first pass keeps fewer than TopK entries.
    The pass then runs once more with the rank scaled by what it kept; where
    that still misses, the row goes to the general selection. The input is
    checked to hold both kinds of row, and every row must equal the
    oracle's."""
    case = synth.make_case(85, [24000, 10000, 9500], [5, 3, 4], N=64, ratio=2, topk=2048,
                           cand_mode="source", cand_blocks=1024, name="prefill-misjudged")
    assert case.T > 2 * case.B
    prep = oracle.prepare(case)
    vis = oracle.run(prep, rows=np.arange(case.T), want_scores=False)["visible"]
    owner = np.searchsorted(case.cu_seqlens_q, np.arange(case.T), side="right") - 1
    for b in range(case.B):
        L = int(case.k_lens[b])
        ks = case.k_scale[case.k_row_start[b]:case.k_row_start[b] + L].view(np.float16)
        hit = np.zeros(L, bool)
        for t in np.flatnonzero(owner == b):
            idx = _sample_runs(int(vis[t]))
            hit[idx[idx < L]] = True
        ks[hit] = (ks[hit].astype(np.float32) * 1.5).astype(np.float16)
    prep = oracle.prepare(case)
    ora = oracle.run(prep, rows=np.arange(case.T), want_scores=True,
                     score_stride=int(case.k_lens.max()))
    kinds = set()
    for t in range(case.T):
        V = int(ora["visible"][t])
        if V > 4608:
            got = _threshold_attempts(ora["scores"][t][:V], case.topk)
            kinds.add((len(got), case.topk <= got[-1] <= 4608))
    assert (2, True) in kinds and (2, False) in kinds, kinds
    check(case)


def test_prefill_rows_between_32k_and_the_shared_memory_limit():
    """Prefill rows of 32K-45K positions: the many-rows-per-SM selection
    still takes them (position bitmaps of up to 1408 words, 16-bit
    positions); the candidate rows are longer than C."""
    case = synth.make_case(86, [90000, 70000], [3, 2], N=32, ratio=2, topk=2048,
                           cand_mode="source", cand_blocks=2048, name="prefill-44k")
    assert case.T > 2 * case.B
    assert 32768 < int(case.k_lens.max()) <= 44 * 1024
    check(case)


def test_prefill_rows_past_the_shared_memory_limit_take_the_long_row_passes():
    """Prefill rows longer than one CTA's shared memory (45056 keys) are
    listed by the many-rows-per-SM selection and ranked by the chunked
    long-row passes and the general selection."""
    case = synth.make_case(87, [120000, 3000], [3, 2], N=64, ratio=2, topk=2048,
                           cand_mode="source", cand_blocks=1024, name="prefill-long")
    assert case.T > 2 * case.B
    assert int(case.k_lens.max()) > 44 * 1024
    check(case)


def _fuzz_cases(n=40, seed=20261203):
    """A seeded sweep of small batches beyond the hand-picked ones: ratio 1
    or 2, 32 or 64 heads, every candidate mode, one to four requests of
    contexts from empty to 9000 raw tokens (some shorter than their query
    run), decode-shaped (one query per request) or prefill-shaped (up to 24),
    TopK from 1 to 2048 and 64 to 1024 candidate blocks, consumer lists valid
    or messy. Together they take the small-batch, stream and group paths."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 5))
        ratio = int(rng.integers(1, 3))
        N = int(rng.choice([32, 64]))
        mode = str(rng.choice(["none", "source", "consumer"]))
        raw = rng.integers(0, 9001, size=B)
        tiny = rng.random(B) < 0.2
        raw[tiny] = rng.integers(0, 40, size=int(tiny.sum()))
        ql = np.ones(B, dtype=np.int64) if rng.random() < 0.5 else rng.integers(1, 25, size=B)
        topk = int(rng.choice([1, 7, 64, 300, 1024, 2048]))
        C = int(rng.integers(1, 17)) * 64 if mode != "none" else 0
        policy = "messy" if mode == "consumer" and rng.random() < 0.5 else "valid"
        out.append(("fuzz%02d-%s-r%d-n%d" % (i, mode, ratio, N), int(rng.integers(0, 1 << 30)),
                    raw.tolist(), ql.tolist(), N, ratio, topk, mode, C, policy))
    return out


FUZZ = _fuzz_cases()


@pytest.mark.parametrize("p", FUZZ, ids=[p[0] for p in FUZZ])
def test_parity_seeded_sweep(p):
    name, seed, raw, ql, N, ratio, topk, mode, C, policy = p
    case = synth.make_case(seed, raw, ql, N=N, ratio=ratio, topk=topk, cand_mode=mode,
                           cand_blocks=C, cand_policy=policy, name=name)
    check(case)
