"""GPU parity of the single-launch path for small decode batches (INT8,
none/source mode, at most 64 tokens and 64 requests, at most 4096 positions
per request): a one-CTA kernel that zeroes the counters, then one kernel that
plans, scores and selects, launched to overlap it. Each
case first checks, through qli_launch_count, that the call takes that path;
the results must match the oracle under the same rule as every other parity
test (bit-equal scores, selections equal up to boundary ties).
"""
import zlib

import numpy as np
import pytest

from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth
from test_parity_gpu import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    qli.lib()


def is_small(case):
    call = qli.Call(**synth.upload(case, "cuda"))
    return (call.launches(0) == 2 and call.launches(qli.STAGE_PLAN) == 1
            and call.launches(qli.STAGE_SCORE) == 1 and call.launches(qli.STAGE_SELECT) == 0)


CASES = [
    # name, raw_lens, q_lens, N, ratio, topk, mode, C, extra
    ("small-none-r2-n64", [3000, 700, 8100], [1, 1, 2], 64, 2, 512, "none", 0, {}),
    ("small-none-r1-n32", [4000, 1, 130], [1, 1, 1], 32, 1, 300, "none", 0, {}),
    ("small-none-r1-n64-r64", [2000, 4090], [2, 1], 64, 1, 2048, "none", 0,
     dict(rows_per_page=64)),
    ("small-source-r2-n64", [7000, 3000], [2, 1], 64, 2, 200, "source", 64, {}),
    ("small-source-r1-n32-few-blocks", [500, 900, 2], [1, 2, 1], 32, 1, 64, "source", 128, {}),
    ("small-source-r2-n32-c2048", [8192, 4000], [1, 1], 32, 2, 2048, "source", 2048, {}),
    ("small-empty", [0, 0, 1], [1, 2, 1], 64, 2, 16, "source", 64, {}),
    ("small-topk1", [2000, 777], [1, 2], 64, 2, 1, "source", 64, {}),
    ("small-tile-exact", [256, 128, 512], [1, 1, 1], 64, 1, 64, "none", 0, {}),
    ("small-many-tokens", [900] * 32, [2] * 32, 64, 2, 100, "source", 64, {}),
]


@pytest.mark.parametrize("p", CASES, ids=[p[0] for p in CASES])
def test_small_path_parity(p):
    name, raw, ql, N, r, K, mode, C, extra = p
    case = synth.make_case(zlib.crc32(name.encode()) % 1000, raw, ql, N=N, ratio=r, topk=K,
                           cand_mode=mode, cand_blocks=C, name=name, **extra)
    assert is_small(case), name
    check(case)


def test_workload_1_takes_the_small_path():
    case = synth.config(1)
    assert is_small(case)
    check(case)


@pytest.mark.parametrize("what", ["over-positions", "fp8", "consumer", "prefill"])
def test_just_outside_the_limits_takes_the_staged_path(what):
    if what == "over-positions":
        case = synth.make_case(3, [8194 + 128, 100], [1, 1], N=64, ratio=2, topk=64)
    elif what == "fp8":
        case = synth.to_fp8(synth.make_case(3, [2000, 100], [1, 1], N=64, ratio=2, topk=64))
    elif what == "consumer":
        case = synth.make_case(3, [2000, 900], [1, 1], N=64, ratio=2, topk=64,
                               cand_mode="consumer", cand_blocks=64)
    else:
        case = synth.make_case(3, [2000, 900], [5, 1], N=64, ratio=2, topk=64)
    assert not is_small(case)
    if what == "fp8":
        from test_fp8_gpu import check as check_fp8   # FP8 scores: to a tolerance
        check_fp8(case)
    else:
        check(case)


def test_small_path_flags_bad_metadata():
    """The metadata is read as the planning stage reads it: lengths clamped
    and flagged, tokens assigned to requests by the same search; a page past
    the pool is flagged and read as page 0."""
    import torch
    case = synth.make_case(8, [500, 300, 900], [1, 1, 1], N=64, ratio=2, topk=16)
    assert is_small(case)
    kw = synth.upload(case, "cuda")
    kw["k_lens"] = torch.tensor([250, 10 ** 6, 450], dtype=torch.int32, device="cuda")
    kw["residual"] = torch.tensor([0, 0, 5], dtype=torch.int32, device="cuda")
    call = qli.Call(**kw)
    ws = call.alloc_workspace()
    call.run(ws)
    err = call.device_error(ws)
    assert err & 2 and err & 4                         # k_lens and residual clamped
    idx = call.indices.cpu().numpy()[:, 0, :]
    assert np.all(idx[idx >= 0] < case.bt_stride * case.rows_per_page)
    # a block-table entry past the pool, in the visible range of token 0
    kw = synth.upload(case, "cuda")
    bt = kw["block_table"].clone()
    bt[0, 1] = 10 ** 7
    kw["block_table"] = bt
    call = qli.Call(**kw)
    call.run(ws)
    assert call.device_error(ws) & 8
    # and a clean call on the same workspace starts from a clear error word
    call = qli.Call(**synth.upload(case, "cuda"))
    call.run(ws)
    assert call.device_error(ws) == 0


def test_small_path_stages_graphs_and_dirty_workspace():
    """PLAN (the zeroing kernel), SCORE (the one kernel) and SELECT (nothing) queued one
    by one, a CUDA graph of the call replayed, and a workspace full of
    garbage all give what one plain call gives."""
    import torch
    case = synth.make_case(32, [3000, 2500, 900], [1, 2, 1], N=64, ratio=2, topk=256,
                           cand_mode="source", cand_blocks=64)
    assert is_small(case)
    call = qli.Call(**synth.upload(case, "cuda"))
    ws = call.alloc_workspace()
    ws.fill_(0xFF)
    idx, cand = call.run(ws)
    torch.cuda.synchronize()
    want = (idx.clone(), cand.clone())
    check(case)

    def same():
        torch.cuda.synchronize()
        assert torch.equal(call.indices, want[0]) and torch.equal(call.cand, want[1])

    for rep in range(2):
        call.indices.fill_(-7)
        call.cand.fill_(-7)
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
    for rep in range(5):
        call.indices.fill_(-7)
        g.replay()
        same()
    assert call.device_error(ws) == 0


def test_small_path_static_entry():
    """The fixed-scratch entry point takes the same path."""
    import torch
    case = synth.make_case(33, [2000, 1500], [1, 1], N=32, ratio=2, topk=128)
    assert is_small(case)
    call = qli.Call(**synth.upload(case, "cuda"))
    ws = call.alloc_workspace()
    a = call.run(ws)[0].clone()
    call.indices.fill_(-7)
    call.run_static()
    torch.cuda.synchronize()
    assert torch.equal(call.indices, a)
    assert call.static_device_error() == 0
