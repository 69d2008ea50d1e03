"""qli_run_static: the entry point for callers that cannot allocate device
memory when they call the indexer (for example a serving engine that gave all
free device memory to its KV-cache pool at start-up, or a C program with no
device allocator). It runs the same kernels on a fixed scratch array inside
the library instead of a caller workspace.

Checked through the C ABI against qli_run, the entry point with a caller
workspace: results must be identical (the tolerance every parity test here
uses: exact, as both sides run the same kernels). The static entry point is
called twice in a row on different inputs, so the second call starts from the
first call's leftover scratch contents. This file is collected last so that a
failure here cannot hide any other test; it also passes alone in a fresh
process.
"""
import numpy as np
import pytest

from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    qli.lib()


def _cases():
    return [
        synth.make_case(71, [9000, 3100, 20000, 640], [1, 1, 1, 1], N=64, ratio=1, topk=2048,
                        name="decode-none"),
        synth.make_case(72, [30000, 5000, 777], [1, 2, 1], N=64, ratio=2, topk=512,
                        cand_mode="source", cand_blocks=256, name="source"),
        synth.make_case(73, [20000, 9000], [1, 2], N=32, ratio=2, topk=1024,
                        cand_mode="consumer", cand_blocks=512, cand_policy="messy",
                        name="consumer"),
    ]


def test_static_entry_matches_workspace_entry():
    import torch
    cases = _cases()
    calls = [qli.Call(**synth.upload(c, "cuda")) for c in cases]
    want = []
    for call in calls:
        ws = call.alloc_workspace()
        idx, cand = call.run(ws)
        torch.cuda.synchronize()
        want.append((idx.clone(), None if cand is None else cand.clone()))
        idx.fill_(-7)                          # the static call must rewrite every output
        if cand is not None:
            cand.fill_(-7)
    # the static entry point, called on each case in a row
    for call, (w_idx, w_cand) in zip(calls, want):
        g_idx, g_cand = call.run_static()
        torch.cuda.synchronize()
        assert torch.equal(g_idx, w_idx)
        if w_cand is not None:
            assert torch.equal(g_cand, w_cand)
    # and the first case again, after the others left their scratch behind
    calls[0].indices.fill_(-7)
    g_idx, _ = calls[0].run_static()
    torch.cuda.synchronize()
    assert torch.equal(g_idx, want[0][0])


def test_static_entry_rejects_calls_beyond_its_scratch():
    # a 4.5M-position capacity needs ~18 MB of score scratch: above the array
    case = synth.make_case(74, [300], [1], N=64, ratio=2, topk=64, bt_stride=70000)
    call = qli.Call(**synth.upload(case, "cuda"))
    assert call.workspace_bytes() > 16 * 1024 * 1024
    with pytest.raises(qli.QLIError) as e:
        call.run_static()
    assert e.value.status == 5                 # QLI_ERR_WORKSPACE_TOO_SMALL, nothing launched


def test_static_entry_reports_device_side_errors():
    # a k_len past the block table's capacity is clamped on the device and
    # flagged in the error word, which the static caller reads back without a
    # workspace of its own
    import torch
    case = synth.make_case(75, [500, 300], [1, 1], N=64, ratio=2, topk=16)
    kw = synth.upload(case, "cuda")
    kw["k_lens"] = torch.tensor([250, 10 ** 6], dtype=torch.int32, device="cuda")
    call = qli.Call(**kw)
    call.run_static()
    assert call.static_device_error() & 2          # QLI_DEVERR_KLEN
    idx = call.indices.cpu().numpy()[:, 0, :]
    assert np.all(idx[idx >= 0] < case.bt_stride * case.rows_per_page)
    # the next call resets the word
    good = qli.Call(**synth.upload(case, "cuda"))
    good.run_static()
    assert good.static_device_error() == 0

