"""The give-up path of the kernels' on-chip waits, exercised on the GPU
without a hang.

A test build of the library (QLI_WAIT_LIMIT_NS = 1 ms, QLI_TEST_STALL_EPILOGUE)
makes the stream kernel's epilogue wait on a barrier nothing arrives on. The
epilogue gives up after 1 ms; the MMA issuers, converters and the producer,
which wait on it in turn, give up too; each role drains the copies and MMAs it
started (those complete by themselves) before the CTA frees its tensor memory
and exits. The call must return, report QLI_DEVERR_TIMEOUT in the device error
word, and leave the context usable: the normal build then gives the oracle's
result on the same (dirty) workspace.
"""
import ctypes
import os
import time

import numpy as np
import pytest

import oracle
from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli, synth

pytestmark = pytest.mark.gpu

STALL_DIR = os.path.join(os.path.dirname(libbuild.LIB), "stall")
DEVERR_TIMEOUT = 16


@pytest.fixture(scope="module")
def stall_lib():
    libbuild.build()
    qli.lib()
    path = libbuild.build(out_dir=STALL_DIR,
                          defines=("QLI_WAIT_LIMIT_NS=1000000ull", "QLI_TEST_STALL_EPILOGUE"))
    return qli.lib(path)


def test_a_wait_that_runs_out_reports_and_leaves_the_context_usable(stall_lib):
    import torch
    # one context past 4096 compressed positions, so that the call takes the
    # streaming kernel (not the single-launch path for small batches)
    case = synth.make_case(91, [9000, 1200, 777], [1, 1, 1], N=64, ratio=2, topk=128,
                           name="stall")
    assert case.bt_stride * case.rows_per_page > 4096
    call = qli.Call(**synth.upload(case, "cuda"))
    ws = call.alloc_workspace()
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    st = stall_lib.qli_run(ctypes.byref(call.args), ws.data_ptr(), ws.numel(), stream)
    assert st == qli.OK
    word = ctypes.c_uint32(0)
    assert stall_lib.qli_read_device_error(ws.data_ptr(), ctypes.byref(word), stream) == qli.OK
    assert time.perf_counter() - t0 < 5.0
    assert word.value & DEVERR_TIMEOUT
    # the normal build on the same workspace: correct, and no flag left over
    want = oracle.run(oracle.prepare(case))
    for _ in range(2):
        call.indices.fill_(-7)
        idx, _ = call.run(ws)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy()[:, 0, :], want["indices"])
        assert call.device_error(ws) == 0
