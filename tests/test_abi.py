"""C-ABI library checks that need no GPU: it builds for sm_103a, loads, exports
every function include/qli.h declares, matches the binding's struct layout, and
its host validation enforces the contract of the guide "DeepSeek V4.1 QLI V2
与候选集成" (sections 数据流, 当前 A3 契约, 构建与回归覆盖). No call here reaches
the device: validation returns before any CUDA call, and the pointers are
never dereferenced."""
import ctypes
import json
import os
import re
import subprocess

import pytest

from sparse_attention_indexer_qli_gb300 import build as libbuild
from sparse_attention_indexer_qli_gb300 import qli

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qli.h")


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return qli.lib()


def declared_functions():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(qli_\w+)\s*\(", txt, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert set(qli.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", libbuild.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (qli_\w+)$", out, re.M))
    missing = set(declared_functions()) - exported
    assert not missing, missing
    assert L.qli_abi_version() == 1


def test_struct_layout_matches_header(tmp_path):
    fields = [f for f, _ in qli.Args._fields_]
    src = ['#include <stddef.h>', '#include <stdio.h>', '#include "qli.h"', 'int main(void){',
           'printf("%zu\\n", sizeof(qli_args));']
    src += ['printf("%%zu\\n", offsetof(qli_args, %s));' % f for f in fields]
    src += ['return 0;}']
    c = tmp_path / "probe.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(c), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(qli.Args)
    for f, off in zip(fields, vals[1:]):
        assert getattr(qli.Args, f).offset == off, f


def good_args(mode="none", T=4, B=2, N=64, ratio=2, K=16, C=64):
    a = qli.Args()
    p = 0x100000          # fake, 16-byte aligned; validation never dereferences
    R, stride = (64, 131072) if ratio == 2 else (128, 147712)
    a.q = p; a.q_stride_t = N * 128; a.q_stride_h = 128
    a.T, a.N, a.D = T, N, 128
    a.cu_seqlens_q = p; a.B = B; a.k_lens = p
    a.residual = p if ratio == 2 else None
    a.cache = p; a.page_stride = stride; a.rows_per_page = R
    a.k_offset = R * 1024; a.scale_offset = R * 1024 + R * 128; a.num_pages = 100
    a.block_table = p; a.bt_stride = 8
    a.head_weights = p; a.q_scale = p
    a.ratio = ratio; a.mask_mode = 3; a.quant_mode = 2; a.layout_q = 1; a.layout_k = 2
    a.topk = K; a.cand_mode = qli.CAND_MODES[mode]; a.cand_blocks = C if mode != "none" else 0
    a.block_size = 8
    if mode == "consumer":
        a.cand_in = p; a.cand_in_numel = T * C
    if mode == "source":
        a.cand_out = p; a.cand_out_numel = T * C
    a.indices_out = p; a.indices_numel = T * K
    return a


def status(L, a):
    return L.qli_validate(ctypes.byref(a))


@pytest.mark.parametrize("mode", ["none", "source", "consumer"])
@pytest.mark.parametrize("ratio", [1, 2])
@pytest.mark.parametrize("N", [32, 64])
def test_contract_accepts(L, mode, ratio, N):
    assert status(L, good_args(mode, ratio=ratio, N=N)) == 0


def test_fp8_quant_mode_is_accepted(L):
    a = good_args("source")
    a.quant_mode = qli.QUANT_FP8
    assert status(L, a) == 0


def _with(mode="none", **kw):
    a = good_args(mode, **{k: v for k, v in kw.items() if k in ("T", "B", "N", "ratio", "K", "C")})
    for k, v in kw.items():
        if k not in ("T", "B", "N", "ratio", "K", "C"):
            setattr(a, k, v)
    return a


REJECT = [
    # (mode, overrides, expected status) — contract of section 当前 A3 契约
    ("none", dict(layout_q=3), 2),                     # BSND query rejected
    ("none", dict(layout_k=3), 2),                     # non-paged key rejected
    ("none", dict(quant_mode=3), 2),                   # quant modes other than 1 (FP8) and 2 (INT8)
    ("none", dict(quant_mode=4), 2),
    ("none", dict(mask_mode=1), 2),
    ("none", dict(N=16), 2),
    ("none", dict(D=64), 2),
    ("none", dict(ratio=4), 2),
    ("none", dict(block_size=16), 2),
    ("none", dict(rows_per_page=32), 2),
    ("none", dict(cand_mode=4), 2),
    ("none", dict(K=0), 1),
    ("none", dict(K=2049), 1),
    ("source", dict(C=32), 1),                         # below 64
    ("source", dict(C=2112), 1),                       # above 2048
    ("source", dict(C=100), 1),                        # not a multiple of 64
    ("consumer", dict(cand_in=None), 3),               # consumer without a source
    ("source", dict(cand_out=None), 1),
    ("none", dict(indices_numel=5), 1),
    ("none", dict(q=0x100008), 6),                     # misaligned
    ("none", dict(page_stride=131080), 6),
    ("none", dict(k_offset=65544), 6),
    ("none", dict(q_stride_h=136), 6),
    ("none", dict(k_offset=131072 - 100), 1),          # index K past the page end
    ("none", dict(num_pages=0), 1),
    ("none", dict(B=0), 1),
]


@pytest.mark.parametrize("mode,over,want", REJECT)
def test_contract_rejects(L, mode, over, want):
    assert status(L, _with(mode, **over)) == want


@pytest.mark.parametrize("mode,over,want", REJECT)
def test_static_entry_rejects_like_the_workspace_entry(L, mode, over, want):
    # host validation runs before either entry point touches the device
    a = _with(mode, **over)
    assert L.qli_run_static(ctypes.byref(a), None) == want
    assert L.qli_run(ctypes.byref(a), 0x100000, 1 << 40, None) == want


def test_residual_with_ratio_one_is_rejected(L):
    a = good_args(ratio=1)
    a.residual = 0x100000
    assert status(L, a) == 4          # "residual must be absent when ratio is 1"
    assert L.qli_run_static(ctypes.byref(a), None) == 4


def test_candidate_extent_is_tokens_times_blocks(L):
    # section 构建与回归覆盖: a TND candidate tensor holds T * N_k * blocks
    # elements; multiplying by the batch size again would wrongly reject a
    # mixed-request consumer.
    a = good_args("consumer", T=6, B=3, C=128)
    assert status(L, a) == 0
    a.cand_in_numel = 6 * 3 * 128
    assert status(L, a) == 1


def test_contract_ranges_match_the_page(L):
    with open(os.path.join(ROOT, "tests", "golden", "contract.json")) as f:
        c = json.load(f)["contract"]
    lo, hi = c["topk_range"]
    for K, ok in ((lo, True), (hi, True), (lo - 1, False), (hi + 1, False)):
        assert (status(L, _with("none", K=K)) == 0) == ok
    lo, hi = c["cand_blocks_range"]
    for C, ok in ((lo, True), (hi, True), (lo - c["cand_blocks_multiple"], False),
                  (hi + c["cand_blocks_multiple"], False), (lo + 1, False)):
        assert (status(L, _with("source", C=C)) == 0) == ok
    for N in (16, 32, 48, 64, 128):
        assert (status(L, _with("none", N=N)) == 0) == (N in c["heads"])


def test_workspace_size_and_launch_counts(L):
    a = good_args("source", T=4, B=2)
    n = ctypes.c_size_t(0)
    assert L.qli_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    # at least the FP32 score rows: T * bt_stride * rows_per_page * 4 bytes
    assert n.value >= 4 * 8 * 64 * 4
    cnt = ctypes.c_int32(0)
    # a small decode batch: two kernels (the plan stage zeroes counters, the
    # score stage's kernel also selects)
    assert L.qli_launch_count(ctypes.byref(a), 0, ctypes.byref(cnt)) == 0
    assert cnt.value == 2
    for stage, want in ((1, 1), (2, 1), (3, 0)):
        assert L.qli_launch_count(ctypes.byref(a), stage, ctypes.byref(cnt)) == 0
        assert cnt.value == want
    # more tokens than two per request: the staged path, three stages or more
    big = good_args("source", T=5, B=2)
    assert L.qli_launch_count(ctypes.byref(big), 0, ctypes.byref(cnt)) == 0
    assert cnt.value >= 3
    off, stride = ctypes.c_size_t(0), ctypes.c_int64(0)
    assert L.qli_scores_layout(ctypes.byref(a), ctypes.byref(off), ctypes.byref(stride)) == 0
    assert stride.value >= 8 * 64 and off.value % 256 == 0
    # T == 0: nothing to do, no workspace
    z = good_args("none", T=0, K=16)
    z.indices_numel = 0
    assert L.qli_workspace_size(ctypes.byref(z), ctypes.byref(n)) == 0 and n.value == 0


def test_status_strings(L):
    for s in range(9):
        assert L.qli_status_string(s)
    assert L.qli_status_string(123) == b"unknown status"


def test_torch_packing_matches_numpy_packing():
    torch = pytest.importorskip("torch")
    from sparse_attention_indexer_qli_gb300 import synth
    case = synth.make_case(3, [300, 70, 0], [2, 1, 1], N=32, ratio=2, topk=8)
    a = case.pack_pages_numpy(filler=False)
    b = case.pack_pages_torch("cpu", filler=False).numpy()
    assert (a == b).all()


# ---- query quantiser and index-K writer: host validation only --------------

A16 = 1 << 20          # a fake, 16-byte-aligned address (never dereferenced)


def test_quantize_q_validation(L):
    f = L.qli_quantize_q
    assert f(None, 0, None, None, None) == qli.OK             # nothing to do, nothing launched
    assert f(A16, -1, A16, A16, None) == 1                    # QLI_ERR_INVALID_ARG
    assert f(None, 4, A16, A16, None) == 1
    assert f(A16, 4, None, A16, None) == 1
    assert f(A16 + 8, 4, A16, A16, None) == 6                 # QLI_ERR_ALIGNMENT
    assert f(A16, 4, A16 + 4, A16, None) == 6
    assert f(A16, 4, A16, A16 + 1, None) == 6


def _w(L, **kw):
    a = dict(k=A16, n=4, slot=A16, cache=A16, num_pages=10, page_stride=131072,
             R=64, k_off=65536, s_off=65536 + 8192, err=None)
    a.update(kw)
    return L.qli_write_index_k(a["k"], a["n"], a["slot"], a["cache"], a["num_pages"],
                               a["page_stride"], a["R"], a["k_off"], a["s_off"], a["err"], None)


def test_write_index_k_validation(L):
    assert _w(L, n=0, k=None, slot=None, cache=None) == qli.OK
    assert _w(L, n=-1) == 1
    assert _w(L, k=None) == 1
    assert _w(L, slot=None) == 1
    assert _w(L, cache=None) == 1
    assert _w(L, num_pages=-1) == 1
    assert _w(L, R=32) == 2                                     # QLI_ERR_UNSUPPORTED
    assert _w(L, k_off=131072 - 64 * 128 + 16) == 1             # index K past the page
    assert _w(L, s_off=131072 - 64 * 2 + 2) == 1                # scales past the page
    assert _w(L, k=A16 + 8) == 6
    assert _w(L, cache=A16 + 8) == 6
    assert _w(L, page_stride=131072 + 8) == 6
    assert _w(L, k_off=65536 + 8) == 6
    assert _w(L, s_off=65536 + 8192 + 1) == 6
    assert _w(L, slot=A16 + 4) == 6
    assert _w(L, err=A16 + 2) == 6


# ---- attention over the selected positions: layout and host validation ------

def test_attn_struct_layout_matches_header(tmp_path):
    fields = [f for f, _ in qli.AttnArgs._fields_]
    src = ['#include <stddef.h>', '#include <stdio.h>', '#include "qli.h"', 'int main(void){',
           'printf("%zu\\n", sizeof(qli_attn_args));']
    src += ['printf("%%zu\\n", offsetof(qli_attn_args, %s));' % f for f in fields]
    src += ['return 0;}']
    c = tmp_path / "probe.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(c), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(qli.AttnArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(qli.AttnArgs, f).offset == off, f


def good_attn(T=4, B=2, H=64, K=256):
    a = qli.AttnArgs()
    p = 0x100000
    a.q = p; a.q_stride_t = H * 512; a.q_stride_h = 512
    a.T, a.H, a.D = T, H, 512
    a.cu_seqlens_q = p; a.B = B
    a.cache = p; a.page_stride = 147712; a.num_pages = 100; a.rows_per_page = 128
    a.kv_offset = 0; a.block_table = p; a.bt_stride = 8
    a.indices = p; a.K = K; a.scale = 0.044
    a.out = p; a.out_stride_t = H * 512; a.out_stride_h = 512
    a.lse = p; a.err_word = None
    return a


ATTN_REJECT = [
    (dict(D=576), 2), (dict(H=16), 2), (dict(H=48), 2), (dict(H=160), 2),
    (dict(rows_per_page=32), 2), (dict(K=0), 1), (dict(K=2049), 1),
    (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(q=None), 1), (dict(indices=None), 1), (dict(out=None), 1),
    (dict(kv_offset=147712 - 128 * 1024 + 16), 1),     # KV rows past the page end
    (dict(q=0x100008), 6), (dict(q_stride_h=500), 1), (dict(q_stride_h=524), 6),
    (dict(page_stride=147720), 6), (dict(kv_offset=8), 6), (dict(out=0x100001), 6),
    (dict(B=0), 1), (dict(num_pages=0), 1),
]


@pytest.mark.parametrize("over,want", ATTN_REJECT)
def test_attention_contract_rejects(L, over, want):
    a = good_attn()
    for k, v in over.items():
        setattr(a, k, v)
    assert L.qli_sparse_attention(ctypes.byref(a), None) == want


def test_attention_nothing_to_do(L):
    a = good_attn(T=0)
    assert L.qli_sparse_attention(ctypes.byref(a), None) == qli.OK
