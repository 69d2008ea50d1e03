"""Pins of the attention consumer's oracle (oracle/csa.py) to things other
than itself: PyTorch's BF16 type and its scaled-dot-product attention, closed
forms and invariants. CPU only.

The definition (blog "DeepSeek V4.1-Flash 登陆昇腾 · 需求故事（PR 16925）",
section 四; guide "DeepSeek V4.1 QLI V2 与候选集成", section 编译范围): softmax
attention of each query head over the KV rows of the positions the indexer
selected, one shared KV head, BF16 inputs, -1 entries skipped.
"""
import importlib.util
import os

import numpy as np
import pytest

from sparse_attention_indexer_qli_gb300 import synth

if os.environ.get("CSA_ORACLE_PATH"):
    # the mutation check points the pins at a mutated copy of the oracle
    _spec = importlib.util.spec_from_file_location("csa_under_test", os.environ["CSA_ORACLE_PATH"])
    csa = importlib.util.module_from_spec(_spec)
    _spec.loader.exec_module(csa)
else:
    from oracle import csa

torch = pytest.importorskip("torch")
SCALE = 1.0 / np.sqrt(512.0)


def small_case(seed=5, raw=(700, 260), ql=(3, 2), H=4, ratio=2, topk=64, count=None):
    case = synth.make_case(seed, list(raw), list(ql), N=32, ratio=ratio, topk=8)
    return synth.add_attention(case, H=H, topk=topk, count=count)


def test_bf16_decoding_matches_torch():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = csa.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def sdpa(q_bits, kv_bits, scale):
    """PyTorch's scaled-dot-product attention, float64, one KV head shared by
    every query head."""
    q = torch.from_numpy(csa.bf16_to_f64(q_bits))[None, :, None, :]          # [1, H, 1, D]
    kv = torch.from_numpy(csa.bf16_to_f64(kv_bits))[None, None, :, :]        # [1, 1, n, D]
    kv = kv.expand(1, q.shape[1], kv.shape[2], kv.shape[3])
    return torch.nn.functional.scaled_dot_product_attention(q, kv, kv, scale=scale)[0, :, 0, :].numpy()


@pytest.mark.parametrize("ratio", [1, 2])
def test_all_positions_equal_dense_attention(ratio):
    # every position of the request listed, in shuffled order with -1 holes:
    # the same as dense attention over the request's rows (a library routine)
    case = small_case(ratio=ratio, topk=1024)
    rng = np.random.default_rng(1)
    for t in range(case.T):
        b = csa.request_of(case.cu_seqlens_q, t)
        lk = int(case.k_lens[b])
        row = np.full(1024, -1, np.int32)
        perm = rng.permutation(lk)
        slots = np.sort(rng.choice(1024, size=lk, replace=False))
        row[slots] = perm
        case.attn_indices[t, 0] = row
    o, lse = csa.attention(case, SCALE)
    for t in range(case.T):
        b = csa.request_of(case.cu_seqlens_q, t)
        want = sdpa(case.q_attn[t], case.kv_of(b), SCALE)
        assert np.allclose(o[t], want, rtol=1e-12, atol=1e-12)


def test_one_position_returns_its_row_exactly():
    case = small_case()
    case.attn_indices[:] = -1
    for t in range(case.T):
        case.attn_indices[t, 0, 5] = 17 + t
    o, lse = csa.attention(case, SCALE)
    for t in range(case.T):
        b = csa.request_of(case.cu_seqlens_q, t)
        row = csa.bf16_to_f64(case.kv_of(b)[17 + t])
        assert np.array_equal(o[t], np.broadcast_to(row, o[t].shape))
        q = csa.bf16_to_f64(case.q_attn[t])
        assert np.allclose(lse[t], SCALE * (q @ row), rtol=1e-14, atol=0)


def test_a_position_listed_twice_counts_twice():
    case = small_case()
    case.attn_indices[:] = -1
    case.attn_indices[:, 0, 0] = 9
    o1, lse1 = csa.attention(case, SCALE)
    case.attn_indices[:, 0, 1] = 9
    o2, lse2 = csa.attention(case, SCALE)
    assert np.allclose(o1, o2, rtol=1e-14, atol=1e-14)
    assert np.allclose(lse2, lse1 + np.log(2.0), rtol=1e-14, atol=1e-14)


def test_order_and_holes_do_not_matter():
    case = small_case(topk=64)
    o1, lse1 = csa.attention(case, SCALE)
    rng = np.random.default_rng(2)
    for t in range(case.T):
        row = case.attn_indices[t, 0].copy()
        case.attn_indices[t, 0] = row[rng.permutation(row.size)]   # -1 now in the middle
    o2, lse2 = csa.attention(case, SCALE)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse1, lse2, rtol=1e-12, atol=1e-12)


def test_empty_list_gives_zeros_and_minus_infinity():
    case = small_case()
    case.attn_indices[1] = -1
    o, lse = csa.attention(case, SCALE)
    assert np.all(o[1] == 0.0) and np.all(lse[1] == -np.inf)
    assert np.all(np.isfinite(lse[0]))


def test_zero_scale_averages_the_rows():
    case = small_case(topk=40)
    o, lse = csa.attention(case, 0.0)
    for t in range(case.T):
        b = csa.request_of(case.cu_seqlens_q, t)
        js = case.attn_indices[t, 0]
        js = js[js >= 0]
        mean = csa.bf16_to_f64(case.kv_of(b)[js]).mean(axis=0)
        assert np.allclose(o[t], np.broadcast_to(mean, o[t].shape), rtol=1e-13, atol=1e-13)
        assert np.allclose(lse[t], np.log(js.size), rtol=1e-14)


def test_a_dominant_score_selects_its_row_without_overflow():
    # scores spread by thousands: exp(s) alone would overflow; the result is
    # the best row exactly and lse its score
    case = small_case(topk=16)
    o, lse = csa.attention(case, 1.0e4)
    for t in range(case.T):
        b = csa.request_of(case.cu_seqlens_q, t)
        js = case.attn_indices[t, 0]
        js = js[js >= 0]
        rows = csa.bf16_to_f64(case.kv_of(b)[js])
        s = 1.0e4 * (rows @ csa.bf16_to_f64(case.q_attn[t]).T)      # [n, H]
        assert np.all(np.isfinite(o[t])) and np.all(np.isfinite(lse[t]))
        for h in range(s.shape[1]):
            top = np.sort(s[:, h])
            if top[-1] - top[-2] > 800.0:
                assert np.array_equal(o[t, h], rows[np.argmax(s[:, h])])
                assert lse[t, h] == top[-1]


def test_paging_does_not_matter():
    case = small_case(ratio=1, raw=(300, 1000), topk=100)
    o1, lse1 = csa.attention(case, SCALE)                       # through the pages
    o2, lse2 = csa.attention(case, SCALE, rows=csa.rows_from_logical(case))
    assert np.array_equal(o1, o2) and np.array_equal(lse1, lse2)


def test_tokens_read_their_own_request():
    # two requests with different rows: each token's output must come from
    # its own request's rows (dense attention over that request)
    case = small_case(raw=(64, 64), ql=(1, 1), topk=32)
    for t in range(2):
        case.attn_indices[t, 0] = np.arange(32)
    o, _ = csa.attention(case, SCALE)
    for t in range(2):
        want = sdpa(case.q_attn[t], case.kv_of(t)[:32], SCALE)
        assert np.allclose(o[t], want, rtol=1e-12, atol=1e-12)
        other = sdpa(case.q_attn[t], case.kv_of(1 - t)[:32], SCALE)
        assert not np.allclose(o[t], other, rtol=1e-6, atol=1e-6)
