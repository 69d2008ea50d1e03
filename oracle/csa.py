"""CPU oracle of the sparse attention consumer of the indexer's output (the
compressed-attention stage) — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the bench's CPU-baseline leg may import
this module. It shares no code with the CUDA library and reads nothing the
CUDA path produced.

What is computed (sources are web pages, cited by title and section):
  * blog "DeepSeek V4.1-Flash 登陆昇腾 · 需求故事（PR 16925）", section 四
    (the attention forward): the indexer's compressed indices feed the
    sparse attention call that follows it; the attention output is then
    inverse-rotated in place on its tail [nope_head_dim, head_dim), so the
    output lives in the space of the cached rows;
  * guide "DeepSeek V4.1 QLI V2 与候选集成", section 编译范围, and blog
    "DeepSeek V4.1-Flash CED·CSA2 架构拆解 × vllm-ascend 性能协助点"
    (architecture table): the sparse attention is compiled only for BF16
    TND queries over the PA_BBND paged cache, with a single-KV-head CSA
    specialisation;
  * guide section 数据流 and the blog's page-packing code: each page holds
    the KV rows first, then the index K and its FP16 scales.

Readings taken where the pages are silent (each is listed in the design
notes):
  * one KV row per compressed position: 1024 bytes = 512 BF16 values at the
    start of its page row (147712 = 128 * (1024 + 128 + 2) for ratio-1 pages);
    the row serves as both key and value (one shared KV head);
  * for query token t and head h, over the listed positions J(t) (entries
    >= 0 of the token's index row; -1 entries are skipped; a position listed
    twice counts twice):
        s_j   = scale * sum_d q[t,h,d] * kv_j[d]
        o     = sum_j exp(s_j - m) kv_j / sum_j exp(s_j - m),  m = max_j s_j
        lse   = m + log(sum_j exp(s_j - m))      (natural logarithm)
    an empty J gives o = 0 and lse = -inf;
  * the softmax scale is a caller argument (the pages print none; the tests
    and the bench use 1/sqrt(512));
  * the sliding-window stage, the attention sinks and the way the two stages
    combine are not described on the pages and are not part of this op (the
    log-sum-exp output is what such a combination would need).

Everything here is float64 (numpy); BF16 inputs decode exactly.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) to float64: the pattern is the top half of
    the FP32 pattern of the same value."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rows_from_pages(pages: np.ndarray, kv_offset: int, rows_per_page: int,
                    block_table: np.ndarray) -> Callable[[int, np.ndarray], np.ndarray]:
    """Row reader over a page pool ([num_pages, page_stride] uint8): position j
    of request b is row j % R of page block_table[b, j // R]; its 512 BF16
    values start at byte kv_offset + (j % R) * 1024 of the page."""
    R = int(rows_per_page)

    def read(b: int, js: np.ndarray) -> np.ndarray:
        out = np.empty((len(js), 512), dtype=np.uint16)
        for i, j in enumerate(js):
            page = int(block_table[b, int(j) // R])
            at = kv_offset + (int(j) % R) * 1024
            out[i] = pages[page, at:at + 1024].view(np.uint16)
        return out

    return read


def rows_from_logical(case) -> Callable[[int, np.ndarray], np.ndarray]:
    """Row reader over the case's logical (unpaged) KV rows."""
    def read(b: int, js: np.ndarray) -> np.ndarray:
        return case.kv_of(b)[np.asarray(js, dtype=np.int64)]
    return read


def request_of(cu_seqlens: np.ndarray, t: int) -> int:
    """The request whose query range [cu[b], cu[b+1]) holds token t."""
    b = 0
    while b + 1 < len(cu_seqlens) - 1 and cu_seqlens[b + 1] <= t:
        b += 1
    return b


def attention_token(q_bits: np.ndarray, kv_bits: np.ndarray, scale: float):
    """One token: q_bits [H, 512] BF16, kv_bits [n, 512] BF16 (the listed rows,
    in list order). Returns (o [H, 512], lse [H]) in float64."""
    q = bf16_to_f64(q_bits)
    H = q.shape[0]
    if kv_bits.shape[0] == 0:
        return np.zeros((H, q.shape[1])), np.full(H, -np.inf)
    kv = bf16_to_f64(kv_bits)
    s = scale * (kv @ q.T)                 # [n, H]
    m = s.max(axis=0)                      # [H]
    p = np.exp(s - m)                      # [n, H]
    l = p.sum(axis=0)
    o = (p.T @ kv) / l[:, None]
    return o, m + np.log(l)


def attention(case, scale: float, tokens: Optional[Sequence[int]] = None,
              rows: Optional[Callable] = None):
    """The consumer over the case's attention inputs (synth.add_attention):
    q_attn [T, H, 512], attn_indices [T, 1, K], KV rows read by `rows`
    (default: through the block table from the case's own page packing).
    Returns (o [n, H, 512] float64, lse [n, H] float64) for the listed tokens."""
    if rows is None:
        pages = case.pack_pages_numpy(filler=False)
        rows = rows_from_pages(pages, 0, case.rows_per_page, case.block_table)
    tokens = range(case.T) if tokens is None else tokens
    outs, lses = [], []
    for t in tokens:
        b = request_of(case.cu_seqlens_q, int(t))
        js = case.attn_indices[int(t), 0]
        js = js[js >= 0]
        o, lse = attention_token(case.q_attn[int(t)], rows(b, js), scale)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)
