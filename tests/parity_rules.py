"""The rule a GPU selection row is checked with against the oracle's row.

Guide "DeepSeek V4.1 QLI V2 与候选集成", section 数据流: a selection row holds
the chosen position (or block) IDs in ascending order with the -1 padding at
the end; a position is eligible only while visible (and, for a consumer,
inside one of the token's given candidate blocks); the last visible block is
always a candidate. Two rows may differ only where the differing elements'
oracle scores tie the selection boundary within REL_TIE_TOL relative.

The boundary is the lowest oracle score among the oracle's ranked elements.
For a candidate row the pinned last block is not ranked (it is in the row
whatever its score), so it is left out of the boundary and checked on its own.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np

REL_TIE_TOL = 1e-3


def assert_selection(gpu_row, ora_row, score_of: Callable[[int], float],
                     eligible: Callable[[int], bool], what, pinned: Optional[int] = None):
    """Raises AssertionError unless gpu_row is an acceptable selection given
    the oracle's ora_row.

    score_of(j): the oracle score of element j; eligible(j): whether j may be
    selected at all; pinned: an element both rows must hold regardless of its
    score (the last visible block of a candidate row), or None.
    """
    gpu_row = np.asarray(gpu_row)
    ora_row = np.asarray(ora_row)
    assert gpu_row.shape == ora_row.shape, (what, gpu_row.shape, ora_row.shape)
    # layout of the GPU row: valid IDs first, ascending, then -1 only
    valid = gpu_row >= 0
    n = int(valid.sum())
    assert np.all(valid[:n]) and np.all(gpu_row[n:] == -1), (what, "padding not at the tail")
    assert np.all(np.diff(gpu_row[:n]) > 0), (what, "not strictly ascending")
    if np.array_equal(gpu_row, ora_row):
        return
    g = set(gpu_row[:n].tolist())
    o = set(ora_row[ora_row >= 0].tolist())
    assert len(g) == len(o), (what, "count", len(g), len(o))
    for j in g - o:
        assert eligible(j), (what, "ineligible element selected", j)
    if pinned is not None:
        assert pinned in g and pinned in o, (what, "pinned element missing", pinned)
    ranked = o - ({pinned} if pinned is not None else set())
    assert ranked, (what, "rows differ with nothing ranked")
    bound = min(score_of(j) for j in ranked)
    for j in g ^ o:
        s = score_of(j)
        assert abs(s - bound) <= REL_TIE_TOL * abs(bound), (what, "not a boundary tie", j, s, bound)
