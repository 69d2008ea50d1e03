"""The GPU parity rule (tests/parity_rules.py) rejects every kind of wrong
selection row it is meant to catch, and accepts a genuine boundary tie.

Hand-made rows against a hand-made oracle row (guide "DeepSeek V4.1 QLI V2 与
候选集成", section 数据流: ascending IDs, -1 only at the end, eligibility, the
pinned last visible block)."""
import numpy as np
import pytest

from parity_rules import assert_selection

# ten positions; 7 and 8 tie the boundary (score 5.0) within 1e-3 relative
SCORES = {0: 1.0, 1: 9.0, 2: 8.0, 3: 5.0, 4: 2.0, 5: 7.0, 6: 0.5, 7: 5.0004, 8: 4.9998, 9: 3.0}
ORACLE = np.array([1, 2, 3, 5, -1, -1])    # best four: 9, 8, 7, 5.0 (3 wins the tie by position)


def score_of(j):
    return SCORES[j]


def all_eligible(j):
    return 0 <= j < 10


def check(row, eligible=all_eligible, pinned=None, oracle=ORACLE, score=score_of):
    assert_selection(np.array(row), oracle, score, eligible, "row", pinned=pinned)


def test_identical_rows_pass():
    check(ORACLE)


def test_a_boundary_tie_passes():
    check([1, 2, 5, 7, -1, -1])            # 7 (5.0004) instead of 3 (5.0)


def test_a_clearly_worse_element_fails():
    with pytest.raises(AssertionError):
        check([1, 2, 4, 5, -1, -1])        # 4 scores 2.0


def test_an_ineligible_near_tie_fails():
    # 7 ties the boundary but is not eligible (e.g. outside the consumer's blocks)
    with pytest.raises(AssertionError, match="ineligible"):
        check([1, 2, 5, 7, -1, -1], eligible=lambda j: j != 7)


def test_a_hole_in_the_padding_fails():
    with pytest.raises(AssertionError, match="padding"):
        check([1, 2, -1, 3, 5, -1])


def test_descending_order_fails():
    with pytest.raises(AssertionError, match="ascending"):
        check([2, 1, 3, 5, -1, -1])


def test_duplicates_fail():
    with pytest.raises(AssertionError):
        check([1, 1, 3, 5, -1, -1])


def test_a_missing_element_fails():
    with pytest.raises(AssertionError):
        check([1, 2, 3, -1, -1, -1])


# candidate rows: blocks 0..5, block 5 is the pinned last block with a low score
BLOCK_SCORES = {0: 9.0, 1: 5.0, 2: 4.9999, 3: 1.0, 4: 8.0, 5: 0.1}
BLOCK_ORACLE = np.array([0, 1, 4, 5])      # best three of 0..4, plus the pinned 5


def bscore(k):
    return BLOCK_SCORES[k]


def test_candidate_tie_at_the_ranked_boundary_passes():
    check([0, 2, 4, 5], oracle=BLOCK_ORACLE, score=bscore, pinned=5)


def test_a_low_pinned_block_does_not_widen_the_tolerance():
    # measured from the pinned block's 0.1, block 3 (1.0) would be far off
    # anyway; measured from a pinned score near it, it would pass: the bound
    # must come from the ranked blocks only (5.0), where 3 is clearly worse
    scores = dict(BLOCK_SCORES)
    scores[5] = 1.0005
    with pytest.raises(AssertionError, match="tie"):
        check([0, 3, 4, 5], oracle=BLOCK_ORACLE, score=lambda k: scores[k], pinned=5)


def test_a_missing_pinned_block_fails():
    with pytest.raises(AssertionError):
        check([0, 1, 2, 4], oracle=BLOCK_ORACLE, score=bscore, pinned=5)
