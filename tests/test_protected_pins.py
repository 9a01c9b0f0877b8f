"""Pins of the oracle's protected-row rule against row sets written out by hand.

RedKnot-MLA paper, protected-set paragraph: the protected set is the union of
the query rows Q, the new rows N, the dirty rows D, the first and last rows of
every relocated segment (B_128), the Indexer's rows (I_top) and the recent
tail; a controller widens it to a fixed share (10 / 20 / 25 %) of the
candidate rows.  The Indexer's rows are stood in for by seeded draws: a
uniform per row (Bernoulli rule) or a row permutation (budget rule).

Each expected set below was worked out by hand from that rule on a geometry
small enough to check by eye; none comes from running a builder.  They catch
the plausible slips of an implementation: boundary rows dropped from the
Bernoulli branch, u <= p instead of u < p, the permutation walked backwards,
boundary rows counted against the fill, the fill taken from boundary or new
rows, the target rounded down, dirty rows charged to the budget.
"""
import numpy as np

import oracle as O


def _rows(mask):
    return set(np.nonzero(mask)[0].tolist())


def test_bernoulli_branch_hand_set():
    # two cached segments (10 rows at 0, 8 rows at 10) and 4 new rows at 18;
    # boundary 2: rows 0,1,8,9 and 10,11,16,17
    segs = [(10, 0, False), (8, 10, False), (4, 18, True)]
    T = 22
    u = np.full(T, 0.5)
    u[[0, 1, 8, 9, 10, 11, 16, 17]] = 0.95   # boundary rows drawn high: kept anyway
    u[3] = 0.10                               # below p: protected
    u[6] = 0.2999                             # below p: protected
    u[7] = 0.30                               # equal to p: not protected (u < p)
    u[13] = 0.0                               # below p: protected
    u[18:22] = 0.99                           # new rows: protected whatever u says
    got = O.build_protected(T, segs, boundary=2, p_random=0.30, budget=0.0, none=False,
                            u=u, perm=np.arange(T))
    assert _rows(got) == {0, 1, 8, 9, 10, 11, 16, 17, 3, 6, 13, 18, 19, 20, 21}


def test_bernoulli_ignores_the_permutation():
    segs = [(10, 0, False), (8, 10, False), (4, 18, True)]
    T = 22
    u = np.full(T, 0.5)
    u[4] = 0.01
    a = O.build_protected(T, segs, 2, 0.10, 0.0, False, u, np.arange(T))
    b = O.build_protected(T, segs, 2, 0.10, 0.0, False, u, np.arange(T)[::-1].copy())
    assert _rows(a) == _rows(b) == {0, 1, 8, 9, 10, 11, 16, 17, 4, 18, 19, 20, 21}


# budget geometry: cached segments of 6 rows at 0 and 12 rows at 6, 3 new rows
# at 18; boundary 1 -> rows 0, 5, 6, 17; C = 18 cached rows
BUDGET_SEGS = [(6, 0, False), (12, 6, False), (3, 18, True)]
BUDGET_T = 21
# a permutation that starts with a new row, a boundary row, then a mix
BUDGET_PERM = np.array([20, 17, 3, 12, 0, 9, 4, 14, 2, 11, 7, 1, 8, 10, 13, 15, 16, 5,
                        6, 18, 19])


def test_budget_fill_in_permutation_order():
    # 50 %: target = ceil(50 * 18 / 100) = 9; 4 boundary rows, then 5 fill rows
    # taken from the permutation, skipping new (20) and boundary (17, 0) rows:
    # 3, 12, 9, 4, 14
    got = O.build_protected(BUDGET_T, BUDGET_SEGS, 1, 0.0, 0.50, False,
                            np.zeros(BUDGET_T), BUDGET_PERM)
    assert _rows(got) == {0, 5, 6, 17} | {3, 12, 9, 4, 14} | {18, 19, 20}


def test_budget_target_rounds_up():
    # 25 %: target = ceil(25 * 18 / 100) = ceil(4.5) = 5: one fill row (3)
    got = O.build_protected(BUDGET_T, BUDGET_SEGS, 1, 0.0, 0.25, False,
                            np.zeros(BUDGET_T), BUDGET_PERM)
    assert _rows(got) == {0, 5, 6, 17, 3, 18, 19, 20}


def test_budget_reversed_permutation_picks_other_rows():
    # the same rule walked over the reversed permutation: 19, 18 (new), 6, 5
    # (boundary), then 16, 15, 13, 10, 8
    got = O.build_protected(BUDGET_T, BUDGET_SEGS, 1, 0.0, 0.50, False,
                            np.zeros(BUDGET_T), BUDGET_PERM[::-1].copy())
    assert _rows(got) == {0, 5, 6, 17} | {16, 15, 13, 10, 8} | {18, 19, 20}


def test_budget_boundary_alone_exceeds_target():
    # cached 4 rows at 0 and 10 rows at 4, new rows 14, 15; boundary 2:
    # the 4-row segment is all boundary (0..3), the other gives 4, 5, 12, 13:
    # 8 boundary rows against a target of ceil(25 * 14 / 100) = 4.  All 8 are
    # kept and nothing else, although the permutation lists 6..11 first.
    segs = [(4, 0, False), (10, 4, False), (2, 14, True)]
    T = 16
    perm = np.array([6, 7, 8, 9, 10, 11, 0, 1, 2, 3, 4, 5, 12, 13, 14, 15])
    got = O.build_protected(T, segs, 2, 0.0, 0.25, False, np.zeros(T), perm)
    assert _rows(got) == {0, 1, 2, 3, 4, 5, 12, 13, 14, 15}


def test_budget_full_share_protects_every_row():
    got = O.build_protected(BUDGET_T, BUDGET_SEGS, 1, 0.0, 1.0, False,
                            np.zeros(BUDGET_T), BUDGET_PERM)
    assert got.all()


def test_dirty_rows_outside_the_budget():
    # dirty rows 7 and 10 join on top of the 50 % fill of the test above; the
    # fill still takes 3, 12, 9, 4, 14 (dirty rows do not use up the budget);
    # dirty row 3 (which the fill takes anyway) and dirty new row 19 add nothing
    dirty = np.zeros(BUDGET_T, bool)
    dirty[[7, 10, 3, 19]] = True
    got = O.build_protected(BUDGET_T, BUDGET_SEGS, 1, 0.0, 0.50, False,
                            np.zeros(BUDGET_T), BUDGET_PERM, dirty=dirty)
    assert _rows(got) == {0, 5, 6, 17} | {3, 12, 9, 4, 14} | {7, 10} | {18, 19, 20}


def test_dirty_rows_with_the_bernoulli_rule():
    segs = [(10, 0, False), (8, 10, False), (4, 18, True)]
    T = 22
    u = np.full(T, 0.5)
    u[13] = 0.0
    dirty = np.zeros(T, bool)
    dirty[[5, 14]] = True
    got = O.build_protected(T, segs, 2, 0.3, 0.0, False, u, np.arange(T), dirty=dirty)
    assert _rows(got) == {0, 1, 8, 9, 10, 11, 16, 17, 13, 5, 14, 18, 19, 20, 21}


def test_no_rule_keeps_only_new_and_dirty_rows():
    segs = [(10, 0, False), (8, 10, False), (4, 18, True)]
    T = 22
    dirty = np.zeros(T, bool)
    dirty[2] = True
    got = O.build_protected(T, segs, 2, 0.3, 0.0, True, np.zeros(T), np.arange(T), dirty=dirty)
    assert _rows(got) == {2, 18, 19, 20, 21}


def test_boundary_only_rule_on_short_segment():
    # boundary 3 on a 4-row segment covers it whole: [0, 3) u [1, 4)
    segs = [(4, 0, False), (9, 4, False), (1, 13, True)]
    got = O.build_protected(14, segs, 3, 0.0, 0.0, False, np.zeros(14), np.arange(14))
    assert _rows(got) == {0, 1, 2, 3, 4, 5, 6, 10, 11, 12, 13}


def test_bitmap_words_hand_values():
    prot = np.zeros(40, bool)
    prot[[0, 3, 31, 32, 39]] = True
    w = O.bitmap_words(prot)
    assert w.tolist() == [(1 << 0) | (1 << 3) | (1 << 31), (1 << 0) | (1 << 7)]
