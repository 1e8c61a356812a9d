"""Pins of the oracle's n-gram fill of the candidate tree (AdaSpark sec. 2.2:
chains branch from the anchor and from each pick and may run past the block;
sec. 3.3 "N-gram candidates": read on along an earlier passage of the
request's text, else the most frequent follower of the last three tokens;
the parameter table: three-token follower context, 32 tokens below the
anchor).

Hand-worked texts fix each branch of the step rule (passage, longest match,
recency ties, the follower fallback and its ties, the pick's context, the
depth limit, nothing proposed).  On seeded texts with repeats, every token is
checked against what its evidence claims: a passage token continues an
earlier copy of the stated length, and a follower token has the stated count,
which no other follower of the same three tokens exceeds."""
import numpy as np
import pytest


def _fill(orc, x, picks=(), n_min=1, Lg=8, max_depth=32, copy_cap=256):
    x = np.asarray(x, np.int32)[None]
    ct = np.asarray(picks, np.int32).reshape(1, len(picks), 1) if len(picks) else np.zeros((1, 0, 1), np.int32)
    return orc.ngram_fill(x, [x.shape[1]], ct, n_min, copy_cap, max_depth, Lg)


def _chain(f, c=0):
    n = int(f.len[0, c])
    return f.tok[0, c, :n].tolist(), f.ev[0, c, :n].tolist()


def test_chain_reads_along_an_earlier_passage(orc):
    # the suffix 1 2 3 occurred at positions 1..3: read 9 8 7 1 2 3 from there;
    # at the text's end the passage stops, and the lookup finds 1 2 3 again
    f = _fill(orc, [5, 1, 2, 3, 9, 8, 7, 1, 2, 3], n_min=2)
    assert _chain(f) == ([9, 8, 7, 1, 2, 3, 9, 8], [3, 4, 5, 6, 7, 8, 3, 4])
    assert f.status == 0


def test_the_passage_is_read_on_even_where_a_new_lookup_would_leave_it(orc):
    # with copies capped at two tokens, "3 4" matches at two places after the
    # first steps; a fresh lookup would take the more recent one (then 8), but
    # the chain keeps reading the passage it is on (then 9)
    f = _fill(orc, [1, 2, 3, 4, 9, 3, 4, 8, 1, 2], n_min=2, Lg=3, copy_cap=2)
    assert _chain(f) == ([3, 4, 9], [2, 2, 2])


def test_longest_match_wins_over_a_more_recent_one(orc):
    x = [1, 2, 3, 4, 50, 9, 2, 3, 4, 60, 9, 7, 1, 2, 3, 4]
    assert _chain(_fill(orc, x, n_min=2, Lg=3)) == ([50, 9, 2], [4, 5, 6])


def test_equal_matches_go_to_the_most_recent(orc):
    x = [7, 2, 3, 4, 50, 8, 2, 3, 4, 60, 9, 2, 3, 4]
    assert _chain(_fill(orc, x, n_min=2, Lg=2)) == ([60, 9], [3, 4])


def test_follower_fallback_takes_the_most_frequent(orc):
    # no earlier 4-token match: the followers of 1 2 3 are 10 (twice) and 11;
    # then 1 2 3 10 matches at two places (the most recent wins) and is read on
    x = [1, 2, 3, 10, 5, 1, 2, 3, 11, 6, 1, 2, 3, 10, 7, 9, 1, 2, 3]
    assert _chain(_fill(orc, x, n_min=4, Lg=4)) == ([10, 7, 9, 1], [-2, 4, 5, 6])


def test_follower_ties_go_to_the_most_recent(orc):
    x = [1, 2, 3, 10, 5, 1, 2, 3, 11, 6, 9, 1, 2, 3]
    assert _chain(_fill(orc, x, n_min=4, Lg=1)) == ([11], [-1])


def test_chain_from_a_pick_continues_the_pick(orc):
    # the drafter picks 8 after the anchor 7: "7 8" occurred before, followed by 20 21 5
    f = _fill(orc, [7, 8, 20, 21, 5, 9, 7], picks=[8], n_min=1, Lg=3)
    assert _chain(f, 0)[0] == [8, 20, 21]
    assert _chain(f, 1)[0] == [20, 21, 5]


def test_depth_limit_counts_from_the_anchor(orc):
    f = _fill(orc, [1, 2, 3, 4] * 5, picks=[1, 2], n_min=1, Lg=8, max_depth=3)
    assert [_chain(f, c)[0] for c in range(3)] == [[1, 2, 3], [2, 3], [3]]


def test_nothing_proposed_stops_the_chain(orc):
    f = _fill(orc, [1, 2, 3], picks=[4], n_min=1)
    assert f.len.tolist() == [[0, 0]]
    assert np.all(f.tok == -1)
    f = orc.ngram_fill(np.zeros((1, 4), np.int32), [0], np.zeros((1, 1, 1), np.int32), 1, 256, 32, 4)
    assert f.len.tolist() == [[0, 0]]


def _text(rng, T, V=12, repeats=0.5):
    """a small-alphabet text with planted repeats"""
    x = list(rng.integers(0, V, 16))
    while len(x) < T:
        if rng.random() < repeats and len(x) > 8:
            a = int(rng.integers(0, len(x) - 4))
            x += x[a:a + int(rng.integers(3, 9))]
        else:
            x.append(int(rng.integers(0, V)))
    return np.array(x[:T], np.int32)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("n_min,V,repeats", [(1, 12, 0.5), (4, 12, 0.5), (4, 5, 0.0)])
def test_every_token_is_backed_by_its_evidence(orc, seed, n_min, V, repeats):
    # the plain 5-letter text makes most 4-token contexts new and most
    # 3-token ones old: the follower branch
    rng = np.random.default_rng(seed)
    T, P = 120, 3
    x = _text(rng, T, V, repeats)
    picks = rng.integers(0, V, P)
    f = orc.ngram_fill(x[None], [T], picks.reshape(1, P, 1), n_min, 256, 32, 32)
    for c in range(P + 1):
        n = int(f.len[0, c])
        assert n <= 32 - c
        ctx = list(x) + list(picks[:c])
        for k in range(n):
            y, e = int(f.tok[0, c, k]), int(f.ev[0, c, k])
            if e > 0:  # continues an earlier copy of length e
                assert e >= n_min
                assert any(x[j + 1] == y and list(x[j - e + 1:j + 1]) == ctx[len(ctx) - e:]
                           for j in range(e - 1, T - 1)), (c, k)
            else:      # the most frequent follower of the last three tokens
                assert e < 0 and n_min > 3
                tri = ctx[-3:]
                cnt = {}
                for j in range(2, T - 1):
                    if list(x[j - 2:j + 1]) == tri:
                        cnt[int(x[j + 1])] = cnt.get(int(x[j + 1]), 0) + 1
                assert cnt.get(y) == -e and max(cnt.values()) == -e, (c, k)
            ctx.append(y)
