"""Pins of the oracle's n-gram lookup (Hybrid Spark sec. 4.1, sec. 4.2 features,
sec. 5.1, where the longest match is the one used): hand-built histories whose match is known by
construction, and an independent restatement by substring search on tiny inputs."""
import numpy as np
import pytest


def _one(orc, x, n_min=5, n_max=15, L=15, cap=256, stride=None):
    x = np.asarray(x, np.int32)
    stride = stride or max(len(x), 1)
    h = np.zeros((1, stride), np.int32)
    h[0, :len(x)] = x
    out = orc.ngram_propose(h, np.array([len(x)], np.int32), n_min, n_max, L, cap)
    return (out.g[0, :out.g_len[0]].tolist(), int(out.match_n[0]), int(out.agree[0]),
            int(out.copy_len[0]), out.status)


def test_exact_copy_gives_its_continuation(orc):
    prog = list(range(100, 160))  # 60 distinct tokens
    x = prog + prog[:40]  # the output is copying the program, 40 tokens in
    g, n, a, m, st = _one(orc, x)
    assert st == 0
    assert g == prog[40:55]  # the next 15 program tokens
    assert n == 15 and m == 40 and a == 1  # no runner-up => agreement


def test_no_repeat_gives_no_proposal(orc):
    g, n, a, m, st = _one(orc, list(range(200)))
    assert g == [] and n == a == m == 0 and st == 0


def test_runner_up_with_different_follower_disagrees(orc):
    ctx = [1, 2, 3, 4, 5, 6]
    x = [90] + ctx + [7] + [91, 92] + ctx + [8] + [93, 94] + ctx
    g, n, a, m, st = _one(orc, x)
    assert n == 6 and m == 6
    assert g[0] == 8  # the most recent occurrence wins the tie
    assert a == 0  # the runner-up continues with 7


def test_runner_up_with_same_follower_agrees(orc):
    ctx = [1, 2, 3, 4, 5, 6]
    x = [90] + ctx + [7, 50] + [91, 92] + ctx + [7, 51] + [93, 94] + ctx
    g, n, a, m, st = _one(orc, x)
    assert g[:2] == [7, 51] and a == 1


def test_longer_match_beats_more_recent_shorter_one(orc):
    long_ctx = [11, 12, 13, 14, 15, 16, 17, 18, 19, 20]
    x = [1] + long_ctx + [70, 71] + [2, 3] + long_ctx[-6:] + [80, 81] + [4] + long_ctx
    g, n, a, m, st = _one(orc, x)
    assert m == 10 and g[:2] == [70, 71]
    assert a == 0  # the shorter runner-up continues with 80


def test_match_length_capped_at_n_max_and_copy_length_at_cap(orc):
    prog = list(range(1000, 1400))
    x = prog + prog[:300]
    g, n, a, m, st = _one(orc, x, n_max=15, cap=256)
    assert n == 15 and m == 256 and g == prog[300:315]


def test_periodic_text_continues_the_period(orc):
    period = [5, 9, 2, 7]
    x = period * 20 + period[:3]
    g, n, a, m, st = _one(orc, x, n_min=2, n_max=15, cap=256)
    T = len(x)
    # every occurrence of the suffix is followed by the same token: agreement
    assert a == 1
    assert g == (period * 10)[3:3 + 15][:len(g)]
    assert m == min(256, T - 4)  # the most recent full repeat reaches back to the start


def test_short_history_and_bad_length(orc):
    assert _one(orc, [])[0] == []
    assert _one(orc, [3])[0] == []
    assert _one(orc, [3, 3], n_min=1, n_max=3)[0] == [3]  # j=0 matches, continuation x[1]
    h = np.zeros((1, 8), np.int32)
    out = orc.ngram_propose(h, np.array([9], np.int32), 1, 3, 15, 256)
    assert out.status & orc.ST_BAD_LENGTH and out.g_len[0] == 0


def test_proposal_may_run_into_the_suffix(orc):
    x = [4, 4, 4, 4, 4, 4]
    g, n, a, m, st = _one(orc, x, n_min=1, n_max=3, L=15)
    assert g == [4]  # j = T-2 is the most recent longest match: one token to copy
    assert m == 5


def _search_reference(x, n_min, n_max, L, cap):
    """Independent restatement by substring search: for each length from the longest
    down, the most recent occurrence (rfind) of the suffix that ends at or before
    position T-2 gives the best match; runner-up = the best other end position."""
    T = len(x)
    s = bytes(x)
    if T < 2:
        return [], 0, 0, 0
    best = None
    for l in range(min(cap, T - 1), n_min - 1, -1):
        pos = s.rfind(s[T - l:], 0, T - 1)
        if pos >= 0:
            best = (l, pos + l - 1)
            break
    if best is None:
        return [], 0, 0, 0
    lb, jb = best
    second = None
    for l in range(lb, n_min - 1, -1):
        ends = []
        start = 0
        while True:
            pos = s.find(s[T - l:], start, T - 1)
            if pos < 0:
                break
            ends.append(pos + l - 1)
            start = pos + 1
        ends = [j for j in ends if j != jb]
        if ends:
            second = max(ends)
            break
    g = list(x[jb + 1:jb + 1 + min(L, T - 1 - jb)])
    a = 1 if second is None or x[second + 1] == x[jb + 1] else 0
    return g, min(lb, n_max), a, lb


@pytest.mark.parametrize("cap", [256, 4])
def test_matches_substring_search_on_small_alphabets(orc, cap):
    rng = np.random.default_rng(5)
    for trial in range(400):
        T = int(rng.integers(0, 64))
        x = rng.integers(0, 3, T).astype(np.int32).tolist()
        n_min = int(rng.integers(1, 4))
        n_max = int(rng.integers(n_min, n_min + 3))
        cap_ = max(cap, n_max)
        g, n, a, m, st = _one(orc, x, n_min, n_max, 6, cap_, stride=64)
        assert (g, n, a, m) == _search_reference(x, n_min, n_max, 6, cap_), (x, n_min, n_max)
