"""Copy drafts (host only, no GPU): the guesses that tfl_copy_draft proposes
for hand-made token sequences, against the rule stated in include/tfl.h (the
longest recurring suffix of 1..3 tokens, its latest earlier occurrence, the
tokens that followed it, continued periodically)."""
import numpy as np
import pytest

from gqa_decoder_forward_gb300 import build, tfl


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    tfl.lib()


def draft(tokens, k):
    return list(tfl.tfl_copy_draft(tokens, k))


def test_nothing_recurs_gives_no_guess():
    assert draft([7], 5) == []
    assert draft([1, 2, 3, 4, 5], 5) == []
    assert draft([1, 2, 3, 1], 0) == []


def test_a_repeated_token_continues_the_repeat():
    assert draft([9, 4, 4], 6) == [4] * 6
    assert draft([5, 5, 5, 5, 5], 3) == [5, 5, 5]


def test_a_cycle_continues_periodically():
    # period 3: ... 1 2 3 1 2 -> 3 1 2 3 1
    assert draft([1, 2, 3, 1, 2, 3, 1, 2], 5) == [3, 1, 2, 3, 1]
    # period 2 with a long max_draft
    assert draft([8, 6, 7, 6, 7], 7) == [6, 7, 6, 7, 6, 7, 6]


def test_latest_occurrence_wins_at_equal_length():
    # suffix [2, 3] occurs at 1 (then 9) and at 5 (then 8): the later one
    t = [1, 2, 3, 9, 5, 2, 3, 8, 6, 2, 3]
    assert draft(t, 3) == [8, 6, 2]
    # period 4 past the end: 8 6 2 3 | 8 6 ...
    assert draft(t, 6) == [8, 6, 2, 3, 8, 6]


def test_longer_suffix_wins_over_a_later_shorter_one():
    # [1, 2, 3] recurs from 0 (then 9); [2, 3] also at 5 (then 8), later but shorter
    t = [1, 2, 3, 9, 5, 2, 3, 8, 1, 2, 3]
    assert draft(t, 4) == [9, 5, 2, 3]
    # a 4-token suffix match is not looked for: only 1..3 tokens
    t2 = [4, 1, 2, 3, 7, 0, 1, 2, 3, 5, 4, 1, 2, 3]
    assert draft(t2, 2) == [5, 4]          # [1, 2, 3] latest at 6 -> 5 4 (not 7 0 from the 4-gram at 0)


def test_guess_is_a_continuation_that_keeps_the_match():
    """On random sequences over a small alphabet: whenever guesses are made, the
    suffix recurs P tokens earlier, and the extended sequence keeps period P."""
    rng = np.random.default_rng(5)
    for _ in range(300):
        n = int(rng.integers(1, 40))
        t = [int(x) for x in rng.integers(0, 4, n)]
        g = draft(t, 6)
        if not g:
            assert all(t[n - 1] != t[j] for j in range(n - 1))   # not even one token recurs
            continue
        assert len(g) == 6
        ext = t + g
        # the period: distance from the latest earlier occurrence of the matched suffix
        ok = False
        for m in range(min(3, n - 1), 0, -1):
            occ = [j for j in range(n - m) if t[j:j + m] == t[n - m:]]
            if occ:
                P = n - m - occ[-1]
                ok = all(ext[n + i] == ext[n + i - P] for i in range(6))
                break
        assert ok, (t, g)


def test_bad_arguments_are_refused():
    with pytest.raises(tfl.TflError):
        tfl.tfl_copy_draft([], 3)
    with pytest.raises(tfl.TflError):
        tfl.tfl_copy_draft([1, 2], -1)
