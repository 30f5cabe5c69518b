"""n-gram drafting of speculative decoding (kimi-k3-in-c k3_run.c,
``spec_draft``): the oracle on worked cases that the rule fixes, and the
library's k2_spec_draft against the oracle on many sequences, without a GPU."""
import numpy as np
import pytest

from oracle import k2_spec as SP


@pytest.fixture(scope="module")
def k2():
    from dense_gqa_decoder_gb300 import build
    build.build()
    from dense_gqa_decoder_gb300 import k2 as mod
    return mod


def test_worked_cases_of_the_rule():
    # a 4-gram seen once: its continuation, up to the end of the sequence
    assert SP.spec_draft([1, 2, 3, 4, 9, 8, 1, 2, 3, 4]) == [9, 8, 1, 2, 3, 4]
    # capped
    assert SP.spec_draft([1, 2, 3, 4, 9, 8, 7, 6, 5, 4, 3, 2, 1, 2, 3, 4], cap=3) == [9, 8, 7]
    # no 4-gram repeat, but a 3-gram: [7, 8, 9] occurs earlier, followed by 5
    assert SP.spec_draft([7, 8, 9, 5, 6, 1, 7, 8, 9]) == [5, 6, 1, 7, 8, 9]
    # nothing repeats
    assert SP.spec_draft([1, 2, 3, 4, 5, 6]) == []
    assert SP.spec_draft([1, 2, 3]) == []
    # two occurrences that agree on two ids, then differ
    seq = [1, 2, 3, 4, 10, 11, 12, 0, 1, 2, 3, 4, 10, 11, 13, 0, 1, 2, 3, 4]
    assert SP.spec_draft(seq) == [10, 11]
    # the 4-gram twice with different continuations (21 vs 20): no 4-gram draft;
    # the 3-gram [2, 3, 4] likewise: no draft at all
    assert SP.spec_draft([1, 2, 3, 4, 20, 9, 1, 2, 3, 4, 21, 9, 1, 2, 3, 4]) == []
    # a 4-gram seen once elsewhere: its continuation up to the end
    assert SP.spec_draft([5, 1, 2, 3, 20, 6, 1, 2, 3, 21, 6, 1, 2, 3]) == [21, 6, 1, 2, 3]
    # the older continuation may not run into the newer occurrence
    # (4-gram: newest at 4, older at 0, and 0 + 4 reaches 4 at once: nothing;
    # 3-gram [2, 3, 4]: newest at 5, older at 1: one agreeing id, then 1 + 3 + 1 reaches 5)
    assert SP.spec_draft([1, 2, 3, 4, 1, 2, 3, 4, 1, 2, 3, 4]) == [1]


def test_the_library_drafts_like_the_oracle(k2):
    rng = np.random.default_rng(12)
    for case in range(400):
        vocab = int(rng.integers(2, 9))
        T = int(rng.integers(0, 60))
        seq = rng.integers(0, vocab, size=T).tolist()
        cap = int(rng.integers(1, 10))
        assert k2.spec_draft(seq, cap) == SP.spec_draft(seq, cap), (seq, cap)
    assert k2.spec_draft([], 8) == []


def test_the_library_drafts_like_the_oracle_on_structured_sequences(k2):
    # repeated units with sparse edits (long matches, overlapping and
    # periodic occurrences, disagreeing continuations), up to 3000 ids
    rng = np.random.default_rng(13)
    for case in range(300):
        unit = rng.integers(0, int(rng.integers(2, 40)), size=int(rng.integers(1, 24))).tolist()
        T = int(rng.integers(4, 3000 if case % 10 == 0 else 200))
        seq = (unit * (T // len(unit) + 1))[:T]
        for _ in range(int(rng.integers(0, 6))):
            seq[int(rng.integers(0, T))] = int(rng.integers(0, 50))
        cap = int(rng.integers(1, 10))
        assert k2.spec_draft(seq, cap) == SP.spec_draft(seq, cap), (case, cap)
