"""The comparison rules themselves, on the CPU: the oracle's own answers pass
and answers with a planted mistake (in a copy of the oracle's output) fail."""

import numpy as np
import pytest

import oracle
import parity
import workloads


@pytest.fixture(scope="module")
def case():
    X, C = workloads.blobs(200, 150, 32, seed=11)
    k = 6
    idx, s = oracle.topk(X, C, k)
    return X, C, k, idx, s


def test_topk_oracle_answers_pass(case):
    X, C, k, idx, s = case
    rep = parity.compare_topk(X, C, idx, s.astype(np.float32), k)
    assert rep.ok() and rep.idx_mismatches == 0, rep
    d = oracle.sqdist(X, C, np.repeat(np.arange(200), k), idx.ravel()).reshape(-1, k)
    rep = parity.compare_topk(X, C, idx, d.astype(np.float32), k, distances=True)
    assert rep.ok(), rep


def test_topk_integer_answers_pass_exactly():
    X, C = workloads.integers(100, 40, 16, seed=2)
    idx, s = oracle.topk(X, C, 5)
    rep = parity.compare_topk(X, C, idx, s, 5, integer=True)
    assert rep.ok() and rep.idx_mismatches == 0, rep


@pytest.mark.parametrize("mistake", ["swap", "wrong_index", "duplicate", "out_of_range",
                                     "skip_second", "score_off", "unsorted_scores"])
def test_topk_planted_mistakes_fail(case, mistake):
    X, C, k, idx, s = case
    idx = idx.copy()
    s = s.astype(np.float32).copy()
    r = 17
    if mistake == "swap":                     # two picks in the wrong order
        idx[r, [0, k - 1]] = idx[r, [k - 1, 0]]
        s[r, [0, k - 1]] = s[r, [k - 1, 0]]
    elif mistake == "wrong_index":            # a far centroid in place of the 3rd nearest
        far = int(np.argmax(oracle.scores(X, C, np.full(150, r), np.arange(150))))
        idx[r, 2] = far
    elif mistake == "duplicate":
        idx[r, 1] = idx[r, 0]
    elif mistake == "out_of_range":
        idx[r, 0] = 150
    elif mistake == "skip_second":            # shifted list: the 2nd nearest is missing
        idx[r, 1:-1] = idx[r, 2:]
        idx[r, -1] = int(np.argsort(oracle.scores(X, C, np.full(150, r), np.arange(150)))[k])
    elif mistake == "score_off":
        s[r, 3] += 0.5
    elif mistake == "unsorted_scores":
        s[r, 1], s[r, 2] = s[r, 2] + 1.0, s[r, 1]
    rep = parity.compare_topk(X, C, idx, s, k)
    assert not rep.ok(), (mistake, rep)
