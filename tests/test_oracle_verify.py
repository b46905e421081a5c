"""Pins of the oracle's LM-head argmax, acceptance and commit (CPU only).

"dflash-mlx" (dpshk.com) 单次前向验证 ⑤–⑧ and 保证二; worked cases are in
tests/golden/acceptance_worked_cases.txt with their citation.
"""
import itertools
import os

import numpy as np
import pytest

from oracle.dflash_oracle import (acceptance_length, lm_head_argmax, near_tie_mask,
                                  verify_accept)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "acceptance_worked_cases.txt")


def load_worked_cases():
    cases = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, blk, post, a, commit, nxt = [p.strip() for p in line.split("|")]
            cases.append((name, [int(t) for t in blk.split()], [int(t) for t in post.split()],
                          int(a), [int(t) for t in commit.split()], int(nxt)))
    return cases


def _planted_hidden(post, V=128, H=16, seed=0):
    """Hidden rows and a W_lm whose argmax at row i is post[i] (planted maxima)."""
    rng = np.random.default_rng(seed)
    T = len(post)
    h = rng.standard_normal((T, H))
    w = 0.01 * rng.standard_normal((V, H))
    for i, p in enumerate(post):
        w[p] += 3.0 * h[i] / np.linalg.norm(h[i]) ** 2 * 1.0
    return h, w


def test_worked_cases_from_the_pages():
    for name, blk, post, a, commit, nxt in load_worked_cases():
        assert acceptance_length(blk[1:], post[:15]) == a, name
        # drive the whole epilogue through planted logits
        h, w = _planted_hidden(post, V=128)
        r = verify_accept(h[None], w, np.array([blk]), np.array([3]), out_cap=40)
        assert list(r["posterior"][0]) == post, name
        assert r["accept"][0] == a, name
        assert list(r["out_tokens"][0, 3:3 + a + 1]) == commit, name
        assert r["commit_len"][0] == 3 + len(commit), name
        assert r["next_staged"][0] == nxt, name


def first_mismatch_definition(drafted, posterior):
    """Accepted prefix length: walk until the first disagreement (保证二 prose)."""
    n = 0
    while n < len(drafted) and drafted[n] == posterior[n]:
        n += 1
    return n


def test_acceptance_exhaustive_patterns():
    post = list(range(100, 115))
    for bits in itertools.product((0, 1), repeat=15):
        drafted = [p if m else p + 1 for p, m in zip(post, bits)]
        assert acceptance_length(drafted, post) == first_mismatch_definition(drafted, post)


def brute_argmax(h, w):
    V = len(w)
    out = []
    for row in h:
        logits = [sum(a * b for a, b in zip(row, w[v])) for v in range(V)]
        best, idx = logits[0], 0
        for v in range(1, V):
            if logits[v] > best:
                best, idx = logits[v], v
        srt = sorted(logits, reverse=True)
        out.append((idx, srt[0] - srt[1], srt[0]))
    return out


@pytest.mark.parametrize("chunk", [1, 3, 7, 50, 1000])
def test_lm_head_argmax_brute_force_and_chunking(chunk):
    rng = np.random.default_rng(1)
    h = rng.standard_normal((6, 12))
    w = rng.standard_normal((50, 12))
    w[17] = w[33]                              # duplicate row: tie in every position
    h[2] = w[17] * 5.0                         # row 2 maxima are the tie 17 / 33
    r = lm_head_argmax(h, w, chunk=chunk)
    for i, (idx, gap, mx) in enumerate(brute_argmax(h, w)):
        assert r["posterior"][i] == idx
        assert abs(r["gap"][i] - gap) < 1e-12
        assert abs(r["max"][i] - mx) < 1e-12
    assert r["posterior"][2] == 17 and r["gap"][2] == 0.0


def test_exact_ties_take_the_lowest_index():
    h = np.ones((3, 4))
    w = np.zeros((10, 4))
    w[[2, 5, 9]] = 1.0
    r = lm_head_argmax(h, w, chunk=4)
    assert list(r["posterior"]) == [2, 2, 2]
    assert list(r["gap"]) == [0.0, 0.0, 0.0]
    r = lm_head_argmax(np.zeros((2, 4)), w, chunk=3)      # all logits zero
    assert list(r["posterior"]) == [0, 0]


def test_planted_maxima():
    rng = np.random.default_rng(2)
    post = rng.integers(0, 300, size=16)
    h, w = _planted_hidden(post, V=300, H=24, seed=3)
    r = lm_head_argmax(h, w, chunk=64)
    assert list(r["posterior"]) == list(post)


def test_commit_position_and_overflow():
    post = list(range(20, 36))
    blk = [5] + post[:15]                       # all drafts match
    h, w = _planted_hidden(post, V=64)
    prev = np.full((2, 30), -7, dtype=np.int32)
    r = verify_accept(np.stack([h, h]), w, np.array([blk, blk]), np.array([4, 20]),
                      out_tokens=prev)
    assert list(r["accept"]) == [15, 15]
    assert list(r["out_tokens"][0, 4:20]) == blk and r["commit_len"][0] == 20
    assert np.all(r["out_tokens"][0, :4] == -7) and np.all(r["out_tokens"][0, 20:] == -7)
    # second sequence would need 20 + 16 > 30 slots: not committed, flagged
    assert r["overflow"][1] and np.all(r["out_tokens"][1] == -7) and r["commit_len"][1] == 20


def test_near_tie_mask():
    gap = np.array([0.0, 1e-4, 1e-2, 5e-3])
    mx = np.array([1.0, 1.0, 1.0, -5.0])
    assert list(near_tie_mask(gap, mx)) == [True, True, False, True]
