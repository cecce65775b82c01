"""Pins of the oracle's SpecCache span completion, global budget control and
cross-tokenizer alignment (SpecCache notes, "2.3 Semantic span completion" and
"2.4 Cross-tokenizer alignment") against values and properties fixed by the pages
and by arithmetic, independent of the oracle's own code."""
import json
import os

import numpy as np
import pytest

from oracle import blend_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "span_completion.json")


def test_hand_worked_case():
    g = json.load(open(GOLDEN))
    s = np.array(g["scores"], dtype=np.float32)
    assert [list(p) for p in O.span_segments(s, g["tau_smooth"], g["max_span"])] == g["spans"]
    for c in g["cases"]:
        got = sorted(O.span_complete(s, c["k"], g["tau_smooth"], c["tau_cover_bp"], g["max_span"]))
        assert got == c["set"], c


def test_descending_ramp_closed_form():
    """scores 2.0 - 0.01 i (i < 40): normalised (39 - i) / 39, so delta_i = 1 / (39 - i),
    below 0.4 exactly for i <= 36.  Greedy spans of at most 16: [0,15], [16,31], [32,37],
    then [38] and [39] (delta_37 = 0.5 and delta_38 = 1 end their spans)."""
    s = (2.0 - 0.01 * np.arange(40)).astype(np.float32)
    assert O.span_segments(s, 0.4, 16) == [(0, 15), (16, 31), (32, 37), (38, 38), (39, 39)]
    # max_span 8 cuts the long run every 8 tokens
    assert O.span_segments(s, 0.4, 8)[:5] == [(0, 7), (8, 15), (16, 23), (24, 31), (32, 37)]


def test_minimum_token_ends_its_span_and_equal_scores_never_merge():
    s = np.array([0.5, 0.5, 0.5], dtype=np.float32)
    assert O.span_segments(s, 0.4, 16) == [(0, 0), (1, 1), (2, 2)]
    # normalised [1, 0, 0.025, 0.05]: delta_0 = 1, delta_1 = 0.025 / 0 (infinite),
    # delta_2 = 1 -> every token is its own span
    s = np.array([3.0, 1.0, 1.05, 1.1], dtype=np.float32)
    assert O.span_segments(s, 0.4, 16) == [(0, 0), (1, 1), (2, 2), (3, 3)]


def _rand_scores(rng, n, kind):
    if kind == "walk":  # locally smooth: spans of several tokens form
        return (5.0 + np.cumsum(rng.normal(0, 0.05, n))).astype(np.float32)
    if kind == "phrases":
        out, i = [], 0
        while i < n:
            ln = int(rng.integers(1, 9))
            lvl = rng.lognormal(0, 0.6)
            out += list(lvl * (1 + rng.normal(0, 0.03, ln)))
            i += ln
        return np.array(out[:n], dtype=np.float32)
    return rng.random(n).astype(np.float32)


@pytest.mark.parametrize("kind", ["walk", "phrases", "iid"])
def test_completion_invariants(kind):
    rng = np.random.default_rng(3)
    for trial in range(20):
        n = int(rng.integers(1, 120))
        s = _rand_scores(rng, n, kind)
        k = int(rng.integers(0, n + 1))
        tc = int(rng.choice([3000, 5000, 7000, 10000]))
        init = set(O.topk(s, k))
        spans = O.span_segments(s, 0.4, 16)
        # spans partition 0..n-1 in order, each 1..16 long
        flat = [t for u, v in spans for t in range(u, v + 1)]
        assert flat == list(range(n)) and all(1 <= v - u + 1 <= 16 for u, v in spans)
        T = O.span_complete(s, k, 0.4, tc, 16)
        assert init <= T
        for u, v in spans:
            members = set(range(u, v + 1))
            c = len(members & init)
            if c * 10000 >= tc * len(members):
                assert members <= T
            else:
                assert (members & T) == (members & init)


def test_degenerate_thresholds_leave_topk():
    rng = np.random.default_rng(4)
    s = _rand_scores(rng, 200, "walk")
    init = set(O.topk(s, 40))
    assert O.span_complete(s, 40, 0.0, 7000, 16) == init       # nothing merges
    assert O.span_complete(s, 40, 0.4, 7000, 1) == init        # spans of one token
    assert O.span_complete(s, 40, 0.4, 10000, 16) == init      # only fully covered spans


def test_final_budget_is_maximal_and_cap_keeps_highest():
    rng = np.random.default_rng(5)
    for trial in range(10):
        n = int(rng.integers(20, 150))
        s = _rand_scores(rng, n, "walk")
        B = int(rng.integers(1, n))
        got = O.span_select(s, B, 0.4, 7000, 16, "final")
        assert len(got) <= B
        # brute force over every k: the result is the completed set of the largest k that fits
        best = max(k for k in range(0, B + 1) if len(O.span_complete(s, k, 0.4, 7000, 16)) <= B)
        assert list(got) == sorted(O.span_complete(s, best, 0.4, 7000, 16))
        cap = int(rng.integers(B, n + 1))
        cand = O.span_select(s, B, 0.4, 5000, 16, "candidate", cap=cap)
        full = O.span_complete(s, B, 0.4, 5000, 16)
        assert len(cand) == min(cap, len(full)) and set(cand) <= full
        dropped = full - set(cand)
        if dropped:  # every kept token outranks every dropped one
            worst_kept = max(O._order_key(s[t], t) for t in cand)
            assert all(O._order_key(s[t], t) > worst_kept for t in dropped)


def test_rank_cover_formulation_matches():
    """The form the GPU evaluates: per span the c-th smallest rank r_c with
    c = ceil(tau * |span|); cover(p) = min(rank p, r_c of p's span); the set at k is
    {p : cover(p) < k} for every k."""
    rng = np.random.default_rng(6)
    for trial in range(15):
        n = int(rng.integers(1, 200))
        s = _rand_scores(rng, n, ["walk", "phrases", "iid"][trial % 3])
        order = O.topk(s, n)
        rank = np.empty(n, dtype=np.int64)
        rank[order] = np.arange(n)
        tc = int(rng.choice([2500, 7000, 10000]))
        cover = rank.copy()
        for u, v in O.span_segments(s, 0.4, 16):
            ln = v - u + 1
            c = (tc * ln + 9999) // 10000
            rc = np.sort(rank[u:v + 1])[c - 1]
            cover[u:v + 1] = np.minimum(rank[u:v + 1], rc)
        for k in range(0, n + 1, max(1, n // 17)):
            assert set(np.nonzero(cover < k)[0]) == O.span_complete(s, k, 0.4, tc, 16)


def test_align_expand():
    sel = [0, 2, 3]
    ident = np.arange(6)
    assert list(O.align_expand(sel, ident, ident + 1)) == sel
    # every speculative token split into two target tokens
    st = np.arange(6) * 2
    assert list(O.align_expand(sel, st, st + 2)) == [0, 1, 4, 5, 6, 7]
    # two speculative tokens covering the same target token count it once
    a0, a1 = np.array([0, 1, 1, 3]), np.array([1, 2, 3, 4])
    assert list(O.align_expand([1, 2], a0, a1)) == [1, 2]
    assert list(O.align_expand([], a0, a1)) == []


def test_final_bisection_matches_linear_scan():
    rng = np.random.default_rng(7)
    for trial in range(12):
        n = int(rng.integers(1, 160))
        s = _rand_scores(rng, n, ["walk", "phrases", "iid"][trial % 3])
        B = int(rng.integers(0, n + 1))
        assert list(O.span_select_final_bisect(s, B, 0.4, 7000, 16, base=5)) == \
            list(O.span_select(s, B, 0.4, 7000, 16, "final", base=5))
