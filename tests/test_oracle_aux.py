"""Pins of the oracle's auxiliary-model attention scoring (CacheClip blog "6.2
Auxiliary-model-guided token selection": the column mean over the query rows of the
last-layer attention; CacheClip paper 4.2) against closed forms and against full prefill."""
import math

import numpy as np

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import synth

from blendcase import f64, oracle_cfg


def test_probs_uniform_for_zero_query_and_causal_zeros():
    rng = np.random.default_rng(0)
    K = rng.normal(size=(7, 2, 8))
    q = np.zeros((3, 4, 8))
    P = O.attention_probs(q, np.array([0, 3, 6]), K)
    for i, p in enumerate([0, 3, 6]):
        assert np.allclose(P[i, :, :p + 1], 1.0 / (p + 1)) and np.all(P[i, :, p + 1:] == 0)


def test_probs_two_keys_logistic_and_gqa_heads():
    d = 4
    K = np.zeros((2, 2, d))
    K[0, 0, 0], K[1, 0, 0] = 1.0, -1.0     # kv head 0
    K[0, 1, 1], K[1, 1, 1] = 2.0, 0.0      # kv head 1
    q = np.zeros((1, 4, d))
    q[0, :, 0] = 3.0                       # heads 0, 1 read kv head 0; heads 2, 3 kv head 1
    q[0, :, 1] = 0.5
    P = O.attention_probs(q, np.array([1]), K)
    a = (3.0 * 1.0 - 3.0 * -1.0) / math.sqrt(d)       # logit gap on kv head 0
    b = (0.5 * 2.0 - 0.0) / math.sqrt(d)               # logit gap on kv head 1
    assert np.isclose(P[0, 0, 0], 1 / (1 + math.exp(-a))) and np.isclose(P[0, 1, 0], P[0, 0, 0])
    assert np.isclose(P[0, 2, 0], 1 / (1 + math.exp(-b))) and np.isclose(P[0, 3, 0], P[0, 2, 0])
    assert np.allclose(P.sum(axis=2), 1.0)


def _tiny(seed=0, L=2):
    sh = synth.ModelShape("aux-tiny", L, 128, 4, 2, 64, 256, 97, 1e4, dtype="f32", init="fan_in")
    w = {k: f64(v) for k, v in synth.model_weights(sh, seed).items()}
    return sh, w


def test_zero_last_query_projection_gives_closed_form_means():
    """With the last layer's query projection zero every query row attends uniformly:
    row i (position P+L_c+i) gives each of its P+L_c+i+1 keys the weight 1/(P+L_c+i+1), so
    every chunk column scores mean_i 1/(P+L_c+i+1)."""
    sh, w = _tiny()
    w["wq"][sh.n_layers - 1][:] = 0.0
    cfg = oracle_cfg(sh)
    rng = np.random.default_rng(1)
    P, lens, Q = 5, [9, 4], 3
    prefix = rng.integers(0, sh.vocab, P)
    chunks = [rng.integers(0, sh.vocab, n) for n in lens]
    query = rng.integers(0, sh.vocab, Q)
    ek, ev = zip(*[O.precompute_chunk(w, cfg, prefix, c) for c in chunks])
    s = O.aux_attention_scores(w, cfg, ek, ev, chunks, prefix, [1, 0], query)
    want = []
    for c in [1, 0]:
        Lc = lens[c]
        want += [np.mean([1.0 / (P + Lc + i + 1) for i in range(Q)])] * Lc
    assert np.allclose(s, want, rtol=1e-12)


def test_query_forward_equals_full_prefill_of_the_sequence():
    """The chunk side comes from the exact precompute of [prefix + chunk], so the query rows
    computed on top of it are the full prefill of [prefix + chunk + query]: the last layer's
    keys of every row agree."""
    sh, w = _tiny(2, L=3)
    cfg = oracle_cfg(sh)
    rng = np.random.default_rng(2)
    P, Lc, Q = 4, 11, 5
    prefix, chunk, query = (rng.integers(0, sh.vocab, n) for n in (P, Lc, Q))
    ek, ev = O.precompute_chunk(w, cfg, prefix, chunk)
    q, K = O.aux_query_forward(w, cfg, ek, ev, P, query)
    _, Kf, _ = O.full_prefill(w, cfg, np.concatenate([prefix, chunk, query]))
    assert np.allclose(K, Kf[sh.n_layers - 1], rtol=1e-10, atol=1e-12)
    assert q.shape == (Q, sh.n_q_heads, sh.head_dim)


def test_scores_are_a_share_of_each_row():
    """Each query row's weights over all keys sum to one, so the chunk columns' scores of one
    chunk sum to at most one, and a permutation of the chunks permutes the score blocks."""
    sh, w = _tiny(3)
    cfg = oracle_cfg(sh)
    rng = np.random.default_rng(3)
    P, lens, Q = 3, [6, 8, 5], 4
    prefix = rng.integers(0, sh.vocab, P)
    chunks = [rng.integers(0, sh.vocab, n) for n in lens]
    query = rng.integers(0, sh.vocab, Q)
    ek, ev = zip(*[O.precompute_chunk(w, cfg, prefix, c) for c in chunks])
    a = O.aux_attention_scores(w, cfg, ek, ev, chunks, prefix, [0, 1, 2], query)
    b = O.aux_attention_scores(w, cfg, ek, ev, chunks, prefix, [2, 0, 1], query)
    blocks = np.split(a, np.cumsum(lens)[:-1])
    assert np.allclose(b, np.concatenate([blocks[2], blocks[0], blocks[1]]))
    for blk in blocks:
        assert 0.0 < blk.sum() < 1.0 and np.all(blk > 0)


def test_column_means_closed_forms():
    """Direct pins of the column mean: a zero query attends uniformly over the keys at or
    before its position, so every column below the smallest query position has the mean of
    1 / (pos + 1) over the rows; and when the columns cover every key any row sees, the
    means add up to one (each row's weights do)."""
    rng = np.random.default_rng(3)
    K = rng.normal(size=(20, 2, 8))
    qpos = np.array([9, 14, 19])
    zero = O.column_mean_scores(np.zeros((3, 4, 8)), qpos, K, 0, 10)
    assert np.allclose(zero, np.mean(1.0 / (qpos + 1)))
    q = rng.normal(size=(3, 4, 8))
    full = O.column_mean_scores(q, qpos, K, 0, 20)
    assert np.isclose(full.sum(), 1.0) and np.all(full >= 0)
    # columns past every query position get no weight
    assert np.all(O.column_mean_scores(q, np.array([3, 4, 5]), K, 6, 20) == 0)
