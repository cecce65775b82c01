"""EPIC's static selection in the oracle (SpecCache notes, background and Figure 1(c):
the first tokens of every chunk are recomputed, the rest reused)."""
import numpy as np

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import synth

from blendcase import f64, oracle_cfg


def test_positions_closed_form():
    # P = 5; chunks of 3, 10, 4 tokens start at blended positions 5, 8, 18
    assert O.epic_positions(5, [3, 10, 4], 4).tolist() == [5, 6, 7, 8, 9, 10, 11, 18, 19, 20, 21]
    assert O.epic_positions(5, [3, 10, 4], 0).tolist() == []
    assert O.epic_positions(0, [2, 2], 99).tolist() == [0, 1, 2, 3]


def test_all_tokens_equals_recomputing_every_chunk_row():
    """With m at least every chunk's length EPIC recomputes every chunk row: the same as a
    forced stage holding all of them."""
    sh = synth.ModelShape("epic-tiny", 2, 128, 4, 2, 64, 256, 97, 1e4, dtype="f32", init="fan_in")
    w = {k: f64(v) for k, v in synth.model_weights(sh, 0).items()}
    cfg = oracle_cfg(sh)
    rng = np.random.default_rng(0)
    P, lens, Q = 4, [9, 6], 3
    prefix = rng.integers(0, sh.vocab, P)
    chunks = [rng.integers(0, sh.vocab, n) for n in lens]
    query = rng.integers(0, sh.vocab, Q)
    ek, ev = zip(*[O.precompute_chunk(w, cfg, prefix, c) for c in chunks])
    a = O.blend_prefill(w, cfg, ek, ev, chunks, prefix, [1, 0], query, "epic", epic_m=50)
    allrows = np.arange(P, P + sum(lens))
    b = O.blend_prefill(w, cfg, ek, ev, chunks, prefix, [1, 0], query, "forced", forced=[(0, allrows)])
    assert np.array_equal(a["stages"][0][1], allrows)
    assert np.allclose(a["hidden"], b["hidden"], rtol=0, atol=0) and np.allclose(a["K"], b["K"], rtol=0, atol=0)


def test_focused_chunks_closed_form():
    """Cache-Craft 3.2.2 reading: a chunk is focused when its summed question attention is
    at least focus_bp of the total.  Masses 0.5, 0.3, 0.2 (of 1.0) over chunks of 2, 3, 1."""
    s = np.array([0.25, 0.25, 0.1, 0.1, 0.1, 0.2])
    assert O.focused_chunks(s, [2, 3, 1], 2500).tolist() == [True, True, False]
    assert O.focused_chunks(s, [2, 3, 1], 2000).tolist() == [True, True, True]
    assert O.focused_chunks(s, [2, 3, 1], 5001).tolist() == [False, False, False]
    assert O.focused_chunks(s, [2, 3, 1], 0).tolist() == [True, True, True]


def test_focus_filter_shrinks_the_set_at_the_detection_layer():
    sh = synth.ModelShape("focus-tiny", 3, 128, 4, 2, 64, 256, 97, 1e4, dtype="f32", init="fan_in")
    w = {k: f64(v) for k, v in synth.model_weights(sh, 1).items()}
    cfg = oracle_cfg(sh)
    rng = np.random.default_rng(1)
    P, lens, Q = 4, [12, 9, 10], 3
    prefix = rng.integers(0, sh.vocab, P)
    chunks = [rng.integers(0, sh.vocab, n) for n in lens]
    query = rng.integers(0, sh.vocab, Q)
    ek, ev = zip(*[O.precompute_chunk(w, cfg, prefix, c) for c in chunks])
    base = O.blend_prefill(w, cfg, ek, ev, chunks, prefix, [0, 1, 2], query, "epic", epic_m=5)
    same = O.blend_prefill(w, cfg, ek, ev, chunks, prefix, [0, 1, 2], query, "epic", epic_m=5, focus_layer=1,
                           focus_bp=0)
    assert np.array_equal(base["hidden"], same["hidden"]) and len(same["stages"]) == 1
    # a threshold no chunk reaches: every chunk row stops at layer 1, only the query continues
    none = O.blend_prefill(w, cfg, ek, ev, chunks, prefix, [0, 1, 2], query, "epic", epic_m=5, focus_layer=1,
                           focus_bp=10000)
    assert none["stages"][1][0] == 1 and len(none["stages"][1][1]) == 0
    # layer-0 K of the chunk rows is recomputed in both runs; the last layer's only in base
    assert np.array_equal(none["K"][0], base["K"][0]) and not np.allclose(none["K"][2], base["K"][2])
