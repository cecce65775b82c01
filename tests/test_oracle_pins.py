"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own formulas: closed forms,
invariants the pages state, a hand-derived worked case of the grouping rule, and
brute force on tiny inputs.  No GPU is used.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import blend_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- tiny fp64 model

def tiny_cfg(n_layers=2):
    return dict(n_layers=n_layers, hidden=32, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn=48,
                vocab=64, rope_theta=1e4, rms_eps=1e-6)


def tiny_weights(cfg, seed=0):
    r = np.random.default_rng(seed)
    L, H, F = cfg["n_layers"], cfg["hidden"], cfg["ffn"]
    qd = cfg["n_q_heads"] * cfg["head_dim"]
    kvd = cfg["n_kv_heads"] * cfg["head_dim"]
    n = lambda *s: r.standard_normal(s) / math.sqrt(s[-1])
    return dict(embed=r.standard_normal((cfg["vocab"], H)), wq=n(L, qd, H), wk=n(L, kvd, H),
                wv=n(L, kvd, H), wo=n(L, H, qd), wg=n(L, F, H), wu=n(L, F, H), wd=n(L, H, F),
                attn_norm=np.ones((L, H)), mlp_norm=np.ones((L, H)), final_norm=np.ones(H))


def tiny_request(cfg, P=4, lens=(8, 8, 8), Q=4, seed=1):
    r = np.random.default_rng(seed)
    prefix = r.integers(0, cfg["vocab"], P)
    chunks = [r.integers(0, cfg["vocab"], lc) for lc in lens]
    query = r.integers(0, cfg["vocab"], Q)
    return prefix, chunks, query


def precompute_pool(w, cfg, prefix, chunks):
    ks, vs = [], []
    for c in chunks:
        k, v = O.precompute_chunk(w, cfg, prefix, c)
        ks.append(k)
        vs.append(v)
    return ks, vs


# ---------------------------------------------------------------- RoPE

def test_rope_basis_closed_form():
    d, theta = 8, 1e4
    for i in range(d // 2):
        e = np.zeros((1, 1, d))
        e[0, 0, i] = 1.0
        p = 37
        out = O.rope_rotate(e, np.array([p]), theta)[0, 0]
        a = p * theta ** (-2.0 * i / d)
        want = np.zeros(d)
        want[i] = math.cos(a)
        want[i + d // 2] = math.sin(a)
        np.testing.assert_allclose(out, want, atol=1e-15)


def test_rope_composition_and_identity():
    r = np.random.default_rng(0)
    x = r.standard_normal((5, 3, 16))
    p = np.array([0, 3, 100, 4095, 17])
    delta = np.array([0, 512, 7, 12000, 31])
    once = O.rope_rotate(x, p + delta, 1e6)
    twice = O.realign_keys(O.rope_rotate(x, p, 1e6), delta, 1e6)
    np.testing.assert_allclose(twice, once, atol=1e-12)
    np.testing.assert_array_equal(O.rope_rotate(x, np.zeros(5, int), 1e6), x)
    # rotation keeps the norm of each head vector
    np.testing.assert_allclose(np.linalg.norm(once, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_relative_position():
    """q.k after RoPE depends only on the distance between the two positions."""
    r = np.random.default_rng(1)
    q = r.standard_normal((1, 1, 16))
    k = r.standard_normal((1, 1, 16))
    dots = []
    for shift in (0, 5, 900):
        qr = O.rope_rotate(q, np.array([40 + shift]), 1e4)
        kr = O.rope_rotate(k, np.array([13 + shift]), 1e4)
        dots.append(float(np.sum(qr * kr)))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-11)


# ---------------------------------------------------------------- norm, activation

def test_rmsnorm_constant_vector():
    for c in (0.5, -3.0, 1e-4):
        x = np.full((2, 10), c)
        g = np.linspace(0.5, 2.0, 10)
        want = c / math.sqrt(c * c + 1e-6) * g
        np.testing.assert_allclose(O.rmsnorm(x, g, 1e-6)[1], want, rtol=1e-14)


def test_silu_closed_form():
    np.testing.assert_array_equal(O.silu(np.array([0.0])), [0.0])
    np.testing.assert_allclose(O.silu(np.array([1.0, -2.0, 40.0])),
                               [1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2)), 40.0], rtol=1e-14)


# ---------------------------------------------------------------- attention

def test_attention_single_key_returns_value():
    r = np.random.default_rng(2)
    q = r.standard_normal((1, 4, 8))
    K = r.standard_normal((6, 2, 8))
    V = r.standard_normal((6, 2, 8))
    out = O.attention(q, np.array([0]), K, V)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], V[0, h // 2], rtol=1e-14)


def test_attention_two_keys_closed_form():
    r = np.random.default_rng(3)
    d = 16
    q = r.standard_normal((1, 1, d))
    K = r.standard_normal((2, 1, d))
    V = r.standard_normal((2, 1, d))
    s0 = float(q[0, 0] @ K[0, 0]) / 4.0          # 1/sqrt(16)
    s1 = float(q[0, 0] @ K[1, 0]) / 4.0
    a1 = 1.0 / (1.0 + math.exp(s0 - s1))
    want = (1 - a1) * V[0, 0] + a1 * V[1, 0]
    np.testing.assert_allclose(O.attention(q, np.array([1]), K, V)[0, 0], want, rtol=1e-12)


def test_attention_gqa_equals_mha_with_repeated_kv():
    r = np.random.default_rng(4)
    q = r.standard_normal((3, 6, 8))
    K = r.standard_normal((9, 2, 8))
    V = r.standard_normal((9, 2, 8))
    pos = np.array([2, 5, 8])
    gqa = O.attention(q, pos, K, V)
    Kr = np.repeat(K, 3, axis=1)          # head h uses kv head h // 3
    Vr = np.repeat(V, 3, axis=1)
    np.testing.assert_allclose(gqa, O.attention(q, pos, Kr, Vr), rtol=1e-13)


def test_attention_is_causal():
    r = np.random.default_rng(5)
    q = r.standard_normal((2, 2, 8))
    K = r.standard_normal((10, 1, 8))
    V = r.standard_normal((10, 1, 8))
    pos = np.array([3, 6])
    a = O.attention(q, pos, K, V)
    K2, V2 = K.copy(), V.copy()
    K2[7:] = 1e3
    V2[7:] = -1e3
    np.testing.assert_array_equal(O.attention(q, pos, K2, V2), a)
    K2[4:] = 50.0
    assert not np.allclose(O.attention(q, pos, K2, V2)[1], a[1])


def test_attention_matches_row_by_row_brute_force():
    """Against the definition written out one row and one head at a time, with more
    rows than one block of the oracle's loop, positions in no particular order and a
    wide logit range (scaled queries)."""
    r = np.random.default_rng(12)
    n, hq, hkv, d, N = 300, 6, 2, 4, 320
    q = r.standard_normal((n, hq, d)) * 4.0
    K = r.standard_normal((N, hkv, d))
    V = r.standard_normal((N, hkv, d))
    pos = r.integers(0, N, n)
    got = O.attention(q, pos, K, V)
    for i in range(n):
        for h in range(hq):
            g = h // (hq // hkv)
            logits = [sum(q[i, h, c] * K[j, g, c] for c in range(d)) / math.sqrt(d) for j in range(pos[i] + 1)]
            m = max(logits)
            wts = [math.exp(x - m) for x in logits]
            tot = sum(wts)
            want = [sum(wts[j] * V[j, g, c] for j in range(pos[i] + 1)) / tot for c in range(d)]
            np.testing.assert_allclose(got[i, h], want, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- prefill, assembly

def test_full_prefill_is_causal():
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    toks = np.random.default_rng(6).integers(0, 64, 20)
    h, K, V = O.full_prefill(w, cfg, toks)
    h2, K2, V2 = O.full_prefill(w, cfg, toks[:13])
    np.testing.assert_allclose(K2, K[:, :13], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(V2, V[:, :13], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(h2, h[:13], rtol=1e-10, atol=1e-12)


def test_assemble_keeps_one_prefix_and_realigns():
    cfg = tiny_cfg()
    w = tiny_weights(cfg)
    prefix, chunks, query = tiny_request(cfg, lens=(8, 5, 8))
    ks, vs = precompute_pool(w, cfg, prefix, chunks)
    # every entry's prefix rows are identical (the prefix is encoded first each time)
    for c in range(1, 3):
        np.testing.assert_allclose(ks[c][:, :4], ks[0][:, :4], rtol=1e-12, atol=1e-14)
    order = [2, 0, 1]
    lens = [len(chunks[c]) for c in order]
    K, V = O.assemble(ks, vs, order, 4, lens, 4, cfg["rope_theta"])
    assert K.shape[1] == 4 + 21 + 4
    np.testing.assert_array_equal(K[:, :4], ks[2][:, :4])
    off = 0
    for c, lc in zip(order, lens):
        # rotate back by -off gives the cached rows; the value rows are copied unchanged
        back = np.stack([O.rope_rotate(K[layer, 4 + off:4 + off + lc], np.full(lc, -off), 1e4)
                         for layer in range(2)])
        np.testing.assert_allclose(back, ks[c][:, 4:4 + lc], atol=1e-12)
        np.testing.assert_array_equal(V[:, 4 + off:4 + off + lc], vs[c][:, 4:4 + lc])
        off += lc
    assert np.all(K[:, 4 + 21:] == 0)


def test_realigned_chunk_keys_equal_keys_encoded_at_the_new_position():
    """Realigning a chunk's cached keys equals encoding the same pre-RoPE keys at the
    new positions (the rotation composes); only cross-chunk attention is missing."""
    r = np.random.default_rng(7)
    raw = r.standard_normal((12, 2, 8))
    local = np.arange(4, 16)
    cached = O.rope_rotate(raw, local, 1e4)
    moved = O.realign_keys(cached, np.full(12, 100), 1e4)
    np.testing.assert_allclose(moved, O.rope_rotate(raw, local + 100, 1e4), atol=1e-12)


# ---------------------------------------------------------------- selection

def _scores_for(cands, n):
    s = np.zeros(n)
    s[list(cands)] = 1.0
    return s


def test_grouping_worked_cases():
    with open(os.path.join(GOLDEN, "fig6_grouping.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = O.group_windows(c["candidates"], c["n"], c["w"], c["tau"])
        assert sorted(got) == c["expected"], c
        # through select(): candidates as the top-k of scores
        s = _scores_for(c["candidates"], c["n"])
        sel = O.select(s, len(c["candidates"]), c["w"], c["tau"], "candidate")
        assert sel.tolist() == c["expected"]


def test_topk_tie_order_nan_and_signed_zero():
    s = np.array([1.0, 2.0, 1.0, np.nan, -0.0, 0.0, 2.0, -1.0])
    assert O.topk(s, 8) == [1, 6, 0, 2, 4, 5, 7, 3]
    assert O.topk(s, 3) == [1, 6, 0]
    assert O.topk(s, 0) == []


def _cover_rank_select(scores, budget, w, tau, mode):
    """Independent formulation: position p is in the grouped set of the top-k iff some
    window start t in (p-w, p] (t <= n-w) has qualify(t) < k, where qualify(t) is the
    larger of t's rank and the tau-th smallest rank inside [t, t+w)."""
    n = len(scores)
    order = sorted(range(n), key=lambda t: (-scores[t], t))
    rank = np.empty(n, int)
    rank[order] = np.arange(n)
    INF = 10 ** 9
    qual = np.full(n, INF)
    for t in range(n - w + 1):
        qual[t] = max(rank[t], sorted(rank[t:t + w])[tau - 1])
    cover = np.array([min([qual[t] for t in range(max(0, p - w + 1), p + 1)]) for p in range(n)])
    if mode == "candidate":
        k = min(budget, n)
    else:
        k = min(budget, n)
        srt = np.sort(cover)
        if n > budget:
            k = min(k, srt[budget])
    return sorted(np.nonzero(cover < k)[0].tolist())


@pytest.mark.parametrize("seed", range(40))
def test_select_matches_cover_rank_formulation(seed):
    r = np.random.default_rng(100 + seed)
    n = int(r.integers(1, 40))
    w = int(r.integers(1, 6))
    tau = int(r.integers(1, w + 1))
    budget = int(r.integers(0, n + 1))
    s = r.integers(0, 5, n).astype(float)        # many ties
    for mode in ("candidate", "final"):
        got = O.select(s, budget, w, tau, mode).tolist()
        assert got == _cover_rank_select(s, budget, w, tau, mode), (n, w, tau, budget, mode)
    np.testing.assert_array_equal(O.select_final_bisect(s, budget, w, tau),
                                  O.select(s, budget, w, tau, "final"))


def test_select_final_bruteforce_over_k():
    r = np.random.default_rng(9)
    for _ in range(30):
        n = int(r.integers(2, 30))
        s = r.standard_normal(n)
        w, tau = int(r.integers(1, 5)), 1
        budget = int(r.integers(0, n + 1))
        sizes = [len(O.group_windows(O.topk(s, k), n, w, tau)) for k in range(n + 1)]
        assert all(a <= b for a, b in zip(sizes, sizes[1:]))   # grows with k
        kstar = max([k for k in range(min(budget, n) + 1) if sizes[k] <= budget])
        want = sorted(O.group_windows(O.topk(s, kstar), n, w, tau))
        assert O.select(s, budget, w, tau, "final").tolist() == want


def test_select_final_monotone_in_budget():
    r = np.random.default_rng(10)
    s = r.standard_normal(300)
    prev = set()
    for b in range(0, 301, 15):
        cur = set(O.select_final_bisect(s, b, 4, 1).tolist())
        assert len(cur) <= b and prev <= cur
        prev = cur


def test_select_allowed_mask():
    r = np.random.default_rng(11)
    s = r.standard_normal(50)
    allowed = r.random(50) < 0.4
    got = O.select(s, 10, 3, 1, "final", allowed=allowed, base=7)
    assert len(got) <= 10 and all(allowed[t - 7] for t in got)


def test_importance_scores_closed_form():
    h = np.ones((3, 4, 16)) * np.array([1.0, 2.0, -3.0])[:, None, None]
    np.testing.assert_allclose(O.importance_scores(h), [4.0, 8.0, 12.0])
    h2 = np.zeros((1, 2, 4))
    h2[0, 0, 0] = 3.0
    h2[0, 1, :2] = [3.0, 4.0]
    np.testing.assert_allclose(O.importance_scores(h2), [(3.0 + 5.0) / 2])


# ---------------------------------------------------------------- blended prefill

@pytest.fixture(scope="module")
def tiny_setup():
    cfg = tiny_cfg(n_layers=4)
    w = tiny_weights(cfg, seed=3)
    prefix, chunks, query = tiny_request(cfg, P=4, lens=(8, 8, 8), Q=4, seed=2)
    ks, vs = precompute_pool(w, cfg, prefix, chunks)
    return cfg, w, prefix, chunks, query, ks, vs


def test_rho_100_equals_full_prefill(tiny_setup):
    cfg, w, prefix, chunks, query, ks, vs = tiny_setup
    order = [1, 2, 0]
    scores = np.random.default_rng(0).standard_normal(24)
    for wnd in (1, 4):
        out = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "ext", rho_bp=10000,
                              window=wnd, tau=1, scores=scores)
        assert out["stages"][0][1].tolist() == list(range(4, 28))
        h, K, V = O.full_prefill(w, cfg, out["tokens"])
        np.testing.assert_allclose(out["hidden"], h[-4:], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(out["K"], K, rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(out["V"], V, rtol=1e-9, atol=1e-11)


def test_rho_0_reuses_every_chunk_row(tiny_setup):
    cfg, w, prefix, chunks, query, ks, vs = tiny_setup
    order = [0, 2, 1]
    out = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "ext", rho_bp=0,
                          scores=np.zeros(24))
    K0, V0 = O.assemble(ks, vs, order, 4, [8, 8, 8], 4, cfg["rope_theta"])
    np.testing.assert_array_equal(out["K"][:, :28], K0[:, :28])
    np.testing.assert_array_equal(out["V"][:, :28], V0[:, :28])
    assert np.all(out["K"][:, 28:] != 0)


def test_first_layer_kv_needs_no_recompute(tiny_setup):
    """A token's first-layer K, V depend only on the token and its position, so after
    realignment the cached first-layer rows equal the fresh ones for every chunk."""
    cfg, w, prefix, chunks, query, ks, vs = tiny_setup
    order = [2, 0, 1]
    K, V = O.assemble(ks, vs, order, 4, [8, 8, 8], 4, cfg["rope_theta"])
    toks = np.concatenate([prefix] + [chunks[c] for c in order] + [query])
    rows = np.arange(4, 28)
    x = w["embed"][toks[rows]]
    _, dev = O.layer_kv(w, cfg, 0, x, rows, K[0].copy(), V[0].copy(), np.ones(24, bool))
    assert np.max(dev) < 1e-24


def test_hkvd_chunk0_has_zero_deviation_and_schedule(tiny_setup):
    cfg, w, prefix, chunks, query, ks, vs = tiny_setup
    order = [2, 0, 1]
    out = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "hkvd", rho_bp=2000,
                          r1_bp=4000, window=2, tau=1)
    dev1, dev2 = out["dev1"], out["dev2"]
    # chunk 0 sits right behind the prefix, exactly where it was encoded: same context,
    # same KV on every layer; later chunks miss their cross-chunk attention
    assert np.max(dev1[:8]) <= 1e-20 * np.max(dev1)
    assert np.min(dev1[8:]) > 1e-6
    c1 = out["stages"][1][1]
    s = out["stages"][2][1]
    assert out["stages"][1][0] == 1 and out["stages"][2][0] == 2
    assert len(c1) == O.ceil_bp(4000, 24)
    assert set(s.tolist()) <= set(c1.tolist()) and len(s) <= O.ceil_bp(2000, 24)
    # stage-1 set is the top of the layer-1 deviation; layer 2 checked only C1 rows
    assert set(c1.tolist()) == set((4 + np.argsort(-dev1, kind="stable")[:len(c1)]).tolist())
    assert set((4 + np.nonzero(dev2)[0]).tolist()) <= set(c1.tolist())
    # the rows outside C1 still got their fresh layer-1 KV, rows outside S keep the
    # realigned cache from layer 3 on
    K0, V0 = O.assemble(ks, vs, order, 4, [8, 8, 8], 4, cfg["rope_theta"])
    rest = sorted(set(range(4, 28)) - set(s.tolist()))
    if cfg["n_layers"] > 3:
        np.testing.assert_array_equal(out["K"][3:, rest], K0[3:, rest])


def test_forced_schedule_reproduces_hkvd(tiny_setup):
    cfg, w, prefix, chunks, query, ks, vs = tiny_setup
    order = [1, 0, 2]
    a = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "hkvd", rho_bp=2500,
                        r1_bp=5000, window=1, tau=1)
    b = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "forced", forced=a["stages"])
    np.testing.assert_array_equal(a["hidden"], b["hidden"])
    np.testing.assert_array_equal(a["K"], b["K"])
    np.testing.assert_array_equal(a["dev1"], b["dev1"])
    np.testing.assert_array_equal(a["dev2"], b["dev2"])


# ---------------------------------------------------------------- layer wiring, closed forms
# These pin the decoder layer's composition (residuals, O projection orientation, which
# SwiGLU branch carries the SiLU, RMSNorm before the MLP) and the deviation's magnitude
# with weights chosen so that every intermediate has a closed form (CacheBlend blog,
# "Selective KV recompute": the recomputed rows go through the ordinary layer;
# "Picking the tokens to recompute": the deviation between fresh and cached KV).

def _layer_setup(seed=20):
    cfg = tiny_cfg(n_layers=1)
    w = tiny_weights(cfg, seed)
    r = np.random.default_rng(seed)
    N = 9
    K = r.standard_normal((N, 2, 8))
    V = r.standard_normal((N, 2, 8))
    pos = np.array([2, 5, 8])
    x = r.standard_normal((3, 32))
    q = r.standard_normal((3, 4, 8))
    return cfg, w, K, V, pos, x, q


def test_layer_rest_is_identity_without_output_projections():
    """wo = 0 and wd = 0: attention and MLP contribute nothing, so the two residual
    connections return the input rows unchanged, bit for bit."""
    cfg, w, K, V, pos, x, q = _layer_setup()
    w["wo"][0] = 0.0
    w["wd"][0] = 0.0
    np.testing.assert_array_equal(O.layer_rest(w, cfg, 0, x, q, pos, K, V), x)


def test_layer_rest_zero_query_adds_mean_value_through_wo():
    """q = 0 makes every logit 0, so each row's attention output is the plain mean of
    its kv head's values over keys 0..pos; with wo a permutation (row i picks o's column
    perm[i]) and wd = 0, output column i gains that mean's column perm[i]."""
    cfg, w, K, V, pos, x, q = _layer_setup(21)
    q = np.zeros_like(q)
    perm = np.random.default_rng(3).permutation(32)
    wo = np.zeros((32, 32))
    wo[np.arange(32), perm] = 1.0
    w["wo"][0] = wo
    w["wd"][0] = 0.0
    out = O.layer_rest(w, cfg, 0, x, q, pos, K, V)
    want = x.copy()
    for i, p in enumerate(pos):
        o = np.zeros(32)
        for h in range(4):                          # query head h reads kv head h // 2
            o[h * 8:(h + 1) * 8] = V[:p + 1, h // 2].sum(axis=0) / (p + 1)
        for col in range(32):
            want[i, col] += o[perm[col]]
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-14)


def test_layer_rest_one_hot_mlp_adds_silu_gate_times_up():
    """wo = 0; gate row f reads input column a, up row f reads column b, down sends unit
    f to output column j: column j gains silu(n_a) * n_b with n the RMS-normalised row
    (unit gains), every other column is unchanged."""
    cfg, w, K, V, pos, x, q = _layer_setup(22)
    a, bcol, f, j = 3, 17, 5, 29
    w["wo"][0] = 0.0
    w["wg"][0] = 0.0
    w["wu"][0] = 0.0
    w["wd"][0] = 0.0
    w["wg"][0][f, a] = 1.0
    w["wu"][0][f, bcol] = 1.0
    w["wd"][0][j, f] = 1.0
    out = O.layer_rest(w, cfg, 0, x, q, pos, K, V)
    want = x.copy()
    for i in range(3):
        rms = math.sqrt(sum(v * v for v in x[i]) / 32 + 1e-6)
        na, nb = x[i, a] / rms, x[i, bcol] / rms
        want[i, j] += na / (1.0 + math.exp(-na)) * nb
    np.testing.assert_allclose(out, want, rtol=1e-13, atol=1e-14)
    # the SiLU sits on the gate branch: swapping the branches changes the result
    w["wg"][0][f, a], w["wg"][0][f, bcol] = 0.0, 1.0
    w["wu"][0][f, bcol], w["wu"][0][f, a] = 0.0, 1.0
    assert not np.allclose(O.layer_rest(w, cfg, 0, x, q, pos, K, V), want)


def test_deviation_of_constant_offsets():
    """wk = wv = 0 makes the fresh K and V rows zero at every position (a rotation of zero
    is zero), so against caches holding the constants cK and cV the deviation is
    hkv*d*(cK^2 + cV^2) in KV mode and hkv*d*cV^2 in V mode, taken before the overwrite
    (the cache rows are zero afterwards); rows outside dev_rows report 0."""
    cfg, w, K, V, pos, x, q = _layer_setup(23)
    w["wk"][0] = 0.0
    w["wv"][0] = 0.0
    cK, cV = 0.75, -2.5
    for mode, want in (("kv", 2 * 8 * (cK * cK + cV * cV)), ("v", 2 * 8 * cV * cV)):
        Kc = np.full((9, 2, 8), cK)
        Vc = np.full((9, 2, 8), cV)
        rows = np.array([True, False, True])
        _, dev = O.layer_kv(w, cfg, 0, x, pos, Kc, Vc, rows, mode)
        np.testing.assert_allclose(dev, [want, 0.0, want], rtol=1e-15)
        assert np.all(Kc[pos] == 0) and np.all(Vc[pos] == 0)
        untouched = np.setdiff1d(np.arange(9), pos)
        assert np.all(Kc[untouched] == cK) and np.all(Vc[untouched] == cV)


def test_deviation_of_a_known_value_row():
    """wv picks input column c for every value unit and wk = 0: the fresh V row is the
    normalised x[c] everywhere (values are not rotated), so against a zero cache the KV
    deviation is hkv*d*n_c^2, at any position."""
    cfg, w, K, V, pos, x, q = _layer_setup(24)
    c = 11
    w["wk"][0] = 0.0
    w["wv"][0] = 0.0
    w["wv"][0][:, c] = 1.0
    _, dev = O.layer_kv(w, cfg, 0, x, pos, np.zeros((9, 2, 8)), np.zeros((9, 2, 8)), np.ones(3, bool))
    for i in range(3):
        n_c = x[i, c] / math.sqrt(sum(v * v for v in x[i]) / 32 + 1e-6)
        assert abs(dev[i] - 16 * n_c * n_c) <= 1e-12 * 16 * n_c * n_c


# ---------------------------------------------------------------- bf16 operand rounding

def test_round_bf16_closed_forms():
    """bf16 keeps 8 significant bits: near 1 the spacing is 2^-7, halfway cases go to
    the even neighbour, signs are kept, and the exponent is untouched."""
    u = 2.0 ** -7
    cases = [(1.0, 1.0), (1 + u / 2, 1.0), (1 + 1.5 * u, 1 + 2 * u), (1 + u / 2 + 2.0 ** -30, 1 + u),
             (-(1 + u / 2), -1.0), (1 + u, 1 + u), (0.0, 0.0), (3.0 * 2.0 ** 100, 3.0 * 2.0 ** 100),
             (2.0 - u / 4, 2.0), (255.5, 256.0), (254.5, 254.0), (1e-30, None)]
    for x, want in cases:
        got = float(O.round_bf16(np.array([x]))[0])
        if want is None:       # any value: 8 significant bits, within half a spacing
            m, e = math.frexp(x)
            assert abs(got - x) <= 2.0 ** (e - 9) and float(O.round_bf16(np.array([got]))[0]) == got
        else:
            assert got == want, (x, got, want)


def test_round_bf16_matches_torch_conversion():
    """Against torch's float32 -> bfloat16 conversion (round to nearest even) on float32
    values, which float64 holds exactly, over a wide exponent range."""
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(30)
    x = (r.standard_normal(200000) * np.exp2(r.integers(-60, 60, 200000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), want)


def test_operand_rounding_mode(tiny_setup):
    """operand_round="bf16": the cache rows written and the output are bf16 values, the
    residual stream is not rounded (wo = wd = 0 returns the input exactly), and the
    result stays within a few bf16 spacings of the exact one; None is the exact oracle."""
    cfg, w, prefix, chunks, query, ks, vs = tiny_setup
    order = [1, 2, 0]
    scores = np.random.default_rng(4).standard_normal(24)
    kw = dict(rho_bp=5000, window=2, tau=1, scores=scores)
    ex = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "ext", **kw)
    rb = O.blend_prefill(w, cfg, ks, vs, chunks, prefix, order, query, "ext", operand_round="bf16", **kw)
    rows = np.concatenate([ex["stages"][0][1], np.arange(28, 32)])
    for t in (rb["K"][:, rows], rb["V"][:, rows], rb["hidden"]):
        np.testing.assert_array_equal(O.round_bf16(t), t)
    for a, e in ((rb["hidden"], ex["hidden"]), (rb["K"], ex["K"]), (rb["V"], ex["V"])):
        err = np.max(np.abs(a - e)) / np.max(np.abs(e))
        assert 0 < err < 3e-2
    w0 = {k: v.copy() for k, v in w.items()}
    w0["wo"][0] = 0.0
    w0["wd"][0] = 0.0
    x = np.random.default_rng(5).standard_normal((3, 32)) * 7.3
    q = np.random.default_rng(6).standard_normal((3, 4, 8))
    Kc = np.random.default_rng(7).standard_normal((9, 2, 8))
    np.testing.assert_array_equal(
        O.layer_rest(w0, cfg, 0, x, q, np.array([2, 5, 8]), Kc, Kc.copy(), operand_round="bf16"), x)
