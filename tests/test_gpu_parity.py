"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Bars: bit-exact for index work (selection sets, gather/scatter maps, copied rows);
max|gpu - ref| / max|ref| <= 2e-2 for bf16 hidden states and K/V, <= 1e-4 for the fp32
model, <= 1e-3 for fp32 scores and deviations.  Selection sets decided by floating
point on each side (HKVD) are compared as sets that may differ only at near-ties, and
the values are then compared with the GPU forced onto the oracle's sets.
"""
import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import (GpuRunner, assert_hkvd_sets_replay, f64, make_case, maxrel, oracle_cfg, run_oracle, set_diff_is_near_tie,
                       stages_to_device)

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F32 = 1e-4
TOL_SCORE = 1e-3

SMALL_BF16 = synth.ModelShape("small-bf16", 3, 512, 8, 2, 128, 1024, 1000, 1e6)
SMALL_BF16_D64 = synth.ModelShape("small-bf16-d64", 3, 384, 6, 3, 64, 768, 500, 1e4)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


def dev():
    return torch.device("cuda:0")


# ---------------------------------------------------------------- step kernels

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_rope_realign(dtype, d):
    sh = synth.ModelShape("t", 2, 256, 4, 2, d, 688, 64, 1e6, dtype=dtype)
    case = make_case(sh, 4, [8], pool="random")
    r = GpuRunner(case, 64, 4096, 64)
    g = torch.Generator().manual_seed(5)
    L, n = 3, 133
    k = torch.randn(L, n, 2, d, generator=g).to(synth.torch_dtype(sh))
    delta = torch.randint(-4095, 4096, (n,), generator=g, dtype=torch.int32)
    delta[:5] = torch.tensor([0, 1, -1, 4095, -4095], dtype=torch.int32)
    kd = k.to(dev())
    out = torch.empty_like(kd)
    b.rope_realign(r.h, kd, out, n, delta.to(dev()), L, n, n)
    torch.cuda.synchronize()
    ref = np.stack([O.realign_keys(f64(k[l]), delta.numpy(), 1e6) for l in range(L)])
    assert maxrel(f64(out), ref) <= (TOL_BF16 if dtype == "bf16" else 1e-6)
    assert torch.equal(out[:, 0], kd[:, 0])           # shift 0 is the identity, bit for bit
    # in place, and a shift back returns the original within rounding
    back = out.clone()
    b.rope_realign(r.h, back, back, n, (-delta).to(dev()), L, n, n)
    torch.cuda.synchronize()
    assert maxrel(f64(back), f64(k)) <= (TOL_BF16 if dtype == "bf16" else 1e-6)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_assemble(dtype):
    sh = synth.ModelShape("t", 3, 256, 4, 2, 64, 688, 64, 1e4, dtype=dtype)
    lens = [37, 128, 5, 64, 100]
    case = make_case(sh, 9, lens, pool="random")
    r = GpuRunner(case, 64, 4096, 1024)
    order = [3, 0, 4, 1]
    q = torch.randint(0, 64, (7,), dtype=torch.int32, device=dev())
    req = b.RequestRef(order, q, mode="full")
    n_c = sum(lens[c] for c in order)
    N = 9 + n_c + 7
    out = r.outputs(N, 7, n_c)
    b.blend_assemble(r.h, [req], r.pool, out)
    b.blend_device_status(r.h)
    K, V = O.assemble(case.entries_k, case.entries_v, order, 9, [lens[c] for c in order], 7, 1e4)
    gk, gv = f64(out["k"]), f64(out["v"])
    np.testing.assert_array_equal(gv[:, :N - 7], V[:, :N - 7])           # values are copied
    np.testing.assert_array_equal(gk[:, :9], K[:, :9])                   # prefix kept once
    np.testing.assert_array_equal(gk[:, 9:9 + lens[3]], K[:, 9:9 + lens[3]])  # first chunk: shift 0
    assert maxrel(gk[:, :N - 7], K[:, :N - 7]) <= (TOL_BF16 if dtype == "bf16" else 1e-6)


def _select_cases():
    rng = np.random.default_rng(0)
    cases = []
    for i in range(60):
        n = int(rng.integers(1, 300))
        w = int(rng.integers(1, 9))
        tau = int(rng.integers(1, w + 1))
        budget = int(rng.integers(0, n + 2))
        mode = "final" if i % 2 == 0 else "candidate"
        cases.append((n, w, tau, budget, mode, i % 3 == 0))
    cases += [(4000, 8, 5, 800, "final", False), (4000, 8, 5, 800, "candidate", True),
              (15872, 4, 1, 3175, "final", False), (32256, 4, 1, 6452, "final", False),
              (4096, 1, 1, 615, "final", False), (4096, 64, 64, 4096, "final", False)]
    return cases


def test_topk_select_dilate_matches_oracle_exactly():
    sh = synth.ModelShape("t", 1, 256, 4, 2, 64, 688, 64, 1e4, dtype="f32")
    case = make_case(sh, 4, [8], pool="random")
    r = GpuRunner(case, 64, 64, 32768)
    rng = np.random.default_rng(1)
    for (n, w, tau, budget, mode, use_mask) in _select_cases():
        s = rng.integers(0, 7, n).astype(np.float32)            # many exact ties
        if n < 1000:
            s[rng.random(n) < 0.05] = np.nan
            s[rng.random(n) < 0.1] = -0.0
        else:
            s = rng.standard_normal(n).astype(np.float32)
        allowed = (rng.random(n) < 0.6) if use_mask else None
        base = int(rng.integers(0, 100))
        st = torch.from_numpy(s).to(dev())
        al = None if allowed is None else torch.from_numpy(allowed.astype(np.uint8)).to(dev())
        idx = torch.full((n,), -7, dtype=torch.int32, device=dev())
        cnt = torch.zeros(1, dtype=torch.int32, device=dev())
        b.topk_select_dilate(r.h, st, n, base, budget, w, tau, b.BUDGETS[mode], al, idx, cnt)
        torch.cuda.synchronize()
        got = idx[:int(cnt.item())].cpu().numpy().tolist()
        sd = s.astype(np.float64)
        if mode == "candidate":
            want = O.select(sd, budget, w, tau, "candidate", allowed=allowed, base=base)
        else:
            want = O.select_final_bisect(sd, budget, w, tau, allowed=allowed, base=base)
        assert got == want.tolist(), (n, w, tau, budget, mode, use_mask)


def test_topk_select_tile_boundaries_and_ties_across_tiles():
    """The rank kernels sort 2048-position tiles and merge them: sizes around a tile edge and
    the 32768 maximum, with integer scores (exact ties in every tile, broken by position
    across tiles), NaN and -0, with and without a mask, both budget modes."""
    sh = synth.ModelShape("t", 1, 256, 4, 2, 64, 688, 64, 1e4, dtype="f32")
    case = make_case(sh, 4, [8], pool="random")
    r = GpuRunner(case, 64, 64, 32768)
    rng = np.random.default_rng(7)
    for n, w, tau, mode, use_mask in ((2047, 4, 1, "final", False), (2048, 4, 2, "candidate", True),
                                      (2049, 3, 1, "final", True), (6144, 8, 5, "final", False),
                                      (32768, 4, 1, "final", False), (32768, 2, 1, "candidate", True)):
        s = rng.integers(0, 5, n).astype(np.float32)
        s[rng.random(n) < 0.01] = np.nan
        s[rng.random(n) < 0.05] = -0.0
        budget = int(rng.integers(n // 10, n // 4))
        allowed = (rng.random(n) < 0.7) if use_mask else None
        st = torch.from_numpy(s).to(dev())
        al = None if allowed is None else torch.from_numpy(allowed.astype(np.uint8)).to(dev())
        idx = torch.full((n,), -7, dtype=torch.int32, device=dev())
        cnt = torch.zeros(1, dtype=torch.int32, device=dev())
        b.topk_select_dilate(r.h, st, n, 11, budget, w, tau, b.BUDGETS[mode], al, idx, cnt)
        torch.cuda.synchronize()
        got = idx[:int(cnt.item())].cpu().numpy().tolist()
        sd = s.astype(np.float64)
        want = (O.select(sd, budget, w, tau, "candidate", allowed=allowed, base=11) if mode == "candidate"
                else O.select_final_bisect(sd, budget, w, tau, allowed=allowed, base=11))
        assert got == want.tolist(), (n, w, tau, budget, mode, use_mask)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_deviation_scatter_gather(dtype):
    sh = synth.ModelShape("t", 1, 256, 4, 2, 128, 688, 64, 1e4, dtype=dtype)
    case = make_case(sh, 4, [8], pool="random")
    r = GpuRunner(case, 64, 64, 64)
    dt = synth.torch_dtype(sh)
    g = torch.Generator().manual_seed(3)
    n_ctx, n = 300, 77
    kc = torch.randn(n_ctx, 2, 128, generator=g).to(dt).to(dev())
    vc = torch.randn(n_ctx, 2, 128, generator=g).to(dt).to(dev())
    kn = torch.randn(n, 2, 128, generator=g).to(dt).to(dev())
    vn = torch.randn(n, 2, 128, generator=g).to(dt).to(dev())
    pos = torch.sort(torch.randperm(n_ctx, generator=g)[:n]).values.to(torch.int32).to(dev())
    nd = torch.tensor([n], dtype=torch.int32, device=dev())
    for mode in (b.DEV_KV, b.DEV_V):
        dv = torch.zeros(n, device=dev())
        b.kv_deviation(r.h, kn, vn, kc, vc, pos, nd, n, mode, dv)
        torch.cuda.synchronize()
        p = pos.cpu().numpy()
        ref = np.sum((f64(vn) - f64(vc)[p]).reshape(n, -1) ** 2, axis=1)
        if mode == b.DEV_KV:
            ref += np.sum((f64(kn) - f64(kc)[p]).reshape(n, -1) ** 2, axis=1)
        assert maxrel(f64(dv), ref) <= 1e-5
    k2, v2 = kc.clone(), vc.clone()
    b.scatter_kv(r.h, kn, vn, pos, nd, n, k2, v2)
    torch.cuda.synchronize()
    want_k = kc.clone()
    want_k[pos.long()] = kn
    assert torch.equal(k2, want_k)
    rows = torch.empty_like(kn)
    b.gather_rows(r.h, k2, kn[0].numel() * kn.element_size(), pos, nd, n, rows)
    torch.cuda.synchronize()
    assert torch.equal(rows, kn)


# (tokens, layers, dim): the 4 x 2048 shape of the workloads, more layers than a block's
# warps, a width without 16-byte vectors, a single layer
@pytest.mark.parametrize("n,n_layers,dim", [(301, 4, 2048), (37, 11, 72), (19, 3, 70), (5, 1, 3)])
def test_importance_scores(n, n_layers, dim):
    for dt in (torch.float32, torch.bfloat16):
        h = synth.hidden_states(n, n_layers, dim, seed=4, dtype=dt)
        out = torch.empty(n, device=dev())
        b.importance_scores(h.to(dev()), n, n_layers, dim, out)
        torch.cuda.synchronize()
        assert maxrel(f64(out), O.importance_scores(f64(h))) <= 1e-5


def test_importance_scores_unaligned():
    """Rows that start off a 16-byte boundary take the scalar loads."""
    n, n_layers, dim = 23, 4, 256
    for dt in (torch.float32, torch.bfloat16):
        h = synth.hidden_states(n, n_layers, dim, seed=6, dtype=dt)
        buf = torch.zeros(h.numel() + 1, dtype=dt, device=dev())
        buf[1:].copy_(h.reshape(-1).to(dev()))
        hv = buf[1:].view(n, n_layers, dim)
        out = torch.empty(n, device=dev())
        b.importance_scores(hv, n, n_layers, dim, out)
        torch.cuda.synchronize()
        assert maxrel(f64(out), O.importance_scores(f64(h))) <= 1e-5


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_BF16], ids=["f32", "bf16"])
def test_selective_layer(shape):
    case = make_case(shape, 4, [8], pool="random")
    r = GpuRunner(case, 256, 1024, 64)
    g = torch.Generator().manual_seed(9)
    n_ctx, n = 400, 97
    dt = synth.torch_dtype(shape)
    kc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt)
    vc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt)
    x = torch.randn(n, shape.hidden, generator=g)
    pos = torch.sort(torch.randperm(n_ctx, generator=g)[:n]).values.to(torch.int32)
    xg, kg, vg = x.to(dev()), kc.to(dev()), vc.to(dev())
    devo = torch.zeros(n, device=dev())
    b.selective_layer(r.h, 1, xg, pos.to(dev()), n, kg, vg, n_ctx, devo)
    b.blend_device_status(r.h)
    K, V = f64(kc), f64(vc)
    xo, dv = O.layer_forward(case.w_np, oracle_cfg(shape), 1, f64(x), pos.numpy(), K, V,
                             np.ones(n, dtype=bool))
    tol = TOL_BF16 if shape.dtype == "bf16" else TOL_F32
    assert maxrel(f64(kg), K) <= tol and maxrel(f64(vg), V) <= tol
    assert maxrel(f64(xg), xo) <= tol
    assert maxrel(f64(devo), dv) <= (TOL_BF16 if shape.dtype == "bf16" else TOL_SCORE)


# ---------------------------------------------------------------- whole prefill

def _ext_scores(n_c, seed):
    h = synth.hidden_states(n_c, 4, 2048, seed=seed)
    return O.importance_scores(f64(h)).astype(np.float32)


@pytest.mark.parametrize("shape,wnd,tau,budget", [(synth.TINY, 2, 1, "final"), (synth.TINY4, 8, 5, "candidate"),
                                                 (SMALL_BF16, 4, 1, "final"),
                                                 (SMALL_BF16_D64, 4, 2, "candidate")],
                         ids=["f32-w2", "f32-w8t5-cand", "bf16-w4", "bf16d64-w4t2-cand"])
def test_prefill_ext(shape, wnd, tau, budget):
    lens = [128, 128, 128, 128] if shape.dtype == "f32" else [96, 128, 77]
    P, Q = 16, 32
    case = make_case(shape, P, lens, seed=1)
    order = list(range(len(lens)))[::-1]
    n_c = sum(lens)
    N = P + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c)
    query = synth.token_ids(Q, shape.vocab, torch.Generator().manual_seed(77)).numpy()
    scores = _ext_scores(n_c, seed=2)
    req = b.RequestRef(order, torch.from_numpy(query).to(dev()), mode="ext", rho_bp=2000, window=wnd,
                       tau=tau, budget_mode=budget, scores=torch.from_numpy(scores).to(dev()))
    out = r.prefill([req], N, Q, n_c)
    ref = run_oracle(case, order, query, mode="ext", rho_bp=2000, window=wnd, tau=tau, budget_mode=budget,
                     scores=scores.astype(np.float64))
    sel = ref["stages"][0][1]
    ns = int(out["n_sel"][0].item())
    assert out["sel"][:ns].cpu().numpy().tolist() == sel.tolist()
    tol = TOL_BF16 if shape.dtype == "bf16" else TOL_F32
    assert maxrel(f64(out["hidden"]), ref["hidden"]) <= tol
    assert maxrel(f64(out["k"]), ref["K"]) <= tol
    assert maxrel(f64(out["v"]), ref["V"]) <= tol
    # rows neither recomputed nor prefix keep their realigned cache rows on every layer
    K0, V0 = O.assemble(case.entries_k, case.entries_v, order, P, [lens[c] for c in order], Q,
                        shape.rope_theta)
    untouched = sorted(set(range(P, P + n_c)) - set(sel.tolist()))
    np.testing.assert_array_equal(f64(out["v"])[:, untouched], V0[:, untouched])


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY4, SMALL_BF16], ids=["f32-2L", "f32-4L", "bf16-3L"])
def test_prefill_hkvd(shape):
    lens = [128, 128, 128, 128] if shape.dtype == "f32" else [128, 96, 128]
    P, Q = 16, 32
    case = make_case(shape, P, lens, seed=3)
    order = [2, 0, 1] + ([3] if len(lens) == 4 else [])
    n_c = sum(lens)
    N = P + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c)
    query = synth.token_ids(Q, shape.vocab, torch.Generator().manual_seed(78)).numpy()
    qd = torch.from_numpy(query).to(dev())
    kw = dict(rho_bp=2000, r1_bp=3000, window=2, tau=1, budget_mode="final")
    ref = run_oracle(case, order, query, mode="hkvd", **kw)
    out = r.prefill([b.RequestRef(order, qd, mode="hkvd", **kw)], N, Q, n_c)
    score_tol = TOL_BF16 if shape.dtype == "bf16" else TOL_SCORE
    # layer-1 deviation of every chunk row, and the first-stage set
    assert maxrel(f64(out["dev1"]), ref["dev1"]) <= score_tol
    c1_ref = ref["stages"][1][1]
    n1 = int(out["n_c1"][0].item())
    c1 = out["c1"][:n1].cpu().numpy()
    assert n1 == len(c1_ref)
    assert set_diff_is_near_tie(c1 - P, c1_ref - P, ref["dev1"], n1, rel=score_tol)
    # values: the GPU forced onto the oracle's stage sets
    forced = stages_to_device(ref["stages"], dev())
    out2 = r.prefill([b.RequestRef(order, qd, mode="forced", stages=forced)], N, Q, n_c)
    tol = TOL_BF16 if shape.dtype == "bf16" else TOL_F32
    assert maxrel(f64(out2["hidden"]), ref["hidden"]) <= tol
    assert maxrel(f64(out2["k"]), ref["K"]) <= tol
    assert maxrel(f64(out2["v"]), ref["V"]) <= tol
    assert maxrel(f64(out2["dev1"]), ref["dev1"]) <= score_tol
    if shape.n_layers > 2:
        assert maxrel(f64(out2["dev2"]), ref["dev2"]) <= score_tol
        # the GPU's own sets are the oracle's top-k / selection of the GPU's own deviations
        assert_hkvd_sets_replay(out, P, n_c, kw["r1_bp"], kw["rho_bp"], kw["window"], kw["tau"], kw["budget_mode"])


def test_prefill_full_equals_rho_100():
    sh = SMALL_BF16
    lens = [64, 64]
    P, Q = 8, 16
    case = make_case(sh, P, lens, seed=4)
    n_c = sum(lens)
    N = P + n_c + Q
    r = GpuRunner(case, N, N, n_c)
    query = synth.token_ids(Q, sh.vocab, torch.Generator().manual_seed(79)).numpy()
    qd = torch.from_numpy(query).to(dev())
    scores = torch.from_numpy(_ext_scores(n_c, 3)).to(dev())
    a = r.prefill([b.RequestRef([0, 1], qd, mode="ext", rho_bp=10000, window=4, scores=scores)], N, Q, n_c)
    f = r.prefill([b.RequestRef([0, 1], qd, mode="full")], N, Q, n_c)
    ref_h, ref_k, ref_v = O.full_prefill(case.w_np, oracle_cfg(sh),
                                         np.concatenate([case.prefix, case.chunks[0], case.chunks[1], query]))
    for o in (a, f):
        assert maxrel(f64(o["hidden"]), ref_h[-Q:]) <= TOL_BF16
        assert maxrel(f64(o["k"]), ref_k) <= TOL_BF16
        assert maxrel(f64(o["v"]), ref_v) <= TOL_BF16


@pytest.mark.parametrize("sh", [SMALL_BF16_D64, SMALL_BF16], ids=["d64-cuda-cores", "d128-tensor-cores"])
def test_prefill_batch_of_requests_matches_single_runs(sh):
    lens = [64, 48, 64, 32, 64]
    P, Q = 8, 12
    case = make_case(sh, P, lens, seed=5)
    orders = [[4, 1, 2], [0, 3], [2, 4, 0, 1]]
    g = torch.Generator().manual_seed(80)
    queries = [synth.token_ids(Q, sh.vocab, g) for _ in orders]
    ncs = [sum(lens[c] for c in o) for o in orders]
    Ns = [P + n + Q for n in ncs]
    r = GpuRunner(case, sum(ncs) + 3 * Q, sum(Ns), max(ncs), max_batch=3)
    reqs = []
    for o, q, n in zip(orders, queries, ncs):
        s = torch.from_numpy(_ext_scores(n, len(o))).to(dev())
        reqs.append(b.RequestRef(o, q.to(dev()), mode="ext", rho_bp=1500, window=1, scores=s))
    out = r.prefill(reqs, sum(Ns), 3 * Q, sum(ncs))
    tok = 0
    for i, (o, q, n, N) in enumerate(zip(orders, queries, ncs, Ns)):
        ref = run_oracle(case, o, q.numpy(), mode="ext", rho_bp=1500, window=1,
                         scores=f64(reqs[i].scores))
        assert maxrel(f64(out["k"][:, tok:tok + N]), ref["K"]) <= TOL_BF16
        assert maxrel(f64(out["hidden"][i * Q:(i + 1) * Q]), ref["hidden"]) <= TOL_BF16
        nc_off = sum(ncs[:i])
        ns = int(out["n_sel"][i].item())
        assert out["sel"][nc_off:nc_off + ns].cpu().numpy().tolist() == ref["stages"][0][1].tolist()
        tok += N


def test_cache_miss_and_bad_arguments_launch_nothing():
    sh = synth.TINY
    case = make_case(sh, 4, [16, 16], pool="random")
    r = GpuRunner(case, 64, 256, 64)
    q = torch.zeros(4, dtype=torch.int32, device=dev())
    pool = b.PoolRef(r.pool.k, r.pool.v, r.pool.tokens, 4, [16, 16], case.entry_row, present=[1, 0])
    out = r.outputs(40, 4, 32)
    before = out["k"].clone()
    with pytest.raises(b.BlendError) as e:
        b.blend_prefill(r.h, [b.RequestRef([0, 1], q, mode="full")], pool, out)
    assert e.value.code == b.EMISS
    with pytest.raises(b.BlendError) as e:
        b.blend_prefill(r.h, [b.RequestRef([0, 7], q, mode="full")], r.pool, out)
    assert e.value.code == b.EINVAL
    with pytest.raises(b.BlendError) as e:
        b.blend_prefill(r.h, [b.RequestRef([0], q, mode="ext", rho_bp=2000)], r.pool, out)  # no scores
    assert e.value.code == b.EINVAL
    torch.cuda.synchronize()
    assert torch.equal(out["k"], before)


def test_forced_set_out_of_range_is_reported_on_device():
    sh = synth.TINY
    case = make_case(sh, 4, [16, 16], pool="random")
    r = GpuRunner(case, 64, 256, 64)
    q = torch.zeros(4, dtype=torch.int32, device=dev())
    bad = torch.tensor([5, 3, 90], dtype=torch.int32, device=dev())   # unsorted, 90 outside the chunks
    out = r.outputs(40, 4, 32)
    b.blend_prefill(r.h, [b.RequestRef([0, 1], q, mode="forced", stages=[(0, bad)])], r.pool, out)
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(r.h)
    assert e.value.code == b.EDEVICE
    b.blend_device_status(r.h)      # the word was cleared


def test_deterministic():
    sh = SMALL_BF16
    lens = [64, 64, 64]
    P, Q = 8, 16
    case = make_case(sh, P, lens, seed=6, pool="random", pool_std=0.3)
    n_c = sum(lens)
    N = P + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c)
    qd = torch.randint(0, sh.vocab, (Q,), dtype=torch.int32, device=dev())
    req = b.RequestRef([0, 1, 2], qd, mode="hkvd", rho_bp=2000, r1_bp=3000, window=2)
    a = r.prefill([req], N, Q, n_c)
    c = r.prefill([req], N, Q, n_c)
    for k in ("k", "v", "hidden", "sel", "dev1", "dev2"):
        assert torch.equal(a[k], c[k]), k


def test_step_calls_check_positions_on_the_device():
    """kv_deviation, scatter_kv and gather_rows take the cache / source row count: a
    position or index outside it touches no memory and is reported as BLEND_EDEVICE, as is
    a device count above max_n (clamped); the valid rows are still done."""
    sh = SMALL_BF16
    case = make_case(sh, 4, [8], pool="random")
    r = GpuRunner(case, 64, 64, 64)
    g = torch.Generator().manual_seed(21)
    n_ctx, hkv, d = 300, sh.n_kv_heads, sh.head_dim
    kc = torch.randn(n_ctx, hkv, d, generator=g).to(torch.bfloat16).to(dev())
    vc = torch.randn(n_ctx, hkv, d, generator=g).to(torch.bfloat16).to(dev())
    kn = torch.randn(4, hkv, d, generator=g).to(torch.bfloat16).to(dev())
    vn = torch.randn(4, hkv, d, generator=g).to(torch.bfloat16).to(dev())
    pos = torch.tensor([3, n_ctx, 7, -2], dtype=torch.int32, device=dev())
    nd = torch.tensor([4], dtype=torch.int32, device=dev())

    dv = torch.full((4,), -1.0, device=dev())
    b.kv_deviation(r.h, kn, vn, kc, vc, pos, nd, 4, b.DEV_KV, dv)
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(r.h)
    assert e.value.code == b.EDEVICE
    want = [float(np.sum((f64(kn[i]) - f64(kc[p])) ** 2) + np.sum((f64(vn[i]) - f64(vc[p])) ** 2))
            for i, p in ((0, 3), (2, 7))]
    got = dv.cpu().numpy()
    assert got[1] == 0.0 and got[3] == 0.0
    np.testing.assert_allclose(got[[0, 2]], want, rtol=1e-5)

    k2, v2 = kc.clone(), vc.clone()
    b.scatter_kv(r.h, kn, vn, pos, nd, 4, k2, v2)
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(r.h)
    assert e.value.code == b.EDEVICE
    want_k, want_v = kc.clone(), vc.clone()
    want_k[[3, 7]] = kn[[0, 2]]
    want_v[[3, 7]] = vn[[0, 2]]
    assert torch.equal(k2, want_k) and torch.equal(v2, want_v)

    idx = torch.tensor([1, 400, 5], dtype=torch.int32, device=dev())
    dst = torch.full((3, hkv, d), 7.0, dtype=torch.bfloat16, device=dev())
    b.gather_rows(r.h, kc, hkv * d * 2, idx, torch.tensor([3], dtype=torch.int32, device=dev()), 3, dst)
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(r.h)
    assert e.value.code == b.EDEVICE
    assert torch.equal(dst[0], kc[1]) and torch.equal(dst[2], kc[5]) and bool((dst[1] == 7.0).all())

    # a device count above max_n: clamped to max_n, reported
    k3 = kc.clone()
    ok_pos = torch.tensor([10, 11, 12, 13], dtype=torch.int32, device=dev())
    b.scatter_kv(r.h, kn, vn, ok_pos, torch.tensor([9], dtype=torch.int32, device=dev()), 2, k3, vc.clone())
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(r.h)
    assert e.value.code == b.EDEVICE
    assert torch.equal(k3[[10, 11]], kn[[0, 1]]) and torch.equal(k3[[12, 13]], kc[[12, 13]])
    b.blend_device_status(r.h)      # the word was cleared


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_BF16], ids=["f32", "bf16"])
def test_selective_layer_with_a_device_count(shape):
    """The row count of selective_layer can come straight from a device-side selection
    (no host round trip): the set and its size from topk_select_dilate drive the layer,
    with max_n above the count, and give the same rows as a call with the count on the host."""
    case = make_case(shape, 4, [8], pool="random")
    r = GpuRunner(case, 256, 1024, 512)
    g = torch.Generator().manual_seed(13)
    n_ctx, cap = 400, 200
    dt = synth.torch_dtype(shape)
    kc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt).to(dev())
    vc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt).to(dev())
    scores = torch.randn(n_ctx, generator=g).to(dev())
    idx = torch.zeros(n_ctx, dtype=torch.int32, device=dev())
    cnt = torch.zeros(1, dtype=torch.int32, device=dev())
    b.topk_select_dilate(r.h, scores, n_ctx, 0, 97, 2, 1, b.BUDGET_FINAL, None, idx, cnt)
    x = torch.randn(cap, shape.hidden, generator=g).to(dev())
    xa, ka, va = x.clone(), kc.clone(), vc.clone()
    b.selective_layer(r.h, 1, xa, idx, cnt, ka, va, n_ctx, max_n=cap)
    b.blend_device_status(r.h)
    n = int(cnt.item())
    assert 0 < n <= 97
    xb, kb, vb = x.clone(), kc.clone(), vc.clone()
    b.selective_layer(r.h, 1, xb, idx[:n].clone(), n, kb, vb, n_ctx)
    b.blend_device_status(r.h)
    assert torch.equal(xa[:n], xb[:n]) and torch.equal(ka, kb) and torch.equal(va, vb)
    assert torch.equal(xa[n:], x[n:])
    # an empty selection on the device (count 0 under a positive bound) changes nothing
    xc, kc2, vc2 = x.clone(), kc.clone(), vc.clone()
    b.selective_layer(r.h, 1, xc, idx, torch.zeros(1, dtype=torch.int32, device=dev()), kc2, vc2, n_ctx,
                      max_n=cap)
    b.blend_device_status(r.h)
    assert torch.equal(xc, x) and torch.equal(kc2, kc) and torch.equal(vc2, vc)
