"""Degenerate inputs of the CUDA path against the oracle, through the C ABI.

A recompute ratio of 0 (no chunk row is chosen; only the query rows are recomputed and
every chunk row keeps its realigned cache value, CacheClip paper "direct reuse"); one
chunk behind the prefix with a one-token query; and selection over an empty score array,
with a zero budget, and with a window wider than the scored span (no window can start).
Bars as in the other parity tests: exact for index sets and copied rows, 2e-2 (bf16) /
1e-4 (fp32) relative to max|ref| for values.
"""
import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import GpuRunner, f64, make_case, maxrel, run_oracle

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}
SMALL_BF16 = synth.ModelShape("small-bf16", 2, 512, 8, 2, 128, 1024, 1000, 1e6)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


def dev():
    return torch.device("cuda:0")


def _scores(n, seed):
    return O.importance_scores(f64(synth.hidden_states(n, 4, 256, seed=seed))).astype(np.float32)


def _run(shape, P, lens, Q, rho_bp, window, seed):
    case = make_case(shape, P, lens, seed=seed)
    order = list(range(len(lens)))[::-1]
    n_c = sum(lens)
    N = P + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c)
    query = synth.token_ids(Q, shape.vocab, torch.Generator().manual_seed(5 + seed)).numpy()
    scores = _scores(n_c, seed)
    req = b.RequestRef(order, torch.from_numpy(query).to(dev()), mode="ext", rho_bp=rho_bp, window=window,
                       scores=torch.from_numpy(scores).to(dev()))
    out = r.prefill([req], N, Q, n_c)
    ref = run_oracle(case, order, query, mode="ext", rho_bp=rho_bp, window=window,
                     scores=scores.astype(np.float64))
    return case, order, out, ref, n_c


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_BF16], ids=["f32", "bf16"])
def test_rho_zero_recomputes_only_the_query(shape):
    P, lens, Q = 16, [128, 96, 128], 32
    case, order, out, ref, n_c = _run(shape, P, lens, Q, 0, 4, seed=3)
    assert int(out["n_sel"][0].item()) == 0 and len(ref["stages"][0][1]) == 0
    tol = TOL[shape.dtype]
    assert maxrel(f64(out["hidden"]), ref["hidden"]) <= tol
    assert maxrel(f64(out["k"]), ref["K"]) <= tol
    # every chunk row (and the prefix) is the realigned cache row, on every layer
    K0, V0 = O.assemble(case.entries_k, case.entries_v, order, P, [lens[c] for c in order], Q,
                        shape.rope_theta)
    np.testing.assert_array_equal(f64(out["v"])[:, :P + n_c], V0[:, :P + n_c])
    assert maxrel(f64(out["k"])[:, :P + n_c], K0[:, :P + n_c]) <= tol


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_BF16], ids=["f32", "bf16"])
def test_one_chunk_and_a_one_token_query(shape):
    case, order, out, ref, n_c = _run(shape, 8, [40], 1, 2000, 4, seed=4)
    n = int(out["n_sel"][0].item())
    assert out["sel"][:n].cpu().numpy().tolist() == ref["stages"][0][1].tolist() and n > 0
    tol = TOL[shape.dtype]
    assert maxrel(f64(out["hidden"]), ref["hidden"]) <= tol
    assert maxrel(f64(out["k"]), ref["K"]) <= tol
    assert maxrel(f64(out["v"]), ref["V"]) <= tol


def test_selection_empty_zero_budget_and_wide_window():
    case = make_case(synth.TINY, 4, [8], pool="random")
    r = GpuRunner(case, 64, 64, 1024)
    rng = np.random.default_rng(6)
    for n, budget, w, tau, mode in [(0, 10, 1, 1, "final"), (0, 0, 4, 2, "candidate"), (100, 0, 1, 1, "final"),
                                    (100, 0, 4, 1, "candidate"), (5, 3, 8, 1, "final"), (5, 3, 8, 1, "candidate"),
                                    (7, 7, 7, 7, "final")]:
        s = rng.standard_normal(max(n, 1)).astype(np.float32)[:n]
        st = torch.from_numpy(s.copy() if n else np.zeros(1, np.float32)).to(dev())
        idx = torch.full((max(n, 1),), -7, dtype=torch.int32, device=dev())
        cnt = torch.full((1,), -7, dtype=torch.int32, device=dev())
        b.topk_select_dilate(r.h, st, n, 10, budget, w, tau, b.BUDGETS[mode], None, idx, cnt)
        torch.cuda.synchronize()
        got = idx[:int(cnt.item())].cpu().numpy().tolist()
        sd = s.astype(np.float64)
        want = (O.select(sd, budget, w, tau, "candidate", base=10) if mode == "candidate"
                else O.select_final_bisect(sd, budget, w, tau, base=10))
        assert got == list(want), (n, budget, w, tau, mode)
        if n == 0 or budget == 0 or w > n:
            assert got == []
