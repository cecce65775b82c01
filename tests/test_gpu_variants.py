"""Selection variants on the GPU against the oracle: EPIC's static first-m-tokens rule
(SpecCache notes, background and Figure 1(c)) and Cache-Craft's early termination of
unfocused chunks (Cache-Craft notes, 3.2.2; readings in oracle.focused_chunks)."""
import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import GpuRunner, f64, make_case, maxrel, oracle_cfg, relerr, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


def _tol(sh):
    return 1e-4 if sh.dtype == "f32" else 2e-2


@pytest.mark.parametrize("dtype,m", [("f32", 5), ("bf16", 24), ("bf16", 0), ("bf16", 1000)])
def test_epic_matches_oracle(dtype, m):
    if dtype == "f32":
        sh = synth.ModelShape("epic-f32", 3, 256, 4, 2, 64, 688, 300, 1e4, dtype="f32", init="fan_in")
    else:
        sh = synth.ModelShape("epic-bf16", 2, 256, 4, 2, 128, 512, 300, 1e6)
    case = make_case(sh, 8, [64, 30, 96, 48], seed=5)
    order = [3, 0, 2, 1]
    n_c = sum(len(case.chunks[c]) for c in order)
    Q = 16
    N = len(case.prefix) + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c, max_pos=N)
    g = torch.Generator().manual_seed(7)
    query = synth.token_ids(Q, sh.vocab, g).numpy()
    req = b.RequestRef(order, torch.from_numpy(query).to("cuda:0"), mode="epic", epic_m=m)
    out = r.prefill([req], N, Q, n_c)
    ref = run_oracle(case, order, query, mode="epic", epic_m=m)
    n = int(out["n_sel"][0].item())
    assert out["sel"][:n].cpu().numpy().tolist() == ref["stages"][0][1].tolist()
    t = _tol(sh)
    assert maxrel(f64(out["hidden"]), ref["hidden"]) <= t
    assert maxrel(f64(out["k"]), ref["K"]) <= t and maxrel(f64(out["v"]), ref["V"]) <= t


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_focus_filter_matches_oracle(dtype):
    if dtype == "f32":
        sh = synth.ModelShape("focus-f32", 4, 256, 4, 2, 64, 688, 300, 1e4, dtype="f32", init="fan_in")
    else:
        sh = synth.ModelShape("focus-bf16", 4, 256, 4, 2, 128, 512, 300, 1e6)
    lens = [40, 64, 24, 48, 56]
    case = make_case(sh, 8, lens, seed=6)
    order = [1, 4, 0, 3, 2]
    n_c = sum(len(case.chunks[c]) for c in order)
    Q = 12
    N = len(case.prefix) + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c, max_pos=N)
    g = torch.Generator().manual_seed(8)
    query = synth.token_ids(Q, sh.vocab, g).numpy()
    layer = 2
    # the threshold sits in the middle of the widest gap between the oracle's chunk shares,
    # so rounding cannot move a chunk across it
    shares = _shares_at_layer(case, oracle_cfg(sh), order, query, layer, 20)
    srt = np.sort(shares)
    gap = np.argmax(np.diff(srt))
    thr_bp = int(round(10000 * (srt[gap] + srt[gap + 1]) / 2))
    req = b.RequestRef(order, torch.from_numpy(query).to("cuda:0"), mode="epic", epic_m=20, focus_layer=layer,
                       focus_bp=thr_bp)
    out = r.prefill([req], N, Q, n_c)
    ref = run_oracle(case, order, query, mode="epic", epic_m=20, focus_layer=layer, focus_bp=thr_bp)
    n = int(out["n_sel"][0].item())
    got = out["sel"][:n].cpu().numpy().tolist()
    want = ref["stages"][-1][1].tolist()
    assert 0 < len(want) < len(ref["stages"][0][1]), "the threshold should keep some chunks and drop others"
    assert got == want
    t = _tol(sh)
    assert relerr(f64(out["hidden"]), ref["hidden"]) <= t and maxrel(f64(out["hidden"]), ref["hidden"]) <= t
    assert maxrel(f64(out["k"]), ref["K"]) <= t and maxrel(f64(out["v"]), ref["V"]) <= t


def _shares_at_layer(case, cfg, order, query, layer, epic_m):
    """Chunk shares of the question attention at `layer` in an EPIC run, from the oracle's
    own pieces: the EPIC stage runs layers 0..layer-1, then layer's q and K give the column
    means."""
    w = case.w_np
    P = len(case.prefix)
    lens = [len(case.chunks[c]) for c in order]
    n_c = sum(lens)
    Q = len(query)
    K, V = O.assemble(case.entries_k, case.entries_v, order, P, lens, Q, cfg["rope_theta"])
    tokens = np.concatenate([case.prefix] + [case.chunks[c] for c in order] + [query])
    rows = np.concatenate([O.epic_positions(P, lens, epic_m), np.arange(P + n_c, P + n_c + Q)])
    x = np.asarray(w["embed"], dtype=np.float64)[tokens[rows]]
    for l in range(layer + 1):
        q, _ = O.layer_kv(w, cfg, l, x, rows, K[l], V[l])
        if l < layer:
            x = O.layer_rest(w, cfg, l, x, q, rows, K[l], V[l])
    sc = O.column_mean_scores(q[len(rows) - Q:], rows[len(rows) - Q:], K[layer], P, P + n_c)
    mass = np.array([sc[a:a + L].sum() for a, L in zip(np.cumsum([0] + lens[:-1]), lens)])
    return mass / mass.sum()
