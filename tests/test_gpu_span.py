"""SpecCache span completion, global budget and cross-tokenizer alignment on the GPU
(span_select, align_expand, and blend_prefill with the span rule) against the oracle
(SpecCache notes, "2.3 Semantic span completion", "2.4 Cross-tokenizer alignment").

Selections are integer results: they must match the oracle exactly.  Both sides take
every merge decision in fp32 (the oracle in numpy float32), so no tolerance applies.
"""
import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import GpuRunner, f64, make_case, maxrel, run_oracle, stages_to_device

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


@pytest.fixture(scope="module")
def runner():
    sh = synth.ModelShape("t", 1, 256, 4, 2, 64, 688, 64, 1e4, dtype="f32")
    case = make_case(sh, 4, [8], pool="random")
    return GpuRunner(case, 64, 64, 32768)


def _scores(rng, n, kind):
    if kind == "walk":  # locally smooth, so spans of several tokens form
        return (5.0 + np.cumsum(rng.normal(0, 0.05, n))).astype(np.float32)
    if kind == "phrases":  # runs of 1..8 tokens of similar importance
        out = []
        while len(out) < n:
            ln = int(rng.integers(1, 9))
            out += list(rng.lognormal(0, 0.6) * (1 + rng.normal(0, 0.03, ln)))
        return np.array(out[:n], dtype=np.float32)
    if kind == "ties":  # exact ties, zeros of both signs, negatives, NaN
        s = rng.integers(-3, 4, n).astype(np.float32)
        s[rng.random(n) < 0.1] = -0.0
        s[rng.random(n) < 0.03] = np.nan
        return s
    if kind == "flat":
        return np.full(n, 0.75, dtype=np.float32)
    return rng.random(n).astype(np.float32)


CASES = [
    # n, kind, budget fraction, mode, tau_smooth, tau_cover_bp, max_span, cap fraction
    (1, "iid", 1.0, "final", 0.4, 7000, 16, 1.0),
    (7, "walk", 0.5, "final", 0.4, 7000, 16, 1.0),
    (100, "walk", 0.2, "final", 0.4, 7000, 16, 1.0),
    (100, "phrases", 0.2, "candidate", 0.4, 7000, 16, 0.3),
    (257, "ties", 0.3, "final", 0.4, 5000, 8, 1.0),
    (257, "ties", 0.3, "candidate", 0.4, 5000, 8, 0.35),
    (1000, "phrases", 0.15, "final", 0.4, 7000, 16, 1.0),
    (1000, "walk", 0.15, "candidate", 0.6, 6000, 32, 0.25),
    (1000, "flat", 0.2, "final", 0.4, 7000, 16, 1.0),
    (1000, "iid", 0.2, "candidate", 0.4, 7000, 16, 0.2),
    (4097, "phrases", 0.2, "final", 0.4, 7000, 16, 1.0),
    (4097, "walk", 0.2, "candidate", 0.4, 10000, 64, 0.5),
    (4097, "walk", 0.0, "final", 0.4, 7000, 16, 1.0),
    (4097, "walk", 1.0, "final", 0.4, 7000, 16, 1.0),
    (4097, "phrases", 0.2, "final", 0.4, 7000, 1, 1.0),
    (15872, "phrases", 0.2, "final", 0.4, 7000, 16, 1.0),
    (32768, "walk", 0.2, "final", 0.4, 7000, 16, 1.0),
    (32768, "phrases", 0.1, "candidate", 0.4, 7000, 16, 0.12),
]


@pytest.mark.parametrize("n,kind,bf,mode,ts,tc,ms,cf", CASES)
def test_span_select_matches_oracle_exactly(runner, n, kind, bf, mode, ts, tc, ms, cf):
    rng = np.random.default_rng(n + int(1000 * bf) + tc + ms)
    s = _scores(rng, n, kind)
    budget = int(round(bf * n))
    cap = int(round(cf * n))
    base = 37
    dev = torch.device("cuda:0")
    idx = torch.full((n,), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    b.span_select(runner.h, torch.from_numpy(s).to(dev), n, base, budget, cap, ts, tc, ms, b.BUDGETS[mode], idx, cnt)
    torch.cuda.synchronize()
    got = idx[:int(cnt.item())].cpu().numpy().tolist()
    if mode == "candidate":
        want = O.span_select(s, budget, ts, tc, ms, "candidate", cap=cap, base=base)
    else:
        want = O.span_select_final_bisect(s, budget, ts, tc, ms, base=base)
    assert got == want.tolist()
    if mode == "final":
        assert len(got) <= budget


def test_span_select_empty_and_argument_checks(runner):
    dev = torch.device("cuda:0")
    idx = torch.zeros(4, dtype=torch.int32, device=dev)
    cnt = torch.full((1,), 99, dtype=torch.int32, device=dev)
    s = torch.zeros(4, device=dev)
    b.span_select(runner.h, s, 0, 0, 0, 0, 0.4, 7000, 16, b.BUDGET_FINAL, idx, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 0
    for bad in [dict(ts=float("nan")), dict(ts=-1.0), dict(tc=0), dict(tc=10001), dict(ms=0), dict(ms=65)]:
        a = dict(ts=0.4, tc=7000, ms=16)
        a.update(bad)
        with pytest.raises(b.BlendError):
            b.span_select(runner.h, s, 4, 0, 2, 2, a["ts"], a["tc"], a["ms"], b.BUDGET_FINAL, idx, cnt)


@pytest.mark.parametrize("n_spec,split,n_sel", [(1, 1, 1), (100, 2, 30), (5000, 3, 1200), (40000, 3, 9000)])
def test_align_expand_matches_oracle(runner, n_spec, split, n_sel):
    """Random alignments: each speculative token covers 0..split target tokens, some
    ranges overlapping their neighbour (two tokenizations of the same text)."""
    rng = np.random.default_rng(n_spec)
    widths = rng.integers(0, split + 1, n_spec)
    start = np.concatenate([[0], np.cumsum(widths)[:-1]]).astype(np.int32)
    end = (start + widths).astype(np.int32)
    ov = rng.random(n_spec) < 0.2
    start = np.where(ov & (start > 0), start - 1, start).astype(np.int32)
    n_target = int(end.max()) if n_spec else 0
    assert n_target <= b.MAX_ALIGN_TARGETS
    sel = np.sort(rng.choice(n_spec, size=min(n_sel, n_spec), replace=False)).astype(np.int32)
    dev = torch.device("cuda:0")
    sel_base, out_base = 11, 500
    out = torch.full((max(n_target, 1),), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    b.align_expand(runner.h, torch.from_numpy(sel + sel_base).to(dev),
                   torch.tensor([len(sel)], dtype=torch.int32, device=dev), len(sel), sel_base,
                   torch.from_numpy(start).to(dev), torch.from_numpy(end).to(dev), n_spec, n_target, out_base,
                   out, cnt)
    b.blend_device_status(runner.h)
    got = out[:int(cnt.item())].cpu().numpy().tolist()
    want = (O.align_expand(sel, start, end) + out_base).tolist()
    assert got == want


def test_align_expand_reports_bad_ranges(runner):
    dev = torch.device("cuda:0")
    start = torch.tensor([0, 2, 5], dtype=torch.int32, device=dev)
    end = torch.tensor([2, 9, 6], dtype=torch.int32, device=dev)  # token 1 runs past n_target
    sel = torch.tensor([0, 1], dtype=torch.int32, device=dev)
    out = torch.zeros(8, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    b.align_expand(runner.h, sel, torch.tensor([2], dtype=torch.int32, device=dev), 2, 0, start, end, 3, 8, 0,
                   out, cnt)
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(runner.h)
    assert e.value.code == b.EDEVICE
    assert out[:int(cnt.item())].cpu().tolist() == [0, 1]  # the bad range is skipped


@pytest.mark.parametrize("budget_mode", ["final", "candidate"])
def test_blend_prefill_with_span_rule(budget_mode):
    """A bf16 2-layer EXT prefill whose set comes from span completion: the set equals
    the oracle's, the hidden state and blended K/V are within the bf16 bound."""
    sh = synth.ModelShape("span-bf16", 2, 256, 4, 2, 128, 512, 300, 1e6)
    case = make_case(sh, 8, [64, 48, 96, 64], seed=3)
    order = [3, 1, 0, 2]
    n_c = sum(len(case.chunks[c]) for c in order)
    Q = 16
    g = torch.Generator().manual_seed(5)
    query = synth.token_ids(Q, sh.vocab, g).numpy()
    rng = np.random.default_rng(9)
    s = _scores(rng, n_c, "phrases")
    N = len(case.prefix) + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c, max_pos=N)
    dev = torch.device("cuda:0")
    req = b.RequestRef(order, torch.from_numpy(query).to(dev), mode="ext", rho_bp=2000,
                       budget_mode=budget_mode, scores=torch.from_numpy(s).to(dev), group_rule="span",
                       tau_smooth=0.4, tau_cover_bp=7000, max_span=16, cap_bp=3000)
    out = r.prefill([req], N, Q, n_c)
    ref = run_oracle(case, order, query, mode="ext", rho_bp=2000, budget_mode=budget_mode,
                     scores=s.astype(np.float64), group_rule="span", tau_smooth=0.4, tau_cover_bp=7000,
                     max_span=16, cap_bp=3000)
    n = int(out["n_sel"][0].item())
    want = ref["stages"][0][1]
    assert out["sel"][:n].cpu().numpy().tolist() == want.tolist()
    assert maxrel(f64(out["hidden"]), ref["hidden"]) <= TOL_BF16
    assert maxrel(f64(out["k"]), ref["K"]) <= TOL_BF16
    assert maxrel(f64(out["v"]), ref["V"]) <= TOL_BF16
