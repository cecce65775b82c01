"""Parity at full depth: every layer of the Llama-3-8B-shaped HKVD request (32 layers), of
the Mistral-7B-shaped batch (32 layers), of the 14B-shaped sweep's 4K context at 10 % (48
layers) and, behind BLEND_FULL_DEPTH_48, of the 14B-shaped 16K request (48 layers), through
blend_prefill in the configuration the benchmark times, against the CPU oracle, with the
error reported per layer.

What is checked, and against what:
  * integer outputs exactly: the HKVD stage sets are the oracle's top-k and selection
    (CacheBlend blog, "Implementation": check layers pick the tokens with the largest KV
    deviation) replayed on the GPU's own deviation arrays; the batch's sets are the
    oracle's selection on the same score arrays;
  * the GPU's deviations against the oracle's, and its sets against the oracle's up to
    near-ties of the oracle's deviations;
  * values (hidden state, every layer's K and V) with the GPU forced onto the oracle's
    sets, against the exact float64 oracle.  bf16 operands (the GEMM inputs, q, the
    attention weights, the cache rows) put a floor under that error which grows with
    depth; the oracle's operand_round="bf16" run measures the floor on the same request,
    and the GPU must stay within FLOOR_RATIO of it.  The 2e-2 bar (max relative error of
    bf16 outputs) is checked at full depth as an explicit expected failure: bf16 arithmetic
    alone exceeds it beyond roughly eight layers of these random-weight models.

The chunk pools are seeded Gaussian (precomputing 32-layer chunk caches in float64 on the
host would take minutes); the HKVD deviations then compare fresh rows with those values.
The tensors of both sides come from the same seeded generators.
"""
import dataclasses
import time

import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import (f64, layerwise_weights, maxrel, oracle_cfg, per_layer_errors, relerr,
                       set_diff_is_near_tie, stages_to_device)

pytestmark = pytest.mark.gpu

TOL = 2e-2            # max relative error of bf16 hidden states and K/V
FLOOR_RATIO = 1.3     # GPU error / error of the same request with bf16 operands in the oracle


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


def dev():
    return torch.device("cuda:0")


class PoolEntries:
    """Entry c of a device pool ([L][P+L_c][hkv][d]) as float64, converted when the oracle
    reads it (a 64-entry pool never exists in float64 all at once)."""

    def __init__(self, t, row_off, rows):
        self.t, self.row_off, self.rows = t, row_off, rows

    def __getitem__(self, c):
        return f64(self.t[:, self.row_off[c]:self.row_off[c] + self.rows[c]])

    def __len__(self):
        return len(self.rows)


class Request:
    """One workload at its full depth: device weights, their layer-by-layer float64 view
    for the oracle, a seeded Gaussian pool on the device and its float64 entries."""

    def __init__(self, wl: synth.Workload):
        self.wl, self.sh = wl, wl.model
        sh = self.sh
        w = synth.model_weights(sh, wl.seed, device=dev())
        self.w_or = layerwise_weights(w)
        self.packed = b.pack_weights(w)
        self.pool_tok, self.reqs = synth.workload_tokens(wl)
        n_entries = len(self.pool_tok.chunks)
        self.P, self.lens = wl.prefix_len, [wl.chunk_len] * n_entries
        k, v, row_off = synth.random_pool_kv(sh, self.P, self.lens, wl.seed, device=dev())
        self.entries_k = PoolEntries(k, row_off, [self.P + L for L in self.lens])
        self.entries_v = PoolEntries(v, row_off, [self.P + L for L in self.lens])
        tok = torch.cat([torch.cat([self.pool_tok.prefix, c]) for c in self.pool_tok.chunks]).to(dev())
        self.pool = b.PoolRef(k, v, tok, self.P, self.lens, row_off)
        self.chunks = [c.numpy() for c in self.pool_tok.chunks]
        self.prefix = self.pool_tok.prefix.numpy()
        self.N, self.n_c, self.Q = wl.n_ctx, wl.n_chunk_rows, wl.query_len
        self.cfg = oracle_cfg(sh)

    def handle(self, max_rows, batch=1):
        return b.blend_init(b.model_cfg(self.sh, self.N), self.packed,
                            b.Limits(max_rows, self.N * batch, self.n_c, batch))

    def outputs(self, batch=1):
        sh, L, d = self.sh, self.sh.n_layers, dev()
        z32 = lambda n: torch.zeros(n, dtype=torch.float32, device=d)
        neg = lambda n: torch.full((n,), -1, dtype=torch.int32, device=d)
        return b.OutputsRef(
            k=torch.zeros(L, self.N * batch, sh.n_kv_heads, sh.head_dim, dtype=torch.bfloat16, device=d),
            v=torch.zeros(L, self.N * batch, sh.n_kv_heads, sh.head_dim, dtype=torch.bfloat16, device=d),
            hidden=torch.zeros(self.Q * batch, sh.hidden, dtype=torch.bfloat16, device=d),
            sel=neg(self.n_c * batch), n_sel=torch.zeros(b.MAX_BATCH, dtype=torch.int32, device=d),
            c1=neg(self.n_c * batch), n_c1=torch.zeros(b.MAX_BATCH, dtype=torch.int32, device=d),
            dev1=z32(self.n_c * batch), dev2=z32(self.n_c * batch))

    def oracle(self, r, **kw):
        req = self.reqs[r]
        t0 = time.time()
        out = O.blend_prefill(self.w_or, self.cfg, self.entries_k, self.entries_v, self.chunks, self.prefix,
                              req.chunk_ids, req.query.numpy(), **kw)
        print(f"[fulldepth] oracle {kw.get('mode')} {kw.get('operand_round') or 'exact'}: {time.time() - t0:.1f} s")
        return out


def whole_errors(got_k, got_v, got_hidden, ref):
    """2-norm and max-norm relative errors of the hidden rows and of K and V over every
    layer (converted one layer at a time), plus the per-layer table."""
    layers = per_layer_errors(got_k, got_v, ref["K"], ref["V"])
    out = {"layers": layers}
    gh = got_hidden if isinstance(got_hidden, np.ndarray) else f64(got_hidden)
    out["hidden"] = (relerr(gh, ref["hidden"]), maxrel(gh, ref["hidden"]))
    for name, gt, rt in (("K", got_k, ref["K"]), ("V", got_v, ref["V"])):
        num = den = 0.0
        mx_d = mx_r = 0.0
        for l in range(rt.shape[0]):
            g = gt[l] if isinstance(gt, np.ndarray) else f64(gt[l])
            d = g - rt[l]
            num += float(np.sum(d * d))
            den += float(np.sum(rt[l] * rt[l]))
            mx_d = max(mx_d, float(np.max(np.abs(d))))
            mx_r = max(mx_r, float(np.max(np.abs(rt[l]))))
        out[name] = (np.sqrt(num / den), mx_d / mx_r)
    return out


def report(tag, gpu, floor):
    print(f"[fulldepth] {tag}: per layer, GPU vs exact oracle (2-norm / max-norm), bf16-operand oracle vs exact (2-norm)")
    for l, (g, f) in enumerate(zip(gpu["layers"], floor["layers"])):
        print(f"[fulldepth] {tag} L{l:2d}  K {g[0]:.3e} / {g[1]:.3e}  V {g[2]:.3e} / {g[3]:.3e}"
              f"   floor K {f[0]:.3e} V {f[2]:.3e}")
    for k in ("hidden", "K", "V"):
        print(f"[fulldepth] {tag} {k}: GPU {gpu[k][0]:.3e} / {gpu[k][1]:.3e}, floor {floor[k][0]:.3e} / "
              f"{floor[k][1]:.3e}, ratio {gpu[k][0] / floor[k][0]:.2f}")


# ---------------------------------------------------------------- Llama-3-8B shape, HKVD 15 %

@pytest.fixture(scope="module")
def llama8b():
    wl = synth.WORKLOADS["llama8b-3k-hkvd15"]
    rq = Request(wl)
    req = rq.reqs[0]
    kw = dict(rho_bp=wl.rho_bp, r1_bp=wl.r1_bp, window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode)
    h = rq.handle(rq.n_c + rq.Q)
    qd = req.query.to(dev())
    sel_run = rq.outputs()
    b.blend_prefill(h, [b.RequestRef(req.chunk_ids, qd, mode="hkvd", **kw)], rq.pool, sel_run)
    b.blend_device_status(h)
    ref = rq.oracle(0, mode="hkvd", **kw)
    forced = rq.outputs()
    b.blend_prefill(h, [b.RequestRef(req.chunk_ids, qd, mode="forced", stages=stages_to_device(ref["stages"], dev()))],
                    rq.pool, forced)
    b.blend_device_status(h)
    torch.cuda.synchronize()
    floor = rq.oracle(0, mode="forced", forced=ref["stages"], operand_round="bf16")
    res = dict(rq=rq, wl=wl, sel_run=sel_run, ref=ref, forced=forced,
               gpu=whole_errors(forced["k"], forced["v"], forced["hidden"], ref),
               floor=whole_errors(floor["K"], floor["V"], floor["hidden"], ref))
    report("8B HKVD 32 layers", res["gpu"], res["floor"])
    return res


def test_llama8b_hkvd_32_layers_sets(llama8b):
    """The GPU's stage sets are the oracle's top-k / selection of the GPU's own
    deviation arrays, exactly; its deviations match the oracle's; its first-stage set
    differs from the oracle's only at near-ties of the oracle's deviations."""
    rq, wl, o, ref = llama8b["rq"], llama8b["wl"], llama8b["sel_run"], llama8b["ref"]
    P, n_c = rq.P, rq.n_c
    n1, ns = int(o["n_c1"][0].item()), int(o["n_sel"][0].item())
    c1 = o["c1"][:n1].cpu().numpy().astype(np.int64)
    sel = o["sel"][:ns].cpu().numpy().astype(np.int64)
    d1, d2 = f64(o["dev1"]), f64(o["dev2"])
    assert n1 == O.ceil_bp(wl.r1_bp, n_c)
    assert c1.tolist() == sorted(P + t for t in O.topk(d1, n1))
    allowed = np.zeros(n_c, dtype=bool)
    allowed[c1 - P] = True
    budget = O.ceil_bp(wl.rho_bp, n_c)
    dscore = np.where(allowed, d2, -np.inf)
    want = (O.select(dscore, budget, wl.window, wl.tau, "candidate", allowed=allowed, base=P)
            if wl.budget_mode == "candidate"
            else O.select_final_bisect(dscore, budget, wl.window, wl.tau, allowed=allowed, base=P))
    assert sel.tolist() == want.tolist()
    assert np.all(d2[~allowed] == 0)
    e2, em = relerr(d1, ref["dev1"]), maxrel(d1, ref["dev1"])
    print(f"[fulldepth] 8B HKVD dev1 vs oracle {e2:.3e} / {em:.3e}; C1 overlap "
          f"{len(set(c1) & set(ref['stages'][1][1])) / n1:.4f}, S overlap "
          f"{len(set(sel) & set(ref['stages'][2][1])) / max(1, ns):.4f}")
    assert e2 <= TOL and em <= TOL
    assert set_diff_is_near_tie(c1 - P, ref["stages"][1][1] - P, ref["dev1"], n1, rel=TOL)
    fd2 = f64(llama8b["forced"]["dev2"])
    assert relerr(fd2, ref["dev2"]) <= TOL and maxrel(fd2, ref["dev2"]) <= TOL


def test_llama8b_hkvd_32_layers_at_the_bf16_floor(llama8b):
    """Hidden state and every layer's K/V with the GPU on the oracle's sets: the error
    against the exact oracle is at most FLOOR_RATIO times the error bf16 operands alone
    give on the same request."""
    gpu, floor = llama8b["gpu"], llama8b["floor"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= FLOOR_RATIO * floor[k][0], (k, gpu[k], floor[k])
    assert np.all(np.isfinite(f64(llama8b["forced"]["hidden"])))


@pytest.mark.xfail(strict=True, reason="fails the 2e-2 bar at full depth: bf16 operand rounding alone "
                                       "(the oracle's operand_round run) exceeds it beyond ~8 of 32 layers")
def test_llama8b_hkvd_32_layers_2e2_bar(llama8b):
    gpu = llama8b["gpu"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= TOL and gpu[k][1] <= TOL, (k, gpu[k])


# ---------------------------------------------------------------- Mistral-7B shape, batch of 8, EXT 15 %

def ext_scores(n_c, seed):
    h = synth.hidden_states(n_c, 4, 2048, seed)
    return O.importance_scores(f64(h)).astype(np.float32)


@pytest.fixture(scope="module")
def mistral7b():
    wl = synth.WORKLOADS["mistral7b-b8-ext15"]
    rq = Request(wl)
    Bn = wl.batch
    budget = O.ceil_bp(wl.rho_bp, rq.n_c)
    h = rq.handle(Bn * (budget + rq.Q), batch=Bn)
    scores, reqs = [], []
    for r in range(Bn):
        s = ext_scores(rq.n_c, wl.seed + r)
        scores.append(s)
        reqs.append(b.RequestRef(rq.reqs[r].chunk_ids, rq.reqs[r].query.to(dev()), mode="ext", rho_bp=wl.rho_bp,
                                 window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode,
                                 scores=torch.from_numpy(s).to(dev())))
    out = rq.outputs(batch=Bn)
    b.blend_prefill(h, reqs, rq.pool, out)
    b.blend_device_status(h)
    torch.cuda.synchronize()
    kw = dict(mode="ext", rho_bp=wl.rho_bp, window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode,
              scores=scores[0].astype(np.float64))
    ref = rq.oracle(0, **kw)
    floor = rq.oracle(0, operand_round="bf16", **kw)
    N, Q = rq.N, rq.Q
    res = dict(rq=rq, wl=wl, out=out, scores=scores, ref=ref,
               gpu=whole_errors(out["k"][:, :N], out["v"][:, :N], out["hidden"][:Q], ref),
               floor=whole_errors(floor["K"], floor["V"], floor["hidden"], ref))
    report("7B batch req0 32 layers", res["gpu"], res["floor"])
    return res


def test_mistral7b_batch8_32_layers_sets(mistral7b):
    """Every request's set is the oracle's selection of its score array, exactly."""
    rq, wl, out = mistral7b["rq"], mistral7b["wl"], mistral7b["out"]
    budget = O.ceil_bp(wl.rho_bp, rq.n_c)
    for r in range(wl.batch):
        s = mistral7b["scores"][r].astype(np.float64)
        want = (O.select(s, budget, wl.window, wl.tau, "candidate", base=rq.P) if wl.budget_mode == "candidate"
                else O.select_final_bisect(s, budget, wl.window, wl.tau, base=rq.P))
        ns = int(out["n_sel"][r].item())
        c0 = r * rq.n_c
        assert out["sel"][c0:c0 + ns].cpu().numpy().tolist() == want.tolist(), r
    assert mistral7b["ref"]["stages"][0][1].tolist() == out["sel"][:int(out["n_sel"][0].item())].cpu().numpy().tolist()


def test_mistral7b_batch8_32_layers_at_the_bf16_floor(mistral7b):
    """Request 0 of the batch (its rows share every weight pass with seven others): hidden
    state and every layer's K/V within FLOOR_RATIO of the bf16-operand floor."""
    gpu, floor = mistral7b["gpu"], mistral7b["floor"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= FLOOR_RATIO * floor[k][0], (k, gpu[k], floor[k])


@pytest.mark.xfail(strict=True, reason="fails the 2e-2 bar at full depth: bf16 operand rounding alone "
                                       "(the oracle's operand_round run) exceeds it beyond ~8 of 32 layers")
def test_mistral7b_batch8_32_layers_2e2_bar(mistral7b):
    gpu = mistral7b["gpu"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= TOL and gpu[k][1] <= TOL, (k, gpu[k])


# ---------------------------------------------------------------- 14B shape, 16K context, EXT 20 %, all 48 layers

RUN_48 = bool(int(__import__("os").environ.get("BLEND_FULL_DEPTH_48", "0")))


@pytest.fixture(scope="module")
def qwen14b():
    if not RUN_48:
        pytest.skip("48-layer 16K oracle runs take ~10 minutes on 16 host cores: set BLEND_FULL_DEPTH_48=1")
    wl = synth.WORKLOADS["qwen14b-16k-ext20"]
    rq = Request(wl)
    req = rq.reqs[0]
    s = ext_scores(rq.n_c, wl.seed)
    h = rq.handle(rq.n_c + rq.Q)
    out = rq.outputs()
    b.blend_prefill(h, [b.RequestRef(req.chunk_ids, req.query.to(dev()), mode="ext", rho_bp=wl.rho_bp,
                                     window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode,
                                     scores=torch.from_numpy(s).to(dev()))], rq.pool, out)
    b.blend_device_status(h)
    torch.cuda.synchronize()
    kw = dict(mode="ext", rho_bp=wl.rho_bp, window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode,
              scores=s.astype(np.float64))
    ref = rq.oracle(0, **kw)
    gpu = whole_errors(out["k"], out["v"], out["hidden"], ref)
    floor = rq.oracle(0, operand_round="bf16", **kw)
    res = dict(rq=rq, out=out, ref=ref, gpu=gpu, floor=whole_errors(floor["K"], floor["V"], floor["hidden"], ref))
    report("14B 16K 48 layers", res["gpu"], res["floor"])
    return res


def test_qwen14b_16k_48_layers_set_and_floor(qwen14b):
    out, ref = qwen14b["out"], qwen14b["ref"]
    ns = int(out["n_sel"][0].item())
    assert out["sel"][:ns].cpu().numpy().tolist() == ref["stages"][0][1].tolist()
    gpu, floor = qwen14b["gpu"], qwen14b["floor"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= FLOOR_RATIO * floor[k][0], (k, gpu[k], floor[k])


@pytest.mark.xfail(strict=True, reason="fails the 2e-2 bar at full depth: bf16 operand rounding alone "
                                       "(the oracle's operand_round run) exceeds it at 48 layers")
def test_qwen14b_16k_48_layers_2e2_bar(qwen14b):
    gpu = qwen14b["gpu"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= TOL and gpu[k][1] <= TOL, (k, gpu[k])


# ---------------------------------------------------------------- the sweep's 4K context at 10 %, all 48 layers

@pytest.fixture(scope="module")
def sweep4k():
    wl = synth.sweep_workload(7, 1000)
    rq = Request(wl)
    req = rq.reqs[0]
    s = ext_scores(rq.n_c, 9)
    h = rq.handle(rq.n_c + rq.Q)
    out = rq.outputs()
    b.blend_prefill(h, [b.RequestRef(req.chunk_ids, req.query.to(dev()), mode="ext", rho_bp=wl.rho_bp,
                                     window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode,
                                     scores=torch.from_numpy(s).to(dev()))], rq.pool, out)
    b.blend_device_status(h)
    torch.cuda.synchronize()
    kw = dict(mode="ext", rho_bp=wl.rho_bp, window=wl.window, tau=wl.tau, budget_mode=wl.budget_mode,
              scores=s.astype(np.float64))
    ref = rq.oracle(0, **kw)
    floor = rq.oracle(0, operand_round="bf16", **kw)
    res = dict(rq=rq, out=out, ref=ref, gpu=whole_errors(out["k"], out["v"], out["hidden"], ref),
               floor=whole_errors(floor["K"], floor["V"], floor["hidden"], ref))
    report("14B 4K 10 % 48 layers", res["gpu"], res["floor"])
    return res


def test_sweep_4k_10pct_48_layers_set_and_floor(sweep4k):
    """The context x ratio sweep's 4K context at 10 % on the 14B shape, every layer: the
    set exactly, values within FLOOR_RATIO of the bf16-operand floor."""
    out, ref = sweep4k["out"], sweep4k["ref"]
    ns = int(out["n_sel"][0].item())
    assert out["sel"][:ns].cpu().numpy().tolist() == ref["stages"][0][1].tolist()
    gpu, floor = sweep4k["gpu"], sweep4k["floor"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= FLOOR_RATIO * floor[k][0], (k, gpu[k], floor[k])


@pytest.mark.xfail(strict=True, reason="fails the 2e-2 bar at full depth: bf16 operand rounding alone "
                                       "(the oracle's operand_round run) exceeds it at 48 layers")
def test_sweep_4k_10pct_48_layers_2e2_bar(sweep4k):
    gpu = sweep4k["gpu"]
    for k in ("hidden", "K", "V"):
        assert gpu[k][0] <= TOL and gpu[k][1] <= TOL, (k, gpu[k])
