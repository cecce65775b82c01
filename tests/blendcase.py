"""Test harness: builds one blended-prefill case for both the CUDA path (through the
C ABI binding) and the CPU oracle, from the same seeded inputs (synth).  It holds no
arithmetic of the method: it only moves arrays between torch, numpy and the two sides.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import synth


def oracle_cfg(shape: synth.ModelShape) -> dict:
    return dict(n_layers=shape.n_layers, hidden=shape.hidden, n_q_heads=shape.n_q_heads,
                n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, ffn=shape.ffn, vocab=shape.vocab,
                rope_theta=shape.rope_theta, rms_eps=shape.rms_eps)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def relerr(got, ref) -> float:
    """Norm-wise relative error ||got - ref||_2 / ||ref||_2."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.sum(ref * ref))
    return float(np.sqrt(np.sum((got - ref) ** 2)) / (den if den > 0 else 1.0))


def maxrel(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


@dataclasses.dataclass
class Case:
    shape: synth.ModelShape
    w_t: dict            # plain weights (torch, CPU, storage dtype)
    w_np: dict           # the same as float64 numpy (oracle side)
    prefix: np.ndarray
    chunks: list         # per pool entry token ids
    pool_k: torch.Tensor  # [L][rows][hkv][d] storage dtype (CPU)
    pool_v: torch.Tensor
    entry_row: list
    entries_k: list      # per entry float64 [L][P+L_c][hkv][d] (oracle side)
    entries_v: list


def make_case(shape: synth.ModelShape, P: int, lens, seed: int = 0, pool: str = "oracle",
              pool_std: float = 1.0) -> Case:
    w_t = synth.model_weights(shape, seed)
    w_np = {k: f64(v) for k, v in w_t.items()}
    g = torch.Generator().manual_seed(10 + seed)
    prefix = synth.token_ids(P, shape.vocab, g).numpy()
    chunks = [synth.token_ids(lc, shape.vocab, g).numpy() for lc in lens]
    dt = synth.torch_dtype(shape)
    if pool == "oracle":
        cfg = oracle_cfg(shape)
        ks, vs = [], []
        for c in chunks:
            k, v = O.precompute_chunk(w_np, cfg, prefix, c)
            ks.append(torch.from_numpy(k).to(dt))
            vs.append(torch.from_numpy(v).to(dt))
        pool_k = torch.cat(ks, dim=1)
        pool_v = torch.cat(vs, dim=1)
    else:
        pool_k, pool_v, _ = synth.random_pool_kv(shape, P, list(lens), seed, std=pool_std)
    rows = [P + lc for lc in lens]
    entry_row = [int(sum(rows[:i])) for i in range(len(rows))]
    entries_k = [f64(pool_k[:, r:r + n]) for r, n in zip(entry_row, rows)]
    entries_v = [f64(pool_v[:, r:r + n]) for r, n in zip(entry_row, rows)]
    return Case(shape, w_t, w_np, prefix, chunks, pool_k, pool_v, entry_row, entries_k, entries_v)


class GpuRunner:
    """A libblend handle on cuda:0 for one case."""

    def __init__(self, case: Case, max_rows: int, max_tokens: int, max_chunk_rows: int, max_batch: int = 1,
                 max_pos: int = 0, tensor_cores: bool = True):
        self.case = case
        dev = torch.device("cuda:0")
        self.dev = dev
        sh = case.shape
        self.packed = b.pack_weights({k: v.to(dev) for k, v in case.w_t.items()})
        self.cfg = b.model_cfg(sh, max_pos or max_tokens)
        self.lim = b.Limits(max_rows, max_tokens, max_chunk_rows, max_batch)
        self.h = b.blend_init(self.cfg, self.packed, self.lim)
        b.blend_set_tensor_cores(self.h, tensor_cores)
        tok = np.concatenate([np.concatenate([case.prefix, c]) for c in case.chunks]).astype(np.int32)
        self.pool = b.PoolRef(case.pool_k.to(dev), case.pool_v.to(dev), torch.from_numpy(tok).to(dev),
                              len(case.prefix), [len(c) for c in case.chunks], case.entry_row)

    def outputs(self, n_tokens: int, n_q: int, n_c: int):
        sh = self.case.shape
        dt = synth.torch_dtype(sh)
        d = self.dev
        L = sh.n_layers
        return b.OutputsRef(
            k=torch.zeros(L, n_tokens, sh.n_kv_heads, sh.head_dim, dtype=dt, device=d),
            v=torch.zeros(L, n_tokens, sh.n_kv_heads, sh.head_dim, dtype=dt, device=d),
            hidden=torch.zeros(n_q, sh.hidden, dtype=dt, device=d),
            sel=torch.full((n_c,), -1, dtype=torch.int32, device=d),
            n_sel=torch.zeros(b.MAX_BATCH, dtype=torch.int32, device=d),
            c1=torch.full((n_c,), -1, dtype=torch.int32, device=d),
            n_c1=torch.zeros(b.MAX_BATCH, dtype=torch.int32, device=d),
            dev1=torch.zeros(n_c, dtype=torch.float32, device=d),
            dev2=torch.zeros(n_c, dtype=torch.float32, device=d))

    def prefill(self, reqs, n_tokens, n_q, n_c):
        out = self.outputs(n_tokens, n_q, n_c)
        b.blend_prefill(self.h, reqs, self.pool, out)
        b.blend_device_status(self.h)
        return out


def run_oracle(case: Case, chunk_ids, query, **kw):
    return O.blend_prefill(case.w_np, oracle_cfg(case.shape), case.entries_k, case.entries_v, case.chunks,
                           case.prefix, chunk_ids, query, **kw)


def stages_to_device(stages, dev):
    return [(int(f), torch.as_tensor(np.asarray(p, dtype=np.int32), device=dev)) for f, p in stages]


def set_diff_is_near_tie(got, want, score, k, rel=1e-3) -> bool:
    """Two top-k sets over `score` may differ only at positions whose score sits within
    rel * max|score| of the k-th largest score (rounding decides near-ties)."""
    got, want = set(got), set(want)
    if got == want:
        return True
    s = np.asarray(score, dtype=np.float64)
    kth = np.sort(s)[::-1][k - 1]
    tol = rel * np.max(np.abs(s))
    return all(abs(s[p] - kth) <= tol for p in got ^ want)


class LayerwiseF64:
    """A stacked torch weight ([layer][...] or [vocab][H]) that the oracle reads one slice
    at a time as float64, so a full-depth model never needs a float64 copy of every
    layer at once.  Indexing converts only the requested rows or layer."""

    def __init__(self, t: torch.Tensor):
        self.t = t

    def __getitem__(self, i):
        if isinstance(i, np.ndarray):
            i = torch.from_numpy(i.astype(np.int64)).to(self.t.device)
        return f64(self.t[i])

    @property
    def shape(self):
        return tuple(self.t.shape)


def layerwise_weights(w: dict) -> dict:
    """Oracle view of model_weights(): every stacked tensor converted on access; the
    final norm gain (one vector) as float64."""
    return {k: (f64(v) if k == "final_norm" else LayerwiseF64(v)) for k, v in w.items()}


def per_layer_errors(got_k, got_v, ref_k, ref_v):
    """Per layer: (2-norm relative, max-norm relative) of K and of V; got_* are device
    tensors [L][N][hkv][d], converted one layer at a time (or float64 arrays)."""
    rows = []
    conv = lambda t: t if isinstance(t, np.ndarray) else f64(t)
    for l in range(ref_k.shape[0]):
        gk, gv = conv(got_k[l]), conv(got_v[l])
        rows.append((relerr(gk, ref_k[l]), maxrel(gk, ref_k[l]), relerr(gv, ref_v[l]), maxrel(gv, ref_v[l])))
    return rows


def assert_hkvd_sets_replay(out, P, n_c, r1_bp, rho_bp, window, tau, budget_mode, r=0):
    """The GPU's HKVD stage sets of request r (chunk rows r*n_c.. of the outputs) equal the
    oracle's top-k and selection run on the GPU's own deviation arrays, bit for bit: C1 =
    topk(dev1, ceil(r1 N_c)), S = select(dev2 over C1) within C1.  Returns (c1, sel) as
    absolute positions."""
    c0 = r * n_c
    n1, ns = int(out["n_c1"][r].item()), int(out["n_sel"][r].item())
    c1 = out["c1"][c0:c0 + n1].cpu().numpy().astype(np.int64)
    sel = out["sel"][c0:c0 + ns].cpu().numpy().astype(np.int64)
    d1 = f64(out["dev1"][c0:c0 + n_c])
    d2 = f64(out["dev2"][c0:c0 + n_c])
    assert n1 == O.ceil_bp(r1_bp, n_c)
    assert c1.tolist() == sorted(P + t for t in O.topk(d1, n1))
    allowed = np.zeros(n_c, dtype=bool)
    allowed[c1 - P] = True
    assert np.all(d2[~allowed] == 0)
    budget = O.ceil_bp(rho_bp, n_c)
    ds = np.where(allowed, d2, -np.inf)
    want = (O.select(ds, budget, window, tau, "candidate", allowed=allowed, base=P) if budget_mode == "candidate"
            else O.select_final_bisect(ds, budget, window, tau, allowed=allowed, base=P))
    assert sel.tolist() == want.tolist()
    return c1, sel
