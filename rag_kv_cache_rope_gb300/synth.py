"""Seeded synthetic inputs for blended (selective KV-recompute) prefill.

This module only draws random numbers: model weights, token ids, chunk-pool
contents, chunk-reuse draws and the small-model hidden states that importance
scores are reduced from.  It holds none of the method's arithmetic (no RoPE, no
attention, no selection), so the CUDA path and the CPU oracle can both take
their inputs from here without sharing any computation.

Shapes follow the workloads the pages measure: 4K-16K token RAG contexts built
from 512-token chunks behind one shared prefix (CacheBlend "Results"; SpecCache
"experimental setup"), 15-20 % recompute (CacheClip Table 6; SpecCache
"experimental results"), decoders shaped like Llama-3-8B, Mistral-7B and
Qwen2.5-14B with random weights (no trained checkpoints are available).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-6
    dtype: str = "bf16"          # "f32" or "bf16": storage type of weights / KV / activations
    init: str = "std0.02"        # "fan_in": N(0, 1/fan_in) weights, N(0,1) embeddings

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def params_per_layer(self) -> int:
        h = self.hidden
        return h * (self.q_dim + 2 * self.kv_dim) + self.q_dim * h + 3 * h * self.ffn


TINY = ModelShape("tiny-2L", 2, 256, 4, 2, 64, 688, 1024, 1e4, dtype="f32", init="fan_in")
TINY4 = dataclasses.replace(TINY, name="tiny-4L", n_layers=4)
LLAMA8B = ModelShape("llama3-8b-shape", 32, 4096, 32, 8, 128, 14336, 128256, 5e5)
MISTRAL7B = ModelShape("mistral-7b-shape", 32, 4096, 32, 8, 128, 14336, 32000, 1e6)
QWEN14B = ModelShape("qwen2.5-14b-shape", 48, 5120, 40, 8, 128, 13824, 152064, 1e6)
# CacheClip's auxiliary model (SmolLM2-135M widths: 30 layers, H 576, 9/3 heads of 64)
SMOL135M = ModelShape("smollm2-135m-shape", 30, 576, 9, 3, 64, 1536, 49152, 1e5)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One blended-prefill request shape (or a batch of identical shapes)."""
    name: str
    model: ModelShape
    prefix_len: int
    chunk_len: int
    n_chunks: int
    query_len: int
    mode: str                    # "ext" | "hkvd" | "forced" | "full"
    rho_bp: int                  # recompute ratio of chunk rows, basis points
    r1_bp: int = 0               # HKVD first-stage ratio, basis points
    window: int = 1
    tau: int = 1
    budget_mode: str = "final"   # "final" | "candidate"
    batch: int = 1
    pool_size: int = 0           # >0: chunks are drawn from a pool of this many entries
    zipf_s: float = 0.0
    seed: int = 0
    score_layers: int = 4        # small-model hidden states [tokens, score_layers, score_dim]
    score_dim: int = 2048
    score_phrase_max: int = 0    # >0: hidden-state scales shared within runs of 1..this many tokens
    group_rule: str = "window"   # "window" (CacheClip grouping) | "span" (SpecCache span completion)
    epic_m: int = 0              # mode "epic": tokens recomputed at the start of every chunk
    focus_layer: int = 0         # focus_bp > 0: Cache-Craft early termination at this layer
    focus_bp: int = 0
    aux_model: Optional["ModelShape"] = None  # CacheClip: scores from this auxiliary model

    @property
    def n_ctx(self) -> int:
        return self.prefix_len + self.n_chunks * self.chunk_len + self.query_len

    @property
    def n_chunk_rows(self) -> int:
        return self.n_chunks * self.chunk_len


def ceil_bp(rho_bp: int, n: int) -> int:
    """ceil(rho * n) for a ratio given in basis points, in integer arithmetic."""
    return (rho_bp * n + 9999) // 10000


WORKLOADS = {
    # 2-layer fp32 decoder; HKVD with a 30 % first stage narrowed to 20 %, window 2.
    "tiny-fp32-hkvd": Workload("tiny-fp32-hkvd", TINY, 16, 128, 4, 32, "hkvd", 2000, 3000, 2, 1, seed=0),
    # same shapes, 4 layers, so the narrowed set is used on layers >= 2
    "tiny4-fp32-hkvd": Workload("tiny4-fp32-hkvd", TINY4, 16, 128, 4, 32, "hkvd", 2000, 3000, 2, 1, seed=0),
    # Llama-3-8B shape, 6 x 512 chunks, 15 % by KV deviation with gradual filtering
    "llama8b-3k-hkvd15": Workload("llama8b-3k-hkvd15", LLAMA8B, 32, 512, 6, 64, "hkvd", 1500, 2250, 1, 1, seed=1),
    # Mistral-7B shape, a batch of 8 requests of 8 chunks drawn from a 64-entry pool (Zipf 1.1)
    "mistral7b-b8-ext15": Workload("mistral7b-b8-ext15", MISTRAL7B, 32, 512, 8, 128, "ext", 1500, 0, 1, 1,
                                   batch=8, pool_size=64, zipf_s=1.1, seed=3),
    # Qwen2.5-14B shape, 16K context (64 + 31 x 512 + 128), 20 % with window-4 dilation
    "qwen14b-16k-ext20": Workload("qwen14b-16k-ext20", QWEN14B, 64, 512, 31, 128, "ext", 2000, 0, 4, 1, seed=4),
    # the same request selected by SpecCache span completion (tau_smooth 0.4, tau_cover 0.7,
    # spans <= 16) over scores with phrase structure (runs of 1..8 tokens of similar scale)
    "qwen14b-16k-span20": Workload("qwen14b-16k-span20", QWEN14B, 64, 512, 31, 128, "ext", 2000, 0, 1, 1, seed=4,
                                   score_phrase_max=8, group_rule="span"),
    # the same context with EPIC's static rule: the first 103 tokens (~20 %) of every chunk
    "qwen14b-16k-epic20": Workload("qwen14b-16k-epic20", QWEN14B, 64, 512, 31, 128, "epic", 2000, seed=4,
                                   epic_m=103),
    # the main request plus Cache-Craft early termination: at layer 16 chunks under a 3 %
    # share of the question attention stop being recomputed
    "qwen14b-16k-ext20-focus": Workload("qwen14b-16k-ext20-focus", QWEN14B, 64, 512, 31, 128, "ext", 2000, 0, 4, 1,
                                        seed=4, focus_layer=16, focus_bp=300),
    # CacheClip end to end: scores from the auxiliary model's last-layer attention (one
    # [prefix + chunk + query] sequence per chunk), window 8, density 5, final budget 20 %
    "qwen14b-16k-aux20": Workload("qwen14b-16k-aux20", QWEN14B, 64, 512, 31, 128, "ext", 2000, 0, 8, 5, seed=4,
                                  aux_model=SMOL135M),
}


def sweep_workload(n_chunks: int, rho_bp: int) -> Workload:
    """The 14B-shaped context x ratio sweep: 7/15/31/63 chunks (4K..32K) x 5..100 %."""
    return Workload(f"qwen14b-{n_chunks}c-ext{rho_bp // 100}", QWEN14B, 64, 512, n_chunks, 128, "ext",
                    rho_bp, 0, 4, 1, seed=5)


def torch_dtype(shape: ModelShape) -> torch.dtype:
    return torch.float32 if shape.dtype == "f32" else torch.bfloat16


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, g: torch.Generator, device, dtype) -> torch.Tensor:
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)


def model_weights(shape: ModelShape, seed: int, device="cpu", layers: Optional[int] = None) -> dict:
    """Random decoder weights in the plain (unpacked) layout, rounded to the storage dtype.

    Linear weights are [out_features, in_features].  RMSNorm gains are 1.  With
    init "fan_in" linear weights are N(0, 1/fan_in) and embeddings N(0, 1);
    otherwise every weight and embedding is N(0, 0.02^2).
    """
    L = shape.n_layers if layers is None else layers
    dt = torch_dtype(shape)
    g = _gen(1000 + seed, device)
    H, F, qd, kvd = shape.hidden, shape.ffn, shape.q_dim, shape.kv_dim

    def lin(out_f, in_f):
        std = (1.0 / math.sqrt(in_f)) if shape.init == "fan_in" else 0.02
        return _normal((L, out_f, in_f), std, g, device, dt)

    emb_std = 1.0 if shape.init == "fan_in" else 0.02
    w = {
        "embed": _normal((shape.vocab, H), emb_std, g, device, dt),
        "wq": lin(qd, H),
        "wk": lin(kvd, H),
        "wv": lin(kvd, H),
        "wo": lin(H, qd),
        "wg": lin(F, H),
        "wu": lin(F, H),
        "wd": lin(H, F),
        "attn_norm": torch.ones(L, H, device=device, dtype=dt),
        "mlp_norm": torch.ones(L, H, device=device, dtype=dt),
        "final_norm": torch.ones(H, device=device, dtype=dt),
    }
    return w


def token_ids(n: int, vocab: int, g: torch.Generator) -> torch.Tensor:
    return torch.randint(0, vocab, (n,), generator=g, dtype=torch.int64).to(torch.int32)


@dataclasses.dataclass
class RequestTokens:
    prefix: torch.Tensor            # [P] int32
    chunk_ids: list                 # pool entry of each chunk, in request order
    query: torch.Tensor             # [Q] int32


@dataclasses.dataclass
class PoolTokens:
    prefix: torch.Tensor            # [P] int32, shared by every entry
    chunks: list                    # per entry [L_c] int32


def zipf_draw(pool_size: int, n: int, s: float, g: torch.Generator) -> list:
    """n distinct pool entries drawn without replacement with P(rank r) ~ r^-s, then shuffled."""
    ranks = torch.arange(1, pool_size + 1, dtype=torch.float64)
    p = ranks.pow(-s)
    picked = torch.multinomial(p, n, replacement=False, generator=g).tolist()
    perm = torch.randperm(n, generator=g).tolist()
    return [picked[i] for i in perm]


def workload_tokens(wl: Workload):
    """Token ids of the pool and of each request of a workload (CPU, seeded by the workload)."""
    g = _gen(wl.seed, "cpu")
    vocab = wl.model.vocab
    prefix = token_ids(wl.prefix_len, vocab, g)
    n_entries = wl.pool_size if wl.pool_size else wl.n_chunks * wl.batch
    chunks = [token_ids(wl.chunk_len, vocab, g) for _ in range(n_entries)]
    pool = PoolTokens(prefix, chunks)
    reqs = []
    for r in range(wl.batch):
        if wl.pool_size:
            gr = _gen(wl.seed + r, "cpu")
            ids = zipf_draw(wl.pool_size, wl.n_chunks, wl.zipf_s, gr)
        else:
            ids = list(range(r * wl.n_chunks, (r + 1) * wl.n_chunks))
        query = token_ids(wl.query_len, vocab, g)
        reqs.append(RequestTokens(prefix, ids, query))
    return pool, reqs


def hidden_states(n_tokens: int, n_layers: int, dim: int, seed: int, device="cpu",
                  dtype=torch.float32, phrase_max: int = 0) -> torch.Tensor:
    """Stand-in for a small model's deep-layer hidden states, [tokens, layers, dim].

    Each token gets its own scale (log-normal), so that the per-token norms spread
    out the way importance scores do, plus unit Gaussian directions.  With phrase_max
    > 0 the scale is shared within runs of 1..phrase_max tokens (a stand-in for
    multi-token entities, SpecCache 2.3) with a 3 % per-token jitter.
    """
    g = _gen(2000 + seed, device)
    scale = torch.exp(0.5 * torch.randn(n_tokens, 1, 1, generator=g, device=device))
    if phrase_max > 0:
        gp = _gen(2500 + seed, "cpu")
        lens = torch.randint(1, phrase_max + 1, (n_tokens,), generator=gp)
        run = torch.repeat_interleave(torch.arange(n_tokens), lens)[:n_tokens].to(device)
        jitter = 1.0 + 0.03 * torch.randn(n_tokens, 1, 1, generator=g, device=device)
        scale = scale[run] * jitter
    h = torch.randn(n_tokens, n_layers, dim, generator=g, device=device) * scale
    return h.to(dtype)


def random_pool_kv(shape: ModelShape, prefix_len: int, chunk_lens: list, seed: int, device="cpu",
                   std: float = 1.0):
    """A chunk-KV pool with random contents, [layers][rows][kv_heads][head_dim] for K and V.

    Entries are packed along rows; entry c occupies rows row_off[c] .. row_off[c]+P+L_c.
    Every entry holds the same prefix rows (a deterministic precompute of one shared
    prefix gives identical rows).  Used where precomputing the pool with the oracle
    would take too long; the hot path's cost does not depend on the values.
    """
    dt = torch_dtype(shape)
    g = _gen(3000 + seed, device)
    L, hk, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    P = prefix_len
    rows = [P + lc for lc in chunk_lens]
    row_off = [0]
    for r in rows[:-1]:
        row_off.append(row_off[-1] + r)
    total = sum(rows)
    k = torch.empty(L, total, hk, d, device=device, dtype=dt)
    v = torch.empty(L, total, hk, d, device=device, dtype=dt)
    pk = _normal((L, P, hk, d), std, g, device, dt)
    pv = _normal((L, P, hk, d), std, g, device, dt)
    for c, lc in enumerate(chunk_lens):
        o = row_off[c]
        k[:, o:o + P] = pk
        v[:, o:o + P] = pv
        k[:, o + P:o + P + lc] = _normal((L, lc, hk, d), std, g, device, dt)
        v[:, o + P:o + P + lc] = _normal((L, lc, hk, d), std, g, device, dt)
    return k, v, row_off
