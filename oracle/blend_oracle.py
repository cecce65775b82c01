"""CPU oracle for blended (selective KV-recompute) RAG prefill.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module: only
the tests, the smoke check of the package entry script and the CPU-baseline leg
of the benchmark do.  It shares no code with the CUDA path.

Plain numpy in float64, written to be read against the pages rather than to be
fast.  Matrix products use numpy's matmul (a library primitive); everything else
is written out step by step.  Where the pages are silent, the reading taken is
stated next to the function.

Sources (page title, section):
  * CacheClip blog, "6.1 Shared prefix and position IDs", "6.2 Auxiliary-model-guided
    token selection" (steps 1-6 and the column-mean formula), "6.3 Sliding-window grouping"
    (with Figure 6 and its rule list).
  * CacheClip paper (arXiv 2510.10129), "4.1 KV Cache Calibration with Shared Prefix",
    "4.3 Sliding-Window Grouping and KV Cache Update".
  * CacheBlend blog, "Prefill and the KV cache", "Selective KV recompute",
    "Picking the tokens to recompute", "The chicken-and-egg problem", "Implementation".
  * SpecCache notes, "2.2 Importance score estimation" (the I_i formula and TopK with
    K = ceil(rho N)), "2.3 Semantic span completion" (span segmentation, coverage,
    global budget control) and "2.4 Cross-tokenizer alignment".

Parity pins (what each function is checked against, in tests/test_oracle_*.py):
  rope / realign      : rotation composition R(d)R(p)x = R(p+d)x, identity at 0, closed
                        form on basis vectors, relative-position invariance of q.k
  rmsnorm / silu      : closed forms on constant vectors
  layer_rest /        : closed forms with chosen weights: wo = wd = 0 is the identity; a zero
  layer_kv deviation    query adds the mean value row through a permuted wo; one-hot SwiGLU
                        weights add silu(gate) * up on one column; zero K/V projections
                        against constant caches give hkv*d*(cK^2 + cV^2) (V only in V mode)
  attention           : row-by-row brute force over several row blocks; single key -> that value row; two keys -> closed-form softmax
                        weights with the 1/sqrt(d) scale; GQA with duplicated K/V heads
                        equals MHA; causal mask by brute force
  full_prefill        : causality (a prefix of the input gives the same rows)
  assemble            : prefix kept once, chunk rows are the realigned pool rows
  select              : the Figure 6 worked case (tests/golden), brute force over all
                        candidate subsets on tiny inputs, monotonicity in the budget
  blend_prefill       : rho=100 % equals full prefill; rho=0 leaves every chunk row at its
                        realigned cache value; chunk 0 (shift 0) has zero layer-0 deviation
  importance_scores   : closed form on constant hidden states
  round_bf16 /        : closed-form halfway and exponent cases, torch's float32 -> bfloat16
  operand_round         conversion on 200 000 values; the mode's outputs are bf16 values,
                        its residual stream is exact (only used to measure the floor of
                        bf16 arithmetic, never as the parity reference)
  span_segments /     : a hand-worked case (tests/golden/span_completion.json), closed-form
  span_complete /       span lengths on a smooth ramp, invariants (T_init inside T, every
  span_select           covered span complete, nothing else added), degenerate thresholds,
                        budget cap and final-budget maximality
  align_expand        : identity alignment, one-to-two splits, overlapping ranges
  ratio_controller /  : hand-computed delays (matching ratio, the floor, the 100 % cap); the
  pick_storage          cheapest device that hides the load, none when no device does
  attention_probs /   : uniform weights for a zero query, the two-key logistic closed form,
  column_mean_scores /  rows summing to one with zeros past the causal limit; a zero query
  aux_attention_scores  projection gives closed-form column means; the query rows' final
                        state equals blend_prefill on the same single-chunk request
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------------
# bf16 operand rounding (used only to measure the floor of bf16 arithmetic)
# ----------------------------------------------------------------------------------

def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value, ties to even: 8 significant bits (one
    implicit, seven stored) and the float32 exponent range.  x = m 2^e with
    0.5 <= |m| < 1, so m 2^8 lies in [128, 256) and is rounded to an integer (half to
    even); values below 2^-126 keep 8 significant bits instead of bf16's subnormal
    spacing (they do not occur in the models here)."""
    m, e = np.frexp(np.asarray(x, dtype=F64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def _rnd(x, operand_round):
    """x unchanged, or rounded to bf16 when operand_round == "bf16"."""
    if operand_round is None:
        return x
    if operand_round == "bf16":
        return round_bf16(x)
    raise ValueError(operand_round)


# ----------------------------------------------------------------------------------
# Rotary position embedding and KV realignment
# ----------------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2i/d) for i = 0..d/2-1 (rotary embedding frequencies).

    Reading: the pages only say RoPE (CacheBlend blog, "Selective KV recompute", the
    footnote on positional correctness); we take the rotate-half pairing (i, i+d/2).
    """
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * i / head_dim)


def rope_rotate(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate every head vector of x[..., n, heads, d] by the angle pos[n] * inv_freq.

    Pair (i, i+d/2) is rotated by angle a: (x_i cos a - x_{i+d/2} sin a,
    x_{i+d/2} cos a + x_i sin a).  pos may be any integer (negative allowed).
    """
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, dtype=F64)[:, None] * rope_inv_freq(d, theta)[None, :]   # [n, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1 = x[..., :h]
    x2 = x[..., h:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def realign_keys(k_cached: np.ndarray, delta: np.ndarray, theta: float) -> np.ndarray:
    """Move cached keys by delta positions: one more rotation by delta * inv_freq.

    Cached keys were rotated at their precompute position p; RoPE rotations compose,
    so rotating by delta gives the key at p + delta (CacheBlend blog, "Selective KV
    recompute", positional-correctness footnote; CacheClip "Position ID rearrangement").
    """
    return rope_rotate(k_cached, delta, theta)


# ----------------------------------------------------------------------------------
# Decoder layer pieces
# ----------------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=F64)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def attention(q: np.ndarray, qpos: np.ndarray, K: np.ndarray, V: np.ndarray,
              operand_round: Optional[str] = None) -> np.ndarray:
    """Causal grouped-query attention of a set of query rows over a full KV.

    q[n, hq, d] at positions qpos[n]; K, V [N, hkv, d] indexed by position.  Query
    head h reads KV head h // (hq/hkv).  Row i attends keys 0..qpos[i] inclusive with
    softmax(q.k / sqrt(d)).  Each row is complete even though only a few rows are
    computed (CacheBlend blog, "Selective KV recompute": expand K and V back to full
    length, then run ordinary attention).

    Written as the textbook masked softmax: for each KV head and a block of query rows,
    all logits against keys 0..max(qpos) of the block, the keys past a row's own
    position set to -inf, the row maximum subtracted, exponentiated, normalised and
    multiplied by V.  Blocks only bound the size of the logit array; every row is
    computed on its own.  With operand_round the exponentials are rounded before their
    product with V (the normalising sum is taken on the unrounded ones).
    """
    n, hq, d = q.shape
    hkv = K.shape[1]
    group = hq // hkv
    out = np.zeros((n, hq, d), dtype=F64)
    scale = 1.0 / math.sqrt(d)
    qpos = np.asarray(qpos, dtype=np.int64)
    block = 256
    Ks = [np.ascontiguousarray(K[:, g, :], dtype=F64) for g in range(hkv)]   # [N, d] per kv head
    Vs = [np.ascontiguousarray(V[:, g, :], dtype=F64) for g in range(hkv)]

    def piece(g, i0):
        heads = slice(g * group, (g + 1) * group)               # query heads of kv head g
        i1 = min(n, i0 + block)
        b = i1 - i0
        top = int(qpos[i0:i1].max()) + 1                       # keys any row of the block sees
        qb = np.asarray(q[i0:i1, heads, :], dtype=F64).reshape(b * group, d)
        s = ((qb @ Ks[g][:top].T) * scale).reshape(b, group, top)
        # keys after the row's own position: -inf
        for r in range(b):
            s[r, :, int(qpos[i0 + r]) + 1:] = -np.inf
        s -= np.max(s, axis=2, keepdims=True)
        e = np.exp(s, out=s)
        pv = (_rnd(e, operand_round).reshape(b * group, top) @ Vs[g][:top]).reshape(b, group, d)
        out[i0:i1, heads, :] = pv / np.sum(e, axis=2, keepdims=True)

    # the (kv head, row block) pieces are independent and write disjoint parts of out; large
    # ones run four at a time (numpy releases the interpreter lock on large arrays), which
    # changes nothing in the arithmetic of any piece
    tasks = [(g, i0) for g in range(hkv) for i0 in range(0, n, block)]
    if len(tasks) > 1 and n * K.shape[0] >= (1 << 22):
        with ThreadPoolExecutor(max_workers=4) as ex:
            list(ex.map(lambda t: piece(*t), tasks))
    else:
        for t in tasks:
            piece(*t)
    return out


def attention_probs(q: np.ndarray, qpos: np.ndarray, K: np.ndarray) -> np.ndarray:
    """The attention weights behind attention(): P[n, hq, N] with P[i, h, j] =
    softmax_j(q_i,h . K_j,g / sqrt(d)) over keys j <= qpos[i] (g = h // (hq/hkv)), and 0 for
    j > qpos[i]."""
    n, hq, d = q.shape
    N, hkv = K.shape[0], K.shape[1]
    group = hq // hkv
    out = np.zeros((n, hq, N), dtype=F64)
    scale = 1.0 / math.sqrt(d)
    for i in range(n):
        p = int(qpos[i])
        for h in range(hq):
            s = (K[:p + 1, h // group, :] @ q[i, h, :]) * scale
            e = np.exp(s - np.max(s))
            out[i, h, :p + 1] = e / np.sum(e)
    return out


def layer_kv(w: dict, cfg: dict, layer: int, x: np.ndarray, pos: np.ndarray,
             K: np.ndarray, V: np.ndarray, dev_rows: Optional[np.ndarray] = None,
             dev_mode: str = "kv", operand_round: Optional[str] = None):
    """First half of a pre-norm decoder layer on the rows x[n, H] at positions pos[n]:
    RMSNorm, Q/K/V projection, RoPE at the blended positions, and the overwrite of this
    layer's cache rows K[pos], V[pos] with the fresh keys and values.

    These are the first steps of selective recompute (CacheBlend blog, "Selective KV
    recompute"): the layer input is already reduced to the selected rows; they are
    projected to Q, K, V; K and V are expanded back to full length with the reused
    rows of the other tokens.

    If dev_rows (bool[n]) is given, the KV deviation of those rows is returned: the
    squared L2 distance between the fresh and the cached K and V rows at the same
    position, taken before the overwrite (CacheBlend blog, "Selective KV recompute":
    how far the cached KV sits from the recomputed one; "Implementation": the largest
    deviation between newly computed and loaded KV).  dev_mode "v" compares V only
    (CacheClip paper, "Related work": CacheBlend compares the value matrix).
    operand_round "bf16" rounds the normalised rows, q and the fresh k, v (after the
    deviation, before the overwrite) to bf16: the operands of bf16 matrix products and
    the cache's storage type (used only to measure the floor of bf16 arithmetic).
    Returns q [n, hq, d] and dev [n] (or None).
    """
    hq, hkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["rms_eps"], cfg["rope_theta"]
    n = x.shape[0]
    h = _rnd(rmsnorm(x, w["attn_norm"][layer], eps), operand_round)
    q = (h @ w["wq"][layer].T).reshape(n, hq, d)
    k = (h @ w["wk"][layer].T).reshape(n, hkv, d)
    v = (h @ w["wv"][layer].T).reshape(n, hkv, d)
    q = rope_rotate(q, pos, theta)
    k = rope_rotate(k, pos, theta)
    dev = None
    if dev_rows is not None:
        dk = (k - K[pos]).reshape(n, -1)
        dv = (v - V[pos]).reshape(n, -1)
        full = np.sum(dv * dv, axis=1)
        if dev_mode == "kv":
            full = full + np.sum(dk * dk, axis=1)
        dev = np.where(dev_rows, full, 0.0)
    K[pos] = _rnd(k, operand_round)
    V[pos] = _rnd(v, operand_round)
    return _rnd(q, operand_round), dev


def layer_rest(w: dict, cfg: dict, layer: int, x: np.ndarray, q: np.ndarray, pos: np.ndarray,
               K: np.ndarray, V: np.ndarray, operand_round: Optional[str] = None) -> np.ndarray:
    """Second half of the layer for the rows that continue: causal attention of their
    queries over this layer's full K, V, O-projection and residual, RMSNorm, SwiGLU MLP
    and residual ("run the ordinary attention module to get the next layer's input").
    operand_round "bf16" rounds the operands of the products (attention weights, the
    attention output, the normalised rows, the SwiGLU output) to bf16; the residual
    stream stays exact."""
    hq, d = cfg["n_q_heads"], cfg["head_dim"]
    eps = cfg["rms_eps"]
    n = x.shape[0]
    o = _rnd(attention(q, pos, K, V, operand_round).reshape(n, hq * d), operand_round)
    x = np.asarray(x, dtype=F64) + o @ w["wo"][layer].T
    h2 = _rnd(rmsnorm(x, w["mlp_norm"][layer], eps), operand_round)
    hmlp = _rnd(silu(h2 @ w["wg"][layer].T) * (h2 @ w["wu"][layer].T), operand_round)
    return x + hmlp @ w["wd"][layer].T


def layer_forward(w: dict, cfg: dict, layer: int, x: np.ndarray, pos: np.ndarray,
                  K: np.ndarray, V: np.ndarray, dev_rows: Optional[np.ndarray] = None,
                  dev_mode: str = "kv"):
    """A whole decoder layer on rows x at positions pos (layer_kv then layer_rest)."""
    q, dev = layer_kv(w, cfg, layer, x, pos, K, V, dev_rows, dev_mode)
    return layer_rest(w, cfg, layer, x, q, pos, K, V), dev


def full_prefill(w: dict, cfg: dict, tokens: np.ndarray):
    """Standard causal prefill of every token (the quality reference, CacheBlend blog,
    "Prefill and the KV cache").  Returns final-norm hidden rows, K, V [L, N, hkv, d]."""
    N = len(tokens)
    L, hkv, d = cfg["n_layers"], cfg["n_kv_heads"], cfg["head_dim"]
    K = np.zeros((L, N, hkv, d), dtype=F64)
    V = np.zeros((L, N, hkv, d), dtype=F64)
    pos = np.arange(N)
    x = np.asarray(w["embed"][np.asarray(tokens)], dtype=F64)
    for layer in range(L):
        x, _ = layer_forward(w, cfg, layer, x, pos, K[layer], V[layer])
    return rmsnorm(x, w["final_norm"], cfg["rms_eps"]), K, V


def precompute_chunk(w: dict, cfg: dict, prefix_tokens, chunk_tokens):
    """Offline encoding of [shared prefix + chunk] at positions 0..P+L-1 (CacheClip
    "4.1 KV Cache Calibration with Shared Prefix").  Returns K, V [L, P+L, hkv, d]."""
    toks = np.concatenate([np.asarray(prefix_tokens), np.asarray(chunk_tokens)])
    _, K, V = full_prefill(w, cfg, toks)
    return K, V


# ----------------------------------------------------------------------------------
# Cache preparation
# ----------------------------------------------------------------------------------

def assemble(entries_k, entries_v, chunk_ids, prefix_len: int, chunk_lens, query_len: int,
             theta: float):
    """Concatenate the retrieved chunk caches behind one prefix copy and realign keys.

    entries_k[c], entries_v[c]: [L, P+L_c, hkv, d] of pool entry c (each holds its own
    prefix copy).  Only the first chunk's prefix rows are kept (CacheClip "6.1 Shared
    prefix and position IDs", steps 2-3).  Chunk j, precomputed at positions P..P+L_j-1,
    moves to P+off_j..P+off_j+L_j-1 with off_j = sum of earlier chunk lengths, so its keys
    are rotated by delta = off_j and its values copied (step 4; CacheClip "Position ID
    rearrangement").  Query rows are left zero: they are always recomputed.
    Returns K, V [L, N, hkv, d] with N = P + sum(L_j) + Q.
    """
    P = prefix_len
    first = chunk_ids[0]
    L, _, hkv, d = entries_k[first].shape
    n_c = int(sum(chunk_lens))
    N = P + n_c + query_len
    K = np.zeros((L, N, hkv, d), dtype=F64)
    V = np.zeros((L, N, hkv, d), dtype=F64)
    K[:, :P] = entries_k[first][:, :P]
    V[:, :P] = entries_v[first][:, :P]
    off = 0
    for c, lc in zip(chunk_ids, chunk_lens):
        src_k = np.asarray(entries_k[c], dtype=F64)[:, P:P + lc]
        src_v = np.asarray(entries_v[c], dtype=F64)[:, P:P + lc]
        delta = np.full(lc, off)
        for layer in range(L):
            K[layer, P + off:P + off + lc] = realign_keys(src_k[layer], delta, theta)
        V[:, P + off:P + off + lc] = src_v
        off += lc
    return K, V


# ----------------------------------------------------------------------------------
# Token selection
# ----------------------------------------------------------------------------------

def _order_key(score: float, t: int):
    """Candidates are ranked by score (descending), ties by position (ascending).
    -0.0 counts as +0.0; NaN ranks below every number (reading: pages are silent)."""
    s = float(score)
    if math.isnan(s):
        return (1, 0.0, t)
    if s == 0.0:
        s = 0.0
    return (0, -s, t)


def topk(scores: np.ndarray, k: int, allowed: Optional[np.ndarray] = None) -> list:
    """Positions of the k highest scores among the allowed ones (SpecCache 2.2,
    TopK(I, K); CacheClip 6.2 step 6), ranked as in _order_key."""
    n = len(scores)
    idx = [t for t in range(n) if allowed is None or allowed[t]]
    idx.sort(key=lambda t: _order_key(scores[t], t))
    return idx[:max(0, min(k, len(idx)))]


def group_windows(candidates, n: int, w: int, tau: int) -> set:
    """CacheClip sliding-window grouping (blog "6.3 Sliding-window grouping", the rule
    list and Figure 6; paper 4.3).  Scan window starts t = 0..n-w with step 1; a window
    [t, t+w) is evaluated only if t is a candidate; if it holds at least tau candidates
    every position in it joins the recompute set, gaps included.  Candidates not covered
    by a passing window are dropped."""
    cand = set(candidates)
    out = set()
    for t in range(n - w + 1):
        if t not in cand:
            continue
        density = 0
        for j in range(t, t + w):
            if j in cand:
                density += 1
        if density >= tau:
            out.update(range(t, t + w))
    return out


def select(scores: np.ndarray, budget: int, w: int, tau: int, budget_mode: str = "final",
           allowed: Optional[np.ndarray] = None, base: int = 0) -> np.ndarray:
    """Recompute set from per-token scores over the chunk region (positions base..base+n-1).

    candidate mode: the top-`budget` scores are the candidates, grouped as above (the
      CacheClip pseudocode literally: k = ratio x N candidates).
    final mode: the largest k <= budget whose grouped set has at most `budget` rows, so
      the ratio bounds the rows actually recomputed (CacheBlend: recomputing r % of the
      tokens costs about r % of a prefill; SpecCache 2.3: a global budget after span
      completion).  The grouped set grows with k, so the first k found scanning down
      from the budget is the largest.
    allowed (bool[n]): only these positions may be candidates or be returned (gradual
      filtering never adds a token outside the previous stage's set).
    Returns sorted absolute positions (int64).
    """
    n = len(scores)

    def grouped(k):
        s = group_windows(topk(scores, k, allowed), n, w, tau)
        if allowed is not None:
            s = {t for t in s if allowed[t]}
        return s

    if budget_mode == "candidate":
        res = grouped(budget)
    elif budget_mode == "final":
        res = set()
        k = budget
        while k > 0:
            s = grouped(k)
            if len(s) <= budget:
                res = s
                break
            k -= 1
    else:
        raise ValueError(budget_mode)
    return np.array(sorted(base + t for t in res), dtype=np.int64)


def select_final_bisect(scores, budget, w, tau, allowed=None, base=0) -> np.ndarray:
    """Same result as select(..., 'final') using bisection on k (the grouped set grows
    with k), for sizes where the linear scan is slow."""
    n = len(scores)
    order = topk(scores, n, allowed)
    n_ok = len(order)

    def grouped(k):
        s = group_windows(order[:k], n, w, tau)
        if allowed is not None:
            s = {t for t in s if allowed[t]}
        return s

    lo, hi = 0, min(budget, n_ok)          # invariant: |grouped(lo)| <= budget
    if len(grouped(hi)) <= budget:
        lo = hi
    else:
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if len(grouped(mid)) <= budget:
                lo = mid
            else:
                hi = mid
    return np.array(sorted(base + t for t in grouped(lo)), dtype=np.int64)


# ----------------------------------------------------------------------------------
# SpecCache semantic span completion (SpecCache notes, "2.3 Semantic span completion")
# and cross-tokenizer alignment ("2.4 Cross-tokenizer alignment")
# ----------------------------------------------------------------------------------

F32 = np.float32


def span_segments(scores: np.ndarray, tau_smooth: float, max_span: int) -> list:
    """Spans [u, v] (inclusive) of SpecCache 2.3, left to right.

    Scores are min-max normalised, I~_i = (I_i - min I) / (max I - min I); the relative
    change to the next token is delta_i = |I~_{i+1} - I~_i| / I~_i, and token i+1 joins
    the span of token i while delta_i < tau_smooth, up to max_span tokens per span.
    Readings (the pages are silent): every step is one fp32 operation rounded to
    nearest (the scores are fp32), so a GPU kernel can take each merge decision
    identically; -0 counts as +0; min and max skip NaN; a NaN or infinite delta
    (I~_i = 0, or all scores equal) is not below the threshold, so it ends the span;
    a span that reaches max_span tokens ends there and the next token starts a new one.
    """
    x = np.asarray(scores, dtype=F32).copy()
    x[x == 0] = F32(0.0)
    n = len(x)
    if n == 0:
        return []
    finite = x[~np.isnan(x)]
    lo = F32(np.min(finite)) if len(finite) else F32(np.nan)
    hi = F32(np.max(finite)) if len(finite) else F32(np.nan)
    rng = F32(hi - lo)
    with np.errstate(divide="ignore", invalid="ignore"):
        norm = [F32(F32(x[i] - lo) / rng) for i in range(n)]
        spans = []
        u = 0
        for i in range(n - 1):
            delta = F32(F32(abs(F32(norm[i + 1] - norm[i]))) / norm[i])
            merge = bool(delta < F32(tau_smooth))
            if not merge or (i + 1 - u) >= max_span:
                spans.append((u, i))
                u = i + 1
        spans.append((u, n - 1))
    return spans


def span_complete(scores: np.ndarray, k: int, tau_smooth: float, tau_cover_bp: int, max_span: int) -> set:
    """T = T_init U (every span p_j with coverage r_j >= tau_cover), SpecCache 2.3, with
    T_init = the top-k scores (2.2; ranked as in _order_key).  The coverage test
    |T_init n p_j| / |p_j| >= tau_cover is taken exactly in integers with tau_cover in
    basis points: count * 10000 >= tau_cover_bp * |p_j|."""
    init = set(topk(scores, k))
    out = set(init)
    for u, v in span_segments(scores, tau_smooth, max_span):
        members = range(u, v + 1)
        count = sum(1 for t in members if t in init)
        if count * 10000 >= tau_cover_bp * (v - u + 1):
            out.update(members)
    return out


def span_select(scores: np.ndarray, budget: int, tau_smooth: float, tau_cover_bp: int, max_span: int,
                budget_mode: str = "final", cap: Optional[int] = None, base: int = 0) -> np.ndarray:
    """SpecCache selection with its global budget control (2.3, last paragraph).

    candidate mode: T_init = top-`budget`, spans completed, then if |T| > cap only the
      cap tokens of T with the highest scores are kept (the pages' "maximum size limit";
      reading: a caller-given cap >= budget, since a cap equal to the TopK size would
      undo every completion).
    final mode (reading, as for window grouping): the largest k <= budget whose completed
      set has at most `budget` tokens, so the ratio bounds the rows recomputed; the
      completed set grows with k, so scanning k down from the budget finds it.
    Returns sorted absolute positions (int64)."""
    n = len(scores)
    if budget_mode == "candidate":
        res = span_complete(scores, min(budget, n), tau_smooth, tau_cover_bp, max_span)
        c = budget if cap is None else cap
        if len(res) > c:
            keep = sorted(res, key=lambda t: _order_key(scores[t], t))[:c]
            res = set(keep)
    elif budget_mode == "final":
        res = set()
        k = min(budget, n)
        while k > 0:
            s = span_complete(scores, k, tau_smooth, tau_cover_bp, max_span)
            if len(s) <= budget:
                res = s
                break
            k -= 1
    else:
        raise ValueError(budget_mode)
    return np.array(sorted(base + t for t in res), dtype=np.int64)


def span_select_final_bisect(scores: np.ndarray, budget: int, tau_smooth: float, tau_cover_bp: int,
                             max_span: int, base: int = 0) -> np.ndarray:
    """Same result as span_select(..., 'final') using bisection on k (the completed set
    grows with k), for sizes where the linear scan is slow."""
    n = len(scores)

    def size(k):
        return len(span_complete(scores, k, tau_smooth, tau_cover_bp, max_span))

    lo, hi = 0, min(budget, n)               # invariant: size(lo) <= budget
    if size(hi) <= budget:
        lo = hi
    else:
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if size(mid) <= budget:
                lo = mid
            else:
                hi = mid
    res = span_complete(scores, lo, tau_smooth, tau_cover_bp, max_span)
    return np.array(sorted(base + t for t in res), dtype=np.int64)


def align_expand(selected, a_start, a_end) -> np.ndarray:
    """SpecCache 2.4: T = union over selected speculative tokens i of Psi(i), where
    Psi(i) = target tokens a_start[i] .. a_end[i]-1 (the target sub-tokens covering the
    same text).  Returns the sorted distinct target indices."""
    out = set()
    for i in selected:
        out.update(range(int(a_start[i]), int(a_end[i])))
    return np.array(sorted(out), dtype=np.int64)


def column_mean_scores(q: np.ndarray, qpos: np.ndarray, K: np.ndarray, col_lo: int, col_hi: int) -> np.ndarray:
    """CacheClip blog 6.2, "the scoring step is just a column mean": score(j) = mean over the
    query rows i (and, reading, over the heads) of the attention weight A[i, j], for the
    columns j in [col_lo, col_hi)."""
    probs = attention_probs(q, qpos, K)
    return np.mean(probs[:, :, col_lo:col_hi], axis=(0, 1))


def aux_query_forward(w: dict, cfg: dict, ek, ev, P: int, query_tokens):
    """The auxiliary model on one [prefix + chunk + query] sequence whose prefix and chunk
    rows are its precomputed cache ek, ev [L, P+L_c, hkv, d] (CacheClip blog 6.2 step 2: only
    the query tokens are computed, the chunk side is loaded from cache).  The query rows go
    through every layer at positions P+L_c ..; returns the last layer's query projections
    q [Q, hq, d] (after RoPE) and its keys K [P+L_c+Q, hkv, d] (cache rows, then the query's)."""
    L = cfg["n_layers"]
    Q = len(query_tokens)
    ek, ev = np.asarray(ek, dtype=F64), np.asarray(ev, dtype=F64)
    Lc = ek.shape[1] - P
    K = np.concatenate([ek, np.zeros((L, Q) + ek.shape[2:], dtype=F64)], axis=1)
    V = np.concatenate([ev, np.zeros((L, Q) + ev.shape[2:], dtype=F64)], axis=1)
    pos = np.arange(P + Lc, P + Lc + Q)
    x = np.asarray(w["embed"][np.asarray(query_tokens)], dtype=F64)
    q = None
    for layer in range(L):
        q, _ = layer_kv(w, cfg, layer, x, pos, K[layer], V[layer])
        if layer < L - 1:
            x = layer_rest(w, cfg, layer, x, q, pos, K[layer], V[layer])
    return q, K[L - 1]


def aux_attention_scores(w: dict, cfg: dict, entries_k, entries_v, entry_tokens, prefix_tokens, chunk_ids,
                         query_tokens) -> np.ndarray:
    """Auxiliary-model importance scores (CacheClip blog "6.2 Auxiliary-model-guided token
    selection", steps 1-5; CacheClip paper 4.2).

    For every retrieved chunk c, in request order, the auxiliary model reads [prefix + chunk_c
    + query] (aux_query_forward).  From the last layer's attention the query rows and chunk_c's
    columns are kept (attention among query tokens and to the prefix is dropped after the
    softmax, which covers all of them) and each column is averaged over the query rows and the
    heads (reading: the pages speak of one attention matrix per layer; a multi-head model's is
    taken as the mean over its heads).  Returns the scores of all chunk tokens [sum L_c].
    """
    P = len(prefix_tokens)
    Q = len(query_tokens)
    out = []
    for c in chunk_ids:
        Lc = len(entry_tokens[c])
        q, K = aux_query_forward(w, cfg, entries_k[c], entries_v[c], P, query_tokens)
        out.append(column_mean_scores(q, np.arange(P + Lc, P + Lc + Q), K, P, P + Lc))
    return np.concatenate(out) if out else np.zeros(0, dtype=F64)


# ----------------------------------------------------------------------------------
# CacheBlend loading controller (CacheBlend blog, "Making the recompute free")
# ----------------------------------------------------------------------------------

def ratio_controller(full_prefill_s: float, kv_bytes: float, load_bytes_per_s: float, floor_bp: int) -> int:
    """Recompute delay = rho x (offline-profiled full prefill time); load delay = KV size of
    the context / the device's throughput.  rho is where the two delays are equal, then the
    larger of that and the quality floor (15 % on the pages), at most 100 %.  Returned in
    basis points, rounded up (reading: the pages give no rounding)."""
    load_s = kv_bytes / load_bytes_per_s
    r = math.ceil(10000.0 * (load_s / full_prefill_s))
    return int(min(10000, max(floor_bp, r)))


def pick_storage(full_prefill_s: float, kv_bytes: float, floor_bp: int, bytes_per_s, cost_per_byte) -> int:
    """The estimators run backwards: fix the ratio at the floor, keep the devices on which
    the recompute takes at least as long as the load, and take the cheapest survivor
    (reading: ties go to the first listed).  -1 when none qualifies."""
    budget_s = (floor_bp / 10000.0) * full_prefill_s
    best = -1
    for i, (bw, cost) in enumerate(zip(bytes_per_s, cost_per_byte)):
        if kv_bytes / bw <= budget_s and (best < 0 or cost < cost_per_byte[best]):
            best = i
    return best


def importance_scores(hidden: np.ndarray) -> np.ndarray:
    """SpecCache 2.2: I_i = mean over the deep layers of ||h_i^(l)||_2.
    hidden: [tokens, layers, dim] (the deep-layer slices of a small model)."""
    h = np.asarray(hidden, dtype=F64)
    return np.mean(np.sqrt(np.sum(h * h, axis=-1)), axis=-1)


# ----------------------------------------------------------------------------------
# Blended prefill
# ----------------------------------------------------------------------------------

def epic_positions(prefix_len: int, chunk_lens, m: int) -> np.ndarray:
    """EPIC's static selection (SpecCache notes, background: EPIC recomputes the first few
    tokens of every chunk): blended positions P + off_j + t for t < min(m, L_j)."""
    out, off = [], 0
    for L in chunk_lens:
        out.extend(prefix_len + off + t for t in range(min(m, L)))
        off += L
    return np.array(out, dtype=np.int64)


def focused_chunks(scores: np.ndarray, chunk_lens, focus_bp: int) -> np.ndarray:
    """Cache-Craft notes, 3.2.2 (adaptive early recomputation termination): the query's
    attention identifies focused chunks and recomputation stops for the others.  Readings
    (the notes give no formula): a chunk's question attention is the sum over its tokens of
    the column-mean scores (column_mean_scores at the detection layer); it is focused when
    that share of the total is at least focus_bp basis points."""
    s = np.asarray(scores, dtype=F64)
    mass = np.array([s[a:a + L].sum() for a, L in zip(np.cumsum([0] + list(chunk_lens)[:-1]), chunk_lens)])
    return mass * 10000.0 >= focus_bp * mass.sum()


def ceil_bp(rho_bp: int, n: int) -> int:
    """ceil(rho * n) with rho in basis points (SpecCache 2.2, K = ceil(rho N))."""
    return (rho_bp * n + 9999) // 10000


CHECK_LAYERS = (1, 2)


def blend_prefill(w: dict, cfg: dict, entries_k, entries_v, entry_tokens, prefix_tokens,
                  chunk_ids, query_tokens, mode: str, rho_bp: int = 0, r1_bp: int = 0,
                  window: int = 1, tau: int = 1, budget_mode: str = "final",
                  scores: Optional[np.ndarray] = None, forced: Optional[list] = None,
                  dev_mode: str = "kv", group_rule: str = "window", tau_smooth: float = 0.4,
                  tau_cover_bp: int = 7000, max_span: int = 16, cap_bp: int = 0, epic_m: int = 0,
                  focus_layer: int = 0, focus_bp: int = 0, operand_round: Optional[str] = None):
    """Selective KV-recompute prefill of one request.

    1. Assemble the blended cache (see assemble()).
    2. Run every layer on a set of chunk rows plus the query rows (always recomputed),
       in ascending position order.  The schedule is a list of stages
       (first_layer, positions): from first_layer on, the rows that go through attention
       and the MLP are `positions` + query.  A layer projects K, V for the rows that
       entered it (the previous layer's rows) and writes them into the cache; when a
       new stage starts at that layer, only the new (smaller) set continues.
       * "ext":   one stage [(0, S)] with S = select(scores, ceil(rho N_c), w, tau, mode)
                  from external per-chunk-token scores (CacheClip 6.2-6.3; SpecCache 2.2),
                  or with group_rule "span" S = span_select(...) (SpecCache 2.3; in
                  candidate mode the cap is ceil(cap_bp N_c)).
       * "hkvd":  gradual filtering (CacheBlend blog, "The chicken-and-egg problem"; the
                  CacheClip paper's summary: the first layer is recomputed in full, the
                  second partially, and its fresh KV is compared with the loaded one).
                  Stage 0 = every chunk row.  The first layer's K, V depend only on a
                  token and its realigned position, so it has no deviation to rank; the
                  checks are at layers 1 and 2 (CHECK_LAYERS, counted from 0):
                  layer 1 ranks every chunk row by deviation and keeps the top
                  ceil(r1 N_c) as C1; layer 2 ranks the C1 rows and keeps
                  S = select(dev2 over C1, ceil(rho N_c), w, tau, mode), within C1.
                  The set only shrinks; S is used from layer 2's attention onward.
       * "forced": the caller's stages (deviations are still reported at the check layers).
       * "full":  every row 0..N-1 at every layer (full prefill through the same steps).
       * "epic":  one stage [(0, S)] with S = the first epic_m tokens of every chunk
                  (EPIC's static rule as SpecCache describes it: a fixed number of tokens at
                  the start of each chunk is recomputed, the rest reused).
       With focus_bp > 0 (ext and epic): early termination for unfocused chunks (Cache-Craft
       notes, 3.2.2; see focused_chunks) at focus_layer, after that layer's K/V projection.
    3. Output the final RMSNorm of the query rows and the blended K, V of every layer.

    operand_round None (the reference) computes every step exactly in float64.  "bf16"
    rounds every operand of a matrix product, the cache rows written and the output to
    bf16 (see layer_kv, layer_rest): not a reading of the method but the arithmetic of a
    bf16 tensor-core implementation, run only to measure how far that arithmetic alone
    moves the result away from the exact one.

    Positions in sets are absolute positions in the blended sequence.
    Returns a dict: hidden [Q, H], K, V [L, N, hkv, d], stages, dev1, dev2 ([N_c] each,
    zero outside the rows checked).
    """
    L = cfg["n_layers"]
    P = len(prefix_tokens)
    lens = [len(entry_tokens[c]) for c in chunk_ids]
    n_c = int(sum(lens))
    Q = len(query_tokens)
    N = P + n_c + Q
    K, V = assemble(entries_k, entries_v, chunk_ids, P, lens, Q, cfg["rope_theta"])
    K = _rnd(K, operand_round)          # the realigned keys as a bf16 cache stores them
    tokens = np.concatenate([np.asarray(prefix_tokens)] + [np.asarray(entry_tokens[c]) for c in chunk_ids]
                            + [np.asarray(query_tokens)])
    lo, hi = P, P + n_c
    qrows = np.arange(hi, N)
    budget = ceil_bp(rho_bp, n_c)

    if mode == "ext" and group_rule == "span":
        s = np.asarray(scores)
        sel = (span_select(s, budget, tau_smooth, tau_cover_bp, max_span, "candidate",
                           cap=ceil_bp(cap_bp, n_c), base=lo) if budget_mode == "candidate"
               else span_select_final_bisect(s, budget, tau_smooth, tau_cover_bp, max_span, base=lo))
        stages = [(0, sel)]
    elif mode == "ext":
        s = np.asarray(scores)
        sel = (select(s, budget, window, tau, budget_mode, base=lo) if budget_mode == "candidate"
               else select_final_bisect(s, budget, window, tau, base=lo))
        stages = [(0, sel)]
    elif mode == "hkvd":
        stages = [(0, np.arange(lo, hi))]
    elif mode == "forced":
        stages = [(int(f), np.asarray(p, dtype=np.int64)) for f, p in forced]
    elif mode == "full":
        stages = [(0, np.arange(0, hi))]
    elif mode == "epic":
        stages = [(0, epic_positions(P, lens, epic_m))]
    else:
        raise ValueError(mode)

    def rows_at(layer):
        cur = None
        for f, p in stages:
            if f <= layer:
                cur = p
        return np.concatenate([cur, qrows]).astype(np.int64)

    devs = {}
    rows = rows_at(0)
    x = np.asarray(w["embed"][tokens[rows]], dtype=F64)
    for layer in range(L):
        check = mode in ("hkvd", "forced") and layer in CHECK_LAYERS
        dev_rows = ((rows >= lo) & (rows < hi)) if check else None
        q, dev = layer_kv(w, cfg, layer, x, rows, K[layer], V[layer], dev_rows, dev_mode, operand_round)
        if dev is not None:
            full = np.zeros(n_c, dtype=F64)
            full[rows[dev_rows] - lo] = dev[dev_rows]
            devs[layer] = full
        if focus_bp > 0 and mode in ("ext", "epic") and layer == focus_layer:
            qq = q[len(rows) - Q:]                     # the query rows are the last Q rows
            sc = column_mean_scores(qq, qrows, K[layer], lo, hi)
            keep = focused_chunks(sc, lens, focus_bp)
            starts = np.cumsum([0] + lens[:-1])
            crow = rows[rows < hi]
            chunk_of = np.searchsorted(starts, crow - lo, side="right") - 1
            stages.append((layer, crow[keep[chunk_of]].astype(np.int64)))
        if mode == "hkvd" and layer == CHECK_LAYERS[0]:
            c1 = np.array(sorted(lo + t for t in topk(devs[layer], ceil_bp(r1_bp, n_c))), dtype=np.int64)
            stages.append((layer, c1))
        if mode == "hkvd" and layer == CHECK_LAYERS[1]:
            allowed = np.zeros(n_c, dtype=bool)
            allowed[stages[1][1] - lo] = True
            dscore = np.where(allowed, devs[layer], -np.inf)
            sel = (select(dscore, budget, window, tau, budget_mode, allowed=allowed, base=lo)
                   if budget_mode == "candidate"
                   else select_final_bisect(dscore, budget, window, tau, allowed=allowed, base=lo))
            stages.append((layer, sel))
        new_rows = rows_at(layer)
        if not np.array_equal(new_rows, rows):
            where = {int(p): i for i, p in enumerate(rows)}
            keep = [where[int(p)] for p in new_rows]
            x, q, rows = x[keep], q[keep], new_rows
        x = layer_rest(w, cfg, layer, x, q, rows, K[layer], V[layer], operand_round)
    qi = np.searchsorted(rows, qrows)
    hidden = _rnd(rmsnorm(x[qi], w["final_norm"], cfg["rms_eps"]), operand_round)
    return {"hidden": hidden, "K": K, "V": V, "stages": stages,
            "dev1": devs.get(CHECK_LAYERS[0]), "dev2": devs.get(CHECK_LAYERS[1]),
            "tokens": tokens, "N": N, "n_c": n_c}
