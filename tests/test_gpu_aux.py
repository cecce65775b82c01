"""CacheClip auxiliary-model scoring on the GPU against the oracle (CacheClip blog, "6.2
Auxiliary-model-guided token selection", steps 1-6; CacheClip paper 4.2).

* the column-mean kernel alone: random last-layer q and keys, several requests;
* the whole auxiliary step: blend_prefill on the auxiliary model in FORCED mode with an
  empty stage (only the query rows are computed over each chunk's cached rows) with the
  last-layer q exported, then aux_attention_scores, against the oracle's
  aux_attention_scores; then top-k + window grouping of those scores.
"""
import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import GpuRunner, f64, make_case, maxrel, relerr, set_diff_is_near_tie

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


def _batch(r, case, Q, query, dev):
    """One request per pool entry: [prefix + chunk_c + query], only the query recomputed."""
    empty = torch.zeros(0, dtype=torch.int32, device=dev)
    q = torch.from_numpy(query.astype(np.int32)).to(dev)
    return [b.RequestRef([c], q, mode="forced", stages=[(0, empty)]) for c in range(len(case.chunks))]


def _outputs(sh, lens, P, Q, dev):
    dt = synth.torch_dtype(sh)
    n_req = len(lens)
    N = sum(P + n + Q for n in lens)
    return b.OutputsRef(k=torch.zeros(sh.n_layers, N, sh.n_kv_heads, sh.head_dim, dtype=dt, device=dev),
                        v=torch.zeros(sh.n_layers, N, sh.n_kv_heads, sh.head_dim, dtype=dt, device=dev),
                        hidden=torch.zeros(n_req * Q, sh.hidden, dtype=dt, device=dev),
                        q_last=torch.zeros(n_req * Q, sh.n_q_heads, sh.head_dim, dtype=dt, device=dev))


# (dtype, d, P, chunk lengths, Q): short contexts, then contexts of several 1024-key spans
# per row (the tensor-core statistics pass merges span partials) with more than 128
# (row, head) pairs per kv head
COLMEAN_CASES = [("f32", 64, 7, [40, 95, 33], 12), ("bf16", 64, 7, [40, 95, 33], 12),
                 ("bf16", 128, 7, [40, 95, 33], 12), ("bf16", 128, 64, [2500, 700], 40),
                 ("bf16", 64, 33, [1100, 3000, 9], 50)]


@pytest.mark.parametrize("dtype,d,P,lens,Q", COLMEAN_CASES)
def test_column_mean_kernel_matches_oracle(dtype, d, P, lens, Q):
    hq, hkv = (9, 3) if d == 64 else (8, 2)
    sh = synth.ModelShape("aux-k", 1, hq * d if d == 64 else 1024, hq, hkv, d, 1536, 64, 1e4, dtype=dtype)
    case = make_case(sh, P, lens, pool="random")
    dev = torch.device("cuda:0")
    N = sum(P + n + Q for n in lens)
    r = GpuRunner(case, len(lens) * Q, N, max(lens), max_batch=len(lens), max_pos=N)
    reqs = _batch(r, case, Q, np.zeros(Q, dtype=np.int32), dev)
    out = _outputs(sh, lens, P, Q, dev)
    g = torch.Generator().manual_seed(3)
    dt = synth.torch_dtype(sh)
    k = torch.randn(N, hkv, d, generator=g).to(dt)
    ql = (0.6 * torch.randn(len(lens) * Q, hq, d, generator=g)).to(dt)
    out.t["k"][0].copy_(k.to(dev))
    out.t["q_last"].copy_(ql.to(dev))
    scores = torch.full((sum(lens),), -1.0, device=dev)
    b.aux_attention_scores(r.h, reqs, r.pool, out, scores)
    b.blend_device_status(r.h)
    got = scores.cpu().numpy().astype(np.float64)
    want, tok = [], 0
    for i, n in enumerate(lens):
        Kr = f64(k[tok:tok + P + n + Q])
        qr = f64(ql[i * Q:(i + 1) * Q])
        want.append(O.column_mean_scores(qr, np.arange(P + n, P + n + Q), Kr, P, P + n))
        tok += P + n + Q
    want = np.concatenate(want)
    assert maxrel(got, want) <= 1e-5
    # deterministic: a second call gives the same bits
    s2 = torch.zeros_like(scores)
    b.aux_attention_scores(r.h, reqs, r.pool, out, s2)
    torch.cuda.synchronize()
    assert torch.equal(scores, s2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_aux_pipeline_matches_oracle(dtype):
    """SmolLM2-135M-shaped auxiliary model (H 576, 9/3 heads, d 64, F 1536), 2 layers: query
    rows over each chunk's cached rows, scores of every chunk token."""
    sh = synth.ModelShape("aux-smol", 2, 576, 9, 3, 64, 1536, 300, 1e5, dtype=dtype,
                          init="fan_in" if dtype == "f32" else "std0.02")
    P, lens, Q = 8, [64, 48, 80, 64], 16
    case = make_case(sh, P, lens, seed=4)
    dev = torch.device("cuda:0")
    N = sum(P + n + Q for n in lens)
    r = GpuRunner(case, len(lens) * Q, N, max(lens), max_batch=len(lens), max_pos=N)
    g = torch.Generator().manual_seed(6)
    query = synth.token_ids(Q, sh.vocab, g).numpy()
    reqs = _batch(r, case, Q, query, dev)
    out = _outputs(sh, lens, P, Q, dev)
    b.blend_prefill(r.h, reqs, r.pool, out)
    scores = torch.zeros(sum(lens), device=dev)
    b.aux_attention_scores(r.h, reqs, r.pool, out, scores)
    b.blend_device_status(r.h)
    got = scores.cpu().numpy().astype(np.float64)
    want = O.aux_attention_scores(case.w_np, dict(n_layers=sh.n_layers, hidden=sh.hidden, n_q_heads=sh.n_q_heads,
                                                  n_kv_heads=sh.n_kv_heads, head_dim=sh.head_dim, ffn=sh.ffn,
                                                  vocab=sh.vocab, rope_theta=sh.rope_theta, rms_eps=sh.rms_eps),
                                  case.entries_k, case.entries_v, case.chunks, case.prefix, list(range(len(lens))),
                                  query)
    if dtype == "f32":
        assert maxrel(got, want) <= 1e-4
    else:
        assert relerr(got, want) <= 2e-2 and maxrel(got, want) <= 2e-2
    # CacheClip 6.2 step 6 and 6.3: top-k of the scores, window grouping (w 8, tau 5)
    n_c = sum(lens)
    k = O.ceil_bp(2000, n_c)
    idx = torch.zeros(n_c, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    b.topk_select_dilate(r.h, scores, n_c, 0, k, 8, 5, b.BUDGET_CANDIDATE, None, idx, cnt)
    torch.cuda.synchronize()
    gsel = idx[:int(cnt.item())].cpu().numpy().tolist()
    wsel = O.select(want, k, 8, 5, "candidate").tolist()
    if dtype == "f32":
        # the candidates themselves may differ only at near-ties of the oracle's scores
        gc = O.topk(got, k)
        assert set_diff_is_near_tie(gc, O.topk(want, k), want, k, rel=1e-4)
        if set(gc) == set(O.topk(want, k)):
            assert gsel == wsel
