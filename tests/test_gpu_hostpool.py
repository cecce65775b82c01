"""A chunk-KV pool in pinned host memory (CacheBlend blog, "Making the recompute free":
loading overlaps recompute; each layer's recompute waits only for that layer's KV).

The same kernels read the pool in place from host memory, one layer at a time on a side
stream, so the outputs must be bitwise identical to a run with the pool in device memory.
"""
import numpy as np
import pytest
import torch

from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import GpuRunner, make_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


def _host_pool(r, case, pinned=True):
    tok = np.concatenate([np.concatenate([case.prefix, c]) for c in case.chunks]).astype(np.int32)
    k, v, t = case.pool_k.clone(), case.pool_v.clone(), torch.from_numpy(tok)
    if pinned:
        k, v, t = k.pin_memory(), v.pin_memory(), t.pin_memory()
    return b.PoolRef(k, v, t, len(case.prefix), [len(c) for c in case.chunks], case.entry_row, location="host")


def _run(r, reqs, pool, n_tok, n_q, n_c):
    out = r.outputs(n_tok, n_q, n_c)
    b.blend_prefill(r.h, reqs, pool, out)
    b.blend_device_status(r.h)
    return {k: v.cpu() for k, v in out.t.items() if v is not None}


@pytest.mark.parametrize("kind", ["bf16-ext", "f32-hkvd"])
def test_host_pool_gives_identical_results(kind):
    dev = torch.device("cuda:0")
    if kind == "bf16-ext":
        sh = synth.ModelShape("hp-bf16", 3, 256, 4, 2, 128, 512, 300, 1e6)
        case = make_case(sh, 8, [64, 48, 96, 40], seed=2, pool="random")
        mode = dict(mode="ext", rho_bp=2000, window=4)
    else:
        sh = synth.ModelShape("hp-f32", 4, 256, 4, 2, 64, 688, 300, 1e4, dtype="f32", init="fan_in")
        case = make_case(sh, 8, [64, 48, 96, 40], seed=3, pool="random")
        mode = dict(mode="hkvd", rho_bp=2000, r1_bp=3000, window=2)
    order = [2, 0, 3, 1]
    n_c = sum(len(case.chunks[c]) for c in order)
    Q = 16
    N = len(case.prefix) + n_c + Q
    r = GpuRunner(case, n_c + Q, N, n_c, max_pos=N)
    g = torch.Generator().manual_seed(4)
    query = synth.token_ids(Q, sh.vocab, g).to(dev)
    scores = torch.rand(n_c, generator=g).to(dev) if mode["mode"] == "ext" else None
    req = b.RequestRef(order, query, scores=scores, **mode)
    want = _run(r, [req], r.pool, N, Q, n_c)
    hp = _host_pool(r, case)
    for _ in range(2):  # the per-layer events are reused from call to call
        got = _run(r, [req], hp, N, Q, n_c)
        for k in want:
            assert torch.equal(got[k], want[k]), k


def test_pageable_host_pool_is_rejected():
    sh = synth.ModelShape("hp-rej", 1, 256, 4, 2, 64, 688, 300, 1e4, dtype="f32")
    case = make_case(sh, 4, [32, 32], pool="random")
    r = GpuRunner(case, 80, 100, 64, max_pos=100)
    hp = _host_pool(r, case, pinned=False)
    dev = torch.device("cuda:0")
    req = b.RequestRef([0, 1], torch.zeros(4, dtype=torch.int32, device=dev), mode="full")
    with pytest.raises(b.BlendError) as e:
        b.blend_prefill(r.h, [req], hp, r.outputs(4 + 64 + 4, 4, 64))
    assert e.value.code == b.EINVAL
