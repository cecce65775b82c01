"""The tcgen05 tensor-core path (GEMMs and attention) against the oracle and against the
CUDA-core path.

One decoder layer through selective_layer with the tensor cores on and off: row
counts that span several 128-row tiles with a ragged tail, widths that give several
256-column tiles and many 64-wide k-blocks per tile, and more tiles than SMs.
"""
import math

import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B
from rag_kv_cache_rope_gb300 import synth

from blendcase import GpuRunner, f64, make_case, maxrel, oracle_cfg

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    b.lib()


SHAPES = [
    (synth.ModelShape("tc-small", 2, 512, 8, 2, 128, 1024, 300, 1e6), 300, 700),
    (synth.ModelShape("tc-wide", 2, 2048, 16, 4, 128, 5632, 300, 1e6), 1000, 1500),
    # 5 query heads per kv head (the 14B grouping), contexts spanning ~60 key blocks
    (synth.ModelShape("tc-gqa5", 2, 1280, 10, 2, 128, 2560, 300, 1e6), 700, 4000),
    # SmolLM2-135M widths: projections of 960 and 576 columns end in partial 256-wide tiles
    (synth.ModelShape("tc-smol", 2, 576, 9, 3, 64, 1536, 300, 1e5), 500, 900),
    # CTA pairs at their edges: 90 rows x 4 heads = 3 attention tiles per kv head, so the
    # last item has no second tile; 129 rows put one live row in the second CTA of a 256-row
    # GEMM tile; 257 rows leave the second 256-row tile one row
    (synth.ModelShape("tc-pair-odd", 2, 512, 8, 2, 128, 1024, 300, 1e6), 90, 300),
    (synth.ModelShape("tc-pair-129", 2, 512, 8, 2, 128, 1024, 300, 1e6), 129, 500),
    (synth.ModelShape("tc-pair-257", 2, 1280, 10, 2, 128, 2560, 300, 1e6), 257, 2000),
    # one query head per kv head (plain multi-head attention) and eight (a tile of 128 pairs
    # then holds 16 rows)
    (synth.ModelShape("tc-mha", 2, 512, 4, 4, 128, 1024, 300, 1e6), 300, 900),
    (synth.ModelShape("tc-gqa8", 2, 2048, 16, 2, 128, 2048, 300, 1e6), 200, 1200),
    # 525 rows with an 8B-wide MLP (the few-row regime of the 8B HKVD request: 336 CTA-pair
    # gate/up tiles, a last wave run as K halves)
    (synth.ModelShape("tc-mlp-525", 2, 512, 8, 2, 128, 14336, 300, 1e6), 525, 900),
]


@pytest.mark.parametrize("shape,n,n_ctx", SHAPES, ids=[s[0].name for s in SHAPES])
def test_layer_tensor_cores_match_oracle_and_cuda_cores(shape, n, n_ctx):
    dev = torch.device("cuda:0")
    case = make_case(shape, 4, [8], pool="random")
    r = GpuRunner(case, max(n, 128), n_ctx, 64, max_pos=n_ctx)
    assert b.blend_set_tensor_cores(r.h, True) == 1, "tcgen05 path unavailable on this GPU"
    g = torch.Generator().manual_seed(11)
    dt = synth.torch_dtype(shape)
    kc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt)
    vc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt)
    x = torch.randn(n, shape.hidden, generator=g)
    pos = torch.sort(torch.randperm(n_ctx, generator=g)[:n]).values.to(torch.int32)
    outs = {}
    for tc in (True, False):
        b.blend_set_tensor_cores(r.h, tc)
        xg, kg, vg = x.to(dev), kc.to(dev), vc.to(dev)
        dv = torch.zeros(n, device=dev)
        b.selective_layer(r.h, 1, xg, pos.to(dev), n, kg, vg, n_ctx, dv)
        b.blend_device_status(r.h)
        outs[tc] = (f64(xg), f64(kg), f64(vg), f64(dv))
    # without a deviation output the projection, RoPE and cache write run as one fused kernel
    b.blend_set_tensor_cores(r.h, True)
    xg, kg, vg = x.to(dev), kc.to(dev), vc.to(dev)
    b.selective_layer(r.h, 1, xg, pos.to(dev), n, kg, vg, n_ctx, None)
    b.blend_device_status(r.h)
    fused = (f64(xg), f64(kg), f64(vg))
    K, V = f64(kc), f64(vc)
    xo, dref = O.layer_forward(case.w_np, oracle_cfg(shape), 1, f64(x), pos.numpy(), K, V,
                               np.ones(n, dtype=bool))
    for tc, (xg, kg, vg, dv) in outs.items():
        assert maxrel(kg, K) <= TOL_BF16, tc
        assert maxrel(vg, V) <= TOL_BF16, tc
        assert maxrel(xg, xo) <= TOL_BF16, tc
        assert maxrel(dv, dref) <= TOL_BF16, tc
    assert maxrel(fused[1], K) <= TOL_BF16 and maxrel(fused[2], V) <= TOL_BF16
    assert maxrel(fused[0], xo) <= TOL_BF16
    # the GPU paths differ only by fp32 summation order and where bf16 rounding happens
    assert maxrel(outs[True][0], outs[False][0]) <= 1e-2
    assert maxrel(fused[0], outs[True][0]) <= 1e-2


@pytest.mark.parametrize("shape,n,n_ctx", SHAPES[:2], ids=[s[0].name for s in SHAPES[:2]])
def test_split_tail_gemm_is_deterministic(shape, n, n_ctx):
    """Shapes whose projections run as column halves (fewer tiles than half the SMs, or a
    last wave at most half full): two runs of the same layer give bitwise identical
    outputs."""
    dev = torch.device("cuda:0")
    case = make_case(shape, 4, [8], pool="random")
    r = GpuRunner(case, max(n, 128), n_ctx, 64, max_pos=n_ctx)
    g = torch.Generator().manual_seed(12)
    dt = synth.torch_dtype(shape)
    kc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt)
    vc = (0.5 * torch.randn(n_ctx, shape.n_kv_heads, shape.head_dim, generator=g)).to(dt)
    x = torch.randn(n, shape.hidden, generator=g)
    pos = torch.sort(torch.randperm(n_ctx, generator=g)[:n]).values.to(torch.int32).to(dev)
    runs = []
    for _ in range(3):
        xg, kg, vg = x.to(dev), kc.to(dev), vc.to(dev)
        b.selective_layer(r.h, 1, xg, pos, n, kg, vg, n_ctx, None)
        b.blend_device_status(r.h)
        runs.append((xg.cpu(), kg.cpu(), vg.cpu()))
    for other in runs[1:]:
        for a, c in zip(runs[0], other):
            assert torch.equal(a, c)


# Attention at large logits.  Each shape has hq * d == H, so with wo the identity and
# wd = 0 the layer's output is x + o: the attention output itself is read back against
# the oracle's causal softmax (CacheBlend blog, "Selective KV recompute": ordinary
# attention over the expanded K/V).  The reused cache rows of 128-key block b hold
# beta_b * r_g (one random unit direction per kv head), so a row's logits step from
# block to block by tens of nats: they rise ("rise": the running maximum grows on every
# block, the exponentials against the old reference pass 2^50 and the exact path with its
# rescale runs), fall ("fall": a huge first block, then small ones), or jump once in the
# middle ("spike").  Ten rows sit at positions 0..9 ahead of rows past position 1500, so
# in the same warp some lanes have every later block masked while others take the exact
# path.
LOGIT_SHAPES = [
    (synth.ModelShape("big-logit-d128", 2, 1024, 8, 2, 128, 1024, 300, 1e6), 300, 3000),
    (synth.ModelShape("big-logit-gqa5", 2, 1280, 10, 2, 128, 2560, 300, 1e6), 200, 2200),
    (synth.ModelShape("big-logit-d64", 2, 384, 6, 3, 64, 768, 300, 1e4), 250, 2000),
]


@pytest.mark.parametrize("profile", ["rise", "fall", "spike"])
@pytest.mark.parametrize("shape,n,n_ctx", LOGIT_SHAPES, ids=[s[0].name for s in LOGIT_SHAPES])
def test_attention_large_logits_match_oracle(shape, n, n_ctx, profile):
    dev = torch.device("cuda:0")
    H, hkv, d = shape.hidden, shape.n_kv_heads, shape.head_dim
    assert shape.n_q_heads * d == H
    case = make_case(shape, 4, [8], pool="random")
    eye = torch.eye(H, dtype=case.w_t["wo"].dtype)
    case.w_t["wo"][1] = eye
    case.w_t["wd"][1] = 0
    case.w_np["wo"][1] = f64(eye)
    case.w_np["wd"][1] = 0.0
    r = GpuRunner(case, max(n, 128), n_ctx, 64, max_pos=n_ctx)
    assert b.blend_set_tensor_cores(r.h, True) == 1
    g = torch.Generator().manual_seed(31)
    nblk = (n_ctx + 127) // 128
    # q's entries have std 0.02 sqrt(H) (unit-RMS rows through N(0, 0.02^2) weights), so
    # q.r / sqrt(d) ~ 0.02 sqrt(H / d) per unit of beta: steps of ~12 nats per block
    step = 12.0 / (0.02 * math.sqrt(H / d))
    blk = torch.arange(n_ctx) // 128
    if profile == "rise":
        beta = step * blk.double()
    elif profile == "fall":
        beta = torch.where(blk == 0, step * nblk, step * 0.05 * blk.double())
    else:
        beta = torch.where(blk == nblk // 2, step * nblk, 0.5 * step * (blk % 3).double())
    rdir = torch.randn(hkv, d, generator=g, dtype=torch.float64)
    rdir = rdir / rdir.norm(dim=1, keepdim=True)
    kc = (beta[:, None, None] * rdir[None]).to(torch.bfloat16)
    vc = (0.5 * torch.randn(n_ctx, hkv, d, generator=g)).to(torch.bfloat16)
    x = 1e-2 * torch.randn(n, H, generator=g)
    late = torch.sort(torch.randperm(n_ctx - 1500, generator=g)[:n - 10]).values + 1500
    pos = torch.cat([torch.arange(10), late]).to(torch.int32)
    xg, kg, vg = x.to(dev), kc.to(dev), vc.to(dev)
    b.selective_layer(r.h, 1, xg, pos.to(dev), n, kg, vg, n_ctx, None)
    b.blend_device_status(r.h)
    K, V = f64(kc), f64(vc)
    xo, _ = O.layer_forward(case.w_np, oracle_cfg(shape), 1, f64(x), pos.numpy(), K, V)
    o_gpu, o_ref = f64(xg) - f64(x), xo - f64(x)
    assert np.all(np.isfinite(o_gpu))
    assert maxrel(o_gpu, o_ref) <= TOL_BF16, (profile, maxrel(o_gpu, o_ref))
    assert maxrel(f64(kg), K) <= TOL_BF16 and maxrel(f64(vg), V) <= TOL_BF16
