"""The allocation-free selection call against the workspace-backed one.

topk_select_dilate_noalloc serves callers that cannot allocate device memory while
they select tokens (a serving loop that reserved all HBM up front, or a hot path that
must not call cudaMalloc/cudaFree because they may synchronise the device).  It keeps
its scratch (ranks and sorted keys) in fixed device arrays instead of a handle's
workspace.  Here it is called through the C ABI several times in a row, with different
inputs, and each result must equal topk_select_dilate's exactly (index sets are compared
bit for bit, as in the other selection tests).  This file is collected last on purpose.
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


def _run_both(r, s, allowed, base, budget, w, tau, mode):
    dev = torch.device("cuda:0")
    n = s.numel()
    al = None if allowed is None else allowed.to(dev)
    ref_idx = torch.full((n,), -1, dtype=torch.int32, device=dev)
    ref_n = torch.zeros(1, dtype=torch.int32, device=dev)
    b.topk_select_dilate(r.h, s, n, base, budget, w, tau, mode, al, ref_idx, ref_n)
    got_idx = torch.full((n,), -2, dtype=torch.int32, device=dev)
    got_n = torch.zeros(1, dtype=torch.int32, device=dev)
    b.topk_select_dilate_noalloc(s, n, base, budget, w, tau, mode, al, got_idx, got_n)
    torch.cuda.synchronize()
    k = int(ref_n.item())
    assert int(got_n.item()) == k
    assert torch.equal(got_idx[:k], ref_idx[:k])
    return k


def test_noalloc_selection_equals_workspace_selection_on_two_calls():
    dev = torch.device("cuda:0")
    case = make_case(synth.ModelShape("t", 1, 256, 4, 2, 64, 688, 64, 1e4, dtype="f32"), 4, [8], pool="random")
    r = GpuRunner(case, 64, 64, 32768)
    g = torch.Generator().manual_seed(21)
    # call 1: the 16K-context shape, window-4 dilation under a final-row budget
    s1 = torch.randn(15872, generator=g).to(dev)
    k1 = _run_both(r, s1, None, 64, 3175, 4, 1, b.BUDGET_FINAL)
    assert 0 < k1 <= 3175
    # call 2 straight after: ties, an allowed mask, CacheClip's (8, 5) grouping by candidates
    s2 = torch.randint(0, 5, (9000,), generator=g).float().to(dev)
    allowed = (torch.rand(9000, generator=g) < 0.7).to(torch.uint8)
    k2 = _run_both(r, s2, allowed, 7, 1800, 8, 5, b.BUDGET_CANDIDATE)
    assert k2 > 0
    # call 3: the largest size the fixed scratch holds, every entry of it in use
    s3 = torch.randn(32768, generator=g).to(dev)
    k3 = _run_both(r, s3, None, 0, 6554, 2, 1, b.BUDGET_FINAL)
    assert 0 < k3 <= 6554


def test_noalloc_rejects_sizes_above_its_scratch():
    dev = torch.device("cuda:0")
    n = 32769
    s = torch.zeros(n, device=dev)
    idx = torch.full((n,), -3, dtype=torch.int32, device=dev)
    cnt = torch.full((1,), -3, dtype=torch.int32, device=dev)
    with pytest.raises(b.BlendError) as e:
        b.topk_select_dilate_noalloc(s, n, 0, 10, 1, 1, b.BUDGET_FINAL, None, idx, cnt)
    assert e.value.code == b.EINVAL and "32768" in str(e.value)
    torch.cuda.synchronize()
    assert int(cnt.item()) == -3 and int(idx.min().item()) == -3
