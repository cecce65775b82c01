"""Failure detection on the GPU without a fault: a bounded device-side wait on a flag that
nothing sets runs out, records BLEND_ETIMEOUT in the handle's error word, the host reads it
through blend_device_status, and the handle and the CUDA context keep working afterwards.
No test here traps, faults or hangs the GPU: the wait is bounded (a few thousand polls)."""
import numpy as np
import pytest
import torch

from oracle import blend_oracle as O
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


def test_bounded_wait_times_out_and_the_context_stays_usable():
    dev = torch.device("cuda:0")
    r = GpuRunner(make_case(synth.TINY, 4, [8], pool="random"), 64, 64, 1024)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    b.blend_wait_flag(r.h, flag, 2000)              # nothing ever sets the flag
    with pytest.raises(b.BlendError) as e:
        b.blend_device_status(r.h)
    assert e.value.code == b.ETIMEOUT
    b.blend_device_status(r.h)                      # the word was cleared on read
    flag.fill_(1)
    b.blend_wait_flag(r.h, flag, 2000)              # set: the wait ends at once
    b.blend_device_status(r.h)
    # the same handle and context still compute: a selection checked against the oracle
    s = np.random.default_rng(2).standard_normal(500).astype(np.float32)
    idx = torch.full((500,), -1, dtype=torch.int32, device=dev)
    cnt = torch.zeros(1, dtype=torch.int32, device=dev)
    b.topk_select_dilate(r.h, torch.from_numpy(s).to(dev), 500, 7, 60, 4, 1, b.BUDGET_FINAL, None, idx, cnt)
    b.blend_device_status(r.h)
    got = idx[:int(cnt.item())].cpu().numpy().tolist()
    assert got == O.select_final_bisect(s.astype(np.float64), 60, 4, 1, base=7).tolist()


def test_bounded_wait_rejects_bad_arguments_before_launching():
    dev = torch.device("cuda:0")
    r = GpuRunner(make_case(synth.TINY, 4, [8], pool="random"), 64, 64, 1024)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    raw = torch.zeros(8, dtype=torch.uint8, device=dev)
    for f, polls in [(flag, -1), (flag, (1 << 24) + 1), (raw[1:], 10)]:
        with pytest.raises(b.BlendError) as e:
            b.blend_wait_flag(r.h, f, polls)
        assert e.value.code == b.EINVAL
    b.blend_device_status(r.h)                      # nothing was launched, nothing recorded
