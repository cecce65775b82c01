"""CacheBlend's loading controller (CacheBlend blog, "Making the recompute free"): the
oracle's formulas against hand-computed cases, and the C ABI's host implementation
against the oracle (host arithmetic only; no GPU involved)."""
import math
import random

import pytest

from oracle import blend_oracle as O
from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build()
    return b.lib()


def test_hand_cases():
    # full prefill 1.0 s; 2 GB of KV at 4 GB/s loads in 0.5 s -> the delays match at 50 %
    assert O.ratio_controller(1.0, 2e9, 4e9, 1500) == 5000
    # a fast device: 0.1 s of loading would suggest 10 %, below the 15 % floor
    assert O.ratio_controller(1.0, 1e9, 1e10, 1500) == 1500
    # a slow device: 2 s of loading caps at 100 %
    assert O.ratio_controller(1.0, 2e9, 1e9, 1500) == 10000
    # 0.37 s of 1 s -> 3700 basis points
    assert O.ratio_controller(1.0, 3.7e9, 1e10, 1500) == 3700


def test_storage_choice_hand_case():
    """At the 15 % floor a 2 s prefill gives 0.3 s to hide the load of 6 GB: devices of
    30 GB/s (0.2 s) and 25 GB/s (0.24 s) qualify, 10 GB/s (0.6 s) does not; the cheaper of
    the two qualifying ones wins."""
    bw = [10e9, 30e9, 25e9]
    cost = [0.1, 3.0, 2.0]
    assert O.pick_storage(2.0, 6e9, 1500, bw, cost) == 2
    assert O.pick_storage(2.0, 6e9, 1500, [10e9], [0.1]) == -1
    assert O.pick_storage(2.0, 6e9, 1500, [30e9, 30e9], [1.0, 1.0]) == 0


def test_library_matches_oracle(lib):
    rnd = random.Random(5)
    for _ in range(200):
        full = 10 ** rnd.uniform(-3, 1)
        kv = 10 ** rnd.uniform(6, 11)
        bw = 10 ** rnd.uniform(8, 12)
        fl = rnd.choice([0, 1500, 2000, 10000])
        assert b.blend_ratio_controller(full, kv, bw, fl) == O.ratio_controller(full, kv, bw, fl)
        n = rnd.randint(0, 6)
        bws = [10 ** rnd.uniform(8, 12) for _ in range(n)]
        costs = [rnd.choice([0.5, 1.0, 2.0, 3.0]) for _ in range(n)]
        assert b.blend_pick_storage(full, kv, fl, bws, costs) == O.pick_storage(full, kv, fl, bws, costs)


def test_library_rejects_bad_inputs(lib):
    for args in [(0.0, 1e9, 1e9, 1500), (1.0, -1.0, 1e9, 1500), (1.0, 1e9, 0.0, 1500), (1.0, 1e9, 1e9, 10001),
                 (math.inf, 1e9, 1e9, 1500)]:
        with pytest.raises(b.BlendError):
            b.blend_ratio_controller(*args)
    with pytest.raises(b.BlendError):
        b.blend_pick_storage(1.0, 1e9, 1500, [0.0], [1.0])
