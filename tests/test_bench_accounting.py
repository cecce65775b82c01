"""Host-side checks of the benchmark's work accounting (no GPU): the algorithmic FLOP and
byte counts that every roofline fraction divides by.

The GEMM total at the 14B shape is pinned to the figure derived by hand from the model
shape (2 x rows x parameters per layer x layers: 8.73e13 FLOP at 3 303 rows per layer),
the attention count to its causal-pair definition on a hand-sized case, and the
per-layer schedules (HKVD gradual filtering, the focus filter) to the layers each set
is used on.
"""
import importlib.util
import os

import pytest

from rag_kv_cache_rope_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def gemm_flop(sh, rows):
    H, F, qd, kvd = sh.hidden, sh.ffn, sh.q_dim, sh.kv_dim
    return 2.0 * rows * (H * (qd + 2 * kvd) + qd * H + 3 * H * F)


def test_14b_gemm_flop_matches_hand_count(bench):
    wl = synth.WORKLOADS["qwen14b-16k-ext20"]
    L = wl.model.n_layers
    work = bench.step_work(wl, [(3303, 3303, 0)] * L)
    gemm = sum(work[k][1] for k in ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down"))
    assert abs(gemm - 8.73e13) / 8.73e13 < 2e-3
    assert all(work[k][2] == L for k in ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down", "attention"))
    assert work["assemble"][2] == 1


def test_attention_counts_causal_pairs_only(bench):
    wl = synth.WORKLOADS["qwen14b-16k-ext20"]
    sh = wl.model
    # two rows at positions 9 and 99: 10 + 100 causal pairs per head
    work = bench.step_work(wl, [(2, 2, 110)] * sh.n_layers)
    assert work["attention"][1] == 4.0 * sh.head_dim * sh.n_q_heads * 110 * sh.n_layers


def test_roofline_takes_the_larger_bound(bench):
    wl = synth.WORKLOADS["qwen14b-16k-ext20"]
    sh = wl.model
    one_row = bench.algorithmic(sh, 1, 1, wl)["gemm_gate_up"]
    many = bench.algorithmic(sh, 3303, 1, wl)["gemm_gate_up"]
    bw, tc = bench.PEAKS["hbm_gbs"] * 1e9, bench.PEAKS["bf16_tflops_sustained"] * 1e12
    # one row: reading the 283 MB of gate/up weights dominates; 3 303 rows: the FLOP
    assert bench.ideal_launch_ms(one_row) == pytest.approx(one_row[2] / bw * 1e3)
    assert one_row[2] >= 2 * sh.hidden * 2 * sh.ffn
    assert bench.ideal_launch_ms(many) == pytest.approx(many[1] / tc * 1e3)


def test_hkvd_schedule_projects_more_rows_than_it_attends(bench):
    wl = synth.WORKLOADS["llama8b-3k-hkvd15"]
    sh = wl.model
    L = sh.n_layers
    r0, r1, r2 = 3136, 756, 525
    layers = [(r0, r0, 10), (r0, r1, 5), (r1, r2, 3)] + [(r2, r2, 3)] * (L - 3)
    work = bench.step_work(wl, layers)
    H, qd, kvd = sh.hidden, sh.q_dim, sh.kv_dim
    want_qkv = 2.0 * H * (qd + 2 * kvd) * (2 * r0 + r1 + (L - 3) * r2)
    want_o = 2.0 * qd * H * (r0 + r1 + (L - 2) * r2)
    assert work["gemm_qkv"][1] == want_qkv
    assert work["gemm_o"][1] == want_o
    assert work["attention"][1] == 4.0 * sh.head_dim * sh.n_q_heads * (10 + 5 + 3 * (L - 2))


def test_batch_scales_assembly_and_kv_bytes(bench):
    wl = synth.WORKLOADS["mistral7b-b8-ext15"]
    sh = wl.model
    a = bench.algorithmic(sh, 100, 100, wl)
    es = 2
    assert a["assemble"][1] == 2 * 2 * sh.n_layers * wl.batch * (wl.prefix_len + wl.n_chunk_rows) * sh.kv_dim * es
    assert a["attention"][2] >= 2 * wl.batch * wl.n_ctx * sh.kv_dim * es
