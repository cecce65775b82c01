"""Host-side checks of the C ABI: the library builds and loads, exports every function
include/blend.h declares, the ctypes mirrors of the structs match the C layout (checked
by compiling a small C probe with gcc), and argument validation rejects bad calls
before touching the GPU.  No GPU is needed."""
import ctypes as C
import os
import re
import subprocess
import tempfile

import pytest

from rag_kv_cache_rope_gb300 import binding as b
from rag_kv_cache_rope_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "blend.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return b.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for n in ("blend_init", "rope_realign", "kv_deviation", "topk_select_dilate", "gather_rows",
              "selective_layer", "scatter_kv", "blend_prefill"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(b.EXPORTED) == set(declared_functions())


PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "blend.h"
#define P(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("blend_model_cfg %zu\n", sizeof(blend_model_cfg));
  P(blend_model_cfg, rope_theta) P(blend_model_cfg, rms_eps) P(blend_model_cfg, max_pos)
  printf("blend_weights %zu\n", sizeof(blend_weights));
  printf("blend_limits %zu\n", sizeof(blend_limits));
  printf("blend_pool %zu\n", sizeof(blend_pool));
  P(blend_pool, entry_len) P(blend_pool, n_rows) P(blend_pool, tokens) P(blend_pool, location)
  printf("blend_request %zu\n", sizeof(blend_request));
  P(blend_request, chunk_ids) P(blend_request, query_tokens) P(blend_request, scores)
  P(blend_request, n_stages) P(blend_request, stage_layer) P(blend_request, stage_pos) P(blend_request, stage_n)
  P(blend_request, group_rule) P(blend_request, tau_smooth) P(blend_request, tau_cover_bp)
  P(blend_request, max_span) P(blend_request, cap_bp) P(blend_request, epic_m)
  P(blend_request, focus_layer) P(blend_request, focus_bp)
  printf("blend_outputs %zu\n", sizeof(blend_outputs));
  P(blend_outputs, dev2) P(blend_outputs, q_last)
  return 0;
}
"""


def test_struct_layout_matches_c():
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        open(src, "w").write(PROBE)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        got = dict(line.rsplit(" ", 1) for line in subprocess.run([exe], capture_output=True,
                                                                    text=True).stdout.splitlines())
    got = {k: int(v) for k, v in got.items()}
    mirror = {"blend_model_cfg": b.ModelCfg, "blend_weights": b.Weights, "blend_limits": b.Limits,
              "blend_pool": b.Pool, "blend_request": b.Request, "blend_outputs": b.Outputs}
    for k, v in got.items():
        if "." in k:
            s, f = k.split(".")
            assert getattr(mirror[s], f).offset == v, k
        else:
            assert C.sizeof(mirror[k]) == v, k


def _cfg(**kw):
    base = dict(n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=688, vocab=1024,
                dtype=b.F32, rope_theta=1e4, rms_eps=1e-6, max_pos=1024)
    base.update(kw)
    return b.ModelCfg(**base)


def test_workspace_size_and_validation(lib):
    lim = b.Limits(1024, 4096, 512, 2)
    n = b.blend_workspace_size(_cfg(), lim)
    assert n > 0 and n % 256 == 0
    # grows with the limits
    assert b.blend_workspace_size(_cfg(), b.Limits(2048, 4096, 512, 2)) > n
    for bad in (dict(head_dim=96), dict(n_kv_heads=3), dict(ffn=100), dict(dtype=7), dict(max_pos=0),
                dict(n_layers=0), dict(rope_theta=-1.0)):
        assert b.blend_workspace_size(_cfg(**bad), lim) == 0, bad
    assert b.blend_workspace_size(_cfg(), b.Limits(1, 1, 40000, 1)) == 0
    assert b.blend_workspace_size(_cfg(), b.Limits(1, 1, 1, 65)) == 0


def test_init_rejects_bad_arguments_without_a_gpu(lib):
    out = C.c_void_p()
    w = b.Weights(*([1 << 20] * 8))
    lim = b.Limits(64, 256, 128, 1)
    rc = lib.blend_init(C.byref(_cfg(head_dim=80)), C.byref(w), C.byref(lim), C.c_void_p(1 << 20), 1 << 30,
                        None, C.byref(out))
    assert rc == b.EINVAL and b"head_dim" in lib.blend_last_error(None)
    rc = lib.blend_init(C.byref(_cfg()), C.byref(w), C.byref(lim), C.c_void_p((1 << 20) + 8), 1 << 30,
                        None, C.byref(out))
    assert rc == b.EINVAL and b"aligned" in lib.blend_last_error(None)
    rc = lib.blend_init(C.byref(_cfg()), C.byref(w), C.byref(lim), C.c_void_p(1 << 20), 100, None,
                        C.byref(out))
    assert rc == b.ENOMEM
    w0 = b.Weights(*([1 << 20] * 7 + [0]))
    rc = lib.blend_init(C.byref(_cfg()), C.byref(w0), C.byref(lim), C.c_void_p(1 << 20), 1 << 30, None,
                        C.byref(out))
    assert rc == b.EINVAL
    assert lib.blend_destroy(None) == b.EINVAL
    vp = C.c_void_p(1 << 20)
    assert lib.gather_rows(None, vp, 16, 4, vp, vp, 1, vp, None) == b.EINVAL          # no handle
    assert lib.scatter_kv(None, vp, vp, vp, vp, 1, 4, vp, vp, None) == b.EINVAL
    assert lib.kv_deviation(None, vp, vp, vp, vp, vp, vp, 1, 4, b.DEV_KV, vp, None) == b.EINVAL
    assert lib.selective_layer(None, 0, vp, vp, vp, 1, vp, vp, 4, None, b.DEV_KV, None) == b.EINVAL
    assert lib.importance_scores(C.c_void_p(1 << 20), 4, 0, 8, b.F32, C.c_void_p(1 << 20), None) == b.EINVAL
    assert lib.importance_scores(C.c_void_p(1 << 20), 4, 4097, 8, b.F32, C.c_void_p(1 << 20), None) == b.EINVAL
    vp = C.c_void_p(1 << 20)
    assert lib.span_select(None, vp, 8, 0, 4, 4, 0.4, 7000, 16, b.BUDGET_FINAL, vp, vp, None) == b.EINVAL
    assert lib.align_expand(None, vp, vp, 4, 0, vp, vp, 4, 8, 0, vp, vp, None) == b.EINVAL
    assert lib.blend_wait_flag(None, vp, 10, None) == b.EINVAL


def test_pack_weights_layout():
    import torch
    L, F, H = 2, 32, 8
    w = {"embed": torch.zeros(4, H), "wq": torch.randn(L, 16, H), "wk": torch.randn(L, 8, H),
         "wv": torch.randn(L, 8, H), "wo": torch.randn(L, H, 16), "wg": torch.randn(L, F, H),
         "wu": torch.randn(L, F, H), "wd": torch.randn(L, H, F), "attn_norm": torch.ones(L, H),
         "mlp_norm": torch.ones(L, H), "final_norm": torch.ones(H)}
    p = b.pack_weights(w)
    assert torch.equal(p["w_qkv"][:, :16], w["wq"]) and torch.equal(p["w_qkv"][:, 24:], w["wv"])
    g = b.GU_BLOCK
    for j in range(F // g):
        assert torch.equal(p["w_gu"][:, 2 * g * j:2 * g * j + g], w["wg"][:, g * j:g * (j + 1)])
        assert torch.equal(p["w_gu"][:, 2 * g * j + g:2 * g * (j + 1)], w["wu"][:, g * j:g * (j + 1)])
