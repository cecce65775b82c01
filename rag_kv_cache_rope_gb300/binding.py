"""Thin Python binding of libblend's C ABI (include/blend.h).

Functions carry the C names and only marshal arguments: torch tensors become device
pointers, Python lists become host arrays, and a non-zero status raises BlendError.
Every step of the method runs in the library's CUDA kernels.  If libblend.so is
missing, lib() raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libblend.so")

OK, EINVAL, ENOMEM, ECUDA, EMISS, ETIMEOUT, EDEVICE, EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6, -7
F32, BF16 = 0, 1
SEL_EXT, SEL_HKVD, SEL_FORCED, SEL_FULL, SEL_EPIC = 0, 1, 2, 3, 4
BUDGET_FINAL, BUDGET_CANDIDATE = 0, 1
DEV_KV, DEV_V = 0, 1
GROUP_WINDOW, GROUP_SPAN = 0, 1
POOL_DEVICE, POOL_HOST = 0, 1
MAX_BATCH = 64
MAX_SPAN = 64
MAX_ALIGN_TARGETS = 131072
GU_BLOCK = 16

MODES = {"ext": SEL_EXT, "hkvd": SEL_HKVD, "forced": SEL_FORCED, "full": SEL_FULL, "epic": SEL_EPIC}
BUDGETS = {"final": BUDGET_FINAL, "candidate": BUDGET_CANDIDATE}
DEVMODES = {"kv": DEV_KV, "v": DEV_V}
GROUP_RULES = {"window": GROUP_WINDOW, "span": GROUP_SPAN}


class BlendError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libblend error {code}: {msg}")
        self.code = code


# ---------------------------------------------------------------- C structs
class ModelCfg(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("dtype", C.c_int32), ("rope_theta", C.c_double),
                ("rms_eps", C.c_float), ("max_pos", C.c_int32)]


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("embed", "attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gu",
                                          "w_down", "final_norm")]


class Limits(C.Structure):
    _fields_ = [("max_rows", C.c_int32), ("max_tokens", C.c_int32), ("max_chunk_rows", C.c_int32),
                ("max_batch", C.c_int32)]


class Pool(C.Structure):
    _fields_ = [("n_entries", C.c_int32), ("prefix_len", C.c_int32),
                ("entry_len", C.POINTER(C.c_int32)), ("entry_row", C.POINTER(C.c_int64)),
                ("present", C.POINTER(C.c_uint8)), ("n_rows", C.c_int64), ("k", C.c_void_p),
                ("v", C.c_void_p), ("tokens", C.c_void_p), ("location", C.c_int32)]


class Request(C.Structure):
    _fields_ = [("n_chunks", C.c_int32), ("chunk_ids", C.POINTER(C.c_int32)),
                ("query_len", C.c_int32), ("query_tokens", C.c_void_p), ("mode", C.c_int32),
                ("rho_bp", C.c_int32), ("r1_bp", C.c_int32), ("window", C.c_int32),
                ("tau", C.c_int32), ("budget_mode", C.c_int32), ("dev_mode", C.c_int32),
                ("scores", C.c_void_p), ("n_stages", C.c_int32), ("stage_layer", C.c_int32 * 3),
                ("stage_pos", C.c_void_p * 3), ("stage_n", C.c_int32 * 3), ("group_rule", C.c_int32),
                ("tau_smooth", C.c_float), ("tau_cover_bp", C.c_int32), ("max_span", C.c_int32),
                ("cap_bp", C.c_int32), ("epic_m", C.c_int32), ("focus_layer", C.c_int32),
                ("focus_bp", C.c_int32)]


class Outputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("k", "v", "hidden", "sel", "n_sel", "c1", "n_c1", "dev1",
                                          "dev2", "q_last")]


_lib = None


def lib() -> C.CDLL:
    """Loads libblend.so (built by build.build()); raises if it is not there."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "rag_kv_cache_rope_gb300.build.build() (needs nvcc)")
        L = C.CDLL(LIB_PATH)
        vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
        sig = {
            "blend_workspace_size": (C.c_size_t, [C.POINTER(ModelCfg), C.POINTER(Limits)]),
            "blend_init": (C.c_int, [C.POINTER(ModelCfg), C.POINTER(Weights), C.POINTER(Limits), vp,
                                     C.c_size_t, vp, C.POINTER(vp)]),
            "blend_destroy": (C.c_int, [vp]),
            "blend_last_error": (C.c_char_p, [vp]),
            "blend_device_status": (C.c_int, [vp, vp]),
            "blend_set_tensor_cores": (C.c_int, [vp, C.c_int]),
            "rope_realign": (C.c_int, [vp, vp, vp, i32, vp, i32, i64, i64, vp]),
            "blend_assemble": (C.c_int, [vp, i32, C.POINTER(Request), C.POINTER(Pool),
                                         C.POINTER(Outputs), vp]),
            "kv_deviation": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, vp, vp]),
            "topk_select_dilate": (C.c_int, [vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp]),
            "gather_rows": (C.c_int, [vp, vp, i64, i64, vp, vp, i32, vp, vp]),
            "scatter_kv": (C.c_int, [vp, vp, vp, vp, vp, i32, i64, vp, vp, vp]),
            "selective_layer": (C.c_int, [vp, i32, vp, vp, vp, i32, vp, vp, i32, vp, i32, vp]),
            "blend_prefill": (C.c_int, [vp, i32, C.POINTER(Request), C.POINTER(Pool),
                                        C.POINTER(Outputs), vp]),
            "importance_scores": (C.c_int, [vp, i32, i32, i32, i32, vp, vp]),
            "blend_profile": (C.c_int, [vp, C.c_int]),
            "blend_profile_stages": (C.c_int, [vp, C.c_uint32]),
            "blend_wait_flag": (C.c_int, [vp, vp, i64, vp]),
            "blend_profile_read": (C.c_int, [vp, C.POINTER(C.c_double), C.POINTER(C.c_int64), i32]),
            "blend_profile_name": (C.c_char_p, [i32]),
            "blend_launch_count": (C.c_int64, []),
            "topk_select_dilate_noalloc": (C.c_int, [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp]),
            "span_select": (C.c_int, [vp, vp, i32, i32, i32, i32, C.c_float, i32, i32, i32, vp, vp, vp]),
            "aux_attention_scores": (C.c_int, [vp, i32, C.POINTER(Request), C.POINTER(Pool),
                                               C.POINTER(Outputs), vp, vp]),
            "blend_ratio_controller": (C.c_int, [C.c_double, C.c_double, C.c_double, i32, C.POINTER(i32)]),
            "blend_pick_storage": (C.c_int, [C.c_double, C.c_double, i32, i32, C.POINTER(C.c_double),
                                             C.POINTER(C.c_double), C.POINTER(i32)]),
            "align_expand": (C.c_int, [vp, vp, vp, i32, i32, vp, vp, i32, i32, i32, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


EXPORTED = ("blend_workspace_size", "blend_init", "blend_destroy", "blend_last_error",
            "blend_device_status", "blend_set_tensor_cores", "rope_realign", "blend_assemble",
            "kv_deviation", "topk_select_dilate", "gather_rows", "scatter_kv", "selective_layer",
            "blend_prefill", "importance_scores", "blend_profile", "blend_profile_stages", "blend_wait_flag", "blend_profile_read",
            "blend_profile_name", "blend_launch_count", "topk_select_dilate_noalloc", "span_select",
            "align_expand", "aux_attention_scores", "blend_ratio_controller", "blend_pick_storage")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(rc: int, h=None):
    if rc != OK:
        msg = lib().blend_last_error(h.ptr if h is not None else None)
        raise BlendError(rc, msg.decode() if msg else "")
    return rc


# ---------------------------------------------------------------- handle
class Handle:
    """A libblend handle plus the tensors it points into (kept alive here)."""

    def __init__(self, ptr, cfg: ModelCfg, lim: Limits, keep):
        self.ptr = ptr
        self.cfg = cfg
        self.lim = lim
        self._keep = keep

    def __del__(self):
        if getattr(self, "ptr", None) and _lib is not None:
            _lib.blend_destroy(self.ptr)
            self.ptr = None


def model_cfg(shape, max_pos: int) -> ModelCfg:
    return ModelCfg(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                    shape.ffn, shape.vocab, F32 if shape.dtype == "f32" else BF16,
                    float(shape.rope_theta), float(shape.rms_eps), int(max_pos))


def blend_workspace_size(cfg: ModelCfg, lim: Limits) -> int:
    return int(lib().blend_workspace_size(C.byref(cfg), C.byref(lim)))


def blend_init(cfg: ModelCfg, packed: dict, lim: Limits, workspace: Optional[torch.Tensor] = None,
               stream=None) -> Handle:
    need = blend_workspace_size(cfg, lim)
    if need == 0:
        raise BlendError(EINVAL, "bad model configuration or limits")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=packed["embed"].device)
    w = Weights(*[packed[k].data_ptr() for k in ("embed", "attn_norm", "w_qkv", "w_o", "mlp_norm",
                                                  "w_gu", "w_down", "final_norm")])
    out = C.c_void_p()
    rc = lib().blend_init(C.byref(cfg), C.byref(w), C.byref(lim), _ptr(workspace), workspace.numel(),
                          _stream(stream), C.byref(out))
    _check(rc)
    return Handle(out, cfg, lim, (packed, workspace))


def blend_destroy(h: Handle):
    if h.ptr:
        _check(lib().blend_destroy(h.ptr))
        h.ptr = None


def blend_device_status(h: Handle, stream=None) -> int:
    return _check(lib().blend_device_status(h.ptr, _stream(stream)), h)


def blend_wait_flag(h: Handle, flag: torch.Tensor, max_polls: int, stream=None):
    """Bounded device-side wait until flag (device int32 scalar) is nonzero; on expiry the
    handle's error word records BLEND_ETIMEOUT (raised by blend_device_status)."""
    _check(lib().blend_wait_flag(h.ptr, _ptr(flag), int(max_polls), _stream(stream)), h)


def blend_set_tensor_cores(h: Handle, on: bool) -> int:
    return int(lib().blend_set_tensor_cores(h.ptr, 1 if on else 0))


def blend_profile(h: Handle, enable: bool):
    _check(lib().blend_profile(h.ptr, 1 if enable else 0), h)


def blend_profile_stages(h: Handle, stages: Sequence[str]):
    """Record only the named stages (an empty list stops recording)."""
    names = [lib().blend_profile_name(i).decode() for i in range(32)]
    mask = 0
    for st in stages:
        if st not in names:
            raise ValueError(f"unknown profiler stage {st!r}")
        mask |= 1 << names.index(st)
    _check(lib().blend_profile_stages(h.ptr, mask), h)


def blend_profile_read(h: Handle) -> dict:
    """{stage: (total ms, kernel launches)} since blend_profile(h, True)."""
    n = 32
    ms = (C.c_double * n)()
    cnt = (C.c_int64 * n)()
    k = lib().blend_profile_read(h.ptr, ms, cnt, n)
    if k < 0:
        _check(k, h)
    return {lib().blend_profile_name(i).decode(): (ms[i], int(cnt[i])) for i in range(k)}


def blend_launch_count() -> int:
    return int(lib().blend_launch_count())


def rope_realign(h, k_src, k_dst, n_rows, delta, n_layers, src_layer_rows, dst_layer_rows, stream=None):
    _check(lib().rope_realign(h.ptr, _ptr(k_src), _ptr(k_dst), n_rows, _ptr(delta), n_layers,
                              src_layer_rows, dst_layer_rows, _stream(stream)), h)


def kv_deviation(h, k_new, v_new, k_cache, v_cache, pos, n_rows, max_rows, mode, dev_out, stream=None):
    """n_rows: device int32 count; the cache row count is taken from k_cache's first dimension."""
    _check(lib().kv_deviation(h.ptr, _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(pos),
                              _ptr(n_rows), max_rows, k_cache.shape[0], mode, _ptr(dev_out), _stream(stream)), h)


def span_select(h, scores, n, base, budget, cap, tau_smooth, tau_cover_bp, max_span, budget_mode, idx_out,
                n_out, stream=None):
    _check(lib().span_select(h.ptr, _ptr(scores), n, base, budget, cap, float(tau_smooth), tau_cover_bp, max_span,
                             budget_mode, _ptr(idx_out), _ptr(n_out), _stream(stream)), h)


def align_expand(h, sel, n_sel, max_sel, sel_base, a_start, a_end, n_spec, n_target, out_base, idx_out, n_out,
                 stream=None):
    _check(lib().align_expand(h.ptr, _ptr(sel), _ptr(n_sel), max_sel, sel_base, _ptr(a_start), _ptr(a_end), n_spec,
                              n_target, out_base, _ptr(idx_out), _ptr(n_out), _stream(stream)), h)


def topk_select_dilate(h, scores, n, base, budget, window, tau, budget_mode, allowed, idx_out, n_out,
                       stream=None):
    _check(lib().topk_select_dilate(h.ptr, _ptr(scores), n, base, budget, window, tau, budget_mode,
                                    _ptr(allowed), _ptr(idx_out), _ptr(n_out), _stream(stream)), h)


def topk_select_dilate_noalloc(scores, n, base, budget, window, tau, budget_mode, allowed, idx_out, n_out,
                               stream=None):
    """topk_select_dilate without a handle or any allocation (fixed 32768-entry device
    scratch shared by every call; see include/blend.h)."""
    _check(lib().topk_select_dilate_noalloc(_ptr(scores), n, base, budget, window, tau, budget_mode,
                                            _ptr(allowed), _ptr(idx_out), _ptr(n_out), _stream(stream)))


def gather_rows(h, src, row_bytes, idx, n, max_n, dst, stream=None):
    """src's first dimension is its row count (src_rows of the C call)."""
    _check(lib().gather_rows(h.ptr, _ptr(src), row_bytes, src.shape[0], _ptr(idx), _ptr(n), max_n, _ptr(dst),
                             _stream(stream)), h)


def scatter_kv(h, k_new, v_new, pos, n, max_n, k_cache, v_cache, stream=None):
    """The cache row count (n_ctx of the C call) is k_cache's first dimension."""
    _check(lib().scatter_kv(h.ptr, _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(n), max_n, k_cache.shape[0],
                            _ptr(k_cache), _ptr(v_cache), _stream(stream)), h)


def selective_layer(h, layer, x, pos, n, k_cache, v_cache, n_ctx, dev_out=None, dev_mode=DEV_KV,
                    stream=None, max_n=None):
    """n: a device int32 count (then max_n bounds it) or a host int (copied into a device
    scalar, max_n = n)."""
    if isinstance(n, torch.Tensor):
        n_dev = n
        if max_n is None:
            raise ValueError("max_n is required with a device count")
    else:
        n_dev = torch.tensor([int(n)], dtype=torch.int32, device=x.device)
        max_n = int(n) if max_n is None else max_n
    _check(lib().selective_layer(h.ptr, layer, _ptr(x), _ptr(pos), _ptr(n_dev), max_n, _ptr(k_cache),
                                 _ptr(v_cache), n_ctx, _ptr(dev_out), dev_mode, _stream(stream)), h)


def importance_scores(hidden, n, n_layers, dim, out, stream=None):
    dt = BF16 if hidden.dtype == torch.bfloat16 else F32
    _check(lib().importance_scores(_ptr(hidden), n, n_layers, dim, dt, _ptr(out), _stream(stream)))


# ---------------------------------------------------------------- pool / requests / outputs
class PoolRef:
    """Host-side description of a chunk-KV pool (see blend_pool): tensors on the GPU, or
    pinned CPU tensors (location "host") that the GPU reads in place."""

    def __init__(self, k, v, tokens, prefix_len, entry_len, entry_row, present=None, location: str = "device"):
        self.k, self.v, self.tokens = k, v, tokens
        self._len = (C.c_int32 * len(entry_len))(*entry_len)
        self._row = (C.c_int64 * len(entry_row))(*entry_row)
        self._present = None if present is None else (C.c_uint8 * len(present))(*present)
        self.c = Pool(len(entry_len), prefix_len, self._len, self._row, self._present, k.shape[1],
                      k.data_ptr(), v.data_ptr(), tokens.data_ptr(),
                      {"device": POOL_DEVICE, "host": POOL_HOST}[location])
        self.entry_len = list(entry_len)
        self.prefix_len = prefix_len


class RequestRef:
    def __init__(self, chunk_ids: Sequence[int], query_tokens: torch.Tensor, mode: str = "ext",
                 rho_bp: int = 0, r1_bp: int = 0, window: int = 1, tau: int = 1,
                 budget_mode: str = "final", dev_mode: str = "kv", scores: Optional[torch.Tensor] = None,
                 stages: Optional[list] = None, group_rule: str = "window", tau_smooth: float = 0.4,
                 tau_cover_bp: int = 7000, max_span: int = 16, cap_bp: int = 0, epic_m: int = 0,
                 focus_layer: int = 0, focus_bp: int = 0):
        self.chunk_ids = list(chunk_ids)
        self._ids = (C.c_int32 * len(self.chunk_ids))(*self.chunk_ids)
        self.query = query_tokens
        self.scores = scores
        self.stages = stages or []
        st_layer = (C.c_int32 * 3)(*([int(f) for f, _ in self.stages] + [0] * (3 - len(self.stages))))
        st_pos = (C.c_void_p * 3)(*([p.data_ptr() if p.numel() else None for _, p in self.stages]
                                     + [None] * (3 - len(self.stages))))
        st_n = (C.c_int32 * 3)(*([int(p.numel()) for _, p in self.stages] + [0] * (3 - len(self.stages))))
        self.c = Request(len(self.chunk_ids), self._ids, int(query_tokens.numel()), query_tokens.data_ptr(),
                         MODES[mode], rho_bp, r1_bp, window, tau, BUDGETS[budget_mode], DEVMODES[dev_mode],
                         scores.data_ptr() if scores is not None else None, len(self.stages), st_layer,
                         st_pos, st_n, GROUP_RULES[group_rule], float(tau_smooth), tau_cover_bp, max_span, cap_bp,
                         epic_m, focus_layer, focus_bp)


class OutputsRef:
    def __init__(self, k, v, hidden, sel=None, n_sel=None, c1=None, n_c1=None, dev1=None, dev2=None,
                 q_last=None):
        self.t = dict(k=k, v=v, hidden=hidden, sel=sel, n_sel=n_sel, c1=c1, n_c1=n_c1, dev1=dev1, dev2=dev2,
                      q_last=q_last)
        self.c = Outputs(*[None if self.t[n] is None else self.t[n].data_ptr()
                           for n in ("k", "v", "hidden", "sel", "n_sel", "c1", "n_c1", "dev1", "dev2",
                                     "q_last")])

    def __getitem__(self, k):
        return self.t[k]


def _req_array(reqs):
    arr = (Request * len(reqs))()
    for i, r in enumerate(reqs):
        arr[i] = r.c
    return arr


def blend_assemble(h, reqs: Sequence[RequestRef], pool: PoolRef, out: OutputsRef, stream=None):
    _check(lib().blend_assemble(h.ptr, len(reqs), _req_array(reqs), C.byref(pool.c), C.byref(out.c),
                                _stream(stream)), h)


def blend_prefill(h, reqs: Sequence[RequestRef], pool: PoolRef, out: OutputsRef, stream=None):
    _check(lib().blend_prefill(h.ptr, len(reqs), _req_array(reqs), C.byref(pool.c), C.byref(out.c),
                               _stream(stream)), h)


def aux_attention_scores(h, reqs: Sequence[RequestRef], pool: PoolRef, out: OutputsRef, scores: torch.Tensor,
                         stream=None):
    _check(lib().aux_attention_scores(h.ptr, len(reqs), _req_array(reqs), C.byref(pool.c), C.byref(out.c),
                                      _ptr(scores), _stream(stream)), h)


def blend_ratio_controller(full_prefill_s: float, kv_bytes: float, load_bytes_per_s: float,
                           floor_bp: int = 1500) -> int:
    out = C.c_int32()
    _check(lib().blend_ratio_controller(full_prefill_s, kv_bytes, load_bytes_per_s, floor_bp, C.byref(out)))
    return out.value


def blend_pick_storage(full_prefill_s: float, kv_bytes: float, floor_bp: int, bytes_per_s, cost_per_byte) -> int:
    n = len(bytes_per_s)
    bw = (C.c_double * max(n, 1))(*bytes_per_s)
    cost = (C.c_double * max(n, 1))(*cost_per_byte)
    out = C.c_int32()
    _check(lib().blend_pick_storage(full_prefill_s, kv_bytes, floor_bp, n, bw, cost, C.byref(out)))
    return out.value


# ---------------------------------------------------------------- weight layout
def pack_weights(w: dict, device=None) -> dict:
    """Plain per-layer weights (synth.model_weights layout) -> the layout blend_weights
    documents: fused [q; k; v] rows, gate/up rows interleaved in blocks of GU_BLOCK."""
    dev = device or w["embed"].device
    wq, wk, wv = w["wq"], w["wk"], w["wv"]
    L, F, H = w["wg"].shape
    gu = torch.stack([w["wg"].reshape(L, F // GU_BLOCK, GU_BLOCK, H),
                      w["wu"].reshape(L, F // GU_BLOCK, GU_BLOCK, H)], dim=2).reshape(L, 2 * F, H)
    return {
        "embed": w["embed"].to(dev).contiguous(),
        "attn_norm": w["attn_norm"].to(dev).contiguous(),
        "w_qkv": torch.cat([wq, wk, wv], dim=1).to(dev).contiguous(),
        "w_o": w["wo"].to(dev).contiguous(),
        "mlp_norm": w["mlp_norm"].to(dev).contiguous(),
        "w_gu": gu.to(dev).contiguous(),
        "w_down": w["wd"].to(dev).contiguous(),
        "final_norm": w["final_norm"].to(dev).contiguous(),
    }
