"""Thin ctypes binding of libmoe_gb300.so: argument marshalling only.

Every function here has the name of the C entry point it calls and takes
torch tensors (device memory) where the C call takes device pointers. There is
no compute in Python and no fallback: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from .build import LIB_PATH

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
                6: "MOE_ERR_DEVICE_CHECK", 7: "MOE_ERR_STASH_FULL"}

# every exported entry point of include/moe_abi.h
ENTRY_POINTS = (
    "moe_query_sizes", "moe_route", "moe_route_replay", "moe_route_aux", "moe_route_aux_bwd",
    "moe_permute", "moe_permute_noalloc", "moe_permute_noalloc_status",
    "moe_quantize_weights", "moe_load_fp8_weights", "moe_grouped_ffn_fwd", "moe_unpermute",
    "moe_unpermute_bwd", "moe_grouped_ffn_dgrad", "moe_grouped_ffn_wgrad", "moe_grouped_ffn_bwd",
    "moe_grouped_ffn_fwd_reordered", "moe_unpermute_bwd_reordered",
    "moe_grouped_ffn_dgrad_reordered", "moe_route_bwd", "moe_permute_bwd",
    "moe_router_wgrad", "moe_layer_fwd", "moe_layer_bwd", "moe_stash_release",
    "moe_last_device_status",
    "moe_clear_device_status", "moe_check_bounded_wait", "moe_status_string",
)


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}: {status_string(code)}")


class MoEConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("F", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("topk_groups", ctypes.c_int32), ("group_score", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("row_align", ctypes.c_int32),
                ("weights_in_expert", ctypes.c_int32), ("recompute_h", ctypes.c_int32),
                ("stash_pool_pages", ctypes.c_int32)]


class MoESizes(ctypes.Structure):
    _fields_ = [("rows_max", ctypes.c_int64), ("groups", ctypes.c_int64),
                ("capacity", ctypes.c_int64), ("scratch_bytes", ctypes.c_int64),
                ("stash_table_len", ctypes.c_int64)]


_P = ctypes.c_void_p


class MoEParams(ctypes.Structure):
    _fields_ = [("W_r", _P), ("bias", _P), ("W13", _P), ("W2", _P)]


FWD_FIELDS = ("logits", "idx", "w", "counts", "offsets", "row_of", "token_of", "sel_offsets",
              "sel_tokens", "x_perm", "GU", "h", "y_perm")
BWD_FIELDS = ("dO_perm", "dw", "dlogits", "dGU", "dX_perm")


# the paged stash's per-layer page table and the pool's page counter
STASH_FIELDS = ("stash_table", "stash_top")


class MoEFwdState(ctypes.Structure):
    _fields_ = [(n, _P) for n in FWD_FIELDS + STASH_FIELDS]


class MoEBwdState(ctypes.Structure):
    _fields_ = [(n, _P) for n in BWD_FIELDS]


_lib = None


def lib():
    """Loads the library once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m routing_dispatch_expert_router_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name in ENTRY_POINTS:
            f = getattr(L, name)
            f.restype = ctypes.c_int
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(name: str, code: int):
    if code != MOE_OK:
        raise MoEError(name, code)


def config(shape) -> MoEConfig:
    """moe_config from any object with the layer's fields (e.g. workloads.MoEShape)."""
    return MoEConfig(T=shape.T, H=shape.H, E=shape.E, k=shape.k, F=shape.F,
                     n_shared=getattr(shape, "n_shared", 0),
                     score_fn=getattr(shape, "score_fn", 0),
                     n_groups=getattr(shape, "n_groups", 1),
                     topk_groups=getattr(shape, "topk_groups", 1),
                     group_score=getattr(shape, "group_score", 0),
                     route_scale=getattr(shape, "route_scale", 1.0),
                     dtype=getattr(shape, "dtype", 0),
                     capacity_factor=getattr(shape, "capacity_factor", 0.0),
                     row_align=getattr(shape, "row_align", 128),
                     weights_in_expert=getattr(shape, "weights_in_expert", 0),
                     recompute_h=getattr(shape, "recompute_h", 0),
                     stash_pool_pages=getattr(shape, "stash_pool_pages", 0))


def _cfg(c) -> MoEConfig:
    return c if isinstance(c, MoEConfig) else config(c)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name, *args):
    f = getattr(lib(), name)
    conv = []
    for a in args:
        if isinstance(a, ctypes.Structure):
            conv.append(ctypes.byref(a))
        elif isinstance(a, float):
            conv.append(ctypes.c_float(a))
        elif a is None or isinstance(a, int):
            conv.append(ctypes.c_void_p(a))
        else:
            conv.append(ctypes.c_void_p(_ptr(a)))
    _check(name, f(*conv))


# ------------------------------------------------------------------ entry points
def moe_query_sizes(cfg) -> MoESizes:
    out = MoESizes()
    _check("moe_query_sizes", lib().moe_query_sizes(ctypes.byref(_cfg(cfg)), ctypes.byref(out)))
    return out


def moe_route(cfg, x, W_r, bias, logits, idx, w, scratch, stream=None):
    _call("moe_route", _cfg(cfg), x, W_r, bias, logits, idx, w, scratch, _stream(stream))


def moe_route_replay(cfg, x, W_r, bias, idx, logits, w, scratch, stream=None):
    """Router Replay: the given experts idx [T,k] (input) instead of the top-k."""
    _call("moe_route_replay", _cfg(cfg), x, W_r, bias, idx, logits, w, scratch, _stream(stream))


def moe_route_aux(cfg, logits, bias, idx, coeff, bias_rate, sel_counts, p_mean, loss, bias_out,
                  scratch, stream=None):
    """Load-balancing loss statistics, loss and (bias_out not None) the bias update."""
    _call("moe_route_aux", _cfg(cfg), logits, bias, idx, float(coeff), float(bias_rate),
          sel_counts, p_mean, loss, bias_out, scratch, _stream(stream))


def moe_route_aux_bwd(cfg, x, logits, bias, W_r, sel_counts, coeff, dloss, dlogits_aux, dx,
                      dW_r, scratch, stream=None):
    """The loss's gradient: writes dlogits_aux, adds into dx and dW_r."""
    _call("moe_route_aux_bwd", _cfg(cfg), x, logits, bias, W_r, sel_counts, float(coeff),
          float(dloss), dlogits_aux, dx, dW_r, scratch, _stream(stream))


def moe_permute(cfg, x, idx, counts, offsets, row_of, token_of, sel_offsets, sel_tokens, x_perm,
                scratch, stream=None):
    _call("moe_permute", _cfg(cfg), x, idx, counts, offsets, row_of, token_of, sel_offsets,
          sel_tokens, x_perm, scratch, _stream(stream))


def moe_permute_noalloc(cfg, x, idx, counts, offsets, row_of, token_of, sel_offsets, sel_tokens,
                        x_perm, stream=None):
    """moe_permute with the library's own fixed scratch array (allocates nothing)."""
    _call("moe_permute_noalloc", _cfg(cfg), x, idx, counts, offsets, row_of, token_of,
          sel_offsets, sel_tokens, x_perm, _stream(stream))


def moe_quantize_weights(cfg, W13, W2, scratch, stream=None):
    """FP8 mode: the E4M3 weights (and scales) in scratch; no-op in bf16 mode."""
    _call("moe_quantize_weights", _cfg(cfg), W13, W2, scratch, _stream(stream))


def moe_load_fp8_weights(cfg, W13_e4m3, W13_scale, W2_e4m3, W2_scale, scratch, stream=None):
    _call("moe_load_fp8_weights", _cfg(cfg), W13_e4m3, W13_scale, W2_e4m3, W2_scale, scratch,
          _stream(stream))


def moe_permute_noalloc_status(stream=None) -> int:
    """The status word the last moe_permute_noalloc call left (synchronises)."""
    code = ctypes.c_int32(0)
    _check("moe_permute_noalloc_status",
           lib().moe_permute_noalloc_status(ctypes.byref(code), ctypes.c_void_p(_stream(stream))))
    return code.value


def moe_grouped_ffn_fwd(cfg, x_perm, counts, offsets, W13, W2, GU, h, y_perm, scratch,
                        stream=None):
    _call("moe_grouped_ffn_fwd", _cfg(cfg), x_perm, counts, offsets, W13, W2, GU, h, y_perm,
          scratch, _stream(stream))


def moe_unpermute(cfg, y_perm, row_of, w, offsets, out, stream=None):
    _call("moe_unpermute", _cfg(cfg), y_perm, row_of, w, offsets, out, _stream(stream))


def moe_unpermute_bwd(cfg, dY, y_perm, row_of, w, counts, offsets, dO_perm, dw, scratch,
                      stream=None):
    _call("moe_unpermute_bwd", _cfg(cfg), dY, y_perm, row_of, w, counts, offsets, dO_perm, dw,
          scratch, _stream(stream))


def moe_grouped_ffn_bwd(cfg, dO_perm, x_perm, GU, h, counts, offsets, token_of, dlogits, W_r,
                        W13, W2, dGU, dX_perm, dW13, dW2, scratch, stream=None):
    _call("moe_grouped_ffn_bwd", _cfg(cfg), dO_perm, x_perm, GU, h, counts, offsets, token_of,
          dlogits, W_r, W13, W2, dGU, dX_perm, dW13, dW2, scratch, _stream(stream))


def moe_grouped_ffn_dgrad(cfg, dO_perm, GU, h, counts, offsets, token_of, dlogits, W_r, W13, W2,
                          dGU, dX_perm, scratch, stream=None):
    """h: None, or the buffer to rewrite h into from GU (fine-grained recompute)."""
    _call("moe_grouped_ffn_dgrad", _cfg(cfg), dO_perm, GU, h, counts, offsets, token_of, dlogits,
          W_r, W13, W2, dGU, dX_perm, scratch, _stream(stream))


def moe_grouped_ffn_wgrad(cfg, dO_perm, x_perm, h, dGU, counts, offsets, dW13, dW2, scratch,
                          stream=None):
    _call("moe_grouped_ffn_wgrad", _cfg(cfg), dO_perm, x_perm, h, dGU, counts, offsets, dW13,
          dW2, scratch, _stream(stream))


def moe_grouped_ffn_fwd_reordered(cfg, x_perm, counts, offsets, token_of, row_of, w, W13, W2,
                                  GU, h, y_perm, scratch, stream=None):
    """Forward GEMMs with the routing weight inside the expert (h = w silu(G) U)."""
    _call("moe_grouped_ffn_fwd_reordered", _cfg(cfg), x_perm, counts, offsets, token_of, row_of,
          w, W13, W2, GU, h, y_perm, scratch, _stream(stream))


def moe_unpermute_bwd_reordered(cfg, dY, row_of, counts, offsets, dO_perm, stream=None):
    _call("moe_unpermute_bwd_reordered", _cfg(cfg), dY, row_of, counts, offsets, dO_perm,
          _stream(stream))


def moe_grouped_ffn_dgrad_reordered(cfg, dO_perm, GU, h, counts, offsets, token_of, row_of,
                                    logits, idx, w, W_r, W13, W2, dGU, dX_perm, dw, dlogits,
                                    scratch, stream=None):
    _call("moe_grouped_ffn_dgrad_reordered", _cfg(cfg), dO_perm, GU, h, counts, offsets,
          token_of, row_of, logits, idx, w, W_r, W13, W2, dGU, dX_perm, dw, dlogits, scratch,
          _stream(stream))


def moe_route_bwd(cfg, logits, idx, w, dw, dlogits, stream=None):
    _call("moe_route_bwd", _cfg(cfg), logits, idx, w, dw, dlogits, _stream(stream))


def moe_permute_bwd(cfg, dX_perm, row_of, offsets, idx, dlogits, W_r, dx, stream=None):
    _call("moe_permute_bwd", _cfg(cfg), dX_perm, row_of, offsets, idx, dlogits, W_r, dx,
          _stream(stream))


def moe_router_wgrad(cfg, x, sel_offsets, sel_tokens, dlogits, dW_r, scratch, stream=None):
    _call("moe_router_wgrad", _cfg(cfg), x, sel_offsets, sel_tokens, dlogits, dW_r, scratch,
          _stream(stream))


def moe_layer_fwd(cfg, params: MoEParams, x, out, fwd: MoEFwdState, scratch, stream=None):
    _call("moe_layer_fwd", _cfg(cfg), params, x, out, fwd, scratch, _stream(stream))


def moe_layer_bwd(cfg, params: MoEParams, x, dY, fwd: MoEFwdState, bwd: MoEBwdState, dx, dW_r,
                  dW13, dW2, scratch, stream=None):
    _call("moe_layer_bwd", _cfg(cfg), params, x, dY, fwd, bwd, dx, dW_r, dW13, dW2, scratch,
          _stream(stream))


def moe_stash_release(cfg, fwd: MoEFwdState, stream=None):
    _call("moe_stash_release", _cfg(cfg), fwd, _stream(stream))


def moe_last_device_status(scratch, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check("moe_last_device_status",
           lib().moe_last_device_status(ctypes.c_void_p(_ptr(scratch)), ctypes.byref(code),
                                        ctypes.c_void_p(_stream(stream))))
    return code.value


def moe_check_bounded_wait(scratch, budget_cycles: int, stream=None):
    f = lib().moe_check_bounded_wait
    _check("moe_check_bounded_wait",
           f(ctypes.c_void_p(_ptr(scratch)), ctypes.c_int64(int(budget_cycles)),
             ctypes.c_void_p(_stream(stream))))


def moe_clear_device_status(scratch, stream=None):
    _call("moe_clear_device_status", scratch, _stream(stream))


# ------------------------------------------------------------------ buffers
@dataclass
class LayerBuffers:
    """Caller-owned device buffers of one layer, sized by moe_query_sizes."""
    sizes: MoESizes
    fwd: dict
    bwd: dict
    scratch: torch.Tensor
    fwd_struct: MoEFwdState
    bwd_struct: MoEBwdState


@dataclass
class StashPool:
    """The rows layers keep for their backward, in pages of 128 rows shared by
    the layers of a step: x_perm, GU, h, y_perm with (pages + 1) * 128 rows
    (the last page is the spill page) and the device page counter."""
    pages: int
    tensors: dict
    top: torch.Tensor


def alloc_stash_pool(cfg, pages: int, device="cuda") -> StashPool:
    c = _cfg(cfg)
    if int(pages) < 1:
        raise ValueError("a stash pool has at least one page (stash_pool_pages = 0 means no pool)")
    rows = (int(pages) + 1) * 128
    bf = torch.bfloat16
    e = lambda *s: torch.empty(*s, dtype=bf, device=device)  # noqa: E731
    t = dict(x_perm=e(rows, c.H), GU=e(rows, 2 * c.F), h=e(rows, c.F), y_perm=e(rows, c.H))
    return StashPool(int(pages), t, torch.zeros(1, dtype=torch.int32, device=device))


def alloc_buffers(cfg, device="cuda", backward: bool = True,
                  pool: StashPool | None = None) -> LayerBuffers:
    """Allocates (torch.empty / zeros) every buffer the layer calls need; with
    a stash pool (cfg.stash_pool_pages == pool.pages) the four stashed row
    tensors are the pool's and the layer gets its own page table."""
    c = _cfg(cfg)
    sz = moe_query_sizes(c)
    R, G = int(sz.rows_max), int(sz.groups)
    T, H, E, k, F = c.T, c.H, c.E, c.k, c.F
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    e = lambda *s, dt: torch.empty(*s, dtype=dt, device=device)  # noqa: E731
    fwd = dict(logits=e(T, E, dt=f32), idx=e(T, k, dt=i32), w=e(T, k, dt=f32),
               counts=e(G, dt=i32), offsets=e(G + 1, dt=i32), row_of=e(T, k, dt=i32),
               token_of=e(R, dt=i32), sel_offsets=e(E + 1, dt=i32),
               sel_tokens=e(max(T * k, 1), dt=i32))
    if pool is None:
        fwd.update(x_perm=e(R, H, dt=bf), GU=e(R, 2 * F, dt=bf), h=e(R, F, dt=bf),
                   y_perm=e(R, H, dt=bf))
    else:
        if c.stash_pool_pages < 1 or c.stash_pool_pages != pool.pages:
            raise ValueError("cfg.stash_pool_pages must equal the pool's pages (at least 1)")
        fwd.update(pool.tensors)
        fwd.update(stash_table=e(int(sz.stash_table_len), dt=i32), stash_top=pool.top)
    bwd = {}
    if backward:
        bwd = dict(dO_perm=e(R, H, dt=bf), dw=e(T, k, dt=f32), dlogits=e(T, E, dt=f32),
                   dGU=e(R, 2 * F, dt=bf), dX_perm=e(R, H, dt=bf))
    scratch = torch.zeros(int(sz.scratch_bytes), dtype=torch.uint8, device=device)
    fs = MoEFwdState(**{n: (fwd[n].data_ptr() if n in fwd else 0)
                        for n in FWD_FIELDS + STASH_FIELDS})
    bs = MoEBwdState(**{n: (bwd[n].data_ptr() if bwd else 0) for n in BWD_FIELDS})
    return LayerBuffers(sz, fwd, bwd, scratch, fs, bs)


def params(W_r, bias, W13, W2) -> MoEParams:
    return MoEParams(W_r=_ptr(W_r), bias=_ptr(bias), W13=_ptr(W13), W2=_ptr(W2))
