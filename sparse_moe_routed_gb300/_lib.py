"""ctypes binding of libmoe: the same names as include/moe.h, marshalling only.

Every function takes torch tensors that already live on the GPU (PyTorch is
used here only for device memory and streams), passes their raw pointers to
the C ABI on the current stream and raises ``MoEError`` on a non-OK status.
No arithmetic happens in Python.  If the shared library is missing it is
built in-tree; if it cannot be built or loaded the call raises: there is no
CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

from . import build as _build

MOE_OK, MOE_EINVAL, MOE_ESHAPE, MOE_ERANGE, MOE_ECUDA, MOE_ENOTSUP, MOE_EDEVICE_TIMEOUT, MOE_EWORKSPACE = range(8)
MOE_DEV_BAD_EXPERT, MOE_DEV_NONFINITE, MOE_DEV_TIMEOUT, MOE_DEV_CACHE_FULL = 0x1, 0x2, 0x4, 0x8
MOE_W_BF16, MOE_W_INT4_G64, MOE_W_BF16_TILED, MOE_W_INT4_G64_TILED = 0, 1, 2, 3
MOE_CACHE_FIFO, MOE_CACHE_LRU, MOE_CACHE_SCORE = 0, 1, 2

HEADER = os.path.join(_build.INCLUDE, "moe.h")

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def declared_functions():
    """Names of the functions include/moe.h declares (parsed from the header)."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b((?:moe|route)_\w+)\s*\(", txt)))


def load(path: str | None = None):
    """Load (building first if needed) libmoe.so and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if path is None:
            path = _build.build()
        lib = C.CDLL(path)
        p, i, sz = C.c_void_p, C.c_int, C.c_size_t
        f = C.c_float
        sig = {
            "moe_abi_version": ([], i),
            "moe_status_str": ([i], C.c_char_p),
            "moe_device_sm_count": ([], i),
            "moe_route_workspace_size": ([i, i], sz),
            "moe_route": ([p, p, p, i, i, i, i, p, p, p, p, sz, p], i),
            "moe_route_noalloc": ([p, p, p, i, i, i, i, p, p, p, p], i),
            "moe_permute": ([p, i, i, i, p, i, p, p, p, p, p, p, p], i),
            "moe_permute_workspace_size": ([i, i, i], sz),
            "moe_permute_ws": ([p, i, i, i, p, i, p, p, p, p, p, p, sz, p, p], i),
            "moe_expert_gateup": ([p, p, i, i, i, i, i, p, p, p, p, p], i),
            "moe_expert_down": ([p, p, i, i, i, i, i, p, p, p, p, p], i),
            "moe_grouped_swiglu": ([p, p, i, i, i, i, i, p, p, p, p, p, p, p, p], i),
            "moe_expert_swiglu_fused": ([p, i, p, p, p, i, i, i, i, i, p, p, p, p, p, p, p], i),
            "moe_expert_swiglu_fused_weighted": ([p, i, p, p, p, i, i, i, i, i, p, p, p, p, p, p, p, p], i),
            "moe_combine_weighted": ([p, p, i, i, i, p, p, p, p, p], i),
            "moe_expert_int4_slots": ([i, p, p, i, i, i, i, p, i, p, p, p, p], i),
            "moe_expert_int4_fetch": ([p, p, i, i, i, i, p, p, i, p, p, p, p, p, p, p, p, p, p], i),
            "moe_route_permute": ([p, p, p, i, i, i, i, p, p, p, p, p, p, p, p, p], i),
            "moe_combine": ([p, p, p, i, i, i, p, p, p, p, p], i),
            "route_block_dedup": ([p, i, i, i, i, i, i, i, p, p, p, p, p, p], i),
            "moe_rmsnorm": ([p, p, f, i, i, p, p, p], i),
            "moe_pack_size": ([i, i, i, i, i], sz),
            "moe_pack_experts": ([i, p, p, i, i, i, i, p, sz, p], i),
            "moe_route_recall": ([p, p, i, i, p, p], i),
            "moe_cache_plan": ([p, i, p, p, i, p, i, f, p, p, p, p, p, p, p], i),
            "moe_cache_fetch": ([p, p, sz, sz, p, p, p, p, p, p], i),
            "moe_layer_stream": ([p, p, sz, sz, p, p, p], i),
            "moe_sidecar_prepare": ([p, p, i, i, i, p, p], i),
            "moe_sidecar_forward": ([p, p, p, p, i, i, i, i, i, i, p, p, p, p, p], i),
            "moe_stream_mode": ([i, i, C.c_double, C.c_double, C.c_double, C.c_double, p, p], i),
            "moe_expert_swiglu_cached": ([p, i, p, p, p, i, i, i, i, i, p, p, i, p, p, p, p, p, p, i, p, p, p, p, p],
                                         i),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(fn, st):
    if st != MOE_OK:
        msg = load().moe_status_str(st).decode()
        raise MoEError(fn, st, msg)


def status_str(st: int) -> str:
    return load().moe_status_str(st).decode()


def abi_version() -> int:
    return load().moe_abi_version()


def device_sm_count() -> int:
    return load().moe_device_sm_count()


def route_workspace_size(T: int, E: int) -> int:
    return load().moe_route_workspace_size(T, E)


def moe_route(x, w_router, bias, k, topk_ids, topk_w, gap, workspace, stream=None):
    T, H = x.shape
    E = w_router.shape[0]
    st = load().moe_route(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, _ptr(topk_ids), _ptr(topk_w),
                          _ptr(gap), _ptr(workspace), workspace.numel() * workspace.element_size()
                          if workspace is not None else 0, _stream(stream))
    _check("moe_route", st)


def moe_route_noalloc(x, w_router, bias, k, topk_ids, topk_w, gap, stream=None):
    """moe_route without a workspace: scratch lives in a fixed array in the
    library (T <= 64, E <= 1024), for callers that cannot allocate."""
    T, H = x.shape
    E = w_router.shape[0]
    st = load().moe_route_noalloc(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, _ptr(topk_ids), _ptr(topk_w),
                                  _ptr(gap), _stream(stream))
    _check("moe_route_noalloc", st)


def moe_permute(topk_ids, E, x, counts, offsets, perm, inv_perm, x_perm, dev_status, stream=None):
    T, k = topk_ids.shape
    H = x.shape[1] if x is not None else 0
    st = load().moe_permute(_ptr(topk_ids), T, k, E, _ptr(x), H, _ptr(counts), _ptr(offsets), _ptr(perm),
                            _ptr(inv_perm), _ptr(x_perm), _ptr(dev_status), _stream(stream))
    _check("moe_permute", st)


def moe_permute_workspace_size(T, k, E):
    return load().moe_permute_workspace_size(T, k, E)


def moe_permute_ws(topk_ids, E, x, counts, offsets, perm, inv_perm, x_perm, workspace, dev_status, stream=None):
    T, k = topk_ids.shape
    H = x.shape[1] if x is not None else 0
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = load().moe_permute_ws(_ptr(topk_ids), T, k, E, _ptr(x), H, _ptr(counts), _ptr(offsets), _ptr(perm),
                               _ptr(inv_perm), _ptr(x_perm), _ptr(workspace), nbytes, _ptr(dev_status),
                               _stream(stream))
    _check("moe_permute_ws", st)


def moe_expert_gateup(x_perm, offsets, E, H, I, w_gateup, h, dev_status, fmt=MOE_W_BF16, s_gateup=None,
                      stream=None):
    R = x_perm.shape[0]
    st = load().moe_expert_gateup(_ptr(x_perm), _ptr(offsets), R, E, H, I, fmt, _ptr(w_gateup), _ptr(s_gateup),
                                  _ptr(h), _ptr(dev_status), _stream(stream))
    _check("moe_expert_gateup", st)


def moe_expert_down(h, offsets, E, H, I, w_down, y_perm, dev_status, fmt=MOE_W_BF16, s_down=None, stream=None):
    R = h.shape[0]
    st = load().moe_expert_down(_ptr(h), _ptr(offsets), R, E, H, I, fmt, _ptr(w_down), _ptr(s_down),
                                _ptr(y_perm), _ptr(dev_status), _stream(stream))
    _check("moe_expert_down", st)


def moe_grouped_swiglu(x_perm, offsets, E, H, I, w_gateup, w_down, h, y_perm, dev_status, fmt=MOE_W_BF16,
                       s_gateup=None, s_down=None, stream=None):
    R = x_perm.shape[0]
    st = load().moe_grouped_swiglu(_ptr(x_perm), _ptr(offsets), R, E, H, I, fmt, _ptr(w_gateup), _ptr(s_gateup),
                                   _ptr(w_down), _ptr(s_down), _ptr(h), _ptr(y_perm), _ptr(dev_status),
                                   _stream(stream))
    _check("moe_grouped_swiglu", st)


def moe_expert_swiglu_fused(x_perm, offsets, E, H, I, w_gateup, w_down, h, y_perm, sync_ws, dev_status,
                            fmt=MOE_W_BF16_TILED, x=None, perm=None, k=0, stream=None):
    """Gate/up + SwiGLU + down in one launch; with x (and perm, k) it also
    gathers x_perm from x first."""
    R = x_perm.shape[0]
    st = load().moe_expert_swiglu_fused(_ptr(x), k, _ptr(perm), _ptr(x_perm), _ptr(offsets), R, E, H, I, fmt,
                                        _ptr(w_gateup), _ptr(w_down), _ptr(h), _ptr(y_perm), _ptr(sync_ws),
                                        _ptr(dev_status), _stream(stream))
    _check("moe_expert_swiglu_fused", st)


def moe_expert_swiglu_fused_weighted(x_perm, offsets, E, H, I, w_gateup, w_down, topk_w, h, yw_perm, sync_ws,
                                     dev_status, perm, k, fmt=MOE_W_BF16_TILED, x=None, stream=None):
    """moe_expert_swiglu_fused whose down epilogue stores bf16 rows already
    multiplied by their route weights (yw_perm [R, H] bf16)."""
    R = x_perm.shape[0]
    st = load().moe_expert_swiglu_fused_weighted(_ptr(x), k, _ptr(perm), _ptr(x_perm), _ptr(offsets), R, E, H, I,
                                                 fmt, _ptr(w_gateup), _ptr(w_down), _ptr(topk_w), _ptr(h),
                                                 _ptr(yw_perm), _ptr(sync_ws), _ptr(dev_status), _stream(stream))
    _check("moe_expert_swiglu_fused_weighted", st)


def moe_expert_int4_slots(kind, rows, offsets, E, H, I, pool, S, slot_of, out, dev_status, stream=None):
    """int4 gate/up (kind 0) or down (kind 1) with expert e's record at
    record slot_of[e] of an S-record pool (decode-sized launches)."""
    R = rows.shape[0]
    st = load().moe_expert_int4_slots(kind, _ptr(rows), _ptr(offsets), R, E, H, I, _ptr(pool), S, _ptr(slot_of),
                                      _ptr(out), _ptr(dev_status), _stream(stream))
    _check("moe_expert_int4_slots", st)


def moe_cache_plan(counts, slot_of, expert_of, hand, miss_list, miss_slot, stats, dev_status,
                   policy=MOE_CACHE_FIFO, decay=0.9, score=None, last_use=None, stream=None):
    E, S = counts.shape[0], expert_of.shape[0]
    st = load().moe_cache_plan(_ptr(counts), E, _ptr(slot_of), _ptr(expert_of), S, _ptr(hand), policy,
                               C.c_float(decay), _ptr(score), _ptr(last_use), _ptr(miss_list), _ptr(miss_slot),
                               _ptr(stats), _ptr(dev_status), _stream(stream))
    _check("moe_cache_plan", st)


def moe_cache_fetch(host_gateup, host_down, rec_gateup, rec_down, miss_list, miss_slot, stats, pool_gateup,
                    pool_down, stream=None):
    st = load().moe_cache_fetch(_ptr(host_gateup), _ptr(host_down), rec_gateup, rec_down, _ptr(miss_list),
                                _ptr(miss_slot), _ptr(stats), _ptr(pool_gateup), _ptr(pool_down), _stream(stream))
    _check("moe_cache_fetch", st)


def moe_sidecar_prepare(w_head, layer_emb, head_bias, stream=None):
    E, r = w_head.shape
    L = layer_emb.shape[0]
    st = load().moe_sidecar_prepare(_ptr(w_head), _ptr(layer_emb), E, r, L, _ptr(head_bias), _stream(stream))
    _check("moe_sidecar_prepare", st)


def moe_sidecar_forward(feat, w_trunk, w_head, head_bias, N, z, cand, cand_score, dev_status, stream=None):
    T, F = feat.shape
    r = w_trunk.shape[0]
    L, E = head_bias.shape
    st = load().moe_sidecar_forward(_ptr(feat), _ptr(w_trunk), _ptr(w_head), _ptr(head_bias), T, F, r, E, L, N,
                                    _ptr(z), _ptr(cand), _ptr(cand_score), _ptr(dev_status), _stream(stream))
    _check("moe_sidecar_forward", st)


MOE_STREAM_SELECTED, MOE_STREAM_LAYER = 0, 1


def moe_layer_stream(host_gateup, host_down, dev_gateup, dev_down, stream=None):
    """Copy a whole layer's packed records host -> device (copy engines)."""
    bg = host_gateup.numel() * host_gateup.element_size()
    bd = host_down.numel() * host_down.element_size()
    st = load().moe_layer_stream(_ptr(host_gateup), _ptr(host_down), bg, bd, _ptr(dev_gateup), _ptr(dev_down),
                                 _stream(stream))
    _check("moe_layer_stream", st)


def stream_mode(U, E, record_bytes, selected_gbs, layer_gbs, selected_overhead_us=0.0):
    """(mode, t_selected_us, t_layer_us) from moe_stream_mode."""
    ts, tl = C.c_double(), C.c_double()
    m = load().moe_stream_mode(U, E, float(record_bytes), float(selected_gbs), float(layer_gbs),
                               float(selected_overhead_us), C.byref(ts), C.byref(tl))
    if m < 0:
        raise ValueError("moe_stream_mode: argument out of range")
    return m, ts.value, tl.value


def moe_expert_swiglu_cached(x_perm, offsets, E, H, I, pool_gateup, pool_down, S, slot_of, h, y_perm, sync_ws,
                             dev_status, host_gateup=None, host_down=None, miss_list=None, miss_slot=None,
                             stats=None, wave=1 << 20, fmt=MOE_W_BF16_TILED, x=None, perm=None, k=0, stream=None):
    """moe_expert_swiglu_fused over slot pools; with host records it also
    fetches the planned misses in the same launch."""
    R = x_perm.shape[0]
    st = load().moe_expert_swiglu_cached(_ptr(x), k, _ptr(perm), _ptr(x_perm), _ptr(offsets), R, E, H, I, fmt,
                                         _ptr(pool_gateup), _ptr(pool_down), S, _ptr(slot_of), _ptr(host_gateup),
                                         _ptr(host_down), _ptr(miss_list), _ptr(miss_slot), _ptr(stats), wave,
                                         _ptr(h), _ptr(y_perm), _ptr(sync_ws), _ptr(dev_status), _stream(stream))
    _check("moe_expert_swiglu_cached", st)


def moe_route_permute(x, w_router, bias, k, topk_ids, topk_w, gap, counts, offsets, perm, inv_perm, dev_status,
                      stream=None):
    T, H = x.shape
    E = w_router.shape[0]
    st = load().moe_route_permute(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, _ptr(topk_ids), _ptr(topk_w),
                                  _ptr(gap), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv_perm),
                                  _ptr(dev_status), _stream(stream))
    _check("moe_route_permute", st)


def moe_combine(y_perm, inv_perm, topk_w, residual, out_bf16, out_f32, dev_status, stream=None):
    T, k = topk_w.shape
    H = y_perm.shape[1]
    st = load().moe_combine(_ptr(y_perm), _ptr(inv_perm), _ptr(topk_w), T, k, H, _ptr(residual), _ptr(out_bf16),
                            _ptr(out_f32), _ptr(dev_status), _stream(stream))
    _check("moe_combine", st)


def moe_combine_weighted(yw_perm, inv_perm, T, k, residual, out_bf16, out_f32, dev_status, stream=None):
    H = yw_perm.shape[1]
    st = load().moe_combine_weighted(_ptr(yw_perm), _ptr(inv_perm), T, k, H, _ptr(residual), _ptr(out_bf16),
                                     _ptr(out_f32), _ptr(dev_status), _stream(stream))
    _check("moe_combine_weighted", st)


def route_block_dedup(ids, E, block, H, I, mask, U, bytes2, bytes4, dev_status, stream=None):
    L, Tt, k = ids.shape
    st = load().route_block_dedup(_ptr(ids), L, Tt, k, E, block, H, I, _ptr(mask), _ptr(U), _ptr(bytes2),
                                  _ptr(bytes4), _ptr(dev_status), _stream(stream))
    _check("route_block_dedup", st)


def moe_rmsnorm(x, gamma, eps, out, raw_bf16=None, stream=None):
    T, H = x.shape
    st = load().moe_rmsnorm(_ptr(x), _ptr(gamma), float(eps), T, H, _ptr(out), _ptr(raw_bf16), _stream(stream))
    _check("moe_rmsnorm", st)


def moe_route_recall(pred_ids, ref_ids, hits, stream=None):
    T, k = ref_ids.shape
    st = load().moe_route_recall(_ptr(pred_ids), _ptr(ref_ids), T, k, _ptr(hits), _stream(stream))
    _check("moe_route_recall", st)


def pack_size(fmt_in: int, E: int, H: int, I: int, which: int) -> int:
    return load().moe_pack_size(fmt_in, E, H, I, which)


def moe_pack_experts(fmt_in, w, s, E, H, I, which, out=None, stream=None):
    """Pack one expert component (which = 0 gate/up, 1 down) into tile order;
    returns the packed uint8 tensor (allocated with torch if out is None)."""
    import torch
    n = pack_size(fmt_in, E, H, I, which)
    if out is None:
        out = torch.empty((n,), dtype=torch.uint8, device=w.device)
    st = load().moe_pack_experts(fmt_in, _ptr(w), _ptr(s), E, H, I, which, _ptr(out), out.numel(), _stream(stream))
    _check("moe_pack_experts", st)
    return out

