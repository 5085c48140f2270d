"""The allocation-free router entry point against the regular one.

moe_route_noalloc serves callers that are handed inputs and outputs but
cannot allocate device memory for a workspace (a host framework that owns
every device buffer, or a path on which allocating is not allowed).  Its
scratch lives in a fixed array inside the library.  This test calls it
through the C ABI twice in a row, on two different inputs, and checks each
result against moe_route (which takes a caller-allocated workspace): expert
IDs must be identical and weights / decision gaps within the route tolerance
the other parity tests use.  Kept in a file of its own that pytest collects
last; it builds its own inputs so it also passes when run alone.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as wl
from parity import W_ATOL
from sparse_moe_routed_gb300 import _lib

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(which):
    if which == "decode":
        x = wl.token_batch(wl.DECODE, DEV, index=3)
        wr = wl.predictor_weights(wl.DECODE.H, wl.DECODE.E, layer=7, device=DEV)  # an [E,H] N(0,0.02) matrix
        bias = wl.zipf_bias(wl.DECODE.E, seed=11).to(DEV)
        return x, wr, bias, wl.DECODE.k
    d = wl.layer_inputs(wl.TINY, DEV)
    return d["x"], d["w_router"], None, wl.TINY.k


def _regular(x, wr, bias, k):
    T, E = x.shape[0], wr.shape[0]
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    gap = torch.empty((T,), dtype=torch.float32, device=DEV)
    ws = torch.empty((_lib.route_workspace_size(T, E),), dtype=torch.uint8, device=DEV)
    _lib.moe_route(x, wr, bias, k, ids, w, gap, ws)
    return ids, w, gap


def _noalloc_via_c_abi(x, wr, bias, k):
    T, H = x.shape
    E = wr.shape[0]
    ids = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device=DEV)
    gap = torch.full((T,), float("nan"), dtype=torch.float32, device=DEV)
    P = lambda t: None if t is None else C.c_void_p(t.data_ptr())
    st = _lib.load().moe_route_noalloc(P(x), P(wr), P(bias), T, H, E, k, P(ids), P(w), P(gap),
                                       C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.MOE_OK, _lib.status_str(st)
    return ids, w, gap


def test_noalloc_route_matches_regular_route_twice():
    for which in ("decode", "tiny"):
        x, wr, bias, k = _inputs(which)
        ref_ids, ref_w, ref_gap = _regular(x, wr, bias, k)
        got_ids, got_w, got_gap = _noalloc_via_c_abi(x, wr, bias, k)
        torch.cuda.synchronize()
        assert torch.equal(got_ids, ref_ids), which
        assert np.abs(got_w.cpu().numpy() - ref_w.cpu().numpy()).max() <= W_ATOL, which
        assert np.allclose(got_gap.cpu().numpy(), ref_gap.cpu().numpy(), rtol=0, atol=W_ATOL), which


def test_noalloc_route_rejects_sizes_beyond_its_array():
    x = torch.zeros((65, 256), dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros((64, 256), dtype=torch.bfloat16, device=DEV)
    ids = torch.full((65, 4), -7, dtype=torch.int32, device=DEV)
    w = torch.zeros((65, 4), dtype=torch.float32, device=DEV)
    with pytest.raises(_lib.MoEError) as ei:
        _lib.moe_route_noalloc(x, wr, None, 4, ids, w, None)
    assert ei.value.status == _lib.MOE_EWORKSPACE
    torch.cuda.synchronize()
    assert bool((ids == -7).all())
