"""The allocation-free router entry point against the regular one.

moe_route_noalloc serves callers that are handed inputs and outputs but
cannot allocate device memory for a workspace (a host framework that owns
every device buffer, or a path on which allocating is not allowed).  Its
scratch lives in a fixed array inside the library.  This test calls it
through the C ABI twice in a row, on two different inputs, and checks each
result against moe_route (which takes a caller-allocated workspace): expert
IDs must be identical and weights / decision gaps within the route tolerance
the other parity tests use.  A second case fills the array to its limit
(T = 64 tokens, E = 1024 experts: every byte of it) and then makes a one-token
call, which must ignore the larger call's leftovers; both are also checked
against the CPU oracle's top-k.  Kept in a file of its own that pytest
collects last; it builds its own inputs so it also passes when run alone.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity import W_ATOL, compare_routes
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


def test_noalloc_route_at_its_limit_then_one_token():
    """T = 64, E = 1024 (the whole 256 KB array), then T = 1 on the same array."""
    H, E, k = 1024, 1024, 10
    g = torch.Generator(device="cpu").manual_seed(2024)
    wr = (torch.randn((E, H), generator=g) * 0.02).to(torch.bfloat16).to(DEV)
    bias = (torch.randn((E,), generator=g) * 0.1).to(DEV)
    x64 = torch.randn((64, H), generator=g).to(torch.bfloat16).to(DEV)
    x1 = torch.randn((1, H), generator=g).to(torch.bfloat16).to(DEV)
    wr_bits = oracle.bf16_bits(wr)
    b_np = bias.cpu().numpy()
    for x in (x64, x1):
        ref_ids, ref_w, ref_gap = _regular(x, wr, bias, k)
        got_ids, got_w, got_gap = _noalloc_via_c_abi(x, wr, bias, k)
        torch.cuda.synchronize()
        assert torch.equal(got_ids, ref_ids), x.shape
        assert np.abs(got_w.cpu().numpy() - ref_w.cpu().numpy()).max() <= W_ATOL, x.shape
        o_ids, o_w, o_gap, o_L = oracle.route(oracle.bf16_bits(x), wr_bits, b_np, k)
        rep = compare_routes(got_ids.cpu().numpy(), got_w.cpu().numpy(), o_ids, o_w, o_gap, o_L)
        assert rep["checked"] + rep["near_tie"] == x.shape[0]
        assert rep["checked"] >= 0.9 * x.shape[0], rep


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
    # more experts than the router supports at all: rejected by that limit first
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros((1056, 256), dtype=torch.bfloat16, device=DEV)
    ids = torch.full((4, 4), -7, dtype=torch.int32, device=DEV)
    w = torch.zeros((4, 4), dtype=torch.float32, device=DEV)
    with pytest.raises(_lib.MoEError) as ei:
        _lib.moe_route_noalloc(x, wr, None, 4, ids, w, None)
    assert ei.value.status == _lib.MOE_ENOTSUP
    torch.cuda.synchronize()
    assert bool((ids == -7).all())
