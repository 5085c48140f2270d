"""Failure detection without a GPU fault.

- A bounded device wait that runs out: the cached contraction is handed a
  fetch plan whose miss entry names no expert, so the landed-piece word of
  the expert it would have fetched is never written.  The producer waiting
  on it gives up after its limit (two seconds), flags MOE_DEV_TIMEOUT, every
  other role of the launch sees the abort and leaves, the last CTA out still
  resets the sync words, and the next call on the same buffers is correct.
- Errors injected on the host between calls (a call the library rejects, an
  allocation that fails) leave the layer usable.
"""
import pytest
import torch

import workloads as wl
from sparse_moe_routed_gb300 import MoELayer, _lib, pack_layer_experts

pytestmark = pytest.mark.gpu
DEV = "cuda"
CFG = wl.LayerConfig("fail_small", T=8, H=256, E=64, k=4, I=128, bias=None, seed=41)


def packed():
    d = wl.layer_inputs(CFG, DEV, with_x=False)
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, CFG.E, CFG.H, CFG.I)
    torch.cuda.synchronize()
    return d, gu, dn


def test_bounded_wait_runs_out_and_the_next_call_is_clean():
    d, gu, dn = packed()
    E, H, I = CFG.E, CFG.H, CFG.I
    # rows of experts 0, 7, 21 and the last one (which the bad plan marks as
    # being fetched)
    counts = torch.zeros(E, dtype=torch.int32)
    counts[[0, 7, 21, E - 1]] = torch.tensor([3, 2, 1, 2], dtype=torch.int32)
    R = int(counts.sum())
    offsets = torch.zeros(E + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0)
    offsets = offsets.to(DEV)
    x_perm = torch.randn((R, H), device=DEV).to(torch.bfloat16)
    S = E
    slot_of = torch.arange(E, dtype=torch.int32, device=DEV)  # every expert resident in slot e
    host_gu = gu.cpu().pin_memory()
    host_dn = dn.cpu().pin_memory()
    miss_list = torch.tensor([E + 5], dtype=torch.int32, device=DEV)  # names no expert
    miss_slot = torch.tensor([0], dtype=torch.int32, device=DEV)
    stats = torch.tensor([0, 1, 0, 0], dtype=torch.int32, device=DEV)
    sync = torch.zeros(E * (1 + I // 64 + H // 128) + 4, dtype=torch.int32, device=DEV)
    h = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((R, H), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    _lib.moe_expert_swiglu_cached(x_perm, offsets, E, H, I, gu, dn, S, slot_of, h, y, sync, st,
                                  host_gateup=host_gu, host_down=host_dn, miss_list=miss_list,
                                  miss_slot=miss_slot, stats=stats, wave=1)
    torch.cuda.synchronize()  # returns: the wait was bounded
    s = int(st.item())
    assert s & _lib.MOE_DEV_TIMEOUT and s & _lib.MOE_DEV_BAD_EXPERT
    assert int(sync.abs().sum().item()) == 0  # sync words reset on the way out

    # the context and the buffers are usable: a clean call matches the
    # resident contraction bit for bit
    st.zero_()
    stats.zero_()
    _lib.moe_expert_swiglu_cached(x_perm, offsets, E, H, I, gu, dn, S, slot_of, h, y, sync, st,
                                  host_gateup=host_gu, host_down=host_dn, miss_list=miss_list,
                                  miss_slot=miss_slot, stats=stats, wave=1)
    h2 = torch.empty_like(h)
    y2 = torch.empty_like(y)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    sync2 = torch.zeros(E + 3, dtype=torch.int32, device=DEV)
    _lib.moe_expert_swiglu_fused(x_perm, offsets, E, H, I, gu, dn, h2, y2, sync2, st2)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))


def test_rejected_call_between_calls_leaves_the_layer_usable():
    d, gu, dn = packed()
    lay = MoELayer(d["w_router"], d["bias"], gu, dn, CFG.k, CFG.T, fmt=_lib.MOE_W_BF16_TILED, I=CFG.I)
    x = wl.token_batch(CFG, DEV, index=1, T=CFG.T)
    want = lay.forward(x).clone()
    # inject: a call the library rejects on the host (no experts), between
    # two layer calls on the same buffers
    with pytest.raises(_lib.MoEError) as ei:
        _lib.moe_permute(lay.ids, 0, None, lay.counts, lay.offsets, lay.perm, lay.inv, None, lay.status)
    assert ei.value.status == _lib.MOE_ESHAPE
    got = lay.forward(x).clone()
    torch.cuda.synchronize()
    assert lay.read_status() == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_allocation_denial_is_an_error_not_a_half_built_layer(monkeypatch):
    d, gu, dn = packed()
    real_empty = torch.empty
    calls = {"n": 0}

    def deny(*a, **kw):
        calls["n"] += 1
        if calls["n"] == 5:
            raise torch.cuda.OutOfMemoryError("allocation denied (injected)")
        return real_empty(*a, **kw)

    monkeypatch.setattr(torch, "empty", deny)
    with pytest.raises(torch.cuda.OutOfMemoryError):
        MoELayer(d["w_router"], d["bias"], gu, dn, CFG.k, CFG.T, fmt=_lib.MOE_W_BF16_TILED, I=CFG.I)
    monkeypatch.setattr(torch, "empty", real_empty)
    lay = MoELayer(d["w_router"], d["bias"], gu, dn, CFG.k, CFG.T, fmt=_lib.MOE_W_BF16_TILED, I=CFG.I)
    out = lay.forward(wl.token_batch(CFG, DEV, index=2, T=CFG.T))
    torch.cuda.synchronize()
    assert lay.read_status() == 0 and torch.isfinite(out.float()).all()
