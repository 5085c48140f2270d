"""GPU checks of the fused contraction's row gather (moe_expert_swiglu_fused
with x given).

With x, the persistent launch first writes x_perm[s] = x[perm[s] / k] itself
and then runs gate/up + SwiGLU + down.  The gather is integer data movement
and the contraction's arithmetic is unchanged, so x_perm, h and y_perm must
equal, bit for bit, what moe_permute's gather followed by the same launch
without x produces on the same seeded routes.  The contraction itself is
graded against the oracle in test_gpu_layer.py.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from parity import assert_output_close
from sparse_moe_routed_gb300 import _lib, pack_layer_experts

pytestmark = pytest.mark.gpu

DEV = "cuda"
_W = {}


def weights(name):
    if name not in _W:
        cfg = wl.CONFIGS[name]
        d = wl.layer_inputs(cfg, DEV)
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
        torch.cuda.synchronize()
        _W[name] = (cfg, gu, dn)
    return _W[name]


def permuted(cfg, T, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(cfg.E, size=cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    R = T * cfg.k
    b = {"ids": torch.from_numpy(ids).to(DEV), "R": R,
         "counts": torch.empty((cfg.E,), dtype=torch.int32, device=DEV),
         "offsets": torch.empty((cfg.E + 1,), dtype=torch.int32, device=DEV),
         "perm": torch.empty((R,), dtype=torch.int32, device=DEV),
         "inv": torch.empty((R,), dtype=torch.int32, device=DEV),
         "st": torch.zeros((1,), dtype=torch.int32, device=DEV),
         "x": wl.token_batch(cfg, DEV, index=seed, T=T)}
    _lib.moe_permute(b["ids"], cfg.E, None, b["counts"], b["offsets"], b["perm"], b["inv"], None, b["st"])
    return b


def run(cfg, gu, dn, b, gather, perm=None, sync=None):
    R, E, H, I = b["R"], cfg.E, cfg.H, cfg.I
    xp = torch.full((R, H), -7.0, dtype=torch.bfloat16, device=DEV)
    h = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((R, H), dtype=torch.float32, device=DEV)
    if sync is None:
        sync = torch.zeros((E + 3,), dtype=torch.int32, device=DEV)
    perm = b["perm"] if perm is None else perm
    if gather:
        _lib.moe_expert_swiglu_fused(xp, b["offsets"], E, H, I, gu, dn, h, y, sync, b["st"], x=b["x"], perm=perm,
                                     k=cfg.k)
    else:
        _lib.moe_permute(b["ids"], E, b["x"], b["counts"], b["offsets"], b["perm"], b["inv"], xp, b["st"])
        _lib.moe_expert_swiglu_fused(xp, b["offsets"], E, H, I, gu, dn, h, y, sync, b["st"])
    torch.cuda.synchronize()
    return xp, h, y, sync


def same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16)) if a.dtype == torch.bfloat16 else \
        torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("name,T", [("tiny", 16), ("tiny", 3), ("decode", 16), ("decode", 37), ("decode", 1),
                                    ("decode", 409)])
def test_gather_in_launch_bitwise(name, T):
    cfg, gu, dn = weights(name)
    b = permuted(cfg, T, seed=T + 11)
    xp0, h0, y0, _ = run(cfg, gu, dn, b, gather=False)
    sync = torch.zeros((cfg.E + 3,), dtype=torch.int32, device=DEV)
    for _ in range(2):  # two calls in a row on one sync_ws
        xp1, h1, y1, sync = run(cfg, gu, dn, b, gather=True, sync=sync)
        assert b["st"].item() == 0
        assert same(xp1, xp0) and same(h1, h0) and same(y1, y0)
        assert int(sync.abs().sum().item()) == 0


def test_gather_skips_out_of_range_perm_entry():
    """A permutation entry out of range leaves that row of x_perm untouched
    (as moe_permute's gather does); every other row is gathered."""
    cfg, gu, dn = weights("tiny")
    b = permuted(cfg, 16, seed=4)
    bad = b["perm"].clone()
    bad[5] = b["R"] + 3
    xp, _, _, sync = run(cfg, gu, dn, b, gather=True, perm=bad)
    assert b["st"].item() == 0
    perm = b["perm"].cpu().numpy()
    x = b["x"]
    for s in range(b["R"]):
        if s == 5:
            assert torch.all(xp[s] == -7.0)
        else:
            assert same(xp[s], x[perm[s] // cfg.k])
    assert int(sync.abs().sum().item()) == 0


@pytest.mark.parametrize("name,T,gather", [("decode", 16, True), ("decode", 410, False), ("prefill", 4096, False),
                                           ("tiny", 16, False), ("prefill", 13108, False)])
def test_weighted_outputs_carry_the_route_weights(name, T, gather):
    """moe_expert_swiglu_fused_weighted applies each slot's route weight in
    the gate/up epilogue (h' = bf16(w * silu(g) * u)) and stores the down
    projection of h' as bf16 rows.  Against the unweighted launch on the same
    routes: h' is within two bf16 roundings (2^-8 relative each) of w * h, and the rows within the
    layer tolerance of w * y; the launch is deterministic (two calls, same
    bits) and leaves its sync words zero."""
    cfg = wl.with_tokens(wl.CONFIGS[name], T) if name != "tiny" else wl.TINY
    if name == "prefill":
        d = wl.layer_inputs(wl.with_tokens(cfg, 16), DEV, with_x=False)
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
        del d
    else:
        _, gu, dn = weights(name)
    b = permuted(cfg, T, seed=T + 5)
    R, E, H, I = b["R"], cfg.E, cfg.H, cfg.I
    xp0, h0, y0, _ = run(cfg, gu, dn, b, gather=False)
    topk_w = torch.rand((T, cfg.k), device=DEV)
    w_slot = topk_w.view(-1)[b["perm"].long()].unsqueeze(1)
    xp = xp0.clone() if not gather else torch.empty_like(xp0)
    h = torch.empty_like(h0)
    yw = torch.full((R, H), -3.0, dtype=torch.bfloat16, device=DEV)
    sync = torch.zeros((E + 3,), dtype=torch.int32, device=DEV)
    prev = None
    for _ in range(2):
        _lib.moe_expert_swiglu_fused_weighted(xp, b["offsets"], E, H, I, gu, dn, topk_w, h, yw, sync, b["st"],
                                              perm=b["perm"], k=cfg.k, x=b["x"] if gather else None)
        torch.cuda.synchronize()
        assert b["st"].item() == 0
        assert int(sync.abs().sum().item()) == 0
        wh = (h0.float() * w_slot).double()
        assert bool(((h.double() - wh).abs() <= wh.abs() * 2.0 ** -7 * 1.01 + 1e-30).all())
        assert_output_close(yw.float().cpu().numpy(), (y0 * w_slot).cpu().numpy(), what="weighted rows")
        if prev is not None:
            assert same(yw, prev) and same(h, prev_h)
        prev, prev_h = yw.clone(), h.clone()


@pytest.mark.parametrize("T,k,H,residual", [(16, 10, 2560, False), (129, 10, 2560, True), (7, 32, 256, True)])
def test_combine_weighted_against_oracle(T, k, H, residual):
    """moe_combine_weighted sums already weighted bf16 rows in rank order:
    the oracle's combine of the same rows (as fp32) with unit weights."""
    import oracle
    rng = np.random.default_rng(T * 3 + k)
    E = 64 if k <= 10 else 128
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, _, inv_r = oracle.permute(ids, E)
    yw_bits = oracle.round_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32))
    res_np = rng.standard_normal((T, H)).astype(np.float32) if residual else None
    ref = oracle.combine(oracle.bits_to_f32(yw_bits), inv_r, np.ones((T, k), np.float32), res_np)
    yw = torch.from_numpy(yw_bits.view(np.int16)).to(DEV).view(torch.bfloat16)
    out_b = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    out_f = torch.empty((T, H), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_combine_weighted(yw, torch.from_numpy(inv_r).to(DEV), T, k,
                              torch.from_numpy(res_np).to(DEV) if residual else None, out_b, out_f, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.allclose(out_f.cpu().numpy(), ref, rtol=1e-5, atol=1e-5)
    assert same(out_b, out_f.to(torch.bfloat16))
