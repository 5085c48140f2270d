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
