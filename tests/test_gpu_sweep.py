"""GPU checks of the route-prediction / dedup sweep.

The recall kernel is compared bit for bit with the oracle on seeded routes.
The sweep itself runs on the GPU's own stack; its outputs are checked by
properties that hold at any size: U equals the size of the union of the
block's routes, U <= min(k*B, E), bytes follow U exactly, the native router
on the pre-normalisation representation recovers the native route (a
positive per-token scale does not change the top-k, up to bf16 near-ties),
and a random linear predictor sits near the chance recall k/E.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from sparse_moe_routed_gb300 import MoELayer, MoEStack, _lib, pack_layer_experts
from sparse_moe_routed_gb300.sweep import route_sweep

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("T,k,E", [(512, 10, 512), (37, 4, 64), (3, 32, 1024)])
def test_recall_bit_exact(T, k, E):
    rng = np.random.default_rng(T + k)
    a = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    b = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    b[: T // 3] = a[: T // 3][:, ::-1]  # some full matches in another order
    ref = oracle.recall_hits(a, b)
    hits = torch.full((T,), -1, dtype=torch.int32, device=DEV)
    _lib.moe_route_recall(torch.from_numpy(a).to(DEV), torch.from_numpy(b).to(DEV), hits)
    torch.cuda.synchronize()
    assert np.array_equal(hits.cpu().numpy(), ref)


def test_sweep_small_stack_properties():
    cfg = wl.STACK48
    L, T = 3, 64
    mls = []
    for l in range(L):
        w = wl.stack_layer_weights(l, DEV)
        gu, dn = pack_layer_experts(w["w_gateup_q"], w["w_down_q"], _lib.MOE_W_INT4_G64, cfg.E, cfg.H, cfg.I,
                                    s_gateup=w["s_gateup"], s_down=w["s_down"])
        mls.append(MoELayer(w["w_router"], None, gu, dn, cfg.k, T, fmt=_lib.MOE_W_INT4_G64_TILED, I=cfg.I))
    stack = MoEStack(mls, T)
    preds = [wl.predictor_weights(cfg.H, cfg.E, l, DEV) for l in range(L)]
    x0 = wl.token_batch(cfg, DEV, index=21, T=T).float()
    res = route_sweep(stack, x0, preds, blocks=(1, 4, 16, 64))
    assert res["status"] == 0
    native = res["native"].cpu().numpy()
    for B, d in res["dedup"].items():
        U = d["U"].cpu().numpy()
        mask = d["mask"].cpu().numpy().view(np.uint32)
        nb = (T + B - 1) // B
        for l in range(L):
            for b in range(nb):
                ref = set(native[l, b * B:(b + 1) * B].reshape(-1).tolist())
                got = {w * 32 + i for w in range(mask.shape[2]) for i in range(32) if (int(mask[l, b, w]) >> i) & 1}
                assert got == ref and U[l, b] == len(ref) <= min(cfg.k * B, cfg.E)
        P = 3 * cfg.H * cfg.I
        assert np.array_equal(d["bytes2"].cpu().numpy(), U.sum(0).astype(np.int64) * P * 2 // 8)
        assert np.array_equal(d["bytes4"].cpu().numpy(), U.sum(0).astype(np.int64) * P * 4 // 8)
    s = res["summary"]
    assert s["blocks"][1]["mean_U_per_layer"] == cfg.k  # one token: ten distinct experts per layer
    assert s["recall_native_router_on_prenorm"] >= 0.97, s
    assert 0.002 <= s["recall_linear_predictor"] <= 0.06, s
    print(s)
