"""GPU checks of macro-prefill layer streaming (moe_layer_stream, PrefillRing).

Whole layers of packed records move from pinned host memory into a
two-layer HBM ring on the copy engines while the previous layer computes.
Copying is byte work and the contraction is unchanged, so a stack run
through the ring must equal, bit for bit, MoEStack over the same records
resident in HBM, with the ring slots reused several times.
"""
import pytest
import torch

import workloads as wl
from sparse_moe_routed_gb300 import MoELayer, MoEStack, PrefillRing, _lib, pack_layer_experts

pytestmark = pytest.mark.gpu

DEV = "cuda"
CFG = wl.LayerConfig("ring_small", T=64, H=256, E=64, k=4, I=128, bias=None, seed=31)


def test_layer_stream_copies_exactly():
    n1, n2 = 3 * 65536 + 16, 4096
    h1 = torch.randint(0, 256, (n1,), dtype=torch.uint8).pin_memory()
    h2 = torch.randint(0, 256, (n2,), dtype=torch.uint8).pin_memory()
    d1 = torch.zeros(n1, dtype=torch.uint8, device=DEV)
    d2 = torch.zeros(n2, dtype=torch.uint8, device=DEV)
    _lib.moe_layer_stream(h1, h2, d1, d2)
    torch.cuda.synchronize()
    assert torch.equal(d1.cpu(), h1) and torch.equal(d2.cpu(), h2)


@pytest.mark.parametrize("L,T", [(5, 64), (2, 16), (1, 64)])
def test_ring_equals_resident_stack(L, T):
    routers, host, dev_layers = [], [], []
    for l in range(L):
        d = wl.layer_inputs(CFG, DEV, layer=l, with_x=False)
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, CFG.E, CFG.H, CFG.I)
        torch.cuda.synchronize()
        routers.append((d["w_router"], d["bias"]))
        host.append((gu.cpu().pin_memory(), dn.cpu().pin_memory()))
        dev_layers.append(MoELayer(d["w_router"], d["bias"], gu, dn, CFG.k, T, fmt=_lib.MOE_W_BF16_TILED, I=CFG.I))
    ref = MoEStack(dev_layers, T)
    ring = PrefillRing(routers, host, CFG.k, T, CFG.I)
    for rep in range(2):  # the second pass refills ring slots the first one used
        x0 = wl.token_batch(CFG, DEV, index=rep, T=T).float()
        want = ref.forward(x0.clone())
        got = ring.forward(x0.clone())
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), rep
        for ml in ring.stack.layers:
            assert ml.read_status() == 0
