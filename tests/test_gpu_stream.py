"""GPU checks of macro-prefill layer streaming (moe_layer_stream, PrefillRing).

Whole layers of packed records move from pinned host memory into a
two-layer HBM ring on the copy engines while the previous layer computes.
Copying is byte work and the contraction is unchanged, so a stack run
through the ring must equal, bit for bit, MoEStack over the same records
resident in HBM, with the ring slots reused several times.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity import assert_output_close, compare_routes
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


def test_ring_two_layers_against_oracle():
    """One PrefillRing pass over two layers of the Qwen4Exp geometry (uniform
    router, 512 tokens: nearly every expert routed) graded against the CPU
    oracle.  Each layer is x <- x + MoE(bf16(RMSNorm(x))); the oracle runs
    both layers from the same x0 on a sample of tokens (tokens are
    independent), and every sampled token whose routes the oracle confirms
    in both layers is graded on the two-layer residual update."""
    cfg = wl.with_tokens(wl.PREFILL, 512)
    L, T = 2, cfg.T
    routers, host, orc = [], [], []
    for l in range(L):
        d = wl.layer_inputs(cfg, DEV, layer=l, with_x=False)
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
        torch.cuda.synchronize()
        routers.append((d["w_router"], d["bias"]))
        host.append((gu.cpu().pin_memory(), dn.cpu().pin_memory()))
        orc.append((oracle.bf16_bits(d["w_router"]), oracle.bf16_bits(d["w_gateup"]), oracle.bf16_bits(d["w_down"])))
        del gu, dn, d
    ring = PrefillRing(routers, host, cfg.k, T, cfg.I)
    x0 = wl.token_batch(cfg, DEV, index=3, T=T).float()
    got = ring.forward(x0.clone())
    torch.cuda.synchronize()
    for ml in ring.stack.layers:
        assert ml.read_status() == 0
    rng = np.random.default_rng(7)
    toks = np.sort(np.concatenate([rng.choice(T - 1, size=127, replace=False), [T - 1]]))
    # teacher forcing: layer 0 reads x0; layer 1 reads the GPU's own
    # normalised input of that layer (the stack's bf16 input buffer holds the
    # last layer's), so a legitimate difference in x_1 cannot flip a route
    inputs = [oracle.round_bf16_bits(oracle.rmsnorm(x0.cpu().numpy()[toks], None, eps=1e-6)),
              oracle.bf16_bits(ring.stack.n[:T])[toks]]
    ok = np.ones(len(toks), bool)
    update = np.zeros((len(toks), cfg.H))
    for l in range(L):
        wr, wgu, wdn = orc[l]
        n_bits = inputs[l]
        ids_r, w_r, gap_r, L_r = oracle.route(n_bits, wr, None, cfg.k)
        ml = ring.stack.layers[l]
        rep = compare_routes(ml.ids[:T].cpu().numpy()[toks], ml.w[:T].cpu().numpy()[toks], ids_r, w_r, gap_r, L_r)
        m = np.zeros(len(toks), bool)
        m[rep["exact_rows"]] = True
        ok &= m
        update += oracle.experts_combine(oracle.bits_to_f32(n_bits), ids_r, w_r, cfg.H, cfg.I, wgu_bits=wgu,
                                         wd_bits=wdn)
    # a token is graded when both of its layers' routes match the oracle in
    # rank order (near-ties and allowed rank swaps in either layer are not)
    assert ok.sum() >= 0.8 * len(toks)
    x0_np = x0.cpu().numpy()[toks].astype(np.float64)
    got_np = got.cpu().numpy()[toks].astype(np.float64)
    rel_max, mean_rel = assert_output_close(got_np[ok] - x0_np[ok], update[ok], what="two-layer ring residual update")
    print(f"ring L=2 T={T}: {ok.sum()}/{len(toks)} tokens graded, max err {rel_max:.2e}, mean rel {mean_rel:.2e}")
