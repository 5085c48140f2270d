"""GPU parity: every step of the layer through the C ABI against the CPU oracle.

Inputs are the seeded synthetic workloads (workloads/): x ~ N(0,1) bf16,
weights ~ N(0,0.02) bf16, Zipf router bias for the decode block.  The oracle
always computes from those seeded inputs; nothing the GPU produced is fed to
it.  Tolerances: tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity import GAP_TOL, assert_output_close, compare_routes
from sparse_moe_routed_gb300 import MoELayer, _lib, pack_layer_experts

pytestmark = pytest.mark.gpu

DEV = "cuda"
_CACHE = {}


def bits(t):
    return oracle.bf16_bits(t)


def f32_of_bits(b):
    return oracle.bits_to_f32(b)


def case(name, T=None):
    """Seeded layer inputs on the GPU plus host copies for the oracle."""
    key = (name, T)
    if key in _CACHE:
        return _CACHE[key]
    cfg = wl.CONFIGS[name]
    if T is not None:
        cfg = wl.with_tokens(cfg, T)
    d = wl.layer_inputs(cfg, DEV)
    torch.cuda.synchronize()
    host = {
        "x": bits(d["x"]),
        "wr": bits(d["w_router"]),
        "bias": None if d["bias"] is None else d["bias"].cpu().numpy(),
        "wgu": bits(d["w_gateup"]),
        "wd": bits(d["w_down"]),
    }
    _CACHE[key] = (cfg, d, host)
    return _CACHE[key]


def run_layer(cfg, d, tiled=False):
    if tiled:
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
        layer = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
    else:
        layer = MoELayer(d["w_router"], d["bias"], d["w_gateup"], d["w_down"], cfg.k, cfg.T)
    layer.clear_status()
    out = layer.forward(d["x"]).clone()
    torch.cuda.synchronize()
    assert layer.read_status() == 0
    return layer, out


def sample_tokens(T, n, seed=0):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    pick = rng.choice(T - 1, size=n - 1, replace=False)
    return np.sort(np.concatenate([pick, [T - 1]]))  # always include the ragged tail token


# --------------------------------------------------------------------------
# Router
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,T,nsample", [("tiny", None, 16), ("decode", None, 16), ("decode", 37, 37),
                                            ("prefill", None, 4096)])
def test_route_parity(name, T, nsample):
    cfg, d, host = case(name, T)
    layer, _ = run_layer(cfg, d)
    ids = layer.ids[:cfg.T].cpu().numpy()
    w = layer.w[:cfg.T].cpu().numpy()
    gap = layer.gap[:cfg.T].cpu().numpy()
    toks = sample_tokens(cfg.T, nsample)
    ids_r, w_r, gap_r, L_r = oracle.route(host["x"][toks], host["wr"], host["bias"], cfg.k)
    rep = compare_routes(ids[toks], w[toks], ids_r, w_r, gap_r, L_r)
    # the decision gap itself agrees to fp32 accumulation error
    assert np.allclose(gap[toks], gap_r, atol=5e-5)
    assert rep["near_tie"] <= max(2, len(toks) // 10), rep
    print(f"{name} T={cfg.T}: checked {rep['checked']} tokens, near-ties {rep['near_tie']}, "
          f"rank swaps {rep['rank_swaps']}")


@pytest.mark.parametrize("name,T", [("tiny", None), ("decode", None), ("decode", 1), ("decode", 5), ("tiny", 16)])
def test_route_permute_one_launch(name, T):
    """moe_route_permute (one cluster launch for a decode block): routes graded
    against the oracle like moe_route's, and its grouping bit-exact against the
    oracle's stable counting sort of the routes it chose."""
    cfg, d, host = case(name, T)
    E, k, Tn = cfg.E, cfg.k, cfg.T
    R = Tn * k
    ids = torch.full((Tn, k), -1, dtype=torch.int32, device=DEV)
    w = torch.full((Tn, k), float("nan"), dtype=torch.float32, device=DEV)
    gap = torch.full((Tn,), float("nan"), dtype=torch.float32, device=DEV)
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    perm = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    for _ in range(2):  # twice in a row: nothing carries over between calls
        _lib.moe_route_permute(d["x"], d["w_router"], d["bias"], k, ids, w, gap, counts, offsets, perm, inv, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ids_np, w_np, gap_np = ids.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy()
    ids_r, w_r, gap_r, L_r = oracle.route(host["x"], host["wr"], host["bias"], k)
    rep = compare_routes(ids_np, w_np, ids_r, w_r, gap_r, L_r)
    assert np.allclose(gap_np, gap_r, atol=5e-5)
    assert rep["near_tie"] <= max(2, Tn // 10), rep
    counts_r, offsets_r, perm_r, inv_r = oracle.permute(ids_np, E)
    assert np.array_equal(counts.cpu().numpy(), counts_r)
    assert np.array_equal(offsets.cpu().numpy(), offsets_r)
    assert np.array_equal(perm.cpu().numpy(), perm_r)
    assert np.array_equal(inv.cpu().numpy(), inv_r)


def test_route_tie_contract_on_gpu():
    """All-zero router weights: every logit equals its bias; ties go to lower IDs."""
    E, H, k, T = 64, 256, 4, 3
    x = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    wr = torch.zeros((E, H), device=DEV, dtype=torch.bfloat16)
    bias = torch.zeros((E,), device=DEV)
    bias[[5, 9, 40]] = 1.0  # three experts tie at the top, the rest tie at zero
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    gap = torch.empty((T,), dtype=torch.float32, device=DEV)
    ws = torch.empty((_lib.route_workspace_size(T, E),), dtype=torch.uint8, device=DEV)
    _lib.moe_route(x, wr, bias, k, ids, w, gap, ws)
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [[5, 9, 40, 0]] * T
    e1 = np.exp(1.0)
    ref_w = np.array([e1, e1, e1, 1.0]) / (3 * e1 + 1.0)
    assert np.allclose(w.cpu().numpy(), ref_w, atol=1e-6)
    assert np.all(gap.cpu().numpy() == 0.0)


def test_route_k_equals_e_is_full_softmax():
    E, H, k, T = 32, 128, 32, 5
    x = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    wr = (0.3 * torch.randn((E, H), device=DEV)).to(torch.bfloat16)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    gap = torch.empty((T,), dtype=torch.float32, device=DEV)
    ws = torch.empty((_lib.route_workspace_size(T, E),), dtype=torch.uint8, device=DEV)
    _lib.moe_route(x, wr, None, k, ids, w, gap, ws)
    torch.cuda.synchronize()
    ids_r, w_r, gap_r, L_r = oracle.route(bits(x), bits(wr), None, k)
    rep = compare_routes(ids.cpu().numpy(), w.cpu().numpy(), ids_r, w_r, np.full(T, np.inf), L_r)
    assert rep["checked"] == T
    assert np.all(np.isinf(gap.cpu().numpy()))


@pytest.mark.parametrize("T,H,E,k", [(5, 2560, 1024, 32), (70, 1024, 1024, 32), (3, 256, 100, 7),
                                     (4, 128, 33, 32), (64, 384, 96, 31)])
def test_route_at_the_largest_accepted_shape(T, H, E, k):
    """The last accepted expert count and route width (E = 1024, k = 32), on
    the small-T path (T <= 64) and on the tcgen05 router path (T > 64); and
    odd shapes: E not a multiple of 32, k + 1 = E, k = 31."""
    g = torch.Generator(device=DEV).manual_seed(T + H)
    x = torch.randn((T, H), device=DEV, generator=g).to(torch.bfloat16)
    wr = (0.02 * torch.randn((E, H), device=DEV, generator=g)).to(torch.bfloat16)
    bias = (0.1 * torch.randn((E,), device=DEV, generator=g)).float()
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    gap = torch.empty((T,), dtype=torch.float32, device=DEV)
    ws = torch.empty((_lib.route_workspace_size(T, E),), dtype=torch.uint8, device=DEV)
    _lib.moe_route(x, wr, bias, k, ids, w, gap, ws)
    torch.cuda.synchronize()
    ids_r, w_r, gap_r, L_r = oracle.route(bits(x), bits(wr), bias.cpu().numpy(), k)
    rep = compare_routes(ids.cpu().numpy(), w.cpu().numpy(), ids_r, w_r, gap_r, L_r)
    assert rep["near_tie"] <= max(2, T // 10), rep
    assert np.allclose(gap.cpu().numpy(), gap_r, atol=5e-5)


# --------------------------------------------------------------------------
# Grouping by expert (integer: bit-exact)
# --------------------------------------------------------------------------
def seeded_ids(T, k, E, seed, zipf=False):
    rng = np.random.default_rng(seed)
    if zipf:
        p = 1.0 / np.arange(1, E + 1)
        p /= p.sum()
        return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


PERMUTE_CASES = [(1, 4, 64, 256, False), (16, 10, 512, 2560, True), (37, 10, 512, 2560, False),
                 (4096, 10, 512, 2560, False), (300, 32, 1024, 128, False), (64, 8, 8, 128, False),
                 (8191, 10, 512, 128, True), (32768, 10, 512, 128, False),
                 # chunk edges: exactly 4 chunks of 2,048 routes; one route past
                 # them; 1,024 experts (fewer route warps per chunk)
                 (2048, 4, 1024, 128, False), (2049, 4, 64, 128, True), (4100, 10, 1024, 128, True)]


def permute_call(chunked, ids, E, x, counts, offsets, perm, inv, xp, st):
    """moe_permute (one CTA) or moe_permute_ws (chunks on many CTAs): the
    same outputs bit for bit."""
    if not chunked:
        _lib.moe_permute(ids, E, x, counts, offsets, perm, inv, xp, st)
        return
    T, k = ids.shape
    ws = torch.full((_lib.moe_permute_workspace_size(T, k, E) // 4,), -3, dtype=torch.int32, device=DEV)
    _lib.moe_permute_ws(ids, E, x, counts, offsets, perm, inv, xp, ws, st)


@pytest.mark.parametrize("chunked", [False, True])
@pytest.mark.parametrize("T,k,E,H,zipf", PERMUTE_CASES)
def test_permute_bit_exact(T, k, E, H, zipf, chunked):
    ids_np = seeded_ids(T, k, E, seed=T * 7 + E, zipf=zipf)
    counts_r, offsets_r, perm_r, inv_r = oracle.permute(ids_np, E)
    R = T * k
    ids = torch.from_numpy(ids_np).to(DEV)
    x = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    perm = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    xp = torch.zeros((R, H), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    permute_call(chunked, ids, E, x, counts, offsets, perm, inv, xp, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(counts.cpu().numpy(), counts_r)
    assert np.array_equal(offsets.cpu().numpy(), offsets_r)
    assert np.array_equal(perm.cpu().numpy(), perm_r)
    assert np.array_equal(inv.cpu().numpy(), inv_r)
    xb = bits(x)
    assert np.array_equal(bits(xp), xb[perm_r // k])


@pytest.mark.parametrize("chunked,T,bad_t", [(False, 8, 5), (True, 8, 5), (True, 3000, 1), (True, 3000, 2999)])
def test_permute_bad_id_flags_and_writes_nothing(chunked, T, bad_t):
    k, E = 4, 16
    ids_np = seeded_ids(T, k, E, 3)
    ids_np[bad_t, 2] = E  # out of range (first or last of several chunks)
    R = T * k
    ids = torch.from_numpy(ids_np).to(DEV)
    sentinel = -12345
    counts = torch.full((E,), sentinel, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), sentinel, dtype=torch.int32, device=DEV)
    # perm and inv hold valid entries from an earlier call: the row gather
    # must not follow them
    perm = torch.arange(R, dtype=torch.int32, device=DEV)
    inv = torch.arange(R, dtype=torch.int32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    H = 128
    x = torch.randn((T, H), device=DEV).to(torch.bfloat16)
    xp = torch.full((R, H), 7.0, dtype=torch.bfloat16, device=DEV)
    permute_call(chunked, ids, E, x, counts, offsets, perm, inv, xp, st)
    torch.cuda.synchronize()
    assert st.item() & _lib.MOE_DEV_BAD_EXPERT
    for t in (counts, offsets):
        assert bool((t == sentinel).all())
    assert torch.equal(perm.cpu(), torch.arange(R, dtype=torch.int32))
    assert torch.equal(inv.cpu(), torch.arange(R, dtype=torch.int32))
    assert bool((xp == 7.0).all())


# --------------------------------------------------------------------------
# Expert contractions (tcgen05) against the oracle's expert, slot by slot
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,T,nslots", [("tiny", None, 64), ("decode", None, 160), ("decode", 37, 370),
                                           ("prefill", None, 4096)])
def test_expert_stage_parity(name, T, nslots):
    cfg, d, host = case(name, T)
    E, H, I, k = cfg.E, cfg.H, cfg.I, cfg.k
    ids_np = seeded_ids(cfg.T, k, E, seed=11 + cfg.T, zipf=(cfg.bias == "zipf"))
    counts_r, offsets_r, perm_r, inv_r = oracle.permute(ids_np, E)
    R = cfg.T * k
    ids = torch.from_numpy(ids_np).to(DEV)
    counts = torch.empty((E,), dtype=torch.int32, device=DEV)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((R,), dtype=torch.int32, device=DEV)
    inv = torch.empty((R,), dtype=torch.int32, device=DEV)
    xp = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    y = torch.full((R, H), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_permute(ids, E, d["x"], counts, offsets, perm, inv, xp, st)
    _lib.moe_grouped_swiglu(xp, offsets, E, H, I, d["w_gateup"], d["w_down"], h, y, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    slots = sample_tokens(R, nslots, seed=5)
    seg_expert = np.searchsorted(offsets_r, slots, side="right") - 1
    y_gpu = y.cpu().numpy()
    xin = f32_of_bits(host["x"])
    # each sampled slot through its expert alone (a one-route combine with weight 1)
    ref = oracle.experts_combine(xin[perm_r[slots] // k], seg_expert.reshape(-1, 1).astype(np.int32),
                                 np.ones((len(slots), 1), np.float32), H, I, wgu_bits=host["wgu"], wd_bits=host["wd"])
    assert_output_close(y_gpu[slots], ref, what=f"{name} expert outputs")
    assert np.isfinite(y_gpu).all()


# --------------------------------------------------------------------------
# Combine
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,H,residual", [(16, 10, 2560, False), (5, 4, 256, True), (129, 10, 2560, True),
                                             (7, 32, 256, True)])
def test_combine_parity(T, k, H, residual):
    rng = np.random.default_rng(T + k)
    E = 64 if k <= 10 else 128
    ids_np = seeded_ids(T, k, E, seed=T)
    _, _, perm_r, inv_r = oracle.permute(ids_np, E)
    y_np = rng.standard_normal((T * k, H)).astype(np.float32)
    w_np = rng.random((T, k)).astype(np.float32)
    res_np = rng.standard_normal((T, H)).astype(np.float32) if residual else None
    ref = oracle.combine(y_np, inv_r, w_np, res_np)
    y = torch.from_numpy(y_np).to(DEV)
    inv = torch.from_numpy(inv_r).to(DEV)
    w = torch.from_numpy(w_np).to(DEV)
    res = torch.from_numpy(res_np).to(DEV) if residual else None
    out_b = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    out_f = torch.empty((T, H), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_combine(y, inv, w, res, out_b, out_f, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    # fp32 fused multiply-add over k terms in rank order vs fp64
    assert np.allclose(out_f.cpu().numpy(), ref, rtol=1e-5, atol=1e-5)
    assert np.array_equal(bits(out_b), bits(out_f.to(torch.bfloat16)))


@pytest.mark.parametrize("T,k,H", [(16, 10, 2560), (3, 20, 384), (40, 32, 256)])
def test_combine_right_after_the_grouping(T, k, H):
    """moe_combine reads the routes' slots and weights before it waits on
    the launch before it and checks them after; when that launch is the
    grouping that rewrites the slots (here several groupings in a row, each
    followed at once by a combine), the rows must still be the ones the new
    slots name."""
    rng = np.random.default_rng(T * k)
    E = 64
    R = T * k
    y_np = rng.standard_normal((R, H)).astype(np.float32)
    y = torch.from_numpy(y_np).to(DEV)
    counts = torch.empty((E,), dtype=torch.int32, device=DEV)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((R,), dtype=torch.int32, device=DEV)
    inv = torch.empty((R,), dtype=torch.int32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    outs, refs = [], []
    for rep in range(6):
        ids_np = seeded_ids(T, k, E, seed=1000 * rep + T)
        _, _, _, inv_r = oracle.permute(ids_np, E)
        w_np = rng.random((T, k)).astype(np.float32)
        w = torch.from_numpy(w_np).to(DEV)
        ids = torch.from_numpy(ids_np).to(DEV)
        torch.cuda.synchronize()
        out = torch.empty((T, H), dtype=torch.float32, device=DEV)
        _lib.moe_permute(ids, E, None, counts, offsets, perm, inv, None, st)
        _lib.moe_combine(y, inv, w, None, None, out, st)
        outs.append(out)
        refs.append(oracle.combine(y_np, inv_r, w_np, None))
    torch.cuda.synchronize()
    assert st.item() == 0
    for out, ref in zip(outs, refs):
        assert np.allclose(out.cpu().numpy(), ref, rtol=1e-5, atol=1e-5)


def test_combine_nonfinite_flag():
    T, k, H = 2, 2, 128
    y = torch.zeros((T * k, H), device=DEV)
    y[1, 7] = float("inf")
    inv = torch.arange(T * k, dtype=torch.int32, device=DEV)
    w = torch.full((T, k), 0.5, device=DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_combine(y, inv, w, None, out, None, st)
    torch.cuda.synchronize()
    assert st.item() & _lib.MOE_DEV_NONFINITE


# --------------------------------------------------------------------------
# Whole layer
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name,T,nsample,tiled", [("tiny", None, 16, False), ("decode", None, 16, False),
                                                  ("decode", 37, 37, False), ("prefill", None, 24, False),
                                                  ("tiny", None, 16, True), ("decode", None, 16, True),
                                                  ("decode", 37, 37, True), ("decode", 1, 1, True),
                                                  ("prefill", None, 4096, True),
                                                  # edges of the launch choices: token rows per tile
                                                  # (R 320 / 330, 1,280 / 1,290), the router's small-T path
                                                  # (T 64 / 65), the in-launch gather and tile queue
                                                  # (R 4,090 / 4,100)
                                                  ("decode", 32, 12, True), ("decode", 33, 12, True),
                                                  ("decode", 64, 12, True), ("decode", 65, 12, True),
                                                  ("decode", 128, 12, True), ("decode", 129, 12, True),
                                                  ("decode", 409, 12, True), ("decode", 410, 12, True),
                                                  # 256-row token tiles (from 131,072 routes)
                                                  ("prefill", 16384, 96, True)])
def test_layer_parity(name, T, nsample, tiled):
    cfg, d, host = case(name, T)
    layer, out = run_layer(cfg, d, tiled)
    ids = layer.ids[:cfg.T].cpu().numpy()
    toks = sample_tokens(cfg.T, nsample, seed=1)
    ids_r, w_r, gap_r, L_r = oracle.route(host["x"][toks], host["wr"], host["bias"], cfg.k)
    xin = f32_of_bits(host["x"][toks])
    ref = oracle.experts_combine(xin, ids_r, w_r, cfg.H, cfg.I, wgu_bits=host["wgu"], wd_bits=host["wd"])
    same = np.array([np.array_equal(ids[t], ids_r[n]) for n, t in enumerate(toks)])
    # tokens whose route legitimately differs (near-tie) are reported, not graded
    assert np.all(same | (gap_r <= GAP_TOL) | ~same & _adjacent_swap_ok(ids[toks], ids_r, L_r))
    keep = same
    assert keep.sum() >= 0.9 * len(toks)
    got = out.float().cpu().numpy()[toks][keep]
    rel_max, mean_rel = assert_output_close(got, ref[keep], what=f"{name} layer output")
    print(f"{name} T={cfg.T} tiled={tiled}: {keep.sum()}/{len(toks)} tokens graded, max err {rel_max:.2e} "
          f"of max|ref|, mean rel {mean_rel:.2e}")


@pytest.mark.parametrize("T,H,E,k,I,tiled", [(16, 1024, 1024, 16, 256, True), (16, 1024, 1024, 16, 256, False),
                                              (37, 256, 100, 7, 128, True), (5, 512, 1024, 32, 128, True)])
def test_layer_parity_at_the_expert_count_limits(T, H, E, k, I, tiled):
    """The whole layer at the largest accepted expert count (E = 1,024: the
    fused launch's tile prefix and tile search over 32 expert groups, 256
    routes, and k = 32) and at an expert count that is not a multiple of
    32, against the oracle on every token."""
    cfg = wl.LayerConfig("limits", T=T, H=H, E=E, k=k, I=I, bias="zipf", seed=43 + E + k)
    d = wl.layer_inputs(cfg, DEV)
    torch.cuda.synchronize()
    layer, out = run_layer(cfg, d, tiled)
    xb, wrb = bits(d["x"]), bits(d["w_router"])
    ids_r, w_r, gap_r, L_r = oracle.route(xb, wrb, d["bias"].cpu().numpy(), k)
    ids = layer.ids[:T].cpu().numpy()
    same = np.array([np.array_equal(ids[t], ids_r[t]) for t in range(T)])
    assert np.all(same | (gap_r <= GAP_TOL) | _adjacent_swap_ok(ids, ids_r, L_r))
    assert same.sum() >= 0.9 * T
    ref = oracle.experts_combine(f32_of_bits(xb), ids_r, w_r, H, I, wgu_bits=bits(d["w_gateup"]),
                                 wd_bits=bits(d["w_down"]))
    rel_max, mean_rel = assert_output_close(out.float().cpu().numpy()[same], ref[same],
                                            what=f"layer E={E} k={k} tiled={tiled}")
    print(f"E={E} k={k} T={T} tiled={tiled}: {same.sum()}/{T} tokens graded, max err {rel_max:.2e} of max|ref|, "
          f"mean rel {mean_rel:.2e}")


@pytest.mark.parametrize("T,H,E,k,I", [(8191, 2560, 64, 8, 640), (4096, 1024, 1024, 16, 256)])
def test_layer_parity_prefill_shapes(T, H, E, k, I):
    """Prefill-sized layers off the main geometry, 48 sampled tokens (the
    last always) against the oracle: 1,024 rows per expert (256-row tiles,
    four row chunks per expert with a ragged last one) and 1,024 experts
    with 64 rows each (the levelled static tile order, the chunked grouping
    and route-weighted outputs over 32 expert groups)."""
    cfg = wl.LayerConfig("prefill_shape", T=T, H=H, E=E, k=k, I=I, bias=None, seed=53 + E)
    d = wl.layer_inputs(cfg, DEV)
    torch.cuda.synchronize()
    layer, out = run_layer(cfg, d, tiled=True)
    toks = sample_tokens(T, 48, seed=3)
    xb = bits(d["x"])
    ids_r, w_r, gap_r, L_r = oracle.route(xb[toks], bits(d["w_router"]), None, k)
    ids = layer.ids[:T].cpu().numpy()[toks]
    same = np.array([np.array_equal(ids[n], ids_r[n]) for n in range(len(toks))])
    assert np.all(same | (gap_r <= GAP_TOL) | _adjacent_swap_ok(ids, ids_r, L_r))
    assert same.sum() >= 0.9 * len(toks)
    ref = oracle.experts_combine(f32_of_bits(xb[toks]), ids_r, w_r, H, I, wgu_bits=bits(d["w_gateup"]),
                                 wd_bits=bits(d["w_down"]))
    rel_max, mean_rel = assert_output_close(out.float().cpu().numpy()[toks][same], ref[same],
                                            what=f"prefill-shaped layer T={T} E={E}")
    print(f"T={T} E={E} k={k}: {same.sum()}/{len(toks)} tokens graded, max err {rel_max:.2e} of max|ref|, "
          f"mean rel {mean_rel:.2e}")


def test_layer_with_one_launch_routing():
    """The layer with routing and grouping in one launch (moe_route_permute)
    against the oracle, as test_layer_parity grades the default chain."""
    cfg, d, host = case("decode")
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
    layer = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
    layer.ROUTE_PERMUTE_ONE_LAUNCH = True
    assert [c[0] for c in layer.bound_calls(d["x"])][0] == "moe_route_permute"
    out = layer.forward(d["x"]).clone()
    torch.cuda.synchronize()
    assert layer.read_status() == 0
    ids = layer.ids[:cfg.T].cpu().numpy()
    ids_r, w_r, gap_r, L_r = oracle.route(host["x"], host["wr"], host["bias"], cfg.k)
    ref = oracle.experts_combine(f32_of_bits(host["x"]), ids_r, w_r, cfg.H, cfg.I, wgu_bits=host["wgu"],
                                 wd_bits=host["wd"])
    same = np.array([np.array_equal(ids[t], ids_r[t]) for t in range(cfg.T)])
    assert same.sum() >= 0.9 * cfg.T
    assert_output_close(out.float().cpu().numpy()[same], ref[same], what="decode layer, one-launch routing")


def _adjacent_swap_ok(ids_gpu, ids_ref, L_ref):
    ok = np.zeros(len(ids_ref), bool)
    for n in range(len(ids_ref)):
        g, r = list(ids_gpu[n]), list(ids_ref[n])
        if set(g) != set(r):
            continue
        ok[n] = all(abs(float(L_ref[n, a]) - float(L_ref[n, b])) <= GAP_TOL for a, b in zip(g, r) if a != b)
    return ok


def test_layer_deterministic():
    cfg, d, _ = case("decode")
    layer = MoELayer(d["w_router"], d["bias"], d["w_gateup"], d["w_down"], cfg.k, cfg.T)
    a = layer.forward(d["x"]).clone()
    b = layer.forward(d["x"]).clone()
    tl, _ = run_layer(cfg, d, tiled=True)
    c = tl.forward(d["x"]).clone()
    c2 = tl.forward(d["x"]).clone()
    torch.cuda.synchronize()
    # the fused contraction leaves its readiness counters zeroed for the next call
    assert int(tl.sync_ws.abs().sum().item()) == 0
    assert torch.equal(c.view(torch.int16), c2.view(torch.int16))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # packing changes where weights live, not the arithmetic: identical bits
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_forward_host_graph_matches_eager():
    """The graph-replayed host round trip gives the eager layer's bits, call
    after call, with new inputs written into the same pinned buffer."""
    cfg, d, _ = case("decode")
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
    layer = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
    x_host = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    out_host = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    for i in range(3):
        xi = wl.token_batch(cfg, DEV, index=40 + i)
        ref = layer.forward(xi).clone()
        torch.cuda.synchronize()
        x_host.copy_(xi.cpu())
        got = layer.forward_host_graph(x_host, out_host)
        assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16)), i
    assert layer.read_status() == 0
    assert int(layer.sync_ws.abs().sum().item()) == 0


def test_forward_host_submit_two_in_flight():
    """Calls queued before the previous one is waited for (two pinned buffer
    pairs, two layers) finish in order with the eager layer's bits."""
    cfg, d, _ = case("decode")
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
    layers = [MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
              for _ in range(2)]
    xs = [wl.token_batch(cfg, DEV, index=60 + i) for i in range(6)]
    refs = [layers[0].forward(x).clone().cpu() for x in xs]
    torch.cuda.synchronize()
    x_host = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    out_host = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    prev = None
    for i, x in enumerate(xs):
        x_host[i % 2].copy_(x.cpu())
        done = layers[i % 2].forward_host_submit(x_host[i % 2], out_host[i % 2])
        if prev is not None:
            MoELayer.wait(prev[0])
            assert torch.equal(out_host[prev[1] % 2].view(torch.int16), refs[prev[1]].view(torch.int16)), prev[1]
        prev = (done, i)
    MoELayer.wait(prev[0])
    assert torch.equal(out_host[prev[1] % 2].view(torch.int16), refs[prev[1]].view(torch.int16))
    assert all(l.read_status() == 0 for l in layers)


@pytest.mark.parametrize("nlayers", [1, 2])
def test_forward_host_pipelined_two_in_flight(nlayers):
    """The pipelined host round trip (input copy on a copy stream, the layer's
    graph on the compute stream, the result copy on another copy stream,
    alternating device buffers) gives the eager layer's bits for every call,
    with the next call queued before the previous one is waited for."""
    cfg, d, _ = case("decode")
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
    layers = [MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
              for _ in range(nlayers)]
    xs = [wl.token_batch(cfg, DEV, index=80 + i) for i in range(7)]
    refs = [layers[0].forward(x).clone().cpu() for x in xs]
    torch.cuda.synchronize()
    x_host = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    out_host = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    prev = None
    for i, x in enumerate(xs):
        x_host[i % 2].copy_(x.cpu())
        done = layers[i % nlayers].forward_host_pipelined(x_host[i % 2], out_host[i % 2])
        if prev is not None:
            MoELayer.wait(prev[0])
            assert torch.equal(out_host[prev[1] % 2].view(torch.int16), refs[prev[1]].view(torch.int16)), prev[1]
        prev = (done, i)
    MoELayer.wait(prev[0])
    assert torch.equal(out_host[prev[1] % 2].view(torch.int16), refs[prev[1]].view(torch.int16))
    assert all(l.read_status() == 0 for l in layers)


@pytest.mark.parametrize("tiled", [False, True])
def test_layer_single_token_and_empty(tiled):
    cfg, d, host = case("tiny")
    if tiled:
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
        layer = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
    else:
        layer = MoELayer(d["w_router"], d["bias"], d["w_gateup"], d["w_down"], cfg.k, cfg.T)
    x1 = d["x"][3:4].contiguous()
    out1 = layer.forward(x1).clone()
    empty = layer.forward(d["x"][:0])
    torch.cuda.synchronize()
    assert empty.shape[0] == 0
    if tiled:
        assert int(layer.sync_ws.abs().sum().item()) == 0
    ids_r, w_r, _, _ = oracle.route(host["x"][3:4], host["wr"], None, cfg.k)
    ref = oracle.experts_combine(f32_of_bits(host["x"][3:4]), ids_r, w_r, cfg.H, cfg.I, wgu_bits=host["wgu"],
                                 wd_bits=host["wd"])
    assert_output_close(out1.float().cpu().numpy(), ref, what="single token")


# --------------------------------------------------------------------------
# Block dedup (integer: bit-exact)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L,Tt,k,E,B", [(48, 512, 10, 512, 1), (48, 512, 10, 512, 4), (48, 512, 10, 512, 16),
                                       (48, 512, 10, 512, 64), (3, 37, 4, 64, 5), (2, 50, 32, 1024, 7)])
def test_dedup_bit_exact(L, Tt, k, E, B):
    ids_np = np.stack([seeded_ids(Tt, k, E, seed=100 + l) for l in range(L)])
    mask_r, U_r, b2_r, b4_r = oracle.dedup(ids_np, E, B, 2560, 640)
    nb = (Tt + B - 1) // B
    W = (E + 31) // 32
    ids = torch.from_numpy(ids_np).to(DEV)
    mask = torch.empty((L, nb, W), dtype=torch.int32, device=DEV)
    U = torch.empty((L, nb), dtype=torch.int32, device=DEV)
    b2 = torch.empty((nb,), dtype=torch.int64, device=DEV)
    b4 = torch.empty((nb,), dtype=torch.int64, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.route_block_dedup(ids, E, B, 2560, 640, mask, U, b2, b4, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), mask_r)
    assert np.array_equal(U.cpu().numpy(), U_r)
    assert np.array_equal(b2.cpu().numpy(), b2_r)
    assert np.array_equal(b4.cpu().numpy(), b4_r)


# --------------------------------------------------------------------------
# RMSNorm
# --------------------------------------------------------------------------
def test_rmsnorm_parity():
    rng = np.random.default_rng(9)
    T, H = 33, 2560
    x_np = (3.0 * rng.standard_normal((T, H))).astype(np.float32)
    g_np = (0.1 * rng.standard_normal(H)).astype(np.float32)
    ref = oracle.rmsnorm(x_np, g_np, eps=1e-6)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    _lib.moe_rmsnorm(torch.from_numpy(x_np).to(DEV), torch.from_numpy(g_np).to(DEV), 1e-6, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    # bf16 output: within one bf16 rounding (2^-8 relative) of the fp64 value
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
