"""GPU parity of the int4 g64 path and of the residual stack.

A stack layer is x <- x + MoE(RMSNorm(x)) with int4 g64 expert weights and a
bf16 router (the 48-layer workload of the Qwen4Exp routed stack).  The oracle
dequantises exactly and runs in fp64; the router and experts on both sides
read the RMS-normalised residual rounded to bf16.  Tolerances: tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity import GAP_TOL, assert_output_close, compare_routes
from sparse_moe_routed_gb300 import MoELayer, MoEStack, _lib, pack_layer_experts

pytestmark = pytest.mark.gpu

DEV = "cuda"
CFG = wl.STACK48
_W = {}


def layer_weights(l):
    if l not in _W:
        w = wl.stack_layer_weights(l, DEV)
        torch.cuda.synchronize()
        w["host"] = {
            "wr": oracle.bf16_bits(w["w_router"]),
            "wgu_q": w["w_gateup_q"].cpu().numpy(), "sgu": oracle.bf16_bits(w["s_gateup"]),
            "wd_q": w["w_down_q"].cpu().numpy(), "sd": oracle.bf16_bits(w["s_down"]),
        }
        _W[l] = w
    return _W[l]


def make_stack(L, T):
    mls = []
    for l in range(L):
        w = layer_weights(l)
        gu, dn = pack_layer_experts(w["w_gateup_q"], w["w_down_q"], _lib.MOE_W_INT4_G64, CFG.E, CFG.H, CFG.I,
                                    s_gateup=w["s_gateup"], s_down=w["s_down"])
        mls.append(MoELayer(w["w_router"], None, gu, dn, CFG.k, T, fmt=_lib.MOE_W_INT4_G64_TILED, I=CFG.I))
    return MoEStack(mls, T)


def oracle_layer(x_np, l, ids=None, w=None):
    """One oracle stack layer on fp32 residual rows x_np: (x + MoE(n), ids, w, gap, logits)."""
    h = layer_weights(l)["host"]
    n_bits = oracle.round_bf16_bits(oracle.rmsnorm(x_np, None, eps=1e-6))
    ids_r, w_r, gap_r, L_r = oracle.route(n_bits, h["wr"], None, CFG.k)
    if ids is None:
        ids, w = ids_r, w_r
    moe = oracle.experts_combine(oracle.bits_to_f32(n_bits), ids, w, CFG.H, CFG.I, wgu_q=h["wgu_q"],
                                 sgu_bits=h["sgu"], wd_q=h["wd_q"], sd_bits=h["sd"])
    return (x_np.astype(np.float64) + moe).astype(np.float32), moe, ids_r, w_r, gap_r, L_r


@pytest.mark.parametrize("T", [16, 37])
def test_int4_stack_layer_parity(T):
    stack = make_stack(1, T)
    x0 = wl.token_batch(CFG, DEV, index=5, T=T).float()
    x = x0.clone()
    stack.forward(x)
    torch.cuda.synchronize()
    L0 = stack.layers[0]
    assert L0.read_status() == 0
    x0_np = x0.cpu().numpy()
    x_ref, moe_ref, ids_r, w_r, gap_r, L_r = oracle_layer(x0_np, 0)
    rep = compare_routes(L0.ids[:T].cpu().numpy(), L0.w[:T].cpu().numpy(), ids_r, w_r, gap_r, L_r)
    keep = np.array(rep["exact_rows"])
    assert len(keep) >= 0.9 * T, rep
    moe_gpu = (x.cpu().numpy().astype(np.float64) - x0_np)[keep]
    rel_max, mean_rel = assert_output_close(moe_gpu, moe_ref[keep], what="int4 stack layer MoE output")
    print(f"T={T}: {len(keep)}/{T} tokens graded, max err {rel_max:.2e} of max|ref|, mean rel {mean_rel:.2e}")


@pytest.mark.parametrize("T", [512, 1024])
def test_int4_stack_layer_parity_many_routes(T):
    """int4 layers with many routes run on the tensor-core kernels (64-row
    token tiles at 5,120 routes, 128-row tiles at 10,240) instead of the
    CUDA-core one: 48 sampled tokens (the last one always) against the
    oracle."""
    stack = make_stack(1, T)
    x0 = wl.token_batch(CFG, DEV, index=7, T=T).float()
    x = x0.clone()
    stack.forward(x)
    torch.cuda.synchronize()
    L0 = stack.layers[0]
    assert L0.read_status() == 0
    rng = np.random.default_rng(T)
    toks = np.sort(np.concatenate([rng.choice(T - 1, size=47, replace=False), [T - 1]]))
    x0_np = x0.cpu().numpy()
    _, moe_ref, ids_r, w_r, gap_r, L_r = oracle_layer(x0_np[toks], 0)
    rep = compare_routes(L0.ids[:T].cpu().numpy()[toks], L0.w[:T].cpu().numpy()[toks], ids_r, w_r, gap_r, L_r)
    keep = np.array(rep["exact_rows"])
    assert len(keep) >= 0.9 * len(toks), rep
    moe_gpu = (x.cpu().numpy().astype(np.float64) - x0_np)[toks][keep]
    rel_max, mean_rel = assert_output_close(moe_gpu, moe_ref[keep], what=f"int4 layer MoE output, T={T}")
    print(f"T={T}: {len(keep)}/{len(toks)} tokens graded, max err {rel_max:.2e} of max|ref|, mean rel {mean_rel:.2e}")


def test_int4_expert_stage_tiny_geometry():
    """int4 contraction on the tiny geometry (two 128-row down blocks, K = 256 / 64)."""
    cfg = wl.TINY
    d = wl.layer_inputs(cfg, DEV)
    q_gu, s_gu = wl.quantize_int4_g64(d["w_gateup"])
    q_d, s_d = wl.quantize_int4_g64(d["w_down"])
    rng = np.random.default_rng(3)
    ids_np = np.stack([rng.choice(cfg.E, size=cfg.k, replace=False) for _ in range(cfg.T)]).astype(np.int32)
    _, offsets_r, perm_r, _ = oracle.permute(ids_np, cfg.E)
    R = cfg.T * cfg.k
    ids = torch.from_numpy(ids_np).to(DEV)
    counts = torch.empty((cfg.E,), dtype=torch.int32, device=DEV)
    offsets = torch.empty((cfg.E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((R,), dtype=torch.int32, device=DEV)
    inv = torch.empty((R,), dtype=torch.int32, device=DEV)
    xp = torch.empty((R, cfg.H), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((R, cfg.I), dtype=torch.bfloat16, device=DEV)
    y = torch.full((R, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_permute(ids, cfg.E, d["x"], counts, offsets, perm, inv, xp, st)
    gu, dn = pack_layer_experts(q_gu, q_d, _lib.MOE_W_INT4_G64, cfg.E, cfg.H, cfg.I, s_gateup=s_gu, s_down=s_d)
    _lib.moe_grouped_swiglu(xp, offsets, cfg.E, cfg.H, cfg.I, gu, dn, h, y, st, fmt=_lib.MOE_W_INT4_G64_TILED)
    torch.cuda.synchronize()
    assert st.item() == 0
    xin = oracle.bits_to_f32(oracle.bf16_bits(d["x"]))
    wgu = oracle.dequant_int4(q_gu.cpu().numpy(), oracle.bf16_bits(s_gu))
    wdn = oracle.dequant_int4(q_d.cpu().numpy(), oracle.bf16_bits(s_d))
    # expected per slot through the oracle's int4 expert (one route per row, weight 1)
    seg_e = np.searchsorted(offsets_r, np.arange(R), side="right") - 1
    tok = perm_r // cfg.k
    ref = oracle.experts_combine(xin[tok], seg_e.reshape(R, 1).astype(np.int32), np.ones((R, 1), np.float32),
                                 cfg.H, cfg.I, wgu_q=q_gu.cpu().numpy(), sgu_bits=oracle.bf16_bits(s_gu),
                                 wd_q=q_d.cpu().numpy(), sd_bits=oracle.bf16_bits(s_d))
    assert np.isfinite(wgu).all() and np.isfinite(wdn).all()
    assert_output_close(y.cpu().numpy(), ref, what="int4 expert outputs (tiny)")


# an odd number of 128-row blocks on both sides (H = 384, 2I = 384): the down
# launch cannot pair its blocks into 256-row tiles and takes the four-group split
ODD = wl.LayerConfig("int4_odd", T=16, H=384, E=64, k=4, I=192, bias=None, seed=19)
# unpaired down blocks whose record has a multiple of four (I = 256) or of two
# (I = 128) K steps: a ring slot holds four or two steps of one block
ODD_K4 = wl.LayerConfig("int4_odd_k4", T=16, H=384, E=64, k=4, I=256, bias=None, seed=29)
ODD_K2 = wl.LayerConfig("int4_odd_k2", T=16, H=384, E=64, k=4, I=128, bias=None, seed=31)
# down tiles of four blocks with one K step per slot (H = 512, I = 192), and
# of two blocks with two steps per slot (H = 768: six blocks, I = 128)
QUAD_K1 = wl.LayerConfig("int4_quad_k1", T=16, H=512, E=64, k=4, I=192, bias=None, seed=37)
PAIR_K2 = wl.LayerConfig("int4_pair_k2", T=16, H=768, E=64, k=4, I=128, bias=None, seed=41)
# the largest accepted expert count: the tile schedule over 1,024 experts, 256 routes
WIDE_E = wl.LayerConfig("int4_e1024", T=16, H=1024, E=1024, k=16, I=256, bias=None, seed=47)
GEOM = {"odd": ODD, "odd_k4": ODD_K4, "odd_k2": ODD_K2, "quad_k1": QUAD_K1, "pair_k2": PAIR_K2, "e1024": WIDE_E}


@pytest.mark.parametrize("name", ["tiny", "decode", "odd", "odd_k4", "odd_k2", "quad_k1", "pair_k2", "e1024"])
def test_int4_skewed_routes_split_tiles(name):
    """Decode-sized int4 launches run on the CUDA-core kernel, which splits an
    expert's rows into tiles of 4: routes skewed so that one expert gets 9
    rows (three tiles), others 1-5, graded row by row against the oracle.
    Down tiles span four, two or one 128-row blocks (by the block count) and
    ring slots hold four, two or one K steps: every combination the
    geometries allow is covered (gate/up 4 and 2 steps; down four blocks with
    2 and 1, two blocks with 2 and 1, one block with 4, 2 and 1)."""
    cfg = GEOM[name] if name in GEOM else wl.CONFIGS[name]
    T, k, E = 16, cfg.k, cfg.E
    d = wl.layer_inputs(cfg, DEV)
    q_gu, s_gu = wl.quantize_int4_g64(d["w_gateup"])
    q_d, s_d = wl.quantize_int4_g64(d["w_down"])
    rng = np.random.default_rng(17)
    ids_np = np.empty((T, k), np.int32)
    for t in range(T):
        pool = rng.permutation(np.arange(4, E))[:k].astype(np.int32)
        if t < 9:
            pool[0] = 1                       # expert 1: 9 rows
        if t % 3 == 0:
            pool[1] = 2                       # expert 2: 6 rows
        if t in (4, 5, 6, 7, 8):
            pool[2] = 3                       # expert 3: 5 rows
        ids_np[t] = pool
    assert all(len(set(r)) == k for r in ids_np)
    R = T * k
    assert R <= 320  # the CUDA-core path
    _, offsets_r, perm_r, _ = oracle.permute(ids_np, E)
    ids = torch.from_numpy(ids_np).to(DEV)
    counts = torch.empty((E,), dtype=torch.int32, device=DEV)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((R,), dtype=torch.int32, device=DEV)
    inv = torch.empty((R,), dtype=torch.int32, device=DEV)
    x = wl.token_batch(cfg, DEV, index=23, T=T)
    xp = torch.empty((R, cfg.H), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((R, cfg.I), dtype=torch.bfloat16, device=DEV)
    y = torch.full((R, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_permute(ids, E, x, counts, offsets, perm, inv, xp, st)
    gu, dn = pack_layer_experts(q_gu, q_d, _lib.MOE_W_INT4_G64, E, cfg.H, cfg.I, s_gateup=s_gu, s_down=s_d)
    _lib.moe_grouped_swiglu(xp, offsets, E, cfg.H, cfg.I, gu, dn, h, y, st, fmt=_lib.MOE_W_INT4_G64_TILED)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert int(counts[1].item()) == 9 and int(counts[2].item()) == 6 and int(counts[3].item()) == 5
    xin = oracle.bits_to_f32(oracle.bf16_bits(x))
    seg_e = np.searchsorted(offsets_r, np.arange(R), side="right") - 1
    tok = perm_r // k
    ref = oracle.experts_combine(xin[tok], seg_e.reshape(R, 1).astype(np.int32), np.ones((R, 1), np.float32),
                                 cfg.H, cfg.I, wgu_q=q_gu.cpu().numpy(), sgu_bits=oracle.bf16_bits(s_gu),
                                 wd_q=q_d.cpu().numpy(), sd_bits=oracle.bf16_bits(s_d))
    assert_output_close(y.cpu().numpy(), ref, what=f"int4 expert outputs, skewed routes ({name})")


def test_int4_launches_right_after_a_grouping_read_the_new_routes():
    """The int4 contractions start their weight stream before the launch in
    front of them ends only when that launch left their offsets as its
    token (the gate/up launch before a down launch, the row gather before a
    gate/up launch).  Here a grouping rewrites the offsets (other routes)
    right before a down launch, and right before a gate/up launch, on the
    same stream with nothing in between: the outputs must be those of the
    new routes, bit for bit (against the same launches after a full
    synchronisation)."""
    cfg = QUAD_K1
    T, k, E, H, I = 16, cfg.k, cfg.E, cfg.H, cfg.I
    d = wl.layer_inputs(cfg, DEV)
    q_gu, s_gu = wl.quantize_int4_g64(d["w_gateup"])
    q_d, s_d = wl.quantize_int4_g64(d["w_down"])
    gu, dn = pack_layer_experts(q_gu, q_d, _lib.MOE_W_INT4_G64, E, H, I, s_gateup=s_gu, s_down=s_d)
    fmt = _lib.MOE_W_INT4_G64_TILED
    R = T * k
    rng = np.random.default_rng(61)
    idsA = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)).to(DEV)
    idsB = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)).to(DEV)
    x = wl.token_batch(cfg, DEV, index=31, T=T)
    counts = torch.empty((E,), dtype=torch.int32, device=DEV)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((R,), dtype=torch.int32, device=DEV)
    inv = torch.empty((R,), dtype=torch.int32, device=DEV)
    xp = torch.empty((R, H), dtype=torch.bfloat16, device=DEV)
    hB = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    hA = torch.empty((R, I), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    # h of routes B, and the reference down outputs after a full sync
    _lib.moe_permute(idsB, E, x, counts, offsets, perm, inv, xp, st)
    _lib.moe_expert_gateup(xp, offsets, E, H, I, gu, hB, st, fmt=fmt)
    torch.cuda.synchronize()
    xpB = xp.clone()
    y_ref = torch.empty((R, H), dtype=torch.float32, device=DEV)
    _lib.moe_expert_down(hB, offsets, E, H, I, dn, y_ref, st, fmt=fmt)
    torch.cuda.synchronize()
    offsB = offsets.clone()
    for rep in range(3):
        # the gate/up -> down pair of routes A leaves the offsets of A ...
        _lib.moe_permute(idsA, E, x, counts, offsets, perm, inv, xp, st)
        _lib.moe_expert_gateup(xp, offsets, E, H, I, gu, hA, st, fmt=fmt)
        yA = torch.full((R, H), float("nan"), dtype=torch.float32, device=DEV)
        _lib.moe_expert_down(hA, offsets, E, H, I, dn, yA, st, fmt=fmt)
        # ... then the grouping of routes B and the down launch right after it
        _lib.moe_permute(idsB, E, None, counts, offsets, perm, inv, None, st)
        y = torch.full((R, H), float("nan"), dtype=torch.float32, device=DEV)
        _lib.moe_expert_down(hB, offsets, E, H, I, dn, y, st, fmt=fmt)
        # and routes A regrouped (no row gather) right before a gate/up
        # launch over routes B's rows: it must wait, and then read B's offsets
        _lib.moe_permute(idsA, E, None, counts, offsets, perm, inv, None, st)
        _lib.moe_permute(idsB, E, None, counts, offsets, perm, inv, None, st)
        h2 = torch.full((R, I), float("nan"), dtype=torch.bfloat16, device=DEV)
        _lib.moe_expert_gateup(xpB, offsets, E, H, I, gu, h2, st, fmt=fmt)
        torch.cuda.synchronize()
        assert st.item() == 0
        assert torch.equal(offsets, offsB)
        assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32)), rep
        assert torch.equal(h2.view(torch.int16), hB.view(torch.int16)), rep
        assert torch.isfinite(yA).all()


def test_int4_stack_forced_routes_six_layers():
    """Six layers free-running with the oracle's routes imposed on the GPU:
    the residual streams must agree to the stated tolerance."""
    T, L = 16, 6
    stack = make_stack(L, T)
    x0 = wl.token_batch(CFG, DEV, index=9, T=T).float()
    x = x0.clone()
    x_o = x0.cpu().numpy()
    for l in range(L):
        x_o_next, _, ids_r, w_r, _, _ = oracle_layer(x_o, l)
        ml = stack.layers[l]
        ml.ids[:T].copy_(torch.from_numpy(ids_r))
        ml.w[:T].copy_(torch.from_numpy(w_r))
        for call in stack.layer_calls(x, l, route=False):
            MoELayer.issue(call)
        x_o = x_o_next
    torch.cuda.synchronize()
    for ml in stack.layers:
        assert ml.read_status() == 0
    x0_np = x0.cpu().numpy().astype(np.float64)
    rel_max, mean_rel = assert_output_close(x.cpu().numpy() - x0_np, x_o - x0_np, what="6-layer residual update")
    print(f"6 layers forced routes: max err {rel_max:.2e} of max|ref|, mean rel {mean_rel:.2e}")


def _used_experts_host(w, ids):
    """Host copies of only the experts that ids name (the oracle reads whole
    records), and ids renumbered into that subset."""
    used = np.unique(ids)
    sel = torch.from_numpy(used.astype(np.int64)).to(DEV)
    host = {"wgu_q": w["w_gateup_q"].index_select(0, sel).cpu().numpy(),
            "sgu": oracle.bf16_bits(w["s_gateup"].index_select(0, sel)),
            "wd_q": w["w_down_q"].index_select(0, sel).cpu().numpy(),
            "sd": oracle.bf16_bits(w["s_down"].index_select(0, sel))}
    return host, np.searchsorted(used, ids).astype(np.int32)


def test_int4_stack_all_48_layers_teacher_forced():
    """Every layer of the 48-layer int4 stack (its own router and experts),
    one decode block of 16 tokens, graded per layer with teacher forcing: the
    oracle's layer l is fed the GPU's residual x_l (and, for the router and
    experts, the GPU's bf16 normalised input of it), so a legitimate near-tie
    flip in one layer cannot cascade.  Routes are graded as everywhere else;
    the residual update of every token whose route matches is graded against
    the oracle's int4 experts.  One layer's weights are held at a time."""
    T = 16
    x = wl.token_batch(CFG, DEV, index=11, T=T).float()
    graded = near = 0
    worst = (0.0, 0.0)
    for l in range(wl.STACK_LAYERS):
        w = wl.stack_layer_weights(l, DEV)
        gu, dn = pack_layer_experts(w["w_gateup_q"], w["w_down_q"], _lib.MOE_W_INT4_G64, CFG.E, CFG.H, CFG.I,
                                    s_gateup=w["s_gateup"], s_down=w["s_down"])
        ml = MoELayer(w["w_router"], None, gu, dn, CFG.k, T, fmt=_lib.MOE_W_INT4_G64_TILED, I=CFG.I)
        stack = MoEStack([ml], T)
        x_l = x.cpu().numpy()
        stack.forward(x)
        torch.cuda.synchronize()
        assert ml.read_status() == 0, l
        # RMSNorm graded on its own (within one bf16 rounding of the fp64
        # value); the router and experts are then graded on the GPU's own
        # normalised input, so a last-bit difference of that rounding cannot
        # move a logit
        n_bits = oracle.bf16_bits(stack.n[:T])
        n_ref = oracle.rmsnorm(x_l, None, eps=1e-6).astype(np.float64)
        n_gpu = oracle.bits_to_f32(n_bits).astype(np.float64)
        assert np.all(np.abs(n_gpu - n_ref) <= np.abs(n_ref) * 2.0 ** -8 + 1e-30), l
        ids_r, w_r, gap_r, L_r = oracle.route(n_bits, oracle.bf16_bits(w["w_router"]), None, CFG.k)
        rep = compare_routes(ml.ids[:T].cpu().numpy(), ml.w[:T].cpu().numpy(), ids_r, w_r, gap_r, L_r)
        keep = np.array(rep["exact_rows"], dtype=np.int64)
        assert len(keep) >= T - 3, (l, rep)
        host, local_ids = _used_experts_host(w, ids_r[keep])
        moe_ref = oracle.experts_combine(oracle.bits_to_f32(n_bits[keep]), local_ids, w_r[keep], CFG.H, CFG.I,
                                         wgu_q=host["wgu_q"], sgu_bits=host["sgu"], wd_q=host["wd_q"],
                                         sd_bits=host["sd"])
        moe_gpu = x.cpu().numpy().astype(np.float64)[keep] - x_l.astype(np.float64)[keep]
        rel_max, mean_rel = assert_output_close(moe_gpu, moe_ref, what=f"int4 stack layer {l} MoE output")
        worst = (max(worst[0], rel_max), max(worst[1], mean_rel))
        graded += len(keep)
        near += rep["near_tie"]
        del stack, ml, gu, dn, w
    print(f"48 layers teacher-forced: {graded}/{48 * T} token-layers graded, {near} near-ties; worst max err "
          f"{worst[0]:.2e} of max|ref|, worst mean rel {worst[1]:.2e}")


def test_stack_is_deterministic():
    T = 16
    stack = make_stack(3, T)
    x0 = wl.token_batch(CFG, DEV, index=2, T=T).float()
    a = x0.clone()
    b = x0.clone()
    stack.forward(a)
    stack.forward(b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def _repack_codes(codes):
    """Packed int4 word order: code + 8, nibble j holds element 0,2,4,6,1,3,5,7."""
    words = codes.reshape(codes.shape[0], -1, 4).view(np.uint32)[..., 0].astype(np.uint64)
    out = np.zeros_like(words)
    for e in range(8):
        n = ((words >> np.uint64(4 * e)) & np.uint64(0xF)) ^ np.uint64(8)
        pos = 4 + e // 2 if e % 2 else e // 2
        out |= n << np.uint64(4 * pos)
    return out.astype(np.uint32).view(np.uint8).reshape(codes.shape)


def _expected_pack(w_np, E, rows, K, I, which, s_np=None):
    """Test-side restatement of the packed layout (see include/moe.h)."""
    MB = (I // 64) if which == 0 else (rows // 128)
    KS = K // 64
    out = []
    for e in range(E):
        for mb in range(MB):
            for ks in range(KS):
                tile_rows = []
                for r in range(128):
                    if which == 0:
                        src = ((r >> 4) & 1) * I + mb * 64 + (r >> 5) * 16 + (r & 15)
                    else:
                        src = mb * 128 + r
                    tile_rows.append(src)
                if s_np is None:  # bf16: swizzled 128-byte rows
                    t = np.zeros((128, 64), np.uint16)
                    for r, src in enumerate(tile_rows):
                        row = w_np[e, src, ks * 64:(ks + 1) * 64].reshape(8, 8)
                        for c in range(8):
                            t[r, (c ^ (r & 7)) * 8:(c ^ (r & 7)) * 8 + 8] = row[c]
                    out.append(t.view(np.uint8).reshape(-1))
                else:
                    codes = np.stack([w_np[e, src, ks * 32:(ks + 1) * 32] for src in tile_rows])
                    codes = _repack_codes(codes)
                    sc = np.array([s_np[e, src, ks] for src in tile_rows], np.uint16)
                    out.append(np.concatenate([codes.reshape(-1), sc.view(np.uint8)]))
    return np.concatenate(out)


@pytest.mark.parametrize("which", [0, 1])
def test_pack_layouts_bit_exact(which):
    cfg = wl.TINY
    d = wl.layer_inputs(cfg, DEV)
    w = d["w_gateup"] if which == 0 else d["w_down"]
    rows, K = (2 * cfg.I, cfg.H) if which == 0 else (cfg.H, cfg.I)
    got = _lib.moe_pack_experts(_lib.MOE_W_BF16, w, None, cfg.E, cfg.H, cfg.I, which).cpu().numpy()
    exp = _expected_pack(oracle.bf16_bits(w), cfg.E, rows, K, cfg.I, which)
    assert np.array_equal(got, exp)
    q, sc = wl.quantize_int4_g64(w)
    got4 = _lib.moe_pack_experts(_lib.MOE_W_INT4_G64, q, sc, cfg.E, cfg.H, cfg.I, which).cpu().numpy()
    exp4 = _expected_pack(q.cpu().numpy(), cfg.E, rows, K, cfg.I, which, s_np=oracle.bf16_bits(sc))
    assert np.array_equal(got4, exp4)

