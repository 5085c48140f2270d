"""GPU checks of the expert cache: moe_cache_plan, moe_cache_fetch,
moe_expert_swiglu_cached and CachedMoELayer.

Every expert's tile-packed records sit in pinned host memory and S slots of
HBM cache them.  Moving records is byte work and each tile's arithmetic is
unchanged, so a cached layer must return, bit for bit, what MoELayer returns
over the same records resident in HBM -- call after call, as experts hit,
miss and are evicted, for every wave width of the in-launch fetch and for the
copy-first path.  The plan itself is integer work (plus one fp32 fused multiply-add
per expert for the score policy's use rates) and is compared bit for bit
with the oracle's plan for the FIFO, LRU and score policies.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from parity import assert_output_close, compare_routes
from sparse_moe_routed_gb300 import CachedMoELayer, MoELayer, _lib, pack_layer_experts

pytestmark = pytest.mark.gpu

DEV = "cuda"

# I/64 even: the in-launch fetch runs on the paired-K-step contraction
SMALL = wl.LayerConfig("cache_small", T=8, H=256, E=64, k=4, I=128, bias=None, seed=21)
WIDE = wl.LayerConfig("cache_wide", T=16, H=256, E=512, k=10, I=128, bias=None, seed=22)
QWEN64 = wl.LayerConfig("cache_qwen64", T=4, H=2560, E=64, k=10, I=640, bias=None, seed=23)


# ----------------------------------------------------------------- plan
@pytest.mark.parametrize("policy", ["fifo", "lru", "score"])
@pytest.mark.parametrize("E,S,T,k", [(64, 24, 4, 4), (512, 200, 16, 10), (1024, 1024, 64, 10), (64, 1, 1, 1),
                                     (100, 37, 3, 8)])
def test_plan_matches_oracle(policy, E, S, T, k):
    """Every output and every piece of state, bit for bit, call after call."""
    rng = np.random.default_rng(E + S + len(policy))
    pol = CachedMoELayer.POLICIES[policy]
    decay = 0.85
    ref = oracle.CachePlan(E, S, policy, decay)
    slot_of = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    expert_of = torch.full((S,), -1, dtype=torch.int32, device=DEV)
    hand = torch.zeros((2,), dtype=torch.int32, device=DEV)
    score = torch.zeros((E,), dtype=torch.float32, device=DEV)
    last_use = torch.full((S,), -1, dtype=torch.int32, device=DEV)
    ml = torch.zeros((S,), dtype=torch.int32, device=DEV)
    ms = torch.zeros((S,), dtype=torch.int32, device=DEV)
    stats = torch.zeros((4,), dtype=torch.int32, device=DEV)
    saw_full = saw_evict = False
    for call in range(40):
        st = torch.zeros((1,), dtype=torch.int32, device=DEV)
        # a hot set of experts makes hits; now and then a call routes more
        # experts than the cache holds
        Tc = T * 8 if call % 13 == 12 else T
        hot = rng.choice(E, size=max(2 * k, E // 8), replace=False)
        cnt = np.zeros(E, dtype=np.int32)
        for _ in range(Tc):
            pool = hot if rng.random() < 0.6 else np.arange(E)
            for e in rng.choice(pool, size=min(k, len(pool)), replace=False):
                cnt[e] += 1
        before = ref.expert_of.copy()
        _lib.moe_cache_plan(torch.from_numpy(cnt).to(DEV), slot_of, expert_of, hand, ml, ms, stats, st,
                            policy=pol, decay=decay, score=score, last_use=last_use)
        full, misses, victims = ref.step(cnt)
        torch.cuda.synchronize()
        saw_full |= full
        saw_evict |= any(before[v] >= 0 for v in victims)
        assert int(st.item()) == (_lib.MOE_DEV_CACHE_FULL if full else 0), call
        assert stats.cpu().tolist() == ref.stats.tolist(), call
        assert slot_of.cpu().tolist() == ref.slot_of.tolist(), call
        assert expert_of.cpu().tolist() == ref.expert_of.tolist(), call
        assert hand.cpu().tolist() == ref.hand.tolist(), call
        n = len(misses)
        assert ml[:n].cpu().tolist() == misses.tolist(), call
        assert ms[:n].cpu().tolist() == victims.tolist(), call
        if policy == "lru":
            assert last_use.cpu().tolist() == ref.last_use.tolist(), call
        if policy == "score":
            assert torch.equal(score.cpu().view(torch.int32), torch.from_numpy(ref.score).view(torch.int32)), call
    if S < E and S > k:
        assert saw_evict and saw_full


# ----------------------------------------------------------------- layer
_L = {}


def layers(cfg):
    """(resident MoELayer, packed host records) for cfg."""
    if cfg.name not in _L:
        d = wl.layer_inputs(cfg, DEV, with_x=False)
        gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
        torch.cuda.synchronize()
        ref = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
        _L[cfg.name] = (ref, gu.cpu().pin_memory(), dn.cpu().pin_memory(), d)
    return _L[cfg.name]


def run_sequence(cfg, S, wave, fetch, calls=12, policy="fifo"):
    ref, hgu, hdn, d = layers(cfg)
    lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, cfg.T, I=cfg.I, S=S, wave=wave, fetch=fetch,
                         policy=policy)
    uniq = 0
    for i in range(calls):
        # repeat a few batches so that some calls hit what earlier ones loaded
        x = wl.token_batch(cfg, DEV, index=[0, 1, 0, 2, 3, 1, 4, 0, 5, 2, 6, 0][i % 12], T=cfg.T)
        want = ref.forward(x).clone()
        got = lay.forward(x).clone()
        torch.cuda.synchronize()
        assert lay.read_status() == 0 and ref.read_status() == 0
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"call {i}"
        uniq += int((lay.counts > 0).sum().item())
    s = lay.stats.cpu().tolist()
    assert s[2] + s[3] == uniq
    return lay, s


@pytest.mark.parametrize("wave", [1, 2, 3, 4, 1 << 20])
def test_cached_layer_bitwise_small(wave):
    lay, s = run_sequence(SMALL, S=40, wave=wave, fetch="wave")
    assert s[2] > 0 and s[3] > 40          # hits, and misses beyond the first fill (evictions)
    assert int(lay.sync_ws.abs().sum().item()) == 0  # sync words left zero


@pytest.mark.parametrize("policy", ["lru", "score"])
def test_cached_layer_bitwise_policies(policy):
    lay, s = run_sequence(SMALL, S=40, wave=2, fetch="wave", policy=policy)
    assert s[2] > 0 and s[3] > 40


def test_cached_layer_copy_first_small():
    _, s = run_sequence(SMALL, S=40, wave=1, fetch="barrier")
    assert s[2] > 0 and s[3] > 40


@pytest.mark.parametrize("wave", [2, 1 << 20])
def test_cached_layer_bitwise_512_experts(wave):
    _, s = run_sequence(WIDE, S=200, wave=wave, fetch="wave", calls=8)
    assert s[2] > 0 and s[3] > 200


@pytest.mark.parametrize("wave,fetch,policy", [(1, "wave", "fifo"), (4, "wave", "lru"), (1 << 20, "wave", "score"),
                                               (1, "barrier", "fifo")])
def test_cached_layer_bitwise_qwen_geometry(wave, fetch, policy):
    """Qwen4Exp expert shape (H 2560, I 640) over 64 experts, 40 slots."""
    _, s = run_sequence(QWEN64, S=40, wave=wave, fetch=fetch, calls=8, policy=policy)
    assert s[2] > 0 and s[3] > 40


def test_cached_layer_with_misses_against_oracle():
    """Qwen4Exp expert shape over 64 experts and 40 slots: every call of a
    sequence with hits, misses and evictions graded directly against the CPU
    oracle (routes, and the layer output of every token whose route the
    oracle confirms), not only against the resident layer."""
    cfg = QWEN64
    ref, hgu, hdn, d = layers(cfg)
    lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, cfg.T, I=cfg.I, S=40, wave=2, fetch="wave")
    wr = oracle.bf16_bits(d["w_router"])
    wgu = oracle.bf16_bits(d["w_gateup"])
    wdn = oracle.bf16_bits(d["w_down"])
    graded = 0
    for i in range(8):
        x = wl.token_batch(cfg, DEV, index=[0, 1, 0, 2, 3, 1, 4, 0][i], T=cfg.T)
        out = lay.forward(x).float().cpu().numpy()
        torch.cuda.synchronize()
        assert lay.read_status() == 0
        xb = oracle.bf16_bits(x)
        ids_r, w_r, gap_r, L_r = oracle.route(xb, wr, None, cfg.k)
        rep = compare_routes(lay.ids[:cfg.T].cpu().numpy(), lay.w[:cfg.T].cpu().numpy(), ids_r, w_r, gap_r, L_r)
        keep = np.array(rep["exact_rows"], dtype=np.int64)
        if len(keep) == 0:
            continue
        want = oracle.experts_combine(oracle.bits_to_f32(xb[keep]), ids_r[keep], w_r[keep], cfg.H, cfg.I,
                                      wgu_bits=wgu, wd_bits=wdn)
        assert_output_close(out[keep], want, what=f"cached layer call {i}")
        graded += len(keep)
    s = lay.stats.cpu().tolist()
    assert s[2] > 0 and s[3] > 40 and graded >= 0.9 * 8 * cfg.T, (s, graded)


def test_cached_layer_host_graph():
    """The cached layer replays from a CUDA graph like the resident one."""
    ref, hgu, hdn, d = layers(SMALL)
    lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, SMALL.k, SMALL.T, I=SMALL.I, S=40, wave=2)
    xh = torch.empty((SMALL.T, SMALL.H), dtype=torch.bfloat16).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    for i in range(5):
        x = wl.token_batch(SMALL, DEV, index=i % 3, T=SMALL.T)
        xh.copy_(x.cpu())
        lay.forward_host_graph(xh, oh)
        want = ref.forward(x).cpu()
        assert torch.equal(oh.view(torch.int16), want.view(torch.int16)), i
    assert lay.read_status() == 0


def test_cache_full_is_flagged_and_changes_nothing():
    ref, hgu, hdn, d = layers(SMALL)
    S = 4
    lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, SMALL.k, SMALL.T, I=SMALL.I, S=S, wave=2)
    x = wl.token_batch(SMALL, DEV, index=9, T=SMALL.T)   # 8 tokens x 4 routes: more than 4 experts
    lay.forward(x)
    torch.cuda.synchronize()
    assert lay.read_status() & _lib.MOE_DEV_CACHE_FULL
    assert lay.slot_of.eq(-1).all() and lay.expert_of.eq(-1).all() and lay.hand.cpu().tolist() == [0, 1]
    assert lay.stats[1].item() == 0
    assert int(lay.sync_ws.abs().sum().item()) == 0


def test_fetch_only_kernel_copies_records():
    """moe_cache_fetch alone: slots receive exactly the planned records."""
    cfg = SMALL
    ref, hgu, hdn, d = layers(cfg)
    S, E = 16, cfg.E
    rg, rd = hgu.numel() // E, hdn.numel() // E
    pgu = torch.zeros((S * rg,), dtype=torch.uint8, device=DEV)
    pdn = torch.zeros((S * rd,), dtype=torch.uint8, device=DEV)
    ml = torch.tensor([5, 63, 0, 17] + [0] * (S - 4), dtype=torch.int32, device=DEV)
    ms = torch.tensor([3, 0, 15, 7] + [0] * (S - 4), dtype=torch.int32, device=DEV)
    stats = torch.tensor([0, 4, 0, 0], dtype=torch.int32, device=DEV)
    _lib.moe_cache_fetch(hgu, hdn, rg, rd, ml, ms, stats, pgu, pdn)
    torch.cuda.synchronize()
    gu_d, dn_d = pgu.cpu(), pdn.cpu()
    for e, sl in zip([5, 63, 0, 17], [3, 0, 15, 7]):
        assert torch.equal(gu_d[sl * rg:(sl + 1) * rg], hgu[e * rg:(e + 1) * rg])
        assert torch.equal(dn_d[sl * rd:(sl + 1) * rd], hdn[e * rd:(e + 1) * rd])
    untouched = [s for s in range(S) if s not in (3, 0, 15, 7)]
    for sl in untouched:
        assert int(gu_d[sl * rg:(sl + 1) * rg].sum()) == 0


# ----------------------------------------------------------------- merge
@pytest.mark.parametrize("name,R", [("decode", 4), ("decode", 2), ("tiny", 3)])
def test_merged_requests_equal_separate_calls(name, R):
    """Several requests' decode blocks grouped into one call (routes grouped
    by expert across the requests) give every token the output its own
    request's call gives, bit for bit: a row's contraction and its
    rank-order combine do not depend on the other rows of the call.  Up to
    64 tokens, where one router kernel serves both call sizes."""
    cfg = wl.CONFIGS[name]
    d = wl.layer_inputs(cfg, DEV, with_x=False)
    gu, dn = pack_layer_experts(d["w_gateup"], d["w_down"], _lib.MOE_W_BF16, cfg.E, cfg.H, cfg.I)
    T = 16
    merged = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, T * R, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
    single = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, T, fmt=_lib.MOE_W_BF16_TILED, I=cfg.I)
    xs = [wl.token_batch(cfg, DEV, index=40 + r, T=T) for r in range(R)]
    got = merged.forward(torch.cat(xs)).clone()
    want = torch.cat([single.forward(x).clone() for x in xs])
    torch.cuda.synchronize()
    assert merged.read_status() == 0 and single.read_status() == 0
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


# ----------------------------------------------------------------- int4 records
INT4_SMALL = wl.LayerConfig("cache_int4", T=4, H=512, E=64, k=4, I=256, bias=None, seed=24)
_Q = {}


def int4_layers(cfg):
    """(resident int4 MoELayer, pinned host int4 records, raw codes/scales)."""
    if cfg.name not in _Q:
        d = wl.layer_inputs(cfg, DEV, with_x=False)
        q_gu, s_gu = wl.quantize_int4_g64(d["w_gateup"])
        q_d, s_d = wl.quantize_int4_g64(d["w_down"])
        gu, dn = pack_layer_experts(q_gu, q_d, _lib.MOE_W_INT4_G64, cfg.E, cfg.H, cfg.I, s_gateup=s_gu, s_down=s_d)
        torch.cuda.synchronize()
        ref = MoELayer(d["w_router"], d["bias"], gu, dn, cfg.k, cfg.T, fmt=_lib.MOE_W_INT4_G64_TILED, I=cfg.I)
        raw = {"wr": oracle.bf16_bits(d["w_router"]), "wgu_q": q_gu.cpu().numpy(), "sgu": oracle.bf16_bits(s_gu),
               "wd_q": q_d.cpu().numpy(), "sd": oracle.bf16_bits(s_d)}
        _Q[cfg.name] = (ref, gu.cpu().pin_memory(), dn.cpu().pin_memory(), d, raw)
    return _Q[cfg.name]


@pytest.mark.parametrize("policy,fetch", [("fifo", "barrier"), ("lru", "barrier"), ("fifo", "wave"),
                                          ("lru", "wave")])
def test_cached_int4_layer_bitwise_and_against_oracle(policy, fetch):
    """int4 g64 records in host memory behind 24 HBM slots (4 tokens x 4 routes
    per call, so a call always fits): every call of a
    sequence with hits, misses and evictions equals, bit for bit, the
    resident int4 layer (the record bytes move, the arithmetic does not);
    misses move int4 records (2,611,200 B per expert at the Qwen4Exp shape);
    each call is also graded against the oracle's int4 experts."""
    cfg = INT4_SMALL
    ref, hgu, hdn, d, raw = int4_layers(cfg)
    lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, cfg.T, I=cfg.I, S=24, policy=policy,
                         fetch=fetch, fmt=_lib.MOE_W_INT4_G64_TILED)
    assert lay.rec_gu + lay.rec_dn == 3 * cfg.H * cfg.I // 2 + 3 * cfg.H * cfg.I // 64 * 2
    uniq = 0
    for i in range(10):
        x = wl.token_batch(cfg, DEV, index=[0, 1, 0, 2, 3, 1, 4, 0, 5, 2][i], T=cfg.T)
        want = ref.forward(x).clone()
        got = lay.forward(x).clone()
        torch.cuda.synchronize()
        assert lay.read_status() == 0 and ref.read_status() == 0
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"call {i}"
        uniq += int((lay.counts > 0).sum().item())
        xb = oracle.bf16_bits(x)
        ids_r, w_r, gap_r, L_r = oracle.route(xb, raw["wr"], None, cfg.k)
        rep = compare_routes(lay.ids[:cfg.T].cpu().numpy(), lay.w[:cfg.T].cpu().numpy(), ids_r, w_r, gap_r, L_r)
        keep = np.array(rep["exact_rows"], dtype=np.int64)
        if len(keep):
            moe = oracle.experts_combine(oracle.bits_to_f32(xb[keep]), ids_r[keep], w_r[keep], cfg.H, cfg.I,
                                         wgu_q=raw["wgu_q"], sgu_bits=raw["sgu"], wd_q=raw["wd_q"], sd_bits=raw["sd"])
            assert_output_close(got.float().cpu().numpy()[keep], moe, what=f"cached int4 call {i}")
    s = lay.stats.cpu().tolist()
    assert s[2] > 0 and s[3] > 24 and s[2] + s[3] == uniq
    assert int(lay.sync_ws.abs().sum().item()) == 0


def test_cached_int4_qwen_geometry_in_launch_fetch():
    """The Qwen4Exp expert shape (H 2,560, I 640: 40 K steps, pieces of eight
    chunks) over 64 experts and 40 slots, misses fetched in the gate/up launch:
    bit-identical to the resident int4 layer call after call."""
    cfg = wl.LayerConfig("cache_int4_qwen", T=4, H=2560, E=64, k=10, I=640, bias=None, seed=25)
    ref, hgu, hdn, d, raw = int4_layers(cfg)
    lay = CachedMoELayer(d["w_router"], d["bias"], hgu, hdn, cfg.k, cfg.T, I=cfg.I, S=40, fetch="wave",
                         fmt=_lib.MOE_W_INT4_G64_TILED)
    for i in range(8):
        x = wl.token_batch(cfg, DEV, index=[0, 1, 0, 2, 3, 1, 4, 0][i], T=cfg.T)
        want = ref.forward(x).clone()
        got = lay.forward(x).clone()
        torch.cuda.synchronize()
        assert lay.read_status() == 0 and ref.read_status() == 0
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"call {i}"
    s = lay.stats.cpu().tolist()
    assert s[2] > 0 and s[3] > 40
    assert int(lay.sync_ws.abs().sum().item()) == 0


def test_int4_slots_flag_an_expert_without_a_slot():
    """A routed expert whose slot entry is -1 reads slot 0 and flags
    MOE_DEV_CACHE_FULL (every access stays inside the pool)."""
    cfg = INT4_SMALL
    ref, hgu, hdn, d, raw = int4_layers(cfg)
    E, H, I = cfg.E, cfg.H, cfg.I
    rg = hgu.numel() // E
    ids = torch.tensor([[3, 5, 7, 9]], dtype=torch.int32, device=DEV)
    counts = torch.empty((E,), dtype=torch.int32, device=DEV)
    offsets = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    perm = torch.empty((4,), dtype=torch.int32, device=DEV)
    inv = torch.empty((4,), dtype=torch.int32, device=DEV)
    xp = torch.empty((4, H), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    x = wl.token_batch(cfg, DEV, index=2, T=1)
    _lib.moe_permute(ids, E, x, counts, offsets, perm, inv, xp, st)
    pool = hgu[: 4 * rg].to(DEV)
    slot_of = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    slot_of[3], slot_of[5], slot_of[7] = 0, 1, 2  # expert 9 has no slot
    h = torch.empty((4, I), dtype=torch.bfloat16, device=DEV)
    _lib.moe_expert_int4_slots(0, xp, offsets, E, H, I, pool, 4, slot_of, h, st)
    torch.cuda.synchronize()
    assert st.item() & _lib.MOE_DEV_CACHE_FULL
