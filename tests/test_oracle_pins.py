"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test names what fixes the expected value: a figure the pages print
(tests/golden/page_figures.json, each with its note and section), a closed
form, brute force on tiny inputs, or a special case that reduces to a library
routine.  A plausible slip in the oracle (dropped term, wrong sign or index,
transposed operand, unstable grouping, wrong tie order) fails at least one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
GEO = GOLD["geometry"]


def bf16_round_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (test-side helper)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def bits_f64(b):
    return oracle.bits_to_f32(b).astype(np.float64)


# --------------------------------------------------------------------------
# Figures the pages print
# --------------------------------------------------------------------------
def test_page_params_per_expert_and_uses():
    H, I = GEO["hidden"], GEO["intermediate"]
    # one expert record through the oracle's byte accounting: bytes at 8 bits = params
    ids = np.arange(1, dtype=np.int32).reshape(1, 1, 1)
    _, U, b2, b4 = oracle.dedup(ids, E=GEO["experts"], block=1, H=H, I=I)
    assert U[0, 0] == 1
    assert b4[0] * 2 == GOLD["params_per_expert"]["value"]
    assert b2[0] * 4 == GOLD["params_per_expert"]["value"]
    assert GEO["layers"] * GEO["top_k"] * b4[0] * 2 == GOLD["param_uses_per_token"]["value"]


def test_page_cold_payload_per_token():
    """T=1, 48 layers, 10 distinct experts per layer -> 562.5 MiB / 1.0986 GiB."""
    L, E, k = GEO["layers"], GEO["experts"], GEO["top_k"]
    rng = np.random.default_rng(0)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(L)]).astype(np.int32)
    ids = ids.reshape(L, 1, k)
    mask, U, b2, b4 = oracle.dedup(ids, E=E, block=1, H=GEO["hidden"], I=GEO["intermediate"])
    assert (U == k).all()
    mib = b2[0] / 2**20
    gib = b4[0] / 2**30
    g2, g4 = GOLD["cold_payload_2bit_mib"], GOLD["cold_payload_4bit_gib"]
    assert round(mib, g2["digits"]) == g2["value"]
    assert round(gib, g4["digits"]) == g4["value"]


def test_page_label_and_intermediate_sizes():
    """Route label = int32 ID + fp32 weight; intermediate [k, I] fp32."""
    rng = np.random.default_rng(1)
    x = bf16_round_bits(rng.standard_normal((2, 64)).astype(np.float32))
    wr = bf16_round_bits((0.02 * rng.standard_normal((GEO["experts"], 64))).astype(np.float32))
    ids, w, gap, _ = oracle.route(x, wr, None, GEO["top_k"])
    per_layer = ids.shape[1] * (ids.itemsize + w.itemsize)
    assert per_layer * GEO["layers"] == GOLD["label_bytes_per_token"]["value"]
    f = GOLD["f32_intermediate_bytes"]
    assert GEO["top_k"] * GEO["intermediate"] * 4 == f["per_layer_token"]
    assert f["per_layer_token"] * GEO["layers"] == f["per_token"]


def test_page_break_even_worst_case():
    """Block of 5 with all-distinct routes reaches the worst case 50 = 10 * 5."""
    be = GOLD["break_even_example"]
    E, k = GEO["experts"], GEO["top_k"]
    ids = np.arange(be["block"] * k, dtype=np.int32).reshape(1, be["block"], k)
    _, U, _, _ = oracle.dedup(ids, E=E, block=be["block"], H=8, I=8)
    assert U[0, 0] == be["worst_case"]
    assert k * be["tau"] == be["bound"]
    # a block whose five tokens share one route: U = 10 < 40
    same = np.tile(np.arange(k, dtype=np.int32), (be["block"], 1)).reshape(1, be["block"], k)
    _, U2, _, _ = oracle.dedup(same, E=E, block=be["block"], H=8, I=8)
    assert U2[0, 0] == k and U2[0, 0] < be["bound"]


# --------------------------------------------------------------------------
# Router logits: library matmul and closed forms
# --------------------------------------------------------------------------
def test_logits_match_float64_matmul():
    rng = np.random.default_rng(2)
    T, H, E = 5, 96, 24
    x = bf16_round_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = bf16_round_bits((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    b = rng.standard_normal(E).astype(np.float32)
    L = oracle.router_logits(x, wr, b)
    ref = (bits_f64(x) @ bits_f64(wr).T + b.astype(np.float64)).astype(np.float32)
    assert np.array_equal(L, ref) or np.max(np.abs(L - ref)) <= 1e-6 * np.max(np.abs(ref))
    # rows / columns not swapped: token 0 against expert 3 by hand
    hand = sum(bits_f64(x)[0, h] * bits_f64(wr)[3, h] for h in range(H)) + float(b[3])
    assert abs(float(L[0, 3]) - hand) <= 1e-6 * max(1.0, abs(hand))


def test_logits_zero_weights_equal_bias():
    x = bf16_round_bits(np.ones((3, 32), np.float32))
    wr = np.zeros((7, 32), np.uint16)
    b = np.arange(7, dtype=np.float32) - 3.5
    L = oracle.router_logits(x, wr, b)
    assert np.array_equal(L, np.tile(b, (3, 1)))


# --------------------------------------------------------------------------
# Top-k: brute force rank, tie contract, softmax special case
# --------------------------------------------------------------------------
def _brute_rank_topk(row, k):
    """Expert e has rank #{e': v[e'] > v[e] or (v[e'] == v[e] and e' < e)}."""
    E = len(row)
    rank = [sum(1 for f in range(E) if row[f] > row[e] or (row[f] == row[e] and f < e))
            for e in range(E)]
    out = [None] * k
    for e in range(E):
        if rank[e] < k:
            out[rank[e]] = e
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force(seed):
    rng = np.random.default_rng(10 + seed)
    T, E, k = 8, 12, 5
    # coarse values to force many exact ties
    L = rng.integers(-3, 4, size=(T, E)).astype(np.float32) * 0.5
    ids, w, gap = oracle.topk(L, k)
    for t in range(T):
        assert list(ids[t]) == _brute_rank_topk(list(L[t]), k)
        srt = sorted(L[t], reverse=True)
        assert gap[t] == np.float32(srt[k - 1] - srt[k])


def test_topk_tie_contract():
    """Equal logits: lower ID wins and equal-logit IDs come out in ID order."""
    L = np.zeros((1, 9), np.float32)
    ids, w, gap = oracle.topk(L, 4)
    assert list(ids[0]) == [0, 1, 2, 3]
    assert np.allclose(w, 0.25, atol=0, rtol=0)
    assert gap[0] == 0.0
    L2 = np.array([[1, 5, 5, 2, 5, 0]], np.float32)
    ids2, _, _ = oracle.topk(L2, 4)
    assert list(ids2[0]) == [1, 2, 4, 3]


def test_topk_weights_sum_monotone_and_full_softmax():
    rng = np.random.default_rng(3)
    T, E = 16, 32
    L = rng.standard_normal((T, E)).astype(np.float32)
    ids, w, _ = oracle.topk(L, 10)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= 1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)
    # k == E: renormalised top-k is the full softmax (library routine)
    idsE, wE, gapE = oracle.topk(L, E)
    sm = scipy.special.softmax(L.astype(np.float64), axis=1)
    for t in range(T):
        assert np.allclose(wE[t], sm[t, idsE[t]], rtol=1e-6, atol=1e-9)
    assert np.all(np.isinf(gapE))
    # renormalised top-k equals the full softmax divided by the top-k mass
    for t in range(T):
        mass = sm[t, ids[t]].sum()
        assert np.allclose(w[t], sm[t, ids[t]] / mass, rtol=1e-6, atol=1e-9)


# --------------------------------------------------------------------------
# Grouping by expert
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 3, 5), (16, 4, 64), (33, 10, 512)])
def test_permute_invariants_and_stable_argsort(T, k, E):
    rng = np.random.default_rng(T * 31 + E)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, inv = oracle.permute(ids, E)
    R = T * k
    flat = ids.reshape(-1)
    assert counts.sum() == R and offsets[0] == 0 and offsets[E] == R
    assert np.array_equal(np.bincount(flat, minlength=E), counts)
    assert np.array_equal(perm[inv], np.arange(R)) and np.array_equal(inv[perm], np.arange(R))
    # stable grouping == numpy's stable argsort by expert (library routine)
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    # gather(scatter(x)) == x
    x = rng.standard_normal((T, 3))
    xp = x[perm // k]
    back = xp[inv].reshape(T, k, 3)
    assert np.array_equal(back, np.repeat(x[:, None, :], k, axis=1))


def test_permute_rejects_bad_id():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 5]], np.int32), 5)
    with pytest.raises(ValueError):
        oracle.permute(np.array([[-1, 2]], np.int32), 5)


# --------------------------------------------------------------------------
# Expert SwiGLU and combine
# --------------------------------------------------------------------------
def _rand_expert(rng, E, H, I, std=0.05):
    wgu = bf16_round_bits((std * rng.standard_normal((E, 2 * I, H))).astype(np.float32))
    wd = bf16_round_bits((std * rng.standard_normal((E, H, I))).astype(np.float32))
    return wgu, wd


def test_single_expert_is_dense_swiglu_mlp():
    """E=1, k=1: the layer is one dense SwiGLU MLP (numpy matmuls + scipy expit)."""
    rng = np.random.default_rng(4)
    H, I, n = 48, 80, 6
    wgu, wd = _rand_expert(rng, 1, H, I, std=0.2)
    x = rng.standard_normal((n, H)).astype(np.float32)
    y = oracle.expert_rows(x, wgu, wd, 0, H, I)
    Wg, Wu = bits_f64(wgu[0, :I]), bits_f64(wgu[0, I:])
    Wd = bits_f64(wd[0])
    g = x.astype(np.float64) @ Wg.T
    u = x.astype(np.float64) @ Wu.T
    ref = (g * scipy.special.expit(g) * u) @ Wd.T
    assert np.allclose(y, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())


def test_expert_closed_form_saturated_gate():
    """H = I, Wg = 64*Id, Wu = Id, Wd = Id: y_i = 64 x_i^2 for x_i >= 1, 0 for x_i <= -1."""
    H = I = 16
    one, c = 0x3F80, 0x4280  # bf16 bits of 1.0 and 64.0
    wgu = np.zeros((1, 2 * I, H), np.uint16)
    wd = np.zeros((1, H, I), np.uint16)
    for i in range(I):
        wgu[0, i, i] = c
        wgu[0, I + i, i] = one
        wd[0, i, i] = one
    x = np.array([[1.0, 2.0, -1.0, -3.0] * 4], np.float32)
    y = oracle.expert_rows(x, wgu, wd, 0, H, I)[0]
    expect = np.where(x[0] > 0, 64.0 * x[0] ** 2, 0.0)
    # silu(64) = 64 * (1 - 1.6e-28) and silu(-64) = -1.0e-26: exact to fp32 here
    assert np.allclose(y, expect, rtol=1e-7, atol=1e-20)


def test_combine_rank_order_weights():
    """out = sum_j w_j y_{e_j}; identical experts -> out = y (weights sum to 1)."""
    rng = np.random.default_rng(5)
    H, I, E, k, n = 32, 16, 6, 3, 4
    wgu, wd = _rand_expert(rng, E, H, I, std=0.3)
    x = rng.standard_normal((n, H)).astype(np.float32)
    ids = np.array([[0, 3, 5], [5, 3, 0], [1, 2, 4], [4, 0, 2]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.6, 0.3, 0.1], [1 / 3, 1 / 3, 1 / 3], [0.9, 0.05, 0.05]], np.float32)
    out = oracle.experts_combine(x, ids, w, H, I, wgu_bits=wgu, wd_bits=wd)
    ys = [oracle.expert_rows(x, wgu, wd, e, H, I) for e in range(E)]
    for t in range(n):
        ref = sum(float(w[t, j]) * ys[ids[t, j]][t].astype(np.float64) for j in range(k))
        assert np.allclose(out[t], ref, rtol=1e-5, atol=1e-7)
    same_gu = np.repeat(wgu[:1], E, axis=0)
    same_d = np.repeat(wd[:1], E, axis=0)
    out_same = oracle.experts_combine(x, ids, w, H, I, wgu_bits=same_gu, wd_bits=same_d)
    assert np.allclose(out_same, ys[0], rtol=1e-5, atol=1e-7)


# --------------------------------------------------------------------------
# int4 g64 codec
# --------------------------------------------------------------------------
def test_int4_nibble_order_and_sign():
    q = np.array([[0x8F, 0x70] + [0] * 30], np.uint8)  # K = 64, one group
    s = np.array([[0x3F80]], np.uint16)  # scale 1.0
    w = oracle.dequant_int4(q, s)
    assert w.shape == (1, 64)
    assert list(w[0, :4]) == [-1.0, -8.0, 0.0, 7.0]


def test_int4_roundtrip_and_error_bound():
    import torch
    from workloads import quantize_int4_g64
    rng = np.random.default_rng(6)
    wf = (0.02 * rng.standard_normal((5, 256))).astype(np.float32)
    wt = torch.from_numpy(wf).to(torch.bfloat16)
    q, s = quantize_int4_g64(wt)
    s_bits = oracle.bf16_bits(s)
    deq = oracle.dequant_int4(q.numpy(), s_bits)
    ref = wt.to(torch.float32).numpy()
    sc = np.repeat(oracle.bits_to_f32(s_bits), 64, axis=-1)
    assert np.all(np.abs(deq - ref) <= sc / 2 + 1e-12)
    q2, s2 = quantize_int4_g64(torch.from_numpy(deq).to(torch.bfloat16))
    assert np.array_equal(q2.numpy(), q.numpy())


def _pack_int4(codes):
    """[..., K] signed codes in [-8, 7] -> [..., K/2] bytes, even input in the
    low nibble (test-side packing, written from the codec's statement)."""
    c = (np.asarray(codes, np.int64) & 0xF).astype(np.uint8)
    return np.ascontiguousarray(c[..., 0::2] | (c[..., 1::2] << 4))


def _rand_int4_experts(rng, E, H, I, pow2_scales):
    """Random int4 g64 expert records: codes [E,2I,H/2] / [E,H,I/2] and bf16
    scales [E,2I,H/64] / [E,H,I/64]; with pow2_scales every scale is a power
    of two, so each scale * code is exact in bf16."""
    qgu = rng.integers(-8, 8, size=(E, 2 * I, H))
    qd = rng.integers(-8, 8, size=(E, H, I))
    if pow2_scales:
        sgu = 2.0 ** rng.integers(-9, -4, size=(E, 2 * I, H // 64))
        sd = 2.0 ** rng.integers(-9, -4, size=(E, H, I // 64))
    else:
        sgu = 0.003 * (1 + rng.random((E, 2 * I, H // 64)))
        sd = 0.003 * (1 + rng.random((E, H, I // 64)))
    return (qgu, _pack_int4(qgu), bf16_round_bits(sgu.astype(np.float32)),
            qd, _pack_int4(qd), bf16_round_bits(sd.astype(np.float32)))


def test_int4_experts_equal_bf16_experts_on_exact_dequant():
    """int4 records whose scale * code is exact in bf16 (power-of-two scales):
    the int4 branch of the expert combine must give the same bits as the bf16
    branch fed the dequantised weights.  Several experts and routes, so a
    wrong gate / up / down offset inside an int4 record shows."""
    rng = np.random.default_rng(21)
    E, H, I, k, n = 5, 128, 64, 3, 6
    qgu, pgu, sgu, qd, pd, sd = _rand_int4_experts(rng, E, H, I, pow2_scales=True)
    # dequantised weights, independently of the oracle: code * scale of its group
    wgu_f = (qgu * np.repeat(oracle.bits_to_f32(sgu), 64, axis=-1)).astype(np.float32)
    wd_f = (qd * np.repeat(oracle.bits_to_f32(sd), 64, axis=-1)).astype(np.float32)
    wgu_b = bf16_round_bits(wgu_f)
    wd_b = bf16_round_bits(wd_f)
    assert np.array_equal(oracle.bits_to_f32(wgu_b), wgu_f)  # exact in bf16
    assert np.array_equal(oracle.bits_to_f32(wd_b), wd_f)
    x = rng.standard_normal((n, H)).astype(np.float32)
    ids = np.array([rng.permutation(E)[:k] for _ in range(n)], np.int32)
    w = rng.random((n, k)).astype(np.float32)
    out_q = oracle.experts_combine(x, ids, w, H, I, wgu_q=pgu, sgu_bits=sgu, wd_q=pd, sd_bits=sd)
    out_b = oracle.experts_combine(x, ids, w, H, I, wgu_bits=wgu_b, wd_bits=wd_b)
    assert np.array_equal(out_q, out_b)


def test_int4_experts_match_numpy_layer():
    """General scales: the int4 expert combine against the layer written with
    numpy matmuls over weights dequantised in numpy (code * scale per 64
    inputs of a row), scipy's expit for the sigmoid."""
    rng = np.random.default_rng(22)
    E, H, I, k, n = 4, 192, 128, 2, 5
    qgu, pgu, sgu, qd, pd, sd = _rand_int4_experts(rng, E, H, I, pow2_scales=False)
    Wgu = qgu * np.repeat(bits_f64(sgu), 64, axis=-1)
    Wd = qd * np.repeat(bits_f64(sd), 64, axis=-1)
    x = rng.standard_normal((n, H)).astype(np.float32)
    ids = np.array([rng.permutation(E)[:k] for _ in range(n)], np.int32)
    w = rng.random((n, k)).astype(np.float32)
    out = oracle.experts_combine(x, ids, w, H, I, wgu_q=pgu, sgu_bits=sgu, wd_q=pd, sd_bits=sd)
    xd = x.astype(np.float64)
    for t in range(n):
        ref = np.zeros(H)
        for j in range(k):
            e = ids[t, j]
            g = Wgu[e, :I] @ xd[t]
            u = Wgu[e, I:] @ xd[t]
            ref += float(w[t, j]) * (Wd[e] @ (g * scipy.special.expit(g) * u))
        assert np.allclose(out[t], ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())


def test_logits_f32_input_match_float64_matmul():
    """Router logits of fp32 input rows (the stack's normalised residual):
    float64 numpy matmul, a hand dot product, and the bf16-input entry point
    on rows that are exactly bf16."""
    rng = np.random.default_rng(23)
    T, H, E = 6, 160, 40
    x = rng.standard_normal((T, H)).astype(np.float32)  # not bf16-representable
    wr = bf16_round_bits((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    b = rng.standard_normal(E).astype(np.float32)
    L = oracle.router_logits(x, wr, b)
    ref = (x.astype(np.float64) @ bits_f64(wr).T + b.astype(np.float64)).astype(np.float32)
    assert np.max(np.abs(L.astype(np.float64) - ref)) <= 1e-6 * np.max(np.abs(ref))
    hand = sum(float(x[2, h]) * bits_f64(wr)[7, h] for h in range(H)) + float(b[7])
    assert abs(float(L[2, 7]) - hand) <= 1e-6 * max(1.0, abs(hand))
    xb = bf16_round_bits(x)
    assert np.array_equal(oracle.router_logits(oracle.bits_to_f32(xb), wr, b), oracle.router_logits(xb, wr, b))


# --------------------------------------------------------------------------
# Zero-centred RMSNorm
# --------------------------------------------------------------------------
def test_rmsnorm_closed_form():
    x = np.array([[3.0, 4.0], [-2.0, -2.0]], np.float32)
    out = oracle.rmsnorm(x, None, eps=0.0)
    assert np.allclose(out[0], np.array([3, 4]) / math.sqrt(12.5), rtol=1e-7)
    assert np.allclose(out[1], [-1.0, -1.0], rtol=1e-7)
    g = np.array([0.5, -0.5], np.float32)
    out_g = oracle.rmsnorm(x, g, eps=0.0)
    assert np.allclose(out_g[0], np.array([3 * 1.5, 4 * 0.5]) / math.sqrt(12.5), rtol=1e-7)
    eps = 1e-6
    out_e = oracle.rmsnorm(np.full((1, 8), 1e-3, np.float32), None, eps=eps)
    assert np.allclose(out_e, 1e-3 / math.sqrt(1e-6 + eps), rtol=1e-6)


# --------------------------------------------------------------------------
# Block deduplication
# --------------------------------------------------------------------------
@pytest.mark.parametrize("B", [1, 3, 4, 16])
def test_dedup_brute_force_sets(B):
    rng = np.random.default_rng(7 + B)
    L, Tt, k, E = 3, 17, 4, 40
    ids = np.stack([[rng.choice(E, size=k, replace=False) for _ in range(Tt)] for _ in range(L)]).astype(np.int32)
    mask, U, b2, b4 = oracle.dedup(ids, E, B, H=10, I=6)
    nb = (Tt + B - 1) // B
    assert mask.shape == (L, nb, 2)
    for l, b in itertools.product(range(L), range(nb)):
        ref = set(ids[l, b * B:(b + 1) * B].reshape(-1).tolist())
        got = {w * 32 + bit for w in range(2) for bit in range(32) if (int(mask[l, b, w]) >> bit) & 1}
        assert got == ref and U[l, b] == len(ref)
        assert U[l, b] <= min(k * min(B, Tt - b * B), E)
    P = 3 * 10 * 6
    assert np.array_equal(b2, U.sum(0).astype(np.int64) * P * 2 // 8)
    assert np.array_equal(b4, U.sum(0).astype(np.int64) * P * 4 // 8)


def test_dedup_rejects_bad_id():
    with pytest.raises(ValueError):
        oracle.dedup(np.array([[[0, 9]]], np.int32), 9, 1, 8, 8)


def test_combine_alone_linearity_and_hand_case():
    """Constant expert outputs v: out = v * sum(w) = v; a 2-route case by hand."""
    rng = np.random.default_rng(8)
    T, k, H = 3, 4, 8
    ids = np.array([[0, 1, 2, 3], [3, 2, 1, 0], [1, 3, 0, 2]], np.int32)
    _, _, perm, inv = oracle.permute(ids, 4)
    v = rng.standard_normal(H).astype(np.float32)
    y = np.tile(v, (T * k, 1))
    w = np.full((T, k), 0.25, np.float32)
    out = oracle.combine(y, inv, w)
    assert np.allclose(out, np.tile(v, (T, 1)), rtol=1e-6)
    y2 = np.zeros((2, 2), np.float32)
    y2[0] = [1.0, 2.0]
    y2[1] = [10.0, 20.0]
    out2 = oracle.combine(y2, np.array([1, 0], np.int32), np.array([[0.75, 0.25]], np.float32),
                          residual=np.array([[100.0, 200.0]], np.float32))
    assert np.allclose(out2[0], [100 + 0.75 * 10 + 0.25 * 1, 200 + 0.75 * 20 + 0.25 * 2])


def test_round_bf16_hand_cases_and_library():
    import torch
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 3.0e38, 0.0, -0.0, 1.0 + 2**-8 + 2**-20],
                    np.float32)
    got = oracle.round_bf16_bits(vals)
    assert list(got[:7]) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F62, 0x0000, 0x8000]
    assert got[7] == 0x3F81  # just above the tie rounds up
    rng = np.random.default_rng(12)
    r = (rng.standard_normal(4096) * 10.0 ** rng.integers(-6, 6, 4096)).astype(np.float32)
    ref = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16_bits(r), ref)


def test_recall_brute_force_and_extremes():
    rng = np.random.default_rng(13)
    T, k, E = 50, 10, 64
    a = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    b = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    hits = oracle.recall_hits(a, b)
    assert list(hits) == [len(set(a[t]) & set(b[t])) for t in range(T)]
    assert np.all(oracle.recall_hits(a, a) == k)
    assert np.all(oracle.recall_hits(a, a[:, ::-1]) == k)  # order does not matter
    assert np.all(oracle.recall_hits(a % 32, a % 32 + 32) == 0)
