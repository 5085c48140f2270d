"""CPU oracle for the routed-expert MoE layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference leg may import this package.  The product path (the CUDA library and
its binding) never touches it.  The arithmetic lives in ``moe_oracle.c``
(plain C, fp64); this module only marshals numpy arrays into it.

Functions and the page passages they follow (Hebrus "Agent Field Notes"):

  route(...)            AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus", section
                        "Phase 1: separate math from acceleration" (float32 router
                        softmax and normalized top-10); AFN-021 "Replay decode as
                        prefill", section "The key equivalence -- and where it
                        breaks" (IDs in rank order are the label).
  permute(...)          AFN-019 "Hide SSD misses before the router knows they exist",
                        section "Why overlap alone cannot defeat the byte roofline"
                        (grouping token rows by expert).
  experts_combine(...)  AFN-019, section "Why overlap alone..." (gate + up + down per
                        expert) and section "Hypothesis H4" (SwiGLU order; weighted
                        sum in deterministic route-rank order).
  dedup(...)            AFN-019, sections "Why overlap alone..." (deduplication of
                        repeated routes across a verifier block) and "Hypothesis H7"
                        (48 * U_B * record bytes).
  dequant_int4(...)     AFN-001, section "Phase 2" (affine4, group 64), in the
                        symmetric-scale reading.
  combine(...)          AFN-019, section "Hypothesis H4" (weighted sum in route-rank order).
  rmsnorm(...)          AFN-001, section "Phase 1" (zero-centred RMS normalisation).
  recall_hits(...)      AFN-019, section "Hypothesis H2" (predicted vs exact top-k).
  round_bf16_bits(...)  bf16 rounding of the normalised stack input (reading: the layer's
                        input is bf16 in every workload, and in the stack that input is
                        RMSNorm(x_l); the residual stream stays fp32).

Parity pins: every function above is pinned in tests/test_oracle_pins.py
against closed forms, brute force on tiny inputs, special cases reducing to
textbook routines, and the figures the pages print.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = C.CDLL(path)
        p = C.c_void_p
        i = C.c_int
        lib.oracle_threads.argtypes = [i]
        lib.oracle_threads.restype = i
        lib.oracle_router_logits.argtypes = [p, p, p, i, i, i, p]
        lib.oracle_router_logits_f32.argtypes = [p, p, p, i, i, i, p]
        lib.oracle_topk.argtypes = [p, i, i, i, p, p, p]
        lib.oracle_permute.argtypes = [p, i, i, i, p, p, p, p]
        lib.oracle_permute.restype = i
        lib.oracle_experts_combine.argtypes = [p, i, i, i, i, p, p, p, p, p, p, p, p, p]
        lib.oracle_expert_rows.argtypes = [p, i, i, i, p, p, i, p]
        lib.oracle_dequant_int4.argtypes = [p, p, i, i, p]
        lib.oracle_combine.argtypes = [p, p, p, i, i, i, p, p]
        lib.oracle_rmsnorm.argtypes = [p, p, i, i, C.c_double, p]
        lib.oracle_round_bf16.argtypes = [p, C.c_size_t, p]
        lib.oracle_recall.argtypes = [p, p, i, i, p]
        lib.oracle_dedup.argtypes = [p, i, i, i, i, i, i, i, p, p, p, p]
        lib.oracle_dedup.restype = i
        lib.oracle_cache_plan.argtypes = [i, C.c_float, p, i, p, p, i, p, p, p, p, p, p]
        lib.oracle_cache_plan.restype = i
        lib.oracle_sidecar.argtypes = [p, p, p, p, i, i, i, i, i, i, p, p, p]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def threads(n: int = 0) -> int:
    """Set (n > 0) and return the OpenMP thread count the oracle uses."""
    return _load().oracle_threads(n)


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (or pass through uint16)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def router_logits(x_bits, wr_bits, bias=None):
    """L[t,e] = fp32(sum_h x*Wr (fp64) + b[e]) for bf16 x (uint16 bits) or fp32 x."""
    wr = _c(wr_bits, np.uint16)
    E, H = wr.shape
    if x_bits.dtype == np.uint16:
        x = _c(x_bits, np.uint16)
        fn = _load().oracle_router_logits
    else:
        x = _c(x_bits, np.float32)
        fn = _load().oracle_router_logits_f32
    T = x.shape[0]
    b = _c(bias, np.float32)
    out = np.empty((T, E), np.float32)
    fn(_ptr(x), _ptr(wr), _ptr(b), T, H, E, _ptr(out))
    return out


def topk(logits, k):
    """(ids [T,k] int32 rank order, w [T,k] fp32, gap [T] fp32)."""
    L = _c(logits, np.float32)
    T, E = L.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    gap = np.empty((T,), np.float32)
    _load().oracle_topk(_ptr(L), T, E, k, _ptr(ids), _ptr(w), _ptr(gap))
    return ids, w, gap


def route(x_bits, wr_bits, bias, k):
    L = router_logits(x_bits, wr_bits, bias)
    ids, w, gap = topk(L, k)
    return ids, w, gap, L


def permute(ids, E):
    """Stable counting sort of flat routes by expert: counts, offsets, perm, inv."""
    a = _c(ids, np.int32)
    T, k = a.shape
    R = T * k
    counts = np.empty((E,), np.int32)
    offsets = np.empty((E + 1,), np.int32)
    perm = np.empty((R,), np.int32)
    inv = np.empty((R,), np.int32)
    rc = _load().oracle_permute(_ptr(a), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv))
    if rc != 0:
        raise ValueError("expert id out of range")
    return counts, offsets, perm, inv


def experts_combine(xin, ids, w, H, I, wgu_bits=None, wd_bits=None,
                    wgu_q=None, sgu_bits=None, wd_q=None, sd_bits=None):
    """out[t] = sum_j w[t,j] * SwiGLU-expert_{ids[t,j]}(xin[t]) in rank order j."""
    x = _c(xin, np.float32)
    n = x.shape[0]
    idc = _c(ids, np.int32)
    k = idc.shape[1]
    wc = _c(w, np.float32)
    out = np.empty((n, H), np.float32)
    _load().oracle_experts_combine(
        _ptr(x), n, H, I, k, _ptr(idc), _ptr(wc),
        _ptr(_c(wgu_bits, np.uint16)), _ptr(_c(wd_bits, np.uint16)),
        _ptr(_c(wgu_q, np.uint8)), _ptr(_c(sgu_bits, np.uint16)),
        _ptr(_c(wd_q, np.uint8)), _ptr(_c(sd_bits, np.uint16)), _ptr(out))
    return out


def expert_rows(xin, wgu_bits, wd_bits, e, H, I):
    """One expert (no routing) applied to each fp32 row of xin."""
    x = _c(xin, np.float32)
    n = x.shape[0]
    y = np.empty((n, H), np.float32)
    _load().oracle_expert_rows(_ptr(x), n, H, I, _ptr(_c(wgu_bits, np.uint16)),
                               _ptr(_c(wd_bits, np.uint16)), e, _ptr(y))
    return y


def combine(y, inv, w, residual=None):
    """out[t] = sum_j w[t,j] * y[inv[t*k+j]] (+ residual) in rank order j."""
    yc = _c(y, np.float32)
    H = yc.shape[1]
    wc = _c(w, np.float32)
    T, k = wc.shape
    ic = _c(inv, np.int32)
    out = np.empty((T, H), np.float32)
    _load().oracle_combine(_ptr(yc), _ptr(ic), _ptr(wc), T, k, H, _ptr(_c(residual, np.float32)), _ptr(out))
    return out


def dequant_int4(q, s_bits):
    q = _c(q, np.uint8)
    s = _c(s_bits, np.uint16)
    rows = int(np.prod(q.shape[:-1]))
    K = q.shape[-1] * 2
    w = np.empty(q.shape[:-1] + (K,), np.float32)
    _load().oracle_dequant_int4(_ptr(q), _ptr(s), rows, K, _ptr(w))
    return w


def rmsnorm(x, gamma=None, eps=1e-6):
    xc = _c(x, np.float32)
    T, H = xc.shape
    out = np.empty_like(xc)
    _load().oracle_rmsnorm(_ptr(xc), _ptr(_c(gamma, np.float32)), T, H, float(eps), _ptr(out))
    return out


def recall_hits(pred, ref):
    """hits[t] = |set(pred[t]) & set(ref[t])| for [T,k] routes."""
    pc = _c(pred, np.int32)
    rc = _c(ref, np.int32)
    T, k = rc.shape
    hits = np.empty((T,), np.int32)
    _load().oracle_recall(_ptr(pc), _ptr(rc), T, k, _ptr(hits))
    return hits


def round_bf16_bits(x):
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    xc = _c(x, np.float32)
    out = np.empty(xc.shape, np.uint16)
    _load().oracle_round_bf16(_ptr(xc), xc.size, _ptr(out))
    return out


def dedup(ids, E, block, H, I):
    """ids [L,Ttot,k] -> (mask [L,nb,ceil(E/32)] uint32, U [L,nb], bytes2 [nb], bytes4 [nb])."""
    a = _c(ids, np.int32)
    L, Tt, k = a.shape
    nb = (Tt + block - 1) // block
    W = (E + 31) // 32
    mask = np.empty((L, nb, W), np.uint32)
    U = np.empty((L, nb), np.int32)
    b2 = np.empty((nb,), np.int64)
    b4 = np.empty((nb,), np.int64)
    rc = _load().oracle_dedup(_ptr(a), L, Tt, k, E, block, H, I, _ptr(mask), _ptr(U), _ptr(b2), _ptr(b4))
    if rc != 0:
        raise ValueError("expert id out of range")
    return mask, U, b2, b4


POLICIES = {"fifo": 0, "lru": 1, "score": 2}


class CachePlan:
    """State of one expert cache (E experts, S slots) stepped by the oracle."""

    def __init__(self, E, S, policy="fifo", decay=0.9):
        self.E, self.S = E, S
        self.policy = POLICIES[policy]
        self.decay = np.float32(decay)
        self.slot_of = np.full(E, -1, np.int32)
        self.expert_of = np.full(S, -1, np.int32)
        self.hand = np.zeros(2, np.int32)
        self.score = np.zeros(E, np.float32)
        self.last_use = np.full(S, -1, np.int32)
        self.stats = np.zeros(4, np.int32)

    def step(self, counts):
        """One call; returns (full, miss_list, miss_slot)."""
        c = _c(counts, np.int32)
        ml = np.zeros(max(self.S, 1), np.int32)
        ms = np.zeros(max(self.S, 1), np.int32)
        full = _load().oracle_cache_plan(self.policy, float(self.decay), _ptr(c), self.E, _ptr(self.slot_of),
                                         _ptr(self.expert_of), self.S, _ptr(self.hand), _ptr(self.score),
                                         _ptr(self.last_use), _ptr(ml), _ptr(ms), _ptr(self.stats))
        n = int(self.stats[1])
        return bool(full), ml[:n].copy(), ms[:n].copy()


def sidecar(feat_bits, trunk_bits, emb_bits, head_bits, N, want_scores=False):
    """Route sidecar: (cand [T,L,N] int32, cand_score [T,L,N] f32, scores
    [T,L,E] f64 or None) for bf16 bit arrays feat [T,F], trunk [r,F],
    emb [L,r], head [E,r]."""
    f = _c(feat_bits, np.uint16)
    wt = _c(trunk_bits, np.uint16)
    em = _c(emb_bits, np.uint16)
    wh = _c(head_bits, np.uint16)
    T, F = f.shape
    r = wt.shape[0]
    L = em.shape[0]
    E = wh.shape[0]
    cand = np.empty((T, L, N), np.int32)
    cs = np.empty((T, L, N), np.float32)
    sc = np.empty((T, L, E), np.float64) if want_scores else None
    _load().oracle_sidecar(_ptr(f), _ptr(wt), _ptr(em), _ptr(wh), T, F, r, E, L, N, _ptr(cand), _ptr(cs),
                           _ptr(sc) if sc is not None else None)
    return cand, cs, sc


def moe_layer(x_bits, wr_bits, bias, wgu_bits, wd_bits, k, I):
    """Full layer for bf16 x: route, then experts + rank-order combine."""
    ids, w, gap, L = route(x_bits, wr_bits, bias, k)
    H = wr_bits.shape[1]
    xin = _bits_to_f32(x_bits)
    out = experts_combine(xin, ids, w, H, I, wgu_bits=wgu_bits, wd_bits=wd_bits)
    return out, ids, w, gap


def _bits_to_f32(bits):
    b = np.ascontiguousarray(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


bits_to_f32 = _bits_to_f32
