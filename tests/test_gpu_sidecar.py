"""GPU parity of the route-sidecar forward pass (moe_sidecar_prepare,
moe_sidecar_forward) against the oracle.

Scores are fp32 sums of bf16 products on the GPU and fp64 in the oracle; the
candidates are a ranking decided by those scores.  So: every candidate's
score must match the oracle's score of the same expert within the fp32
rounding bound, the n-th candidate's oracle score must be within that bound
of the oracle's n-th largest score (a valid ranking), and wherever the
oracle's n-th and (n+1)-th scores are further apart than twice the bound the
IDs must be equal.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from sparse_moe_routed_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def bf16_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("T,F,r,E,L,N", [(16, 2560, 256, 512, 48, 16), (1, 2560, 256, 512, 48, 10),
                                         (37, 1280, 64, 100, 5, 32), (3, 256, 24, 40, 70, 7),
                                         (64, 512, 512, 1024, 3, 32)])
def test_sidecar_matches_oracle(T, F, r, E, L, N):
    w = wl.sidecar_weights(F, r, E, L, DEV)
    feat = torch.randn((T, F), generator=torch.Generator(device=DEV).manual_seed(T * 7 + F), device=DEV)
    feat = feat.to(torch.bfloat16)
    hb = torch.empty((L, E), dtype=torch.float32, device=DEV)
    z = torch.empty((T, r), dtype=torch.float32, device=DEV)
    cand = torch.full((T, L, N), -1, dtype=torch.int32, device=DEV)
    cs = torch.empty((T, L, N), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_sidecar_prepare(w["w_head"], w["layer_emb"], hb)
    _lib.moe_sidecar_forward(feat, w["w_trunk"], w["w_head"], hb, N, z, cand, cs, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rc, rs, sc = oracle.sidecar(bf16_bits(feat), bf16_bits(w["w_trunk"]), bf16_bits(w["layer_emb"]),
                                bf16_bits(w["w_head"]), N, want_scores=True)
    got_c, got_s = cand.cpu().numpy(), cs.cpu().numpy()
    # fp32 bound: trunk sums F products, head sums r products; scores are O(1)
    tol = 4e-4
    assert got_c.min() >= 0 and got_c.max() < E
    for t in range(T):
        for l in range(L):
            s = sc[t, l]
            ref_sorted = np.sort(s)[::-1]
            ids = got_c[t, l]
            assert len(set(ids.tolist())) == N
            np.testing.assert_allclose(got_s[t, l], s[ids], rtol=0, atol=tol)
            np.testing.assert_allclose(s[ids], ref_sorted[:N], rtol=0, atol=2 * tol)
            gaps = ref_sorted[:N] - np.append(ref_sorted[1:N + 1], -np.inf)[:N]
            for n in range(N):
                left = n == 0 or ref_sorted[n - 1] - ref_sorted[n] > 2 * tol
                if left and gaps[n] > 2 * tol:
                    assert ids[n] == rc[t, l, n], (t, l, n)


def test_layer_embedding_changes_the_ranking():
    """The layers' candidate lists differ (the embedding is not dropped)."""
    T, F, r, E, L, N = 4, 2560, 256, 512, 48, 16
    w = wl.sidecar_weights(F, r, E, L, DEV)
    feat = wl.token_batch(wl.DECODE, DEV, index=3, T=T)
    hb = torch.empty((L, E), dtype=torch.float32, device=DEV)
    z = torch.empty((T, r), dtype=torch.float32, device=DEV)
    cand = torch.empty((T, L, N), dtype=torch.int32, device=DEV)
    cs = torch.empty((T, L, N), dtype=torch.float32, device=DEV)
    st = torch.zeros((1,), dtype=torch.int32, device=DEV)
    _lib.moe_sidecar_prepare(w["w_head"], w["layer_emb"], hb)
    _lib.moe_sidecar_forward(feat, w["w_trunk"], w["w_head"], hb, N, z, cand, cs, st)
    torch.cuda.synchronize()
    c = cand.cpu().numpy()
    assert len({tuple(c[0, l]) for l in range(L)}) == L
    assert np.all(np.diff(cs.cpu().numpy(), axis=-1) <= 0)  # ranked, best first
