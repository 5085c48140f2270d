"""Pins of the oracle's route-sidecar forward pass (no GPU).

AFN-021 "Replay decode as prefill: a training flywheel for predictive MoE
I/O", section "What feature should the sidecar see?": feature -> shared
low-rank trunk -> plus the target layer's embedding -> shared expert-head
embeddings -> one score per expert -> ranked candidates.  Pinned by a
hand-worked case, a rank-one construction whose ranking is known in closed
form for every layer, the special case without layer embeddings (two plain
matrix products), exact scale covariance, and the tie rule.
"""
import numpy as np

import oracle


def bits(a):
    """float array of bf16-exact values -> bf16 bit patterns."""
    f = np.ascontiguousarray(a, np.float32)
    b = f.view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def test_hand_worked_case():
    # f = (1, 2); trunk rows (1, 0), (1, 1): z = (1, 3)
    # layer 0: z0 = (1, 3); layer 1: z1 = z + (-2, 1) = (-1, 4)
    # head rows (1, 0), (0, 1), (-1, 1):
    #   layer 0 scores (1, 3, 2) -> experts 1, 2 with 3, 2
    #   layer 1 scores (-1, 4, 5) -> experts 2, 1 with 5, 4
    feat = bits([[1, 2]])
    trunk = bits([[1, 0], [1, 1]])
    emb = bits([[0, 0], [-2, 1]])
    head = bits([[1, 0], [0, 1], [-1, 1]])
    cand, cs, sc = oracle.sidecar(feat, trunk, emb, head, N=2, want_scores=True)
    assert cand.tolist() == [[[1, 2], [2, 1]]]
    assert cs.tolist() == [[[3.0, 2.0], [5.0, 4.0]]]
    assert sc.tolist() == [[[1.0, 3.0, 2.0], [-1.0, 4.0, 5.0]]]


def test_rank_one_closed_form():
    """Trunk row 0 picks feature 0 (+1 or -1), the layer embedding adds +4 on
    even and -4 on odd layers, head row e is ((e+1)/64, 0, ...): score
    s_e = (e+1)/64 * z_l[0], so even layers rank the highest IDs first and
    odd layers the lowest, with exact scores."""
    T, F, r, E, L, N = 3, 16, 8, 48, 6, 5
    feat = np.zeros((T, F), np.float32)
    feat[:, 0] = [1, -1, 1]
    feat[:, 1:] = 0.5  # ignored by the trunk
    trunk = np.zeros((r, F), np.float32)
    trunk[0, 0] = 1
    trunk[3, 5] = 1    # a trunk row the head ignores
    emb = np.zeros((L, r), np.float32)
    emb[:, 0] = [4 if l % 2 == 0 else -4 for l in range(L)]
    emb[:, 3] = 2
    head = np.zeros((E, r), np.float32)
    head[:, 0] = (np.arange(E) + 1) / 64
    cand, cs, _ = oracle.sidecar(bits(feat), bits(trunk), bits(emb), bits(head), N)
    for t in range(T):
        for l in range(L):
            zl0 = feat[t, 0] + emb[l, 0]
            want = list(range(E - 1, E - 1 - N, -1)) if zl0 > 0 else list(range(N))
            assert cand[t, l].tolist() == want, (t, l)
            np.testing.assert_array_equal(cs[t, l], [(e + 1) / 64 * zl0 for e in want])


def test_without_layer_embeddings_it_is_two_matrix_products():
    rng = np.random.default_rng(3)
    T, F, r, E, N = 4, 32, 8, 20, 20
    q = lambda *s: np.round(rng.normal(size=s) * 8) / 8  # small dyadic values, exact in bf16
    feat, trunk, head = q(T, F), q(r, F), q(E, r)
    emb = np.zeros((1, r))
    cand, cs, sc = oracle.sidecar(bits(feat), bits(trunk), bits(emb), bits(head), N, want_scores=True)
    want = (head @ (trunk @ feat.T)).T  # [T, E]
    np.testing.assert_allclose(sc[:, 0, :], want, rtol=0, atol=1e-9)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-want[t, e], e))
        assert cand[t, 0].tolist() == order


def test_scale_covariance_and_ties():
    rng = np.random.default_rng(4)
    T, F, r, E, L, N = 2, 16, 8, 12, 3, 6
    q = lambda *s: np.round(rng.normal(size=s) * 4) / 4
    feat, trunk, emb, head = q(T, F), q(r, F), q(L, r), q(E, r)
    c1, s1, _ = oracle.sidecar(bits(feat), bits(trunk), bits(emb), bits(head), N)
    c2, s2, _ = oracle.sidecar(bits(feat), bits(2 * trunk), bits(2 * emb), bits(head), N)
    assert np.array_equal(c1, c2)
    np.testing.assert_array_equal(s2, 2 * s1)
    # identical head rows score equally: the lower ID ranks first
    head2 = head.copy()
    head2[7] = head2[2]
    c3, s3, sc3 = oracle.sidecar(bits(feat), bits(trunk), bits(emb), bits(head2), E, want_scores=True)
    for t in range(T):
        for l in range(L):
            row = c3[t, l].tolist()
            assert sc3[t, l, 2] == sc3[t, l, 7] and row.index(2) < row.index(7)
