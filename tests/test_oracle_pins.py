"""Pins for the fp64 oracle: hand-worked examples, closed forms, library
special cases (dense masked attention, scaled_dot_product_attention, torch
autograd), finite differences and invariants.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rand_graph(rng, N, p, self_loops=True, dups=False):
    """Small random destination-sorted CSR (sources ascending)."""
    rows = []
    for i in range(N):
        src = [j for j in range(N) if (rng.random() < p) or (self_loops and j == i)]
        if dups and src and rng.random() < 0.3:
            src = sorted(src + [src[rng.integers(len(src))]])
        rows.append(src)
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    return indptr, indices


def dense_mask(indptr, indices, N):
    m = torch.zeros(N, N, dtype=torch.bool)
    for i in range(N):
        for e in range(indptr[i], indptr[i + 1]):
            m[i, indices[e]] = True
    return m


def dense_gt(Q, K, V, mask):
    """Brute-force dense masked attention in torch fp64: [N,H,D] tensors."""
    N, H, D = Q.shape
    s = torch.einsum("ihd,jhd->hij", Q, K) / math.sqrt(D)
    s = s.masked_fill(~mask[None], float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                      # [H, N]
    p = torch.exp(s - lse[..., None]).nan_to_num(0.0)      # empty rows -> 0
    out = torch.einsum("hij,jhd->ihd", p, V)
    return out, lse.T


def dense_gatv2(X, Wl, Wr, a, mask, slope=0.2):
    N = X.shape[0]
    H, D = a.shape
    FL = (X @ Wl).reshape(N, H, D)
    FR = (X @ Wr).reshape(N, H, D)
    z = FL[:, None] + FR[None, :]                          # [i, j, H, D]
    e = (torch.nn.functional.leaky_relu(z, slope) * a).sum(-1).permute(2, 0, 1)  # [H, i, j]
    e = e.masked_fill(~mask[None], float("-inf"))
    lse = torch.logsumexp(e, dim=-1)
    p = torch.exp(e - lse[..., None]).nan_to_num(0.0)
    out = torch.einsum("hij,jhd->ihd", p, FR)
    return out, lse.T


# ------------------------------------------------------------ hand examples

def test_gt_hand_example():
    g = load("gt_hand.json")
    q = np.array(g["q"]).reshape(2, 1, 1)
    k = np.array(g["k"]).reshape(2, 1, 1)
    v = np.array(g["v"]).reshape(2, 1, 1)
    out, lse = oracle.gt_fwd(g["indptr"], g["indices"], q, k, v)
    assert out[:, 0, 0] == pytest.approx(g["expected_out"], abs=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(4.0), abs=1e-14)
    assert lse[1, 0] == pytest.approx(2.0 * math.log(3.0), abs=1e-14)


def test_gatv2_hand_example():
    g = load("gatv2_hand.json")
    X = np.array(g["x"]).reshape(3, 1)
    FL, FR, out, lse = oracle.gatv2_fwd(g["indptr"], g["indices"], X, g["W_l"], g["W_r"], g["a"],
                                        g["slope"])
    e1, e2 = g["expected_scores_row0"]
    w1 = math.exp(e1) / (math.exp(e1) + math.exp(e2))
    w2 = 1.0 - w1
    assert out[0, 0, 0] == pytest.approx(-2.0 * w1 + 1.0 * w2, abs=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(-0.2) + math.exp(2.0)), abs=1e-14)
    assert np.all(out[1:] == 0.0)
    assert np.all(np.isneginf(lse[1:]))


def test_five_node_closed_forms():
    """Empty row, degree-1 row, zero query (uniform weights), identical keys."""
    rng = np.random.default_rng(11)
    H, D = 2, 4
    indptr = np.array([0, 3, 3, 4, 6, 8], np.int32)
    indices = np.array([1, 2, 3, 4, 0, 3, 2, 4], np.int32)
    Q = rng.standard_normal((5, H, D)); K = rng.standard_normal((5, H, D))
    V = rng.standard_normal((5, H, D))
    Q[0] = 0.0                      # row 0: uniform weights over {1,2,3}
    K[3] = K[0]                     # row 3: identical keys for {0,3}
    out, lse = oracle.gt_fwd(indptr, indices, Q, K, V)
    np.testing.assert_allclose(out[0], V[[1, 2, 3]].mean(0), atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(3.0), atol=1e-14)
    assert np.all(out[1] == 0.0) and np.all(np.isneginf(lse[1]))
    np.testing.assert_allclose(out[2], V[4], atol=1e-14)
    np.testing.assert_allclose(lse[2], (Q[2] * K[4]).sum(-1) / math.sqrt(D), atol=1e-14)
    np.testing.assert_allclose(out[3], V[[0, 3]].mean(0), atol=1e-14)
    np.testing.assert_allclose(lse[3], (Q[3] * K[0]).sum(-1) / math.sqrt(D) + math.log(2.0),
                               atol=1e-13)
    m = dense_mask(indptr, indices, 5)
    o_ref, l_ref = dense_gt(*(torch.from_numpy(x) for x in (Q, K, V)), m)
    np.testing.assert_allclose(out[4], o_ref[4].numpy(), atol=1e-13)


def test_gatv2_zero_attention_vector_gives_mean():
    rng = np.random.default_rng(5)
    N, F, H, D = 20, 6, 2, 3
    indptr, indices = rand_graph(rng, N, 0.3)
    X = rng.standard_normal((N, F)); Wl = rng.standard_normal((F, H * D))
    Wr = rng.standard_normal((F, H * D)); a = np.zeros((H, D))
    FL, FR, out, lse = oracle.gatv2_fwd(indptr, indices, X, Wl, Wr, a)
    for i in range(N):
        nb = indices[indptr[i]:indptr[i + 1]]
        np.testing.assert_allclose(out[i], FR[nb].mean(0), atol=1e-13)
        np.testing.assert_allclose(lse[i], math.log(len(nb)), atol=1e-13)


# ------------------------------------------------------ library special cases

def test_gt_complete_graph_equals_sdpa():
    rng = np.random.default_rng(1)
    N, H, D = 12, 3, 8
    indptr = np.arange(0, N * N + 1, N, dtype=np.int32)
    indices = np.tile(np.arange(N, dtype=np.int32), N)
    Q, K, V = (rng.standard_normal((N, H, D)) for _ in range(3))
    out, _ = oracle.gt_fwd(indptr, indices, Q, K, V)
    t = lambda x: torch.from_numpy(x).permute(1, 0, 2)[None]  # [1, H, N, D]
    ref = torch.nn.functional.scaled_dot_product_attention(t(Q), t(K), t(V))
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), atol=1e-13)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gt_matches_dense_masked(seed):
    rng = np.random.default_rng(100 + seed)
    N, H, D = 40, 2, 8
    indptr, indices = rand_graph(rng, N, 0.15, self_loops=(seed != 2))
    Q, K, V = (rng.standard_normal((N, H, D)) for _ in range(3))
    out, lse = oracle.gt_fwd(indptr, indices, Q, K, V)
    o_ref, l_ref = dense_gt(*(torch.from_numpy(x) for x in (Q, K, V)),
                            dense_mask(indptr, indices, N))
    np.testing.assert_allclose(out, o_ref.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, l_ref.numpy(), atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_gatv2_matches_dense_masked(seed):
    rng = np.random.default_rng(200 + seed)
    N, F, H, D = 30, 5, 2, 4
    indptr, indices = rand_graph(rng, N, 0.2, self_loops=(seed == 0))
    X = rng.standard_normal((N, F)); Wl = rng.standard_normal((F, H * D))
    Wr = rng.standard_normal((F, H * D)); a = rng.standard_normal((H, D))
    FL, FR, out, lse = oracle.gatv2_fwd(indptr, indices, X, Wl, Wr, a, 0.2)
    t = torch.from_numpy
    o_ref, l_ref = dense_gatv2(t(X), t(Wl), t(Wr), t(a), dense_mask(indptr, indices, N))
    np.testing.assert_allclose(FL.reshape(N, -1), X @ Wl, atol=1e-12)
    np.testing.assert_allclose(out, o_ref.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, l_ref.numpy(), atol=1e-12)


def test_gt_backward_matches_autograd():
    rng = np.random.default_rng(7)
    N, H, D = 36, 2, 8
    indptr, indices = rand_graph(rng, N, 0.2)
    indptr2, indices2 = indptr.copy(), indices.copy()
    indptr2[:] = indptr;
    Q, K, V, dO = (rng.standard_normal((N, H, D)) for _ in range(4))
    # an empty row must contribute nothing
    row = 5
    b, e = indptr[row], indptr[row + 1]
    indices2 = np.concatenate([indices[:b], indices[e:]]).astype(np.int32)
    indptr2[row + 1:] -= (e - b)
    dQ, dK, dV = oracle.gt_bwd(indptr2, indices2, Q, K, V, dO)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (Q, K, V))
    out, _ = dense_gt(tq, tk, tv, dense_mask(indptr2, indices2, N))
    (out * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-12)
    assert np.all(dQ[row] == 0.0)


def test_gatv2_backward_matches_autograd():
    rng = np.random.default_rng(8)
    N, F, H, D = 28, 6, 2, 4
    indptr, indices = rand_graph(rng, N, 0.25)
    X = rng.standard_normal((N, F)); Wl = rng.standard_normal((F, H * D)) * 0.5
    Wr = rng.standard_normal((F, H * D)) * 0.5; a = rng.standard_normal((H, D))
    dO = rng.standard_normal((N, H, D))
    g = oracle.gatv2_bwd(indptr, indices, X, Wl, Wr, a, dO, 0.2)
    tX, tWl, tWr, ta = (torch.from_numpy(x).requires_grad_() for x in (X, Wl, Wr, a))
    out, _ = dense_gatv2(tX, tWl, tWr, ta, dense_mask(indptr, indices, N))
    (out * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(g["dX"], tX.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dW_l"], tWl.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["dW_r"], tWr.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(g["da"], ta.grad.numpy(), atol=1e-11)


def straight_through(Y, store):
    """Y rounded to the storage dtype in value, the identity in gradient."""
    r = Y.detach().float()
    r = r.to(torch.bfloat16).double() if store == "bf16" else r.double()
    return Y + (r - Y).detach()


@pytest.mark.parametrize("store", ["bf16", "f32"])
def test_gatv2_backward_with_stored_projections_matches_straight_through_autograd(store):
    """store='bf16'/'f32' in the backward: the edge stage runs on the rounded
    projections (branches decided on them) and the rounding passes gradients
    unchanged.  torch autograd of the dense form with a straight-through
    rounding step must agree; the projections are made large enough that the
    rounding moves the gradients far beyond the tolerance (a backward that
    ignored the storage mode fails)."""
    rng = np.random.default_rng(24 if store == "bf16" else 25)
    N, F, H, D = 27, 6, 2, 4
    indptr, indices = rand_graph(rng, N, 0.3)
    X = rng.standard_normal((N, F)) * 3.0
    Wl = rng.standard_normal((F, H * D)); Wr = rng.standard_normal((F, H * D))
    a = rng.standard_normal((H, D)); dO = rng.standard_normal((N, H, D))
    g = oracle.gatv2_bwd(indptr, indices, X, Wl, Wr, a, dO, 0.2, store=store)
    g64 = oracle.gatv2_bwd(indptr, indices, X, Wl, Wr, a, dO, 0.2)
    tX, tWl, tWr, ta = (torch.from_numpy(x).requires_grad_() for x in (X, Wl, Wr, a))
    FL = straight_through(tX @ tWl, store).reshape(N, H, D)
    FR = straight_through(tX @ tWr, store).reshape(N, H, D)
    mask = dense_mask(indptr, indices, N)
    z = FL[:, None] + FR[None, :]
    e = (torch.nn.functional.leaky_relu(z, 0.2) * ta).sum(-1).permute(2, 0, 1)
    e = e.masked_fill(~mask[None], float("-inf"))
    p = torch.exp(e - torch.logsumexp(e, dim=-1)[..., None]).nan_to_num(0.0)
    out = torch.einsum("hij,jhd->ihd", p, FR)
    (out * torch.from_numpy(dO)).sum().backward()
    for name, t in (("dX", tX), ("dW_l", tWl), ("dW_r", tWr), ("da", ta)):
        ref = t.grad.numpy()
        np.testing.assert_allclose(g[name], ref, atol=1e-10 * max(1.0, np.abs(ref).max()))
        # the rounding matters: fp64 projections give gradients outside the check
        # (relative ~1e-2 for bf16, ~1e-7 for fp32, both far above 1e-10)
        assert np.abs(g64[name] - ref).max() > (1e-4 if store == "bf16" else 1e-8) * np.abs(ref).max()


# -------------------------------------------------------- finite differences

def test_gt_backward_finite_differences():
    rng = np.random.default_rng(9)
    N, H, D = 15, 2, 4
    indptr, indices = rand_graph(rng, N, 0.3, dups=True)
    Q, K, V, dO = (rng.standard_normal((N, H, D)) for _ in range(4))
    grads = dict(zip("QKV", oracle.gt_bwd(indptr, indices, Q, K, V, dO)))
    eps = 1e-6
    for name in "QKV":
        for _ in range(6):
            idx = tuple(rng.integers(s) for s in Q.shape)
            args = {"Q": Q.copy(), "K": K.copy(), "V": V.copy()}
            args[name][idx] += eps
            lp = (oracle.gt_fwd(indptr, indices, args["Q"], args["K"], args["V"])[0] * dO).sum()
            args[name][idx] -= 2 * eps
            lm = (oracle.gt_fwd(indptr, indices, args["Q"], args["K"], args["V"])[0] * dO).sum()
            fd = (lp - lm) / (2 * eps)
            assert fd == pytest.approx(grads[name][idx], rel=1e-6, abs=1e-8)


def test_gatv2_backward_finite_differences():
    rng = np.random.default_rng(10)
    N, F, H, D = 12, 4, 2, 3
    indptr, indices = rand_graph(rng, N, 0.35)
    args = {"X": rng.standard_normal((N, F)), "Wl": rng.standard_normal((F, H * D)),
            "Wr": rng.standard_normal((F, H * D)), "a": rng.standard_normal((H, D))}
    dO = rng.standard_normal((N, H, D))
    g = oracle.gatv2_bwd(indptr, indices, args["X"], args["Wl"], args["Wr"], args["a"], dO)
    names = {"X": "dX", "Wl": "dW_l", "Wr": "dW_r", "a": "da"}
    eps = 1e-6

    def loss(a_):
        return (oracle.gatv2_fwd(indptr, indices, a_["X"], a_["Wl"], a_["Wr"], a_["a"])[2] * dO).sum()

    for name, gname in names.items():
        for _ in range(5):
            idx = tuple(rng.integers(s) for s in args[name].shape)
            ap = {k: v.copy() for k, v in args.items()}
            ap[name][idx] += eps
            am = {k: v.copy() for k, v in args.items()}
            am[name][idx] -= eps
            fd = (loss(ap) - loss(am)) / (2 * eps)
            assert fd == pytest.approx(g[gname][idx], rel=1e-6, abs=1e-8)


# ---------------------------------------------------------------- invariants

def test_gt_invariants():
    rng = np.random.default_rng(12)
    N, H, D = 50, 3, 4
    indptr, indices = rand_graph(rng, N, 0.12, dups=True)
    Q, K, V = (rng.standard_normal((N, H, D)) for _ in range(3))
    out, lse = oracle.gt_fwd(indptr, indices, Q, K, V)
    # weights sum to one: V = 1 gives out = 1
    ones, _ = oracle.gt_fwd(indptr, indices, Q, K, np.ones_like(V))
    np.testing.assert_allclose(ones, 1.0, atol=1e-14)
    # convex combination: within the neighbours' range; lse bounds
    for i in range(N):
        nb = indices[indptr[i]:indptr[i + 1]]
        assert np.all(out[i] <= V[nb].max(0) + 1e-12) and np.all(out[i] >= V[nb].min(0) - 1e-12)
        s = np.einsum("hd,jhd->jh", Q[i], K[nb]) / math.sqrt(D)
        assert np.all(lse[i] >= s.max(0) - 1e-12)
        assert np.all(lse[i] <= s.max(0) + math.log(len(nb)) + 1e-12)
    # permuting each row's neighbour order changes nothing
    perm = indices.copy()
    for i in range(N):
        perm[indptr[i]:indptr[i + 1]] = rng.permutation(perm[indptr[i]:indptr[i + 1]])
    out_p, lse_p = oracle.gt_fwd(indptr, perm, Q, K, V)
    np.testing.assert_allclose(out_p, out, atol=1e-13)
    np.testing.assert_allclose(lse_p, lse, atol=1e-13)
    # relabelling nodes is equivariant
    pi = rng.permutation(N)                      # new id of old node
    inv = np.argsort(pi)
    rows = [sorted(pi[indices[indptr[inv[n]]:indptr[inv[n] + 1]]]) for n in range(N)]
    indptr_r = np.zeros(N + 1, np.int32)
    indptr_r[1:] = np.cumsum([len(r) for r in rows])
    indices_r = np.array([j for r in rows for j in r], np.int32)
    out_r, lse_r = oracle.gt_fwd(indptr_r, indices_r, Q[inv], K[inv], V[inv])
    np.testing.assert_allclose(out_r, out[inv], atol=1e-13)
    np.testing.assert_allclose(lse_r, lse[inv], atol=1e-13)


def test_sampled_entry_points_match_full():
    rng = np.random.default_rng(13)
    N, H, D = 45, 2, 4
    indptr, indices = rand_graph(rng, N, 0.15, dups=True)
    Q, K, V, dO = (rng.standard_normal((N, H, D)) for _ in range(4))
    out, lse = oracle.gt_fwd(indptr, indices, Q, K, V)
    dQ, dK, dV = oracle.gt_bwd(indptr, indices, Q, K, V, dO)
    rows = np.array([0, 7, 7, 44, 13])
    o, l = oracle.gt_fwd(indptr, indices, Q, K, V, rows=rows)
    np.testing.assert_array_equal(o, out[rows]); np.testing.assert_array_equal(l, lse[rows])
    np.testing.assert_allclose(oracle.gt_bwd_dq_rows(indptr, indices, Q, K, V, dO, rows), dQ[rows],
                               atol=1e-13)
    dk, dv = oracle.gt_bwd_dkdv_srcs(indptr, indices, Q, K, V, dO, rows)
    np.testing.assert_allclose(dk, dK[rows], atol=1e-13)
    np.testing.assert_allclose(dv, dV[rows], atol=1e-13)


# ------------------------------------------------------- graph preprocessing

def test_transpose_matches_scipy_and_roundtrips():
    sp = pytest.importorskip("scipy.sparse")
    rng = np.random.default_rng(14)
    N = 300
    indptr, indices = rand_graph(rng, N, 0.02)
    t_indptr, t_dst = oracle.transpose(indptr, indices)
    A = sp.csr_matrix((np.ones(len(indices)), indices, indptr), shape=(N, N))
    At = A.T.tocsr()
    At.sort_indices()
    np.testing.assert_array_equal(t_indptr, At.indptr)
    np.testing.assert_array_equal(t_dst, At.indices)
    back_ptr, back_idx = oracle.transpose(t_indptr, t_dst)
    np.testing.assert_array_equal(back_ptr, indptr)
    np.testing.assert_array_equal(back_idx, indices)


def test_partition_definition():
    rng = np.random.default_rng(15)
    deg = rng.integers(0, 40, 200)
    deg[[3, 50, 199]] = [300, 97, 1000]
    indptr = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    p = oracle.partition(indptr, threshold=64, chunk=32)
    assert list(p["split_rows"]) == [i for i in range(200) if deg[i] > 64]
    for s, i in enumerate(p["split_rows"]):
        c0, c1 = p["chunk_ptr"][s], p["chunk_ptr"][s + 1]
        assert c1 - c0 == math.ceil(deg[i] / 32)
        assert p["chunk_beg"][c0] == indptr[i] and p["chunk_end"][c1 - 1] == indptr[i + 1]
        assert np.all(p["chunk_beg"][c0 + 1:c1] == p["chunk_end"][c0:c1 - 1])
        assert np.all(p["chunk_end"][c0:c1] - p["chunk_beg"][c0:c1] <= 32)
        assert np.all(p["chunk_row"][c0:c1] == i)


# ------------------------------------------------- storage rounding (GATv2)

def test_round_bf16_matches_torch_conversion():
    """The oracle's bfloat16 rounding (via float, ties to even) equals torch's
    float32 -> bfloat16 conversion, including exact ties and subnormals."""
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal(2000).astype(np.float32),
                        (rng.standard_normal(500) * 1e-39).astype(np.float32),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0,
                                  3.0e38], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in x])
    np.testing.assert_array_equal(got, ref)


def test_gatv2_stored_projection_rounding():
    """store='bf16' is the edge stage run on bf16-rounded projections."""
    rng = np.random.default_rng(22)
    N, F, H, D = 25, 6, 2, 4
    indptr, indices = rand_graph(rng, N, 0.3)
    X = rng.standard_normal((N, F)); Wl = rng.standard_normal((F, H * D))
    Wr = rng.standard_normal((F, H * D)); a = rng.standard_normal((H, D))
    FL, FR, out, lse = oracle.gatv2_fwd(indptr, indices, X, Wl, Wr, a, 0.2, store="bf16")
    rl = torch.from_numpy(X @ Wl).float().to(torch.bfloat16).double().numpy().reshape(N, H, D)
    rr = torch.from_numpy(X @ Wr).float().to(torch.bfloat16).double().numpy().reshape(N, H, D)
    np.testing.assert_array_equal(FL, rl)
    np.testing.assert_array_equal(FR, rr)
    o2, l2 = oracle.gatv2_fwd_rows(indptr, indices, rl, rr, a, np.arange(N))
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(lse, l2)


def test_gatv2_branch_slack_bounds_flipped_branches():
    """Move one source's projection across z = 0 for one edge element: the
    gradient change equals the slack computed on either side (one undecided
    element), and the slack is zero when no element is near z = 0."""
    rng = np.random.default_rng(23)
    N, F, H, D = 6, 3, 1, 2
    indptr = np.array([0, 2, 3, 4, 5, 6, 7], np.int32)
    indices = np.array([1, 2, 2, 3, 4, 5, 0], np.int32)
    X = rng.standard_normal((N, F)); Wl = rng.standard_normal((F, H * D))
    Wr = rng.standard_normal((F, H * D)); a = rng.standard_normal((H, D))
    dO = rng.standard_normal((N, H, D))
    far = oracle.gatv2_branch_slack(indptr, indices, X, Wl, Wr, a, dO, store=None, tau=1e-9)
    for v in far.values():
        assert np.all(v == 0.0)
    # make z of (row 0, source 1, d = 0) straddle zero: fr_1 = -fl_0 +/- eps
    FL = X @ Wl
    FR = X @ Wr
    eps = 1e-9
    res = {}
    for sign in (+1, -1):
        target = -FL[0, 0] + sign * eps
        # adjust X[1] along a direction that only changes FR[1, 0] (solve with the pseudo-inverse)
        X2 = X.copy()
        delta = np.zeros(H * D); delta[0] = target - FR[1, 0]
        X2[1] += np.linalg.lstsq(Wr.T, delta, rcond=None)[0]
        res[sign] = (X2, oracle.gatv2_bwd(indptr, indices, X2, Wl, Wr, a, dO))
    diff = np.abs(res[1][1]["dW_l"] - res[-1][1]["dW_l"])
    sl = oracle.gatv2_branch_slack(indptr, indices, res[1][0], Wl, Wr, a, dO, store=None, tau=1e-6)
    assert diff.max() > 1e-3                       # the branch matters
    assert np.all(diff <= sl["dW_l"] * (1 + 1e-6) + 1e-7)
    assert sl["dW_l"].max() <= diff.max() * (1 + 1e-6) + 1e-7   # and the bound is tight here


# ------------------------------------------------------------ block-sparse tiles

def test_tile_extract_by_brute_force():
    """Tiles, bitmaps and residual against an explicit per-edge loop; the kept
    and residual edges partition the graph."""
    rng = np.random.default_rng(31)
    N = 300
    indptr, indices = rand_graph(rng, N, 0.04)
    # a dense block so that some tiles pass the threshold
    rows = [list(indices[indptr[i]:indptr[i + 1]]) for i in range(N)]
    for i in range(128, 200):
        rows[i] = sorted(set(rows[i]) | set(range(32, 64)))
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    t = oracle.tile_extract(indptr, indices, N, min_nnz=20)
    counts = {}
    for i in range(N):
        for e in range(indptr[i], indptr[i + 1]):
            k = (i // 128, indices[e] // 16)
            counts[k] = counts.get(k, 0) + 1
    kept = sorted(k for k, c in counts.items() if c >= 20)
    assert len(kept) > 0
    got = [(p, c) for p in range(len(t["tile_ptr"]) - 1)
           for c in t["tile_col"][t["tile_ptr"][p]:t["tile_ptr"][p + 1]]]
    assert got == kept
    res_rows = [[] for _ in range(N)]
    for i in range(N):
        for e in range(indptr[i], indptr[i + 1]):
            j = indices[e]
            k = (i // 128, j // 16)
            if k in counts and counts[k] >= 20:
                ti = kept.index(k)
                assert t["tile_bits"][ti, i % 128] >> (j % 16) & 1
            else:
                res_rows[i].append(j)
    assert [list(t["r_indices"][t["r_indptr"][i]:t["r_indptr"][i + 1]]) for i in range(N)] == res_rows
    assert sum(bin(int(b)).count("1") for b in t["tile_bits"].ravel()) + len(t["r_indices"]) == len(indices)


def test_tile_extract_repeated_edges_by_brute_force():
    """Repeated (destination, source) pairs: counted towards the tile's
    threshold; in a kept tile the first occurrence in CSR order sets the mask
    bit and every later one stays in the residual, in CSR order; in a tile
    that is not kept all of them stay.  Checked by an explicit edge loop."""
    rng = np.random.default_rng(32)
    N = 300
    rows = [list(rng.integers(0, N, rng.integers(0, 5))) for _ in range(N)]
    for i in range(128, 190):            # a dense block: kept tiles over sources 32..63
        rows[i] = list(rng.permutation(np.arange(32, 64)))
    rows[130] = rows[130][:5] + [40, 40] + rows[130][5:] + [40]   # source 40 four times in a kept tile
    rows[200] = [7, 7, 7, 250]                                    # repeats in a tile that is not kept
    rows[129] = rows[129] + [33]
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    t = oracle.tile_extract(indptr, indices, N, min_nnz=20)
    counts = {}
    for i in range(N):
        for e in range(indptr[i], indptr[i + 1]):
            k = (i // 128, indices[e] // 16)
            counts[k] = counts.get(k, 0) + 1
    kept = sorted(k for k, c in counts.items() if c >= 20)
    got = [(p, c) for p in range(len(t["tile_ptr"]) - 1)
           for c in t["tile_col"][t["tile_ptr"][p]:t["tile_ptr"][p + 1]]]
    assert got == kept and len(kept) > 0
    bits = np.zeros_like(t["tile_bits"])
    res_rows = [[] for _ in range(N)]
    n_rep = 0
    for i in range(N):
        seen = set()
        for e in range(indptr[i], indptr[i + 1]):
            j = int(indices[e])
            k = (i // 128, j // 16)
            if k in kept and j not in seen:
                bits[kept.index(k), i % 128] |= np.uint16(1 << (j % 16))
            else:
                n_rep += k in kept
                res_rows[i].append(j)
            seen.add(j)
    assert n_rep == 4    # row 130: three repeats of 40; row 129: 33 once more
    np.testing.assert_array_equal(t["tile_bits"], bits)
    assert [list(t["r_indices"][t["r_indptr"][i]:t["r_indptr"][i + 1]]) for i in range(N)] == res_rows
    assert sum(bin(int(b)).count("1") for b in t["tile_bits"].ravel()) + len(t["r_indices"]) == len(indices)


# ------------------------------------------------------- min / max aggregation

def test_agg_hand_example():
    g = load("agg_hand.json")
    ip, ix = np.array(g["indptr"], np.int32), np.array(g["indices"], np.int32)
    X = np.array(g["X"], float)
    for op in ("max", "min"):
        out, arg = oracle.agg_fwd(ip, ix, X, op)
        np.testing.assert_array_equal(out, np.array(g[op + "_out"], float))
        np.testing.assert_array_equal(arg, np.array(g[op + "_arg"]))
    _, arg = oracle.agg_fwd(ip, ix, X, "max")
    np.testing.assert_array_equal(oracle.agg_bwd(arg, np.array(g["dO"], float)),
                                  np.array(g["max_dX"], float))


@pytest.mark.parametrize("op", ["max", "min"])
def test_agg_matches_dense_masked_reduction(op):
    """Duplicate-free graphs with ascending sources: a dense masked max/min,
    and numpy's argmax/argmin (first occurrence, i.e. the smallest source,
    which is the first edge of an ascending row), with values drawn from a
    small set so that ties are frequent."""
    rng = np.random.default_rng(51 if op == "max" else 52)
    N, F = 40, 6
    indptr, indices = rand_graph(rng, N, 0.2, self_loops=False)
    # empty row 5
    deg = np.diff(indptr)
    indices = np.delete(indices, np.arange(indptr[5], indptr[6]))
    deg[5] = 0
    indptr = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    X = rng.integers(-3, 4, (N, F)).astype(float)
    out, arg = oracle.agg_fwd(indptr, indices, X, op)
    mask = dense_mask(indptr, indices, N).numpy()
    fill = -np.inf if op == "max" else np.inf
    dense = np.where(mask[:, :, None], X[None, :, :], fill)   # [i, j, f]
    red = dense.max(1) if op == "max" else dense.min(1)
    who = dense.argmax(1) if op == "max" else dense.argmin(1)
    empty = ~mask.any(1)
    np.testing.assert_array_equal(out[~empty], red[~empty])
    np.testing.assert_array_equal(arg[~empty], who[~empty])
    assert np.all(out[empty] == 0.0) and np.all(arg[empty] == -1)
    assert empty.any() and (~empty).any()


@pytest.mark.parametrize("op", ["max", "min"])
def test_agg_matches_torch_scatter_reduce_and_autograd(op):
    """torch.scatter_reduce (amax / amin over the edges) gives the values;
    with tie-free inputs its autograd gives the gradient of the backward."""
    rng = np.random.default_rng(53 if op == "max" else 54)
    N, F = 60, 5
    indptr, indices = rand_graph(rng, N, 0.1, dups=True)
    X = rng.standard_normal((N, F))
    dO = rng.standard_normal((N, F))
    out, arg = oracle.agg_fwd(indptr, indices, X, op)
    dX = oracle.agg_bwd(arg, dO)
    rows = torch.from_numpy(np.repeat(np.arange(N), np.diff(indptr)).astype(np.int64))
    tX = torch.from_numpy(X).requires_grad_()
    src = tX[torch.from_numpy(indices.astype(np.int64))]
    red = torch.zeros(N, F, dtype=torch.float64).scatter_reduce(
        0, rows[:, None].expand(-1, F), src, reduce="amax" if op == "max" else "amin",
        include_self=False)
    np.testing.assert_array_equal(out, red.detach().numpy())
    (red * torch.from_numpy(dO)).sum().backward()
    # a duplicated edge repeats a value: torch splits the gradient among the
    # copies, the definition sends it once to that source; both sum to the same
    np.testing.assert_allclose(dX, tX.grad.numpy(), atol=1e-12)


def test_agg_invariants():
    """Reordering a row's edges keeps every value; the winner changes only
    among equal values; relabelling nodes is equivariant."""
    rng = np.random.default_rng(55)
    N, F = 50, 4
    indptr, indices = rand_graph(rng, N, 0.15)
    X = rng.integers(-2, 3, (N, F)).astype(float)
    out, arg = oracle.agg_fwd(indptr, indices, X, "max")
    ix2 = indices.copy()
    for i in range(N):
        b, e = indptr[i], indptr[i + 1]
        ix2[b:e] = rng.permutation(ix2[b:e])
    out2, arg2 = oracle.agg_fwd(indptr, ix2, X, "max")
    np.testing.assert_array_equal(out, out2)
    has = arg >= 0
    np.testing.assert_array_equal(X[arg[has], np.nonzero(has)[1]], X[arg2[has], np.nonzero(has)[1]])
    perm = rng.permutation(N)             # node v becomes perm[v]
    inv = np.argsort(perm)
    rows = [perm[indices[indptr[inv[u]]:indptr[inv[u] + 1]]] for u in range(N)]
    ip3 = np.zeros(N + 1, np.int32)
    ip3[1:] = np.cumsum([len(r) for r in rows])
    ix3 = np.concatenate(rows).astype(np.int32)
    X3 = np.empty_like(X)
    X3[perm] = X
    out3, arg3 = oracle.agg_fwd(ip3, ix3, X3, "max")
    np.testing.assert_array_equal(out3[perm], out)
    np.testing.assert_array_equal(np.where(arg >= 0, perm[np.maximum(arg, 0)], -1), arg3[perm])


# ------------------------------------------------------------ graph reordering

def test_reorder_hand_example():
    g = load("reorder_hand.json")
    ip, ix = np.array(g["indptr"], np.int32), np.array(g["indices"], np.int32)
    np.testing.assert_array_equal(oracle.order_rcm(ip, ix), g["rcm_perm"])
    np.testing.assert_array_equal(oracle.order_degree(ip, ix), g["degree_perm"])


def sym_graph(rng, N, p):
    """Symmetric, duplicate-free, without self-loops (sources ascending)."""
    a = rng.random((N, N)) < p
    a = np.triu(a, 1)
    a = a | a.T
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum(a.sum(1))
    return indptr, np.nonzero(a)[1].astype(np.int32)


@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_rcm_matches_scipy_on_symmetric_graphs(seed):
    """On a symmetric graph without self-loops or duplicates, the degree used
    here is twice the matrix row count, so the ordering rules coincide with
    scipy.sparse.csgraph.reverse_cuthill_mckee's (least-degree start,
    children by ascending degree, ties by id).  scipy breaks ties between
    equal-degree start nodes of different components in an unspecified
    order, so the graphs here are connected."""
    sp = pytest.importorskip("scipy.sparse")
    from scipy.sparse.csgraph import connected_components, reverse_cuthill_mckee
    rng = np.random.default_rng(seed)
    N = 60
    indptr, indices = sym_graph(rng, N, 0.12)
    m = sp.csr_matrix((np.ones(len(indices)), indices, indptr), shape=(N, N))
    assert connected_components(m, directed=False)[0] == 1
    order = reverse_cuthill_mckee(m, symmetric_mode=True)
    perm = oracle.order_rcm(indptr, indices)
    # scipy returns the order (position -> node); ours is node -> position
    np.testing.assert_array_equal(np.argsort(perm), order)


def test_rcm_recovers_a_shuffled_path_and_grid_bandwidth():
    rng = np.random.default_rng(5)
    N = 50
    lab = rng.permutation(N)
    rows = [[] for _ in range(N)]
    for t in range(N - 1):                        # path lab[0] - lab[1] - ... - lab[N-1]
        rows[lab[t + 1]].append(lab[t])
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    perm = oracle.order_rcm(indptr, indices)
    new_pos = perm[lab]                           # positions along the path
    assert np.all(np.abs(np.diff(new_pos)) == 1)  # bandwidth 1
    # a 12 x 12 grid under random labels: bandwidth falls to the grid's width order
    W = 12
    lab = rng.permutation(W * W)
    rows = [[] for _ in range(W * W)]
    for r in range(W):
        for c in range(W):
            if c + 1 < W:
                rows[lab[r * W + c]].append(lab[r * W + c + 1])
            if r + 1 < W:
                rows[lab[r * W + c]].append(lab[(r + 1) * W + c])
    indptr = np.zeros(W * W + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    perm = oracle.order_rcm(indptr, indices)
    dst = np.repeat(np.arange(W * W), np.diff(indptr))
    bw_before = np.abs(dst - indices).max()
    bw_after = np.abs(perm[dst] - perm[indices]).max()
    assert bw_after <= W + 1 < bw_before


def test_relabelled_graph_is_equivariant():
    """A relabelled graph with relabelled features gives the relabelled
    attention output (checked through the oracle's Graph Transformer)."""
    rng = np.random.default_rng(6)
    N, H, D = 40, 2, 4
    indptr, indices = rand_graph(rng, N, 0.15, dups=True)
    for perm in (oracle.order_rcm(indptr, indices), oracle.order_degree(indptr, indices)):
        assert sorted(perm.tolist()) == list(range(N))
        ip2, ix2 = oracle.relabel_csr(indptr, indices, perm)
        Q, K, V = (rng.standard_normal((N, H, D)) for _ in range(3))
        P = lambda x: x[np.argsort(perm)]         # row perm[v] of the result = row v
        o1, l1 = oracle.gt_fwd(indptr, indices, Q, K, V)
        o2, l2 = oracle.gt_fwd(ip2, ix2, P(Q), P(K), P(V))
        np.testing.assert_allclose(o2, P(o1), atol=1e-12)
        np.testing.assert_allclose(l2, P(l1), atol=1e-12)


# ------------------------------------- rounding bound of the fp32 GATv2 backward

def fp32_dense_gatv2_grads(indptr, indices, X, Wl, Wr, a, dO, slope=0.2):
    """An independent fp32 evaluation: torch autograd of the dense form,
    every tensor float32 (projections, scores, softmax, gradients)."""
    N = X.shape[0]
    H, D = a.shape
    tX, tWl, tWr, ta = (torch.from_numpy(x).float().requires_grad_() for x in (X, Wl, Wr, a))
    FL = (tX @ tWl).reshape(N, H, D)
    FR = (tX @ tWr).reshape(N, H, D)
    z = FL[:, None] + FR[None, :]
    e = (torch.nn.functional.leaky_relu(z, slope) * ta).sum(-1).permute(2, 0, 1)
    e = e.masked_fill(~dense_mask(indptr, indices, N)[None], float("-inf"))
    p = torch.exp(e - torch.logsumexp(e, -1)[..., None]).nan_to_num(0.0)
    out = torch.einsum("hij,jhd->ihd", p, FR)
    (out * torch.from_numpy(dO).float()).sum().backward()
    return {"dX": tX.grad, "dW_l": tWl.grad, "dW_r": tWr.grad, "da": ta.grad}


@pytest.mark.parametrize("seed,ascale", [(1, 1.0), (2, 4.0), (3, 8.0)])
def test_gatv2_fp32_bound_covers_an_fp32_evaluation_and_is_not_vacuous(seed, ascale):
    """The first-order rounding bound of the fp32 backward holds for an
    independent fp32 evaluation (with the LeakyReLU branch slack of float
    storage) and stays below 5% of the largest gradient.  It adds carried
    errors worst-case, so it is loose (about 10^3 times the errors an fp32
    evaluation shows): at the workloads' attention-vector scale (0.1 per
    element) it still separates a one-edge mistake, at larger scales it no
    longer does -- fp32 GATv2 gradient checks are consistency checks."""
    rng = np.random.default_rng(seed)
    N, F, H, D = 80, 16, 2, 16
    indptr, indices = rand_graph(rng, N, 0.15)
    lim = math.sqrt(6 / (F + H * D))
    f32 = lambda x: x.astype(np.float32).astype(np.float64)
    X = f32(rng.standard_normal((N, F)))
    Wl, Wr = f32(rng.uniform(-lim, lim, (F, H * D))), f32(rng.uniform(-lim, lim, (F, H * D)))
    a = f32(rng.standard_normal((H, D)) * ascale / math.sqrt(D))
    dO = f32(rng.standard_normal((N, H, D)))
    g = oracle.gatv2_bwd(indptr, indices, X, Wl, Wr, a, dO, 0.2, store="f32")
    b = oracle.gatv2_bwd_bound(indptr, indices, X, Wl, Wr, a, dO, 0.2)
    sl = oracle.gatv2_branch_slack(indptr, indices, X, Wl, Wr, a, dO, 0.2, store="f32")
    t = fp32_dense_gatv2_grads(indptr, indices, X, Wl, Wr, a, dO)
    # one edge dropped (row 0 loses its last source): a plausible indexing mistake
    ip2 = indptr.copy()
    ip2[1:] -= 1
    ix2 = np.delete(indices, indptr[1] - 1)
    g2 = oracle.gatv2_bwd(ip2, ix2, X, Wl, Wr, a, dO, 0.2, store="f32")
    for k in ("dX", "dW_l", "dW_r", "da"):
        err = np.abs(t[k].double().numpy() - g[k])
        assert np.all(err <= b[k] + sl[k]), k
        assert b[k].max() < 0.05 * np.abs(g[k]).max(), k
        if ascale == 1.0:
            assert np.any(np.abs(g2[k] - g[k]) > 10 * (b[k] + sl[k])), k


# ------------------------------------------------- Graph Transformer with edge bias

def edge_rows(indptr):
    return np.repeat(np.arange(len(indptr) - 1), np.diff(indptr))


def test_gt_bias_complete_graph_equals_sdpa_with_float_mask():
    """The additive score bias is scaled_dot_product_attention's float
    attn_mask on a complete graph (every row lists every node once)."""
    rng = np.random.default_rng(61)
    N, H, D = 9, 3, 8
    indptr = (np.arange(N + 1) * N).astype(np.int32)
    indices = np.tile(np.arange(N), N).astype(np.int32)
    Q, K, V = (rng.standard_normal((N, H, D)) for _ in range(3))
    B = rng.standard_normal((N * N, H)) * 2.0
    out, lse = oracle.gt_bias_fwd(indptr, indices, Q, K, V, B)
    mask = torch.from_numpy(B.reshape(N, N, H).transpose(2, 0, 1).copy())   # [H, i, j]
    t = lambda x: torch.from_numpy(x).permute(1, 0, 2)                      # [H, N, D]
    ref = torch.nn.functional.scaled_dot_product_attention(t(Q), t(K), t(V), attn_mask=mask)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_gt_bias_backward_matches_autograd():
    rng = np.random.default_rng(62)
    N, H, D = 22, 2, 4
    indptr, indices = rand_graph(rng, N, 0.25)
    E = len(indices)
    Q, K, V, dO = (rng.standard_normal((N, H, D)) for _ in range(4))
    B = rng.standard_normal((E, H)) * 3.0
    dQ, dK, dV, dB = oracle.gt_bias_bwd(indptr, indices, Q, K, V, B, dO)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (Q, K, V))
    tb = torch.from_numpy(B).requires_grad_()
    rows = torch.from_numpy(edge_rows(indptr))
    cols = torch.from_numpy(indices.astype(np.int64))
    s = torch.einsum("ihd,jhd->hij", tq, tk) / math.sqrt(D)
    bias = torch.zeros(H, N, N, dtype=torch.float64).index_put((torch.arange(H)[:, None].expand(H, E),
                                                                 rows[None].expand(H, E),
                                                                 cols[None].expand(H, E)), tb.T)
    mask = dense_mask(indptr, indices, N)
    s = (s + bias).masked_fill(~mask[None], float("-inf"))
    p = torch.exp(s - torch.logsumexp(s, -1)[..., None]).nan_to_num(0.0)
    out = torch.einsum("hij,jhd->ihd", p, tv)
    (out * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dB, tb.grad.numpy(), atol=1e-11)


def test_gt_bias_special_cases():
    """Zero bias is the plain layer; a bias constant over a row (per head)
    leaves the output unchanged and shifts lse by that constant; the bias
    gradient of each row and head sums to zero (softmax Jacobian)."""
    rng = np.random.default_rng(63)
    N, H, D = 30, 2, 4
    indptr, indices = rand_graph(rng, N, 0.2, dups=True)
    E = len(indices)
    Q, K, V, dO = (rng.standard_normal((N, H, D)) for _ in range(4))
    o0, l0 = oracle.gt_fwd(indptr, indices, Q, K, V)
    ob, lb = oracle.gt_bias_fwd(indptr, indices, Q, K, V, np.zeros((E, H)))
    np.testing.assert_array_equal(ob, o0)
    np.testing.assert_array_equal(lb, l0)
    c = rng.standard_normal((N, H))
    oc, lc = oracle.gt_bias_fwd(indptr, indices, Q, K, V, c[edge_rows(indptr)])
    np.testing.assert_allclose(oc, o0, atol=1e-12)
    fin = np.isfinite(l0)
    np.testing.assert_allclose(lc[fin], (l0 + c)[fin], atol=1e-12)
    B = rng.standard_normal((E, H))
    dB = oracle.gt_bias_bwd(indptr, indices, Q, K, V, B, dO)[3]
    sums = np.zeros((N, H))
    np.add.at(sums, edge_rows(indptr), dB)
    np.testing.assert_allclose(sums, 0.0, atol=1e-12)


# --------------------------------------------------- GAT (original attention score)

def dense_gat(X, W, a, mask, slope=0.2, rnd=None):
    N = X.shape[0]
    H, _, D = a.shape
    FL = X @ W
    if rnd is not None:
        FL = rnd(FL)
    FL = FL.reshape(N, H, D)
    el = (FL * a[:, 0]).sum(-1)                          # [N, H]
    er = (FL * a[:, 1]).sum(-1)
    e = torch.nn.functional.leaky_relu(el[:, None, :] + er[None, :, :], slope).permute(2, 0, 1)
    e = e.masked_fill(~mask[None], float("-inf"))
    lse = torch.logsumexp(e, -1)
    p = torch.exp(e - lse[..., None]).nan_to_num(0.0)
    return torch.einsum("hij,jhd->ihd", p, FL), lse.T


def test_gat_hand_example():
    g = load("gat_hand.json")
    FL, out, lse = oracle.gat_fwd(np.array(g["indptr"], np.int32), np.array(g["indices"], np.int32),
                                  np.array(g["X"]), np.array(g["W"]), np.array(g["a"]), 0.2)
    np.testing.assert_allclose(out, np.array(g["out"]), atol=1e-14)
    np.testing.assert_allclose(lse, np.array(g["lse"]), atol=1e-14)


@pytest.mark.parametrize("store", [None, "bf16"])
def test_gat_matches_dense_autograd(store):
    """Forward against the dense masked form; backward against torch autograd
    of it (for bf16 storage through a straight-through rounding step)."""
    rng = np.random.default_rng(71)
    N, F, H, D = 26, 6, 2, 4
    indptr, indices = rand_graph(rng, N, 0.25)
    X = rng.standard_normal((N, F)) * 2.0
    W = rng.standard_normal((F, H * D))
    a = rng.standard_normal((H, 2, D))
    dO = rng.standard_normal((N, H, D))
    FL, out, lse = oracle.gat_fwd(indptr, indices, X, W, a, 0.2, store=store)
    g = oracle.gat_bwd(indptr, indices, X, W, a, dO, 0.2, store=store)
    tX, tW, ta = (torch.from_numpy(x).requires_grad_() for x in (X, W, a))
    rnd = (lambda Y: straight_through(Y, "bf16")) if store == "bf16" else None
    to, tl = dense_gat(tX, tW, ta, dense_mask(indptr, indices, N), rnd=rnd)
    np.testing.assert_allclose(out, to.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, tl.detach().numpy(), atol=1e-12)
    (to * torch.from_numpy(dO)).sum().backward()
    np.testing.assert_allclose(g["dX"], tX.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(g["dW"], tW.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(g["da"], ta.grad.numpy(), atol=1e-10)


def test_gat_closed_forms_and_finite_differences():
    """a = 0 gives the neighbour mean of FL and lse = ln deg; the backward
    matches central differences of the forward."""
    rng = np.random.default_rng(72)
    N, F, H, D = 14, 4, 2, 3
    indptr, indices = rand_graph(rng, N, 0.3, dups=True)
    X = rng.standard_normal((N, F)); W = rng.standard_normal((F, H * D))
    FL, out, lse = oracle.gat_fwd(indptr, indices, X, W, np.zeros((H, 2, D)))
    for i in range(N):
        srcs = indices[indptr[i]:indptr[i + 1]]
        np.testing.assert_allclose(out[i], FL[srcs].mean(0), atol=1e-12)
        np.testing.assert_allclose(lse[i], np.log(len(srcs)), atol=1e-12)
    args = {"X": X, "W": W, "a": rng.standard_normal((H, 2, D))}
    dO = rng.standard_normal((N, H, D))
    g = oracle.gat_bwd(indptr, indices, args["X"], args["W"], args["a"], dO)
    loss = lambda a_: (oracle.gat_fwd(indptr, indices, a_["X"], a_["W"], a_["a"])[1] * dO).sum()
    eps = 1e-6
    for name, gname in (("X", "dX"), ("W", "dW"), ("a", "da")):
        for _ in range(5):
            idx = tuple(rng.integers(s) for s in args[name].shape)
            ap = {k: v.copy() for k, v in args.items()}
            ap[name][idx] += eps
            am = {k: v.copy() for k, v in args.items()}
            am[name][idx] -= eps
            assert (loss(ap) - loss(am)) / (2 * eps) == pytest.approx(g[gname][idx], rel=1e-6, abs=1e-8)


def test_gat_edge_stage_composes_to_the_layer():
    """The edge stage on FL, el = a_l . FL, er = a_r . FL gives the layer's
    output; its gradients, chained through el, er and FL = X W, give the
    layer's dX, dW and da."""
    rng = np.random.default_rng(73)
    N, F, H, D = 24, 5, 2, 3
    indptr, indices = rand_graph(rng, N, 0.3, dups=True)
    X = rng.standard_normal((N, F)); W = rng.standard_normal((F, H * D))
    a = rng.standard_normal((H, 2, D)); dO = rng.standard_normal((N, H, D))
    FL, out, lse = oracle.gat_fwd(indptr, indices, X, W, a)
    el = np.einsum("nhd,hd->nh", FL, a[:, 0])
    er = np.einsum("nhd,hd->nh", FL, a[:, 1])
    o2, l2 = oracle.gat_edge_fwd(indptr, indices, FL, el, er)
    np.testing.assert_allclose(o2, out, atol=1e-12)
    np.testing.assert_allclose(l2, lse, atol=1e-12)
    dFv, de_l, de_r = oracle.gat_edge_bwd(indptr, indices, FL, el, er, dO)
    dFL = dFv + de_l[:, :, None] * a[None, :, 0] + de_r[:, :, None] * a[None, :, 1]
    g = oracle.gat_bwd(indptr, indices, X, W, a, dO)
    np.testing.assert_allclose(dFL, g["dFL"], atol=1e-11)
    np.testing.assert_allclose(dFL.reshape(N, -1) @ W.T, g["dX"], atol=1e-11)
    np.testing.assert_allclose(X.T @ dFL.reshape(N, -1), g["dW"], atol=1e-11)
    da = np.stack([np.einsum("nh,nhd->hd", de_l, FL), np.einsum("nh,nhd->hd", de_r, FL)], 1)
    np.testing.assert_allclose(da, g["da"], atol=1e-11)


def test_projection_matmul_matches_numpy():
    """The oracle's projection product (the X W step of the GATv2 layer) is a
    plain triple loop; numpy's BLAS product computes the same sum."""
    rng = np.random.default_rng(21)
    for n, f, c in ((7, 5, 3), (1, 128, 128), (33, 8, 1)):
        X, W = rng.standard_normal((n, f)), rng.standard_normal((f, c))
        np.testing.assert_allclose(oracle.matmul(X, W), X @ W, rtol=1e-12, atol=1e-12)
    # an identity W returns X; a zero row of X gives a zero row
    X = rng.standard_normal((4, 6))
    X[2] = 0.0
    np.testing.assert_array_equal(oracle.matmul(X, np.eye(6)), X)
    assert not oracle.matmul(X, rng.standard_normal((6, 3)))[2].any()
