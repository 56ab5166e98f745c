"""Block-sparse tensor-core forward (kept 128 x 16 tiles on tcgen05, residual
edges on the CSR kernels, merged by log-sum-exp) vs the fp64 oracle, and the
tile extraction vs its definition, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import compare, dev

pytestmark = pytest.mark.gpu


def sbm_graph(seed, N, block=256, p_in=0.15, inter=4):
    rng = np.random.default_rng(seed)
    return synth.graph_sbm(rng, N, block, p_in, inter) if N % block == 0 else \
        synth.graph_sbm(rng, (N // block) * block, block, p_in, inter)


def ragged_graph(seed, N):
    """Dense diagonal blocks plus random edges, N not a multiple of 128 or 16."""
    rng = np.random.default_rng(seed)
    dst, src = [], []
    for b0 in range(0, N, 96):
        b1 = min(N, b0 + 96)
        m = rng.random((b1 - b0, b1 - b0)) < 0.3
        d, s = np.nonzero(m)
        dst.append(d + b0)
        src.append(s + b0)
    n = 3 * N
    dst.append(rng.integers(0, N, n))
    src.append(rng.integers(0, N, n))
    return synth.csr_from_edges(N, np.concatenate(dst), np.concatenate(src))


def inputs(seed, N, H, D, std):
    g = torch.Generator().manual_seed(seed)
    t = [(torch.randn(N, H, D, generator=g) * std).to(torch.bfloat16) for _ in range(4)]
    return [(x, x.double().numpy()) for x in t]


def check_tiles(plan, indptr, indices, N, tau):
    ref = oracle.tile_extract(indptr, indices, N, tau)
    np.testing.assert_array_equal(plan.array("tile_ptr"), ref["tile_ptr"])
    np.testing.assert_array_equal(plan.array("tile_col"), ref["tile_col"])
    bits = plan.array("tile_bits").view(np.uint16).reshape(-1, 128)
    np.testing.assert_array_equal(bits, ref["tile_bits"])
    np.testing.assert_array_equal(plan.array("r_indptr"), ref["r_indptr"])
    np.testing.assert_array_equal(plan.array("r_indices"), ref["r_indices"])
    return ref


@pytest.mark.parametrize("case", ["sbm_d128", "sbm_d64", "ragged_d128"])
def test_block_sparse_forward_and_backward(case):
    if case.startswith("sbm"):
        N, H, D = 4096, 4, (128 if case.endswith("128") else 64)
        indptr, indices = sbm_graph(7, N)
        tau = 16
    else:
        N, H, D = 1000, 2, 128
        indptr, indices = ragged_graph(8, N)
        tau = 24
    (q, qf), (k, kf), (v, vf), (do, dof) = inputs(3, N, H, D, D ** -0.5)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16, tile_min_nnz=tau)
    inf = plan.info()
    assert inf["n_tiles"] > 0 and inf["E_residual"] > 0
    ref_t = check_tiles(plan, indptr, indices, N, tau)
    # most of the SBM's edges fall in kept tiles
    if case.startswith("sbm"):
        assert inf["E_residual"] < 0.25 * len(indices)
    Q, K, V, dO = (dev(x) for x in (q, k, v, do))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    ro, rl = oracle.gt_fwd(indptr, indices, qf, kf, vf)
    compare(out, ro, "bf16", "out")
    compare(lse, rl, "bf16", "lse")
    # same layer on the CSR path (plan without tiles)
    plan_csr = sga.Plan(ip, ix, H, D, torch.bfloat16)
    out_c, lse_c = sga.gt_attn_fwd(plan_csr, Q, K, V)
    compare(out, out_c.double().cpu().numpy(), "bf16", "out vs CSR path")
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    rq, rk, rv = oracle.gt_bwd(indptr, indices, qf, kf, vf, dof)
    compare(dQ, rq, "bf16", "dQ")
    compare(dK, rk, "bf16", "dK")
    compare(dV, rv, "bf16", "dV")
    # deterministic: a second call gives the same bits
    dQ2, dK2, dV2 = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    assert torch.equal(dQ, dQ2) and torch.equal(dK, dK2) and torch.equal(dV, dV2)
    assert plan.device_error() == 0


def test_block_sparse_is_deterministic_and_handles_empty_panels():
    N, H, D = 2000, 1, 64
    indptr, indices = ragged_graph(9, N)
    # a threshold no tile reaches: everything stays on the CSR path
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16, tile_min_nnz=2048)
    assert plan.info()["n_tiles"] == 0
    (q, qf), (k, kf), (v, vf), _ = inputs(5, N, H, D, 0.125)
    Q, K, V = dev(q), dev(k), dev(v)
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    ro, rl = oracle.gt_fwd(indptr, indices, qf, kf, vf)
    compare(out, ro, "bf16", "out")
    _, dof = inputs(6, N, H, D, 1.0)[0]
    dO = dev(torch.from_numpy(dof).to(torch.bfloat16))
    rq, rk, rv = oracle.gt_bwd(indptr, indices, qf, kf, vf, dof)
    g = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    for t, ref, name in zip(g, (rq, rk, rv), ("dQ", "dK", "dV")):
        compare(t, ref, "bf16", name)
    plan2 = sga.Plan(ip, ix, H, D, torch.bfloat16, tile_min_nnz=20)
    a = sga.gt_attn_fwd(plan2, Q, K, V)
    b = sga.gt_attn_fwd(plan2, Q, K, V)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    compare(a[0], ro, "bf16", "out")
    g2 = sga.gt_attn_bwd(plan2, Q, K, V, a[0], a[1], dO)
    for t, ref, name in zip(g2, (rq, rk, rv), ("dQ", "dK", "dV")):
        compare(t, ref, "bf16", name)


def test_block_sparse_repeated_edges_join_the_residual():
    """A mask holds a (destination, source) pair once: in a kept tile the
    first edge of a pair sets the bit and its repeats go to the residual CSR,
    where they add their own softmax terms; the layer equals the oracle's,
    which counts every edge."""
    N, H, D = 300, 2, 64
    rng = np.random.default_rng(12)
    rows = [list(range(16)) + [3] for _ in range(N)]       # tile (panel, sources 0..15) kept everywhere
    rows[0] = rows[0] + [3, 40, 40]                          # source 3 three times; 40 twice (tile not kept)
    rows[131] = [5, 5] + rows[131]
    for i in range(N):
        rows[i] += list(rng.integers(0, N, 3))
    indptr = np.concatenate([[0], np.cumsum([len(r) for r in rows])]).astype(np.int32)
    indices = np.concatenate(rows).astype(np.int32)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16, tile_min_nnz=8)
    ref = check_tiles(plan, indptr, indices, N, 8)
    assert plan.info()["E_residual"] == len(ref["r_indices"]) >= N + 4
    (q, qf), (k, kf), (v, vf), (do, dof) = inputs(13, N, H, D, 0.5)
    Q, K, V, dO = (dev(x) for x in (q, k, v, do))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    ro, rl = oracle.gt_fwd(indptr, indices, qf, kf, vf)
    compare(out, ro, "bf16", "out")
    compare(lse, rl, "bf16", "lse")
    g = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    for t, r_, name in zip(g, oracle.gt_bwd(indptr, indices, qf, kf, vf, dof), ("dQ", "dK", "dV")):
        compare(t, r_, "bf16", name)
    assert plan.device_error() == 0


def blocky_graph(seed, N, sizes=(16, 48, 96, 200, 384, 520), p_in=0.35, extra=2):
    """Diagonal blocks of mixed sizes (so that panels keep from one to many
    tiles, in groups of four with ragged last groups) plus random edges."""
    rng = np.random.default_rng(seed)
    dst, src = [], []
    b0 = 0
    while b0 < N:
        b1 = min(N, b0 + int(rng.choice(sizes)))
        m = rng.random((b1 - b0, b1 - b0)) < p_in
        d, s_ = np.nonzero(m)
        dst.append(d + b0)
        src.append(s_ + b0)
        b0 = b1
    dst.append(rng.integers(0, N, extra * N))
    src.append(rng.integers(0, N, extra * N))
    return synth.csr_from_edges(N, np.concatenate(dst), np.concatenate(src))


@pytest.mark.parametrize("H,D", [(4, 64), (2, 128)])
def test_block_sparse_many_units_per_cta(H, D):
    """More (panel, head) units than SMs, with unequal tile counts per panel:
    every persistent CTA takes several units, so the buffers, TMEM
    accumulators and barrier phases are handed from unit to unit."""
    N = 24000
    indptr, indices = blocky_graph(21, N)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16, tile_min_nnz=12)
    ref_t = check_tiles(plan, indptr, indices, N, 12)
    per_panel = np.diff(ref_t["tile_ptr"])
    assert (per_panel > 0).sum() * H > 2 * 152 and per_panel.max() > 4 * 4 and (per_panel % 4 != 0).any()
    (q, qf), (k, kf), (v, vf), (do, dof) = inputs(22, N, H, D, 1.5 * D ** -0.5)
    Q, K, V, dO = (dev(x) for x in (q, k, v, do))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    ro, rl = oracle.gt_fwd(indptr, indices, qf, kf, vf)
    compare(out, ro, "bf16", "out")
    compare(lse, rl, "bf16", "lse")
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    rq, rk, rv = oracle.gt_bwd(indptr, indices, qf, kf, vf, dof)
    compare(dQ, rq, "bf16", "dQ")
    compare(dK, rk, "bf16", "dK")
    compare(dV, rv, "bf16", "dV")
    again = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    assert all(torch.equal(x, y) for x, y in zip((dQ, dK, dV), again))
    assert plan.device_error() == 0


def test_block_sparse_beyond_2_18_nodes():
    """N above 2^18 (the tile extraction has no per-panel histogram limit);
    sampled rows and sources against the oracle, tiles bit-exact."""
    N, H, D = (1 << 18) + 3001, 2, 64
    rng = np.random.default_rng(31)
    dst, src = [rng.integers(0, N, 2 * N)], [rng.integers(0, N, 2 * N)]
    for b0 in list(range(0, 4096, 256)) + [N - 300]:   # dense blocks at both ends
        b1 = min(N, b0 + 256)
        m = rng.random((b1 - b0, b1 - b0)) < 0.3
        d, s_ = np.nonzero(m)
        dst.append(d + b0)
        src.append(s_ + b0)
    indptr, indices = synth.csr_from_edges(N, np.concatenate(dst), np.concatenate(src))
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16, tile_min_nnz=16)
    check_tiles(plan, indptr, indices, N, 16)
    assert plan.info()["n_tiles"] > 0
    (q, qf), (k, kf), (v, vf), (do, dof) = inputs(32, N, H, D, D ** -0.5)
    Q, K, V, dO = (dev(x) for x in (q, k, v, do))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([rng.integers(0, N, 500), np.arange(0, 600, 7), [N - 300, N - 1]]))
    ro, rl = oracle.gt_fwd(indptr, indices, qf, kf, vf, rows=rows)
    r = torch.from_numpy(rows).cuda()
    compare(out[r], ro, "bf16", "out")
    compare(lse[r], rl, "bf16", "lse")
    compare(dQ[r], oracle.gt_bwd_dq_rows(indptr, indices, qf, kf, vf, dof, rows), "bf16", "dQ")
    rk, rv = oracle.gt_bwd_dkdv_srcs(indptr, indices, qf, kf, vf, dof, rows)
    compare(dK[r], rk, "bf16", "dK")
    compare(dV[r], rv, "bf16", "dV")
    assert plan.device_error() == 0


def test_block_sparse_rejects_unsupported_shapes():
    indptr = np.array([0, 1, 2], np.int32)
    indices = np.array([0, 1], np.int32)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    for dtype, D in ((torch.float32, 64), (torch.bfloat16, 32)):
        with pytest.raises(sga.SgaError) as ei:
            sga.Plan(ip, ix, 1, D, dtype, tile_min_nnz=4)
        assert ei.value.status == sga.SGA_EUNSUPPORTED


@pytest.mark.slow
def test_workload5_block_sparse_sampled():
    """The SBM workload at full size (N = 262,144, 11.3M edges, H = 4, D = 128)
    in the launch configuration the benchmark times (tile_min_nnz = 16)."""
    w = synth.WORKLOADS[5]
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w)
    h = {k: v[1] for k, v in x.items()}
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, w.H, w.D, torch.bfloat16, tile_min_nnz=16)
    check_tiles(plan, indptr, indices, w.N, 16)
    Q, K, V, dO = (dev(x[n][0]) for n in ("Q", "K", "V", "dOut"))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    torch.cuda.synchronize()
    rng = np.random.default_rng(55)
    rows = np.unique(np.concatenate([rng.integers(0, w.N, 2000), [0, 127, 128, w.N - 1]]))
    srcs = np.unique(np.concatenate([rng.integers(0, w.N, 300), [0, 127, 128, w.N - 1]]))
    ro, rl = oracle.gt_fwd(indptr, indices, h["Q"], h["K"], h["V"], rows=rows)
    r = torch.from_numpy(rows).cuda()
    compare(out[r], ro, "bf16", "out")
    compare(lse[r], rl, "bf16", "lse")
    rq = oracle.gt_bwd_dq_rows(indptr, indices, h["Q"], h["K"], h["V"], h["dOut"], rows)
    compare(dQ[r], rq, "bf16", "dQ")
    rk, rv = oracle.gt_bwd_dkdv_srcs(indptr, indices, h["Q"], h["K"], h["V"], h["dOut"], srcs)
    sj = torch.from_numpy(srcs).cuda()
    compare(dK[sj], rk, "bf16", "dK")
    compare(dV[sj], rv, "bf16", "dV")
    assert plan.device_error() == 0
