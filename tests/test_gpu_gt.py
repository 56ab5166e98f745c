"""Graph Transformer CUDA path vs the fp64 oracle, through the C ABI.

Small seeded graphs that span many warps, split rows and ragged tails; edge
cases (empty rows, degree 1, empty graph, duplicates, every lane layout);
bit-exact preprocessing; determinism; error codes."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import TORCH_DT, compare, dev

pytestmark = pytest.mark.gpu


def csr(rows):
    indptr = np.zeros(len(rows) + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    indices = np.array([j for r in rows for j in r], np.int32)
    return indptr, indices


def random_csr(rng, N, mean_deg, self_loops=True, empty_frac=0.0, hubs=()):
    rows = []
    for i in range(N):
        if rng.random() < empty_frac:
            rows.append([])
            continue
        d = rng.poisson(mean_deg)
        r = set(rng.integers(0, N, d).tolist())
        if self_loops:
            r.add(i)
        rows.append(sorted(r))
    for h, deg in hubs:
        rows[h] = sorted(set(rng.integers(0, N, deg).tolist()) | {h})
    return csr(rows)


def values(rng, N, H, D, dtype, std=1.0):
    x = (rng.standard_normal((N, H, D)) * std).astype(np.float32)
    t = torch.from_numpy(x).to(TORCH_DT[dtype])
    return t, t.to(torch.float64).numpy()


def run_gt(indptr, indices, H, D, dtype, seed=0, std=1.0, backward=True, split=0, chunk=0,
           std_do=1.0):
    rng = np.random.default_rng(seed)
    N = len(indptr) - 1
    (q, qf), (k, kf), (v, vf) = (values(rng, N, H, D, dtype, std) for _ in range(3))
    do, dof = values(rng, N, H, D, dtype, std_do)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, TORCH_DT[dtype], split_threshold=split, chunk_len=chunk)
    Q, K, V, dO = dev(q), dev(k), dev(v), dev(do)
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    ref_out, ref_lse = oracle.gt_fwd(indptr, indices, qf, kf, vf)
    compare(out, ref_out, dtype, "out")
    compare(lse, ref_lse, dtype, "lse")
    if backward:
        dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
        rq, rk, rv = oracle.gt_bwd(indptr, indices, qf, kf, vf, dof)
        compare(dQ, rq, dtype, "dQ")
        compare(dK, rk, dtype, "dK")
        compare(dV, rv, dtype, "dV")
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return plan


@pytest.mark.parametrize("key", [1, 3, 4, 5])
def test_small_workloads_match_oracle(key):
    w = synth.small_workload(key)
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w)
    N = w.N
    if key == 1:
        x["dOut"] = synth.round_to(synth.normal(w.seed, synth.STREAM_DOUT, (N, w.H, w.D)), w.dtype)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, w.H, w.D, TORCH_DT[w.dtype])
    Q, K, V, dO = (dev(x[n][0]) for n in ("Q", "K", "V", "dOut"))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    ro, rl = oracle.gt_fwd(indptr, indices, x["Q"][1], x["K"][1], x["V"][1])
    compare(out, ro, w.dtype, "out")
    compare(lse, rl, w.dtype, "lse")
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    rq, rk, rv = oracle.gt_bwd(indptr, indices, x["Q"][1], x["K"][1], x["V"][1], x["dOut"][1])
    compare(dQ, rq, w.dtype, "dQ")
    compare(dK, rk, w.dtype, "dK")
    compare(dV, rv, w.dtype, "dV")
    assert plan.device_error() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H,D", [(1, 32), (2, 32), (1, 64), (2, 64), (4, 32), (3, 64), (1, 128),
                                 (4, 128), (8, 128), (5, 32), (3, 128), (6, 64)])
def test_every_lane_layout(dtype, H, D):
    """Edge groups of 4..32 lanes and 1..8 chunks per lane; forced splitting."""
    rng = np.random.default_rng(H * 1000 + D)
    indptr, indices = random_csr(rng, 300, 6, hubs=[(7, 250), (299, 120)])
    run_gt(indptr, indices, H, D, dtype, seed=H + D, std=1 / math.sqrt(D) if dtype == "bf16" else 1.0,
           split=40, chunk=16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_rows_degree_one_and_duplicates(dtype):
    rows = [[], [3], [0, 0, 2], [], [1, 2, 3, 4], [4], [], [0, 1, 1, 1, 6]]
    indptr, indices = csr(rows)
    run_gt(indptr, indices, 2, 32, dtype, split=2, chunk=1)
    run_gt(indptr, indices, 2, 32, dtype)


def test_empty_graph_and_single_node():
    run_gt(np.zeros(6, np.int32), np.zeros(0, np.int32), 4, 64, "bf16")
    run_gt(np.array([0, 1], np.int32), np.array([0], np.int32), 4, 32, "f32")


def test_no_self_loops_and_unreferenced_sources():
    rng = np.random.default_rng(3)
    indptr, indices = random_csr(rng, 500, 3, self_loops=False, empty_frac=0.2)
    run_gt(indptr, indices, 4, 64, "bf16", std=0.125)


def test_plan_arrays_bit_exact():
    w = synth.small_workload(4)
    indptr, indices = synth.make_graph(w)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    for T, C in ((256, 128), (17, 5), (1, 1)):
        plan = sga.Plan(ip, ix, 4, 64, torch.bfloat16, split_threshold=T, chunk_len=C)
        t_indptr, t_dst = oracle.transpose(indptr, indices)
        np.testing.assert_array_equal(plan.array("t_indptr"), t_indptr)
        np.testing.assert_array_equal(plan.array("t_dst"), t_dst)
        for prefix, ptr in (("", indptr), ("t_", t_indptr)):
            ref = oracle.partition(ptr, T, C)
            np.testing.assert_array_equal(plan.array(prefix + "split_rows"), ref["split_rows"])
            np.testing.assert_array_equal(plan.array(prefix + "chunk_ptr"), ref["chunk_ptr"])
            for f in ("chunk_row", "chunk_beg", "chunk_end"):
                np.testing.assert_array_equal(plan.array(prefix + f), ref[f])


def test_runs_are_bitwise_reproducible():
    w = synth.small_workload(3)
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, w.H, w.D, torch.bfloat16)
    Q, K, V, dO = (dev(x[n][0]) for n in ("Q", "K", "V", "dOut"))
    a = [sga.gt_attn_fwd(plan, Q, K, V) for _ in range(2)]
    assert torch.equal(a[0][0], a[1][0]) and torch.equal(a[0][1], a[1][1])
    g = [sga.gt_attn_bwd(plan, Q, K, V, a[0][0], a[0][1], dO) for _ in range(2)]
    for x0, x1 in zip(*g):
        assert torch.equal(x0, x1)


def test_invalid_csr_is_rejected():
    good_ptr = np.array([0, 2, 3, 5], np.int32)
    good_idx = np.array([0, 1, 2, 0, 2], np.int32)
    cases = [
        (np.array([1, 2, 3, 5], np.int32), good_idx),        # indptr[0] != 0
        (np.array([0, 3, 2, 5], np.int32), good_idx),        # not monotone
        (np.array([0, 2, 3, 4], np.int32), good_idx),        # indptr[N] != E
        (good_ptr, np.array([0, 1, 3, 0, 2], np.int32)),     # index >= N
        (good_ptr, np.array([0, -1, 2, 0, 2], np.int32)),    # negative index
    ]
    for ptr, idx in cases:
        with pytest.raises(sga.SgaError) as ei:
            sga.Plan(dev(torch.from_numpy(ptr)), dev(torch.from_numpy(idx)), 1, 32, torch.float32)
        assert ei.value.status == sga.SGA_EINVAL
    sga.Plan(dev(torch.from_numpy(good_ptr)), dev(torch.from_numpy(good_idx)), 1, 32, torch.float32)


def test_call_checks():
    indptr, indices = csr([[0, 1], [1], [0, 2]])
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, 2, 32, torch.float32)
    Q = torch.randn(3, 2, 32, device="cuda")
    with pytest.raises(TypeError):
        sga.gt_attn_fwd(plan, Q.bfloat16(), Q.bfloat16(), Q.bfloat16())
    lib = sga.load_library()
    import ctypes
    p = ctypes.c_void_p
    out = torch.empty_like(Q)
    lse = torch.empty(3, 2, device="cuda")
    # wrong head count for this plan
    st = lib.gt_attn_fwd(plan.handle, p(ip.data_ptr()), p(ix.data_ptr()), p(Q.data_ptr()),
                         p(Q.data_ptr()), p(Q.data_ptr()), 3, 5, 1, 32, sga.SGA_F32,
                         p(out.data_ptr()), p(lse.data_ptr()), None)
    assert st == sga.SGA_EINVAL
    # misaligned tensor pointer
    st = lib.gt_attn_fwd(plan.handle, p(ip.data_ptr()), p(ix.data_ptr()), p(Q.data_ptr() + 4),
                         p(Q.data_ptr()), p(Q.data_ptr()), 3, 5, 2, 32, sga.SGA_F32,
                         p(out.data_ptr()), p(lse.data_ptr()), None)
    assert st == sga.SGA_EINVAL
    # a GATv2 call on a Graph Transformer plan
    st = lib.gatv2_fwd(plan.handle, p(ip.data_ptr()), p(ix.data_ptr()), *([p(Q.data_ptr())] * 4),
                       3, 5, 64, 2, 32, ctypes.c_float(0.2), sga.SGA_F32, *([p(out.data_ptr())] * 3),
                       p(lse.data_ptr()), None)
    assert st == sga.SGA_EINVAL


def test_device_range_check_flags_corrupted_indices():
    """An index corrupted after planning is caught by the kernel's own range
    check (the access is skipped, a bit is set, the host reads it)."""
    indptr, indices = csr([[0, 1], [1, 2], [0, 2]])
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, 1, 32, torch.float32)
    Q = torch.randn(3, 1, 32, device="cuda")
    ix[3] = 1000                      # out of range now
    out, lse = sga.gt_attn_fwd(plan, Q, Q, Q)
    assert plan.device_error() == 1
    assert plan.device_error() == 0   # read clears it
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("key", [4, 3])
def test_descending_degree_walking_order_is_bitwise_identical(key):
    """Walking rows by descending degree changes which warp computes a row,
    not the row's arithmetic: outputs and gradients are bit-identical to the
    ascending-id walk; the orders are the stable sort by descending degree.
    (Workload 3's two-chunk rows merge their split rows inside the kernels,
    in chunk order whichever chunk finishes last.)"""
    w = synth.small_workload(key)
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    Q, K, V, dO = (dev(x[n][0]) for n in ("Q", "K", "V", "dOut"))
    res = []
    for ro in (2, 1):   # ascending id, descending degree
        plan = sga.Plan(ip, ix, w.H, w.D, torch.bfloat16, row_order=ro, split_threshold=64,
                        chunk_len=32)
        out, lse = sga.gt_attn_fwd(plan, Q, K, V)
        res.append((out, lse) + tuple(sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)))
        if ro == 1:
            deg = np.diff(indptr.astype(np.int64))
            t_indptr, _ = oracle.transpose(indptr, indices)
            tdeg = np.diff(t_indptr.astype(np.int64))
            N = len(deg)
            np.testing.assert_array_equal(plan.array("row_order"), np.lexsort((np.arange(N), -deg)))
            np.testing.assert_array_equal(plan.array("t_row_order"), np.lexsort((np.arange(N), -tdeg)))
    for a, b in zip(*res):
        assert torch.equal(a, b)
    ro, rl = oracle.gt_fwd(indptr, indices, x["Q"][1], x["K"][1], x["V"][1])
    compare(res[1][0], ro, "bf16", "out")
