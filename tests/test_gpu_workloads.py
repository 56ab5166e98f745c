"""Parity at the five workloads' full sizes, with the plan options bench.py
uses.  Workloads 1-3 are compared element by element on every output; for
the two largest graphs (R-MAT with super nodes, block-dense SBM) the oracle
computes sampled rows and sources one by one: random ones plus the
highest-degree ones, which take the split-and-merge path."""
import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import TORCH_DT, compare, dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def gt_setup(key):
    """Forward and backward of a Graph Transformer workload at full size, with
    the default plan (the one bench.py uses); also returns the plan's split
    threshold, above which rows and sources take the split-and-merge path."""
    w = synth.WORKLOADS[key]
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w)
    if "dOut" not in x:
        x["dOut"] = synth.round_to(synth.normal(w.seed, synth.STREAM_DOUT, (w.N, w.H, w.D)), w.dtype)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, w.H, w.D, TORCH_DT[w.dtype])
    d = {k: dev(v[0]) for k, v in x.items()}
    out, lse = sga.gt_attn_fwd(plan, d["Q"], d["K"], d["V"])
    grads = sga.gt_attn_bwd(plan, d["Q"], d["K"], d["V"], out, lse, d["dOut"])
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return w, indptr, indices, x, out, lse, grads, plan.info()["split_threshold"]


def test_workload1_gt_forward_fp32_full():
    w, indptr, indices, x, out, lse, _, _ = gt_setup(1)
    ro, rl = oracle.gt_fwd(indptr, indices, x["Q"][1], x["K"][1], x["V"][1])
    compare(out, ro, "f32", "out")
    compare(lse, rl, "f32", "lse")


def test_workload2_gatv2_full():
    w = synth.WORKLOADS[2]
    indptr, indices = synth.make_graph(w)
    x = synth.gatv2_inputs(w)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, w.H, w.D, torch.bfloat16, F=w.F)
    d = {k: dev(v[0]) for k, v in x.items()}
    FL, FR, out, lse = sga.gatv2_fwd(plan, d["X"], d["W_l"], d["W_r"], d["a"], 0.2)
    dX, dWl, dWr, da = sga.gatv2_bwd(plan, d["X"], d["W_l"], d["W_r"], d["a"], FL, FR, out, lse,
                                     d["dOut"], 0.2)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    h = {k: v[1] for k, v in x.items()}
    rFL, rFR, ro, rl = oracle.gatv2_fwd(indptr, indices, h["X"], h["W_l"], h["W_r"], h["a"], 0.2,
                                        store="bf16")
    # projections are correctly rounded: bit-exact
    assert np.array_equal(FL.double().cpu().numpy(), rFL)
    assert np.array_equal(FR.double().cpu().numpy(), rFR)
    compare(out, ro, "bf16", "out")
    compare(lse, rl, "bf16", "lse")
    g = oracle.gatv2_bwd(indptr, indices, h["X"], h["W_l"], h["W_r"], h["a"], h["dOut"], 0.2,
                         store="bf16")
    sl = oracle.gatv2_branch_slack(indptr, indices, h["X"], h["W_l"], h["W_r"], h["a"],
                                   h["dOut"], 0.2, store="bf16")
    compare(dX, g["dX"], "bf16", "dX", slack=sl["dX"])
    compare(dWl, g["dW_l"], "bf16", "dW_l", slack=sl["dW_l"])
    compare(dWr, g["dW_r"], "bf16", "dW_r", slack=sl["dW_r"])
    compare(da, g["da"], "bf16", "da", slack=sl["da"])
    # bf16 projections agree bit for bit, so no branch is left undecided
    assert all(not v.any() for v in sl.values())


def test_workload3_gt_full():
    w, indptr, indices, x, out, lse, (dQ, dK, dV), _ = gt_setup(3)
    h = {k: v[1] for k, v in x.items()}
    ro, rl = oracle.gt_fwd(indptr, indices, h["Q"], h["K"], h["V"])
    compare(out, ro, "bf16", "out")
    compare(lse, rl, "bf16", "lse")
    rq, rk, rv = oracle.gt_bwd(indptr, indices, h["Q"], h["K"], h["V"], h["dOut"])
    compare(dQ, rq, "bf16", "dQ")
    compare(dK, rk, "bf16", "dK")
    compare(dV, rv, "bf16", "dV")


@pytest.mark.parametrize("key", [4, 5])
def test_large_workloads_sampled(key):
    """Sampled rows: 1500 random, the 20 of highest degree and up to 400 more
    split rows drawn at random (R-MAT has about 1,350 rows above its split
    threshold, up to 64k edges each).  Sampled sources: 300 random, the 8 of
    highest degree and up to 12 more split sources; the oracle recomputes
    the softmax of every destination row of a source, which bounds how many
    hub sources it can afford."""
    w, indptr, indices, x, out, lse, (dQ, dK, dV), thr = gt_setup(key)
    h = {k: v[1] for k, v in x.items()}
    rng = np.random.default_rng(key)
    deg = np.diff(indptr.astype(np.int64))
    t_indptr, t_dst = oracle.transpose(indptr, indices)
    tdeg = np.diff(t_indptr.astype(np.int64))
    split, tsplit = np.flatnonzero(deg > thr), np.flatnonzero(tdeg > thr)
    rows = np.unique(np.concatenate([rng.integers(0, w.N, 1500), np.argsort(deg)[-20:],
                                     rng.permutation(split)[:400]]))
    srcs = np.unique(np.concatenate([rng.integers(0, w.N, 300), np.argsort(tdeg)[-8:],
                                     rng.permutation(tsplit)[:12]]))
    if key == 4:
        # the super-node path is what this workload is for
        assert np.isin(split, rows).sum() >= min(400, split.size) and split.size > 100
    ro, rl = oracle.gt_fwd(indptr, indices, h["Q"], h["K"], h["V"], rows=rows)
    r = torch.from_numpy(rows).cuda()
    compare(out[r], ro, "bf16", "out")
    compare(lse[r], rl, "bf16", "lse")
    rq = oracle.gt_bwd_dq_rows(indptr, indices, h["Q"], h["K"], h["V"], h["dOut"], rows)
    compare(dQ[r], rq, "bf16", "dQ")
    rk, rv = oracle.gt_bwd_dkdv_srcs(indptr, indices, h["Q"], h["K"], h["V"], h["dOut"], srcs,
                                     transposed=(t_indptr, t_dst))
    sj = torch.from_numpy(srcs).cuda()
    compare(dK[sj], rk, "bf16", "dK")
    compare(dV[sj], rv, "bf16", "dV")
