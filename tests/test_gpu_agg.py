"""Min / max neighbourhood aggregation (the degree-aware reduction layer) on
the GPU vs the fp64 oracle, through the C ABI.

The forward is exact: values and winning sources are compared bit for bit.
Inputs are drawn from a small set of values, so most elements of a row tie
and the first-edge rule is exercised across edge groups, warps and the
chunks of split rows.  The backward is a sum of upstream gradients per
source (fp32 accumulation): compared within the stated tolerances."""
import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import TORCH_DT, compare, dev
from test_gpu_gt import csr, random_csr

pytestmark = pytest.mark.gpu


def tie_values(rng, N, H, D, dtype, levels=7):
    x = rng.integers(-(levels // 2), levels // 2 + 1, (N, H, D)).astype(np.float32) * 0.5
    x += (rng.random((N, H, D)) < 0.2) * rng.standard_normal((N, H, D)).astype(np.float32)
    t = torch.from_numpy(x).to(TORCH_DT[dtype])
    return t, t.to(torch.float64).numpy()


def expected_mask(indptr, indices, arg, dtype):
    """The win mask the forward must write, from the oracle's winners: the
    winning edge of (row i, element f) is the first edge of row i whose
    source is arg[i, f] (equal sources carry equal values, and ties go to the
    first edge); bit f % EL of byte (edge, f // EL)."""
    EL = 8 if dtype == "bf16" else 4
    N = len(indptr) - 1
    a = arg.reshape(N, -1)
    HD = a.shape[1]
    mask = np.zeros((len(indices), HD // EL), np.uint8)
    for i in range(N):
        b, e = indptr[i], indptr[i + 1]
        first = {}
        for x in range(b, e):
            first.setdefault(int(indices[x]), x)
        for f in range(HD):
            if a[i, f] >= 0:
                mask[first[int(a[i, f])], f // EL] |= np.uint8(1 << (f % EL))
    return mask


def run_agg(indptr, indices, H, D, dtype, op, seed=0, split=0, chunk=0, backward=True):
    rng = np.random.default_rng(seed)
    N = len(indptr) - 1
    X, xf = tie_values(rng, N, H, D, dtype)
    dO = torch.from_numpy(rng.standard_normal((N, H, D)).astype(np.float32)).to(TORCH_DT[dtype])
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, TORCH_DT[dtype], split_threshold=split, chunk_len=chunk,
                    layer=sga.SGA_LAYER_MINMAX)
    out, arg, mask = sga.agg_minmax_fwd(plan, dev(X), op)
    ro, ra = oracle.agg_fwd(indptr, indices, xf, op)
    assert np.array_equal(out.double().cpu().numpy(), ro), "values differ"
    assert np.array_equal(arg.cpu().numpy(), ra), "winning sources differ"
    if len(indices):
        assert np.array_equal(mask.cpu().numpy().reshape(len(indices), -1),
                              expected_mask(indptr, indices, ra, dtype)), "win masks differ"
    if backward:
        dX = sga.agg_minmax_bwd(plan, mask, dev(dO))
        rdx = oracle.agg_bwd(ra, dO.double().numpy())
        compare(dX, rdx, dtype, "dX")
        assert torch.equal(dX, sga.agg_minmax_bwd(plan, mask, dev(dO))), "backward not reproducible"
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return plan


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H,D", [(1, 32), (2, 32), (4, 32), (1, 64), (2, 64), (4, 128), (8, 128),
                                 (3, 64), (5, 32)])
@pytest.mark.parametrize("op", ["max", "min"])
def test_every_lane_layout_with_split_rows(dtype, H, D, op):
    """Edge groups of 4..32 lanes and 1..8 chunks per lane; hub rows split
    into chunks of 16 (threshold 40)."""
    rng = np.random.default_rng(H * 100 + D + (1 if op == "min" else 0))
    indptr, indices = random_csr(rng, 400, 9, hubs=[(7, 300), (399, 120), (200, 41)])
    run_agg(indptr, indices, H, D, dtype, op, seed=H + D, split=40, chunk=16)
    run_agg(indptr, indices, H, D, dtype, op, seed=H + D + 1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_empty_rows_degree_one_duplicates_and_empty_graph(dtype):
    rows = [[], [3], [0, 0, 2], [], [1, 2, 3, 4], [4], [], [0, 1, 1, 1, 6]]
    indptr, indices = csr(rows)
    run_agg(indptr, indices, 2, 32, dtype, "max", split=2, chunk=1)
    run_agg(indptr, indices, 2, 32, dtype, "min")
    run_agg(np.zeros(6, np.int32), np.zeros(0, np.int32), 4, 64, dtype, "max")


def test_small_workload_recipe():
    """The aggregation workload's recipe (lognormal citation-like graph with a
    hub, F = 512 as H=4 x D=128, bf16) at reduced size, default plan."""
    w = synth.small_workload(6)
    indptr, indices = synth.make_graph(w)
    x = synth.agg_inputs(w)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, w.H, w.D, torch.bfloat16, layer=sga.SGA_LAYER_MINMAX)
    out, arg, mask = sga.agg_minmax_fwd(plan, dev(x["X"][0]), "min")
    ro, ra = oracle.agg_fwd(indptr, indices, x["X"][1], "min")
    assert np.array_equal(out.double().cpu().numpy(), ro)
    assert np.array_equal(arg.cpu().numpy(), ra)
    # without the winners output, the values and the mask are the same
    out2, none, mask2 = sga.agg_minmax_fwd(plan, dev(x["X"][0]), "min", arg=False)
    assert none is None and torch.equal(out2, out) and torch.equal(mask2, mask)
    dX = sga.agg_minmax_bwd(plan, mask, dev(x["dOut"][0]))
    compare(dX, oracle.agg_bwd(ra, x["dOut"][1]), "bf16", "dX")
    assert plan.device_error() == 0


def test_autograd_function_and_plan_kind_checks():
    rng = np.random.default_rng(4)
    indptr, indices = random_csr(rng, 300, 6, hubs=[(1, 280)])
    N = len(indptr) - 1
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, 2, 64, torch.float32, layer=sga.SGA_LAYER_MINMAX)
    gen = torch.Generator().manual_seed(8)   # seeded: the same draw in every process
    X = torch.randn(N, 2, 64, generator=gen).cuda().requires_grad_()
    out = sga.MinMaxAggregation.apply(X, plan, "max")
    g = torch.randn(tuple(out.shape), generator=gen).cuda()
    out.backward(g)
    ro, ra = oracle.agg_fwd(indptr, indices, X.detach().double().cpu().numpy(), "max")
    assert np.array_equal(out.detach().double().cpu().numpy(), ro)
    compare(X.grad, oracle.agg_bwd(ra, g.double().cpu().numpy()), "f32", "dX")
    # an attention call on an aggregation plan, and the reverse, are refused
    with pytest.raises(sga.SgaError):
        sga.gt_attn_fwd(plan, X.detach(), X.detach(), X.detach())
    gt_plan = sga.Plan(ip, ix, 2, 64, torch.float32)
    with pytest.raises(sga.SgaError):
        sga.agg_minmax_fwd(gt_plan, X.detach())
