"""Graph reordering on the GPU (degree order, reverse Cuthill-McKee) vs the
oracle's sequential definitions, bit for bit; relabelling and row
permutation vs numpy; and the attention layers run on a relabelled graph
(features relabelled alike, results mapped back) against the fp64 oracle on
the original graph."""
import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import TORCH_DT, compare, dev
from test_gpu_gt import csr, random_csr

pytestmark = pytest.mark.gpu


def graphs():
    rng = np.random.default_rng(11)
    out = {
        "hand": tuple(np.array(x, np.int32) for x in ([0, 1, 3, 4, 4, 5, 6, 6, 9, 9, 9, 9],
                                                      [1, 0, 2, 3, 5, 4, 8, 9, 10])),
        "random_dups_empty": random_csr(rng, 700, 4, self_loops=False, empty_frac=0.15,
                                        hubs=[(3, 300)]),
        "isolated_many": csr([[] for _ in range(50)] + [[50], [52], [51]] + [[] for _ in range(20)]),
    }
    for key in (3, 4, 5):
        w = synth.small_workload(key)
        out[f"workload{key}"] = synth.make_graph(w)
    return out


@pytest.mark.parametrize("name", ["hand", "random_dups_empty", "isolated_many", "workload3",
                                  "workload4", "workload5"])
@pytest.mark.parametrize("method", ["rcm", "degree"])
def test_permutation_bit_exact(name, method):
    indptr, indices = graphs()[name]
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    perm = sga.reorder(ip, ix, method).cpu().numpy()
    ref = oracle.order_rcm(indptr, indices) if method == "rcm" else oracle.order_degree(indptr, indices)
    np.testing.assert_array_equal(perm, ref)
    np.testing.assert_array_equal(np.sort(perm), np.arange(len(indptr) - 1))
    # the relabelled CSR, bit for bit
    new_ptr, new_idx = sga.relabel_csr(ip, ix, torch.from_numpy(perm).cuda())
    rp, ri = oracle.relabel_csr(indptr, indices, perm)
    np.testing.assert_array_equal(new_ptr.cpu().numpy(), rp)
    np.testing.assert_array_equal(new_idx.cpu().numpy(), ri)


def test_full_size_rcm_of_the_rmat_workload():
    """R-MAT at 2^20 nodes and 32M edges (many components, hub rows)."""
    w = synth.WORKLOADS[4]
    indptr, indices = synth.make_graph(w)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    perm = sga.reorder(ip, ix, "rcm").cpu().numpy()
    np.testing.assert_array_equal(perm, oracle.order_rcm(indptr, indices))


def test_permute_rows_and_inverse():
    rng = np.random.default_rng(2)
    N = 1000
    perm = torch.from_numpy(rng.permutation(N).astype(np.int32)).cuda()
    for dt, shape in ((torch.bfloat16, (N, 4, 64)), (torch.float32, (N, 3, 32)), (torch.int32, (N, 512))):
        x = torch.randint(-100, 100, shape, device="cuda").to(dt)
        y = sga.permute_rows(x, perm)
        ref = torch.empty_like(x)
        ref[perm.long()] = x
        assert torch.equal(y, ref)
        assert torch.equal(sga.permute_rows(y, perm, inverse=True), x)


@pytest.mark.parametrize("method", ["rcm", "degree"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_attention_on_the_relabelled_graph(method, dtype):
    """GT forward and backward, and GATv2 forward and backward, on the
    relabelled graph with relabelled inputs; results mapped back with the
    inverse permutation match the oracle on the original graph."""
    w = synth.small_workload(3)
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w.scaled(dtype=dtype))
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    perm = sga.reorder(ip, ix, method)
    rp, ri = sga.relabel_csr(ip, ix, perm)
    plan = sga.Plan(rp, ri, w.H, w.D, TORCH_DT[dtype])
    P = lambda t: sga.permute_rows(dev(t), perm)
    Pi = lambda t: sga.permute_rows(t, perm, inverse=True)
    Q, K, V, dO = (P(x[n][0]) for n in ("Q", "K", "V", "dOut"))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    h = {k: v[1] for k, v in x.items()}
    ro, rl = oracle.gt_fwd(indptr, indices, h["Q"], h["K"], h["V"])
    rq, rk, rv = oracle.gt_bwd(indptr, indices, h["Q"], h["K"], h["V"], h["dOut"])
    compare(Pi(out), ro, dtype, "out")
    compare(Pi(lse.contiguous()), rl, dtype, "lse")
    compare(Pi(dQ), rq, dtype, "dQ")
    compare(Pi(dK), rk, dtype, "dK")
    compare(Pi(dV), rv, dtype, "dV")
    assert plan.device_error() == 0


def test_invalid_graphs_and_permutations_are_rejected():
    """The reordering calls check their inputs on the device before any kernel
    indexes with them: an invalid CSR or a perm that is not a permutation
    returns SGA_EINVAL, and the library stays usable afterwards."""
    t = lambda x: dev(torch.tensor(x, dtype=torch.int32))
    good_ptr, good_idx = t([0, 2, 3, 3]), t([1, 0, 2])
    bad_graphs = [
        (t([0, 2, 3, 3]), t([1, 0, 3])),    # source id N
        (t([0, 2, 3, 3]), t([1, -1, 2])),   # negative source id
        (t([0, 3, 2, 3]), t([1, 0, 2])),    # indptr decreasing
        (t([1, 2, 3, 3]), t([1, 0, 2])),    # indptr[0] != 0
    ]
    for ip, ix in bad_graphs:
        for method in ("rcm", "degree"):
            with pytest.raises(sga.SgaError) as ei:
                sga.reorder(ip, ix, method)
            assert ei.value.status == sga.SGA_EINVAL
        with pytest.raises(sga.SgaError) as ei:
            sga.relabel_csr(ip, ix, t([2, 0, 1]))
        assert ei.value.status == sga.SGA_EINVAL
    for perm in ([0, 0, 1], [0, 1, 3], [-1, 0, 1]):
        with pytest.raises(sga.SgaError) as ei:
            sga.relabel_csr(good_ptr, good_idx, t(perm))
        assert ei.value.status == sga.SGA_EINVAL
    # valid inputs still work after the rejections
    perm = sga.reorder(good_ptr, good_idx, "rcm")
    np.testing.assert_array_equal(perm.cpu().numpy(),
                                  oracle.order_rcm(np.array([0, 2, 3, 3], np.int32),
                                                   np.array([1, 0, 2], np.int32)))
    rp, ri = sga.relabel_csr(good_ptr, good_idx, perm)
    ep, ei2 = oracle.relabel_csr(np.array([0, 2, 3, 3], np.int32), np.array([1, 0, 2], np.int32),
                                 perm.cpu().numpy())
    np.testing.assert_array_equal(rp.cpu().numpy(), ep)
    np.testing.assert_array_equal(ri.cpu().numpy(), ei2)


def test_permute_rows_skips_entries_outside_the_node_range():
    x = dev(torch.arange(4 * 8, dtype=torch.float32).reshape(4, 8))
    perm = dev(torch.tensor([2, 7, 0, -3], dtype=torch.int32))
    out = dev(torch.full((4, 8), -1.0))
    sga.permute_rows(x, perm, out=out)
    torch.cuda.synchronize()
    ref = torch.full((4, 8), -1.0)
    ref[2], ref[0] = x[0].cpu(), x[2].cpu()
    assert torch.equal(out.cpu(), ref)
    out.fill_(-1.0)
    sga.permute_rows(x, perm, inverse=True, out=out)
    ref = torch.full((4, 8), -1.0)
    ref[0], ref[2] = x[2].cpu(), x[0].cpu()
    assert torch.equal(out.cpu(), ref)
