"""Graph Transformer with a per-edge, per-head score bias on the GPU vs the
fp64 oracle, through the C ABI: forward (out, lse), backward (dQ, dK, dV and
the bias gradient dB = dS of every edge), over every lane layout, split rows,
duplicate edges and empty rows; a bias staircase that makes scores climb far
past the online softmax's rescale point; the transposed-edge map of the
plan, bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import TORCH_DT, compare, dev
from test_gpu_gt import csr, random_csr, values

pytestmark = pytest.mark.gpu


def run_bias(indptr, indices, H, D, dtype, B, seed=0, std=1.0, split=0, chunk=0):
    rng = np.random.default_rng(seed)
    N = len(indptr) - 1
    (q, qf), (k, kf), (v, vf), (do, dof) = (values(rng, N, H, D, dtype, std) for _ in range(4))
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, TORCH_DT[dtype], split_threshold=split, chunk_len=chunk,
                    edge_bias=True)
    Bt = torch.from_numpy(np.ascontiguousarray(B, dtype=np.float32)).cuda()
    bf = Bt.double().cpu().numpy()
    Q, K, V, dO = dev(q), dev(k), dev(v), dev(do)
    out, lse = sga.gt_attn_bias_fwd(plan, Q, K, V, Bt)
    ro, rl = oracle.gt_bias_fwd(indptr, indices, qf, kf, vf, bf)
    compare(out, ro, dtype, "out")
    compare(lse, rl, dtype, "lse")
    dQ, dK, dV, dB = sga.gt_attn_bias_bwd(plan, Q, K, V, Bt, out, lse, dO)
    rq, rk, rv, rb = oracle.gt_bias_bwd(indptr, indices, qf, kf, vf, bf, dof)
    compare(dQ, rq, dtype, "dQ")
    compare(dK, rk, dtype, "dK")
    compare(dV, rv, dtype, "dV")
    # dB is fp32 for both dtypes; bf16 inputs carry the bf16 bound
    compare(dB, rb, dtype, "dB")
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    return plan


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H,D", [(1, 32), (2, 32), (4, 32), (1, 64), (4, 64), (3, 64), (1, 128),
                                 (4, 128), (8, 128), (5, 32)])
def test_every_lane_layout_with_split_rows(dtype, H, D):
    rng = np.random.default_rng(H * 100 + D)
    indptr, indices = random_csr(rng, 300, 6, hubs=[(7, 250), (299, 120)])
    B = rng.standard_normal((len(indices), H))
    std = 1 / math.sqrt(D) if dtype == "bf16" else 1.0
    run_bias(indptr, indices, H, D, dtype, B, seed=H + D, std=std, split=40, chunk=16)
    run_bias(indptr, indices, H, D, dtype, B, seed=H + D, std=std)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_duplicates_empty_rows_and_edge_map(dtype):
    rows = [[], [3], [0, 0, 2], [], [1, 2, 3, 4], [4], [], [0, 1, 1, 1, 6]]
    indptr, indices = csr(rows)
    rng = np.random.default_rng(1)
    B = rng.standard_normal((len(indices), 2))
    plan = run_bias(indptr, indices, 2, 32, dtype, B, split=2, chunk=1)
    run_bias(indptr, indices, 2, 32, dtype, B)
    # the transposed CSR of an edge-bias plan equals a plain plan's
    t_indptr, t_dst = oracle.transpose(indptr, indices)
    np.testing.assert_array_equal(plan.array("t_indptr"), t_indptr)
    np.testing.assert_array_equal(plan.array("t_dst"), t_dst)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bias_staircase_forces_the_rescale(dtype):
    """Bias levels 7 apart climbing along each row (sources in ascending
    level order), hub rows split into chunks of 16: scores exceed the running
    maximum by more than 2^8 repeatedly, chunk maxima lie levels apart."""
    rng = np.random.default_rng(5)
    N, H, D = 500, 4, 64
    lev = rng.integers(0, 3 if dtype == "f32" else 5, N).astype(np.float64)
    rows = []
    for i in range(N):
        r = set(rng.integers(0, N, rng.poisson(24)).tolist()) | {i}
        if i in (4, 250):
            r |= set(rng.integers(0, N, 400).tolist())
        rows.append(sorted(r, key=lambda j: (lev[j], j)))
    indptr, indices = csr(rows)
    dst = np.repeat(np.arange(N), np.diff(indptr))
    # fp32: |bias| <= 7 (its 1e-5 bound), bf16: up to 28
    B = (lev[indices] * 7.0 - (7.0 if dtype == "f32" else 14.0))[:, None] + \
        0.1 * rng.standard_normal((len(indices), H))
    rise = 0
    for i in range(N):
        b = B[indptr[i]:indptr[i + 1], 0]
        if len(b) > 1 and np.any(b[1:] > np.maximum.accumulate(b)[:-1] + 8 * math.log(2)):
            rise += 1
    assert rise > 0.5 * N
    std = 0.5 / math.sqrt(D) if dtype == "bf16" else 0.25
    run_bias(indptr, indices, H, D, dtype, B, seed=3, std=std, split=48, chunk=16)


def test_small_workload_with_bias():
    w = synth.small_workload(4)
    indptr, indices = synth.make_graph(w)
    rng = np.random.default_rng(7)
    B = rng.standard_normal((len(indices), w.H)) * 0.5
    run_bias(indptr, indices, w.H, w.D, "bf16", B, seed=4)


def test_bias_needs_an_edge_bias_plan():
    indptr, indices = csr([[0, 1], [1]])
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, 1, 32, torch.float32)
    Q = torch.randn(2, 1, 32, device="cuda")
    with pytest.raises(sga.SgaError):
        sga.gt_attn_bias_fwd(plan, Q, Q, Q, torch.zeros(3, 1, device="cuda"))
    with pytest.raises(sga.SgaError):   # block-sparse plans do not take a bias
        sga.Plan(ip, ix, 1, 64, torch.bfloat16, tile_min_nnz=4, edge_bias=True)
