"""The alternative thread mappings of the Graph Transformer forward
(feature-parallel; edge-parallel scores with feature-parallel aggregation)
vs the fp64 oracle, through the C ABI: every lane layout, split rows, rows
whose scores climb past the online softmax's rescale point, and the edge
cases.  The backward is shared with the default schedule."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga
from sparse_graph_attention_csr_gb300 import synth

from helpers import TORCH_DT, compare, dev
from test_gpu_gt import csr, random_csr, values
from test_gpu_rescale import LEVELS, rescale_rows, rounded, staircase_graph, staircase_qk

pytestmark = pytest.mark.gpu

SCHEDULES = [sga.SGA_SCHED_FEATURE, sga.SGA_SCHED_BILEVEL]


def run_fwd(indptr, indices, q, k, v, H, D, dtype, schedule, split=0, chunk=0):
    """q, k, v: (tensor in dtype, float64 copy)."""
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, TORCH_DT[dtype], split_threshold=split, chunk_len=chunk,
                    schedule=schedule)
    out, lse = sga.gt_attn_fwd(plan, dev(q[0]), dev(k[0]), dev(v[0]))
    ro, rl = oracle.gt_fwd(indptr, indices, q[1], k[1], v[1])
    compare(out, ro, dtype, "out")
    compare(lse, rl, dtype, "lse")
    torch.cuda.synchronize()
    assert plan.device_error() == 0


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H,D", [(1, 32), (2, 32), (4, 32), (1, 64), (2, 64), (4, 64), (1, 128),
                                 (4, 128), (8, 128), (3, 64), (5, 32), (32, 32)])
def test_every_shape_with_split_rows(schedule, dtype, H, D):
    rng = np.random.default_rng(H * 1000 + D + 7 * schedule)
    indptr, indices = random_csr(rng, 300, 6, hubs=[(7, 250), (299, 120), (150, 70)])
    std = 1 / math.sqrt(D) if dtype == "bf16" else 1.0
    q, k, v = (values(rng, 300, H, D, dtype, std) for _ in range(3))
    run_fwd(indptr, indices, q, k, v, H, D, dtype, schedule, split=40, chunk=16)
    run_fwd(indptr, indices, q, k, v, H, D, dtype, schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rising_scores(schedule, dtype):
    rng = np.random.default_rng(90 + schedule)
    N, H, D = 600, 4, 64
    t, Qf, Kf = staircase_qk(rng, N, H, D, LEVELS[dtype], neg_frac=0.15)
    indptr, indices = staircase_graph(rng, N, 40, t, hubs=[(5, 400), (321, 150)])
    V = rng.standard_normal((N, H, D))
    q, k, v = rounded(Qf, dtype), rounded(Kf, dtype), rounded(V, dtype)
    assert rescale_rows(indptr, indices, q[1], k[1]) > 0.4 * N
    run_fwd(indptr, indices, q, k, v, H, D, dtype, schedule, split=48, chunk=16)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_edge_cases(schedule):
    rows = [[], [3], [0, 0, 2], [], [1, 2, 3, 4], [4], [], [0, 1, 1, 1, 6]]
    indptr, indices = csr(rows)
    rng = np.random.default_rng(3)
    for dtype in ("f32", "bf16"):
        q, k, v = (values(rng, 8, 2, 32, dtype) for _ in range(3))
        run_fwd(indptr, indices, q, k, v, 2, 32, dtype, schedule, split=2, chunk=1)
        run_fwd(indptr, indices, q, k, v, 2, 32, dtype, schedule)
    z = np.zeros((5, 4, 64))
    zt = (torch.zeros(5, 4, 64, dtype=torch.bfloat16), z)
    run_fwd(np.zeros(6, np.int32), np.zeros(0, np.int32), zt, zt, zt, 4, 64, "bf16", schedule)


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("key", [3, 4])
def test_small_workloads(schedule, key):
    w = synth.small_workload(key)
    indptr, indices = synth.make_graph(w)
    x = synth.gt_inputs(w)
    run_fwd(indptr, indices, x["Q"], x["K"], x["V"], w.H, w.D, w.dtype, schedule)


def test_bad_schedule_is_refused():
    indptr, indices = csr([[0, 1], [1]])
    with pytest.raises(sga.SgaError):
        sga.Plan(dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices)), 1, 32,
                 torch.float32, schedule=7)
