"""The Python binding checks every tensor against the plan before a pointer
reaches the library (which sees pointers only): wrong row counts, element
counts, dtypes or devices raise instead of reaching the kernels."""
import numpy as np
import pytest
import torch

import sparse_graph_attention_csr_gb300 as sga

from helpers import dev
from test_gpu_gt import random_csr

pytestmark = pytest.mark.gpu


def graph(N=300, seed=5):
    rng = np.random.default_rng(seed)
    indptr, indices = random_csr(rng, N, 6, hubs=[(3, 200)])
    return dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))


def test_graph_transformer_shapes():
    ip, ix = graph()
    N, H, D = ip.numel() - 1, 2, 64
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16)
    Q = torch.randn(N, H, D, device="cuda").to(torch.bfloat16)
    short = Q[:-1].contiguous()
    for bad in ((short, Q, Q), (Q, short, Q), (Q, Q, short)):
        with pytest.raises(ValueError):
            sga.gt_attn_fwd(plan, *bad)
    with pytest.raises(TypeError):
        sga.gt_attn_fwd(plan, Q.float(), Q, Q)
    with pytest.raises(ValueError):
        sga.gt_attn_fwd(plan, Q, Q, Q, lse=torch.empty(N, H + 1, device="cuda"))
    out, lse = sga.gt_attn_fwd(plan, Q, Q, Q)
    with pytest.raises(ValueError):
        sga.gt_attn_bwd(plan, Q, Q, Q, out, lse[:-1].contiguous(), Q)
    with pytest.raises(ValueError):
        sga.gt_attn_bwd(plan, Q, Q, Q, out, lse, short)
    with pytest.raises(ValueError):
        sga.gt_attn_bwd(plan, Q, Q, Q, out, lse, Q, dQ=short)
    # a [N, H*D] view of the same storage is accepted
    o2, _ = sga.gt_attn_fwd(plan, Q.view(N, H * D), Q, Q)
    assert torch.equal(o2.view(N, H, D), out)
    assert plan.device_error() == 0


def test_gatv2_and_aggregation_shapes():
    ip, ix = graph(seed=6)
    N, H, D, F = ip.numel() - 1, 2, 64, 128
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16, F=F)
    X = torch.randn(N, F, device="cuda").to(torch.bfloat16)
    W = (torch.randn(F, H * D, device="cuda") * 0.05).to(torch.bfloat16)
    a = (torch.randn(H, D, device="cuda") * 0.1).to(torch.bfloat16)
    with pytest.raises(ValueError):
        sga.gatv2_fwd(plan, X[:, :-8].contiguous(), W, W, a)
    with pytest.raises(ValueError):
        sga.gatv2_fwd(plan, X, W[:-1].contiguous(), W, a)
    with pytest.raises(ValueError):
        sga.gatv2_fwd(plan, X, W, W, a[:1].contiguous())
    sga.gatv2_fwd(plan, X, W, W, a)
    aplan = sga.Plan(ip, ix, H, D, torch.bfloat16, layer=sga.SGA_LAYER_MINMAX)
    Y = torch.randn(N, H, D, device="cuda").to(torch.bfloat16)
    with pytest.raises(ValueError):
        sga.agg_minmax_fwd(aplan, Y[:-1].contiguous())
    out, arg, mask = sga.agg_minmax_fwd(aplan, Y)
    with pytest.raises(ValueError):
        sga.agg_minmax_bwd(aplan, mask[:-1].contiguous(), Y)
    with pytest.raises(ValueError):
        sga.agg_minmax_fwd(aplan, Y, arg=torch.empty(N, H, device="cuda", dtype=torch.int32))
    assert aplan.device_error() == 0

