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


def test_autograd_layers_match_the_direct_calls():
    """GTAttention and GATv2Attention return the direct calls' outputs and
    gradients bit for bit: the kernels are deterministic (no atomics in any
    sum, split rows merged in chunk order), so the autograd layers add nothing
    but the routing of saved tensors and gradients."""
    ip, ix = graph(seed=7)
    N, H, D, F = ip.numel() - 1, 2, 64, 128
    g = torch.Generator().manual_seed(3)
    r = lambda *s: torch.randn(*s, generator=g)
    Q, K, V, dO = (r(N, H, D).to(torch.bfloat16).cuda() for _ in range(4))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16)
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    q, k, v = (t.clone().requires_grad_() for t in (Q, K, V))
    o = sga.GTAttention.apply(q, k, v, plan)
    o.backward(dO)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), out)
    for got, ref in ((q.grad, dQ), (k.grad, dK), (v.grad, dV)):
        assert torch.equal(got, ref)
    assert plan.device_error() == 0

    plan2 = sga.Plan(ip, ix, H, D, torch.bfloat16, F=F)
    X = r(N, F).to(torch.bfloat16).cuda()
    W_l, W_r = ((r(F, H * D) * 0.05).to(torch.bfloat16).cuda() for _ in range(2))
    a = (r(H, D) * 0.1).to(torch.bfloat16).cuda()
    FL, FR, out2, lse2 = sga.gatv2_fwd(plan2, X, W_l, W_r, a, 0.2)
    grads = sga.gatv2_bwd(plan2, X, W_l, W_r, a, FL, FR, out2, lse2, dO, 0.2)
    ins = [t.clone().requires_grad_() for t in (X, W_l, W_r, a)]
    o2 = sga.GATv2Attention.apply(*ins, plan2, 0.2)
    o2.backward(dO)
    torch.cuda.synchronize()
    assert torch.equal(o2.detach(), out2)
    for t, ref in zip(ins, grads):
        assert torch.equal(t.grad, ref)
    assert plan2.device_error() == 0
