"""The autograd layers on the GPU: GTAttention and GATv2Attention against the
direct calls, bit for bit.  Collected after the parity files, so that a
failure here cannot stop them in a run that halts at the first failure."""
import pytest
import torch

import sparse_graph_attention_csr_gb300 as sga

from test_gpu_binding_checks import graph

pytestmark = pytest.mark.gpu


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
