"""Checks of the Python binding that run before any device call (CPU only)."""
import pytest
import torch

import sparse_graph_attention_csr_gb300 as sga


def test_plan_refuses_dtypes_the_layers_do_not_compute_in():
    """Only float32 and bfloat16 layers exist; any other dtype is refused before
    the plan is built (float16 tensors must not be read as bfloat16)."""
    ip, ix = torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)
    for dt in (torch.float16, torch.float64, torch.int32):
        with pytest.raises(TypeError):
            sga.Plan(ip, ix, 1, 32, dt)


def test_host_tensors_are_refused():
    ip, ix = torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sga.Plan(ip, ix, 1, 32, torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sga.gt_attn_fwd_noalloc(ip, ix, *(torch.zeros(1, 1, 32) for _ in range(3)))
    with pytest.raises(ValueError, match="CUDA tensor"):
        sga.reorder(ip, ix)


# ---------------------------------------------------------------------------
# autograd plumbing of the layer classes, with the library calls replaced by
# dense torch stand-ins on the CPU (the kernels themselves are compared with
# the oracle in the GPU tests): each class must route its saved tensors and
# gradients to the right calls and return one gradient per input


class _FakePlan:
    pass


def _dense(indptr, indices, N):
    m = torch.zeros(N, N, dtype=torch.bool)
    for i in range(N):
        m[i, indices[indptr[i]:indptr[i + 1]]] = True
    return m


def _gt_ref(Q, K, V, mask):
    s = torch.einsum("ihd,jhd->hij", Q, K) / Q.shape[-1] ** 0.5
    s = s.masked_fill(~mask[None], float("-inf"))
    lse = torch.logsumexp(s, -1)
    return torch.einsum("hij,jhd->ihd", torch.exp(s - lse[..., None]), V), lse.T.contiguous()


def test_gt_attention_autograd_routes_gradients(monkeypatch):
    torch.manual_seed(0)
    N, H, D = 6, 2, 4
    indptr = [0, 2, 3, 5, 6, 8, 9]
    indices = [0, 1, 1, 2, 3, 3, 4, 5, 0]
    mask = _dense(indptr, indices, N)

    def fwd(plan, Q, K, V):
        return _gt_ref(Q, K, V, mask)

    def bwd(plan, Q, K, V, out, lse, dOut):
        with torch.enable_grad():   # (a Function's backward runs with grad mode off)
            q, k, v = (t.detach().clone().requires_grad_() for t in (Q, K, V))
            o, _ = _gt_ref(q, k, v, mask)
            return torch.autograd.grad(o, (q, k, v), dOut)

    monkeypatch.setattr(sga, "gt_attn_fwd", fwd)
    monkeypatch.setattr(sga, "gt_attn_bwd", bwd)
    Q, K, V = (torch.randn(N, H, D, dtype=torch.float64, requires_grad=True) for _ in range(3))
    dO = torch.randn(N, H, D, dtype=torch.float64)
    out = sga.GTAttention.apply(Q, K, V, _FakePlan())
    out.backward(dO)
    Q2, K2, V2 = (t.detach().clone().requires_grad_() for t in (Q, K, V))
    ref, _ = _gt_ref(Q2, K2, V2, mask)
    ref.backward(dO)
    torch.testing.assert_close(out, ref)
    for a, b in ((Q, Q2), (K, K2), (V, V2)):
        torch.testing.assert_close(a.grad, b.grad)


def test_gatv2_attention_autograd_routes_gradients(monkeypatch):
    torch.manual_seed(1)
    N, F, H, D = 5, 3, 2, 4
    indptr = [0, 2, 3, 5, 6, 7]
    indices = [0, 1, 2, 0, 3, 4, 2]
    mask = _dense(indptr, indices, N)

    def layer(X, Wl, Wr, a, slope):
        FL, FR = (X @ Wl).reshape(N, H, D), (X @ Wr).reshape(N, H, D)
        z = FL[:, None] + FR[None]
        e = (torch.nn.functional.leaky_relu(z, slope) * a).sum(-1).permute(2, 0, 1)
        e = e.masked_fill(~mask[None], float("-inf"))
        lse = torch.logsumexp(e, -1)
        out = torch.einsum("hij,jhd->ihd", torch.exp(e - lse[..., None]), FR)
        return FL, FR, out, lse.T.contiguous()

    def fwd(plan, X, Wl, Wr, a, slope):
        return layer(X, Wl, Wr, a, slope)

    def bwd(plan, X, Wl, Wr, a, FL, FR, out, lse, dOut, slope):
        with torch.enable_grad():
            ins = [t.detach().clone().requires_grad_() for t in (X, Wl, Wr, a)]
            return torch.autograd.grad(layer(*ins, slope)[2], ins, dOut)

    monkeypatch.setattr(sga, "gatv2_fwd", fwd)
    monkeypatch.setattr(sga, "gatv2_bwd", bwd)
    X = torch.randn(N, F, dtype=torch.float64, requires_grad=True)
    Wl, Wr = (torch.randn(F, H * D, dtype=torch.float64, requires_grad=True) for _ in range(2))
    a = torch.randn(H, D, dtype=torch.float64, requires_grad=True)
    dO = torch.randn(N, H, D, dtype=torch.float64)
    out = sga.GATv2Attention.apply(X, Wl, Wr, a, _FakePlan(), 0.2)
    out.backward(dO)
    ins2 = [t.detach().clone().requires_grad_() for t in (X, Wl, Wr, a)]
    ref = layer(*ins2, 0.2)[2]
    ref.backward(dO)
    torch.testing.assert_close(out, ref)
    for t, t2 in zip((X, Wl, Wr, a), ins2):
        torch.testing.assert_close(t.grad, t2.grad)


def test_gt_bias_attention_autograd_routes_gradients(monkeypatch):
    torch.manual_seed(2)
    N, H, D = 5, 2, 4
    indptr = [0, 2, 3, 5, 6, 7]
    indices = [0, 1, 1, 2, 3, 4, 0]
    E = len(indices)
    rows = torch.repeat_interleave(torch.arange(N), torch.tensor(indptr).diff())
    cols = torch.tensor(indices)

    def layer(Q, K, V, B):
        s = torch.full((H, N, N), float("-inf"), dtype=Q.dtype)
        s[:, rows, cols] = (Q[rows] * K[cols]).sum(-1).T / D ** 0.5 + B.T
        lse = torch.logsumexp(s, -1)
        return torch.einsum("hij,jhd->ihd", torch.exp(s - lse[..., None]), V), lse.T.contiguous()

    def fwd(plan, Q, K, V, B):
        return layer(Q, K, V, B)

    def bwd(plan, Q, K, V, B, out, lse, dOut):
        with torch.enable_grad():
            ins = [t.detach().clone().requires_grad_() for t in (Q, K, V, B)]
            return torch.autograd.grad(layer(*ins)[0], ins, dOut)

    monkeypatch.setattr(sga, "gt_attn_bias_fwd", fwd)
    monkeypatch.setattr(sga, "gt_attn_bias_bwd", bwd)
    Q, K, V = (torch.randn(N, H, D, dtype=torch.float64, requires_grad=True) for _ in range(3))
    B = torch.randn(E, H, dtype=torch.float64, requires_grad=True)
    dO = torch.randn(N, H, D, dtype=torch.float64)
    out = sga.GTBiasAttention.apply(Q, K, V, B, _FakePlan())
    out.backward(dO)
    ins2 = [t.detach().clone().requires_grad_() for t in (Q, K, V, B)]
    ref = layer(*ins2)[0]
    ref.backward(dO)
    torch.testing.assert_close(out, ref)
    for t, t2 in zip((Q, K, V, B), ins2):
        torch.testing.assert_close(t.grad, t2.grad)
    assert B.grad.abs().sum() > 0
