"""gt_attn_fwd_noalloc: the Graph Transformer forward for callers that must
not allocate device memory (an engine whose memory is reserved up front, a
plugin whose host runtime owns the device memory, a loop that cannot absorb
cudaMalloc's synchronisation).  Its scratch is a fixed static device array,
so the checks here are: same output as gt_attn_fwd within the tests'
tolerance, on two calls in a row (the second call finds the first call's data
in the shared array), and a clear rejection of inputs beyond the array's
limits.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_graph_attention_csr_gb300 as sga

from helpers import TORCH_DT, compare, dev

pytestmark = pytest.mark.gpu


def graph_with_hubs(seed, N, mean_deg, hubs):
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(N):
        r = set(rng.integers(0, N, rng.poisson(mean_deg)).tolist()) | {i}
        rows.append(sorted(r))
    for h, d in hubs:
        rows[h] = sorted(set(rng.integers(0, N, d).tolist()) | {h})
    indptr = np.zeros(N + 1, np.int32)
    indptr[1:] = np.cumsum([len(r) for r in rows])
    return indptr, np.array([j for r in rows for j in r], np.int32)


def inputs(seed, N, H, D, dtype):
    g = torch.Generator().manual_seed(seed)
    std = 1.0 if dtype == "f32" else D ** -0.5
    return [(torch.randn(N, H, D, generator=g) * std).to(TORCH_DT[dtype]).cuda() for _ in range(3)]


def call_noalloc(ip, ix, Q, K, V, out, lse):
    """Straight through the C ABI (ctypes), with caller-owned outputs."""
    lib = sga.load_library()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    N, H, D = Q.shape
    return lib.gt_attn_fwd_noalloc(p(ip), p(ix), p(Q), p(K), p(V), N, ix.numel(), H, D,
                                   sga.SGA_F32 if Q.dtype == torch.float32 else sga.SGA_BF16,
                                   p(out), p(lse),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,H,D", [("bf16", 4, 64), ("f32", 2, 32)])
def test_matches_planned_forward_on_two_calls_in_a_row(dtype, H, D):
    cases = [
        graph_with_hubs(1, 5000, 6, [(10, 3500), (2000, 1800), (4999, 1100)]),   # 3 split rows
        graph_with_hubs(2, 3000, 4, [(7, 1300)]),                                # 1 split row
    ]
    for seed, (indptr, indices) in enumerate(cases):
        ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
        N = len(indptr) - 1
        Q, K, V = inputs(seed, N, H, D, dtype)
        plan = sga.Plan(ip, ix, H, D, TORCH_DT[dtype])
        ref_out, ref_lse = sga.gt_attn_fwd(plan, Q, K, V)
        out = torch.full_like(Q, float("nan"))
        lse = torch.full((N, H), float("nan"), device="cuda")
        assert call_noalloc(ip, ix, Q, K, V, out, lse) == sga.SGA_OK
        torch.cuda.synchronize()
        compare(out, ref_out.double().cpu().numpy(), dtype, "out")
        compare(lse, ref_lse.double().cpu().numpy(), dtype, "lse")


def test_rejects_inputs_beyond_the_static_limits():
    # 4097 rows of degree 1025: one split row more than the array holds
    n_split, deg = 4097, 1025
    N = n_split
    indptr = (np.arange(N + 1, dtype=np.int64) * deg).astype(np.int32)
    indices = np.tile(np.arange(deg, dtype=np.int32), N)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    Q = torch.zeros(N, 1, 32, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(Q)
    lse = torch.empty(N, 1, device="cuda")
    assert call_noalloc(ip, ix, Q, Q, Q, out, lse) == sga.SGA_ELIMIT
    assert sga.load_library().sga_status_string(sga.SGA_ELIMIT).decode().startswith("input exceeds")
    # an invalid CSR is rejected as well, and a valid call afterwards still works
    bad = ix.clone()
    bad[5] = N + 3
    assert call_noalloc(ip, bad, Q, Q, Q, out, lse) == sga.SGA_EINVAL
    indptr2, indices2 = graph_with_hubs(3, 2000, 5, [(0, 1500)])
    ip2, ix2 = dev(torch.from_numpy(indptr2)), dev(torch.from_numpy(indices2))
    Q2, K2, V2 = inputs(9, 2000, 2, 64, "bf16")
    out2 = torch.empty_like(Q2)
    lse2 = torch.empty(2000, 2, device="cuda")
    assert call_noalloc(ip2, ix2, Q2, K2, V2, out2, lse2) == sga.SGA_OK
    ref = sga.gt_attn_fwd(sga.Plan(ip2, ix2, 2, 64, torch.bfloat16), Q2, K2, V2)
    compare(out2, ref[0].double().cpu().numpy(), "bf16", "out")
