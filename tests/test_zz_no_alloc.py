"""gt_attn_fwd_noalloc: the Graph Transformer forward for callers that must
not allocate device memory (an engine whose memory is reserved up front, a
plugin whose host runtime owns the device memory, a loop that cannot absorb
cudaMalloc's synchronisation).  Its scratch is a fixed static device array,
so the checks here are: the same output as gt_attn_fwd within the tests'
tolerance and against the fp64 oracle, on two calls in a row (the second
call finds the first call's data in the shared array); a clear rejection of
inputs beyond either of the array's limits (split rows, chunk partials),
each followed by a valid call; the Python wrapper's shape checks; and the
range-check word read back.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def valid_call_after(seed=3):
    """A valid call after a rejected one: the shared array still serves."""
    indptr2, indices2 = graph_with_hubs(seed, 2000, 5, [(0, 1500)])
    ip2, ix2 = dev(torch.from_numpy(indptr2)), dev(torch.from_numpy(indices2))
    Q2, K2, V2 = inputs(9, 2000, 2, 64, "bf16")
    out2 = torch.empty_like(Q2)
    lse2 = torch.empty(2000, 2, device="cuda")
    assert call_noalloc(ip2, ix2, Q2, K2, V2, out2, lse2) == sga.SGA_OK
    ref = sga.gt_attn_fwd(sga.Plan(ip2, ix2, 2, 64, torch.bfloat16), Q2, K2, V2)
    compare(out2, ref[0].double().cpu().numpy(), "bf16", "out")
    compare(lse2, ref[1].double().cpu().numpy(), "bf16", "lse")


@pytest.mark.parametrize("dtype,H,D", [("bf16", 4, 64), ("f32", 2, 32)])
def test_matches_planned_forward_and_oracle_on_two_calls_in_a_row(dtype, H, D):
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
        ro, rl = oracle.gt_fwd(indptr, indices, *(t.double().cpu().numpy() for t in (Q, K, V)))
        compare(out, ro, dtype, "out vs oracle")
        compare(lse, rl, dtype, "lse vs oracle")
        assert sga.noalloc_device_error() == 0


def test_rejects_more_split_rows_than_the_array_holds():
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
    valid_call_after()


def test_rejects_more_chunk_partials_than_the_array_holds():
    """Few split rows, but their chunks need more partial space than the array
    has: H = 8, D = 128 leaves room for 24 MiB / ((1024 + 16) * 4 B) = 6049
    chunks; 100 rows of degree 60 * 1024 + 1 need 61 chunks each (6100)."""
    H, D = 8, 128
    cap = (24 << 20) // ((H * D + 2 * H) * 4)
    assert cap == 6049
    N, deg = 100, 60 * 1024 + 1
    assert N * ((deg + 1023) // 1024) > cap and N <= 4096
    indptr = (np.arange(N + 1, dtype=np.int64) * deg).astype(np.int32)
    indices = (np.arange(N * deg, dtype=np.int64) % N).astype(np.int32)
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    Q = torch.zeros(N, H, D, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(Q)
    lse = torch.empty(N, H, device="cuda")
    assert call_noalloc(ip, ix, Q, Q, Q, out, lse) == sga.SGA_ELIMIT
    # one chunk fewer per row fits (60 chunks x 100 rows = 6000 <= 6049)
    deg2 = 60 * 1024
    indptr2 = (np.arange(N + 1, dtype=np.int64) * deg2).astype(np.int32)
    indices2 = (np.arange(N * deg2, dtype=np.int64) % N).astype(np.int32)
    ip2, ix2 = dev(torch.from_numpy(indptr2)), dev(torch.from_numpy(indices2))
    g = torch.Generator().manual_seed(5)
    Q2, K2, V2 = ((torch.randn(N, H, D, generator=g) * D ** -0.5).to(torch.bfloat16).cuda()
                  for _ in range(3))
    assert call_noalloc(ip2, ix2, Q2, K2, V2, out, lse) == sga.SGA_OK
    rows = np.array([0, 37, 99])
    ro, rl = oracle.gt_fwd(indptr2, indices2, *(t.double().cpu().numpy() for t in (Q2, K2, V2)),
                           rows=rows)
    r = torch.from_numpy(rows).cuda()
    compare(out[r], ro, "bf16", "out")
    compare(lse[r], rl, "bf16", "lse")
    valid_call_after(4)


def test_python_wrapper_and_its_shape_checks():
    indptr, indices = graph_with_hubs(6, 1500, 5, [(3, 1200)])
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    N = len(indptr) - 1
    Q, K, V = inputs(7, N, 4, 32, "bf16")
    out, lse = sga.gt_attn_fwd_noalloc(ip, ix, Q, K, V)
    ro, rl = oracle.gt_fwd(indptr, indices, *(t.double().cpu().numpy() for t in (Q, K, V)))
    compare(out, ro, "bf16", "out")
    compare(lse, rl, "bf16", "lse")
    # caller-owned outputs are filled in place
    o2, l2 = torch.empty_like(Q), torch.empty(N, 4, device="cuda")
    r2 = sga.gt_attn_fwd_noalloc(ip, ix, Q, K, V, out=o2, lse=l2)
    assert r2[0] is o2 and r2[1] is l2 and torch.equal(o2, out) and torch.equal(l2, lse)
    # mismatched shapes never reach the library
    with pytest.raises(ValueError):   # Q has more rows than the graph
        sga.gt_attn_fwd_noalloc(ip, ix, torch.cat([Q, Q[:1]]), torch.cat([K, K[:1]]),
                                torch.cat([V, V[:1]]))
    with pytest.raises(ValueError):   # K smaller than Q
        sga.gt_attn_fwd_noalloc(ip, ix, Q, K[:-1], V)
    with pytest.raises(ValueError):   # out of the wrong shape
        sga.gt_attn_fwd_noalloc(ip, ix, Q, K, V, out=torch.empty_like(Q[:, :2]))
    with pytest.raises(ValueError):   # lse of the wrong shape
        sga.gt_attn_fwd_noalloc(ip, ix, Q, K, V, lse=torch.empty(N, 3, device="cuda"))
    with pytest.raises(TypeError):    # lse of the wrong dtype
        sga.gt_attn_fwd_noalloc(ip, ix, Q, K, V, lse=torch.empty(N, 4, device="cuda",
                                                                    dtype=torch.bfloat16))
    with pytest.raises(TypeError):    # V of another dtype
        sga.gt_attn_fwd_noalloc(ip, ix, Q, K, V.float())
    assert sga.noalloc_device_error() == 0
