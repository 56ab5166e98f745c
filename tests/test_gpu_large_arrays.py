"""Node arrays above 4 GB: 8.4M nodes x H=4 x D=64 in bf16 make every
gathered array 4.3 GB, past the range of 32-bit byte offsets, so the edge
stream of the Graph Transformer passes takes its 64-bit address path (arrays
below 4 GB take 32-bit offsets).  Forward and backward run on the whole
graph; the oracle checks sampled rows and sources on small subgraphs cut out
around them (a row's output and dQ depend on the row's own edges only; a
source's dK and dV on every row that gathers it)."""
import numpy as np
import pytest
import torch

import oracle
import sparse_graph_attention_csr_gb300 as sga

from helpers import compare, dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

N, H, D = 8_400_000, 4, 64


def graph(rng):
    deg = rng.poisson(2.0, N).astype(np.int64)
    hubs = rng.choice(N, 6, replace=False)
    deg[hubs] = 5000                       # split rows (default threshold 512 here)
    indptr = np.zeros(N + 1, np.int64)
    np.cumsum(deg, out=indptr[1:])
    indices = rng.integers(0, N, int(indptr[-1]), dtype=np.int64).astype(np.int32)
    return indptr.astype(np.int32), indices, hubs


def subgraph(indptr, indices, rows, extra=()):
    """Rows `rows` with their edges, over the nodes they touch and the nodes
    `extra` (relabelled): (sub_indptr, sub_indices, node ids, position of each
    row).  Only the listed rows keep edges."""
    segs = [indices[indptr[i]:indptr[i + 1]] for i in rows]
    nodes, inv = np.unique(np.concatenate([np.asarray(rows, np.int32)] + segs + [np.asarray(extra, np.int32)]),
                           return_inverse=True)
    pos = inv[:len(rows)]
    sub_ptr = np.zeros(len(nodes) + 1, np.int64)
    lens = np.zeros(len(nodes), np.int64)
    lens[pos] = [len(sg) for sg in segs]
    np.cumsum(lens, out=sub_ptr[1:])
    sub_idx = np.empty(int(sub_ptr[-1]), np.int32)
    k = len(rows)
    for r, sg in enumerate(segs):
        n = len(sg)
        sub_idx[sub_ptr[pos[r]]:sub_ptr[pos[r]] + n] = inv[k:k + n]
        k += n
    return sub_ptr.astype(np.int32), sub_idx, nodes, pos


def test_gt_over_4gb_node_arrays():
    rng = np.random.default_rng(21)
    indptr, indices, hubs = graph(rng)
    assert N * H * D * 2 > 1 << 32
    ip, ix = dev(torch.from_numpy(indptr)), dev(torch.from_numpy(indices))
    plan = sga.Plan(ip, ix, H, D, torch.bfloat16)
    gen = torch.Generator(device="cuda").manual_seed(5)
    Q, K, V, dO = (torch.randn(N, H, D, device="cuda", generator=gen, dtype=torch.bfloat16) * (D ** -0.25)
                   for _ in range(4))
    out, lse = sga.gt_attn_fwd(plan, Q, K, V)
    dQ, dK, dV = sga.gt_attn_bwd(plan, Q, K, V, out, lse, dO)
    torch.cuda.synchronize()
    assert plan.device_error() == 0

    def host(t, nodes):
        return t[torch.from_numpy(nodes.astype(np.int64)).cuda()].double().cpu().numpy()

    # destination rows: output, lse and dQ
    rows = np.unique(np.concatenate([rng.integers(0, N, 400), hubs])).astype(np.int32)
    sp, si, nodes, pos = subgraph(indptr, indices, rows)
    q, k, v, g = (host(t, nodes) for t in (Q, K, V, dO))
    ro, rl = oracle.gt_fwd(sp, si, q, k, v, rows=pos)
    r = torch.from_numpy(rows.astype(np.int64)).cuda()
    compare(out[r], ro, "bf16", "out")
    compare(lse[r], rl, "bf16", "lse")
    compare(dQ[r], oracle.gt_bwd_dq_rows(sp, si, q, k, v, g, pos), "bf16", "dQ")

    # sources: dK and dV need every row that gathers them, with all its edges
    srcs = rng.integers(0, N, 60).astype(np.int32)
    is_src = np.zeros(N, bool)
    is_src[srcs] = True
    hit = np.flatnonzero(is_src[indices])
    dst = np.unique(np.searchsorted(indptr, hit, side="right") - 1).astype(np.int32)
    sp, si, nodes, _ = subgraph(indptr, indices, dst, extra=srcs)   # (a source no row gathers: dK = dV = 0)
    q, k, v, g = (host(t, nodes) for t in (Q, K, V, dO))
    spos = np.searchsorted(nodes, srcs)
    assert np.array_equal(nodes[spos], srcs)
    rk, rv = oracle.gt_bwd_dkdv_srcs(sp, si, q, k, v, g, spos)
    sj = torch.from_numpy(srcs.astype(np.int64)).cuda()
    compare(dK[sj], rk, "bf16", "dK")
    compare(dV[sj], rv, "bf16", "dV")
