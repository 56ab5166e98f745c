"""Seeded synthetic inputs: graphs in destination-sorted CSR form and the dense
feature tensors that feed both the CUDA path and the fp64 oracle.

This module holds no attention arithmetic.  It draws random numbers, builds
CSR arrays from edge lists, and rounds drawn values to the storage dtype.
Both sides of every parity check consume the arrays it returns.

Graph conventions (the plainest reading of "CSR sorted by destination"):
row ``i`` of the CSR is destination node ``i``; ``indices[indptr[i]:indptr[i+1]]``
are its source nodes, ascending, without duplicates; every node carries a
self-loop.

Stand-ins.  The pages evaluate on citation-like and power-law graphs
(Open Graph Benchmark is cited; no dataset is available here).  The five
workloads below are synthetic graphs with the stated size, degree law and
structure:

1. Erdos-Renyi directed, N=1024, mean out-degree 8 (GT forward, fp32, H=4, D=32).
2. Chung-Lu power law, N=100k, exponent 2.5, 1.6M draws (GATv2, bf16, H=2, D=64, F=128).
3. Chung-Lu with lognormal weights (median 7) and one hub of weight 10k,
   N=170k, 1.2M undirected draws made symmetric (GT, bf16, H=4, D=128).
4. R-MAT (0.57, 0.19, 0.19, 0.05), scale 20, 2^25 draws (GT, bf16, H=4, D=64).
5. Stochastic block model, 1024 contiguous communities of 256, p_in=0.15,
   4N inter-community draws (GT, bf16, H=4, D=128).
6. Min / max aggregation over workload 3's graph (N=170k, lognormal
   Chung-Lu with a hub), node rows of 512 bf16 features (read as H=4 x D=128),
   the width of the pages' min-aggregation figure.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

# Streams spawned from one SeedSequence per workload.
STREAM_GRAPH, STREAM_A, STREAM_B, STREAM_C, STREAM_ATT, STREAM_DOUT = range(6)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: graph recipe, layer kind and tensor shapes."""
    key: int
    name: str
    layer: str              # "gt", "gatv2", "agg_min" or "agg_max"
    graph: str              # "er" | "chung_lu" | "lognormal_cl" | "rmat" | "sbm"
    N: int
    H: int
    D: int
    dtype: str              # "f32" | "bf16"
    backward: bool
    seed: int
    params: dict = field(default_factory=dict)
    F: int = 0              # GATv2 input feature width
    qkv_std: float = 1.0    # standard deviation of Q, K, V

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (smaller sizes for parity cases)."""
        params = dict(self.params)
        params.update(kw.pop("params", {}))
        return replace(self, params=params, **kw)


WORKLOADS = {
    1: Workload(1, "gt_fwd_er_n1024_h4_d32_f32", "gt", "er", 1024, 4, 32, "f32",
                False, 1, {"mean_deg": 8.0}),
    2: Workload(2, "gatv2_chunglu_n100k_h2_d64_bf16", "gatv2", "chung_lu", 100_000, 2, 64,
                "bf16", True, 2, {"draws": 1_600_000, "gamma": 2.5}, F=128),
    3: Workload(3, "gt_lognormal_n170k_h4_d128_bf16", "gt", "lognormal_cl", 170_000, 4, 128,
                "bf16", True, 3, {"draws": 1_200_000, "median": 7.0, "sigma": 1.15,
                                  "hub_weight": 10_000.0}, qkv_std=1.0 / math.sqrt(128)),
    4: Workload(4, "gt_rmat_s20_h4_d64_bf16", "gt", "rmat", 1 << 20, 4, 64, "bf16", True, 4,
                {"scale": 20, "draws": 1 << 25, "abcd": (0.57, 0.19, 0.19, 0.05)}),
    5: Workload(5, "gt_sbm_n262k_h4_d128_bf16", "gt", "sbm", 262_144, 4, 128, "bf16", True, 5,
                {"block": 256, "p_in": 0.15, "inter_per_node": 4},
                qkv_std=1.0 / math.sqrt(128)),
    6: Workload(6, "agg_min_lognormal_n170k_f512_bf16", "agg_min", "lognormal_cl", 170_000, 4, 128,
                "bf16", True, 6, {"draws": 1_200_000, "median": 7.0, "sigma": 1.15,
                                  "hub_weight": 10_000.0}),
}


def small_workload(key: int) -> Workload:
    """Reduced copies of the five workloads with the same recipe, sized so the
    oracle finishes in seconds while the CUDA path still spans many warps,
    split rows and a ragged tail."""
    w = WORKLOADS[key]
    if key == 1:
        return w
    if key == 2:
        return w.scaled(N=6000, params={"draws": 96_000})
    if key == 3:
        return w.scaled(N=9000, params={"draws": 63_000, "hub_weight": 2500.0})
    if key == 4:
        return w.scaled(N=1 << 14, params={"scale": 14, "draws": 1 << 19})
    if key == 5:
        return w.scaled(N=4096)
    if key == 6:
        return w.scaled(N=9000, params={"draws": 63_000, "hub_weight": 2500.0})
    raise KeyError(key)


# --------------------------------------------------------------------------
# CSR construction
# --------------------------------------------------------------------------

def csr_from_edges(N: int, dst: np.ndarray, src: np.ndarray, self_loops: bool = True):
    """Destination-sorted CSR from an edge list: duplicates dropped, sources
    ascending within a row, a self-loop added to every node when asked."""
    dst = np.asarray(dst, dtype=np.int64)
    src = np.asarray(src, dtype=np.int64)
    if self_loops:
        ar = np.arange(N, dtype=np.int64)
        dst = np.concatenate([dst, ar])
        src = np.concatenate([src, ar])
    keys = dst * N + src
    keys.sort()
    if len(keys):
        keys = keys[np.concatenate(([True], keys[1:] != keys[:-1]))]
    d = keys // N
    s = keys - d * N
    counts = np.bincount(d, minlength=N)
    indptr = np.zeros(N + 1, dtype=np.int64)
    np.cumsum(counts, out=indptr[1:])
    if indptr[-1] >= 2 ** 31:
        raise ValueError("graph too large for int32 CSR")
    return indptr.astype(np.int32), s.astype(np.int32)


def _weighted_endpoints(rng, cdf: np.ndarray, n: int) -> np.ndarray:
    """n node ids drawn with probability proportional to the weights whose
    normalised cumulative sum is ``cdf``."""
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), len(cdf) - 1)


def graph_er(rng, N: int, mean_deg: float):
    """Directed G(N, p): each ordered pair u != v is an edge with p = mean_deg/(N-1)."""
    p = mean_deg / (N - 1)
    if N <= 8192:
        m = rng.random((N, N)) < p
        np.fill_diagonal(m, False)
        dst, src = np.nonzero(m)
    else:
        n = rng.binomial(N * (N - 1), p)
        dst = rng.integers(0, N, n)
        src = rng.integers(0, N - 1, n)
        src = src + (src >= dst)
    return csr_from_edges(N, dst, src)


def graph_chung_lu(rng, N: int, draws: int, gamma: float):
    """Chung-Lu: weights w_i = i^(-1/(gamma-1)); ``draws`` (dst, src) pairs with
    both endpoints proportional to w; self-pairs and duplicates dropped."""
    w = np.arange(1, N + 1, dtype=np.float64) ** (-1.0 / (gamma - 1.0))
    cdf = np.cumsum(w) / w.sum()
    dst = _weighted_endpoints(rng, cdf, draws)
    src = _weighted_endpoints(rng, cdf, draws)
    keep = dst != src
    return csr_from_edges(N, dst[keep], src[keep])


def graph_lognormal_cl(rng, N: int, draws: int, median: float, sigma: float, hub_weight: float):
    """Chung-Lu with lognormal weights (median, sigma) and the largest weight
    replaced by ``hub_weight``; ``draws`` unordered pairs made symmetric."""
    w = rng.lognormal(mean=math.log(median), sigma=sigma, size=N)
    w[np.argmax(w)] = hub_weight
    cdf = np.cumsum(w) / w.sum()
    u = _weighted_endpoints(rng, cdf, draws)
    v = _weighted_endpoints(rng, cdf, draws)
    keep = u != v
    u, v = u[keep], v[keep]
    return csr_from_edges(N, np.concatenate([u, v]), np.concatenate([v, u]))


def graph_rmat(rng, scale: int, draws: int, abcd, chunk: int = 1 << 22):
    """R-MAT: each draw descends ``scale`` quadrant levels with probabilities
    (a, b, c, d); the row bit is the destination, the column bit the source."""
    a, b, c, _ = abcd
    N = 1 << scale
    dsts, srcs = [], []
    left = draws
    while left > 0:
        n = min(chunk, left)
        left -= n
        dst = np.zeros(n, dtype=np.int32)
        src = np.zeros(n, dtype=np.int32)
        for _level in range(scale):
            r = rng.random(n, dtype=np.float32)
            row = r >= (a + b)
            col = ((r >= a) & (r < a + b)) | (r >= a + b + c)
            dst <<= 1
            dst |= row
            src <<= 1
            src |= col
        dsts.append(dst)
        srcs.append(src)
    return csr_from_edges(N, np.concatenate(dsts), np.concatenate(srcs))


def graph_sbm(rng, N: int, block: int, p_in: float, inter_per_node: int, batch: int = 64):
    """Stochastic block model with contiguous communities of ``block`` nodes:
    every intra-community ordered pair u != v with probability p_in, plus
    ``inter_per_node * N`` inter-community pairs (source uniform, destination
    uniform outside the source's community)."""
    nb = N // block
    dsts, srcs = [], []
    for c0 in range(0, nb, batch):
        cb = min(batch, nb - c0)
        m = rng.random((cb, block, block), dtype=np.float32) < p_in
        idx = np.arange(block)
        m[:, idx, idx] = False
        cc, u, v = np.nonzero(m)
        base = (cc + c0).astype(np.int64) * block
        dsts.append(base + u)
        srcs.append(base + v)
    n_inter = inter_per_node * N
    src = rng.integers(0, N, n_inter)
    dst = rng.integers(0, N - block, n_inter)
    start = (src // block) * block
    dst = dst + (dst >= start) * block
    dsts.append(dst)
    srcs.append(src)
    return csr_from_edges(N, np.concatenate(dsts), np.concatenate(srcs))


def make_graph(w: Workload):
    """(indptr, indices) int32 CSR for a workload, deterministic in its seed."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(w.seed).spawn(6)[STREAM_GRAPH]))
    p = w.params
    if w.graph == "er":
        return graph_er(rng, w.N, p["mean_deg"])
    if w.graph == "chung_lu":
        return graph_chung_lu(rng, w.N, p["draws"], p["gamma"])
    if w.graph == "lognormal_cl":
        return graph_lognormal_cl(rng, w.N, p["draws"], p["median"], p["sigma"], p["hub_weight"])
    if w.graph == "rmat":
        return graph_rmat(rng, p["scale"], p["draws"], p["abcd"])
    if w.graph == "sbm":
        return graph_sbm(rng, w.N, p["block"], p["p_in"], p["inter_per_node"])
    raise ValueError(w.graph)


# --------------------------------------------------------------------------
# Dense inputs
# --------------------------------------------------------------------------

def _rng(seed: int, stream: int):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(6)[stream]))


def round_to(x: np.ndarray, dtype: str):
    """Round float values to the storage dtype.  Returns (torch CPU tensor in
    that dtype, the same values as float64 numpy) so the oracle sees exactly
    what the GPU sees."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    elif dtype != "f32":
        raise ValueError(dtype)
    return t, t.to(torch.float64).numpy()


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """float32 standard normal draws times ``std`` from one seeded stream."""
    x = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def gt_inputs(w: Workload, N: int | None = None):
    """Q, K, V (and dOut when the workload has a backward pass), each as
    (tensor in the workload dtype, float64 copy).  Shapes [N, H, D]."""
    N = w.N if N is None else N
    shape = (N, w.H, w.D)
    out = {
        "Q": round_to(normal(w.seed, STREAM_A, shape, w.qkv_std), w.dtype),
        "K": round_to(normal(w.seed, STREAM_B, shape, w.qkv_std), w.dtype),
        "V": round_to(normal(w.seed, STREAM_C, shape, w.qkv_std), w.dtype),
    }
    if w.backward:
        out["dOut"] = round_to(normal(w.seed, STREAM_DOUT, shape), w.dtype)
    return out


def gatv2_inputs(w: Workload, N: int | None = None):
    """X [N, F] ~ N(0, 1); W_l, W_r [F, H*D] Glorot-uniform; a [H, D] ~ N(0, 0.1^2);
    dOut [N, H, D] ~ N(0, 1).  Each as (tensor in the workload dtype, float64 copy)."""
    N = w.N if N is None else N
    F, HD = w.F, w.H * w.D
    lim = math.sqrt(6.0 / (F + HD))
    wl = _rng(w.seed, STREAM_B).uniform(-lim, lim, size=(F, HD)).astype(np.float32)
    wr = _rng(w.seed, STREAM_C).uniform(-lim, lim, size=(F, HD)).astype(np.float32)
    out = {
        "X": round_to(normal(w.seed, STREAM_A, (N, F)), w.dtype),
        "W_l": round_to(wl, w.dtype),
        "W_r": round_to(wr, w.dtype),
        "a": round_to(normal(w.seed, STREAM_ATT, (w.H, w.D), 0.1), w.dtype),
    }
    if w.backward:
        out["dOut"] = round_to(normal(w.seed, STREAM_DOUT, (N, w.H, w.D)), w.dtype)
    return out


def agg_inputs(w: Workload, N: int | None = None):
    """X [N, H, D] ~ N(0, 1) rounded to the workload dtype (the min / max
    aggregation's node rows) and dOut [N, H, D] ~ N(0, 1)."""
    N = w.N if N is None else N
    shape = (N, w.H, w.D)
    out = {"X": round_to(normal(w.seed, STREAM_A, shape), w.dtype)}
    if w.backward:
        out["dOut"] = round_to(normal(w.seed, STREAM_DOUT, shape), w.dtype)
    return out


def degree_summary(indptr: np.ndarray) -> dict:
    """Row-degree statistics of a CSR (for logs and sanity tests)."""
    deg = np.diff(indptr.astype(np.int64))
    return {"N": int(len(deg)), "E": int(indptr[-1]), "mean": float(deg.mean()),
            "median": float(np.median(deg)), "max": int(deg.max()), "min": int(deg.min())}
