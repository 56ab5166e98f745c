"""fp64 CPU oracle for fused CSR edge attention (Graph Transformer and GATv2).

TEST INFRASTRUCTURE ONLY: the library never imports this package.  The tests,
the package smoke check and the benchmark's CPU-baseline leg are its only
callers.  It shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, doubles, explicit edge loops,
dense softmax per row); this module compiles it with gcc on first use and
wraps it with ctypes.  The row partition below is host logic written from its
definition in plain Python.

Every function follows the definitions on "On Efficient Scaling of GNNs via
IO-Aware Layers Implementations" (abstract; Yandex Research blog post,
"Attention-based layers" paragraph) and the Graph Transformer / GATv2 score
functions the pages cite; ``oracle.c`` states each reading in its header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_I32P = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_I64P = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_F64P = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64, _int, _dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        sig = {
            "oracle_threads": ([], _int),
            "oracle_set_threads": ([_int], None),
            "oracle_transpose": ([_i64, _I32P, _I32P, _I32P, _I32P], _int),
            "oracle_gt_fwd_rows": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P,
                                    _i64, _I64P, _F64P, _F64P], _int),
            "oracle_gt_fwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P,
                               _F64P, _F64P], _int),
            "oracle_gt_bwd_dq_rows": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P,
                                       _F64P, _i64, _I64P, _F64P], _int),
            "oracle_gt_bwd_dkdv_srcs": ([_i64, _I32P, _I32P, _I32P, _I32P, _int, _int, _F64P,
                                         _F64P, _F64P, _F64P, _i64, _I64P, _F64P, _F64P], _int),
            "oracle_gt_bwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P, _F64P,
                               _F64P, _F64P, _F64P], _int),
            "oracle_matmul": ([_i64, _int, _int, _F64P, _F64P, _F64P], _int),
            "oracle_gatv2_fwd_rows": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P,
                                       _dbl, _i64, _I64P, _F64P, _F64P], _int),
            "oracle_gatv2_fwd": ([_i64, _int, _int, _int, _I32P, _I32P, _F64P, _F64P, _F64P,
                                  _F64P, _dbl, _int, _F64P, _F64P, _F64P, _F64P], _int),
            "oracle_gatv2_bwd": ([_i64, _int, _int, _int, _I32P, _I32P, _F64P, _F64P, _F64P,
                                  _F64P, _dbl, _int, _F64P, _F64P, _F64P, _F64P, _F64P, _F64P,
                                  _F64P], _int),
            "oracle_round_bf16": ([_dbl], _dbl),
            "oracle_agg_fwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _I32P], _int),
            "oracle_agg_bwd": ([_i64, _int, _I32P, _F64P, _F64P], _int),
            "oracle_rcm": ([_i64, _I32P, _I32P, _I32P], _int),
            "oracle_gat_edge_fwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P, _dbl, _F64P,
                                     _F64P], _int),
            "oracle_gat_edge_bwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P, _dbl, _F64P,
                                     _F64P, _F64P, _F64P], _int),
            "oracle_gat_fwd": ([_i64, _int, _int, _int, _I32P, _I32P, _F64P, _F64P, _F64P, _dbl, _int,
                                _F64P, _F64P, _F64P], _int),
            "oracle_gat_bwd": ([_i64, _int, _int, _int, _I32P, _I32P, _F64P, _F64P, _F64P, _dbl, _int,
                                _F64P, _F64P, _F64P, _F64P, _F64P], _int),
            "oracle_gt_bias_fwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P, _F64P,
                                    _F64P, _F64P], _int),
            "oracle_gt_bias_bwd": ([_i64, _I32P, _I32P, _int, _int, _F64P, _F64P, _F64P, _F64P,
                                    _F64P, _F64P, _F64P, _F64P, _F64P], _int),
            "oracle_gatv2_bwd_bound": ([_i64, _int, _int, _int, _I32P, _I32P, _F64P, _F64P, _F64P,
                                        _F64P, _dbl, _F64P, _F64P, _F64P, _F64P, _F64P], _int),
            "oracle_gatv2_branch_slack": ([_i64, _int, _int, _int, _I32P, _I32P, _F64P, _F64P,
                                           _F64P, _F64P, _dbl, _int, _dbl, _F64P, _F64P, _F64P,
                                           _F64P, _F64P], _int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.int32)


def _check(rc: int, name: str):
    if rc != 0:
        raise MemoryError(f"oracle {name} failed ({rc})")


def threads() -> int:
    """OpenMP threads the oracle uses."""
    return _load().oracle_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


# ---------------------------------------------------------------- graph steps

def transpose(indptr, indices):
    """Transposed CSR (t_indptr[N+1], t_dst[E]): destinations of each source,
    ascending.  Counting sort in C."""
    indptr, indices = _i32(indptr), _i32(indices)
    N = len(indptr) - 1
    t_indptr = np.zeros(N + 1, np.int32)
    t_dst = np.zeros(max(int(indptr[-1]), 1), np.int32)
    _check(_load().oracle_transpose(N, indptr, indices, t_indptr, t_dst), "transpose")
    return t_indptr, t_dst[: int(indptr[-1])]


def partition(indptr, threshold: int, chunk: int):
    """Row partition by its definition: rows of degree > ``threshold`` are
    split rows (ascending id); each is cut into consecutive edge chunks of
    ``chunk`` edges (the last one shorter).  Returns int32 arrays
    split_rows[S], chunk_ptr[S+1] (chunk range per split row), chunk_row[C],
    chunk_beg[C], chunk_end[C]."""
    indptr = np.asarray(indptr, dtype=np.int64)
    split_rows, chunk_ptr, crow, cbeg, cend = [], [0], [], [], []
    for i in range(len(indptr) - 1):
        b, e = int(indptr[i]), int(indptr[i + 1])
        if e - b <= threshold:
            continue
        split_rows.append(i)
        x = b
        while x < e:
            crow.append(i)
            cbeg.append(x)
            cend.append(min(x + chunk, e))
            x += chunk
        chunk_ptr.append(len(crow))
    as32 = lambda v: np.asarray(v, dtype=np.int32)
    return {"split_rows": as32(split_rows), "chunk_ptr": as32(chunk_ptr),
            "chunk_row": as32(crow), "chunk_beg": as32(cbeg), "chunk_end": as32(cend)}


# ---------------------------------------------------------- Graph Transformer

def gt_fwd(indptr, indices, Q, K, V, rows=None):
    """out [R, H, D], lse [R, H] for the listed rows (all rows if None)."""
    indptr, indices = _i32(indptr), _i32(indices)
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N, H, D = Q.shape
    lib = _load()
    if rows is None:
        out = np.empty((N, H, D)); lse = np.empty((N, H))
        _check(lib.oracle_gt_fwd(N, indptr, indices, H, D, Q, K, V, out, lse), "gt_fwd")
        return out, lse
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), H, D)); lse = np.empty((len(rows), H))
    _check(lib.oracle_gt_fwd_rows(N, indptr, indices, H, D, Q, K, V, len(rows), rows, out, lse),
           "gt_fwd_rows")
    return out, lse


def gt_bwd(indptr, indices, Q, K, V, dO):
    """(dQ, dK, dV), each [N, H, D], by the softmax Jacobian."""
    indptr, indices = _i32(indptr), _i32(indices)
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    N, H, D = Q.shape
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Q), np.empty_like(Q)
    _check(_load().oracle_gt_bwd(N, indptr, indices, H, D, Q, K, V, dO, dQ, dK, dV), "gt_bwd")
    return dQ, dK, dV


def gt_bias_fwd(indptr, indices, Q, K, V, B):
    """GT forward with an additive score bias B [E, H] (CSR edge order):
    s_ij = q_i . k_j / sqrt(D) + B[e, h].  (out [N, H, D], lse [N, H])."""
    indptr, indices = _i32(indptr), _i32(indices)
    Q, K, V, B = _f64(Q), _f64(K), _f64(V), _f64(B)
    N, H, D = Q.shape
    out = np.empty((N, H, D)); lse = np.empty((N, H))
    ix = indices if len(indices) else np.zeros(1, np.int32)
    Bp = B if B.size else np.zeros(1)
    _check(_load().oracle_gt_bias_fwd(N, indptr, ix, H, D, Q, K, V, Bp, out, lse), "gt_bias_fwd")
    return out, lse


def gt_bias_bwd(indptr, indices, Q, K, V, B, dO):
    """(dQ, dK, dV, dB) of the biased GT layer; dB = dS per edge and head."""
    indptr, indices = _i32(indptr), _i32(indices)
    Q, K, V, B, dO = _f64(Q), _f64(K), _f64(V), _f64(B), _f64(dO)
    N, H, D = Q.shape
    E = len(indices)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Q), np.empty_like(Q)
    dB = np.empty((max(E, 1), H))
    ix = indices if E else np.zeros(1, np.int32)
    Bp = B if B.size else np.zeros(1)
    _check(_load().oracle_gt_bias_bwd(N, indptr, ix, H, D, Q, K, V, Bp, dO, dQ, dK, dV, dB),
           "gt_bias_bwd")
    return dQ, dK, dV, dB[:E]


def gt_bwd_dq_rows(indptr, indices, Q, K, V, dO, rows):
    indptr, indices = _i32(indptr), _i32(indices)
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    N, H, D = Q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dq = np.empty((len(rows), H, D))
    _check(_load().oracle_gt_bwd_dq_rows(N, indptr, indices, H, D, Q, K, V, dO, len(rows), rows, dq),
           "gt_bwd_dq_rows")
    return dq


def gt_bwd_dkdv_srcs(indptr, indices, Q, K, V, dO, srcs, transposed=None):
    indptr, indices = _i32(indptr), _i32(indices)
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    N, H, D = Q.shape
    t_indptr, t_dst = transposed if transposed is not None else transpose(indptr, indices)
    t_dst = _i32(t_dst) if len(t_dst) else np.zeros(1, np.int32)
    srcs = np.ascontiguousarray(srcs, dtype=np.int64)
    dk = np.empty((len(srcs), H, D)); dv = np.empty((len(srcs), H, D))
    _check(_load().oracle_gt_bwd_dkdv_srcs(N, indptr, indices, _i32(t_indptr), t_dst, H, D,
                                           Q, K, V, dO, len(srcs), srcs, dk, dv),
           "gt_bwd_dkdv_srcs")
    return dk, dv


# ---------------------------------------------------------------------- GATv2

def matmul(X, W):
    X, W = _f64(X), _f64(W)
    Y = np.empty((X.shape[0], W.shape[1]))
    _load().oracle_matmul(X.shape[0], X.shape[1], W.shape[1], X, W, Y)
    return Y


_STORE = {None: 0, "f64": 0, "f32": 1, "bf16": 2}


def round_bf16(x: float) -> float:
    """Nearest bfloat16 (ties to even) of a double, via float."""
    return _load().oracle_round_bf16(float(x))


def gatv2_fwd(indptr, indices, X, Wl, Wr, a, slope=0.2, store=None):
    """(FL, FR, out, lse): projections [N, H, D], output [N, H, D], lse [N, H].
    ``store`` ("f32" or "bf16") rounds the projections to the layer's storage
    dtype before the edge stage, as the layer stores them; None keeps fp64."""
    indptr, indices = _i32(indptr), _i32(indices)
    X, Wl, Wr, a = _f64(X), _f64(Wl), _f64(Wr), _f64(a)
    N, F = X.shape
    H, D = a.shape
    FL = np.empty((N, H, D)); FR = np.empty((N, H, D))
    out = np.empty((N, H, D)); lse = np.empty((N, H))
    _check(_load().oracle_gatv2_fwd(N, F, H, D, indptr, indices, X, Wl, Wr, a, float(slope),
                                    _STORE[store], FL, FR, out, lse), "gatv2_fwd")
    return FL, FR, out, lse


def gatv2_fwd_rows(indptr, indices, FL, FR, a, rows, slope=0.2):
    indptr, indices = _i32(indptr), _i32(indices)
    FL, FR, a = _f64(FL), _f64(FR), _f64(a)
    N, H, D = FL.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((len(rows), H, D)); lse = np.empty((len(rows), H))
    _check(_load().oracle_gatv2_fwd_rows(N, indptr, indices, H, D, FL, FR, a, float(slope),
                                         len(rows), rows, out, lse), "gatv2_fwd_rows")
    return out, lse


def gatv2_bwd(indptr, indices, X, Wl, Wr, a, dO, slope=0.2, store=None):
    """dict with dX [N, F], dW_l, dW_r [F, H*D], da [H, D], dFL, dFR [N, H, D].
    ``store`` as in gatv2_fwd."""
    indptr, indices = _i32(indptr), _i32(indices)
    X, Wl, Wr, a, dO = _f64(X), _f64(Wl), _f64(Wr), _f64(a), _f64(dO)
    N, F = X.shape
    H, D = a.shape
    dX = np.empty((N, F)); dWl = np.empty((F, H * D)); dWr = np.empty((F, H * D))
    da = np.empty((H, D)); dFL = np.empty((N, H, D)); dFR = np.empty((N, H, D))
    _check(_load().oracle_gatv2_bwd(N, F, H, D, indptr, indices, X, Wl, Wr, a, float(slope),
                                    _STORE[store], dO, dX, dWl, dWr, da, dFL, dFR), "gatv2_bwd")
    return {"dX": dX, "dW_l": dWl, "dW_r": dWr, "da": da, "dFL": dFL, "dFR": dFR}


# Relative width of the band of z = FL + FR in which two correct
# implementations may decide the LeakyReLU branch differently.  Float storage:
# projections accumulated in fp32 differ from the exact ones by a few float
# ulps, far inside 2^-18.  bf16 storage: the projections are the correctly
# rounded values on both sides, so no branch is undecided.
BRANCH_TAU = {"bf16": 0.0, "f32": 2.0 ** -18}


def gatv2_branch_slack(indptr, indices, X, Wl, Wr, a, dO, slope=0.2, store="bf16", tau=None):
    """Largest change of dX, dW_l, dW_r, da that LeakyReLU branches left
    undecided by the projections' storage precision can cause (see
    oracle_gatv2_branch_slack in oracle.c).  dict of nonnegative arrays."""
    indptr, indices = _i32(indptr), _i32(indices)
    X, Wl, Wr, a, dO = _f64(X), _f64(Wl), _f64(Wr), _f64(a), _f64(dO)
    N, F = X.shape
    H, D = a.shape
    tau = BRANCH_TAU[store] if tau is None else tau
    sX = np.empty((N, F)); sWl = np.empty((F, H * D)); sWr = np.empty((F, H * D))
    sda = np.empty((H, D))
    _check(_load().oracle_gatv2_branch_slack(N, F, H, D, indptr, indices, X, Wl, Wr, a,
                                             float(slope), _STORE[store], float(tau), dO,
                                             sX, sWl, sWr, sda), "gatv2_branch_slack")
    return {"dX": sX, "dW_l": sWl, "dW_r": sWr, "da": sda}


# --------------------------------------------------- GAT (original attention score)

def gat_fwd(indptr, indices, X, W, a, slope=0.2, store=None):
    """(FL, out, lse) of the GAT layer: FL = X W [N, H, D] (rounded to
    ``store`` as the layer stores it), e_ij = LeakyReLU(a[h,0] . FL_i +
    a[h,1] . FL_j), softmax over the row, out_i = sum_j p_ij FL_j.
    a: [H, 2, D]."""
    indptr, indices = _i32(indptr), _i32(indices)
    X, W, a = _f64(X), _f64(W), _f64(a)
    N, F = X.shape
    H, _, D = a.shape
    FL = np.empty((N, H, D)); out = np.empty((N, H, D)); lse = np.empty((N, H))
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_gat_fwd(N, F, H, D, indptr, ix, X, W, a, float(slope), _STORE[store],
                                  FL, out, lse), "gat_fwd")
    return FL, out, lse


def gat_bwd(indptr, indices, X, W, a, dO, slope=0.2, store=None):
    """dict with dX [N, F], dW [F, H*D], da [H, 2, D], dFL [N, H, D]."""
    indptr, indices = _i32(indptr), _i32(indices)
    X, W, a, dO = _f64(X), _f64(W), _f64(a), _f64(dO)
    N, F = X.shape
    H, _, D = a.shape
    dX = np.empty((N, F)); dW = np.empty((F, H * D)); da = np.empty((H, 2, D))
    dFL = np.empty((N, H, D))
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_gat_bwd(N, F, H, D, indptr, ix, X, W, a, float(slope), _STORE[store], dO,
                                  dX, dW, da, dFL), "gat_bwd")
    return {"dX": dX, "dW": dW, "da": da, "dFL": dFL}


def gat_edge_fwd(indptr, indices, Fv, el, er, slope=0.2):
    """GAT edge stage: (out [N, H, D], lse [N, H]) from the projected
    features Fv [N, H, D] and the score halves el, er [N, H]."""
    indptr, indices = _i32(indptr), _i32(indices)
    Fv, el, er = _f64(Fv), _f64(el), _f64(er)
    N, H, D = Fv.shape
    out = np.empty((N, H, D)); lse = np.empty((N, H))
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_gat_edge_fwd(N, indptr, ix, H, D, Fv, el, er, float(slope), out, lse),
           "gat_edge_fwd")
    return out, lse


def gat_edge_bwd(indptr, indices, Fv, el, er, dO, slope=0.2):
    """(dFv, del, der) of the GAT edge stage (dFv: the value path only)."""
    indptr, indices = _i32(indptr), _i32(indices)
    Fv, el, er, dO = _f64(Fv), _f64(el), _f64(er), _f64(dO)
    N, H, D = Fv.shape
    dFv = np.empty((N, H, D)); de_l = np.empty((N, H)); de_r = np.empty((N, H))
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_gat_edge_bwd(N, indptr, ix, H, D, Fv, el, er, float(slope), dO, dFv, de_l,
                                       de_r), "gat_edge_bwd")
    return dFv, de_l, de_r


# ------------------------------------------------------- min / max aggregation

def agg_fwd(indptr, indices, X, op="max"):
    """(out, arg) of the min / max aggregation over [N, ...] node rows (any
    trailing shape, flattened per node): out = the extreme of the sources'
    values per element, arg = the source of its first occurrence in CSR
    order (-1 and out = 0 for an empty row)."""
    indptr, indices = _i32(indptr), _i32(indices)
    X = _f64(X)
    N = X.shape[0]
    F = int(np.prod(X.shape[1:])) if X.ndim > 1 else 1
    out = np.empty(X.shape)
    arg = np.empty(X.shape, np.int32)
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_agg_fwd(N, indptr, ix, F, 1 if op == "max" else 0, X, out, arg),
           "agg_fwd")
    return out, arg


def agg_bwd(arg, dO):
    """dX: dO routed to the winning sources (sum over the rows that chose them)."""
    arg = _i32(arg)
    dO = _f64(dO)
    N = dO.shape[0]
    F = int(np.prod(dO.shape[1:])) if dO.ndim > 1 else 1
    dX = np.empty(dO.shape)
    _check(_load().oracle_agg_bwd(N, F, arg, dO, dX), "agg_bwd")
    return dX


# ------------------------------------------------------------ graph reordering

def order_degree(indptr, indices):
    """perm[v] = new id: nodes by descending in-degree (times gathered), ties
    by ascending id."""
    N = len(indptr) - 1
    indeg = np.bincount(np.asarray(indices, dtype=np.int64), minlength=N)
    order = np.lexsort((np.arange(N), -indeg))
    perm = np.empty(N, np.int32)
    perm[order] = np.arange(N, dtype=np.int32)
    return perm


def order_rcm(indptr, indices):
    """perm[v] = new id under reverse Cuthill-McKee (queue-based, in C; see
    oracle_rcm in oracle.c for the tie rules)."""
    indptr, indices = _i32(indptr), _i32(indices)
    N = len(indptr) - 1
    perm = np.empty(max(N, 1), np.int32)
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_rcm(N, indptr, ix, perm), "rcm")
    return perm[:N]


def relabel_csr(indptr, indices, perm):
    """The graph under perm: new row perm[v] = old row v with sources mapped
    through perm, in their original order."""
    indptr = np.asarray(indptr, dtype=np.int64)
    N = len(indptr) - 1
    inv = np.empty(N, np.int64)
    inv[np.asarray(perm, dtype=np.int64)] = np.arange(N)
    deg = np.diff(indptr)[inv]
    new_ptr = np.zeros(N + 1, np.int64)
    new_ptr[1:] = np.cumsum(deg)
    rows = [np.asarray(perm)[indices[indptr[inv[u]]:indptr[inv[u] + 1]]] for u in range(N)]
    new_idx = np.concatenate(rows) if rows else np.zeros(0)
    return new_ptr.astype(np.int32), new_idx.astype(np.int32)


# ------------------------------------------- rounding bound of the fp32 GATv2 backward

def gatv2_bwd_bound(indptr, indices, X, Wl, Wr, a, dO, slope=0.2):
    """Elementwise first-order bound on |fp32 result - exact| of dX, dW_l,
    dW_r, da for a float GATv2 layer (see oracle_gatv2_bwd_bound in
    oracle.c for the arithmetic it covers).  dict of nonnegative arrays."""
    indptr, indices = _i32(indptr), _i32(indices)
    X, Wl, Wr, a, dO = _f64(X), _f64(Wl), _f64(Wr), _f64(a), _f64(dO)
    N, F = X.shape
    H, D = a.shape
    bX = np.empty((N, F)); bWl = np.empty((F, H * D)); bWr = np.empty((F, H * D))
    bda = np.empty((H, D))
    ix = indices if len(indices) else np.zeros(1, np.int32)
    _check(_load().oracle_gatv2_bwd_bound(N, F, H, D, indptr, ix, X, Wl, Wr, a, float(slope), dO,
                                          bX, bWl, bWr, bda), "gatv2_bwd_bound")
    return {"dX": bX, "dW_l": bWl, "dW_r": bWr, "da": bda}


# ------------------------------------------------------------ block-sparse tiles

def tile_extract(indptr, indices, N, min_nnz, panel=128, width=16):
    """Block-sparse split of a CSR by its definition: rows in panels of
    ``panel`` destinations, sources in column tiles of ``width``; a
    (panel, tile) pair with at least ``min_nnz`` edges (repeats counted) is
    kept, with one ``width``-bit mask per panel row (bit b: source width*tile
    + b present).  A mask holds each (destination, source) pair once: the
    first edge of the pair in CSR order sets the bit, and a repeat of it
    (another term of the row's softmax) stays in the residual CSR with every
    edge of a tile that is not kept (same row order and source order).

    Returns dict: tile_ptr [P+1], tile_col [T], tile_bits [T, panel] (uint16),
    r_indptr [N+1], r_indices [E_r]."""
    indptr = np.asarray(indptr, dtype=np.int64)
    indices = np.asarray(indices, dtype=np.int64)
    P = (N + panel - 1) // panel
    rows = np.repeat(np.arange(N), np.diff(indptr))
    pan, col = rows // panel, indices // width
    key = pan * ((N + width - 1) // width) + col
    uniq, counts = np.unique(key, return_counts=True)
    kept_keys = uniq[counts >= min_nnz]
    # first occurrence of every (destination, source) pair in CSR order
    first = np.zeros(len(indices), bool)
    if len(indices):
        _, first_at = np.unique(rows * N + indices, return_index=True)
        first[first_at] = True
    kept = np.isin(key, kept_keys) & first
    tile_ptr = np.zeros(P + 1, np.int64)
    kp = kept_keys // ((N + width - 1) // width)
    np.add.at(tile_ptr, kp + 1, 1)
    tile_ptr = np.cumsum(tile_ptr)
    tile_col = (kept_keys % ((N + width - 1) // width)).astype(np.int32)
    tile_bits = np.zeros((len(kept_keys), panel), np.uint16)
    tix = np.searchsorted(kept_keys, key[kept])
    np.bitwise_or.at(tile_bits, (tix, rows[kept] % panel),
                     (1 << (indices[kept] % width)).astype(np.uint16))
    r_counts = np.bincount(rows[~kept], minlength=N)
    r_indptr = np.zeros(N + 1, np.int64)
    r_indptr[1:] = np.cumsum(r_counts)
    return {"tile_ptr": tile_ptr.astype(np.int32), "tile_col": tile_col,
            "tile_bits": tile_bits, "r_indptr": r_indptr.astype(np.int32),
            "r_indices": indices[~kept].astype(np.int32)}
