"""Fused CSR edge attention (Graph Transformer, GATv2) on sm_103a.

A thin ctypes binding over the C ABI of ``libsga.so`` (declared in
``include/sga.h``).  This module only marshals arguments: every step of the
forward and backward passes runs in the library's CUDA kernels.  PyTorch
provides device memory and the current stream.  There is no CPU fallback: if
the library is missing, every call raises.

Graph convention: destination-sorted CSR (row i = destination, ``indices`` =
sources), int32, on the GPU.  Node tensors are [N, H, D], float32 or bfloat16.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsga.so")

SGA_OK, SGA_EINVAL, SGA_EUNSUPPORTED, SGA_ECUDA, SGA_EWORKSPACE, SGA_EDEVICE_CHECK, SGA_ELIMIT = range(7)
SGA_F32, SGA_BF16 = 0, 1

KERNELS = {
    "gt_fwd": 1, "gt_fwd_merge": 2, "gt_bwd_dq": 3, "gt_bwd_dkdv": 4, "gt_bwd_merge": 5,
    "gatv2_proj": 6, "gatv2_fwd": 7, "gatv2_fwd_merge": 8, "gatv2_bwd_dst": 9,
    "gatv2_bwd_src": 10, "gatv2_bwd_merge": 11, "gatv2_bwd_dx": 12, "gatv2_bwd_dw": 13,
    "gatv2_bwd_reduce": 14, "bsr_fwd": 15, "bsr_bwd_delta": 16, "bsr_bwd_dq": 17,
    "bsr_bwd_dkdv": 18, "agg_fwd": 19, "agg_fwd_merge": 20, "agg_bwd": 21, "agg_bwd_merge": 22,
    "gat_fwd": 23, "gat_bwd_dst": 24, "gat_bwd_src": 25,
}

SGA_LAYER_ATTENTION, SGA_LAYER_MINMAX, SGA_LAYER_GAT = 0, 1, 2
SGA_AGG_MAX, SGA_AGG_MIN = 0, 1
SGA_SCHED_STREAM, SGA_SCHED_FEATURE, SGA_SCHED_BILEVEL = 0, 1, 2
SGA_ORDER_DEGREE, SGA_ORDER_RCM = 0, 1

ARRAYS = {
    "t_indptr": 0, "t_dst": 1, "split_rows": 2, "chunk_ptr": 3, "chunk_row": 4, "chunk_beg": 5,
    "chunk_end": 6, "t_split_rows": 7, "t_chunk_ptr": 8, "t_chunk_row": 9, "t_chunk_beg": 10,
    "t_chunk_end": 11, "tile_ptr": 12, "tile_col": 13, "tile_bits": 14, "r_indptr": 15,
    "r_indices": 16, "row_order": 17, "t_row_order": 18, "t_eid": 19,
}


class SgaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib().sga_status_string(status).decode()
        if status == SGA_ECUDA:
            msg += f" (cudaError {_lib().sga_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")


class PlanOpts(ctypes.Structure):
    _fields_ = [("split_threshold", ctypes.c_int32), ("chunk_len", ctypes.c_int32),
                ("in_features", ctypes.c_int32), ("tile_min_nnz", ctypes.c_int32),
                ("layer", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("edge_bias", ctypes.c_int32), ("row_order", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("E", ctypes.c_int64), ("H", ctypes.c_int32),
                ("D", ctypes.c_int32), ("F", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("split_threshold", ctypes.c_int32), ("chunk_len", ctypes.c_int32),
                ("n_split", ctypes.c_int32), ("n_chunks", ctypes.c_int32),
                ("t_n_split", ctypes.c_int32), ("t_n_chunks", ctypes.c_int32),
                ("plan_device_bytes", ctypes.c_int64), ("n_tiles", ctypes.c_int32),
                ("n_panels", ctypes.c_int32), ("E_residual", ctypes.c_int64),
                ("n_entries", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_LIB = None
_vp, _i64, _int, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float

_SIGNATURES = {
    "sga_status_string": ([_int], ctypes.c_char_p),
    "sga_last_cuda_error": ([], _int),
    "sga_launch_count": ([], _i64),
    "sga_plan_create": ([_vp, _vp, _i64, _i64, _int, _int, _int, ctypes.POINTER(PlanOpts), _vp,
                         ctypes.POINTER(_vp)], _int),
    "sga_plan_workspace_bytes": ([_vp], ctypes.c_size_t),
    "sga_plan_set_workspace": ([_vp, _vp, ctypes.c_size_t], _int),
    "sga_plan_destroy": ([_vp], None),
    "sga_plan_get_info": ([_vp, ctypes.POINTER(PlanInfo)], _int),
    "sga_plan_copy_array": ([_vp, _int, _vp, _i64], _int),
    "sga_read_device_error": ([_vp, _vp, ctypes.POINTER(ctypes.c_int32)], _int),
    "gt_attn_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp, _vp, _vp],
                    _int),
    "gt_attn_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int,
                     _vp, _vp, _vp, _vp], _int),
    "gatv2_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _f32, _int,
                   _vp, _vp, _vp, _vp, _vp], _int),
    "gatv2_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int,
                   _int, _int, _f32, _int, _vp, _vp, _vp, _vp, _vp], _int),
    "gt_attn_bias_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp,
                          _vp, _vp], _int),
    "gt_attn_bias_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int,
                          _int, _vp, _vp, _vp, _vp, _vp], _int),
    "gat_attn_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _f32, _int, _vp, _vp,
                      _vp], _int),
    "gat_attn_bwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _f32,
                      _int, _vp, _vp, _vp, _vp], _int),
    "gt_attn_fwd_noalloc": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp, _vp, _vp],
                            _int),
    "sga_noalloc_scratch_bytes": ([], ctypes.c_size_t),
    "sga_noalloc_read_device_error": ([_vp, ctypes.POINTER(ctypes.c_int32)], _int),
    "agg_minmax_fwd": ([_vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _int, _vp, _vp, _vp,
                        _vp], _int),
    "sga_agg_mask_bytes": ([_vp], ctypes.c_size_t),
    "agg_minmax_bwd": ([_vp, _vp, _vp, _i64, _int, _int, _int, _vp, _vp], _int),
    "sga_reorder": ([_vp, _vp, _i64, _i64, _int, _vp, _vp], _int),
    "sga_relabel_csr": ([_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp], _int),
    "sga_permute_rows": ([_vp, _i64, _i64, _vp, _int, _vp, _vp], _int),
    "sga_profile_start": ([_int], _int),
    "sga_profile_stop": ([ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i64)], _int),
}


def _lib():
    """Load libsga.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run sparse_graph_attention_csr_gb300.build "
                              "(or __graft_entry__.build()) first; there is no CPU fallback")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


def load_library():
    """Load the native library now; returns the ctypes handle."""
    return _lib()


def _check(status: int, what: str):
    if status != SGA_OK:
        raise SgaError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SGA_F32
    if t.dtype == torch.bfloat16:
        return SGA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, numel=None, rows=None, plan=None):
    """Checks a tensor before its pointer reaches the library, which sees
    pointers only: a CUDA tensor, contiguous, of the expected dtype, element
    count and leading dimension, on the plan's device."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {tuple(t.shape)}")
    if rows is not None and (t.dim() == 0 or t.shape[0] != rows):
        raise ValueError(f"{name} must have {rows} rows, got {tuple(t.shape)}")
    if plan is not None and t.device != plan.device:
        raise ValueError(f"{name} is on {t.device}, the plan's graph on {plan.device}")


def _node(t, name, plan, dtype=None):
    """A node tensor [N, H, D] (any contiguous view with N rows and N*H*D elements)."""
    _need(t, name, plan.dtype if dtype is None else dtype, plan.N * plan.H * plan.D, plan.N, plan)


def _head(t, name, plan):
    """A per-head float32 node tensor [N, H]."""
    _need(t, name, torch.float32, plan.N * plan.H, plan.N, plan)


def launch_count() -> int:
    """Kernels launched by the library in this process."""
    return int(_lib().sga_launch_count())


def profile_start(kernel: str):
    _check(_lib().sga_profile_start(KERNELS[kernel]), "sga_profile_start")


def profile_stop():
    """(total device ms, launches) of the kernel kind being profiled."""
    ms, n = ctypes.c_double(), ctypes.c_int64()
    _check(_lib().sga_profile_stop(ctypes.byref(ms), ctypes.byref(n)), "sga_profile_stop")
    return ms.value, n.value


class Plan:
    """A graph plan: validated CSR, transposed CSR and degree partitions on the
    device, plus the caller-owned workspace the kernels need.

    ``indptr``/``indices`` must stay alive and unchanged while the plan is used.
    """

    def __init__(self, indptr: torch.Tensor, indices: torch.Tensor, H: int, D: int,
                 dtype=torch.bfloat16, F: int = 0, split_threshold: int = 0, chunk_len: int = 0,
                 tile_min_nnz: int = 0, layer: int = SGA_LAYER_ATTENTION,
                 schedule: int = SGA_SCHED_STREAM, edge_bias: bool = False,
                 row_order: int = 0, stream=None):
        if dtype not in (torch.float32, torch.bfloat16):
            raise TypeError(f"the layers compute in torch.float32 or torch.bfloat16, not {dtype}")
        _need(indptr, "indptr", torch.int32)
        _need(indices, "indices", torch.int32)
        if indices.device != indptr.device:
            raise ValueError(f"indices on {indices.device}, indptr on {indptr.device}")
        self.indptr, self.indices = indptr, indices
        self.N = indptr.numel() - 1
        self.E = indices.numel()
        self.device = indptr.device
        self.H, self.D, self.F = int(H), int(D), int(F)
        self.dtype = dtype
        self.dt = SGA_F32 if dtype == torch.float32 else SGA_BF16
        self.layer = int(layer)
        # walking order of the edge kernels: 0 (default) / 1 descending degree, 2 ascending id
        self.row_order, self.edge_bias = int(row_order), bool(edge_bias)
        opts = PlanOpts(int(split_threshold), int(chunk_len), int(F), int(tile_min_nnz),
                        self.layer, int(schedule), 1 if edge_bias else 0, int(row_order))
        handle = ctypes.c_void_p()
        self._h = None
        _check(_lib().sga_plan_create(_ptr(indptr), _ptr(indices), self.N, self.E, self.H, self.D,
                                      self.dt, ctypes.byref(opts), _stream(stream),
                                      ctypes.byref(handle)), "sga_plan_create")
        self._h = handle
        nbytes = int(_lib().sga_plan_workspace_bytes(handle))
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=indptr.device)
        _check(_lib().sga_plan_set_workspace(handle, _ptr(self.workspace), nbytes),
               "sga_plan_set_workspace")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _LIB is not None:
            _LIB.sga_plan_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        inf = PlanInfo()
        _check(_lib().sga_plan_get_info(self._h, ctypes.byref(inf)), "sga_plan_get_info")
        return {name: getattr(inf, name) for name, _ in PlanInfo._fields_}

    def array(self, name: str):
        """Copy one plan array (transposed CSR or partition) to a numpy int32 array."""
        import numpy as np
        inf = self.info()
        n = {"t_indptr": self.N + 1, "t_dst": self.E, "split_rows": inf["n_split"],
             "chunk_ptr": inf["n_split"] + 1, "chunk_row": inf["n_chunks"],
             "chunk_beg": inf["n_chunks"], "chunk_end": inf["n_chunks"],
             "t_split_rows": inf["t_n_split"], "t_chunk_ptr": inf["t_n_split"] + 1,
             "t_chunk_row": inf["t_n_chunks"], "t_chunk_beg": inf["t_n_chunks"],
             "t_chunk_end": inf["t_n_chunks"],
             "tile_ptr": inf["n_panels"] + 1 if inf["n_panels"] else 0,
             "tile_col": inf["n_tiles"], "tile_bits": inf["n_tiles"] * 64,
             "r_indptr": self.N + 1 if inf["n_panels"] else 0,
             "r_indices": inf["E_residual"],
             "row_order": self.N if self.row_order != 2 else 0,
             "t_row_order": self.N if self.row_order != 2 else 0,
             "t_eid": self.E if self.edge_bias else 0}[name]
        out = np.zeros(max(n, 1), dtype=np.int32)
        _check(_lib().sga_plan_copy_array(self._h, ARRAYS[name], out.ctypes.data, n),
               "sga_plan_copy_array")
        return out[:n]

    def device_error(self, stream=None) -> int:
        """Read and clear the device range-check word (0 = no failed check)."""
        code = ctypes.c_int32()
        st = _lib().sga_read_device_error(self._h, _stream(stream), ctypes.byref(code))
        if st not in (SGA_OK, SGA_EDEVICE_CHECK):
            _check(st, "sga_read_device_error")
        return int(code.value)

    def _graph(self):
        return _ptr(self.indptr), _ptr(self.indices), self.N, self.E


# ------------------------------------------------------------ Graph Transformer

def gt_attn_fwd(plan: Plan, Q, K, V, out=None, lse=None, stream=None):
    """out [N,H,D] (dtype of Q) and lse [N,H] float32."""
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _node(t, n, plan)
    out = torch.empty_like(Q) if out is None else out
    lse = torch.empty((plan.N, plan.H), dtype=torch.float32, device=Q.device) if lse is None else lse
    _node(out, "out", plan)
    _head(lse, "lse", plan)
    _check(_lib().gt_attn_fwd(plan.handle, *plan._graph()[:2], _ptr(Q), _ptr(K), _ptr(V), plan.N,
                              plan.E, plan.H, plan.D, plan.dt, _ptr(out), _ptr(lse),
                              _stream(stream)), "gt_attn_fwd")
    return out, lse


def gt_attn_bwd(plan: Plan, Q, K, V, out, lse, dOut, dQ=None, dK=None, dV=None, stream=None):
    """(dQ, dK, dV), each [N,H,D]."""
    for n, t in (("Q", Q), ("K", K), ("V", V), ("out", out), ("dOut", dOut)):
        _node(t, n, plan)
    _head(lse, "lse", plan)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        _node(t, n, plan)
    _check(_lib().gt_attn_bwd(plan.handle, *plan._graph()[:2], _ptr(Q), _ptr(K), _ptr(V),
                              _ptr(out), _ptr(lse), _ptr(dOut), plan.N, plan.E, plan.H, plan.D,
                              plan.dt, _ptr(dQ), _ptr(dK), _ptr(dV), _stream(stream)),
           "gt_attn_bwd")
    return dQ, dK, dV


def gt_attn_bias_fwd(plan: Plan, Q, K, V, bias, out=None, lse=None, stream=None):
    """Graph Transformer with a per-edge, per-head score bias [E, H] float32
    (CSR edge order): (out, lse).  The plan needs edge_bias=True."""
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _node(t, n, plan)
    _need(bias, "bias", torch.float32, plan=plan)
    if tuple(bias.shape) != (plan.E, plan.H):
        raise ValueError(f"bias must be [{plan.E}, {plan.H}], got {tuple(bias.shape)}")
    out = torch.empty_like(Q) if out is None else out
    lse = torch.empty((plan.N, plan.H), dtype=torch.float32, device=Q.device) if lse is None else lse
    _node(out, "out", plan)
    _head(lse, "lse", plan)
    _check(_lib().gt_attn_bias_fwd(plan.handle, *plan._graph()[:2], _ptr(Q), _ptr(K), _ptr(V),
                                   _ptr(bias), plan.N, plan.E, plan.H, plan.D, plan.dt, _ptr(out),
                                   _ptr(lse), _stream(stream)), "gt_attn_bias_fwd")
    return out, lse


def gt_attn_bias_bwd(plan: Plan, Q, K, V, bias, out, lse, dOut, dQ=None, dK=None, dV=None,
                     dbias=None, stream=None):
    """(dQ, dK, dV, dbias) of the biased layer; dbias [E, H] float32."""
    for n, t in (("Q", Q), ("K", K), ("V", V), ("out", out), ("dOut", dOut)):
        _node(t, n, plan)
    _head(lse, "lse", plan)
    _need(bias, "bias", torch.float32, plan.E * plan.H, plan.E, plan)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    dbias = torch.empty_like(bias) if dbias is None else dbias
    for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        _node(t, n, plan)
    _need(dbias, "dbias", torch.float32, plan.E * plan.H, plan.E, plan)
    _check(_lib().gt_attn_bias_bwd(plan.handle, *plan._graph()[:2], _ptr(Q), _ptr(K), _ptr(V),
                                   _ptr(bias), _ptr(out), _ptr(lse), _ptr(dOut), plan.N, plan.E,
                                   plan.H, plan.D, plan.dt, _ptr(dQ), _ptr(dK), _ptr(dV),
                                   _ptr(dbias), _stream(stream)), "gt_attn_bias_bwd")
    return dQ, dK, dV, dbias


def gt_attn_fwd_noalloc(indptr, indices, Q, K, V, out=None, lse=None, stream=None):
    """Graph Transformer forward without a plan or workspace, for callers that
    must not allocate device memory (the library uses a fixed static device
    array instead; see include/sga.h).  Passing ``out`` and ``lse`` keeps this
    call free of allocations on the Python side too.  Synchronises the stream
    once; the first call on a device looks up the static array's address, so
    make it before any stream capture.  Returns (out, lse).

    Shapes are checked here before the library sees any pointer: N is taken
    from ``indptr`` (N + 1 entries), Q, K, V (and ``out``) must be [N, H, D] of
    one dtype, ``lse`` [N, H] float32, all on one device."""
    _need(indptr, "indptr", torch.int32)
    _need(indices, "indices", torch.int32)
    if indptr.dim() != 1 or indices.dim() != 1 or indptr.numel() < 1:
        raise ValueError("indptr and indices must be 1-D, indptr with N + 1 entries")
    N = indptr.numel() - 1
    if Q.dim() != 3 or Q.shape[0] != N:
        raise ValueError(f"Q must be [N, H, D] with N = indptr.numel() - 1 = {N}, got {tuple(Q.shape)}")
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _need(t, n, Q.dtype)
        if t.shape != Q.shape:
            raise ValueError(f"{n} must have Q's shape {tuple(Q.shape)}, got {tuple(t.shape)}")
    _, H, D = Q.shape
    if out is None:
        out = torch.empty_like(Q)
    else:
        _need(out, "out", Q.dtype)
        if out.shape != Q.shape:
            raise ValueError(f"out must have Q's shape {tuple(Q.shape)}, got {tuple(out.shape)}")
    if lse is None:
        lse = torch.empty((N, H), dtype=torch.float32, device=Q.device)
    else:
        _need(lse, "lse", torch.float32)
        if tuple(lse.shape) != (N, H):
            raise ValueError(f"lse must be [{N}, {H}], got {tuple(lse.shape)}")
    for n, t in (("indptr", indptr), ("indices", indices), ("K", K), ("V", V), ("out", out),
                 ("lse", lse)):
        if t.device != Q.device:
            raise ValueError(f"{n} is on {t.device}, Q on {Q.device}")
    _check(_lib().gt_attn_fwd_noalloc(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), N,
                                      indices.numel(), H, D, _dtype_code(Q), _ptr(out), _ptr(lse),
                                      _stream(stream)), "gt_attn_fwd_noalloc")
    return out, lse


def noalloc_device_error(stream=None) -> int:
    """Read and clear gt_attn_fwd_noalloc's device range-check word on the
    current device (0 = no failed check).  Synchronises the stream."""
    code = ctypes.c_int32()
    st = _lib().sga_noalloc_read_device_error(_stream(stream), ctypes.byref(code))
    if st not in (SGA_OK, SGA_EDEVICE_CHECK):
        _check(st, "sga_noalloc_read_device_error")
    return int(code.value)


# ----------------------------------------------------------------------- GATv2

def _gatv2_inputs(plan, X, W_l, W_r, a):
    _need(X, "X", plan.dtype, plan.N * plan.F, plan.N, plan)
    for n, t in (("W_l", W_l), ("W_r", W_r)):
        _need(t, n, plan.dtype, plan.F * plan.H * plan.D, plan.F, plan)
    _need(a, "a", plan.dtype, plan.H * plan.D, None, plan)


def gatv2_fwd(plan: Plan, X, W_l, W_r, a, slope: float = 0.2, FL=None, FR=None, out=None,
              lse=None, stream=None):
    """(FL, FR, out, lse): FL = X W_l and FR = X W_r as [N,H,D], out [N,H,D], lse [N,H]."""
    _gatv2_inputs(plan, X, W_l, W_r, a)
    shape = (plan.N, plan.H, plan.D)
    FL = torch.empty(shape, dtype=X.dtype, device=X.device) if FL is None else FL
    FR = torch.empty(shape, dtype=X.dtype, device=X.device) if FR is None else FR
    out = torch.empty(shape, dtype=X.dtype, device=X.device) if out is None else out
    lse = torch.empty(shape[:2], dtype=torch.float32, device=X.device) if lse is None else lse
    for n, t in (("FL", FL), ("FR", FR), ("out", out)):
        _node(t, n, plan)
    _head(lse, "lse", plan)
    _check(_lib().gatv2_fwd(plan.handle, *plan._graph()[:2], _ptr(X), _ptr(W_l), _ptr(W_r),
                            _ptr(a), plan.N, plan.E, plan.F, plan.H, plan.D, float(slope), plan.dt,
                            _ptr(FL), _ptr(FR), _ptr(out), _ptr(lse), _stream(stream)),
           "gatv2_fwd")
    return FL, FR, out, lse


def gatv2_bwd(plan: Plan, X, W_l, W_r, a, FL, FR, out, lse, dOut, slope: float = 0.2,
              dX=None, dW_l=None, dW_r=None, da=None, stream=None):
    """(dX, dW_l, dW_r, da)."""
    _gatv2_inputs(plan, X, W_l, W_r, a)
    for n, t in (("FL", FL), ("FR", FR), ("out", out), ("dOut", dOut)):
        _node(t, n, plan)
    _head(lse, "lse", plan)
    dX = torch.empty_like(X) if dX is None else dX
    dW_l = torch.empty_like(W_l) if dW_l is None else dW_l
    dW_r = torch.empty_like(W_r) if dW_r is None else dW_r
    da = torch.empty_like(a) if da is None else da
    _gatv2_inputs(plan, dX, dW_l, dW_r, da)
    _check(_lib().gatv2_bwd(plan.handle, *plan._graph()[:2], _ptr(X), _ptr(W_l), _ptr(W_r),
                            _ptr(a), _ptr(FL), _ptr(FR), _ptr(out), _ptr(lse), _ptr(dOut), plan.N,
                            plan.E, plan.F, plan.H, plan.D, float(slope), plan.dt, _ptr(dX),
                            _ptr(dW_l), _ptr(dW_r), _ptr(da), _stream(stream)), "gatv2_bwd")
    return dX, dW_l, dW_r, da


# ------------------------------------------------------------ graph reordering

def reorder(indptr, indices, method: str = "rcm", stream=None):
    """perm [N] int32 on the device: the new id of every node under the
    ordering ("rcm": reverse Cuthill-McKee, "degree": descending in-degree).
    The library checks the CSR on the device (SgaError if it is not valid)."""
    _need(indptr, "indptr", torch.int32)
    _need(indices, "indices", torch.int32)
    if indptr.numel() < 1 or indices.device != indptr.device:
        raise ValueError("indptr needs N + 1 entries, on the device of indices")
    N = indptr.numel() - 1
    perm = torch.empty(max(N, 1), dtype=torch.int32, device=indptr.device)
    code = {"degree": SGA_ORDER_DEGREE, "rcm": SGA_ORDER_RCM}[method]
    _check(_lib().sga_reorder(_ptr(indptr), _ptr(indices), N, indices.numel(), code, _ptr(perm),
                              _stream(stream)), "sga_reorder")
    return perm[:N]


def relabel_csr(indptr, indices, perm, stream=None):
    """(new_indptr, new_indices): row perm[v] = old row v, sources mapped.  The
    library checks the CSR and that perm is a permutation (SgaError if not)."""
    for n, t in (("indptr", indptr), ("indices", indices), ("perm", perm)):
        _need(t, n, torch.int32)
    if indptr.numel() < 1 or not (indices.device == perm.device == indptr.device):
        raise ValueError("indptr needs N + 1 entries; indptr, indices and perm on one device")
    N = indptr.numel() - 1
    _need(perm, "perm", torch.int32, N)
    new_ptr = torch.empty_like(indptr)
    new_idx = torch.empty_like(indices)
    _check(_lib().sga_relabel_csr(_ptr(indptr), _ptr(indices), N, indices.numel(), _ptr(perm),
                                  _ptr(new_ptr), _ptr(new_idx), _stream(stream)), "sga_relabel_csr")
    return new_ptr, new_idx


def permute_rows(x, perm, inverse: bool = False, out=None, stream=None):
    """Rows of a node tensor under perm: out[perm[v]] = x[v] (inverse:
    out[v] = x[perm[v]]).  perm should be a permutation of 0..N-1; rows whose
    entry lies outside [0, N) are skipped, not reported."""
    _need(x, "x")
    N = x.shape[0] if x.dim() else 0
    _need(perm, "perm", torch.int32, N)
    out = torch.empty_like(x) if out is None else out
    _need(out, "out", x.dtype, x.numel(), N)
    if not (perm.device == out.device == x.device):
        raise ValueError("x, perm and out must be on one device")
    row_bytes = x.numel() // max(N, 1) * x.element_size()
    _check(_lib().sga_permute_rows(_ptr(x), N, row_bytes, _ptr(perm), 1 if inverse else 0,
                                   _ptr(out), _stream(stream)), "sga_permute_rows")
    return out


# ------------------------------------------------------------------------- GAT

def gat_attn_fwd(plan: Plan, Fv, el, er, slope: float = 0.2, out=None, lse=None, stream=None):
    """GAT edge attention: (out [N,H,D], lse [N,H]) from the projected features
    Fv [N,H,D] and the score halves el, er [N,H] float32.  The plan must be
    built with layer=SGA_LAYER_GAT."""
    _node(Fv, "Fv", plan)
    _head(el, "el", plan)
    _head(er, "er", plan)
    out = torch.empty_like(Fv) if out is None else out
    lse = torch.empty((plan.N, plan.H), dtype=torch.float32, device=Fv.device) if lse is None else lse
    _node(out, "out", plan)
    _head(lse, "lse", plan)
    _check(_lib().gat_attn_fwd(plan.handle, *plan._graph()[:2], _ptr(Fv), _ptr(el), _ptr(er), plan.N,
                               plan.E, plan.H, plan.D, float(slope), plan.dt, _ptr(out), _ptr(lse),
                               _stream(stream)), "gat_attn_fwd")
    return out, lse


def gat_attn_bwd(plan: Plan, Fv, el, er, out, lse, dOut, slope: float = 0.2, stream=None):
    """(dFv, del, der): the value-path gradient of Fv and the gradients of the
    two score halves."""
    for n, t in (("Fv", Fv), ("out", out), ("dOut", dOut)):
        _node(t, n, plan)
    for n, t in (("el", el), ("er", er), ("lse", lse)):
        _head(t, n, plan)
    dFv = torch.empty_like(Fv)
    de_l = torch.empty_like(el)
    de_r = torch.empty_like(er)
    _check(_lib().gat_attn_bwd(plan.handle, *plan._graph()[:2], _ptr(Fv), _ptr(el), _ptr(er),
                               _ptr(out), _ptr(lse), _ptr(dOut), plan.N, plan.E, plan.H, plan.D,
                               float(slope), plan.dt, _ptr(dFv), _ptr(de_l), _ptr(de_r),
                               _stream(stream)), "gat_attn_bwd")
    return dFv, de_l, de_r


# ------------------------------------------------------- min / max aggregation

def agg_minmax_fwd(plan: Plan, X, op: str = "max", out=None, arg=True, mask=True, stream=None):
    """(out, arg, mask): out [N,H,D] = elementwise max (or min) of the sources'
    rows; arg [N,H,D] int32 = the winning source (first edge on ties, -1 for
    an empty row); mask [E, R] uint8 = the win mask the backward takes.
    ``arg``/``mask`` = False skips that output (None in its place), a tensor
    is filled in place.  ``plan`` must be built with layer=SGA_LAYER_MINMAX."""
    _node(X, "X", plan)
    out = torch.empty_like(X) if out is None else out
    _node(out, "out", plan)
    if arg is True:
        arg = torch.empty(X.shape, dtype=torch.int32, device=X.device)
    elif arg is False:
        arg = None
    if arg is not None:
        _node(arg, "arg", plan, torch.int32)
    mask_bytes = int(_lib().sga_agg_mask_bytes(plan.handle))
    if mask is True:
        mask = torch.empty(mask_bytes, dtype=torch.uint8, device=X.device)
    elif mask is False:
        mask = None
    if mask is not None:
        _need(mask, "mask", torch.uint8, mask_bytes, None, plan)
    code = {"max": SGA_AGG_MAX, "min": SGA_AGG_MIN}[op]
    _check(_lib().agg_minmax_fwd(plan.handle, *plan._graph()[:2], _ptr(X), plan.N, plan.E, plan.H,
                                 plan.D, plan.dt, code, _ptr(out), _ptr(arg), _ptr(mask),
                                 _stream(stream)), "agg_minmax_fwd")
    return out, arg, mask


def agg_minmax_bwd(plan: Plan, mask, dOut, dX=None, stream=None):
    """dX [N,H,D]: dOut gathered into the winning sources of the forward."""
    _need(mask, "mask", torch.uint8, int(_lib().sga_agg_mask_bytes(plan.handle)), None, plan)
    _node(dOut, "dOut", plan)
    dX = torch.empty_like(dOut) if dX is None else dX
    _node(dX, "dX", plan)
    _check(_lib().agg_minmax_bwd(plan.handle, _ptr(mask), _ptr(dOut), plan.N, plan.H, plan.D,
                                 plan.dt, _ptr(dX), _stream(stream)), "agg_minmax_bwd")
    return dX


# -------------------------------------------------------------- autograd layers

class GTAttention(torch.autograd.Function):
    """Graph Transformer edge attention as an autograd function:
    ``out = GTAttention.apply(Q, K, V, plan)``."""

    @staticmethod
    def forward(ctx, Q, K, V, plan):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        out, lse = gt_attn_fwd(plan, Q, K, V)
        ctx.plan = plan
        ctx.save_for_backward(Q, K, V, out, lse)
        return out

    @staticmethod
    def backward(ctx, dOut):
        Q, K, V, out, lse = ctx.saved_tensors
        dQ, dK, dV = gt_attn_bwd(ctx.plan, Q, K, V, out, lse, dOut.contiguous())
        return dQ, dK, dV, None


class GTBiasAttention(torch.autograd.Function):
    """Graph Transformer edge attention with a per-edge, per-head score bias
    (e.g. projected edge features), as an autograd function:
    ``out = GTBiasAttention.apply(Q, K, V, bias, plan)`` with bias [E, H]
    float32 in CSR edge order; the plan needs edge_bias=True."""

    @staticmethod
    def forward(ctx, Q, K, V, bias, plan):
        Q, K, V, bias = Q.contiguous(), K.contiguous(), V.contiguous(), bias.contiguous()
        out, lse = gt_attn_bias_fwd(plan, Q, K, V, bias)
        ctx.plan = plan
        ctx.save_for_backward(Q, K, V, bias, out, lse)
        return out

    @staticmethod
    def backward(ctx, dOut):
        Q, K, V, bias, out, lse = ctx.saved_tensors
        dQ, dK, dV, dbias = gt_attn_bias_bwd(ctx.plan, Q, K, V, bias, out, lse, dOut.contiguous())
        return dQ, dK, dV, dbias, None


class MinMaxAggregation(torch.autograd.Function):
    """Min / max neighbourhood aggregation:
    ``out = MinMaxAggregation.apply(X, plan, "max")``."""

    @staticmethod
    def forward(ctx, X, plan, op="max"):
        out, _, mask = agg_minmax_fwd(plan, X.contiguous(), op, arg=False)
        ctx.plan = plan
        ctx.save_for_backward(mask)
        return out

    @staticmethod
    def backward(ctx, dOut):
        (mask,) = ctx.saved_tensors
        return agg_minmax_bwd(ctx.plan, mask, dOut.contiguous()), None, None


class GATEdgeAttention(torch.autograd.Function):
    """GAT edge stage as an autograd function:
    ``out = GATEdgeAttention.apply(Fv, el, er, plan, slope)``; with
    Fv = X @ W and el, er the per-node dots with the attention vector's two
    halves (ordinary torch ops around it), this is the GAT layer."""

    @staticmethod
    def forward(ctx, Fv, el, er, plan, slope=0.2):
        Fv, el, er = Fv.contiguous(), el.contiguous(), er.contiguous()
        out, lse = gat_attn_fwd(plan, Fv, el, er, slope)
        ctx.plan, ctx.slope = plan, slope
        ctx.save_for_backward(Fv, el, er, out, lse)
        return out

    @staticmethod
    def backward(ctx, dOut):
        Fv, el, er, out, lse = ctx.saved_tensors
        dFv, de_l, de_r = gat_attn_bwd(ctx.plan, Fv, el, er, out, lse, dOut.contiguous(), ctx.slope)
        return dFv, de_l, de_r, None, None


class GATv2Attention(torch.autograd.Function):
    """GATv2 layer (projections + edge attention):
    ``out = GATv2Attention.apply(X, W_l, W_r, a, plan, slope)``."""

    @staticmethod
    def forward(ctx, X, W_l, W_r, a, plan, slope=0.2):
        X, W_l, W_r, a = (t.contiguous() for t in (X, W_l, W_r, a))
        FL, FR, out, lse = gatv2_fwd(plan, X, W_l, W_r, a, slope)
        ctx.plan, ctx.slope = plan, slope
        ctx.save_for_backward(X, W_l, W_r, a, FL, FR, out, lse)
        return out

    @staticmethod
    def backward(ctx, dOut):
        X, W_l, W_r, a, FL, FR, out, lse = ctx.saved_tensors
        dX, dWl, dWr, da = gatv2_bwd(ctx.plan, X, W_l, W_r, a, FL, FR, out, lse,
                                     dOut.contiguous(), ctx.slope)
        return dX, dWl, dWr, da, None, None
