"""The C-ABI library builds for sm_103a, loads, and exports every function
include/sga.h declares (no compute call: this runs without a GPU)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "sga.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("sga_plan_create", "sga_plan_workspace_bytes", "sga_plan_set_workspace",
                     "sga_plan_destroy", "gt_attn_fwd", "gt_attn_bwd", "gatv2_fwd", "gatv2_bwd",
                     "sga_status_string", "sga_read_device_error"):
        assert required in names


def test_library_loads_and_exports_every_symbol():
    from sparse_graph_attention_csr_gb300 import build
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    lib.sga_status_string.restype = ctypes.c_char_p
    assert lib.sga_status_string(0) == b"ok"


def test_plan_create_rejects_bad_arguments_without_a_device():
    """Host-side checks run before any CUDA call."""
    import sparse_graph_attention_csr_gb300 as sga
    lib = sga.load_library()
    out = ctypes.c_void_p()
    dummy = ctypes.c_void_p(4096)
    # unsupported head dim
    assert lib.sga_plan_create(dummy, dummy, 4, 4, 1, 48, 0, None, None, ctypes.byref(out)) == sga.SGA_EUNSUPPORTED
    # H*D above 1024
    assert lib.sga_plan_create(dummy, dummy, 4, 4, 16, 128, 0, None, None, ctypes.byref(out)) == sga.SGA_EUNSUPPORTED
    # misaligned indptr
    assert lib.sga_plan_create(ctypes.c_void_p(4097), dummy, 4, 4, 1, 32, 0, None, None, ctypes.byref(out)) == sga.SGA_EINVAL
    # negative sizes
    assert lib.sga_plan_create(dummy, dummy, -1, 4, 1, 32, 0, None, None, ctypes.byref(out)) == sga.SGA_EINVAL
    # null output handle
    assert lib.sga_plan_create(dummy, dummy, 4, 4, 1, 32, 0, None, None, None) == sga.SGA_EINVAL
    # compute calls without a plan
    assert lib.gt_attn_fwd(None, dummy, dummy, dummy, dummy, dummy, 4, 4, 1, 32, 0, dummy, dummy, None) == sga.SGA_EINVAL
