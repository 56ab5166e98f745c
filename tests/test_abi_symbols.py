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


def test_header_is_plain_c_and_links_from_c(tmp_path):
    """A C11 program (strict, warnings as errors) includes the header, takes
    the address of every declared function, links against the library and
    runs host-side rejections that need no GPU: the boundary is usable from C,
    not only through ctypes."""
    import shutil
    import subprocess

    import pytest

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from sparse_graph_attention_csr_gb300 import build
    lib = build.build()
    names = declared_functions()
    table = ",\n    ".join(f"(fn)&{n}" for n in names)
    src = tmp_path / "abi.c"
    src.write_text(f"""#include <stdio.h>
#include <string.h>
#include "sga.h"
typedef void (*fn)(void);
static const fn every[] = {{
    {table}
}};
int main(void) {{
    size_t i;
    sga_plan *p = (sga_plan *)0;
    for (i = 0; i < sizeof every / sizeof every[0]; ++i)
        if (!every[i]) return 10;
    if (strcmp(sga_status_string(SGA_OK), "ok") != 0) return 11;
    /* null indptr, unsupported D, null handle: rejected before any CUDA call */
    if (sga_plan_create(NULL, NULL, 4, 4, 1, 32, SGA_F32, NULL, NULL, &p) != SGA_EINVAL) return 12;
    if (p != NULL) return 13;
    if (sga_plan_create((const int32_t *)4096, (const int32_t *)4096, 4, 4, 1, 48, SGA_BF16, NULL,
                        NULL, &p) != SGA_EUNSUPPORTED) return 14;
    if (sga_plan_create((const int32_t *)4096, (const int32_t *)4096, 4, 4, 1, 32, SGA_F32, NULL,
                        NULL, NULL) != SGA_EINVAL) return 15;
    if (sga_plan_workspace_bytes(NULL) != 0) return 16;
    sga_plan_destroy(NULL);
    printf("%u functions\\n", (unsigned)(sizeof every / sizeof every[0]));
    return 0;
}}
""")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
           os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", libdir, "-lsga",
           f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == f"{len(names)} functions"
