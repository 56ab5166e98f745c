"""Shared helpers for the parity tests (comparison against the fp64 oracle)."""
import numpy as np
import torch

# Tolerances stated by the workloads: fp32 max-abs 1e-5; bf16 inputs with fp32
# accumulation: |gpu - oracle| <= 2e-2 + 1e-2 |oracle|, elementwise.
TOL = {"f32": (1e-5, 0.0), "bf16": (2e-2, 1e-2)}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def compare(gpu, ref, dtype: str, name: str = "", atol=None, rtol=None, norm=0.0, slack=None):
    """Elementwise |gpu - ref| <= atol + rtol |ref| + norm max|ref| (infinities
    must match).  ``norm`` serves sums over many nodes, whose rounding error
    scales with the size of the sum's terms rather than with each result.
    ``slack`` (same shape as ref) widens the bound where the oracle reports
    that several results are correct (undecided LeakyReLU branches)."""
    a0, r0 = TOL[dtype]
    atol = a0 if atol is None else atol
    rtol = r0 if rtol is None else rtol
    g = to_np(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    inf = np.isinf(r)
    assert np.array_equal(np.isinf(g), inf) and np.array_equal(g[inf], r[inf]), \
        f"{name}: infinities differ"
    assert not np.isnan(g).any(), f"{name}: NaN in GPU result"
    fin = ~inf
    err = np.abs(g[fin] - r[fin])
    bound = atol + rtol * np.abs(r[fin]) + (norm * np.abs(r[fin]).max() if err.size else 0.0)
    if slack is not None:
        bound = bound + np.asarray(slack, dtype=np.float64)[fin]
    bad = int((err > bound).sum())
    maxabs = float(err.max()) if err.size else 0.0
    assert bad == 0, f"{name}: {bad}/{err.size} outside tolerance, max abs err {maxabs:.3e}"
    return maxabs


def dev(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().cuda()
