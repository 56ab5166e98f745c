"""Seeded input generators: determinism, well-formed CSR, degree laws."""
import numpy as np
import pytest

from sparse_graph_attention_csr_gb300 import synth


def check_csr(indptr, indices, N):
    assert indptr.dtype == np.int32 and indices.dtype == np.int32
    assert indptr[0] == 0 and len(indptr) == N + 1 and indptr[-1] == len(indices)
    assert np.all(np.diff(indptr) >= 1)                       # self-loop everywhere
    for i in np.random.default_rng(0).integers(0, N, 200):
        row = indices[indptr[i]:indptr[i + 1]]
        assert np.all(np.diff(row) > 0)                       # ascending, no duplicates
        assert i in row
    assert indices.min() >= 0 and indices.max() < N


@pytest.mark.parametrize("key", [1, 2, 3, 4, 5])
def test_small_workloads_deterministic_and_wellformed(key):
    w = synth.small_workload(key)
    a = synth.make_graph(w)
    b = synth.make_graph(w)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    check_csr(*a, w.N)


def test_degree_laws():
    s = synth.degree_summary(synth.make_graph(synth.WORKLOADS[1])[0])
    assert 8.0 < s["mean"] < 10.5                            # ER mean 8 + self-loop
    s = synth.degree_summary(synth.make_graph(synth.small_workload(3))[0])
    assert 6 <= s["median"] <= 10 and s["max"] > 20 * s["median"]   # lognormal + hub
    s = synth.degree_summary(synth.make_graph(synth.small_workload(4))[0])
    assert s["max"] > 50 * s["mean"]                          # R-MAT heavy tail
    ip, ix = synth.make_graph(synth.small_workload(5))
    rows = np.repeat(np.arange(len(ip) - 1), np.diff(ip))
    intra = (rows // 256) == (ix // 256)
    assert intra.mean() > 0.85                                # community-local nonzeros


def test_inputs_rounded_and_seeded():
    import torch
    w = synth.small_workload(3)
    x = synth.gt_inputs(w, N=100)
    y = synth.gt_inputs(w, N=100)
    for k in ("Q", "K", "V", "dOut"):
        t, f = x[k]
        assert t.dtype == torch.bfloat16 and t.shape == (100, w.H, w.D)
        np.testing.assert_array_equal(f, t.to(torch.float64).numpy())
        np.testing.assert_array_equal(f, y[k][1])
    g = synth.gatv2_inputs(synth.small_workload(2), N=50)
    assert g["X"][0].shape == (50, 128) and g["W_l"][0].shape == (128, 128)
    assert g["a"][0].shape == (2, 64)
