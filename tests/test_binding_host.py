"""Checks of the Python binding that run before any device call (CPU only)."""
import pytest
import torch

import sparse_graph_attention_csr_gb300 as sga


def test_plan_refuses_dtypes_the_layers_do_not_compute_in():
    """Only float32 and bfloat16 layers exist; any other dtype is refused before
    the plan is built (float16 tensors must not be read as bfloat16)."""
    ip, ix = torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)
    for dt in (torch.float16, torch.float64, torch.int32):
        with pytest.raises(TypeError):
            sga.Plan(ip, ix, 1, 32, dt)


def test_host_tensors_are_refused():
    ip, ix = torch.zeros(2, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sga.Plan(ip, ix, 1, 32, torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        sga.gt_attn_fwd_noalloc(ip, ix, *(torch.zeros(1, 1, 32) for _ in range(3)))
    with pytest.raises(ValueError, match="CUDA tensor"):
        sga.reorder(ip, ix)
