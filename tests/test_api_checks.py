"""The Python binding refuses tensors the library cannot read as the problem's contiguous device arrays
before any library call: here, host tensors (no GPU needed)."""

import pytest
import torch

import gated_delta_rule_38_gb300 as gdr


def _host_inputs(B=1, T=8, H=2, D=128):
    q = torch.zeros(B, T, H, D, dtype=torch.bfloat16)
    g = torch.zeros(B, T, H, dtype=torch.bfloat16)
    return q, q.clone(), q.clone(), g, g.clone()


def test_host_tensors_are_refused():
    q, k, v, g, beta = _host_inputs()
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdr.chunk_gated_delta_rule_fwd(q, k, v, g, beta)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdr.recurrent_gated_delta_rule(q, k, v, g, beta)
    A = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdr.chunk_gated_delta_rule_bwd(q, k, v, g.float(), beta, A, v.clone())
    with pytest.raises(ValueError, match="CUDA tensor"):
        gdr.prepare_chunks(torch.tensor([0, 8], dtype=torch.int32), total_tokens=8)
