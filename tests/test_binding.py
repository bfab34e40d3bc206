"""The Python binding checks its tensors before anything reaches the library:
a CPU tensor, a wrong dtype or a non-contiguous view is refused with
ValueError (CPU only; no library call is made)."""
import pytest
import torch

from long_context_sparse_moba_gb300 import ops


def bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def test_cpu_tensors_are_refused_before_the_library():
    q = bf(1, 128, 2, 64)
    with pytest.raises(ValueError):
        ops.attn_fwd(q, q, q, 64, 3)
    with pytest.raises(ValueError):
        ops.attn_bwd(q, q, q, q, torch.zeros(1, 2, 128), q, 64, 3)
    with pytest.raises(ValueError):
        ops.kpool(q, 64)
    with pytest.raises(ValueError):
        ops.decode_fwd(bf(1, 2, 64), q, q, torch.zeros(2, 2, 64), torch.ones(1, dtype=torch.int32),
                       64, 3)


def test_wrong_dtype_and_layout_are_refused():
    q32 = torch.zeros(1, 128, 2, 64)
    with pytest.raises(ValueError):
        ops.attn_fwd(q32, q32, q32, 64, 3)
    qt = bf(1, 2, 128, 64).transpose(1, 2)       # [1, 128, 2, 64] view, not contiguous
    with pytest.raises(ValueError):
        ops.attn_fwd(qt, qt, qt, 64, 3)
