"""The no-allocation forward (moba_attn_fwd_noalloc) against moba_attn_fwd.

Some callers cannot allocate device memory (a memory manager owns the whole
device, or the serving loop must not allocate); this entry point runs the same
forward with its scratch in the library's static device array.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from long_context_sparse_moba_gb300 import ops, workloads

from .parity import LSE_MAX, OUT_MAX, OUT_MEAN


@pytest.fixture(scope="module")
def lib():
    from long_context_sparse_moba_gb300 import build
    build.build()
    return ops.lib()


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    need = lib.moba_attn_fwd_workspace_size(1, 32, 32768, 128, 512, 3)
    assert need > ops.noalloc_capacity() == 64 << 20
    fake = ctypes.c_void_p(0x10000)  # rejected before any launch
    rc = lib.moba_attn_fwd_noalloc(fake, fake, fake, fake, fake, 1, 32, 32768, 128, 512, 3, None)
    assert rc == ops.MOBA_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = workloads.custom((4096, 4096), 4, 128, 512, topk=3, seed=21)
    assert ops.workspace_size(2, 4, 4096, 128, 512, 3) <= ops.noalloc_capacity()
    inp = workloads.make_inputs(w, device="cuda")
    ref_out, ref_lse = ops.attn_fwd(inp.q, inp.k, inp.v, 512, 3)
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        out = torch.full_like(inp.q, float("nan"))
        lse = torch.full((2, 4, 4096), float("nan"), dtype=torch.float32, device="cuda")
        ops.attn_fwd_noalloc(inp.q, inp.k, inp.v, 512, 3, out, lse)
        assert ops.get_status() == ops.MOBA_OK
        err = (out.float() - ref_out.float()).abs()
        lerr = (lse - ref_lse).abs()
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all(), call
        assert err.max().item() <= OUT_MAX and err.mean().item() <= OUT_MEAN, call
        assert lerr.max().item() <= LSE_MAX, call
