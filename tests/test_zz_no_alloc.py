"""The no-allocation forward (moba_attn_fwd_noalloc) against moba_attn_fwd.

Some callers cannot allocate device memory: a memory manager that owns the
whole device, or a serving loop that must not allocate on its latency path.
This entry point runs the same forward with its scratch in the library's static
device array.  The file is collected last on purpose, so that a run stopping at
the first failure has run every other test before this one."""
import ctypes

import pytest
import torch

from long_context_sparse_moba_gb300 import ops, workloads


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
    """Two calls in a row share the static array, which keeps the previous
    call's contents.  The first call is the larger problem (more selections,
    longer lists), so a later call that read a scratch area it never rewrote
    would see the first call's values; the second call uses other inputs and
    another top-k.  Both must equal moba_attn_fwd bit for bit (the same kernels
    run in the same order, and the forward is deterministic)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [(workloads.custom((4096, 4096), 4, 128, 256, topk=6, seed=21), 6),
             (workloads.custom((4096, 4096), 4, 128, 512, topk=3, seed=22), 3)]
    for w, topk in cases:
        assert ops.workspace_size(w.B, w.H, w.S, w.D, w.block_size, topk) <= ops.noalloc_capacity()
    for call, (w, topk) in enumerate(cases):
        inp = workloads.make_inputs(w, device="cuda")
        ref_out, ref_lse = ops.attn_fwd(inp.q, inp.k, inp.v, w.block_size, topk)
        out = torch.full_like(inp.q, float("nan"))
        lse = torch.full((w.B, w.H, w.S), float("nan"), dtype=torch.float32, device="cuda")
        ops.attn_fwd_noalloc(inp.q, inp.k, inp.v, w.block_size, topk, out, lse)
        assert ops.get_status() == ops.MOBA_OK
        assert torch.equal(out, ref_out), call
        assert torch.equal(lse, ref_lse), call
