"""Max pooling of each block's keys ("MOBA mixture of block attention for
server-side long context" §3 allows it instead of the mean): the pooled keys
are exact, and the whole forward with max pooling matches the oracle run
with max pooling."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_moba_gb300 import ops, workloads

from .parity import compare, flat, gpu_forward, gpu_select

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_moba_gb300 import build
    build.build()
    oracle.build()
    ops.lib()


@pytest.fixture
def max_pooling():
    ops.set_pooling(ops.POOL_MAX)
    try:
        yield
    finally:
        ops.set_pooling(ops.POOL_MEAN)


@pytest.mark.parametrize("seqlens,H,D,bs", [((2048,), 1, 64, 256), ((1000, 777), 3, 128, 128),
                                            ((4096,), 4, 128, 512)])
def test_max_pooled_keys_are_exact(max_pooling, seqlens, H, D, bs):
    w = workloads.custom(seqlens, H, D, bs, topk=3, seed=41)
    inp = workloads.make_inputs(w, device="cuda")
    if w.varlen:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")
        kbar = ops.kpool_varlen(inp.k, cu, bs)
    else:
        kbar = ops.kpool(inp.k, bs)
    ref = oracle.kpool(flat(inp.k).cpu(), inp.cu_seqlens, H, D, bs, pooling="max")
    assert np.array_equal(kbar.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("name,topk,rows", [("tiny", 3, None), ("train32k", 3, 4096),
                                            ("varlen", 4, 4096)])
def test_forward_with_max_pooling(max_pooling, name, topk, rows):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda")
    _, idx = gpu_select(inp, w, topk)
    out, lse = gpu_forward(inp, w, topk)
    assert ops.get_status() == ops.MOBA_OK
    host = tuple(flat(x).cpu() for x in (inp.q, inp.k, inp.v))
    kbar = oracle.kpool(host[1], inp.cu_seqlens, w.H, w.D, w.block_size, pooling="max")
    sel = None
    if rows is not None:
        sel = workloads.sample_rows(w, rows, seed=5)
    compare(w, inp, topk, out, lse, idx_gpu=idx, rows=sel, host=host, kbar=kbar)


def test_max_pooling_changes_the_selection():
    """On the 32K training shape the two poolings choose differently for a
    sizeable share of rows (so the switch is not a no-op)."""
    w = workloads.WORKLOADS["train32k"]
    inp = workloads.make_inputs(w, device="cuda")
    _, mean_idx = gpu_select(inp, w, 3)
    ops.set_pooling(ops.POOL_MAX)
    try:
        _, max_idx = gpu_select(inp, w, 3)
    finally:
        ops.set_pooling(ops.POOL_MEAN)
    differ = (mean_idx != max_idx).any(dim=-1).float().mean().item()
    assert differ > 0.05
