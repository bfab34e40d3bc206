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


@pytest.mark.parametrize("seqlens,H,D,bs", [((2048,), 1, 64, 256), ((1000, 777), 3, 128, 128),
                                            ((4096,), 4, 128, 512)])
def test_max_pooled_keys_are_exact(seqlens, H, D, bs):
    w = workloads.custom(seqlens, H, D, bs, topk=3, seed=41)
    inp = workloads.make_inputs(w, device="cuda")
    if w.varlen:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")
        kbar = ops.kpool_varlen(inp.k, cu, bs, pooling=ops.POOL_MAX)
    else:
        kbar = ops.kpool(inp.k, bs, pooling=ops.POOL_MAX)
    ref = oracle.kpool(flat(inp.k).cpu(), inp.cu_seqlens, H, D, bs, pooling="max")
    assert np.array_equal(kbar.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("name,topk,rows", [("tiny", 3, None), ("train32k", 3, 4096),
                                            ("varlen", 4, 4096)])
def test_forward_with_max_pooling(name, topk, rows):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, device="cuda")
    _, idx_gate = gpu_select(inp, w, topk, pooling=ops.POOL_MAX)
    out, lse, idx = gpu_forward(inp, w, topk, with_idx=True, pooling=ops.POOL_MAX)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(idx, idx_gate)
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
    _, max_idx = gpu_select(inp, w, 3, pooling=ops.POOL_MAX)
    differ = (mean_idx != max_idx).any(dim=-1).float().mean().item()
    assert differ > 0.05


def test_two_threads_two_streams_mean_and_max():
    """Two host threads, each on its own stream, run the forward at the same
    time with different pooling options; each result matches the oracle run
    with its own pooling (the library holds no process-wide setting)."""
    import threading
    w = workloads.custom((8192,), 4, 128, 512, topk=3, seed=43)
    inp = workloads.make_inputs(w, device="cuda")
    torch.cuda.synchronize()
    results, errors = {}, []

    def run(pool):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                outs = []
                for _ in range(4):  # several calls so that the two streams overlap
                    outs.append(gpu_forward(inp, w, 3, with_idx=True, stream=st, pooling=pool))
            st.synchronize()
            results[pool] = outs
        except Exception as e:  # noqa: BLE001 -- reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(p,)) for p in (ops.POOL_MEAN, ops.POOL_MAX)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert ops.get_status() == ops.MOBA_OK
    host = tuple(flat(x).cpu() for x in (inp.q, inp.k, inp.v))
    rows = workloads.sample_rows(w, 2048, seed=9)
    for pool, name in ((ops.POOL_MEAN, "mean"), (ops.POOL_MAX, "max")):
        kbar = oracle.kpool(host[1], inp.cu_seqlens, w.H, w.D, w.block_size, pooling=name)
        out0, lse0, idx0 = results[pool][0]
        for out, lse, idx in results[pool][1:]:
            assert torch.equal(out, out0) and torch.equal(idx, idx0)
        compare(w, inp, 3, out0, lse0, idx_gpu=idx0, rows=rows, host=host, kbar=kbar)
    assert not torch.equal(results[ops.POOL_MEAN][0][2], results[ops.POOL_MAX][0][2])
