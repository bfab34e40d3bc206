"""The forward on host buffers (moba_attn_fwd_host): its copies in and out and
the per-input waits inside the forward change nothing in the results, which
equal the device-buffer forward's bit for bit, also when two calls run side by
side on two streams."""
import pytest
import torch

from long_context_sparse_moba_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_moba_gb300 import build
    build.build()
    ops.lib()


def host_case(w, topk):
    inp = workloads.make_inputs(w, device="cuda")
    ref_out, ref_lse = ops.attn_fwd(inp.q, inp.k, inp.v, w.block_size, topk)
    assert ops.get_status() == ops.MOBA_OK
    hq, hk, hv = (t.cpu().pin_memory() for t in (inp.q, inp.k, inp.v))
    return inp, ref_out, ref_lse, hq, hk, hv


@pytest.mark.parametrize("S,H,D,bs,topk", [(4096, 4, 128, 512, 3), (3000, 2, 64, 256, 2),
                                           (1024, 2, 128, 256, 8)])
def test_host_forward_equals_device_forward(S, H, D, bs, topk):
    w = workloads.custom((S,), H, D, bs, topk, seed=41, qkv_scale=D ** -0.5)
    inp, ref_out, ref_lse, hq, hk, hv = host_case(w, topk)
    out = torch.empty(hq.shape, dtype=torch.bfloat16).pin_memory()
    lse = torch.empty(ref_lse.shape, dtype=torch.float32).pin_memory()
    scratch = torch.empty(ops.host_scratch_size(1, H, S, D, bs, topk), dtype=torch.uint8,
                          device="cuda")
    ops.attn_fwd_host(hq, hk, hv, bs, topk, out, lse, scratch)
    assert ops.get_status() == ops.MOBA_OK  # synchronises the stream
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())


def test_two_host_forwards_side_by_side():
    w = workloads.custom((8192,), 8, 128, 512, 3, seed=42, qkv_scale=128 ** -0.5)
    inp, ref_out, ref_lse, hq, hk, hv = host_case(w, 3)
    size = ops.host_scratch_size(1, 8, 8192, 128, 512, 3)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    scratch = [torch.empty(size, dtype=torch.uint8, device="cuda") for _ in range(2)]
    outs = [torch.empty(hq.shape, dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    lses = [torch.empty(ref_lse.shape, dtype=torch.float32).pin_memory() for _ in range(4)]
    for i in range(4):  # alternate streams and scratch; calls 2 and 3 reuse them
        ops.attn_fwd_host(hq, hk, hv, 512, 3, outs[i], lses[i], scratch[i % 2],
                          stream=streams[i % 2])
    torch.cuda.synchronize()
    assert ops.get_status() == ops.MOBA_OK
    for i in range(4):
        assert torch.equal(outs[i], ref_out.cpu()) and torch.equal(lses[i], ref_lse.cpu())


def test_host_forward_refuses_short_scratch():
    w = workloads.custom((1024,), 2, 64, 256, 3, seed=43)
    inp, ref_out, ref_lse, hq, hk, hv = host_case(w, 3)
    out = torch.empty(hq.shape, dtype=torch.bfloat16)
    lse = torch.empty(ref_lse.shape, dtype=torch.float32)
    size = ops.host_scratch_size(1, 2, 1024, 64, 256, 3)
    scratch = torch.empty(size - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(Exception):
        ops.attn_fwd_host(hq, hk, hv, 256, 3, out, lse, scratch)
