"""Parity of the CUDA path (through the C ABI) with the CPU oracle."""
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


def run_case(w, topk, rows=None, device="cuda", **options):
    """The forward on one workload, its selection read back through idx_out and
    checked (with the outputs) against the oracle; the standalone gate entry
    point must select the same blocks."""
    inp = workloads.make_inputs(w, device=device)
    kbar_g, idx_gate = gpu_select(inp, w, topk)
    out, lse, idx = gpu_forward(inp, w, topk, with_idx=True, **options)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(idx, idx_gate)
    return inp, kbar_g, idx, out, lse, compare(w, inp, topk, out, lse, idx_gpu=idx, rows=rows)


# ---------------------------------------------------------------------------
# per-kernel parity
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seqlens,H,D,bs", [((2048,), 1, 64, 256), ((1000, 777), 3, 128, 128),
                                            ((4096,), 4, 128, 512)])
def test_kpool_matches_oracle(seqlens, H, D, bs):
    w = workloads.custom(seqlens, H, D, bs, topk=3, seed=11)
    inp = workloads.make_inputs(w, device="cuda")
    if w.varlen:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")
        kbar = ops.kpool_varlen(inp.k, cu, bs)
    else:
        kbar = ops.kpool(inp.k, bs)
    ref = oracle.kpool(flat(inp.k).cpu(), inp.cu_seqlens, H, D, bs)
    got = kbar.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("topk", [1, 2, 3, 5, 8])
def test_gate_matches_oracle(topk):
    w = workloads.custom((3000, 5000), 2, 128, 128, topk=topk, seed=12)
    inp = workloads.make_inputs(w, device="cuda")
    _, idx = gpu_select(inp, w, topk)
    q, k = flat(inp.q).cpu(), flat(inp.k).cpu()
    tok, head = oracle.all_rows(w.total, w.H)
    ref = oracle.moba_rows(q, k, flat(inp.v).cpu(), inp.cu_seqlens, w.H, w.D, w.block_size, topk,
                           tok, head)
    gi = idx.cpu().numpy().reshape(-1, topk)
    differ = (gi != ref["idx"]).any(axis=1)
    assert not (differ & (ref["gap"] >= 1e-5)).any()


# ---------------------------------------------------------------------------
# end-to-end parity on the workloads
# ---------------------------------------------------------------------------

def test_tiny_workload_all_rows():
    w = workloads.WORKLOADS["tiny"]
    *_, st = run_case(w, 3)
    print("tiny", st)


@pytest.mark.parametrize("topk", [3, 64])
def test_train32k_sampled(topk):
    w = workloads.WORKLOADS["train32k"]
    rows = workloads.sample_rows(w, 4096)
    *_, st = run_case(w, topk, rows=rows)
    print("train32k", topk, st)


def test_long128k_sampled_with_needles():
    w = workloads.WORKLOADS["long128k"]
    inp = workloads.make_inputs(w, device="cuda")
    rows = workloads.sample_rows(w, 4096, needle_queries=inp.needle_queries)
    out, lse, idx = gpu_forward(inp, w, 3, with_idx=True)
    st = compare(w, inp, 3, out, lse, idx_gpu=idx, rows=rows)
    print("long128k", st)


def test_prefill1m_sampled():
    w = workloads.WORKLOADS["prefill1m"]
    rows = workloads.sample_rows(w, 4096)
    *_, st = run_case(w, 3, rows=rows)
    print("prefill1m", st)


@pytest.mark.parametrize("topk", [1, 2, 3, 4, 8])
def test_varlen_sampled(topk):
    w = workloads.WORKLOADS["varlen"]
    rows = workloads.sample_rows(w, 4096)
    *_, st = run_case(w, topk, rows=rows)
    print("varlen", topk, st)


# ---------------------------------------------------------------------------
# edge cases: tiny / ragged sizes, k >= n, k = 1, several sequences and heads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seqlens,H,D,bs,topk", [
    ((1,), 1, 64, 64, 3),          # a single token
    ((63,), 2, 64, 64, 3),         # one partial block
    ((65,), 1, 128, 64, 3),        # tail block with one token
    ((64 * 5,), 2, 128, 64, 2),    # several tiles, n > k
    ((700,), 3, 64, 64, 4),        # ragged tail, many blocks
    ((300,), 1, 128, 64, 1),       # top-k 1: own block only
    ((512,), 2, 128, 128, 4),      # top-k == number of blocks (dense)
    ((512,), 2, 64, 128, 9),       # top-k > number of blocks (dense)
    ((200, 1, 64, 129), 2, 128, 64, 3),  # varlen with tiny sequences
    ((4096, 4096), 2, 128, 256, 3),      # B = 2, fixed length
    ((4096,), 2, 128, 64, 32),     # 31 past slots
])
def test_edge_cases(seqlens, H, D, bs, topk):
    w = workloads.custom(seqlens, H, D, bs, topk=topk, seed=13)
    *_, st = run_case(w, topk)
    print(seqlens, st)


def test_deterministic_and_workspace_variant():
    w = workloads.custom((8192,), 4, 128, 512, topk=3, seed=14)
    inp = workloads.make_inputs(w, device="cuda")
    o1, l1 = ops.attn_fwd(inp.q, inp.k, inp.v, 512, 3)
    o2, l2 = ops.attn_fwd(inp.q, inp.k, inp.v, 512, 3)
    ws = torch.empty(ops.workspace_size(1, 4, 8192, 128, 512, 3), dtype=torch.uint8,
                     device="cuda")
    o3, l3 = ops.attn_fwd(inp.q, inp.k, inp.v, 512, 3, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_causality_on_gpu():
    """Changing the future never changes earlier outputs."""
    w = workloads.custom((4096,), 2, 128, 256, topk=3, seed=15)
    inp = workloads.make_inputs(w, device="cuda")
    o1, l1 = ops.attn_fwd(inp.q, inp.k, inp.v, 256, 3)
    i = 2500
    q2, k2, v2 = (x.clone() for x in (inp.q, inp.k, inp.v))
    for x in (q2, k2, v2):
        x[:, i + 1:] = torch.randn_like(x[:, i + 1:].float()).mul(3).to(torch.bfloat16)
    o2, l2 = ops.attn_fwd(q2, k2, v2, 256, 3)
    assert torch.equal(o1[:, :i + 1], o2[:, :i + 1])
    assert torch.equal(l1[:, :, :i + 1], l2[:, :, :i + 1])


def test_workspace_too_small_on_device():
    w = workloads.custom((1024,), 1, 64, 64, topk=3, seed=16)
    inp = workloads.make_inputs(w, device="cuda")
    need = ops.workspace_size(1, 1, 1024, 64, 64, 3)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError, match="WORKSPACE"):
        ops.attn_fwd(inp.q, inp.k, inp.v, 64, 3, workspace=ws)


# ---------------------------------------------------------------------------
# bounded waits, and the warp-level mma.sync baseline kernels
# ---------------------------------------------------------------------------

def test_bounded_wait_reports_timeout_and_context_survives():
    """A producer told to skip its first K/V load leaves the MMA lane waiting on
    an mbarrier nothing will complete: the wait gives up, MOBA_ERR_TIMEOUT is
    recorded, and the next call on the same context is correct."""
    w = workloads.custom((2048,), 1, 128, 256, topk=3, seed=6)
    inp = workloads.make_inputs(w, device="cuda")
    gpu_forward(inp, w, 3, debug_flags=1, wait_limit_cycles=20_000_000)  # ~10 ms per wait
    assert ops.get_status() == ops.MOBA_ERR_TIMEOUT
    out, lse = gpu_forward(inp, w, 3)
    assert ops.get_status() == ops.MOBA_OK
    compare(w, inp, 3, out, lse)


@pytest.mark.parametrize("seqlens,H,D,bs,topk", [
    ((2048,), 1, 64, 256, 3), ((700,), 3, 64, 64, 4), ((4096, 4096), 2, 128, 256, 3),
    ((512,), 2, 128, 128, 4), ((200, 1, 64, 129), 2, 128, 64, 3)])
def test_mma_sync_baseline_path(seqlens, H, D, bs, topk):
    w = workloads.custom(seqlens, H, D, bs, topk=topk, seed=17)
    *_, st = run_case(w, topk, attn_kernel=ops.ATTN_MMA_SYNC)
    print("mma.sync", seqlens, st)


@pytest.mark.parametrize("seqlens,H,D,bs,topk", [
    ((32768,), 4, 128, 512, 3),       # one 128-block chunk
    ((16384,), 2, 128, 64, 5),        # 256 blocks: two chunks in TMEM
    ((3000, 9000), 3, 64, 64, 8),     # varlen, D = 64
    ((20000,), 2, 128, 64, 3),        # 313 blocks: falls back to the CUDA-core gate
    ((65536,), 2, 128, 256, 17),      # wide top-k
])
def test_tensor_core_gate_equals_cuda_core_gate(seqlens, H, D, bs, topk):
    """The tensor-core gate re-scores its candidates exactly, so it must pick
    the very same blocks as the all-CUDA-core gate."""
    w = workloads.custom(seqlens, H, D, bs, topk=topk, seed=31)
    inp = workloads.make_inputs(w, device="cuda")
    _, ref = gpu_select(inp, w, topk, gate_kernel=ops.GATE_CUDA_CORES)
    _, got = gpu_select(inp, w, topk)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(ref, got)
    # and the forward on the CUDA-core gate uses that same selection
    _, _, fidx = gpu_forward(inp, w, topk, with_idx=True, gate_kernel=ops.GATE_CUDA_CORES)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(ref, fidx)


# ---------------------------------------------------------------------------
# device-side lengths that contradict the host arguments
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cu,max_seqlen", [
    ((0, 2048, 4096), 1024),        # max_seqlen below a sequence's length
    ((0, 3000, 2000, 4096), 4096),  # offsets decrease
    ((0, 2048, 4000), 2048),        # last offset is not the token count
    ((16, 2048, 4096), 4096),       # first offset is not 0
])
def test_inconsistent_cu_seqlens_are_reported_not_used(cu, max_seqlen):
    """cu_seqlens lives on the device, so the first kernel of each varlen call
    checks it; when it contradicts the host arguments every later kernel returns
    without touching memory through it and the status word reports
    MOBA_ERR_INVALID_ARG.  The context stays usable: a correct call follows."""
    total, H, D, bs = 4096, 2, 128, 256
    g = torch.Generator(device="cuda").manual_seed(3)
    q, k, v = (torch.randn(total, H, D, generator=g, device="cuda").to(torch.bfloat16)
               for _ in range(3))
    dcu = torch.tensor(cu, dtype=torch.int32, device="cuda")
    assert ops.get_status() == ops.MOBA_OK
    ops.attn_fwd_varlen(q, k, v, dcu, max_seqlen, bs, 3)
    assert ops.get_status() == ops.MOBA_ERR_INVALID_ARG
    # pooling and gate take no max_seqlen: only offsets that contradict the
    # token count make them refuse
    kbar = ops.kpool_varlen(k, dcu, bs)
    bad_alone = cu[0] != 0 or cu[-1] != total or any(b < a for a, b in zip(cu, cu[1:]))
    want = ops.MOBA_ERR_INVALID_ARG if bad_alone else ops.MOBA_OK
    assert ops.get_status() == want
    ops.gate_topk_varlen(q, torch.zeros_like(kbar), dcu, bs, 3)
    assert ops.get_status() == want
    out = torch.zeros_like(q)
    lse = torch.zeros(H, total, dtype=torch.float32, device="cuda")
    ops.attn_bwd_varlen(q, k, v, out, lse, q, dcu, max_seqlen, bs, 3)
    assert ops.get_status() == ops.MOBA_ERR_INVALID_ARG
    # a consistent call on the same context
    w = workloads.custom((2048, 2048), H, D, bs, topk=3, seed=44)
    *_, st = run_case(w, 3)
    print("after invalid offsets", st)


# ---------------------------------------------------------------------------
# query-major fusion of own-block jobs whose rows agree on their past blocks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seqlens,H,bs,topk,coherent", [
    ((4096,), 4, 512, 3, 2),            # every tile's rows agree on 2 blocks: fused
    ((4096, 2500), 2, 256, 3, 2),       # varlen, block 256, partial tail tile
    ((8192,), 2, 1024, 2, 1),           # top-2: a single past block per tile
    ((4096,), 2, 512, 4, 2),            # union 2 <= topk - 1 = 3: fused
    ((4096,), 2, 512, 3, 3),            # union 3 > topk - 1: block-major
    ((6144,), 2, 512, 9, 8),            # the widest union a fused job may hold
])
def test_fused_own_block_jobs(seqlens, H, bs, topk, coherent):
    """Rows of a 256-row tile that agree on their past blocks are attended by
    the own-block pass (query-major, each row masked to its selection): the
    results match the oracle, and the block-major schedule on the same inputs."""
    w = workloads.custom(seqlens, H, 128, bs, topk=topk, seed=51, qkv_scale=128 ** -0.5,
                         coherent=coherent)
    inp, _, idx, out, lse, st = run_case(w, topk)
    o2, l2, i2 = gpu_forward(inp, w, topk, with_idx=True, schedule=ops.SCHEDULE_BLOCK_MAJOR)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(idx, i2)
    compare(w, inp, topk, o2, l2, idx_gpu=i2)
    print(seqlens, bs, topk, coherent, st)


def test_coherent32k_sampled():
    w = workloads.WORKLOADS["coherent32k"]
    rows = workloads.sample_rows(w, 4096)
    *_, st = run_case(w, 3, rows=rows)
    print("coherent32k", st)
