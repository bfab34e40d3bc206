"""Backward pass (dq, dk, dv with the gate's selection held fixed) on the GPU
against the oracle's backward.

Acceptance, per tensor, on the compared elements (ratios of the error to the
oracle's magnitudes):
  dk, dv:  max |gpu - oracle| <= 1.5e-2 * max |oracle|,
           mean |gpu - oracle| <= 6e-3 * mean |oracle|;
  dq:      max <= 5e-2 * max |oracle|,  mean <= 2e-2 * mean |oracle|.
Derivation: the kernel rounds P and dS to bf16 for the tensor-core products,
takes dO . O from the forward's bf16 out, and returns bf16 gradients.  An fp32
model of exactly that rounding, run against the fp64 oracle on every shape
below, gives at most 3.6e-3 (max) and 2.3e-3 (mean) for dk and dv, and
2.3e-2 and 8.6e-3 for dq: dq_i = sum_j dS_ij k_j / sqrt(D) adds terms whose
weights dS_ij sum to zero for every row, so their rounding is large against
the result, worst where a row sees few keys (top-1).  The GPU forward's own
rounding of out and lse comes on top; the bounds leave about a factor 2.
Rows whose selection differs from the oracle's at a near tie (score gap below
1e-5) are valid either way: their dq and the dk, dv of the blocks on which the
two selections disagree are left out of the comparison; any other difference
fails."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_moba_gb300 import ops, workloads

from .parity import TIE_GAP, flat, gpu_forward, tie_masks

pytestmark = pytest.mark.gpu

TOL = {"dq": (5e-2, 2e-2), "dk": (1.5e-2, 6e-3), "dv": (1.5e-2, 6e-3)}  # (max, mean) ratios


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_moba_gb300 import build
    build.build()
    oracle.build()
    ops.lib()


def gpu_backward(inp, w, topk, out, lse, dout, workspace=None):
    if w.varlen:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")
        return ops.attn_bwd_varlen(inp.q, inp.k, inp.v, out, lse, dout, cu, w.S, w.block_size,
                                   topk)
    return ops.attn_bwd(inp.q, inp.k, inp.v, out, lse, dout, w.block_size, topk,
                        workspace=workspace)


def check(name, got, ref, keep=None):
    got = got.astype(np.float64)
    if keep is not None:
        got, ref = got[keep], ref[keep]
    err = np.abs(got - ref)
    mx, mn = err.max() / np.abs(ref).max(), err.mean() / np.abs(ref).mean()
    assert mx <= TOL[name][0] and mn <= TOL[name][1], (name, mx, mn)
    return mx, mn


def run_case(w, topk, dout_scale=1.0):
    inp = workloads.make_inputs(w, device="cuda")
    dout = workloads.make_grad(w, device="cuda", scale=dout_scale)
    out, lse = gpu_forward(inp, w, topk)
    dq, dk, dv = gpu_backward(inp, w, topk, out, lse, dout)
    assert ops.get_status() == ops.MOBA_OK
    q, k, v, g = (flat(t).cpu() for t in (inp.q, inp.k, inp.v, dout))
    cu = w.cu_seqlens()
    ref = oracle.moba_bwd(q, k, v, g, cu, w.H, w.D, w.block_size, topk)
    fwd = oracle.moba_full(q, k, v, cu, w.H, w.D, w.block_size, topk)
    if topk > 1 and topk < max(oracle.num_blocks(L, w.block_size) for L in w.seqlens):
        from .parity import gpu_select
        _, idx = gpu_select(inp, w, topk)
        row_ok, key_ok = tie_masks(w, idx.cpu().numpy(), ref["idx"], fwd["gap"])
    else:
        row_ok = key_ok = np.ones((w.total, w.H), dtype=bool)
    res = {}
    res["dq"] = check("dq", flat(dq).float().cpu().numpy(), ref["dq"], row_ok)
    res["dk"] = check("dk", flat(dk).float().cpu().numpy(), ref["dk"], key_ok)
    res["dv"] = check("dv", flat(dv).float().cpu().numpy(), ref["dv"], key_ok)
    return res


@pytest.mark.parametrize("seqlens,H,D,bs,topk,varlen", [
    ((1000, 1000), 2, 128, 128, 3, False),      # ragged tail block, two sequences
    ((1000, 700, 333), 2, 64, 64, 4, True),     # varlen, partial tails
    ((2048,), 2, 128, 512, 3, False),           # the 32K workload's block size
    ((777,), 1, 64, 64, 1, False),              # top-1: own block only
    ((600,), 2, 128, 128, 8, False),            # top-k covers every block: dense
    ((300,), 1, 128, 64, 3, False),             # early rows: fewer past blocks than slots
])
def test_backward_matches_oracle(seqlens, H, D, bs, topk, varlen):
    w = workloads.custom(seqlens, H, D, bs, topk, seed=31, qkv_scale=D ** -0.5,
                         varlen=varlen)
    res = run_case(w, topk)
    print(seqlens, D, bs, topk, {n: ("%.2e" % a, "%.2e" % b) for n, (a, b) in res.items()})


def test_backward_unit_scale_inputs():
    # larger logits (q, k ~ N(0, 1)): peakier softmax rows
    w = workloads.custom((1500,), 2, 64, 128, 3, seed=32, qkv_scale=1.0)
    run_case(w, 3)


@pytest.mark.parametrize("seqlens,D,varlen", [
    ((1536,), 128, False),          # tcgen05 backward
    ((1100, 900, 300), 64, True),   # mma.sync backward, varlen
])
def test_backward_workspace_variant_and_determinism(seqlens, D, varlen):
    w = workloads.custom(seqlens, 2, D, 128, 3, seed=33, qkv_scale=D ** -0.5, varlen=varlen)
    inp = workloads.make_inputs(w, device="cuda")
    dout = workloads.make_grad(w, device="cuda")
    out, lse = gpu_forward(inp, w, 3)
    a = gpu_backward(inp, w, 3, out, lse, dout)
    if varlen:
        b = gpu_backward(inp, w, 3, out, lse, dout)
    else:
        ws = torch.empty(ops.bwd_workspace_size(w.B, w.H, w.S, w.D, w.block_size, 3),
                         dtype=torch.uint8, device="cuda")
        b = gpu_backward(inp, w, 3, out, lse, dout, workspace=ws)
    assert ops.get_status() == ops.MOBA_OK
    # the regroup lists come out in the same order on every call and every key's
    # dk, dv is summed by one CTA in list order: bit for bit.  dq adds fp32
    # reductions from several CTAs in any order: equal to rounding.
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    d = (a[0].float() - b[0].float()).abs()
    assert d.max() <= 1e-2 * a[0].float().abs().max(), d.max()
    assert d.mean() <= 2e-3 * a[0].float().abs().mean(), d.mean()


@pytest.mark.parametrize("seqlens,D,bs,topk", [((1536,), 128, 128, 3), ((2048,), 64, 256, 4),
                                               ((4096,), 128, 512, 3)])
def test_backward_with_the_forwards_selection(seqlens, D, bs, topk):
    # the forward's idx_out handed back as idx_in: the backward regroups that
    # selection instead of recomputing it, and the gradients are those of the
    # recomputing backward (dk, dv bit for bit; dq to the rounding of its
    # fp32 reductions)
    w = workloads.custom(seqlens, 2, D, bs, topk, seed=34, qkv_scale=D ** -0.5)
    inp = workloads.make_inputs(w, device="cuda")
    dout = workloads.make_grad(w, device="cuda")
    idx = torch.empty(w.B, w.S, w.H, topk, dtype=torch.int32, device="cuda")
    out, lse = ops.attn_fwd(inp.q, inp.k, inp.v, bs, topk, idx_out=idx)
    a = ops.attn_bwd(inp.q, inp.k, inp.v, out, lse, dout, bs, topk)
    b = ops.attn_bwd(inp.q, inp.k, inp.v, out, lse, dout, bs, topk, idx_in=idx)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    d = (a[0].float() - b[0].float()).abs()
    assert d.max() <= 1e-2 * a[0].float().abs().max(), d.max()
    assert d.mean() <= 2e-3 * a[0].float().abs().mean(), d.mean()


def test_backward_varlen_with_the_forwards_selection():
    # the same for packed sequences (a partial tail block in each)
    w = workloads.custom((1100, 900, 300), 2, 128, 128, 3, seed=35, qkv_scale=128 ** -0.5,
                         varlen=True)
    inp = workloads.make_inputs(w, device="cuda")
    dout = workloads.make_grad(w, device="cuda")
    cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device="cuda")
    idx = torch.empty(w.total, w.H, 3, dtype=torch.int32, device="cuda")
    out, lse = ops.attn_fwd_varlen(inp.q, inp.k, inp.v, cu, w.S, w.block_size, 3, idx_out=idx)
    a = ops.attn_bwd_varlen(inp.q, inp.k, inp.v, out, lse, dout, cu, w.S, w.block_size, 3)
    b = ops.attn_bwd_varlen(inp.q, inp.k, inp.v, out, lse, dout, cu, w.S, w.block_size, 3,
                            idx_in=idx)
    assert ops.get_status() == ops.MOBA_OK
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    d = (a[0].float() - b[0].float()).abs()
    assert d.max() <= 1e-2 * a[0].float().abs().max(), d.max()


def test_backward_train32k_sampled_and_identities():
    # the 32K-token training shape: dq of sampled rows against the oracle, and
    # two exact identities of attention gradients over every key
    w = workloads.WORKLOADS["train32k"]
    topk = 3
    inp = workloads.make_inputs(w, device="cuda")
    dout = workloads.make_grad(w, device="cuda")
    out, lse = gpu_forward(inp, w, topk)
    dq, dk, dv = gpu_backward(inp, w, topk, out, lse, dout)
    assert ops.get_status() == ops.MOBA_OK
    q, k, v, g = (flat(t).cpu() for t in (inp.q, inp.k, inp.v, dout))
    cu = w.cu_seqlens()
    toks, heads = workloads.sample_rows(w, 96, seed=5)
    r = oracle.moba_rows(q, k, v, cu, w.H, w.D, w.block_size, topk, toks, heads)
    from .parity import gpu_select
    _, idx = gpu_select(inp, w, topk)
    gi = idx.cpu().numpy()[toks, heads]
    differ = (gi != r["idx"]).any(axis=1)
    assert not (differ & (r["gap"] >= TIE_GAP)).any()
    ref = oracle.moba_bwd_dq_rows(q, k, v, g, cu, w.H, w.D, w.block_size, topk, toks, heads,
                                  r["idx"])
    got = flat(dq).float().cpu().numpy()[toks, heads]
    check("dq", got[~differ], ref[~differ])
    # dq, dk and dv of two whole heads element by element: the oracle's backward
    # on the head's own slice (gate, selection and attention are per head)
    for h in (0, w.H - 1):
        sl = lambda t: t[:, h:h + 1, :].contiguous()
        refh = oracle.moba_bwd(sl(q), sl(k), sl(v), sl(g), cu, 1, w.D, w.block_size, topk)
        fwdh = oracle.moba_full(sl(q), sl(k), sl(v), cu, 1, w.D, w.block_size, topk)
        wh = workloads.Workload(**{**w.__dict__, "H": 1})
        row_ok, key_ok = tie_masks(wh, idx.cpu().numpy()[:, h:h + 1, :], refh["idx"],
                                   fwdh["gap"])
        for name, t, keep in (("dq", dq, row_ok), ("dk", dk, key_ok), ("dv", dv, key_ok)):
            check(name, flat(t)[:, h:h + 1, :].float().cpu().numpy(), refh[name], keep)
    # sum over keys of dv = sum over rows of dO; sum over keys of dk = 0 (per head)
    dvs = flat(dv).double().sum(0)
    gs = flat(dout).double().sum(0)
    dva = flat(dv).double().abs().sum(0)
    assert ((dvs - gs).abs() <= 1e-2 * dva).all()
    dks = flat(dk).double().sum(0)
    dka = flat(dk).double().abs().sum(0)
    assert (dks.abs() <= 1e-2 * dka).all()
