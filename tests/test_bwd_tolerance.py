"""The backward parity bounds against an fp32 model of the kernel's rounding
(CPU): P and dS rounded to bf16 before the tensor-core products, dO . O taken
from the forward's output rounded to bf16, gradients returned in bf16.  The
model, run against the fp64 oracle, must stay well inside the bounds the GPU
tests use, on the shapes where it comes closest (few keys per row: top-1; the
scaled-down inputs of the 32K workload)."""
import numpy as np
import pytest
import torch

from long_context_sparse_moba_gb300 import workloads

from .test_gpu_bwd import TOL

MARGIN = 1.5


def rounding_model(oracle_mod, w, topk):
    inp = workloads.make_inputs(w)
    g = workloads.make_grad(w)
    cu = w.cu_seqlens()
    H, D, bs = w.H, w.D, w.block_size
    q, k, v, go = (t.reshape(w.total, H, D) for t in (inp.q, inp.k, inp.v, g))
    ref = oracle_mod.moba_bwd(q, k, v, go, cu, H, D, bs, topk)
    fwd = oracle_mod.moba_full(q, k, v, cu, H, D, bs, topk)
    model = {n: np.zeros((w.total, H, D)) for n in ("dq", "dk", "dv")}
    l2e = 1.4426950408889634
    for b in range(w.B):
        L = cu[b + 1] - cu[b]
        sl = slice(cu[b], cu[b + 1])
        for h in range(H):
            qh, kh, vh, gh = (t[sl, h].float() for t in (q, k, v, go))
            blk = torch.arange(L) // bs
            sel = torch.as_tensor(ref["idx"][sl, h].astype(np.int64))
            mask = (blk[None, :, None] == sel[:, None, :]).any(-1) & \
                (torch.arange(L)[None, :] <= torch.arange(L)[:, None])
            lse = torch.as_tensor(fwd["lse"][sl, h]).float()
            o = torch.as_tensor(fwd["out"][sl, h]).float().bfloat16().float()
            p = torch.where(mask, torch.exp2((qh @ kh.T) * (D ** -0.5 * l2e) - lse[:, None] * l2e),
                            torch.zeros(()))
            ds = p * ((gh @ vh.T) - (gh * o).sum(-1)[:, None])
            pb, dsb = p.bfloat16().float(), ds.bfloat16().float()
            model["dv"][sl, h] = (pb.T @ gh).bfloat16().float().numpy()
            model["dk"][sl, h] = ((dsb.T @ qh) * D ** -0.5).bfloat16().float().numpy()
            model["dq"][sl, h] = ((dsb @ kh) * D ** -0.5).bfloat16().float().numpy()
    out = {}
    for n in ("dq", "dk", "dv"):
        e, r = np.abs(model[n] - ref[n]), np.abs(ref[n])
        out[n] = (e.max() / r.max(), e.mean() / r.mean())
    return out


@pytest.mark.parametrize("seqlens,H,D,bs,topk", [((777,), 1, 64, 64, 1),
                                                 ((1000, 1000), 1, 128, 128, 3)])
def test_gpu_bounds_cover_the_rounding_model(oracle_mod, seqlens, H, D, bs, topk):
    w = workloads.custom(seqlens, H, D, bs, topk, seed=31, qkv_scale=D ** -0.5)
    got = rounding_model(oracle_mod, w, topk)
    for n, (mx, mn) in got.items():
        assert mx * MARGIN <= TOL[n][0] and mn * MARGIN <= TOL[n][1], (n, mx, mn)
