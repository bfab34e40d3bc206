"""Comparison of the CUDA path with the CPU oracle (shared by the GPU tests).

Acceptance (element by element on the compared rows):
  idx  bit-exact, except rows whose oracle score gap between the last kept
       and the first dropped past block is below 1e-5 (near ties); those rows
       are counted, and their outputs are checked against the oracle run with
       the GPU's own selection;
  out  max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3;
  lse  max |gpu - oracle| <= 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from long_context_sparse_moba_gb300 import ops, workloads

TIE_GAP = 1e-5
OUT_MAX = 2e-2
OUT_MEAN = 2e-3
LSE_MAX = 1e-3


def flat(x):
    """[B, S, H, ...] or [total, H, ...] -> [total, H, ...] (view)."""
    return x.reshape(-1, *x.shape[2:]) if x.dim() == 4 else x


def gpu_select(inp, w: workloads.Workload, topk: int, pooling=ops.POOL_MEAN,
               gate_kernel=ops.GATE_TCGEN05):
    """kbar and idx from the library's pooling and gate entry points."""
    if w.varlen:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device=inp.q.device)
        kbar = ops.kpool_varlen(inp.k, cu, w.block_size, pooling=pooling)
        idx = ops.gate_topk_varlen(inp.q, kbar, cu, w.block_size, topk, gate_kernel=gate_kernel)
    else:
        kbar = ops.kpool(inp.k, w.block_size, pooling=pooling)
        idx = ops.gate_topk(inp.q, kbar, w.block_size, topk, gate_kernel=gate_kernel)
    return kbar, flat(idx)


def gpu_forward(inp, w: workloads.Workload, topk: int, with_idx=False, stream=None, **options):
    """The forward through the C ABI; with ``with_idx`` also the selection the
    forward itself used (its idx_out option), as [total, H, topk]."""
    dev = inp.q.device
    idx = None
    if w.varlen:
        cu = torch.tensor(inp.cu_seqlens, dtype=torch.int32, device=dev)
        if with_idx:
            idx = torch.empty(w.total, w.H, topk, dtype=torch.int32, device=dev)
        out, lse = ops.attn_fwd_varlen(inp.q, inp.k, inp.v, cu, w.S, w.block_size, topk,
                                       idx_out=idx, stream=stream, **options)
    else:
        if with_idx:
            idx = torch.empty(w.B, w.S, w.H, topk, dtype=torch.int32, device=dev)
        out, lse = ops.attn_fwd(inp.q, inp.k, inp.v, w.block_size, topk, idx_out=idx,
                                stream=stream, **options)
    if with_idx:
        return out, lse, flat(idx)
    return out, lse


def lse_at(lse, w: workloads.Workload, tok, head):
    tok = np.asarray(tok)
    head = np.asarray(head)
    l = lse.detach().cpu().numpy()
    if w.varlen:
        return l[head, tok].astype(np.float64)
    b, i = tok // w.S, tok % w.S
    return l[b, head, i].astype(np.float64)


def compare(w: workloads.Workload, inp, topk: int, out, lse, idx_gpu=None, rows=None,
            host=None, kbar=None):
    """Check out / lse (and idx if given) against the oracle on `rows`
    ((tokens, heads); all rows if None).  Returns a stats dict."""
    if host is None:
        host = tuple(flat(x).cpu() for x in (inp.q, inp.k, inp.v))
    q, k, v = host
    H, D, bs = w.H, w.D, w.block_size
    if rows is None:
        tok, head = oracle.all_rows(w.total, H)
    else:
        tok, head = (np.asarray(rows[0], dtype=np.int64), np.asarray(rows[1], dtype=np.int32))
    if kbar is None:
        kbar = oracle.kpool(k, inp.cu_seqlens, H, D, bs)
    ref = oracle.moba_rows(q, k, v, inp.cu_seqlens, H, D, bs, topk, tok, head, kbar=kbar)
    stats = {"rows": int(len(tok)), "near_ties": int((ref["gap"] < TIE_GAP).sum())}
    exp_out, exp_lse = ref["out"], ref["lse"]
    if idx_gpu is not None:
        gi = idx_gpu.cpu().numpy()[tok, head]
        differ = (gi != ref["idx"]).any(axis=1)
        near = ref["gap"] < TIE_GAP
        bad = differ & ~near
        assert not bad.any(), (
            f"{int(bad.sum())} rows select different blocks with a score gap >= {TIE_GAP}: "
            f"first at token {int(tok[bad][0])} head {int(head[bad][0])}: "
            f"gpu {gi[bad][0].tolist()} oracle {ref['idx'][bad][0].tolist()} "
            f"gap {ref['gap'][bad][0]}")
        stats["near_tie_rows_differing"] = int((differ & near).sum())
        if differ.any():
            sub = np.nonzero(differ)[0]
            alt = oracle.moba_rows(q, k, v, inp.cu_seqlens, H, D, bs, topk, tok[sub], head[sub],
                                   given_idx=gi[sub], kbar=kbar)
            exp_out = exp_out.copy()
            exp_lse = exp_lse.copy()
            exp_out[sub] = alt["out"]
            exp_lse[sub] = alt["lse"]
    go = flat(out).float().cpu().numpy()[tok, head].astype(np.float64)
    err = np.abs(go - exp_out)
    gl = lse_at(lse, w, tok, head)
    lerr = np.abs(gl - exp_lse)
    stats.update(out_max=float(err.max()), out_mean=float(err.mean()), lse_max=float(lerr.max()))
    assert np.isfinite(go).all() and np.isfinite(gl).all(), "non-finite GPU output"
    assert stats["out_max"] <= OUT_MAX, stats
    assert stats["out_mean"] <= OUT_MEAN, stats
    assert stats["lse_max"] <= LSE_MAX, stats
    return stats


def tie_masks(w, idx_gpu, ref_idx, gap):
    """Rows (token, head) and keys (token, head) excluded because of near ties."""
    differ = (idx_gpu != ref_idx).any(axis=-1)                       # [total, H]
    assert not (differ & (gap >= TIE_GAP)).any(), "selection differs away from a tie"
    row_ok = ~differ
    key_ok = np.ones((w.total, w.H), dtype=bool)
    cu = w.cu_seqlens()
    bs = w.block_size
    for t, h in zip(*np.nonzero(differ)):
        b = int(np.searchsorted(cu, t, side="right") - 1)
        for c in set(idx_gpu[t, h].tolist()) ^ set(ref_idx[t, h].tolist()):
            if c >= 0:
                key_ok[cu[b] + c * bs: min(cu[b] + (c + 1) * bs, cu[b + 1]), h] = False
    return row_ok, key_ok
