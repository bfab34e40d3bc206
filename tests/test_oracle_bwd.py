"""Pins for the oracle's backward pass (the gradient of the MoBA attention with
the gate's selection held fixed): torch autograd of library attention on the
dense case, autograd of a masked softmax attention on sparse cases, and exact
identities of softmax attention's gradients.  CPU only."""
import numpy as np
import pytest
import torch

from long_context_sparse_moba_gb300 import workloads


def flat(x, w):
    return x.reshape(w.total, w.H, w.D)


def case(seqlens, H, D, bs, topk, seed):
    w = workloads.custom(seqlens, H, D, bs, topk, seed=seed, varlen=True)
    inp = workloads.make_inputs(w)
    dout = workloads.make_grad(w)
    return w, inp, dout


def per_head(x, w, b, h):
    """[len, D] float64 slice of sequence b, head h of a [total, H, D] tensor."""
    cu = w.cu_seqlens()
    return torch.as_tensor(np.asarray(x[cu[b]:cu[b + 1], h], dtype=np.float64))


def autograd_grads(w, inp, dout, allowed):
    """dq, dk, dv [total, H, D] from torch autograd; allowed(b, h, L) gives the
    [L, L] boolean mask of the keys each row attends to, or None for the
    library's causal attention."""
    cu = w.cu_seqlens()
    out = {n: np.zeros((w.total, w.H, w.D)) for n in ("dq", "dk", "dv", "o")}
    for b in range(w.B):
        for h in range(w.H):
            q, k, v, g = (per_head(flat(t, w).to(torch.float64), w, b, h)
                          for t in (inp.q, inp.k, inp.v, dout))
            q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
            L = q.shape[0]
            m = allowed(b, h, L)
            if m is None:
                o = torch.nn.functional.scaled_dot_product_attention(
                    q[None, None], k[None, None], v[None, None], is_causal=True)[0, 0]
            else:
                z = (q @ k.T) / np.sqrt(w.D)
                z = z.masked_fill(~m, float("-inf"))
                o = torch.softmax(z, dim=-1) @ v
            o.backward(g)
            sl = slice(cu[b], cu[b + 1])
            out["dq"][sl, h] = q.grad.numpy()
            out["dk"][sl, h] = k.grad.numpy()
            out["dv"][sl, h] = v.grad.numpy()
            out["o"][sl, h] = o.detach().numpy()
    return out


def test_dense_backward_equals_causal_attention_autograd(oracle_mod):
    # top-k covering every block: MoBA is causal attention (the pages' smooth
    # switch to full attention); the library's causal attention decides
    w, inp, dout = case((200, 77), H=2, D=16, bs=64, topk=8, seed=11)
    got = oracle_mod.moba_bwd(flat(inp.q, w), flat(inp.k, w), flat(inp.v, w), flat(dout, w),
                              w.cu_seqlens(), w.H, w.D, w.block_size, 8)
    ref = autograd_grads(w, inp, dout, lambda b, h, L: None)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(got[n], ref[n], rtol=0, atol=1e-10, err_msg=n)


@pytest.mark.parametrize("seqlens,bs,topk,seed", [((300, 130), 32, 3, 12), ((256,), 16, 2, 13),
                                                  ((190, 64, 5), 32, 4, 14)])
def test_sparse_backward_equals_masked_attention_autograd(oracle_mod, seqlens, bs, topk, seed):
    w, inp, dout = case(seqlens, H=2, D=16, bs=bs, topk=topk, seed=seed)
    q, k, v, g = (flat(t, w) for t in (inp.q, inp.k, inp.v, dout))
    fwd = oracle_mod.moba_full(q, k, v, w.cu_seqlens(), w.H, w.D, bs, topk)
    idx = fwd["idx"]
    cu = w.cu_seqlens()

    def allowed(b, h, L):
        blk = torch.arange(L) // bs
        sel = torch.as_tensor(idx[cu[b]:cu[b + 1], h].astype(np.int64))       # [L, topk]
        in_sel = (blk[None, :, None] == sel[:, None, :]).any(-1)               # [L, L]
        causal = torch.arange(L)[None, :] <= torch.arange(L)[:, None]
        return in_sel & causal

    got = oracle_mod.moba_bwd(q, k, v, g, cu, w.H, w.D, bs, topk)
    assert np.array_equal(got["idx"], idx)
    ref = autograd_grads(w, inp, dout, allowed)
    np.testing.assert_allclose(ref["o"], fwd["out"], rtol=0, atol=1e-12)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(got[n], ref[n], rtol=0, atol=1e-10, err_msg=n)


def test_backward_identities(oracle_mod):
    # Exact consequences of softmax attention, per (sequence, head):
    #  * every row's weights sum to 1        -> sum_j dv_j = sum_i dO_i
    #  * shifting all keys by c shifts each row's logits by a constant and every
    #    gate score equally (selection unchanged) -> sum_j dk_j = 0
    #  * out depends on q, k only through q_i . k_j -> sum <q,dq> = sum <k,dk>
    #  * out is linear in v                  -> sum <v,dv> = sum <dO,out>
    #  * a row with one key has zero dq (the first token of every sequence)
    w, inp, dout = case((512, 300), H=2, D=32, bs=64, topk=3, seed=15)
    q, k, v, g = (flat(t, w) for t in (inp.q, inp.k, inp.v, dout))
    cu = w.cu_seqlens()
    r = oracle_mod.moba_bwd(q, k, v, g, cu, w.H, w.D, w.block_size, 3)
    o = oracle_mod.moba_full(q, k, v, cu, w.H, w.D, w.block_size, 3)["out"]
    qd, kd, vd, gd = (t.to(torch.float64).numpy() for t in (q, k, v, g))
    for b in range(w.B):
        sl = slice(cu[b], cu[b + 1])
        for h in range(w.H):
            dq, dk, dv = r["dq"][sl, h], r["dk"][sl, h], r["dv"][sl, h]
            np.testing.assert_allclose(dv.sum(0), gd[sl, h].sum(0), rtol=0, atol=1e-9)
            assert np.abs(dk.sum(0)).max() <= 1e-9 * np.abs(dk).sum(0).max()
            a, c = (qd[sl, h] * dq).sum(), (kd[sl, h] * dk).sum()
            assert abs(a - c) <= 1e-9 * (np.abs(qd[sl, h] * dq).sum() + 1.0)
            e, f = (vd[sl, h] * dv).sum(), (gd[sl, h] * o[sl, h]).sum()
            assert abs(e - f) <= 1e-9 * (np.abs(vd[sl, h] * dv).sum() + 1.0)
            assert np.all(dq[0] == 0.0)
            # and the second row (two keys) has a non-zero dq
            assert np.abs(dq[1]).max() > 0


def test_sampled_dq_rows_match_the_whole_pass(oracle_mod):
    w, inp, dout = case((400, 150), H=3, D=16, bs=32, topk=3, seed=16)
    q, k, v, g = (flat(t, w) for t in (inp.q, inp.k, inp.v, dout))
    cu = w.cu_seqlens()
    full = oracle_mod.moba_bwd(q, k, v, g, cu, w.H, w.D, w.block_size, 3)
    toks, heads = workloads.sample_rows(w, 40, seed=3)
    sel = full["idx"][toks, heads]
    dq = oracle_mod.moba_bwd_dq_rows(q, k, v, g, cu, w.H, w.D, w.block_size, 3, toks, heads, sel)
    assert np.array_equal(dq, full["dq"][toks, heads])
