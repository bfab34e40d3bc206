"""Decode (one new token per sequence against its KV cache) against the
oracle: a decode step is the prefill forward's row len - 1 of each sequence,
so the oracle's rows at those tokens are the reference, and the selection
must equal the prefill gate's for the same rows."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_moba_gb300 import ops, workloads

from .parity import LSE_MAX, OUT_MAX, OUT_MEAN, TIE_GAP

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_sparse_moba_gb300 import build
    build.build()
    oracle.build()
    ops.lib()


def decode_case(lens, S_max, H, D, bs, topk, seed, use_ws=False):
    B = len(lens)
    w = workloads.custom((S_max,) * B, H, D, bs, topk=topk, seed=seed, qkv_scale=D ** -0.5,
                         offset_std=0.5)
    inp = workloads.make_inputs(w, device="cuda")
    qf, kc, vc = inp.q, inp.k, inp.v                   # [B, S_max, H, D]
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q = torch.stack([qf[b, L - 1] for b, L in enumerate(lens)]).contiguous()
    kbar = ops.kpool(kc, bs)
    ws = None
    if use_ws:
        ws = torch.empty(ops.decode_workspace_size(B, H, D, topk), dtype=torch.uint8, device="cuda")
    out, lse, idx = ops.decode_fwd(q, kc, vc, kbar, lens_t, bs, topk, workspace=ws)
    assert ops.get_status() == ops.MOBA_OK
    # the prefill gate's selection of the same rows
    pidx = ops.gate_topk(qf, kbar, bs, topk)
    want_idx = torch.stack([pidx[b, L - 1] for b, L in enumerate(lens)])
    assert torch.equal(idx, want_idx)
    # oracle rows on the packed caches
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    pack = lambda t: torch.cat([t[b, :L] for b, L in enumerate(lens)]).cpu()
    tok = np.repeat(cu[1:] - 1, H)
    head = np.tile(np.arange(H, dtype=np.int32), B)
    ref = oracle.moba_rows(pack(qf), pack(kc), pack(vc), cu, H, D, bs, topk, tok, head)
    gi = idx.cpu().numpy().reshape(B * H, topk)
    differ = (gi != ref["idx"]).any(axis=1)
    assert not (differ & (ref["gap"] >= TIE_GAP)).any()
    keep = ~differ
    err = np.abs(out.float().cpu().numpy().reshape(B * H, D).astype(np.float64) - ref["out"])[keep]
    lerr = np.abs(lse.cpu().numpy().reshape(B * H).astype(np.float64) - ref["lse"])[keep]
    assert err.max() <= OUT_MAX and err.mean() <= OUT_MEAN, (err.max(), err.mean())
    assert lerr.max() <= LSE_MAX, lerr.max()
    return out, lse, idx


@pytest.mark.parametrize("topk", [1, 2, 3, 5, 8])
def test_decode_matches_oracle(topk):
    decode_case([4096, 1, 2500, 513], 4096, 4, 128, 512, topk, seed=51)


def test_decode_dense_when_topk_covers_every_block():
    decode_case([2048, 700, 1], 2048, 2, 128, 256, 8, seed=52)


def test_decode_head_dim_64_and_small_blocks():
    decode_case([3000, 1234], 3072, 3, 64, 64, 4, seed=53)


def test_decode_with_caller_workspace():
    decode_case([4096, 1000], 4096, 2, 128, 512, 3, seed=54, use_ws=True)


def test_decode_32k_cache():
    decode_case([32768, 20000], 32768, 8, 128, 512, 3, seed=55)


def test_decode_rejects_a_bad_length_on_the_device():
    B, S_max, H, D, bs = 2, 1024, 2, 128, 256
    q = torch.randn(B, H, D, device="cuda").to(torch.bfloat16)
    kc = torch.randn(B, S_max, H, D, device="cuda").to(torch.bfloat16)
    kbar = ops.kpool(kc, bs)
    lens = torch.tensor([0, 500], dtype=torch.int32, device="cuda")
    out, lse, idx = ops.decode_fwd(q, kc, kc, kbar, lens, bs, 3)
    assert ops.get_status() == ops.MOBA_ERR_INVALID_ARG
    assert (out[0] == 0).all() and torch.isinf(lse[0]).all()
    assert torch.isfinite(lse[1]).all()
    # the context stays usable
    lens = torch.tensor([1024, 500], dtype=torch.int32, device="cuda")
    ops.decode_fwd(q, kc, kc, kbar, lens, bs, 3)
    assert ops.get_status() == ops.MOBA_OK
