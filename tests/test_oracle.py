"""Pins for the CPU oracle: checks against numbers the pages print, closed
forms, library routines, brute force and invariants -- never against the
oracle's own formulas retyped.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from long_context_sparse_moba_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_counts.json")


def bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def widen(x):
    return x.to(torch.float64)


def rand_qkv(total, H, D, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return tuple(bf16(torch.randn(total, H, D, generator=g) * scale) for _ in range(3))


# --------------------------------------------------------------------------
# block partition and the sparsity figures printed on the pages
# --------------------------------------------------------------------------

def test_num_blocks_golden(oracle_mod):
    gold = json.load(open(GOLDEN))
    for e in gold["block_counts"]:
        assert oracle_mod.num_blocks(e["seq_len"], e["block_size"]) == e["num_blocks"], e["source"]
    # the workloads' own geometries, by hand: 131072/2048, 1048576/4096, 2048/256
    assert oracle_mod.num_blocks(131072, 2048) == 64
    assert oracle_mod.num_blocks(1048576, 4096) == 256
    assert oracle_mod.num_blocks(2048, 256) == 8
    # partial tail block (the reading taken where a length is not a multiple)
    assert oracle_mod.num_blocks(513, 512) == 2
    assert oracle_mod.num_blocks(1, 512) == 1
    assert oracle_mod.num_blocks(0, 512) == 0


def _selected_fraction_last_row(oracle_mod, S, bs, topk):
    q, k, v = rand_qkv(S, 1, 4, seed=7)
    r = oracle_mod.moba_rows(q, k, v, [0, S], 1, 4, bs, topk, [S - 1], [0])
    nsel = int((r["idx"][0] >= 0).sum())
    return nsel / oracle_mod.num_blocks(S, bs)


def test_sparsity_golden(oracle_mod):
    gold = json.load(open(GOLDEN))
    for e in gold["sparsity"]:
        frac = _selected_fraction_last_row(oracle_mod, e["seq_len"], e["block_size"], e["topk"])
        assert abs((1.0 - frac) - e["sparsity"]) <= e["abs_tol"], e["source"]
    for e in gold["compute_fraction"]:
        frac = _selected_fraction_last_row(oracle_mod, e["seq_len"], e["block_size"], e["topk"])
        assert abs(frac - e["fraction"]) <= e["abs_tol"], e["source"]


# --------------------------------------------------------------------------
# mean-pooled keys
# --------------------------------------------------------------------------

def test_kpool_constant_blocks(oracle_mod):
    """Keys equal to alpha * e_d inside a block pool to exactly alpha * e_d."""
    H, D, bs, S = 2, 8, 4, 22  # 6 blocks, the last one partial (2 tokens)
    alphas = [0.5, -1.25, 3.0, 2.0, -0.75, 1.5]
    k = torch.zeros(S, H, D)
    expect = np.zeros((6, H, D))
    for c in range(6):
        for h in range(H):
            d = (c + 3 * h) % D
            a = alphas[c] * (1 + h)
            k[c * bs:(c + 1) * bs, h, d] = a
            expect[c, h, d] = a
    kbar = oracle_mod.kpool(bf16(k), [0, S], H, D, bs)
    assert np.array_equal(kbar, expect)


def test_kpool_matches_numpy_mean(oracle_mod):
    """Against numpy's mean over each block (two sequences, partial tails)."""
    H, D, bs = 3, 16, 8
    lens = [37, 16]
    total = sum(lens)
    q, k, v = rand_qkv(total, H, D, seed=3)
    kw = widen(k).numpy()
    cu = [0, lens[0], total]
    kbar = oracle_mod.kpool(k, cu, H, D, bs)
    g = 0
    for b, L in enumerate(lens):
        for c in range(oracle_mod.num_blocks(L, bs)):
            t0, t1 = cu[b] + c * bs, cu[b] + min((c + 1) * bs, L)
            np.testing.assert_allclose(kbar[g], kw[t0:t1].mean(axis=0), rtol=0, atol=1e-14)
            g += 1
    assert g == kbar.shape[0]


def test_kpool_permutation_invariant(oracle_mod):
    H, D, bs, S = 2, 8, 16, 64
    q, k, v = rand_qkv(S, H, D, seed=4)
    perm = torch.cat([torch.randperm(bs, generator=torch.Generator().manual_seed(c)) + c * bs
                      for c in range(S // bs)])
    a = oracle_mod.kpool(k, [0, S], H, D, bs)
    b = oracle_mod.kpool(k[perm], [0, S], H, D, bs)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


def test_kpool_max_matches_numpy_max(oracle_mod):
    """Max pooling against numpy's element-wise max over each block (two
    sequences, partial tails, negative and positive keys)."""
    H, D, bs = 3, 16, 8
    lens = [37, 16]
    total = sum(lens)
    q, k, v = rand_qkv(total, H, D, seed=13)
    kw = widen(k).numpy()
    cu = [0, lens[0], total]
    kbar = oracle_mod.kpool(k, cu, H, D, bs, pooling="max")
    g = 0
    for b, L in enumerate(lens):
        for c in range(oracle_mod.num_blocks(L, bs)):
            t0, t1 = cu[b] + c * bs, cu[b] + min((c + 1) * bs, L)
            assert np.array_equal(kbar[g], kw[t0:t1].max(axis=0))
            g += 1
    assert g == kbar.shape[0]


def test_kpool_max_single_spike(oracle_mod):
    """One large key in an otherwise negative block: the max sees it, the mean
    barely moves (worked by hand: keys -1 except one 6, block of 4 -> mean
    0.75, max 6)."""
    bs, D = 4, 8
    k = -torch.ones(8, 1, D)
    k[5, 0, 0] = 6.0
    kb = bf16(k)
    mean = oracle_mod.kpool(kb, [0, 8], 1, D, bs)
    mx = oracle_mod.kpool(kb, [0, 8], 1, D, bs, pooling="max")
    assert mean[1, 0, 0] == pytest.approx((6.0 - 3.0) / 4)
    assert mx[1, 0, 0] == 6.0 and mx[0, 0, 0] == -1.0
    assert (mx[:, 0, 1:] == -1.0).all()


def test_max_pooling_changes_the_selection(oracle_mod):
    """Block 1 holds one key aligned with the queries (spike 8) among keys of
    -1; block 2 is uniformly 1.5.  Mean pooling scores block 1 at 1.25 < 1.5,
    max pooling at 8 > 1.5 (q = e_0), so a row of block 4 with top-k 2 picks
    block 2 under the mean and block 1 under the max."""
    bs, D = 4, 8
    S = 5 * bs
    q = torch.zeros(S, 1, D)
    q[:, 0, 0] = 1.0
    k = torch.zeros(S, 1, D)
    k[0:4, 0, 0] = -2.0
    k[4:8, 0, 0] = -1.0
    k[6, 0, 0] = 8.0
    k[8:12, 0, 0] = 1.5
    k[12:16, 0, 0] = -3.0
    v = torch.randn(S, 1, D, generator=torch.Generator().manual_seed(1))
    q, k, v = bf16(q), bf16(k), bf16(v)
    t = 4 * bs + 1
    mean = oracle_mod.moba_rows(q, k, v, [0, S], 1, D, bs, 2, [t], [0])
    mx = oracle_mod.moba_rows(q, k, v, [0, S], 1, D, bs, 2, [t], [0], pooling="max")
    assert mean["idx"][0].tolist() == [2, 4]
    assert mx["idx"][0].tolist() == [1, 4]
    assert mean["gap"][0] == pytest.approx(1.5 - 1.25)
    assert mx["gap"][0] == pytest.approx(8.0 - 1.5)


# --------------------------------------------------------------------------
# gate and top-k selection
# --------------------------------------------------------------------------

def _hand_built(alphas, bs=4, D=8):
    """Queries all equal e_0; keys of block c equal alpha_c * e_0.  Then the
    score of block c for every query is alpha_c (worked by hand)."""
    n = len(alphas)
    S = n * bs
    q = torch.zeros(S, 1, D)
    q[:, 0, 0] = 1.0
    k = torch.zeros(S, 1, D)
    for c, a in enumerate(alphas):
        k[c * bs:(c + 1) * bs, 0, 0] = a
    v = torch.randn(S, 1, D, generator=torch.Generator().manual_seed(0))
    return bf16(q), bf16(k), bf16(v), S


def test_gate_hand_built(oracle_mod):
    alphas = [0.5, 3.0, 1.0, 2.5, 4.0, 2.0]
    q, k, v, S = _hand_built(alphas)
    bs = 4
    # expected selections with top-k 3 (own block + the 2 best past blocks)
    expect = {0: [0, -1, -1], 1: [0, 1, -1], 2: [0, 1, 2], 3: [1, 2, 3],
              4: [1, 3, 4], 5: [1, 4, 5]}
    expect_gap = {3: 1.0 - 0.5, 4: 2.5 - 1.0, 5: 3.0 - 2.5}
    r = oracle_mod.moba_full(q, k, v, [0, S], 1, 8, bs, 3)
    for t in range(S):
        c = t // bs
        assert r["idx"][t, 0].tolist() == expect[c], (t, c)
        if c in expect_gap:
            assert r["gap"][t, 0] == pytest.approx(expect_gap[c], abs=1e-12)
        else:
            assert math.isinf(r["gap"][t, 0])


def test_gate_ties_go_to_lower_block(oracle_mod):
    q, k, v, S = _hand_built([1.0] * 6)
    r = oracle_mod.moba_full(q, k, v, [0, S], 1, 8, 4, 3)
    for t in range(S):
        c = t // 4
        want = [0, 1, c] if c >= 3 else list(range(c + 1)) + [-1] * (2 - c)
        assert r["idx"][t, 0].tolist() == want
        if c >= 3:
            assert r["gap"][t, 0] == 0.0


def test_gate_topk1_is_own_block(oracle_mod):
    q, k, v = rand_qkv(40, 2, 8, seed=5)
    r = oracle_mod.moba_full(q, k, v, [0, 40], 2, 8, 8, 1)
    for t in range(40):
        assert (r["idx"][t, :, 0] == t // 8).all()


def test_gate_matches_subset_bruteforce(oracle_mod):
    """The selected past set is the (k-1)-subset with the largest score sum
    (scores distinct); found here by enumerating every subset."""
    for seed, (S, bs, topk, D) in enumerate([(56, 8, 3, 8), (63, 7, 4, 16), (80, 16, 2, 4)]):
        q, k, v = rand_qkv(S, 2, D, seed=10 + seed)
        r = oracle_mod.moba_full(q, k, v, [0, S], 2, D, bs, topk)
        kw, qw = widen(k).numpy(), widen(q).numpy()
        n = oracle_mod.num_blocks(S, bs)
        means = np.stack([kw[c * bs:min((c + 1) * bs, S)].mean(axis=0) for c in range(n)])
        for t in range(S):
            ci = t // bs
            for h in range(2):
                if ci <= topk - 1:
                    want = list(range(ci + 1))
                else:
                    sc = means[:ci, h] @ qw[t, h]
                    best = max(itertools.combinations(range(ci), topk - 1),
                               key=lambda s: sum(sc[list(s)]))
                    want = sorted(best) + [ci]
                got = [c for c in r["idx"][t, h] if c >= 0]
                assert got == want, (t, h)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _sdpa_causal(q, k, v, mask=None):
    """torch's scaled_dot_product_attention in float64 + logsumexp of the
    masked scaled logits.  q,k,v: [S, H, D] bf16.  mask: [S, S] bool allowed."""
    S, H, D = q.shape
    qh, kh, vh = (widen(x).permute(1, 0, 2) for x in (q, k, v))
    if mask is None:
        mask = torch.ones(S, S, dtype=torch.bool).tril()
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask)
    logits = (qh @ kh.transpose(1, 2)) / math.sqrt(D)
    lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("S,bs,H,D", [(64, 16, 2, 8), (70, 16, 1, 16), (33, 32, 3, 8), (128, 64, 2, 32)])
def test_topk_covering_all_blocks_is_dense_causal(oracle_mod, S, bs, H, D):
    """The pages' smooth full/sparse switch: with top-k >= number of blocks the
    result is ordinary causal softmax attention."""
    q, k, v = rand_qkv(S, H, D, seed=S)
    n = oracle_mod.num_blocks(S, bs)
    for topk in (n, n + 3):
        r = oracle_mod.moba_full(q, k, v, [0, S], H, D, bs, topk)
        o, lse = _sdpa_causal(q, k, v)
        np.testing.assert_allclose(r["out"], o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["lse"], lse, rtol=0, atol=1e-12)


def test_topk1_is_block_local_causal(oracle_mod):
    S, bs, H, D = 48, 16, 2, 8
    q, k, v = rand_qkv(S, H, D, seed=21)
    r = oracle_mod.moba_full(q, k, v, [0, S], H, D, bs, 1)
    pos = torch.arange(S)
    mask = (pos[:, None] >= pos[None, :]) & (pos[:, None] // bs == pos[None, :] // bs)
    o, lse = _sdpa_causal(q, k, v, mask)
    np.testing.assert_allclose(r["out"], o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["lse"], lse, rtol=0, atol=1e-12)


def test_selected_blocks_as_mask(oracle_mod):
    """Generic top-k: the output equals masked dense attention whose mask is the
    oracle's own selection (pins the attention half independently of the gate)."""
    S, bs, H, D, topk = 96, 8, 2, 16, 3
    q, k, v = rand_qkv(S, H, D, seed=22)
    r = oracle_mod.moba_full(q, k, v, [0, S], H, D, bs, topk)
    pos = torch.arange(S)
    for h in range(H):
        allowed = torch.zeros(S, S, dtype=torch.bool)
        for t in range(S):
            for c in r["idx"][t, h]:
                if c >= 0:
                    allowed[t, c * bs:(c + 1) * bs] = True
        allowed &= pos[:, None] >= pos[None, :]
        o, lse = _sdpa_causal(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], allowed)
        np.testing.assert_allclose(r["out"][:, h], o[:, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["lse"][:, h], lse[:, 0], rtol=0, atol=1e-12)


def test_first_row_closed_form(oracle_mod):
    S, H, D = 32, 2, 16
    q, k, v = rand_qkv(S, H, D, seed=23)
    r = oracle_mod.moba_rows(q, k, v, [0, S], H, D, 8, 3, [0, 0], [0, 1])
    for h in range(H):
        np.testing.assert_array_equal(r["out"][h], widen(v[0, h]).numpy())
        want = float(widen(q[0, h]) @ widen(k[0, h])) / math.sqrt(D)
        assert r["lse"][h] == pytest.approx(want, abs=1e-13)


def test_causality_invariant(oracle_mod):
    """Changing q, k, v after position i changes no output at or before i."""
    S, bs, H, D, topk = 80, 8, 2, 8, 3
    q, k, v = rand_qkv(S, H, D, seed=24)
    base = oracle_mod.moba_full(q, k, v, [0, S], H, D, bs, topk)
    for i in (0, 7, 8, 37, 63):
        q2, k2, v2 = (x.clone() for x in (q, k, v))
        g = torch.Generator().manual_seed(i)
        for x in (q2, k2, v2):
            x[i + 1:] = bf16(torch.randn(S - i - 1, H, D, generator=g) * 3)
        r = oracle_mod.moba_full(q2, k2, v2, [0, S], H, D, bs, topk)
        for key in ("idx", "out", "lse"):
            np.testing.assert_array_equal(r[key][:i + 1], base[key][:i + 1])


def test_sequences_are_independent(oracle_mod):
    """A packed batch gives each sequence the result it gets alone."""
    H, D, bs, topk = 2, 8, 8, 3
    lens = [41, 17, 64]
    total = sum(lens)
    q, k, v = rand_qkv(total, H, D, seed=25)
    cu = [0, 41, 58, 122]
    r = oracle_mod.moba_full(q, k, v, cu, H, D, bs, topk)
    for b in range(3):
        s, e = cu[b], cu[b + 1]
        alone = oracle_mod.moba_full(q[s:e], k[s:e], v[s:e], [0, e - s], H, D, bs, topk)
        for key in ("idx", "out", "lse"):
            np.testing.assert_array_equal(r[key][s:e], alone[key])


def test_given_idx_reproduces(oracle_mod):
    S, bs, H, D, topk = 64, 8, 2, 8, 3
    q, k, v = rand_qkv(S, H, D, seed=26)
    r = oracle_mod.moba_full(q, k, v, [0, S], H, D, bs, topk)
    r2 = oracle_mod.moba_full(q, k, v, [0, S], H, D, bs, topk, given_idx=r["idx"])
    np.testing.assert_array_equal(r2["out"], r["out"])
    np.testing.assert_array_equal(r2["lse"], r["lse"])


def test_needle_queries_find_needle_blocks(oracle_mod):
    """A strong shared direction planted in a few blocks' keys and in some
    queries makes those queries route to the planted blocks."""
    w = workloads.custom([512], H=2, D=32, block_size=32, topk=4, seed=9)
    w = workloads.Workload("needle", w.seqlens, H=2, D=32, block_size=32, topks=(4,), seed=9,
                           offset_std=0.1, needle_block_frac=0.2, needle_query_frac=0.05)
    inp = workloads.make_inputs(w)
    rows = [t for t in inp.needle_queries if t // 32 > max(inp.needle_blocks)]
    assert rows
    r = oracle_mod.moba_rows(inp.q.view(512, 2, 32), inp.k.view(512, 2, 32),
                             inp.v.view(512, 2, 32), [0, 512], 2, 32, 32, 4,
                             rows, [0] * len(rows))
    nb = set(inp.needle_blocks)
    for j, t in enumerate(rows):
        past = [c for c in r["idx"][j] if 0 <= c < t // 32]
        assert set(past) == nb, (t, past, nb)
