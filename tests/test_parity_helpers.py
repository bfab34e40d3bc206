"""The GPU tests' near-tie exclusion, checked on the CPU with hand-made
selections (no GPU, no library)."""
import numpy as np
import pytest

from long_context_sparse_moba_gb300 import workloads

from .parity import TIE_GAP, tie_masks


def test_tie_rows_exclude_their_row_and_the_disputed_blocks():
    w = workloads.custom((256, 128), H=2, D=16, block_size=32, topk=3)
    total, H = w.total, w.H
    ref = np.full((total, H, 3), -1, dtype=np.int32)
    ref[:, :, 0] = 0
    gpu = ref.copy()
    gap = np.full((total, H), np.inf)
    # row 100 of sequence 0, head 1: a near tie between blocks 1 and 2
    ref[100, 1, :2] = (1, 3)
    gpu[100, 1, :2] = (2, 3)
    gap[100, 1] = TIE_GAP / 2
    row_ok, key_ok = tie_masks(w, gpu, ref, gap)
    assert not row_ok[100, 1] and row_ok.sum() == total * H - 1
    # keys of blocks 1 and 2 of sequence 0, head 1 only
    bad = np.zeros((total, H), dtype=bool)
    bad[32:96, 1] = True
    assert np.array_equal(~key_ok, bad)


def test_tie_rows_in_a_later_sequence_map_to_its_own_tokens():
    w = workloads.custom((256, 128), H=1, D=16, block_size=32, topk=2)
    ref = np.zeros((w.total, 1, 2), dtype=np.int32)
    gpu = ref.copy()
    gap = np.full((w.total, 1), np.inf)
    t = 256 + 70                                   # sequence 1, local block 2
    ref[t, 0] = (0, 2)
    gpu[t, 0] = (1, 2)
    gap[t, 0] = 0.0
    _, key_ok = tie_masks(w, gpu, ref, gap)
    bad = np.zeros((w.total, 1), dtype=bool)
    bad[256:256 + 64, 0] = True                    # its blocks 0 and 1
    assert np.array_equal(~key_ok, bad)


def test_a_difference_away_from_a_tie_fails():
    w = workloads.custom((64,), H=1, D=16, block_size=16, topk=2)
    ref = np.zeros((64, 1, 2), dtype=np.int32)
    gpu = ref.copy()
    gpu[40, 0, 0] = 1
    gap = np.full((64, 1), 1.0)
    with pytest.raises(AssertionError):
        tie_masks(w, gpu, ref, gap)
