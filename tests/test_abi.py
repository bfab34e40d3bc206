"""C ABI checks that need no GPU: the library builds and loads, exports every
entry point include/moba.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

from long_context_sparse_moba_gb300 import ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moba.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ops.LIB_PATH):
        if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build the library")
        from long_context_sparse_moba_gb300 import build
        build.build()
    return ops.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moba_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moba_attn_fwd", "moba_kpool", "moba_gate_topk", "moba_attn_fwd_varlen",
                     "moba_get_status", "moba_status_string", "moba_attn_fwd_ws",
                     "moba_attn_fwd_workspace_size"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in ops._SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert ops.status_string(0) == "MOBA_OK"
    assert ops.status_string(5) == "MOBA_ERR_TIMEOUT"
    assert ops.status_string(99) == "MOBA_ERR_UNKNOWN"


def test_options_validate_on_the_host(lib):
    """Out-of-set option values are rejected before any launch (the fake
    pointers are never dereferenced)."""
    fake = ctypes.c_void_p(0x10000)
    for field, bad in (("pooling", 7), ("pooling", -1), ("gate_kernel", 2), ("attn_kernel", 5),
                       ("debug_flags", -1), ("schedule", 2)):
        o = ops.Options()
        setattr(o, field, bad)
        assert lib.moba_kpool_ex(fake, fake, 1, 1, 64, 64, 64, ctypes.byref(o),
                                 None) == ops.MOBA_ERR_INVALID_ARG, field
        assert lib.moba_attn_fwd_ex(fake, fake, fake, fake, fake, 1, 1, 64, 64, 64, 3,
                                    ctypes.byref(o), None, 0, None) == ops.MOBA_ERR_INVALID_ARG
        assert lib.moba_attn_bwd_ex(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 1,
                                    64, 64, 64, 3, ctypes.byref(o), None, 0,
                                    None) == ops.MOBA_ERR_INVALID_ARG
    o = ops.Options()
    o.idx_out = 0x10002  # not 4-byte aligned
    assert lib.moba_attn_fwd_ex(fake, fake, fake, fake, fake, 1, 1, 64, 64, 64, 3,
                                ctypes.byref(o), None, 0, None) == ops.MOBA_ERR_INVALID_ARG
    o = ops.Options()
    o.idx_in = 0x10002  # not 4-byte aligned
    assert lib.moba_attn_bwd_ex(fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 1,
                                64, 64, 64, 3, ctypes.byref(o), None, 0,
                                None) == ops.MOBA_ERR_INVALID_ARG


def test_options_struct_layout():
    """The ctypes mirror of moba_options_t has the C layout (LP64: int x4,
    long long, two pointers, int, padding, pointer = 56 bytes)."""
    assert ctypes.sizeof(ops.Options) == 56
    assert ops.Options.wait_limit_cycles.offset == 16
    assert ops.Options.idx_out.offset == 24 and ops.Options.phase_events.offset == 32
    assert ops.Options.schedule.offset == 40 and ops.Options.idx_in.offset == 48


def test_no_process_wide_switches(lib):
    """Kernel choice, pooling, fault injection and phase timing are per call:
    the library exports no setter for them."""
    for name in ("moba_set_pooling", "moba_set_gate_kernel", "moba_set_attention_kernel",
                 "moba_debug_set", "moba_profile_begin", "moba_profile_end"):
        assert not hasattr(lib, name), name


def test_host_scratch_size(lib):
    # device copies of q, k, v, out (bf16) and lse (fp32), each from a 256-byte
    # boundary, then the forward's own workspace
    B, H, S, D = 1, 32, 32768, 128
    a256 = lambda x: (x + 255) // 256 * 256
    want = 4 * a256(B * S * H * D * 2) + a256(B * S * H * 4) + \
        lib.moba_attn_fwd_workspace_size(B, H, S, D, 512, 3)
    assert lib.moba_attn_fwd_host_scratch_size(B, H, S, D, 512, 3) == want
    assert lib.moba_attn_fwd_host_scratch_size(B, H, S, 96, 512, 3) == 0  # unsupported D


def test_workspace_size_alias(lib):
    assert lib.moba_workspace_size(1, 32, 32768, 128, 512, 3) == \
        lib.moba_attn_fwd_workspace_size(1, 32, 32768, 128, 512, 3) > 0


def test_decode_validates_on_the_host(lib):
    args = lambda **kw: [kw.get(n, FAKE) for n in ("q", "k", "v", "kbar", "lens", "out", "lse")]
    # B, H, S_max, D, bs, topk
    assert lib.moba_decode_fwd(*args(q=None), None, 1, 1, 64, 64, 64, 1, None) == 1
    assert lib.moba_decode_fwd(*args(), None, 0, 1, 64, 64, 64, 1, None) == 1
    assert lib.moba_decode_fwd(*args(), None, 1, 1, 64, 96, 64, 1, None) == 2      # head dim
    assert lib.moba_decode_fwd(*args(), None, 1, 1, 64, 64, 96, 1, None) == 1      # block size
    assert lib.moba_decode_fwd(*args(), None, 1, 1, 64 * 64, 64, 64, 40, None) == 2  # wide top-k
    assert lib.moba_decode_fwd(*args(q=ctypes.c_void_p(0x10002)), None, 1, 1, 64, 64, 64, 1,
                               None) == 1                                           # misaligned
    need = lib.moba_decode_workspace_size(2, 4, 128, 3)
    assert need > 0 and lib.moba_decode_workspace_size(2, 4, 96, 3) == 0
    assert lib.moba_decode_fwd_ws(*args(), None, 2, 4, 1024, 128, 256, 3, FAKE, need - 1,
                                  None) == ops.MOBA_ERR_WORKSPACE


def test_num_blocks(lib):
    assert ops.num_blocks(32768, 512) == 64
    assert ops.num_blocks(131072, 2048) == 64
    assert ops.num_blocks(1048576, 4096) == 256
    assert ops.num_blocks(2049, 256) == 9
    assert ops.num_blocks(0, 256) == 0


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


@pytest.mark.parametrize("B,H,S,D,bs,topk,code", [
    (0, 1, 64, 64, 64, 1, ops.MOBA_ERR_INVALID_ARG),
    (1, 0, 64, 64, 64, 1, ops.MOBA_ERR_INVALID_ARG),
    (1, 1, 0, 64, 64, 1, ops.MOBA_ERR_INVALID_ARG),
    (1, 1, 64, 64, 0, 1, ops.MOBA_ERR_INVALID_ARG),
    (1, 1, 64, 64, 96, 1, ops.MOBA_ERR_INVALID_ARG),     # block size not a multiple of 64
    (1, 1, 64, 64, 64, 0, ops.MOBA_ERR_INVALID_ARG),     # topk < 1
    (1, 1, 64, 96, 64, 1, ops.MOBA_ERR_UNSUPPORTED),     # head dim
    (1, 1, 64 * 64, 64, 64, 40, ops.MOBA_ERR_UNSUPPORTED),  # more than 31 past slots
    (1, 1, 1 << 26, 64, 64, 3, ops.MOBA_ERR_UNSUPPORTED),   # too many tokens
])
def test_attn_rejects_bad_sizes(lib, B, H, S, D, bs, topk, code):
    rc = lib.moba_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, B, H, S, D, bs, topk, None)
    assert rc == code
    assert lib.moba_attn_fwd_workspace_size(B, H, S, D, bs, topk) == 0


def test_null_and_misaligned_pointers(lib):
    assert lib.moba_attn_fwd(None, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 64, 1, None) == 1
    assert lib.moba_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 64, 64, 64, 1, None) == 1
    odd = ctypes.c_void_p(0x10002)
    assert lib.moba_attn_fwd(odd, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 64, 1, None) == 1
    assert lib.moba_kpool(None, FAKE, 1, 1, 64, 64, 64, None) == 1
    assert lib.moba_gate_topk(FAKE, FAKE, None, 1, 1, 64, 64, 64, 3, None) == 1
    assert lib.moba_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 64, 64, 1, 64, 64, 1,
                                    None) == 1


def test_workspace_too_small_is_rejected_before_launch(lib):
    need = lib.moba_attn_fwd_workspace_size(1, 2, 4096, 128, 512, 3)
    assert need > 0
    rc = lib.moba_attn_fwd_ws(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 4096, 128, 512, 3,
                              ctypes.c_void_p(0x100000), need - 1, None)
    assert rc == ops.MOBA_ERR_WORKSPACE


def test_workspace_grows_with_topk_and_dense_needs_little(lib):
    sparse = lib.moba_attn_fwd_workspace_size(1, 32, 32768, 128, 512, 3)
    wider = lib.moba_attn_fwd_workspace_size(1, 32, 32768, 128, 512, 8)
    dense = lib.moba_attn_fwd_workspace_size(1, 32, 32768, 128, 512, 64)
    assert wider > sparse > dense > 0
    # the partial outputs dominate: tokens * heads * (topk - 1) * D bf16 values
    assert sparse >= 32768 * 32 * 2 * 128 * 2


def test_backward_validates_on_the_host(lib):
    F = FAKE
    args = (1, 2, 4096, 128, 512, 3)
    # null and misaligned tensors
    assert lib.moba_attn_bwd(F, F, F, F, F, None, F, F, F, *args, None) == ops.MOBA_ERR_INVALID_ARG
    assert lib.moba_attn_bwd(F, F, F, F, F, F, F, None, F, *args, None) == ops.MOBA_ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x10002)
    assert lib.moba_attn_bwd(F, F, F, F, F, F, odd, F, F, *args, None) == ops.MOBA_ERR_INVALID_ARG
    # the forward's size rules
    assert lib.moba_attn_bwd(F, F, F, F, F, F, F, F, F, 1, 2, 4096, 96, 512, 3,
                             None) == ops.MOBA_ERR_UNSUPPORTED
    assert lib.moba_attn_bwd(F, F, F, F, F, F, F, F, F, 1, 2, 4096, 128, 500, 3,
                             None) == ops.MOBA_ERR_INVALID_ARG
    assert lib.moba_attn_bwd_varlen(F, F, F, F, F, F, F, F, F, None, 1, 64, 64, 1, 64, 64, 1,
                                    None) == ops.MOBA_ERR_INVALID_ARG
    # caller scratch: too small is refused before any launch
    need = lib.moba_attn_bwd_workspace_size(*args)
    assert need > 0
    assert lib.moba_attn_bwd_ws(F, F, F, F, F, F, F, F, F, *args, ctypes.c_void_p(0x100000),
                                need - 1, None) == ops.MOBA_ERR_WORKSPACE
    # no partial outputs, but the fp32 dq accumulator and dO . O per row
    rows = 4096 * 2
    assert need >= rows * 128 * 4 + rows * 4
    # (varlen bounds the block count by total / bs + sequences: at least as much)
    assert lib.moba_attn_bwd_varlen_workspace_size(1, 4096, 4096, 2, 128, 512, 3) >= need
