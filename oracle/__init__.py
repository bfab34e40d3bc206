"""CPU oracle of the MoBA forward and backward passes -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.  The arithmetic lives in ``moba_oracle.c`` (plain C,
double precision, OpenMP over rows); this module only compiles it with gcc and
marshals numpy arrays.

Sources: "Moonshot MoBA paper explained" (gsyq.cn/news/227272) sections 3.1
and 4.1 and "MOBA mixture of block attention for server-side long context"
(hncyxsy.com/news/197418) section 3; the readings taken where those pages are
silent are listed at the top of ``moba_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moba_oracle.c")
_LIB = os.path.join(_HERE, "libmoba_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.moba_oracle_num_blocks.restype = i64
        lib.moba_oracle_num_blocks.argtypes = [i64, i64]
        lib.moba_oracle_max_threads.restype = i32
        lib.moba_oracle_kpool.restype = i32
        lib.moba_oracle_kpool.argtypes = [p, p, i32, i32, i32, i32, p]
        lib.moba_oracle_kpool_max.argtypes = [p, p, i32, i32, i32, i32, p]
        lib.moba_oracle_rows.restype = i32
        lib.moba_oracle_bwd.restype = i32
        lib.moba_oracle_bwd.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, p, p, p, p]
        lib.moba_oracle_bwd_dq_rows.restype = i32
        lib.moba_oracle_bwd_dq_rows.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i64,
                                                p, p, p, p]
        lib.moba_oracle_rows.argtypes = [p, p, p, p, i32, i32, i32, i32, i32, p,
                                         i64, p, p, p, p, p, p, p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch, CPU) or uint16 array -> contiguous uint16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _cu(cu_seqlens) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))


def num_blocks(length: int, block_size: int) -> int:
    return int(_load().moba_oracle_num_blocks(int(length), int(block_size)))


def max_threads() -> int:
    return int(_load().moba_oracle_max_threads())


def kpool(k, cu_seqlens, H: int, D: int, block_size: int, pooling: str = "mean") -> np.ndarray:
    """Pooled keys, float64 ``[num_blocks_total, H, D]``: the mean (default) or
    the element-wise maximum of each block's keys."""
    kb = _bits(k)
    cu = _cu(cu_seqlens)
    nb = sum(num_blocks(cu[b + 1] - cu[b], block_size) for b in range(len(cu) - 1))
    out = np.zeros((nb, H, D), dtype=np.float64)
    fn = {"mean": _load().moba_oracle_kpool, "max": _load().moba_oracle_kpool_max}[pooling]
    rc = fn(_ptr(kb), _ptr(cu), len(cu) - 1, H, D, block_size, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle pooling ({pooling}) failed ({rc})")
    return out


def moba_rows(q, k, v, cu_seqlens, H: int, D: int, block_size: int, topk: int,
              row_tok, row_head, given_idx=None, kbar=None, pooling: str = "mean") -> dict:
    """Gate + attention for the listed (token, head) rows.

    Returns a dict of numpy arrays: ``idx`` int32 [R, topk] (ascending, -1
    padded), ``gap`` float64 [R], ``out`` float64 [R, D], ``lse`` float64 [R].
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cu = _cu(cu_seqlens)
    if kbar is None:
        kbar = kpool(kb, cu, H, D, block_size, pooling)
    kbar = np.ascontiguousarray(kbar, dtype=np.float64)
    rt = np.ascontiguousarray(np.asarray(row_tok, dtype=np.int64))
    rh = np.ascontiguousarray(np.asarray(row_head, dtype=np.int32))
    R = rt.shape[0]
    gi = None
    if given_idx is not None:
        gi = np.ascontiguousarray(np.asarray(given_idx, dtype=np.int32).reshape(R, topk))
    idx = np.empty((R, topk), dtype=np.int32)
    gap = np.empty(R, dtype=np.float64)
    out = np.empty((R, D), dtype=np.float64)
    lse = np.empty(R, dtype=np.float64)
    rc = _load().moba_oracle_rows(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), len(cu) - 1, H, D, block_size, topk,
        _ptr(kbar), R, _ptr(rt), _ptr(rh), _ptr(gi) if gi is not None else None,
        _ptr(idx), _ptr(gap), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"moba_oracle_rows failed ({rc})")
    return {"idx": idx, "gap": gap, "out": out, "lse": lse}


def all_rows(total: int, H: int):
    """Every (token, head) pair, token-major."""
    tok = np.repeat(np.arange(total, dtype=np.int64), H)
    head = np.tile(np.arange(H, dtype=np.int32), total)
    return tok, head


def moba_full(q, k, v, cu_seqlens, H: int, D: int, block_size: int, topk: int,
              given_idx=None, pooling: str = "mean") -> dict:
    """All rows; arrays reshaped to ``[total, H, ...]``."""
    cu = _cu(cu_seqlens)
    total = int(cu[-1])
    tok, head = all_rows(total, H)
    gi = None if given_idx is None else np.asarray(given_idx).reshape(total * H, topk)
    r = moba_rows(q, k, v, cu, H, D, block_size, topk, tok, head, given_idx=gi, pooling=pooling)
    return {"idx": r["idx"].reshape(total, H, topk), "gap": r["gap"].reshape(total, H),
            "out": r["out"].reshape(total, H, D), "lse": r["lse"].reshape(total, H)}


def moba_bwd(q, k, v, dout, cu_seqlens, H: int, D: int, block_size: int, topk: int,
             idx=None, pooling: str = "mean") -> dict:
    """Backward pass with the gate's selection held fixed: ``dq``, ``dk``,
    ``dv`` float64 ``[total, H, D]`` for the upstream gradient ``dout``.
    ``idx`` ([total, H, topk]) defaults to the oracle's own selection."""
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    cu = _cu(cu_seqlens)
    total = int(cu[-1])
    if idx is None:
        idx = moba_full(qb, kb, vb, cu, H, D, block_size, topk, pooling=pooling)["idx"]
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32).reshape(total, H, topk))
    dq = np.empty((total, H, D), dtype=np.float64)
    dk = np.empty((total, H, D), dtype=np.float64)
    dv = np.empty((total, H, D), dtype=np.float64)
    rc = _load().moba_oracle_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), _ptr(cu), len(cu) - 1,
                                 H, D, block_size, topk, _ptr(idx), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError(f"moba_oracle_bwd failed ({rc})")
    return {"dq": dq, "dk": dk, "dv": dv, "idx": idx}


def moba_bwd_dq_rows(q, k, v, dout, cu_seqlens, H: int, D: int, block_size: int, topk: int,
                     row_tok, row_head, idx) -> np.ndarray:
    """dq float64 [R, D] of the listed rows, for their selections idx [R, topk]."""
    qb, kb, vb, gb = _bits(q), _bits(k), _bits(v), _bits(dout)
    cu = _cu(cu_seqlens)
    rt = np.ascontiguousarray(np.asarray(row_tok, dtype=np.int64))
    rh = np.ascontiguousarray(np.asarray(row_head, dtype=np.int32))
    R = rt.shape[0]
    gi = np.ascontiguousarray(np.asarray(idx, dtype=np.int32).reshape(R, topk))
    dq = np.empty((R, D), dtype=np.float64)
    rc = _load().moba_oracle_bwd_dq_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), _ptr(cu),
                                         len(cu) - 1, H, D, block_size, topk, R, _ptr(rt),
                                         _ptr(rh), _ptr(gi), _ptr(dq))
    if rc != 0:
        raise ValueError(f"moba_oracle_bwd_dq_rows failed ({rc})")
    return dq
