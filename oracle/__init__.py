"""CPU oracle for Kara's decode-time KV-cache compression step.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the library and its Python binding never
do.  The arithmetic lives in ``kara_oracle.c`` (plain C, fp64 scoring); this
module compiles it with gcc and marshals numpy/torch CPU arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kara_oracle.c")
_LIB = os.path.join(_HERE, "libkara_oracle.so")

OK, EINVAL, ENOBLOCKS, EDUPBLOCK, EBADBLOCK = 0, -1, -3, -4, -6


class Shape(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int32), ("layers", ctypes.c_int32), ("hq", ctypes.c_int32),
        ("hkv", ctypes.c_int32), ("d", ctypes.c_int32), ("block", ctypes.c_int32),
        ("W", ctypes.c_int32), ("B", ctypes.c_int32), ("K", ctypes.c_int32), ("R", ctypes.c_int32),
        ("lam", ctypes.c_float), ("bt_stride", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("layer_stride", ctypes.c_int64), ("block_stride", ctypes.c_int64),
        ("head_stride", ctypes.c_int64),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        _lib.kro_scores.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, ctypes.c_int]
        _lib.kro_scores_causal.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, ctypes.c_int]
        _lib.kro_select_mode.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_float, P, P, P]
        _lib.kro_select_mode_batch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_float, P, P, P, ctypes.c_int]
        _lib.kro_select.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                    P, P, P, P, P]
        _lib.kro_select_batch.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_float, P, P, P, ctypes.c_int]
        _lib.kro_plan.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, P, P]
        _lib.kro_compact.argtypes = [ctypes.POINTER(Shape), P, P, P, P, P, P, ctypes.c_int64, P, P]
        _lib.kro_max_threads.restype = ctypes.c_int
        _lib.kro_compact_queries.argtypes = [ctypes.POINTER(Shape), P, P, P]
        _lib.kro_decode_attention.argtypes = [ctypes.POINTER(Shape), ctypes.c_int, P, P, P, P, P, P, ctypes.c_int]
    return _lib


def max_threads() -> int:
    return int(lib().kro_max_threads())


def _np(t, dtype):
    """A C-contiguous numpy array of the given dtype (bf16 torch tensors -> uint16 bits)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        if dtype == np.uint16 and a.dtype == np.int16:
            a = a.view(np.uint16)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def make_shape(n_seq, layers, hq, hkv, d, block, W, B, K, R, lam, bt_stride, num_blocks,
               pool_shape=None) -> Shape:
    """Shape record; pool_shape = (layers, num_blocks, hkv, block, d) for dense pools."""
    if pool_shape is None:
        pool_shape = (layers, num_blocks, hkv, block, d)
    _, nb, h, b, dd = pool_shape
    return Shape(n_seq, layers, hq, hkv, d, block, W, B, K, R, lam, bt_stride, num_blocks,
                 nb * h * b * dd, h * b * dd, b * dd)


def shape_of(wl) -> Shape:
    s = wl.spec
    return make_shape(s.n_seq, s.layers, s.hq, s.hkv, s.d, s.block, s.W, s.B, s.K, s.R, s.lam,
                      wl.bt_stride, wl.num_blocks)


def scores(shape: Shape, q, kpool, block_table, lengths, with_colsum=False, nthreads=None, causal=False):
    """fp32 scores [n_seq][layers][hkv][C] (and fp64 full column sums [.., W]).
    causal=True: the unidirectional scoring ablation (kro_scores_causal)."""
    qa = _np(q, np.uint16)
    ka = _np(kpool, np.uint16)
    bt = _np(block_table, np.int32)
    ln = _np(lengths, np.int32)
    C = shape.W - shape.B
    out = np.zeros((shape.n_seq, shape.layers, shape.hkv, C), dtype=np.float32)
    cs = np.zeros((shape.n_seq, shape.layers, shape.hkv, shape.W), dtype=np.float64) if with_colsum else None
    fn = lib().kro_scores_causal if causal else lib().kro_scores
    st = fn(ctypes.byref(shape), _ptr(qa), _ptr(ka), _ptr(bt), _ptr(ln), _ptr(out),
            _ptr(cs) if cs is not None else None, int(nthreads or max_threads()))
    if st != OK:
        raise ValueError(f"oracle scores failed: status {st}")
    return (out, cs) if with_colsum else out


def select(s, K: int, R: int, lam: float, with_chunks=False):
    """One window: cand[K], kept[R] (and chunk scores / taken flags)."""
    sa = _np(s, np.float32).reshape(-1)
    C = sa.shape[0]
    cand = np.zeros(K, np.int32)
    kept = np.zeros(R, np.int32)
    csc = np.zeros(max(K - 1, 1), np.float32)
    tk = np.zeros(max(K - 1, 1), np.uint8)
    st = lib().kro_select(C, K, R, ctypes.c_float(lam), _ptr(sa), _ptr(cand), _ptr(kept),
                          _ptr(csc), _ptr(tk))
    if st != OK:
        raise ValueError(f"oracle select failed: status {st}")
    if with_chunks:
        return cand, kept, csc[:K - 1], tk[:K - 1].astype(bool)
    return cand, kept


def select_batch(scores_arr, K: int, R: int, lam: float, nthreads=None):
    """scores [..., C] -> cand [..., K], kept [..., R]."""
    sa = _np(scores_arr, np.float32)
    lead = sa.shape[:-1]
    C = sa.shape[-1]
    nwin = int(np.prod(lead)) if lead else 1
    cand = np.zeros(lead + (K,), np.int32)
    kept = np.zeros(lead + (R,), np.int32)
    st = lib().kro_select_batch(nwin, C, K, R, ctypes.c_float(lam), _ptr(sa), _ptr(cand),
                                _ptr(kept), int(nthreads or max_threads()))
    if st != OK:
        raise ValueError(f"oracle select failed: status {st}")
    return cand, kept


def decode_attention(shape: Shape, layer: int, q, kpool, vpool, block_table, lengths, nthreads=None):
    """Decode attention of one query per (sequence, query head) over the paged
    cache of one layer: float [n_seq][hq][d]."""
    qa = _np(q, np.uint16)
    ka = _np(kpool, np.uint16)
    va = _np(vpool, np.uint16)
    bt = _np(block_table, np.int32)
    ln = _np(lengths, np.int32)
    out = np.zeros((shape.n_seq, shape.hq, shape.d), np.float32)
    st = lib().kro_decode_attention(ctypes.byref(shape), int(layer), _ptr(qa), _ptr(ka), _ptr(va), _ptr(bt),
                                    _ptr(ln), _ptr(out), int(nthreads or max_threads()))
    if st != OK:
        raise ValueError(f"oracle decode attention failed: status {st}")
    return out


def compact_queries(shape: Shape, q_ring, lengths, kept):
    """The query ring [n_seq][layers][hq][W][d] (bf16 bits) after the step
    moves the kept and buffer queries with K and V; returns a new array."""
    qa = _np(q_ring, np.uint16).copy()
    ln = _np(lengths, np.int32)
    kp = _np(kept, np.int32)
    st = lib().kro_compact_queries(ctypes.byref(shape), _ptr(qa), _ptr(ln), _ptr(kp))
    if st != OK:
        raise ValueError(f"oracle query compaction failed: status {st}")
    return qa


SELECT_TOKEN2CHUNK, SELECT_TOP_R, SELECT_FIXED_CHUNK = 0, 1, 2


def select_mode(s, K: int, R: int, lam: float, mode: int, chunk: int = 0):
    """One window under selection mode 0 (Token2Chunk), 1 (token Top-R) or 2
    (fixed chunks of `chunk` tokens): cand[K], kept[R]."""
    sa = _np(s, np.float32).reshape(-1)
    cand = np.zeros(K, np.int32)
    kept = np.zeros(R, np.int32)
    st = lib().kro_select_mode(int(mode), int(chunk), sa.shape[0], K, R, ctypes.c_float(lam), _ptr(sa),
                               _ptr(cand), _ptr(kept))
    if st != OK:
        raise ValueError(f"oracle select failed: status {st}")
    return cand, kept


def select_mode_batch(scores_arr, K: int, R: int, lam: float, mode: int, chunk: int = 0, nthreads=None):
    """scores [..., C] -> cand [..., K], kept [..., R] under a selection mode."""
    sa = _np(scores_arr, np.float32)
    lead = sa.shape[:-1]
    C = sa.shape[-1]
    nwin = int(np.prod(lead)) if lead else 1
    cand = np.zeros(lead + (K,), np.int32)
    kept = np.zeros(lead + (R,), np.int32)
    st = lib().kro_select_mode_batch(int(mode), int(chunk), nwin, C, K, R, ctypes.c_float(lam), _ptr(sa),
                                     _ptr(cand), _ptr(kept), int(nthreads or max_threads()))
    if st != OK:
        raise ValueError(f"oracle select failed: status {st}")
    return cand, kept


def plan(lengths, W: int, B: int, R: int, block: int, bt_stride: int):
    ln = _np(lengths, np.int32)
    n = ln.shape[0]
    nn = np.zeros(n, np.int32)
    no = np.zeros(n, np.int32)
    st = lib().kro_plan(n, _ptr(ln), W, B, R, block, bt_stride, _ptr(nn), _ptr(no))
    if st != OK:
        raise ValueError(f"oracle plan failed: status {st}")
    return nn, no


def compact(shape: Shape, kpool, vpool, block_table, lengths, kept, fresh):
    """Returns (k', v', bt', freed, new_len) as new numpy arrays; inputs are not modified.

    Returns the status instead of raising when the oracle rejects the inputs:
    (status, None, None, None, None, None)."""
    ka = _np(kpool, np.uint16).copy()
    va = _np(vpool, np.uint16).copy()
    bt = _np(block_table, np.int32).copy()
    ln = _np(lengths, np.int32)
    kp = _np(kept, np.int32)
    fr = _np(fresh, np.int32)
    nn, no = None, None
    n_old_total = 0
    try:
        nn, no = plan(ln, shape.W, shape.B, shape.R, shape.block, shape.bt_stride)
        n_old_total = int(no.sum())
    except ValueError:
        pass
    freed = np.full(max(n_old_total, 1), -1, np.int32)
    new_len = np.zeros(ln.shape[0], np.int32)
    st = lib().kro_compact(ctypes.byref(shape), _ptr(ka), _ptr(va), _ptr(bt), _ptr(ln), _ptr(kp),
                           _ptr(fr), fr.shape[0], _ptr(freed), _ptr(new_len))
    if st != OK:
        return st, None, None, None, None, None
    return OK, ka, va, bt, freed[:n_old_total], new_len
