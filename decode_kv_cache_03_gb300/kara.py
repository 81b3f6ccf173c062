"""ctypes binding of libkara.so: the C entry points under the same names.

Marshalling only: every step of the compression runs in the library's CUDA
kernels.  Tensors are torch tensors on the GPU (host tensors only where the C
signature takes h_* pointers); the library never allocates.  If libkara.so is
missing or cannot be loaded this module raises at import, so no code path can
silently fall back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkara.so")

OK, EINVAL, EUNSUPPORTED, ENOBLOCKS, EDUPBLOCK, ECUDA, EBADBLOCK, ETIMEOUT, EWORKSPACE = (
    0, -1, -2, -3, -4, -5, -6, -7, -8)


class KaraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class Params(ctypes.Structure):
    _fields_ = [("W", ctypes.c_int32), ("B", ctypes.c_int32), ("K", ctypes.c_int32),
                ("R", ctypes.c_int32), ("lam", ctypes.c_float), ("score_mode", ctypes.c_int32),
                ("select_mode", ctypes.c_int32), ("chunk", ctypes.c_int32)]


# kara_score_mode / kara_select_mode
SCORE_BIDIRECTIONAL, SCORE_CAUSAL = 0, 1
SELECT_TOKEN2CHUNK, SELECT_TOP_R, SELECT_FIXED_CHUNK = 0, 1, 2


class Cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("layer_stride", ctypes.c_int64),
                ("block_stride", ctypes.c_int64), ("head_stride", ctypes.c_int64),
                ("num_layers", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32)]


class Batch(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("len", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("bt_stride", ctypes.c_int32), ("q", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libkara.so is not built ({LIB_PATH}); run decode_kv_cache_03_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    PP, PC, PB = ctypes.POINTER(Params), ctypes.POINTER(Cache), ctypes.POINTER(Batch)
    I32, I64, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "kara_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "kara_version": ([], ctypes.c_int),
        "kara_plan": ([PP, I32, I32, P, I32, P, P, P, P], ctypes.c_int),
        "kara_workspace_size": ([PC, PP, I32], SZ),
        "kara_score": ([PC, PP, PB, P, P, SZ, P, P], ctypes.c_int),
        "kara_select": ([PP, I64, P, P, P, P], ctypes.c_int),
        "kara_compact": ([PC, PP, PB, P, P, I64, P, P, P, P, SZ, P], ctypes.c_int),
        "kara_compress_batch": ([PC, PP, PB, P, I64, P, P, P, P, P, P, SZ, P, P, P], ctypes.c_int),
        "kara_get_error": ([P, P], ctypes.c_int),
        "kara_batch_groups": ([PC, PP, PB], I32),
        "kara_compact_static": ([PC, PP, PB, P, P, I64, P, P, P, P], ctypes.c_int),
        "kara_decode_workspace_size": ([PC, I32, I32], SZ),
        "kara_compact_queries": ([PC, PP, PB, P, P, P], ctypes.c_int),
        "kara_append_queries": ([PC, PP, PB, P, P], ctypes.c_int),
        "kara_decode_attention": ([PC, I32, I32, P, P, I32, P, P, P, SZ, P, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()
EXPORTED = ("kara_status_string", "kara_version", "kara_plan", "kara_workspace_size", "kara_score",
            "kara_select", "kara_compact", "kara_compress_batch", "kara_get_error", "kara_compact_static",
            "kara_decode_workspace_size", "kara_decode_attention", "kara_compact_queries", "kara_append_queries",
            "kara_batch_groups")
STATIC_MAX_SEQS = 8192     # KARA_STATIC_MAX_SEQS


def status_string(status: int) -> str:
    return _lib.kara_status_string(int(status)).decode()


def version() -> int:
    return int(_lib.kara_version())


def _check(status: int, where: str):
    if status != OK:
        raise KaraError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def params(W, B, K, R, lam, score_mode=SCORE_BIDIRECTIONAL, select_mode=SELECT_TOKEN2CHUNK, chunk=0) -> Params:
    return Params(int(W), int(B), int(K), int(R), float(lam), int(score_mode), int(select_mode), int(chunk))


def cache(k: torch.Tensor, v: torch.Tensor, num_q_heads: int) -> Cache:
    """Describe bf16 pools laid out [layers][num_blocks][hkv][block][d] (rows contiguous)."""
    assert k.dtype == torch.bfloat16 and v.shape == k.shape and v.stride() == k.stride()
    Lyr, nb, hkv, bs, d = k.shape
    assert k.stride(4) == 1 and k.stride(3) == d
    return Cache(k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2), Lyr, nb, hkv,
                 int(num_q_heads), d, bs)


def batch(lengths: torch.Tensor, block_table: torch.Tensor, q: torch.Tensor) -> Batch:
    assert lengths.dtype == torch.int32 and block_table.dtype == torch.int32
    assert block_table.is_contiguous() and q.is_contiguous() and q.dtype == torch.bfloat16
    return Batch(int(lengths.shape[0]), lengths.data_ptr(), block_table.data_ptr(),
                 int(block_table.shape[1]), q.data_ptr())


def kara_plan(p: Params, block_size: int, h_len: torch.Tensor, bt_stride: int):
    """Host plan: (n_new[n], n_old[n], total_new, total_old) as CPU tensors / ints."""
    h_len = h_len.cpu().to(torch.int32).contiguous()
    n = h_len.shape[0]
    nn = torch.zeros(n, dtype=torch.int32)
    no = torch.zeros(n, dtype=torch.int32)
    tn, to = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(_lib.kara_plan(ctypes.byref(p), block_size, n, _ptr(h_len), bt_stride, _ptr(nn), _ptr(no),
                          ctypes.byref(tn), ctypes.byref(to)), "kara_plan")
    return nn, no, tn.value, to.value


def kara_workspace_size(c: Cache, p: Params, n: int) -> int:
    return int(_lib.kara_workspace_size(ctypes.byref(c), ctypes.byref(p), int(n)))


def kara_score(c: Cache, p: Params, b: Batch, scores: torch.Tensor, ws: torch.Tensor, err: torch.Tensor,
               stream=None):
    _check(_lib.kara_score(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), _ptr(scores), _ptr(ws),
                           ws.numel() * ws.element_size(), _ptr(err), _stream(stream)), "kara_score")


def kara_compact_queries(c: Cache, p: Params, b: Batch, kept: torch.Tensor, err: torch.Tensor, stream=None):
    """Move the kept and buffer queries of the ring b.q with the step's K/V compaction."""
    _check(_lib.kara_compact_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), _ptr(kept), _ptr(err),
                                     _stream(stream)), "kara_compact_queries")


def kara_append_queries(c: Cache, p: Params, b: Batch, q_new: torch.Tensor, stream=None):
    """Write one decode step's queries [n][layers][hq][D] into row len mod W of each ring."""
    assert q_new.dtype == torch.bfloat16 and q_new.is_contiguous()
    _check(_lib.kara_append_queries(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), _ptr(q_new),
                                    _stream(stream)), "kara_append_queries")


def kara_decode_workspace_size(c: Cache, n: int, bt_stride: int) -> int:
    return int(_lib.kara_decode_workspace_size(ctypes.byref(c), int(n), int(bt_stride)))


def kara_decode_attention(c: Cache, layer: int, lengths: torch.Tensor, block_table: torch.Tensor,
                          q: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, err: torch.Tensor, stream=None):
    """Decode attention of q [n][num_q_heads][head_dim] (bf16) over layer `layer`
    of the paged cache, read through block_table [n][bt_stride]; out is float."""
    assert lengths.dtype == torch.int32 and block_table.dtype == torch.int32 and block_table.is_contiguous()
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and out.dtype == torch.float32
    n, bt_stride = block_table.shape
    _check(_lib.kara_decode_attention(ctypes.byref(c), int(layer), int(n), _ptr(lengths), _ptr(block_table),
                                      int(bt_stride), _ptr(q), _ptr(out), _ptr(ws),
                                      ws.numel() * ws.element_size(), _ptr(err), _stream(stream)),
           "kara_decode_attention")


def kara_select(p: Params, n_windows: int, scores: torch.Tensor, cand, kept: torch.Tensor, stream=None):
    _check(_lib.kara_select(ctypes.byref(p), int(n_windows), _ptr(scores), _ptr(cand), _ptr(kept),
                            _stream(stream)), "kara_select")


def kara_compact(c: Cache, p: Params, b: Batch, kept, fresh, freed, new_len, err, ws, stream=None):
    _check(_lib.kara_compact(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), _ptr(kept), _ptr(fresh),
                             int(fresh.numel()), _ptr(freed), _ptr(new_len), _ptr(err), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "kara_compact")


def kara_compact_static(c: Cache, p: Params, b: Batch, kept, fresh, freed, new_len, err, stream=None):
    """kara_compact without a workspace (plan kept in the library's fixed array)."""
    _check(_lib.kara_compact_static(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), _ptr(kept), _ptr(fresh),
                                    int(fresh.numel()), _ptr(freed), _ptr(new_len), _ptr(err), _stream(stream)),
           "kara_compact_static")


def kara_compress_batch(c: Cache, p: Params, b: Batch, fresh, freed, new_len, ws, err, scores_out=None,
                        cand_out=None, kept_out=None, stream=None, phase_events=None):
    """phase_events: None or 5 torch.cuda.Event(enable_timing=True) recorded around the phases."""
    ev = None
    if phase_events is not None:
        assert len(phase_events) == 5
        assert all(e.cuda_event for e in phase_events), "record each event once before passing it"
        ev = (ctypes.c_void_p * 5)(*[e.cuda_event for e in phase_events])
    _check(_lib.kara_compress_batch(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b), _ptr(fresh),
                                    int(fresh.numel()), _ptr(freed), _ptr(new_len), _ptr(scores_out),
                                    _ptr(cand_out), _ptr(kept_out), _ptr(ws), ws.numel() * ws.element_size(),
                                    _ptr(err), _stream(stream), ev), "kara_compress_batch")


def kara_batch_groups(c: Cache, p: Params, b: Batch) -> int:
    """Sequence groups kara_compress_batch pipelines this batch into (1: none)."""
    r = int(_lib.kara_batch_groups(ctypes.byref(c), ctypes.byref(p), ctypes.byref(b)))
    _check(r if r < 0 else OK, "kara_batch_groups")
    return r


def kara_get_error(err: torch.Tensor, stream=None) -> int:
    return int(_lib.kara_get_error(_ptr(err), _stream(stream)))
