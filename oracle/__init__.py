"""ORACLE -- test infrastructure only.

A plain, slow, obviously correct CPU implementation of split-KV GQA decode
attention, used to check the CUDA library.  Only the test suite, the smoke
check and the benchmark's CPU-baseline leg may import it; the product path
never does, and it shares no code with the CUDA library (only the seeded
input generators in `workloads` serve both).

  scheduler.py  the tile scheduler as plain loops (tile counts, stream scan,
                equal budgets, segment table) and the static comparator;
  attention.c   fp64 attention over a paged KV cache (built with gcc);
  combine()     the log-sum-exp merge of split partials, in numpy fp64.

Every function is pinned by tests in tests/test_oracle_*.py against values
the pages print, closed forms, library routines and brute force.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

from . import scheduler  # noqa: F401
from .scheduler import plan, plan_static, plan_weighted, segment_key_ranges  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attention.c with gcc into oracle/_build/liboracle.so."""
    src = os.path.join(_HERE, "attention.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", src,
                           "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            L.oracle_attention.argtypes = [P, P, P, I, P, P, P, P, P, ctypes.c_int64, I, I, I,
                                           I, I, I, D, I, P, I, P, P]
            L.oracle_attention.restype = I
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = D
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = D
            _lib = L
    return _lib


def _np(x, dtype):
    """Host array view (torch tensors are viewed through their raw bits)."""
    if hasattr(x, "numpy"):
        import torch
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.contiguous().numpy()
    return np.ascontiguousarray(x).view(dtype) if np.asarray(x).dtype != dtype else \
        np.ascontiguousarray(x)


def attention(batch, items=None, n_threads: int = 0, sm_scale: float | None = None):
    """fp64 attention of `batch` (a workloads.Batch) over `items`.

    items: list of (req, key_lo, key_hi); default: every request over all of
    its keys (the unsplit result).  Returns (out [n][q_len][Hq][d],
    lse [n][q_len][Hq]) as float64 arrays.
    """
    if items is None:
        items = [(r, 0, int(L)) for r, L in enumerate(batch.seq_lens)]
    it = np.asarray(items, dtype=np.int32).reshape(-1, 3)
    n = it.shape[0]
    q = _np(batch.q, np.uint16)
    kp = _np(batch.k_pool, np.uint16 if batch.kv_dtype == "bf16" else np.uint8)
    vp = _np(batch.v_pool, np.uint16 if batch.kv_dtype == "bf16" else np.uint8)
    ks = None if batch.k_scale is None else np.ascontiguousarray(batch.k_scale, np.float32)
    vs = None if batch.v_scale is None else np.ascontiguousarray(batch.v_scale, np.float32)
    lens = np.ascontiguousarray(batch.seq_lens, np.int32)
    indptr = np.ascontiguousarray(batch.page_indptr, np.int32)
    indices = np.ascontiguousarray(batch.page_indices, np.int32)
    out = np.zeros((n, batch.q_len, batch.Hq, batch.d), np.float64)
    lse = np.zeros((n, batch.q_len, batch.Hq), np.float64)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(batch.d)
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = lib().oracle_attention(
        ptr(q), ptr(kp), ptr(vp), 0 if batch.kv_dtype == "bf16" else 1, ptr(ks), ptr(vs),
        ptr(lens), ptr(indptr), ptr(indices), batch.num_pages, batch.page_size, batch.B,
        batch.q_len, batch.Hq, batch.Hkv, batch.d, float(sm_scale), n, ptr(it), n_threads,
        ptr(out), ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments (code %d)" % rc)
    return out, lse


def combine(partial_o, partial_lse, seg_off):
    """Log-sum-exp merge of split partials into one result per request.

    partial_o [S][q][Hq][d] holds each segment's normalised output, partial_lse
    [S][q][Hq] its log-sum-exp; segments seg_off[r]..seg_off[r+1] belong to
    request r.  Per (r, j, head): M = max_s lse_s, w_s = exp(lse_s - M),
    out = sum w_s o_s / sum w_s, lse = M + ln sum w_s.  A row that no partial
    saw a key for (M = -inf) gives out = 0, lse = -inf.
    """
    B = len(seg_off) - 1
    o = np.asarray(partial_o, np.float64)
    l = np.asarray(partial_lse, np.float64)
    out = np.zeros((B,) + o.shape[1:], np.float64)
    lse = np.zeros((B,) + l.shape[1:], np.float64)
    for r in range(B):
        a, b = int(seg_off[r]), int(seg_off[r + 1])
        M = l[a:b].max(axis=0)
        empty = np.isneginf(M)                       # no partial saw a key
        Ms = np.where(empty, 0.0, M)
        w = np.exp(l[a:b] - Ms)                      # -inf partials weigh 0
        W = w.sum(axis=0)
        Wd = np.where(empty, 1.0, W)
        out[r] = (w[..., None] * o[a:b]).sum(axis=0) / Wd[..., None]
        lse[r] = np.where(empty, -np.inf, Ms + np.log(Wd))
    return out, lse


def split_attention(batch, p, n_threads: int = 0, sm_scale: float | None = None):
    """Every segment of task map `p` as its own partial (a5), in fp64."""
    return attention(batch, segment_key_ranges(p), n_threads, sm_scale)


def split_combine(batch, p, n_threads: int = 0):
    """a5 then a6 on the oracle's own segments: must equal unsplit attention."""
    po, pl = split_attention(batch, p, n_threads)
    return combine(po, pl, p["seg_off"])
