"""Python binding of libhpa (ctypes): the C entry points under the same names.

Argument marshalling only -- every step of the path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors; shapes are taken from them and
checked by the library, which returns an error code (raised here as
HpaError) before launching anything on bad input.  There is no CPU path: if
the shared library is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

KV_BF16, KV_E4M3 = 0, 1
STATUS_BITS = {1: "BAD_SEQLEN", 2: "MISMATCH", 4: "BAD_PAGE", 8: "TIMEOUT", 16: "OVERFLOW",
               32: "BAD_MAP"}
HEADER_WORDS = 16

_lock = threading.Lock()
_lib = None


class HpaError(RuntimeError):
    pass


def lib():
    """Load libhpa.so (building it first if it is missing or older than its sources)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if _build._stale():
                try:
                    path = _build.build()
                except Exception as e:  # no nvcc, or a compile error: fail loudly
                    raise HpaError("libhpa.so is not built and cannot be built: %s" % e)
            L = ctypes.CDLL(path)
            P, I32, I64, SZ, F = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_size_t, ctypes.c_float)
            sig = {
                "hpa_taskmap_bytes": ([I32, I32], SZ),
                "hpa_max_segments": ([I32, I32], I32),
                "hpa_static_num_ctas": ([I32, I32], I32),
                "hpa_static_taskmap_bytes": ([I32, I32], SZ),
                "hpa_default_num_ctas": ([I32, I32, I32, I32], I32),
                "hpa_plan": ([P, I32, I32, I32, P, SZ, P], ctypes.c_int),
                "hpa_plan_static": ([P, I32, I32, I32, P, SZ, P], ctypes.c_int),
                "hpa_plan_weighted": ([P, I32, I32, I32, P, SZ, P], ctypes.c_int),
                "hpa_decode_attn": ([P, P, P, I32, P, P, I64, P, P, I32, I32, I32, I32, I32,
                                     I32, F, P, I32, P, P, P], ctypes.c_int),
                "hpa_decode_attn_tc": ([P, P, P, I32, P, P, I64, P, P, I32, I32, I32, I32, I32,
                                        I32, F, P, I32, P, P, P], ctypes.c_int),
                "hpa_default_num_ctas_tc": ([I32, I32, I32, I32], I32),
                "hpa_decode_attn_mma": ([P, P, P, I32, P, P, I64, P, P, I32, I32, I32, I32, I32,
                                         I32, F, P, I32, P, P, P], ctypes.c_int),
                "hpa_default_num_ctas_mma": ([I32, I32, I32, I32], I32),
                "hpa_decode_attn_allheads": ([P, P, P, I32, P, P, I64, P, P, I32, I32, I32, I32,
                                              I32, I32, F, P, I32, P, P, P, P], ctypes.c_int),
                "hpa_default_num_ctas_allheads": ([I32, I32, I32, I32], I32),
                "hpa_decode_attn_traced": ([P, P, P, I32, P, P, I64, P, P, I32, I32, I32, I32,
                                            I32, I32, F, P, I32, P, P, P, P], ctypes.c_int),
                "hpa_combine": ([P, P, P, I32, I32, I32, I32, I32, P, P, P], ctypes.c_int),
                "hpa_arrivals_elems": ([I32, I32, I32, I32], SZ),
                "hpa_decode_attn_fused": ([P, P, P, I32, P, P, I64, P, P, I32, I32, I32, I32,
                                           I32, I32, F, P, I32, P, P, P, P, P, P],
                                          ctypes.c_int),
                "hpa_selftest_wait_timeout": ([P, I64, P], ctypes.c_int),
                "hpa_decode_attn_combine_noalloc": ([P, P, P, I32, P, P, I64, P, P, I32, I32,
                                                     I32, I32, I32, I32, F, P, I32, P, P, P],
                                                    ctypes.c_int),
                "hpa_store_kv": ([P, P, P, P, P, I64, I32, P, I32, P, F, I32, I32, P, P, P, P,
                                  I32, I32, I32, I32, P, P], ctypes.c_int),
                "hpa_error_string": ([ctypes.c_int], ctypes.c_char_p),
                "hpa_last_cuda_error": ([], ctypes.c_int),
            }
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        L = lib()
        msg = L.hpa_error_string(rc).decode()
        if rc == -5:
            msg += " (cudaError %d)" % L.hpa_last_cuda_error()
        raise HpaError("%s failed: %s (%d)" % (what, msg, rc))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise HpaError("%s must be a contiguous CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise HpaError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


# ----------------------------------------------------------------------------- sizes
def hpa_taskmap_bytes(B: int, num_ctas: int) -> int:
    return int(lib().hpa_taskmap_bytes(B, num_ctas))


def hpa_max_segments(B: int, num_ctas: int) -> int:
    return int(lib().hpa_max_segments(B, num_ctas))


def hpa_static_num_ctas(B: int, splits: int) -> int:
    return int(lib().hpa_static_num_ctas(B, splits))


def hpa_static_taskmap_bytes(B: int, splits: int) -> int:
    return int(lib().hpa_static_taskmap_bytes(B, splits))


def hpa_default_num_ctas(Hkv: int, q_len: int, kv_dtype: int, Hq: int = 64) -> int:
    c = int(lib().hpa_default_num_ctas(Hq, Hkv, q_len, kv_dtype))
    if c <= 0:
        raise HpaError("hpa_default_num_ctas failed (cudaError %d)" % lib().hpa_last_cuda_error())
    return c


def hpa_default_num_ctas_mma(Hkv: int, q_len: int, kv_dtype: int, Hq: int = 64) -> int:
    c = int(lib().hpa_default_num_ctas_mma(Hq, Hkv, q_len, kv_dtype))
    if c <= 0:
        raise HpaError("hpa_default_num_ctas_mma failed (cudaError %d)" %
                       lib().hpa_last_cuda_error())
    return c


def hpa_default_num_ctas_tc(Hkv: int, q_len: int, kv_dtype: int, Hq: int = 64) -> int:
    c = int(lib().hpa_default_num_ctas_tc(Hq, Hkv, q_len, kv_dtype))
    if c <= 0:
        raise HpaError("hpa_default_num_ctas_tc failed (cudaError %d)" %
                       lib().hpa_last_cuda_error())
    return c


def hpa_default_num_ctas_allheads(Hkv: int, q_len: int, kv_dtype: int, Hq: int = 64) -> int:
    c = int(lib().hpa_default_num_ctas_allheads(Hq, Hkv, q_len, kv_dtype))
    if c <= 0:
        raise HpaError("hpa_default_num_ctas_allheads failed (cudaError %d)" %
                       lib().hpa_last_cuda_error())
    return c


# ----------------------------------------------------------------------------- the three calls
def hpa_plan(seq_lens, tile: int, num_ctas: int, taskmap, stream=None):
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(taskmap, "taskmap")
    _check(lib().hpa_plan(_ptr(seq_lens), seq_lens.numel(), tile, num_ctas, _ptr(taskmap),
                          taskmap.numel() * taskmap.element_size(), _stream(stream)), "hpa_plan")


def hpa_plan_weighted(seq_lens, tile: int, num_ctas: int, taskmap, stream=None):
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(taskmap, "taskmap")
    _check(lib().hpa_plan_weighted(_ptr(seq_lens), seq_lens.numel(), tile, num_ctas,
                                   _ptr(taskmap), taskmap.numel() * taskmap.element_size(),
                                   _stream(stream)), "hpa_plan_weighted")


def hpa_plan_static(seq_lens, tile: int, splits: int, taskmap, stream=None):
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(taskmap, "taskmap")
    _check(lib().hpa_plan_static(_ptr(seq_lens), seq_lens.numel(), tile, splits, _ptr(taskmap),
                                 taskmap.numel() * taskmap.element_size(), _stream(stream)),
           "hpa_plan_static")


def _attn_args(q, k_pool, v_pool, page_indptr, page_indices, taskmap, k_scale, v_scale):
    """Checks shared by every attention call; returns (kv, B, q_len, Hq, d, P, Hkv, page)."""
    _dev(q, "q", torch.bfloat16)
    _dev(k_pool, "k_pool")
    _dev(v_pool, "v_pool")
    if k_pool.dtype == torch.bfloat16:
        kv = KV_BF16
    elif k_pool.dtype in (torch.uint8, torch.float8_e4m3fn):
        kv = KV_E4M3
        _dev(k_scale, "k_scale", torch.float32)
        _dev(v_scale, "v_scale", torch.float32)
    else:
        raise HpaError("unsupported KV dtype %s" % k_pool.dtype)
    if v_pool.dtype != k_pool.dtype or v_pool.shape != k_pool.shape:
        raise HpaError("k_pool and v_pool must match")
    for t, n in ((page_indptr, "page_indptr"), (page_indices, "page_indices")):
        _dev(t, n, torch.int32)
    _dev(taskmap, "taskmap")
    if q.dim() != 4 or k_pool.dim() != 4:
        raise HpaError("q must be [B][q_len][Hq][d] and the pools [P][Hkv][page][d]")
    B, q_len, Hq, d = q.shape
    P, Hkv, page, d2 = k_pool.shape
    if d2 != d:
        raise HpaError("head dim mismatch")
    if kv == KV_E4M3 and (k_scale.numel() < Hkv or v_scale.numel() < Hkv):
        raise HpaError("k_scale / v_scale need one fp32 value per KV head")
    return kv, B, q_len, Hq, d, P, Hkv, page


def _partials(partial_o, partial_lse, B, num_ctas, q_len, Hq, d):
    _dev(partial_o, "partial_o", torch.float32)
    _dev(partial_lse, "partial_lse", torch.float32)
    need = hpa_max_segments(B, num_ctas) * q_len * Hq
    if partial_lse.numel() < need or partial_o.numel() < need * d:
        raise HpaError("partial buffers too small: need (B + num_ctas - 1) segments")


def _outputs(out, out_lse, B, q_len, Hq, d):
    _dev(out, "out", torch.bfloat16)
    if tuple(out.shape) != (B, q_len, Hq, d):
        raise HpaError("out must have q's shape %s, got %s" % ((B, q_len, Hq, d),
                                                               tuple(out.shape)))
    if out_lse is not None:
        _dev(out_lse, "out_lse", torch.float32)
        if tuple(out_lse.shape) != (B, q_len, Hq):
            raise HpaError("out_lse must have shape %s" % ((B, q_len, Hq),))


def hpa_decode_attn(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas: int,
                    partial_o, partial_lse, k_scale=None, v_scale=None,
                    sm_scale: float | None = None, stream=None, tc: bool = False,
                    mma: bool = False):
    """q bf16 [B][q_len][Hq][d]; k/v pools bf16 or uint8 (E4M3) [P][Hkv][page][d].

    hpa_decode_attn picks the kernel by query rows per KV head (mma.sync up to 16,
    tcgen05 above); tc=True calls hpa_decode_attn_tc and mma=True hpa_decode_attn_mma
    with the same arguments."""
    kv, B, q_len, Hq, d, P, Hkv, page = _attn_args(q, k_pool, v_pool, page_indptr,
                                                   page_indices, taskmap, k_scale, v_scale)
    _partials(partial_o, partial_lse, B, num_ctas, q_len, Hq, d)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    name = "hpa_decode_attn_tc" if tc else "hpa_decode_attn_mma" if mma else "hpa_decode_attn"
    _check(getattr(lib(), name)(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), kv, _ptr(k_scale), _ptr(v_scale), P,
        _ptr(page_indptr), _ptr(page_indices), page, B, q_len, Hq, Hkv, d, float(sm_scale),
        _ptr(taskmap), num_ctas, _ptr(partial_o), _ptr(partial_lse), _stream(stream)), name)


def hpa_decode_attn_mma(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas: int,
                        partial_o, partial_lse, k_scale=None, v_scale=None,
                        sm_scale: float | None = None, stream=None):
    """hpa_decode_attn computed by the mma.sync kernel at any query-row count."""
    hpa_decode_attn(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas, partial_o,
                    partial_lse, k_scale, v_scale, sm_scale, stream, mma=True)


def hpa_decode_attn_tc(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas: int,
                       partial_o, partial_lse, k_scale=None, v_scale=None,
                       sm_scale: float | None = None, stream=None):
    """hpa_decode_attn computed on the tcgen05 tensor cores (one pass for up to 64 rows)."""
    hpa_decode_attn(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas, partial_o,
                    partial_lse, k_scale, v_scale, sm_scale, stream, tc=True)


def hpa_decode_attn_allheads(q, k_pool, v_pool, page_indptr, page_indices, taskmap,
                             num_ctas: int, partial_o, partial_lse, k_scale=None, v_scale=None,
                             sm_scale: float | None = None, trace=None, stream=None):
    """hpa_decode_attn with every KV head walked inside the CTA of a partition (grid over
    partitions only); num_ctas counts partitions of the whole grid.  trace: optional int64
    [4 * num_ctas * row groups] per-CTA timestamps."""
    kv, B, q_len, Hq, d, P, Hkv, page = _attn_args(q, k_pool, v_pool, page_indptr,
                                                   page_indices, taskmap, k_scale, v_scale)
    _partials(partial_o, partial_lse, B, num_ctas, q_len, Hq, d)
    if trace is not None:
        _dev(trace, "trace", torch.int64)
        if trace.numel() < 4 * num_ctas * ((Hq // Hkv * q_len + 15) // 16):
            raise HpaError("trace buffer too small")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(lib().hpa_decode_attn_allheads(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), kv, _ptr(k_scale), _ptr(v_scale), P,
        _ptr(page_indptr), _ptr(page_indices), page, B, q_len, Hq, Hkv, d, float(sm_scale),
        _ptr(taskmap), num_ctas, _ptr(partial_o), _ptr(partial_lse), _ptr(trace),
        _stream(stream)), "hpa_decode_attn_allheads")


def hpa_decode_attn_traced(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas: int,
                           partial_o, partial_lse, trace, k_scale=None, v_scale=None,
                           sm_scale: float | None = None, stream=None):
    """hpa_decode_attn plus per-CTA timestamps: trace is int64 [num_ctas * Hkv * 4] on device."""
    kv, B, q_len, Hq, d, P, Hkv, page = _attn_args(q, k_pool, v_pool, page_indptr,
                                                   page_indices, taskmap, k_scale, v_scale)
    _partials(partial_o, partial_lse, B, num_ctas, q_len, Hq, d)
    _dev(trace, "trace", torch.int64)
    groups = (Hq // Hkv * q_len + 15) // 16
    if trace.numel() < 4 * num_ctas * Hkv * groups:
        raise HpaError("trace buffer too small")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(lib().hpa_decode_attn_traced(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), kv, _ptr(k_scale), _ptr(v_scale), P,
        _ptr(page_indptr), _ptr(page_indices), page, B, q_len, Hq, Hkv, d, float(sm_scale),
        _ptr(taskmap), num_ctas, _ptr(partial_o), _ptr(partial_lse), _ptr(trace),
        _stream(stream)), "hpa_decode_attn_traced")


def trace_summary(trace, num_ctas: int, Hkv: int, groups: int = 1) -> dict:
    """SM busy and tail figures from a hpa_decode_attn_traced buffer (host-side arithmetic)."""
    import numpy as np
    t = trace.view(-1, 4).cpu().numpy().astype(np.int64)[:num_ctas * Hkv * groups]
    entry, go, end, info = t[:, 0], t[:, 1], t[:, 2], t[:, 3]
    sm = info & 0xffffffff
    busy = t[(info >> 32) > 0]
    t0 = int(entry.min())
    span = int(end.max()) - t0
    ends = np.sort(busy[:, 2]) if len(busy) else np.sort(end)
    per_sm = {}
    for s_, a, b_ in zip(sm, go, end):
        per_sm.setdefault(int(s_), []).append((int(a), int(b_)))
    occ = []
    for iv in per_sm.values():
        iv.sort()
        tot, cur_a, cur_b = 0, iv[0][0], iv[0][1]
        for a, b_ in iv[1:]:
            if a > cur_b:
                tot += cur_b - cur_a
                cur_a, cur_b = a, b_
            else:
                cur_b = max(cur_b, b_)
        occ.append(tot + cur_b - cur_a)
    return {"span_us": span / 1e3,
            "first_go_us": (int(go.min()) - t0) / 1e3,
            "median_cta_end_us": (float(np.median(ends)) - t0) / 1e3,
            "last_cta_tail_us": (float(ends[-1]) - float(np.median(ends))) / 1e3,
            "sm_busy_frac": float(np.mean(occ)) / span if span > 0 else 0.0,
            "sms_used": len(per_sm)}


def hpa_arrivals_elems(B: int, Hq: int, Hkv: int, q_len: int) -> int:
    return int(lib().hpa_arrivals_elems(B, Hq, Hkv, q_len))


def hpa_decode_attn_fused(q, k_pool, v_pool, page_indptr, page_indices, taskmap, num_ctas: int,
                          partial_o, partial_lse, out, arrivals, out_lse=None, k_scale=None,
                          v_scale=None, sm_scale: float | None = None, stream=None):
    """Attention with the combine folded in; arrivals: int32, hpa_arrivals_elems(B, Hq, Hkv,
    q_len) elements, zero between calls."""
    kv, B, q_len, Hq, d, P, Hkv, page = _attn_args(q, k_pool, v_pool, page_indptr,
                                                   page_indices, taskmap, k_scale, v_scale)
    _partials(partial_o, partial_lse, B, num_ctas, q_len, Hq, d)
    _outputs(out, out_lse, B, q_len, Hq, d)
    _dev(arrivals, "arrivals", torch.int32)
    if arrivals.numel() < hpa_arrivals_elems(B, Hq, Hkv, q_len):
        raise HpaError("arrivals has the wrong size")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(lib().hpa_decode_attn_fused(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), kv, _ptr(k_scale), _ptr(v_scale), P,
        _ptr(page_indptr), _ptr(page_indices), page, B, q_len, Hq, Hkv, d, float(sm_scale),
        _ptr(taskmap), num_ctas, _ptr(partial_o), _ptr(partial_lse), _ptr(out), _ptr(out_lse),
        _ptr(arrivals), _stream(stream)), "hpa_decode_attn_fused")


def hpa_combine(partial_o, partial_lse, taskmap, num_ctas: int, out, out_lse=None, stream=None):
    """out bf16 [B][q_len][Hq][d]; out_lse fp32 [B][q_len][Hq] or None."""
    _dev(partial_o, "partial_o", torch.float32)
    _dev(partial_lse, "partial_lse", torch.float32)
    _dev(taskmap, "taskmap")
    _dev(out, "out", torch.bfloat16)
    if out.dim() != 4:
        raise HpaError("out must be [B][q_len][Hq][d]")
    B, q_len, Hq, d = out.shape
    _outputs(out, out_lse, B, q_len, Hq, d)
    _partials(partial_o, partial_lse, B, num_ctas, q_len, Hq, d)
    _check(lib().hpa_combine(_ptr(partial_o), _ptr(partial_lse), _ptr(taskmap), B, num_ctas,
                             q_len, Hq, d, _ptr(out), _ptr(out_lse), _stream(stream)),
           "hpa_combine")


def hpa_selftest_wait_timeout(status, limit_ns: int, stream=None):
    """Run the bounded-wait diagnostic; status: int32 CUDA tensor of >= 1 element."""
    _dev(status, "status", torch.int32)
    _check(lib().hpa_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)),
           "hpa_selftest_wait_timeout")


def hpa_decode_attn_combine_noalloc(q, k_pool, v_pool, page_indptr, page_indices, taskmap,
                                    num_ctas: int, out, out_lse=None, k_scale=None,
                                    v_scale=None, sm_scale: float | None = None, stream=None):
    """Attention + combine with the split partials in the library's fixed device array.

    For callers that cannot allocate device memory during a decode step (a
    plugin inside a runtime that owns the memory pool, a serving loop that
    must not call cudaMalloc/cudaFree).  Calls that overlap on the GPU share
    that array and race; serialise them.
    """
    kv, B, q_len, Hq, d, P, Hkv, page = _attn_args(q, k_pool, v_pool, page_indptr,
                                                   page_indices, taskmap, k_scale, v_scale)
    _outputs(out, out_lse, B, q_len, Hq, d)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    _check(lib().hpa_decode_attn_combine_noalloc(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), kv, _ptr(k_scale), _ptr(v_scale), P,
        _ptr(page_indptr), _ptr(page_indices), page, B, q_len, Hq, Hkv, d, float(sm_scale),
        _ptr(taskmap), num_ctas, _ptr(out), _ptr(out_lse), _stream(stream)),
        "hpa_decode_attn_combine_noalloc")


def hpa_store_kv(k_new, v_new, seq_lens, page_indptr, page_indices, cos_sin, norm_w, k_pool,
                 v_pool, eps: float = 1e-6, use_hadamard: bool = True, k_scale=None,
                 v_scale=None, status=None, stream=None):
    """Fused RoPE + RMSNorm + Hadamard + quantise + paged store of the new tokens' K/V.

    k_new, v_new: bf16 [B][q_len][Hkv][d]; cos_sin: fp32 [max_pos][d]; norm_w: fp32 [d];
    pools: bf16 or uint8 (E4M3) [P][Hkv][page][d] (E4M3 needs k_scale / v_scale)."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _dev(t, n, torch.bfloat16)
    _dev(cos_sin, "cos_sin", torch.float32)
    _dev(norm_w, "norm_w", torch.float32)
    for t, n in ((seq_lens, "seq_lens"), (page_indptr, "page_indptr"),
                 (page_indices, "page_indices")):
        _dev(t, n, torch.int32)
    _dev(k_pool, "k_pool")
    _dev(v_pool, "v_pool")
    kv = KV_BF16 if k_pool.dtype == torch.bfloat16 else KV_E4M3
    B, q_len, Hkv, d = k_new.shape
    P, Hkv2, page, _ = k_pool.shape
    if Hkv2 != Hkv:
        raise HpaError("KV head count mismatch")
    _check(lib().hpa_store_kv(
        _ptr(k_new), _ptr(v_new), _ptr(seq_lens), _ptr(page_indptr), _ptr(page_indices), P,
        page, _ptr(cos_sin), cos_sin.shape[0], _ptr(norm_w), float(eps), int(use_hadamard), kv,
        _ptr(k_scale), _ptr(v_scale), _ptr(k_pool), _ptr(v_pool), B, q_len, Hkv, d,
        _ptr(status), _stream(stream)), "hpa_store_kv")


# ----------------------------------------------------------------------------- workspace helper
class Workspace:
    """Device buffers for one decode step: task map and split partials.

    Sized once for (B, num_ctas, q_len, Hq, d) -- dynamic map by default, or
    the static comparator with `splits`.  Allocation is done with torch; the
    library itself never allocates.  num_ctas (partitions per KV head) is
    normally hpa_default_num_ctas(...), which follows hpa_decode_attn's kernel
    choice (mma.sync up to 16 query rows per KV head, tcgen05 above);
    hpa_default_num_ctas_mma / _tc size for a forced kernel.  Either kernel
    accepts any partition count.
    """

    def __init__(self, B, q_len, Hq, d, num_ctas=None, splits=None, device="cuda", Hkv=8,
                 weighted=False):
        if splits is not None:
            self.num_ctas = hpa_static_num_ctas(B, splits)
            nbytes = hpa_static_taskmap_bytes(B, splits)
        else:
            self.num_ctas = num_ctas
            nbytes = hpa_taskmap_bytes(B, num_ctas)
        cap = hpa_max_segments(B, self.num_ctas)   # partial rows, valid for either map
        if nbytes == 0 or cap == 0:
            raise HpaError("workspace size query failed")
        self.splits = splits
        self.weighted = weighted
        self.capacity = cap
        self.taskmap = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device=device)
        self.partial_o = torch.empty(cap * q_len * Hq * d, dtype=torch.float32, device=device)
        self.partial_lse = torch.empty(cap * q_len * Hq, dtype=torch.float32, device=device)
        self.arrivals = torch.zeros(hpa_arrivals_elems(B, Hq, Hkv, q_len), dtype=torch.int32,
                                    device=device)  # fused combine

    def plan(self, seq_lens, tile=512, stream=None):
        if self.splits is not None:
            hpa_plan_static(seq_lens, tile, self.splits, self.taskmap, stream)
        elif self.weighted:
            hpa_plan_weighted(seq_lens, tile, self.num_ctas, self.taskmap, stream)
        else:
            hpa_plan(seq_lens, tile, self.num_ctas, self.taskmap, stream)

    def status(self) -> int:
        """Status word of the map (synchronises the current stream)."""
        return int(self.taskmap[6].item())


def decode_step(ws: Workspace, q, k_pool, v_pool, seq_lens, page_indptr, page_indices, out,
                out_lse=None, k_scale=None, v_scale=None, tile=512, plan=True, stream=None,
                fused=False, tc=False, sm_scale: float | None = None, allheads=False,
                mma=False):
    """plan (optional) -> split-KV attention -> combine, all enqueued on one stream.

    fused=True runs the attention kernel with the combine folded in (one launch);
    The attention call is hpa_decode_attn, which picks its kernel by query rows per KV
    head (size the workspace with hpa_default_num_ctas); tc=True forces the tcgen05
    kernel (hpa_default_num_ctas_tc), mma=True the mma.sync kernel
    (hpa_default_num_ctas_mma), allheads=True the mma.sync variant with every KV head
    inside the CTA (hpa_default_num_ctas_allheads); sm_scale defaults to 1/sqrt(d)."""
    if fused and tc:
        raise HpaError("the tcgen05 kernel has no fused-combine variant")
    if allheads and (fused or tc):
        raise HpaError("the all-heads variant has no fused or tcgen05 form")
    if plan:
        ws.plan(seq_lens, tile, stream)
    if fused:
        hpa_decode_attn_fused(q, k_pool, v_pool, page_indptr, page_indices, ws.taskmap,
                              ws.num_ctas, ws.partial_o, ws.partial_lse, out, ws.arrivals,
                              out_lse, k_scale, v_scale, sm_scale=sm_scale, stream=stream)
        return
    if allheads:
        hpa_decode_attn_allheads(q, k_pool, v_pool, page_indptr, page_indices, ws.taskmap,
                                 ws.num_ctas, ws.partial_o, ws.partial_lse, k_scale, v_scale,
                                 sm_scale=sm_scale, stream=stream)
    else:
        hpa_decode_attn(q, k_pool, v_pool, page_indptr, page_indices, ws.taskmap, ws.num_ctas,
                        ws.partial_o, ws.partial_lse, k_scale, v_scale, sm_scale=sm_scale,
                        stream=stream, tc=tc, mma=mma)
    hpa_combine(ws.partial_o, ws.partial_lse, ws.taskmap, ws.num_ctas, out, out_lse, stream)
