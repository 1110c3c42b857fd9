"""The no-allocation entry point, hpa_decode_attn_combine_noalloc.

It serves callers that cannot allocate device memory during a decode step
(a plugin inside a runtime that owns the memory pool, a serving loop that
must not call cudaMalloc/cudaFree): the split partials live in a fixed array
inside the library instead of caller buffers.  Here it is called through the
C ABI three times in a row, on three different batches, and each result is
checked against hpa_decode_attn + hpa_combine with caller-allocated partials
and against the fp64 oracle, within the tolerances the other parity tests
use.  The third call needs fewer partial rows than the second, so it runs
over rows a larger earlier call left in the shared array.  This file is
collected last so a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import DeviceBatch, assert_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _existing_path(db, b, ws, out, out_lse):
    hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, ws.num_ctas,
                        ws.partial_o, ws.partial_lse, db.ks, db.vs)
    hpa.hpa_combine(ws.partial_o, ws.partial_lse, ws.taskmap, ws.num_ctas, out, out_lse)


def _noalloc_c_call(db, b, ws, out, out_lse):
    L = hpa.lib()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    kv = hpa.KV_BF16 if b.kv_dtype == "bf16" else hpa.KV_E4M3
    return L.hpa_decode_attn_combine_noalloc(
        p(db.q), p(db.k), p(db.v), kv, p(db.ks), p(db.vs), b.num_pages, p(db.indptr),
        p(db.indices), b.page_size, b.B, b.q_len, b.Hq, b.Hkv, b.d, 1.0 / math.sqrt(b.d),
        p(ws.taskmap), ws.num_ctas, p(out), p(out_lse), stream)


def _partial_rows(b, C):
    return (b.B + C - 1) * b.q_len * b.Hq


# partial rows: 2688, then 3328 (more), then 256 (fewer: stale rows of call 2 remain)
BATCHES = [
    dict(lens=[1024, 5120, 2048, 77, 9000], q_len=1, kv="bf16", C=38),
    dict(lens=[513, 20000, 64, 3000], q_len=2, kv="e4m3", C=23),
    dict(lens=[700, 40], q_len=1, kv="bf16", C=3),
]


def test_noalloc_matches_existing_entry_points_and_oracle_three_calls_in_a_row():
    rows = []
    for i, spec in enumerate(BATCHES):
        b = W.make_batch(spec["lens"], q_len=spec["q_len"], kv_dtype=spec["kv"], seed=40 + i)
        rows.append(_partial_rows(b, spec["C"]))
        db = DeviceBatch(b)
        ws = hpa.Workspace(b.B, b.q_len, b.Hq, b.d, num_ctas=spec["C"])
        ws.plan(db.lens)
        shape = (b.B, b.q_len, b.Hq, b.d)
        ref = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
        _existing_path(db, b, ws, ref, ref_lse)
        out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        out_lse = torch.full(shape[:3], float("nan"), dtype=torch.float32, device="cuda")
        rc = _noalloc_c_call(db, b, ws, out, out_lse)
        assert rc == 0, hpa.lib().hpa_error_string(rc)
        torch.cuda.synchronize()
        assert ws.status() == 0
        got = out.float().cpu().numpy()
        got_lse = out_lse.cpu().numpy()
        what = "call %d" % (i + 1)
        assert_close(got, ref.float().cpu().numpy(), b.kv_dtype, "noalloc out vs caller buffers, " + what)
        assert_lse_close(got_lse, ref_lse.cpu().numpy(), "noalloc lse vs caller buffers, " + what)
        o_ref, l_ref = oracle.attention(b)
        assert_close(got, o_ref, b.kv_dtype, "noalloc out vs oracle, " + what)
        assert_lse_close(got_lse, l_ref, "noalloc lse vs oracle, " + what)
    assert rows[1] > rows[0] and rows[2] < rows[1]


def test_noalloc_through_the_python_binding():
    b = W.make_batch([3000, 64, 9000], q_len=2, kv_dtype="e4m3", seed=47)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, b.q_len, b.Hq, b.d, num_ctas=11)
    ws.plan(db.lens)
    out = torch.empty((b.B, b.q_len, b.Hq, b.d), dtype=torch.bfloat16, device="cuda")
    out_lse = torch.empty((b.B, b.q_len, b.Hq), dtype=torch.float32, device="cuda")
    hpa.hpa_decode_attn_combine_noalloc(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap,
                                        ws.num_ctas, out, out_lse, db.ks, db.vs)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention(b)
    assert_close(out.float().cpu().numpy(), o_ref, "e4m3", "noalloc out (binding)")
    assert_lse_close(out_lse.cpu().numpy(), l_ref, "noalloc lse (binding)")


def test_noalloc_binding_rejects_bad_outputs():
    b = W.make_batch([300], q_len=1, seed=48)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 1, b.Hq, b.d, num_ctas=2)
    out = torch.empty((1, 1, b.Hq, b.d), dtype=torch.bfloat16, device="cuda")
    cases = [
        dict(out=out, out_lse=torch.empty((1, 1, b.Hq), dtype=torch.float32)),      # host lse
        dict(out=out.float(), out_lse=None),                                       # fp32 out
        dict(out=torch.empty((1, 1, b.Hq, b.d // 2), dtype=torch.bfloat16, device="cuda"),
             out_lse=None),                                                        # too small
    ]
    for c in cases:
        with pytest.raises(hpa.HpaError):
            hpa.hpa_decode_attn_combine_noalloc(db.q, db.k, db.v, db.indptr, db.indices,
                                                ws.taskmap, 2, c["out"], c["out_lse"])


def test_noalloc_rejects_problems_beyond_the_fixed_array():
    # 2000 requests x 2 tokens x 64 heads x (128 + 1) floats is ~130 MB of partials,
    # far above the 16 MiB array: rejected on the host, nothing launched.
    L = hpa.lib()
    big = 1 << 20  # aligned, non-null; never dereferenced because the size check fails first
    rc = L.hpa_decode_attn_combine_noalloc(big, big, big, 0, None, None, 100, big, big, 64,
                                           2000, 2, 64, 8, 128, 0.088, big, 38, big, None, None)
    assert rc == -6
    assert b"no-alloc" in L.hpa_error_string(rc)
