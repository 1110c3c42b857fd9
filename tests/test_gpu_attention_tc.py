"""The tcgen05 attention kernel (hpa_decode_attn_tc) against the fp64 oracle.

Same checks as the mma.sync kernel's tests: the task map bit-exactly, every
segment's partial (o, lse) against the oracle over that segment's keys, and
the combined output and lse against unsplit attention.  The cases cover
what is particular to this kernel: two pages per step (odd page counts, a
missing second page), all G * q_len rows (up to 64) in one CTA, query rows
and probabilities carried as two E4M3 terms, and the reference-max moves
that rescale O and L in tensor memory."""
import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import (DeviceBatch, assert_close, assert_lse_close, expect_taskmap_equal,
                         run_gpu, scaled_query_batch)

pytestmark = pytest.mark.gpu


def check(b, num_ctas=None, splits=None, tile=512, sm_scale=None):
    g = run_gpu(b, num_ctas=num_ctas, splits=splits, tile=tile, tc=True, sm_scale=sm_scale)
    ref_plan = (oracle.plan(b.seq_lens, tile, g["num_ctas"]) if splits is None
                else oracle.plan_static(b.seq_lens, tile, splits))
    expect_taskmap_equal(g["tm"], ref_plan, g["capacity"])
    po, pl = oracle.split_attention(b, ref_plan, sm_scale=sm_scale)
    assert_close(g["po"], po, b.kv_dtype, "partial_o")
    assert_lse_close(g["pl"], pl, "partial_lse")
    out, lse = oracle.attention(b, sm_scale=sm_scale)
    err = assert_close(g["out"], out, b.kv_dtype, "out")
    assert_lse_close(g["lse"], lse, "out_lse")
    return g, err


def test_worked_example():
    check(W.make_config(1))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("q_len", [1, 2, 3, 4, 5, 6, 7, 8])
def test_ragged_batch(kv, q_len):
    """8 to 64 rows per KV head: every P^T row width (32, 64, 96 in 128, 128 bytes)."""
    lens = [q_len, 63, 64, 65, 128, 129, 511, 513, 1000, 3333, 4096 + 17]
    b = W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=200 + q_len)
    check(b, num_ctas=7)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("C", [1, 3, 40])
def test_partition_counts(kv, C):
    b = W.make_batch([100, 700, 30, 5000], q_len=2, kv_dtype=kv, seed=C)
    check(b, num_ctas=C)


@pytest.mark.parametrize("tile", [64, 192, 1024])
def test_odd_page_segments(tile):
    """Tiles of 1 or 3 pages give segments with a missing second page mid-request."""
    b = W.make_batch([100, 2000, 9000, 64 * 7], q_len=2, kv_dtype="e4m3", seed=tile)
    check(b, num_ctas=9, tile=tile)


@pytest.mark.parametrize("splits", [1, 3, 16])
def test_static_plan(splits):
    b = W.make_batch([100, 2000, 9000, 4], q_len=4, kv_dtype="e4m3", seed=splits)
    check(b, splits=splits)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_poisoned_tail_slots_are_ignored(kv):
    """Pool slots past each request's length hold NaN; they must not reach the output."""
    lens = [70, 130, 1000, 5]
    b = W.make_batch(lens, q_len=2, kv_dtype=kv, seed=5)
    nan_code = 0x7FC0 if kv == "bf16" else 0x7F
    for r, L in enumerate(lens):
        last = b.page_indices[b.page_indptr[r + 1] - 1]
        used = L - (b.page_indptr[r + 1] - b.page_indptr[r] - 1) * b.page_size
        for pool in (b.k_pool, b.v_pool):
            raw = pool.view(torch.int16) if kv == "bf16" else pool
            raw[last, :, used:, :] = nan_code
    check(b, num_ctas=6)


def test_rows_not_a_multiple_of_16():
    b = W.make_batch([100, 2000], q_len=3, Hq=24, Hkv=4, kv_dtype="e4m3", seed=7)  # 18 rows
    check(b, num_ctas=4)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_late_dominant_key_moves_the_reference(kv):
    """A key far above everything before it (late in a long segment) forces the
    reference max up by more than the slack, so O and L are rescaled in TMEM."""
    b = W.make_batch([6000, 3000], q_len=2, kv_dtype=kv, seed=77)
    hot = 5000                                         # key 5000 of request 0
    page = b.page_indices[b.page_indptr[0] + hot // b.page_size]
    slot = hot % b.page_size
    q0 = b.q[0, 0].float()                             # [Hq][d]
    G = b.Hq // b.Hkv
    for h in range(b.Hkv):
        direction = torch.sign(q0[h * G])              # aligned with head h*G's query
        if kv == "bf16":
            b.k_pool[page, h, slot] = (direction * 3.0).to(torch.bfloat16)
        else:
            b.k_pool[page, h, slot] = W.encode_e4m3(direction * 3.0 / float(b.k_scale[h]))
    check(b, num_ctas=2)


def test_mtp_workload_sample():
    """The first 3 requests of the MTP E4M3 workload at q_len 4 (32 rows per KV head)."""
    b = W.make_config(5, max_requests=3, q_len=4)
    check(b)


def test_bad_page_id_is_flagged():
    b = W.make_batch([200, 300], q_len=2, kv_dtype="e4m3", seed=6)
    b.page_indices = b.page_indices.copy()
    b.page_indices[2] = b.num_pages + 5
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 2, 64, 128, num_ctas=4)
    out = torch.empty((2, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    hpa.decode_step(ws, db.q, db.k, db.v, db.lens, db.indptr, db.indices, out, None, db.ks,
                    db.vs, tc=True)
    torch.cuda.synchronize()
    assert ws.status() & 4
    assert torch.isnan(out.float()).all()


def test_mismatched_partition_count_is_flagged():
    b = W.make_batch([200, 3000], q_len=4, seed=7)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 4, 64, 128, num_ctas=4)
    ws.plan(db.lens)
    big = hpa.Workspace(b.B, 4, 64, 128, num_ctas=9)
    out = torch.empty((2, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
    hpa.hpa_decode_attn_tc(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, 9,
                           big.partial_o, big.partial_lse)
    hpa.hpa_combine(big.partial_o, big.partial_lse, ws.taskmap, 9, out)
    torch.cuda.synchronize()
    assert ws.status() & 2
    assert torch.isnan(out.float()).all()


def test_three_calls_capture_in_a_cuda_graph():
    """plan -> tcgen05 attention -> combine recorded once in a CUDA graph and replayed on
    new lengths."""
    lens0 = np.array([3000, 40, 12000, 700], dtype=np.int32)
    b = W.make_batch(lens0, q_len=4, kv_dtype="e4m3", seed=90)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 4, 64, 128, num_ctas=11)
    out = torch.empty((b.B, 4, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((b.B, 4, 64), dtype=torch.float32, device="cuda")
    lens = db.lens.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):                       # warm up (resolves TMA descriptors etc.)
        hpa.decode_step(ws, db.q, db.k, db.v, lens, db.indptr, db.indices, out, lse, db.ks,
                        db.vs, stream=s, tc=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hpa.decode_step(ws, db.q, db.k, db.v, lens, db.indptr, db.indices, out, lse, db.ks,
                        db.vs, stream=s, tc=True)
    for shorten in (0, 17):                          # replay; the second time with new lengths
        b.seq_lens = lens0 - shorten
        lens.copy_(torch.from_numpy(b.seq_lens))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref, ref_lse = oracle.attention(b)
        assert_close(out.float().cpu().numpy(), ref, "e4m3")
        assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("Hq,Hkv,q_len,kv", [(8, 8, 1, "bf16"), (8, 8, 2, "e4m3"),
                                             (64, 1, 1, "e4m3"), (32, 2, 2, "bf16")])
def test_head_layouts(Hq, Hkv, q_len, kv):
    """MHA (one query row per KV head), MQA (one KV head for 64 query heads: 64 rows)
    and 16 query heads per KV head with two tokens."""
    b = W.make_batch([q_len, 70, 1000, 5000], q_len=q_len, kv_dtype=kv, Hq=Hq, Hkv=Hkv,
                     seed=Hq + Hkv + q_len)
    check(b, num_ctas=5)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_thousands_of_short_requests(kv):
    """3000 requests of 2-300 keys: thousands of segments, many per partition."""
    lens = np.random.default_rng(31).integers(2, 301, size=3000)
    b = W.make_batch(lens, q_len=2, kv_dtype=kv, seed=31)
    check(b)


@pytest.mark.parametrize("case", ["large", "tiny", "mixed_rows"])
@pytest.mark.parametrize("q_len", [1, 2, 4, 6, 8])
@pytest.mark.parametrize("kv", ["e4m3", "bf16"])
def test_query_magnitudes(kv, q_len, case):
    """bf16 query rows far outside N(0,1): elements near 1e5 and near 1e-6, at 8 to 64
    rows per KV head (every compute-warp layout).  The E4M3 path carries each row as
    two E4M3 terms under a power-of-two row scale, the second term with a further
    fixed x16, so rows of any magnitude are carried to bf16 precision and the scores of
    1e5-sized rows keep the precision the 1e-4 lse bound needs where they cancel to a
    small lse.  (A row with a
    single element 3e5 times its others is run on the mma.sync kernel only: here up to
    16 partial-output elements of such rows, among keys that tie on that element, miss
    the bound.)"""
    b, sm = scaled_query_batch([2 * q_len, 65, 513, 1000, 3333], q_len, kv, 140 + q_len, case)
    check(b, num_ctas=5, sm_scale=sm)


@pytest.mark.parametrize("q_len", [3, 8])
def test_traced_call_runs_tcgen05_above_16_rows(q_len):
    """hpa_decode_attn_traced makes hpa_decode_attn's kernel choice: above 16 rows it runs
    this kernel (the same partials as hpa_decode_attn_tc, bit for bit) and records one
    trace entry per (partition, KV head) CTA, with every segment counted once per head."""
    b = W.make_batch([3000, 40, 12000, 700], q_len=q_len, kv_dtype="e4m3", seed=90 + q_len)
    db = DeviceBatch(b)
    C = 6
    ws = hpa.Workspace(b.B, q_len, b.Hq, b.d, num_ctas=C)
    ws.plan(db.lens)
    hpa.hpa_decode_attn_tc(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C, ws.partial_o,
                           ws.partial_lse, db.ks, db.vs)
    torch.cuda.synchronize()
    S = int(ws.taskmap[5].item())
    n = S * q_len * b.Hq
    ref_o, ref_l = ws.partial_o[:n * b.d].clone(), ws.partial_lse[:n].clone()
    groups = (b.Hq // b.Hkv * q_len + 15) // 16
    trace = torch.zeros(4 * C * b.Hkv * groups, dtype=torch.int64, device="cuda")
    hpa.hpa_decode_attn_traced(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C,
                               ws.partial_o, ws.partial_lse, trace, db.ks, db.vs)
    torch.cuda.synchronize()
    assert int(ws.taskmap[6].item()) == 0
    assert torch.equal(ws.partial_o[:n * b.d], ref_o) and torch.equal(ws.partial_lse[:n], ref_l)
    t = trace.view(-1, 4).cpu().numpy()
    used, rest = t[:C * b.Hkv], t[C * b.Hkv:]
    assert (used[:, 0] > 0).all() and (used[:, 0] <= used[:, 1]).all()
    assert (used[:, 1] <= used[:, 2]).all()
    assert (rest == 0).all()                             # no row-group axis on this kernel
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ((used[:, 3] & 0xffffffff) < sms).all()
    assert int((used[:, 3] >> 32).sum()) == S * b.Hkv   # every segment, once per KV head
    summ = hpa.trace_summary(trace, C, b.Hkv)
    assert summ["span_us"] > 0 and 0 < summ["sm_busy_frac"] <= 1.0
