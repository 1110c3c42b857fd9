"""Split-KV attention (the mma.sync kernel) and combine on the GPU against the fp64 oracle.

Every case checks (i) the task map bit-exactly, (ii) every segment's partial
(o, lse) against the oracle's attention over that segment's keys, and (iii)
the combined output and lse against the oracle's unsplit attention."""
import math

import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import (DeviceBatch, assert_close, assert_lse_close, expect_taskmap_equal,
                         run_gpu, scaled_query_batch)

pytestmark = pytest.mark.gpu


def check(b, num_ctas=None, splits=None, tile=512, db=None, check_partials=True, fused=False,
          weighted=False, sm_scale=None, allheads=False, mma=True):
    """This file covers the mma.sync kernel: hpa_decode_attn_mma unless asked otherwise
    (hpa_decode_attn runs the same kernel up to 16 query rows per KV head)."""
    g = run_gpu(b, num_ctas=num_ctas, splits=splits, tile=tile, db=db, fused=fused,
                weighted=weighted, sm_scale=sm_scale, allheads=allheads, mma=mma)
    check_partials = check_partials and not fused  # fused: single-segment partials skipped
    if weighted:
        ref_plan = oracle.plan_weighted(b.seq_lens, tile, g["num_ctas"])
    elif splits is None:
        ref_plan = oracle.plan(b.seq_lens, tile, g["num_ctas"])
    else:
        ref_plan = oracle.plan_static(b.seq_lens, tile, splits)
    expect_taskmap_equal(g["tm"], ref_plan, g["capacity"])
    if check_partials:
        po, pl = oracle.split_attention(b, ref_plan, sm_scale=sm_scale)
        assert_close(g["po"], po, b.kv_dtype, "partial_o")
        assert_lse_close(g["pl"], pl, "partial_lse")
    out, lse = oracle.attention(b, sm_scale=sm_scale)
    err = assert_close(g["out"], out, b.kv_dtype, "out")
    assert_lse_close(g["lse"], lse, "out_lse")
    return g, err


def test_worked_example():
    b = W.make_config(1)
    g, _ = check(b)
    assert list(np.diff(g["tm"]["cta_begin"])) == [4, 4, 4, 4]


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("q_len", [1, 2])
@pytest.mark.parametrize("C", [1, 5, 23])
def test_ragged_batch(kv, q_len, C):
    lens = [2, 63, 64, 65, 511, 512, 513, 1000, 3333, 4096 + 17]
    b = W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=11 + C)
    check(b, num_ctas=C)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_more_partitions_than_tiles(kv):
    b = W.make_batch([100, 700, 30], kv_dtype=kv, seed=2)
    check(b, num_ctas=40)


@pytest.mark.parametrize("L,q_len", [(1, 1), (2, 2), (64, 1), (65, 2), (512, 1), (513, 2)])
def test_tiny_requests(L, q_len):
    b = W.make_batch([L], q_len=q_len, seed=L)
    check(b, num_ctas=3)


@pytest.mark.parametrize("tile", [64, 128, 1024])
def test_tile_sizes(tile):
    b = W.make_batch([100, 2000, 9000, 64 * 7], q_len=2, seed=tile)
    check(b, num_ctas=9, tile=tile)


@pytest.mark.parametrize("splits", [1, 3, 16])
@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_static_plan_same_kernels(splits, kv):
    b = W.make_batch([100, 2000, 9000, 1], kv_dtype=kv, seed=splits)
    check(b, splits=splits)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("q_len", [1, 2])
def test_poisoned_tail_slots_are_ignored(kv, q_len):
    """Pool slots past each request's length hold NaN; they must not reach the output."""
    lens = [70, 130, 1000, 5]
    b = W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=5)
    nan_code = 0x7FC0 if kv == "bf16" else 0x7F
    for r, L in enumerate(lens):
        last = b.page_indices[b.page_indptr[r + 1] - 1]
        used = L - (len(range(b.page_indptr[r], b.page_indptr[r + 1])) - 1) * b.page_size
        for pool in (b.k_pool, b.v_pool):
            raw = pool.view(torch.int16) if kv == "bf16" else pool
            raw[last, :, used:, :] = nan_code
    check(b, num_ctas=6)


def test_gqa_groups_of_four():
    b = W.make_batch([300, 1500], q_len=4, Hq=16, Hkv=4, seed=3)   # 4 heads x 4 tokens = 16 rows
    check(b, num_ctas=5)


def test_map_reused_across_layers():
    b = W.make_batch([3000, 40, 12000], seed=4)
    db = DeviceBatch(b)
    C = 7
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=C)
    ws.plan(db.lens)
    outs = []
    for layer in range(3):
        out = torch.empty((b.B, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
        hpa.decode_step(ws, db.q, db.k, db.v, db.lens, db.indptr, db.indices, out, plan=False)
        outs.append(out.float().cpu().numpy())
    ref, _ = oracle.attention(b)
    for o in outs:
        assert_close(o, ref, "bf16")


def test_bad_page_id_is_flagged():
    b = W.make_batch([200, 300], seed=6)
    b.page_indices = b.page_indices.copy()
    b.page_indices[2] = b.num_pages + 5
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=4)
    out = torch.empty((2, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    hpa.decode_step(ws, db.q, db.k, db.v, db.lens, db.indptr, db.indices, out)
    torch.cuda.synchronize()
    assert ws.status() & 4
    assert torch.isnan(out.float()).all()


def test_mismatched_partition_count_is_flagged():
    b = W.make_batch([200, 3000], seed=7)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=4)
    ws.plan(db.lens)
    big = hpa.Workspace(b.B, 1, 64, 128, num_ctas=9)
    out = torch.empty((2, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, 9, big.partial_o,
                        big.partial_lse)
    hpa.hpa_combine(big.partial_o, big.partial_lse, ws.taskmap, 9, out)
    torch.cuda.synchronize()
    assert ws.status() & 2
    assert torch.isnan(out.float()).all()


def test_sm_scale_argument():
    b = W.make_batch([900], seed=8)
    db = DeviceBatch(b)
    ws = hpa.Workspace(1, 1, 64, 128, num_ctas=3)
    ws.plan(db.lens)
    out = torch.empty((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 1, 64), dtype=torch.float32, device="cuda")
    hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, 3, ws.partial_o,
                        ws.partial_lse, sm_scale=0.05)
    hpa.hpa_combine(ws.partial_o, ws.partial_lse, ws.taskmap, 3, out, lse)
    ref, ref_lse = oracle.attention(b, sm_scale=0.05)
    assert_close(out.float().cpu().numpy(), ref, "bf16")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("case", ["large", "tiny", "mixed_rows", "mixed"])
@pytest.mark.parametrize("q_len", [1, 2])
@pytest.mark.parametrize("kv", ["e4m3", "bf16"])
def test_query_magnitudes(kv, q_len, case):
    """bf16 query rows far outside N(0,1): elements near 1e5 (beyond f16's range, which
    the E4M3 path's f16 MMAs use) and near 1e-6 (f16 subnormals), against the oracle."""
    b, sm = scaled_query_batch([2, 65, 513, 1000, 3333], q_len, kv, 120 + q_len, case)
    check(b, num_ctas=5, sm_scale=sm)
    if kv == "e4m3" and case == "mixed":
        check(b, num_ctas=5, sm_scale=sm, fused=True)


def test_traced_call_matches_and_records_every_cta():
    b = W.make_batch([3000, 40, 12000, 700], seed=9)
    db = DeviceBatch(b)
    C = 6
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=C)
    ws.plan(db.lens)
    hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C, ws.partial_o,
                        ws.partial_lse)
    torch.cuda.synchronize()
    S = int(ws.taskmap[5].item())
    ref_o = ws.partial_o[:S * 64 * 128].clone()
    trace = torch.zeros(4 * C * b.Hkv, dtype=torch.int64, device="cuda")
    hpa.hpa_decode_attn_traced(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C,
                               ws.partial_o, ws.partial_lse, trace)
    torch.cuda.synchronize()
    got = ws.partial_o[:S * 64 * 128]
    assert torch.allclose(got, ref_o, rtol=1e-5, atol=1e-6)
    t = trace.view(-1, 4).cpu().numpy()
    assert (t[:, 0] > 0).all() and (t[:, 0] <= t[:, 1]).all() and (t[:, 1] <= t[:, 2]).all()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ((t[:, 3] & 0xffffffff) < sms).all()
    assert int((t[:, 3] >> 32).sum()) == S * b.Hkv      # every segment, once per KV head
    summ = hpa.trace_summary(trace, C, b.Hkv)
    assert summ["span_us"] > 0 and 0 < summ["sm_busy_frac"] <= 1.0


# ----------------------------------------------------------------------------- fused combine
FUSED_CASES = [
    dict(lens=[2, 63, 64, 65, 511, 512, 513, 1000, 3333, 4113], q_len=1, kv="bf16", C=5),
    dict(lens=[2, 63, 64, 65, 511, 512, 513, 1000, 3333, 4113], q_len=2, kv="e4m3", C=23),
    dict(lens=[100, 700, 30], q_len=1, kv="bf16", C=40),          # surplus partitions
    dict(lens=[196608 // 8], q_len=1, kv="bf16", C=38),           # one request over 38 CTAs
    dict(lens=[3000, 9000, 64 * 7, 2], q_len=2, kv="bf16", C=9),
]


@pytest.mark.parametrize("case", range(len(FUSED_CASES)))
def test_fused_combine(case):
    c = FUSED_CASES[case]
    b = W.make_batch(c["lens"], q_len=c["q_len"], kv_dtype=c["kv"], seed=60 + case)
    check(b, num_ctas=c["C"], fused=True)


@pytest.mark.parametrize("splits", [1, 3])
def test_fused_combine_static_plan(splits):
    b = W.make_batch([100, 2000, 9000, 1], seed=70 + splits)
    check(b, splits=splits, fused=True)


def test_fused_combine_reused_map_and_bad_map():
    b = W.make_batch([3000, 40, 12000], seed=80)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=7)
    ws.plan(db.lens)
    ref, _ = oracle.attention(b)
    for layer in range(3):
        out = torch.empty((b.B, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
        hpa.decode_step(ws, db.q, db.k, db.v, db.lens, db.indptr, db.indices, out, plan=False,
                        fused=True)
        assert_close(out.float().cpu().numpy(), ref, "bf16")
    assert int(ws.arrivals.abs().sum().item()) == 0
    bad = db.lens.clone()
    bad[1] = 0
    ws.plan(bad)
    out = torch.zeros((b.B, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    hpa.decode_step(ws, db.q, db.k, db.v, bad, db.indptr, db.indices, out, plan=False,
                    fused=True)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()


def test_three_calls_capture_in_a_cuda_graph():
    """plan -> attention -> combine recorded once in a CUDA graph and replayed on new lengths."""
    b = W.make_batch([3000, 40, 12000, 700], seed=90)
    db = DeviceBatch(b)
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=11)
    out = torch.empty((b.B, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((b.B, 1, 64), dtype=torch.float32, device="cuda")
    lens = db.lens.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):                       # warm up (resolves TMA descriptors etc.)
        hpa.decode_step(ws, db.q, db.k, db.v, lens, db.indptr, db.indices, out, lse, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hpa.decode_step(ws, db.q, db.k, db.v, lens, db.indptr, db.indices, out, lse, stream=s)
    for shorten in (0, 17):                          # replay; the second time with new lengths
        b2 = W.make_batch([3000, 40, 12000, 700], seed=90)
        b2.seq_lens = b.seq_lens - shorten
        lens.copy_(torch.from_numpy(b2.seq_lens))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        ref, ref_lse = oracle.attention(b2)
        assert_close(out.float().cpu().numpy(), ref, "bf16")
        assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("q_len", [1, 2])
def test_weighted_plan_same_kernels(kv, q_len):
    b = W.make_batch([2, 63, 513, 1000, 3333, 4113, 600], q_len=q_len, kv_dtype=kv, seed=95)
    check(b, num_ctas=7, weighted=True)


@pytest.mark.parametrize("q_len,kv", [(3, "bf16"), (4, "bf16"), (4, "e4m3"), (8, "bf16")])
def test_mtp_more_draft_tokens(q_len, kv):
    """G * q_len up to 64 query rows per KV head, in groups of 16 (grid z)."""
    lens = [q_len, 70, 513, 1000, 3333, 9000]
    b = W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=100 + q_len)
    check(b, num_ctas=6)
    check(b, num_ctas=6, fused=True)


def test_mtp_rows_not_a_multiple_of_16():
    b = W.make_batch([100, 2000], q_len=3, Hq=24, Hkv=4, seed=7)    # 6 heads x 3 tokens = 18 rows
    check(b, num_ctas=4)


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


# ----------------------------------------------------------------------------- all heads in a CTA
ALLHEADS_CASES = [
    dict(lens=[2, 63, 64, 65, 511, 512, 513, 1000, 3333, 4113], q_len=1, kv="bf16", C=23),
    dict(lens=[2, 63, 64, 65, 511, 512, 513, 1000, 3333, 4113], q_len=2, kv="e4m3", C=7),
    dict(lens=[100, 700, 30], q_len=1, kv="e4m3", C=40),              # surplus partitions
    dict(lens=[70, 1000, 9000], q_len=4, kv="bf16", C=5),              # two row groups
]


@pytest.mark.parametrize("case", range(len(ALLHEADS_CASES)))
def test_allheads_variant(case):
    """hpa_decode_attn_allheads: every KV head walked inside the CTA of a partition."""
    c = ALLHEADS_CASES[case]
    b = W.make_batch(c["lens"], q_len=c["q_len"], kv_dtype=c["kv"], seed=170 + case)
    check(b, num_ctas=c["C"], allheads=True)


def test_allheads_variant_static_plan_and_default_count():
    b = W.make_batch([100, 2000, 9000, 2], kv_dtype="e4m3", q_len=2, seed=175)
    check(b, splits=3, allheads=True)
    check(b, allheads=True)            # hpa_default_num_ctas_allheads partitions


def test_allheads_traced():
    b = W.make_batch([3000, 40, 12000, 700], seed=176)
    db = DeviceBatch(b)
    C = 20
    ws = hpa.Workspace(b.B, 1, 64, 128, num_ctas=C)
    ws.plan(db.lens)
    trace = torch.zeros(4 * C, dtype=torch.int64, device="cuda")
    hpa.hpa_decode_attn_allheads(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C,
                                 ws.partial_o, ws.partial_lse, trace=trace)
    torch.cuda.synchronize()
    t = trace.view(-1, 4).cpu().numpy()
    S = int(ws.taskmap[5].item())
    assert int((t[:, 3] >> 32).sum()) == S          # every segment once (all heads inside)
    assert (t[:, 0] <= t[:, 2]).all()
    out = torch.empty((b.B, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    hpa.hpa_combine(ws.partial_o, ws.partial_lse, ws.taskmap, C, out)
    ref, _ = oracle.attention(b)
    assert_close(out.float().cpu().numpy(), ref, "bf16")


@pytest.mark.parametrize("q_len,kv", [(1, "bf16"), (2, "e4m3"), (3, "e4m3"), (8, "bf16")])
def test_hpa_decode_attn_picks_the_kernel_by_row_count(q_len, kv):
    """hpa_decode_attn runs the mma.sync kernel up to 16 query rows per KV head and the
    tcgen05 kernel above: its partials equal those of the forced kernel bit for bit,
    and hpa_default_num_ctas follows the same choice."""
    b = W.make_batch([q_len, 700, 5000], q_len=q_len, kv_dtype=kv, seed=180 + q_len)
    db = DeviceBatch(b)
    kvc = hpa.KV_BF16 if kv == "bf16" else hpa.KV_E4M3
    rows = b.Hq // b.Hkv * q_len
    forced = hpa.hpa_default_num_ctas_tc if rows > 16 else hpa.hpa_default_num_ctas_mma
    C = hpa.hpa_default_num_ctas(b.Hkv, q_len, kvc, b.Hq)
    assert C == forced(b.Hkv, q_len, kvc, b.Hq)
    ws = hpa.Workspace(b.B, q_len, b.Hq, b.d, num_ctas=C)
    ws.plan(db.lens)
    hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C, ws.partial_o,
                        ws.partial_lse, db.ks, db.vs)
    torch.cuda.synchronize()
    S = int(ws.taskmap[5].item())
    auto_o = ws.partial_o[:S * q_len * b.Hq * b.d].clone()
    auto_l = ws.partial_lse[:S * q_len * b.Hq].clone()
    hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, ws.taskmap, C, ws.partial_o,
                        ws.partial_lse, db.ks, db.vs, tc=rows > 16, mma=rows <= 16)
    torch.cuda.synchronize()
    assert torch.equal(auto_o, ws.partial_o[:S * q_len * b.Hq * b.d])
    assert torch.equal(auto_l, ws.partial_lse[:S * q_len * b.Hq])
