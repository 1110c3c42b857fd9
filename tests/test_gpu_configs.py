"""The five decode workloads at full size, in the launch configuration the
benchmark times (device-default partition count), against the fp64 oracle:
task map bit-exact, every split partial, and the combined output and lse.
The static split-KV comparator is checked at its heuristic split count, and
the tcgen05 kernel on the mixed and MTP workloads (the MTP one also at four
query tokens, 32 rows per KV head, where that kernel is the faster one)."""
import math

import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import (DeviceBatch, assert_close, assert_lse_close, expect_taskmap_equal,
                         num_ctas_for, run_gpu)

pytestmark = pytest.mark.gpu


def static_splits_heuristic(b, num_ctas):
    """ceil(partitions that fill the GPU / B), clamped to [1, max tiles of a request]."""
    max_tiles = int((b.seq_lens.max() + b.tile - 1) // b.tile)
    return max(1, min(max_tiles, math.ceil(num_ctas / b.B)))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_config_full_size(cfg):
    b = W.make_config(cfg)
    db = DeviceBatch(b)
    g = run_gpu(b, db=db)
    ref_plan = oracle.plan(b.seq_lens, b.tile, g["num_ctas"])
    expect_taskmap_equal(g["tm"], ref_plan, g["capacity"])
    out, lse = oracle.attention(b)
    e_abs, e_rel = assert_close(g["out"], out, b.kv_dtype, "out")
    assert_lse_close(g["lse"], lse, "out_lse")
    # every segment's partial, against the oracle over the same keys
    po, pl = oracle.split_attention(b, ref_plan)
    assert_close(g["po"], po, b.kv_dtype, "partial_o")
    assert_lse_close(g["pl"], pl, "partial_lse")
    # the static comparator through the same kernels
    splits = static_splits_heuristic(b, g["num_ctas"])
    gs = run_gpu(b, splits=splits, db=db)
    expect_taskmap_equal(gs["tm"], oracle.plan_static(b.seq_lens, b.tile, splits),
                         gs["capacity"])
    assert_close(gs["out"], out, b.kv_dtype, "static out")
    assert_lse_close(gs["lse"], lse, "static out_lse")
    # the fused combine through one attention launch
    gf = run_gpu(b, db=db, fused=True)
    assert_close(gf["out"], out, b.kv_dtype, "fused out")
    assert_lse_close(gf["lse"], lse, "fused out_lse")
    print("cfg%d %s: max|d| %.3g, max rel %.3g" % (cfg, b.name, e_abs, e_rel))


def _check_full(b, tc):
    g = run_gpu(b, tc=tc, mma=not tc)
    ref_plan = oracle.plan(b.seq_lens, b.tile, g["num_ctas"])
    expect_taskmap_equal(g["tm"], ref_plan, g["capacity"])
    out, lse = oracle.attention(b)
    e_abs, e_rel = assert_close(g["out"], out, b.kv_dtype, "out")
    assert_lse_close(g["lse"], lse, "out_lse")
    po, pl = oracle.split_attention(b, ref_plan)
    assert_close(g["po"], po, b.kv_dtype, "partial_o")
    assert_lse_close(g["pl"], pl, "partial_lse")
    return e_abs, e_rel


@pytest.mark.parametrize("cfg,q_len", [(3, None), (5, None), (5, 4)])
def test_config_full_size_tcgen05(cfg, q_len):
    """hpa_decode_attn_tc at full size with its own default partition count."""
    b = W.make_config(cfg, q_len=q_len)
    e_abs, e_rel = _check_full(b, tc=True)
    print("tc cfg%d q_len %d: max|d| %.3g, max rel %.3g" % (cfg, b.q_len, e_abs, e_rel))


def test_config5_four_query_tokens_mma():
    """The MTP workload at q_len 4 (two 16-row groups per KV head) on hpa_decode_attn."""
    b = W.make_config(5, q_len=4)
    e_abs, e_rel = _check_full(b, tc=False)
    print("mma cfg5 q_len 4: max|d| %.3g, max rel %.3g" % (e_abs, e_rel))
