"""GPU task maps (hpa_plan / hpa_plan_static) against the oracle scheduler, bit-exact."""
import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
from gpu_helpers import decode_taskmap, expect_taskmap_equal

pytestmark = pytest.mark.gpu


def gpu_plan(lens, tile, C=None, splits=None, weighted=False):
    lens_d = torch.tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    B = len(lens)
    if splits is None:
        nbytes, cap, CC = hpa.hpa_taskmap_bytes(B, C), hpa.hpa_max_segments(B, C), C
    else:
        nbytes, CC = hpa.hpa_static_taskmap_bytes(B, splits), hpa.hpa_static_num_ctas(B, splits)
        cap = CC
    tm = torch.full(((nbytes + 3) // 4,), 12345, dtype=torch.int32, device="cuda")
    if splits is None and weighted:
        hpa.hpa_plan_weighted(lens_d, tile, C, tm)
    elif splits is None:
        hpa.hpa_plan(lens_d, tile, C, tm)
    else:
        hpa.hpa_plan_static(lens_d, tile, splits, tm)
    torch.cuda.synchronize()
    g = decode_taskmap(tm.cpu().numpy(), B, CC)
    assert g["words"] == tm.numel()
    return g, cap


def test_worked_example():
    g, cap = gpu_plan([1024, 5120, 2048], 512, 4)
    ref = oracle.plan([1024, 5120, 2048], 512, 4)
    expect_taskmap_equal(g, ref, cap)
    assert list(np.diff(g["cta_begin"])) == [4, 4, 4, 4]


CASES = [
    ([1], 512, 1), ([1], 512, 7), ([100, 600], 512, 7), ([512] * 12, 512, 5),
    ([196608], 512, 37), ([8192] * 32, 512, 38), ([1000, 1, 70000, 513, 512, 64], 64, 9),
]


@pytest.mark.parametrize("lens,tile,C", CASES)
def test_fixed_cases(lens, tile, C):
    g, cap = gpu_plan(lens, tile, C)
    expect_taskmap_equal(g, oracle.plan(lens, tile, C), cap)


@pytest.mark.parametrize("seed", range(12))
def test_random(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 3000))          # spans several 1024-thread scan chunks
    tile = int(rng.choice([64, 128, 512, 1024]))
    lens = rng.integers(1, 200000 if tile >= 512 else 20000, size=B)
    C = int(rng.integers(1, 2500))
    g, cap = gpu_plan(lens, tile, C)
    expect_taskmap_equal(g, oracle.plan(lens, tile, C), cap)


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 64])
def test_static(splits):
    rng = np.random.default_rng(splits)
    lens = rng.integers(1, 140000, size=45)
    g, cap = gpu_plan(lens, 512, splits=splits)
    expect_taskmap_equal(g, oracle.plan_static(lens, 512, splits), cap)


def test_bad_length_sets_status():
    g, _ = gpu_plan([100, 0, 5], 512, 4)
    assert g["status"] & 1
    g, _ = gpu_plan([100, -3], 512, 2)
    assert g["status"] & 1


def test_replan_clears_status():
    lens_d = torch.tensor([100, 0], dtype=torch.int32, device="cuda")
    ws = hpa.Workspace(2, 1, 64, 128, num_ctas=3)
    ws.plan(lens_d)
    assert ws.status() & 1
    lens_d[1] = 7
    ws.plan(lens_d)
    assert ws.status() == 0


@pytest.mark.parametrize("seed", range(12))
def test_weighted(seed):
    rng = np.random.default_rng(900 + seed)
    B = int(rng.integers(1, 1500))
    tile = int(rng.choice([64, 256, 512]))
    lens = rng.integers(1, 100000 if tile >= 256 else 20000, size=B)
    C = int(rng.integers(1, 1200))
    g, cap = gpu_plan(lens, tile, C, weighted=True)
    expect_taskmap_equal(g, oracle.plan_weighted(lens, tile, C), cap)


def test_weighted_worked_example_and_partial_tiles():
    for lens, C in (([1024, 5120, 2048], 4), ([513] * 4, 2), ([1025, 1], 2), ([1], 5)):
        g, cap = gpu_plan(lens, 512, C, weighted=True)
        expect_taskmap_equal(g, oracle.plan_weighted(lens, 512, C), cap)


@pytest.mark.parametrize("bmax,cmax", [(32, 32), (128, 128), (256, 256), (32, 300), (300, 32),
                                       (129, 1100), (1100, 100)])
@pytest.mark.parametrize("seed", range(3))
def test_block_sizes(bmax, cmax, seed):
    """Batches and partition counts around each plan block size (32, 128, 256, 1024
    threads: the smallest that covers max(B, C)), for all three planners."""
    rng = np.random.default_rng([bmax, cmax, seed])
    B = int(rng.integers(max(1, bmax // 4), bmax + 1))
    C = int(rng.integers(max(1, cmax // 4), cmax + 1))
    lens = rng.integers(1, 90000, size=B)
    g, cap = gpu_plan(lens, 512, C)
    expect_taskmap_equal(g, oracle.plan(lens, 512, C), cap)
    g, cap = gpu_plan(lens, 256, C, weighted=True)
    expect_taskmap_equal(g, oracle.plan_weighted(lens, 256, C), cap)
    splits = max(1, C // B)
    g, cap = gpu_plan(lens, 512, splits=splits)
    expect_taskmap_equal(g, oracle.plan_static(lens, 512, splits), cap)
