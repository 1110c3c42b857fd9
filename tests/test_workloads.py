"""The seeded input generators: deterministic, shaped as the five workloads state."""
import numpy as np
import torch

import workloads as W


def test_lengths_of_the_five_workloads():
    assert W.config_lens(1).tolist() == [1024, 5120, 2048]
    L2 = W.config_lens(2)
    assert L2.shape == (32,) and (L2 == 8192).all()
    L3 = W.config_lens(3)
    assert L3.shape == (45,) and L3.min() >= 1024 and L3.max() <= 131072
    for x in (1024, 4096, 16384, 65536, 131072):
        assert (L3 == x).sum() >= 1
    assert W.config_lens(4).tolist() == [196608]
    L5 = W.config_lens(5)
    assert L5.shape == (64,) and L5.min() >= 512 and L5.max() <= 196608
    assert abs(L5.mean() - 68000) < 50


def test_lengths_are_seeded():
    assert (W.lens_mixed(0) == W.lens_mixed(0)).all()
    assert not (W.lens_mixed(0) == W.lens_mixed(1)).all()


def test_batch_is_deterministic_and_shaped():
    a = W.make_batch([70, 130], q_len=2, seed=3)
    b = W.make_batch([70, 130], q_len=2, seed=3)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.k_pool.view(torch.int16), b.k_pool.view(torch.int16))
    assert a.q.shape == (2, 2, 64, 128) and a.k_pool.shape == (2 + 3, 8, 64, 128)
    assert a.page_indptr.tolist() == [0, 2, 5]
    assert sorted(a.page_indices.tolist()) == list(range(5))
    assert a.kv_bytes == 200 * 8 * 128 * 2 * 2


def test_e4m3_pool_scale_and_codes():
    b = W.make_batch([300], kv_dtype="e4m3", seed=1)
    assert b.k_pool.dtype == torch.uint8 and b.k_scale.shape == (8,)
    vals = b.k_pool.view(torch.float8_e4m3fn).float()
    assert torch.isfinite(vals).all()
    assert vals.abs().amax().item() == 448.0            # amax maps to the largest code
    assert np.all(b.k_scale > 0)


def test_contiguous_pages_for_the_worked_example():
    b = W.make_config(1)
    assert b.page_indices.tolist() == list(range(b.num_pages))
    assert b.num_ctas == 4
