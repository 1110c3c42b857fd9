"""Pins of the oracle's KV-cache writer (RoPE, RMSNorm, Hadamard, E4M3 encoding,
placement) against library routines, closed forms and invariants."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from oracle import feeder


def test_e4m3_encoder_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10, rng.standard_normal(5000) * 1e-3,
                        np.array([0.0, 448.0, 464.0, 600.0, -1000.0, 2.0 ** -10])])
    grid = feeder.e4m3_grid()
    mids = (grid[1:] + grid[:-1]) / 2                 # exact ties
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).to(torch.float64)
    np.testing.assert_array_equal(feeder.encode_e4m3_value(x), ref.numpy())


def test_rope_is_a_rotation_per_pair():
    cs = W.rope_cos_sin_table(70000)
    x = np.random.default_rng(1).standard_normal(128)
    np.testing.assert_allclose(feeder.rope_rotate_half(x, cs[0].astype(np.float64)), x)
    for pos in (1, 17, 65535):
        y = feeder.rope_rotate_half(x, cs[pos].astype(np.float64))
        # as complex numbers: (x_i + i x_{i+64}) * exp(i theta)
        z = (x[:64] + 1j * x[64:]) * (cs[pos, :64] + 1j * cs[pos, 64:])
        np.testing.assert_allclose(y[:64], z.real, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(y[64:], z.imag, rtol=1e-12, atol=1e-12)


def test_rope_table_angles():
    cs = W.rope_cos_sin_table(5)
    i = np.arange(64)
    ang = 3 * 10000.0 ** (-2 * i / 128)
    np.testing.assert_allclose(cs[3, :64], np.cos(ang), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(cs[3, 64:], np.sin(ang), rtol=1e-6, atol=1e-7)


def test_rms_norm_closed_forms():
    w = np.linspace(0.5, 1.5, 128)
    y = feeder.rms_norm(np.full(128, -2.0), w, 1e-6)
    np.testing.assert_allclose(y, -w * 2.0 / math.sqrt(4.0 + 1e-6), rtol=1e-14)
    x = np.random.default_rng(2).standard_normal(128)
    np.testing.assert_allclose(feeder.rms_norm(7.5 * x, w, 0.0), feeder.rms_norm(x, w, 0.0),
                               rtol=1e-12)


def test_hadamard_is_orthonormal_sylvester():
    H = feeder.hadamard(128)
    np.testing.assert_allclose(H @ H.T, np.eye(128), atol=1e-12)
    np.testing.assert_allclose(H[:, 0], np.full(128, 1 / math.sqrt(128)))
    # Sylvester recursion H_2n = [[H, H], [H, -H]] / sqrt(2)
    h64 = feeder.hadamard(64)
    np.testing.assert_allclose(H, np.block([[h64, h64], [h64, -h64]]) / math.sqrt(2), atol=1e-12)


def test_placement_and_order():
    fi = W.make_feeder_inputs(3, B=2, q_len=2, max_pos=200, Hkv=2, d=128)
    lens = np.array([65, 130])
    indptr = np.array([0, 2, 5])
    indices = np.array([7, 3, 9, 1, 4])
    kn = fi.k_new.to(torch.float64).numpy()
    out = feeder.store_kv(kn, fi.v_new.to(torch.float64).numpy(), lens, indptr, indices,
                          fi.cos_sin, fi.norm_w, fi.eps, True, "bf16")
    # request 0: positions 63 (page 7, slot 63) and 64 (page 3, slot 0)
    # request 1 (pages 9, 1, 4): positions 128 and 129 -> page 4, slots 0 and 1
    assert set(out) == {(7, h, 63) for h in range(2)} | {(3, h, 0) for h in range(2)} | \
        {(4, h, 0) for h in range(2)} | {(4, h, 1) for h in range(2)}
    k, v = out[(3, 1, 0)]
    x = feeder.rope_rotate_half(kn[0, 1, 1], fi.cos_sin[64].astype(np.float64))
    x = feeder.rms_norm(x, fi.norm_w.astype(np.float64), fi.eps)
    np.testing.assert_allclose(k, feeder.hadamard(128) @ x)
    np.testing.assert_array_equal(v, fi.v_new[0, 1, 1].to(torch.float64).numpy())
