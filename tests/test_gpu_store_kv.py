"""The fused KV-cache writer (hpa_store_kv) against the oracle's RoPE + RMSNorm +
Hadamard + quantise + placement, slot by slot.

The kernel works in fp32 and the oracle in fp64, so a value that lies on a
rounding boundary of the output format may round either way: every written
element must be a correctly rounded result of the oracle's value, within half
a step of the output grid plus the fp32 evaluation error (1e-5 of the row's
rms: RoPE differences of O(1) terms can leave a small element with a large
relative error), and everything outside the new tokens' slots must be
untouched."""
import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import DeviceBatch, assert_close, assert_lse_close
from oracle import feeder

pytestmark = pytest.mark.gpu

SLACK = 1e-5


def _slack(x):
    return SLACK * (np.abs(x) + np.sqrt(np.mean(x * x)))


def _bf16_ok(got, x):
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    ulp = 2.0 ** (np.floor(np.log2(ax)) - 7)
    return np.abs(got - x) <= 0.5 * ulp + _slack(x)


def _e4m3_ok(got, x):
    grid = feeder.e4m3_grid()
    a = np.minimum(np.abs(x), 448.0)
    idx = np.clip(np.searchsorted(grid, a), 1, len(grid) - 1)
    step = grid[idx] - grid[idx - 1]
    sat = np.abs(x) >= 448.0 * (1 + SLACK)
    ok = np.abs(got - np.clip(x, -448, 448)) <= 0.5 * step + _slack(x)
    return np.where(sat, got == np.sign(x) * 448.0, ok)


def _run(lens, q_len, kv, hadamard, seed, Hkv=8):
    b = W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=seed, Hq=8 * Hkv, Hkv=Hkv)
    fi = W.make_feeder_inputs(seed, b.B, q_len, max_pos=int(max(lens)) + 1, Hkv=Hkv)
    db = DeviceBatch(b)
    k0, v0 = db.k.clone(), db.v.clone()
    cs = torch.from_numpy(fi.cos_sin).cuda()
    w = torch.from_numpy(fi.norm_w).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hpa.hpa_store_kv(fi.k_new.cuda(), fi.v_new.cuda(), db.lens, db.indptr, db.indices, cs, w,
                     db.k, db.v, eps=fi.eps, use_hadamard=hadamard, k_scale=db.ks,
                     v_scale=db.vs, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = feeder.store_kv(fi.k_new.to(torch.float64).numpy(), fi.v_new.to(torch.float64).numpy(),
                          b.seq_lens, b.page_indptr, b.page_indices, fi.cos_sin, fi.norm_w,
                          fi.eps, hadamard, kv, b.k_scale, b.v_scale)
    return b, db, k0, v0, ref


def _values(pool, kv):
    if kv == "bf16":
        return pool.float().cpu().numpy().astype(np.float64)
    return pool.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def _check_written(db, k0, v0, ref, kv):
    K, V = _values(db.k, kv), _values(db.v, kv)
    ok = _bf16_ok if kv == "bf16" else _e4m3_ok
    written = np.zeros(K.shape[:3], bool)
    for (page, h, slot), (kx, vx) in ref.items():
        gk, gv = K[page, h, slot], V[page, h, slot]
        for what, g, x in (("key", gk, kx), ("value", gv, vx)):
            bad = np.nonzero(~ok(g, x))[0]
            assert len(bad) == 0, (what, page, h, slot, [(int(i), g[i], x[i]) for i in bad[:4]])
        written[page, h, slot] = True
    # every other slot is untouched
    k0v, v0v = _values(k0, kv), _values(v0, kv)
    same_k = (K == k0v) | (np.isnan(K) & np.isnan(k0v))
    same_v = (V == v0v) | (np.isnan(V) & np.isnan(v0v))
    assert same_k[~written].all() and same_v[~written].all()


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("hadamard", [True, False])
@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_store_kv_matches_oracle(kv, hadamard, q_len):
    lens = [q_len, 64, 65, 513, 3000, 131072]
    b, db, k0, v0, ref = _run(lens, q_len, kv, hadamard, seed=q_len + 10 * hadamard)
    _check_written(db, k0, v0, ref, kv)


@pytest.mark.parametrize("Hkv,q_len", [(2, 3), (12, 2), (20, 1)])
def test_store_kv_head_counts(Hkv, q_len):
    """KV head counts that are not a multiple of the kernel's chunk of 8 heads."""
    b, db, k0, v0, ref = _run([q_len, 700, 5000], q_len, "e4m3", True, seed=30 + Hkv, Hkv=Hkv)
    _check_written(db, k0, v0, ref, "e4m3")


def test_store_kv_many_tokens():
    """4096 new tokens of one request: more (token, head chunk) items than resident
    warps, so each warp walks several of them."""
    b, db, k0, v0, ref = _run([6000], 4096, "bf16", True, seed=44)
    _check_written(db, k0, v0, ref, "bf16")


def test_store_then_attend():
    """New tokens written by the feeder are read by the decode path like any others."""
    lens = [70, 3000, 9000]
    b, db, _, _, _ = _run(lens, 2, "e4m3", True, seed=5)
    b.k_pool, b.v_pool = db.k.cpu(), db.v.cpu()          # the pool as the feeder left it
    ws = hpa.Workspace(b.B, 2, 64, 128, num_ctas=7)
    out = torch.empty((b.B, 2, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((b.B, 2, 64), dtype=torch.float32, device="cuda")
    hpa.decode_step(ws, db.q, db.k, db.v, db.lens, db.indptr, db.indices, out, lse, db.ks,
                    db.vs)
    ref, ref_lse = oracle.attention(b)
    assert_close(out.float().cpu().numpy(), ref, "e4m3")
    assert_lse_close(lse.cpu().numpy(), ref_lse)


def test_store_kv_flags_bad_pages_and_positions():
    b = W.make_batch([100, 200], seed=3)
    fi = W.make_feeder_inputs(3, b.B, 1, max_pos=150)         # position 199 is past the table
    db = DeviceBatch(b)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hpa.hpa_store_kv(fi.k_new.cuda(), fi.v_new.cuda(), db.lens, db.indptr, db.indices,
                     torch.from_numpy(fi.cos_sin).cuda(), torch.from_numpy(fi.norm_w).cuda(),
                     db.k, db.v, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    bad = db.indices.clone()
    bad[1] = b.num_pages + 3                                   # request 0's page of position 99
    status.zero_()
    fi = W.make_feeder_inputs(3, b.B, 1, max_pos=300)
    hpa.hpa_store_kv(fi.k_new.cuda(), fi.v_new.cuda(), db.lens, db.indptr, bad,
                     torch.from_numpy(fi.cos_sin).cuda(), torch.from_numpy(fi.norm_w).cuda(),
                     db.k, db.v, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4


def test_store_kv_walk_carries():
    """600 requests x 3 new tokens x 2 chunks of KV heads (12 heads) = 3600 items, more
    than the resident warps: a warp's next item carries across chunks, tokens and
    requests."""
    lens = list(np.random.default_rng(45).integers(3, 900, size=600))
    b, db, k0, v0, ref = _run(lens, 3, "e4m3", True, seed=45, Hkv=12)
    _check_written(db, k0, v0, ref, "e4m3")
