"""Pins of the oracle's fp64 attention and merge against independent facts.

- bit decoders: every bf16 / E4M3 code against torch's own conversions;
- closed forms: one key, identical keys, zero query, a dominant key, two keys
  worked by hand (with the first MTP token's causal row);
- brute force: pure-Python scalar loops on tiny inputs (d <= 4, L <= 8);
- library routines: torch scaled_dot_product_attention and torch.logsumexp in
  float64 on the explicitly expanded (GQA-repeated, page-gathered) tensors;
- invariants: causal MTP rows, page-table permutation, GQA grouping;
- the merge identity: any split then log-sum-exp merge equals unsplit.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

F64 = torch.float64


def small_batch(lens, q_len=1, kv="bf16", seed=0, Hq=16, Hkv=2, d=32, page=16, shuffle=True):
    return W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=seed, shuffle_pages=shuffle,
                        Hq=Hq, Hkv=Hkv, d=d, page_size=page)


def dense_kv(b, which):
    """[B] list of float64 [L][Hkv][d] key or value tensors gathered through the page table."""
    pool = b.k_pool if which == "k" else b.v_pool
    scale = b.k_scale if which == "k" else b.v_scale
    if b.kv_dtype == "bf16":
        pool = pool.to(F64)
    else:
        pool = pool.view(torch.float8_e4m3fn).to(F64) * torch.from_numpy(scale).to(F64).view(
            1, -1, 1, 1)
    out = []
    for r, L in enumerate(b.seq_lens):
        pages = b.page_indices[b.page_indptr[r]:b.page_indptr[r + 1]]
        x = pool[torch.from_numpy(pages.astype(np.int64))]        # [np][Hkv][page][d]
        x = x.permute(0, 2, 1, 3).reshape(-1, b.Hkv, b.d)[:L]
        out.append(x)
    return out


def torch_reference(b):
    """sdpa in float64 with an explicit causal (bottom-right) mask and repeated KV heads."""
    G = b.Hq // b.Hkv
    K, V = dense_kv(b, "k"), dense_kv(b, "v")
    outs, lses = [], []
    for r, L in enumerate(b.seq_lens):
        q = b.q[r].to(F64).permute(1, 0, 2)                       # [Hq][q_len][d]
        k = K[r].permute(1, 0, 2).repeat_interleave(G, dim=0)      # [Hq][L][d]
        v = V[r].permute(1, 0, 2).repeat_interleave(G, dim=0)
        pos = torch.arange(L)
        qpos = L - b.q_len + torch.arange(b.q_len)
        mask = pos[None, :] <= qpos[:, None]                       # [q_len][L]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask)
        s = (q @ k.transpose(-1, -2)) / math.sqrt(b.d)
        s = s.masked_fill(~mask, float("-inf"))
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(torch.logsumexp(s, dim=-1).permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


# ----------------------------------------------------------------------------- decoders
def test_bf16_decoder_exhaustive():
    L = oracle.lib()
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    ref = codes.to(F64).numpy()
    got = np.array([L.oracle_bf16_to_double(c) for c in range(65536)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_e4m3_decoder_exhaustive():
    L = oracle.lib()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(F64).numpy()
    got = np.array([L.oracle_e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# ----------------------------------------------------------------------------- closed forms
def test_single_key():
    b = small_batch([1, 1], Hq=8, Hkv=1, d=8, page=4)
    out, lse = oracle.attention(b)
    K, V = dense_kv(b, "k"), dense_kv(b, "v")
    for r in range(2):
        q = b.q[r, 0].to(F64).numpy()                             # [Hq][d]
        np.testing.assert_array_equal(out[r, 0], np.broadcast_to(V[r][0, 0].numpy(), (8, 8)))
        np.testing.assert_allclose(lse[r, 0], q @ K[r][0, 0].numpy() / math.sqrt(8), rtol=1e-14)


def test_identical_keys_give_mean_of_values():
    b = small_batch([37], Hq=4, Hkv=1, d=16, page=8, shuffle=False)
    b.k_pool[:] = b.k_pool[0, 0, 0]                               # every key equal
    out, lse = oracle.attention(b)
    V = dense_kv(b, "v")[0][:, 0].numpy()                         # [L][d]
    k = dense_kv(b, "k")[0][0, 0].numpy()
    q = b.q[0, 0].to(F64).numpy()
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(V.mean(axis=0), (4, 16)), rtol=1e-12,
                               atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(37) + q @ k / 4.0, rtol=1e-13)


def test_zero_query_gives_uniform_weights():
    b = small_batch([50, 3], Hq=8, Hkv=2, d=16, page=8)
    b.q.zero_()
    out, lse = oracle.attention(b)
    for r, L in enumerate(b.seq_lens):
        V = dense_kv(b, "v")[r].numpy()                           # [L][Hkv][d]
        for g in range(8):
            np.testing.assert_allclose(out[r, 0, g], V[:, g // 4].mean(axis=0), rtol=1e-12,
                                       atol=1e-14)
        np.testing.assert_allclose(lse[r, 0], math.log(L), rtol=1e-14)


def test_dominant_key():
    b = small_batch([40], Hq=8, Hkv=1, d=16, page=8, shuffle=False)
    b.q[:] = 1.0
    b.k_pool.zero_()
    b.k_pool[2, 0, 5] = 8.0                                       # key 21 (page 2, slot 5)
    out, _ = oracle.attention(b)
    v21 = dense_kv(b, "v")[0][21, 0].numpy()
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(v21, (8, 16)), atol=1e-10)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_two_keys_by_hand(kv):
    """d = 4 (scale 1/2), q = (1,1,1,1), k0 = 0, k1 = (1,1,0,0): the scores are 0 and 1,
    so the weights are 1/(1+e) and e/(1+e). With v0 = (1,0,0,0) and v1 = (0,2,0,0)
    the output is (1/(1+e), 2e/(1+e), 0, 0) and lse = ln(1+e). With two new tokens,
    the first sits at position 0 and sees only key 0: out = v0, lse = 0."""
    for q_len in (1, 2):
        b = small_batch([2], q_len=q_len, kv=kv, Hq=1, Hkv=1, d=4, page=4, shuffle=False)
        b.q[:] = 1.0
        if kv == "bf16":
            b.k_pool.zero_()
            b.v_pool.zero_()
            b.k_pool[0, 0, 1, :2] = 1.0
            b.v_pool[0, 0, 0, 0] = 1.0
            b.v_pool[0, 0, 1, 1] = 2.0
        else:
            # E4M3 codes (bias 7): 0x30 = 0.5, 0x38 = 1.0, 0x40 = 2.0; the per-head
            # scales bring k1 to (1,1,0,0), v0 to (1,0,0,0) and v1 to (0,2,0,0)
            b.k_scale[:] = 0.5
            b.v_scale[:] = 2.0
            b.k_pool.zero_()
            b.v_pool.zero_()
            b.k_pool[0, 0, 1, :2] = 0x40
            b.v_pool[0, 0, 0, 0] = 0x30
            b.v_pool[0, 0, 1, 1] = 0x38
        out, lse = oracle.attention(b)
        e = math.e
        last = q_len - 1
        np.testing.assert_allclose(out[0, last, 0], [1 / (1 + e), 2 * e / (1 + e), 0, 0],
                                   rtol=1e-14, atol=1e-16)
        np.testing.assert_allclose(lse[0, last, 0], math.log(1 + e), rtol=1e-14)
        if q_len == 2:
            np.testing.assert_array_equal(out[0, 0, 0], [1.0, 0, 0, 0])
            assert lse[0, 0, 0] == 0.0


def scalar_attention(b):
    """Pure-Python scalar loops over the definition: exp without max-subtraction,
    sums in visiting order, keys decoded by torch (tiny inputs only)."""
    G = b.Hq // b.Hkv
    K, V = dense_kv(b, "k"), dense_kv(b, "v")
    out = np.zeros((b.B, b.q_len, b.Hq, b.d))
    lse = np.zeros((b.B, b.q_len, b.Hq))
    for r, L in enumerate(b.seq_lens):
        Kr, Vr = K[r].tolist(), V[r].tolist()
        for j in range(b.q_len):
            visible = L - b.q_len + 1 + j
            for g in range(b.Hq):
                h = g // G
                q = b.q[r, j, g].to(F64).tolist()
                w = []
                for k in range(visible):
                    dot = 0.0
                    for i in range(b.d):
                        dot += q[i] * Kr[k][h][i]
                    w.append(math.exp(dot / math.sqrt(b.d)))
                Z = sum(w)
                for i in range(b.d):
                    out[r, j, g, i] = sum(w[k] * Vr[k][h][i] for k in range(visible)) / Z
                lse[r, j, g] = math.log(Z)
    return out, lse


@pytest.mark.parametrize("seed", range(8))
def test_brute_force_tiny(seed):
    """d <= 4, L <= 8, one or two new tokens, up to 2 KV heads, both KV types."""
    rng = np.random.default_rng(100 + seed)
    q_len = 1 + seed % 2
    lens = rng.integers(q_len, 9, size=int(rng.integers(1, 4)))
    Hkv = 1 + (seed // 2) % 2
    b = small_batch(lens, q_len=q_len, kv="e4m3" if seed % 4 >= 2 else "bf16", seed=seed,
                    Hq=2 * Hkv, Hkv=Hkv, d=int(rng.choice([2, 4])), page=int(rng.choice([1, 2, 4])))
    out, lse = oracle.attention(b)
    ref_o, ref_l = scalar_attention(b)
    np.testing.assert_allclose(out, ref_o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------- library routine
@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("q_len", [1, 2])
def test_matches_torch_sdpa(kv, q_len):
    b = small_batch([1 + q_len, 17, 64, 100, 257], q_len=q_len, kv=kv, seed=3)
    out, lse = oracle.attention(b)
    ref_o, ref_l = torch_reference(b)
    np.testing.assert_allclose(out, ref_o, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13, atol=1e-13)


def test_model_shape_matches_torch_sdpa():
    b = W.make_batch([70, 300], q_len=2, kv_dtype="bf16", seed=5)   # 64/8 heads, d=128
    out, lse = oracle.attention(b)
    ref_o, ref_l = torch_reference(b)
    np.testing.assert_allclose(out, ref_o, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13)


# ----------------------------------------------------------------------------- invariants
def test_causal_rows_match_shorter_requests():
    """Row j of an MTP pair sees exactly the first L - 1 + j keys (q_len = 2)."""
    b2 = small_batch([30, 65], q_len=2, seed=7)
    o2, l2 = oracle.attention(b2)
    for j, cut in ((0, 1), (1, 0)):
        b1 = small_batch([30, 65], q_len=2, seed=7)
        b1.q = b2.q[:, j:j + 1].contiguous()
        b1.q_len = 1
        b1.seq_lens = b2.seq_lens - cut
        o1, l1 = oracle.attention(b1)
        np.testing.assert_array_equal(o1[:, 0], o2[:, j])
        np.testing.assert_array_equal(l1[:, 0], l2[:, j])


def test_page_permutation_invariance():
    a = small_batch([45, 130], seed=9, shuffle=False)
    b = small_batch([45, 130], seed=9, shuffle=False)
    perm = np.random.default_rng(1).permutation(a.num_pages)
    inv = np.argsort(perm)
    b.k_pool = a.k_pool[torch.from_numpy(inv)].contiguous()      # page p of a -> slot perm[p]
    b.v_pool = a.v_pool[torch.from_numpy(inv)].contiguous()
    b.page_indices = perm[a.page_indices].astype(np.int32)
    oa, la = oracle.attention(a)
    ob, lb = oracle.attention(b)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


def test_gqa_grouping():
    """Query head g reads KV head g // (Hq / Hkv)."""
    b = small_batch([20, 9], Hq=16, Hkv=4, d=8, page=4)
    for h in range(4):
        b.v_pool[:, h] = float(h + 1)
    out, _ = oracle.attention(b)
    for g in range(16):
        np.testing.assert_allclose(out[:, 0, g], g // 4 + 1, rtol=1e-14)


def test_row_without_visible_keys():
    b = small_batch([17], q_len=2, page=16)
    out, lse = oracle.attention(b, items=[(0, 16, 17)])           # only the last key
    assert np.isneginf(lse[0, 0]).all() and (out[0, 0] == 0).all()
    assert np.isfinite(lse[0, 1]).all()


def test_invalid_arguments_rejected():
    b = small_batch([10])
    with pytest.raises(ValueError):
        oracle.attention(b, items=[(0, 0, 11)])
    b.page_indices = b.page_indices + 100
    with pytest.raises(ValueError):
        oracle.attention(b)


# ----------------------------------------------------------------------------- merge identity
@pytest.mark.parametrize("seed", range(6))
def test_split_then_combine_equals_unsplit(seed):
    rng = np.random.default_rng(seed)
    q_len = int(rng.integers(1, 3))
    lens = rng.integers(q_len, 700, size=int(rng.integers(1, 6)))
    kv = "e4m3" if seed % 2 else "bf16"
    b = small_batch(lens, q_len=q_len, kv=kv, seed=seed)
    tile = int(rng.choice([16, 32, 64]))
    p = oracle.plan(lens, tile, int(rng.integers(1, 12)))
    o, l = oracle.split_combine(b, p)
    ref_o, ref_l = oracle.attention(b)
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l, ref_l, rtol=1e-13)
    ps = oracle.plan_static(lens, tile, int(rng.integers(1, 5)))
    o, l = oracle.split_combine(b, ps)
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-14)


def test_combine_closed_forms():
    o = np.array([[[[1.0, 2.0]]], [[[3.0, 6.0]]], [[[5.0, 5.0]]]])      # [S=3][1][1][2]
    l = np.array([[[0.5]], [[0.5]], [[-np.inf]]])
    out, lse = oracle.combine(o, l, [0, 2, 3])
    np.testing.assert_allclose(out[0, 0, 0], [2.0, 4.0])              # equal weights
    np.testing.assert_allclose(lse[0, 0, 0], 0.5 + math.log(2.0))
    assert np.isneginf(lse[1, 0, 0])                                   # lone empty partial
    out, lse = oracle.combine(o[:2], np.array([[[0.0]], [[math.log(3.0)]]]), [0, 2])
    np.testing.assert_allclose(out[0, 0, 0], [(1 + 3 * 3) / 4, (2 + 6 * 3) / 4])
    np.testing.assert_allclose(lse[0, 0, 0], math.log(4.0))
