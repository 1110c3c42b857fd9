"""The C-ABI library builds, loads, exports every entry point include/hpa.h
declares, and rejects bad host-visible arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import load_balanced_split_gb300 as hpa
from load_balanced_split_gb300 import build as hbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "hpa.h")


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hpa_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("hpa_plan", "hpa_decode_attn", "hpa_combine", "hpa_plan_static",
              "hpa_taskmap_bytes", "hpa_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(hbuild.build())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_names_match_c_names():
    skip = {"hpa_error_string", "hpa_last_cuda_error"}   # used inside the binding's error path
    for n in declared_functions():
        if n not in skip:
            assert callable(getattr(hpa, n)), n


def _words(B, C, cap):
    o = 16 + B + (B + 1) + 2 * (C + 1) + (B + 1)
    return ((o + 3) & ~3) + 4 * cap


@pytest.mark.parametrize("B,C", [(1, 1), (3, 4), (45, 38), (1000, 300), (5000, 2000)])
def test_size_queries(B, C):
    assert hpa.hpa_max_segments(B, C) == B + C - 1
    assert hpa.hpa_taskmap_bytes(B, C) == 4 * _words(B, C, B + C - 1)
    assert hpa.hpa_static_num_ctas(B, 3) == 3 * B
    assert hpa.hpa_static_taskmap_bytes(B, 3) == 4 * _words(B, 3 * B, 3 * B)


def test_size_queries_reject_out_of_range():
    assert hpa.hpa_taskmap_bytes(0, 4) == 0
    assert hpa.hpa_taskmap_bytes(4, 0) == 0
    assert hpa.hpa_max_segments(-1, 4) == 0
    assert hpa.hpa_static_num_ctas(4, 0) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null value; never dereferenced by these calls


def test_plan_argument_checks():
    L = hpa.lib()
    nb = hpa.hpa_taskmap_bytes(3, 4)
    assert L.hpa_plan(None, 3, 512, 4, FAKE, nb, None) == -1        # NULL lengths
    assert L.hpa_plan(FAKE, 3, 512, 4, None, nb, None) == -1        # NULL map
    assert L.hpa_plan(FAKE, 0, 512, 4, FAKE, nb, None) == -1        # B < 1
    assert L.hpa_plan(FAKE, 3, 512, 0, FAKE, nb, None) == -1        # C < 1
    assert L.hpa_plan(FAKE, 3, 500, 4, FAKE, nb, None) == -1        # tile not a page multiple
    assert L.hpa_plan(FAKE, 3, 512, 4, FAKE + 4, nb, None) == -4    # misaligned map
    assert L.hpa_plan(FAKE, 3, 512, 4, FAKE, nb - 4, None) == -3    # map too small
    assert L.hpa_plan_static(FAKE, 3, 512, 0, FAKE, nb, None) == -1


@pytest.mark.parametrize("entry", ["hpa_decode_attn", "hpa_decode_attn_tc"])
def test_attention_argument_checks(entry):
    L = hpa.lib()
    args = dict(q=FAKE, k=FAKE, v=FAKE, kv=0, ks=None, vs=None, P=100, indptr=FAKE,
                indices=FAKE, page=64, B=3, q_len=1, Hq=64, Hkv=8, d=128, scale=0.088,
                tm=FAKE, C=4, po=FAKE, pl=FAKE)

    def call(**kw):
        a = dict(args, **kw)
        return getattr(L, entry)(a["q"], a["k"], a["v"], a["kv"], a["ks"], a["vs"], a["P"],
                                 a["indptr"], a["indices"], a["page"], a["B"], a["q_len"],
                                 a["Hq"], a["Hkv"], a["d"], a["scale"], a["tm"], a["C"],
                                 a["po"], a["pl"], None)

    assert call(q=None) == -1
    assert call(kv=7) == -1
    assert call(kv=1) == -1                       # E4M3 without scales
    assert call(B=0) == -1
    assert call(scale=float("nan")) == -1
    assert call(d=64) == -2
    assert call(page=32) == -2
    assert call(Hq=60) == -2                      # Hq not a multiple of Hkv
    assert call(q_len=9) == -2                    # 8 * 9 rows > 64
    assert call(P=1 << 29) == -2                  # page*head index beyond int32
    assert call(k=FAKE + 8) == -4
    assert call(po=FAKE + 4) == -4


def test_combine_argument_checks():
    L = hpa.lib()
    assert L.hpa_combine(None, FAKE, FAKE, 3, 4, 1, 64, 128, FAKE, None, None) == -1
    assert L.hpa_combine(FAKE, FAKE, FAKE, 3, 4, 1, 64, 64, FAKE, None, None) == -2
    assert L.hpa_combine(FAKE, FAKE, FAKE, 3, 4, 1, 64, 128, FAKE + 2, None, None) == -4


def test_error_strings():
    L = hpa.lib()
    for c in (0, -1, -2, -3, -4, -5, 99):
        assert L.hpa_error_string(c)


def test_selftest_argument_checks():
    L = hpa.lib()
    assert L.hpa_selftest_wait_timeout(None, 10**6, None) == -1
    assert L.hpa_selftest_wait_timeout(FAKE, 10, None) == -1
    assert L.hpa_selftest_wait_timeout(FAKE + 2, 10**6, None) == -4


def test_weighted_plan_size_limit():
    L = hpa.lib()
    B, C = 3000, 2000                            # too large to stage the key prefix
    nb = hpa.hpa_taskmap_bytes(B, C)
    assert L.hpa_plan_weighted(FAKE, B, 512, C, FAKE, nb, None) == -2
    assert L.hpa_plan_weighted(None, 3, 512, 4, FAKE, hpa.hpa_taskmap_bytes(3, 4), None) == -1


def test_store_kv_argument_checks():
    L = hpa.lib()

    def call(**kw):
        a = dict(k=FAKE, v=FAKE, lens=FAKE, ip=FAKE, ix=FAKE, P=10, page=64, cs=FAKE, maxpos=100,
                 w=FAKE, eps=1e-6, had=1, kv=0, ks=None, vs=None, kp=FAKE, vp=FAKE, B=2, q=1,
                 Hkv=8, d=128, st=None)
        a.update(kw)
        return L.hpa_store_kv(a["k"], a["v"], a["lens"], a["ip"], a["ix"], a["P"], a["page"],
                              a["cs"], a["maxpos"], a["w"], a["eps"], a["had"], a["kv"], a["ks"],
                              a["vs"], a["kp"], a["vp"], a["B"], a["q"], a["Hkv"], a["d"],
                              a["st"], None)

    assert call(k=None) == -1
    assert call(kv=1) == -1                      # E4M3 without scales
    assert call(eps=-1.0) == -1
    assert call(d=64) == -2
    assert call(page=16) == -2
    assert call(cs=FAKE + 4) == -4
    assert call(k=FAKE + 8) == -4
