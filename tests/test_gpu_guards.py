"""Guard bands and corrupted task maps (the stand-ins for a memory checker, which
this pool does not offer).

Guard bands: every buffer the kernels write -- the task map, partial_o,
partial_lse, out, out_lse and the fused combine's arrival counters -- is a
view into a larger allocation whose head and tail hold a sentinel pattern.
After a step, the results must match the fp64 oracle and every sentinel byte
must be unchanged, so no kernel wrote outside the extent the C ABI states.

Corrupted maps: a map written by hpa_plan is altered on the host (a segment
row pointing at a request that does not exist, a tile range past its
request's end, a row owned by another partition, a partition's segment range
past the map's segments, a request's segment range past the partials) and
the step is run again.  The kernels must report HPA_STATUS_BAD_MAP, make the
affected outputs NaN, and write nothing outside their buffers.
"""
import numpy as np
import pytest
import torch

import load_balanced_split_gb300 as hpa
import oracle
import workloads as W
from gpu_helpers import DeviceBatch, assert_close, assert_lse_close, decode_taskmap

pytestmark = pytest.mark.gpu

GUARD = 1024          # elements of sentinel before and after each buffer
BAD_MAP = 32
_SENTINEL = {torch.float32: (torch.int32, 0x7FA5A5A5), torch.int32: (torch.int32, 0x5A5A5A5A),
             torch.bfloat16: (torch.int16, 0x7FA5)}


class Guarded:
    """A device tensor of n elements inside an allocation with sentinel bands around it."""

    def __init__(self, n, dtype, shape=None, zero=False):
        self.n = n
        self.raw = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        ity, fill = _SENTINEL[dtype]
        self.ity, self.fill = ity, fill
        self.raw.view(ity).fill_(fill)
        self.t = self.raw[GUARD:GUARD + n]
        if zero:
            self.t.zero_()
        if shape is not None:
            self.t = self.t.view(shape)

    def intact(self) -> bool:
        r = self.raw.view(self.ity)
        return bool((r[:GUARD] == self.fill).all()) and bool((r[GUARD + self.n:] == self.fill).all())


class Step:
    """Task map, partials and outputs of one decode step, all guarded."""

    def __init__(self, b, C):
        self.b, self.C = b, C
        cap = hpa.hpa_max_segments(b.B, C)
        self.tm = Guarded(hpa.hpa_taskmap_bytes(b.B, C) // 4, torch.int32)
        self.po = Guarded(cap * b.q_len * b.Hq * b.d, torch.float32)
        self.pl = Guarded(cap * b.q_len * b.Hq, torch.float32)
        self.out = Guarded(b.B * b.q_len * b.Hq * b.d, torch.bfloat16, (b.B, b.q_len, b.Hq, b.d))
        self.lse = Guarded(b.B * b.q_len * b.Hq, torch.float32, (b.B, b.q_len, b.Hq))
        self.arr = Guarded(hpa.hpa_arrivals_elems(b.B, b.Hq, b.Hkv, b.q_len), torch.int32,
                           zero=True)

    def buffers(self):
        return [self.tm, self.po, self.pl, self.out, self.lse, self.arr]

    def plan(self, db):
        hpa.hpa_plan(db.lens, self.b.tile, self.C, self.tm.t)

    def attend(self, db, kernel):
        if kernel == "fused":
            hpa.hpa_decode_attn_fused(db.q, db.k, db.v, db.indptr, db.indices, self.tm.t, self.C,
                                      self.po.t, self.pl.t, self.out.t, self.arr.t, self.lse.t,
                                      db.ks, db.vs)
            return
        hpa.hpa_decode_attn(db.q, db.k, db.v, db.indptr, db.indices, self.tm.t, self.C,
                            self.po.t, self.pl.t, db.ks, db.vs, tc=kernel == "tc",
                            mma=kernel == "mma")
        hpa.hpa_combine(self.po.t, self.pl.t, self.tm.t, self.C, self.out.t, self.lse.t)

    def status(self) -> int:
        return int(self.tm.t[6].item())


GUARD_CASES = [
    dict(lens=[2, 63, 64, 65, 511, 512, 513, 1000, 3333, 4113], q_len=2, kv="bf16", C=23),
    dict(lens=[100, 700, 30], q_len=1, kv="e4m3", C=40),                    # surplus partitions
    dict(lens=list(np.random.default_rng(31).integers(2, 301, size=3000)), q_len=2, kv="e4m3",
         C=None),                                                           # thousands of segments
]


@pytest.mark.parametrize("kernel", ["mma", "tc", "fused"])
@pytest.mark.parametrize("case", range(len(GUARD_CASES)))
def test_guard_bands_untouched(case, kernel):
    c = GUARD_CASES[case]
    b = W.make_batch(c["lens"], q_len=c["q_len"], kv_dtype=c["kv"], seed=150 + case)
    db = DeviceBatch(b)
    kv = hpa.KV_BF16 if b.kv_dtype == "bf16" else hpa.KV_E4M3
    C = c["C"] or (hpa.hpa_default_num_ctas_tc if kernel == "tc" else hpa.hpa_default_num_ctas_mma)(
        b.Hkv, b.q_len, kv, b.Hq)
    st = Step(b, C)
    st.plan(db)
    st.attend(db, kernel)
    torch.cuda.synchronize()
    assert st.status() == 0
    ref, ref_lse = oracle.attention(b)
    assert_close(st.out.t.float().cpu().numpy(), ref, b.kv_dtype, "out")
    assert_lse_close(st.lse.t.cpu().numpy(), ref_lse, "out_lse")
    for name, g in zip(("taskmap", "partial_o", "partial_lse", "out", "out_lse", "arrivals"),
                       st.buffers()):
        assert g.intact(), "%s: sentinel band overwritten" % name


def _corrupt(tm_host, b, C, how):
    """Alter one part of a decoded map in place (int32 words of the blob)."""
    m = decode_taskmap(tm_host, b.B, C)
    B, S = b.B, m["S"]
    o_cta_seg = 16 + B + (B + 1) + (C + 1)
    o_seg_off = o_cta_seg + (C + 1)
    o_segs = (o_seg_off + B + 1 + 3) & ~3
    seg = 1                                              # a row in the middle of the table
    r = int(m["segs"][seg][0])
    if how == "request":
        tm_host[o_segs + 4 * seg + 0] = B + 1000
    elif how == "tile_hi":
        n_r = int(m["cu_tiles"][r + 1] - m["cu_tiles"][r])
        tm_host[o_segs + 4 * seg + 2] = n_r + 5
    elif how == "owner":
        tm_host[o_segs + 4 * seg + 3] = (int(m["segs"][seg][3]) + 1) % C
    elif how == "cta_seg":
        tm_host[o_cta_seg + 1] = S + 7                    # partition 0's range past the map
    elif how == "seg_off":
        tm_host[o_seg_off + 2] = S + 100                  # request 1's range past the partials
        return 1
    else:
        raise ValueError(how)
    return None


@pytest.mark.parametrize("kernel", ["mma", "tc"])
@pytest.mark.parametrize("how", ["request", "tile_hi", "owner", "cta_seg", "seg_off"])
def test_corrupted_map_is_reported_not_followed(how, kernel):
    b = W.make_batch([3000, 40, 12000, 700], q_len=2, kv_dtype="e4m3", seed=160)
    db = DeviceBatch(b)
    C = 6
    st = Step(b, C)
    st.plan(db)
    torch.cuda.synchronize()
    host = st.tm.t.cpu().numpy().copy()
    bad_req = _corrupt(host, b, C, how)
    st.tm.t.copy_(torch.from_numpy(host))
    st.attend(db, kernel)
    torch.cuda.synchronize()
    assert st.status() & BAD_MAP, "status %d" % st.status()
    out = st.out.t.float()
    if bad_req is None:       # the attention kernel flagged it: the combine writes NaN everywhere
        assert torch.isnan(out).all()
    else:                     # the combine flagged one request's range: that request is NaN
        assert torch.isnan(out[bad_req]).all()
    for name, g in zip(("taskmap", "partial_o", "partial_lse", "out", "out_lse"), st.buffers()):
        assert g.intact(), "%s: sentinel band overwritten" % name


def test_corrupted_map_fused_combine():
    """The fused kernel reports a bad row (and its request's segment range) without
    following it; the caller re-zeroes the arrival counters after a bad status."""
    b = W.make_batch([3000, 40, 12000, 700], q_len=1, seed=161)
    db = DeviceBatch(b)
    C = 6
    for how in ("request", "owner", "seg_off"):
        st = Step(b, C)
        st.plan(db)
        torch.cuda.synchronize()
        host = st.tm.t.cpu().numpy().copy()
        _corrupt(host, b, C, how)
        st.tm.t.copy_(torch.from_numpy(host))
        st.attend(db, "fused")
        torch.cuda.synchronize()
        assert st.status() & BAD_MAP, (how, st.status())
        for name, g in zip(("taskmap", "partial_o", "partial_lse", "out", "out_lse", "arrivals"),
                           st.buffers()):
            assert g.intact(), "%s (%s): sentinel band overwritten" % (name, how)
    # the context is still good: a clean step afterwards matches the oracle
    st = Step(b, C)
    st.plan(db)
    st.attend(db, "fused")
    torch.cuda.synchronize()
    assert st.status() == 0
    ref, _ = oracle.attention(b)
    assert_close(st.out.t.float().cpu().numpy(), ref, "bf16", "out after bad maps")
