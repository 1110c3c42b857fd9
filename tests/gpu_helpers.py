"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on a
workloads.Batch, decode the task map blob (format stated in include/hpa.h),
and compare against the oracle with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import load_balanced_split_gb300 as hpa
import workloads as W

HEADER = 16

# Output tolerance: |d| <= ABS (+ half an ulp of bf16 at ref, for outputs stored as bf16)
# and |d| <= REL * max(|ref|, rms of the ref row of d values).
TOL = {"bf16": (1e-2, 2e-2), "e4m3": (5e-2, 5e-2)}
LSE_REL = 1e-4  # |d lse| <= 1e-4 * max(|ref lse|, 1)


def decode_taskmap(tm: np.ndarray, B: int, C: int) -> dict:
    tm = np.asarray(tm, dtype=np.int32)
    h = tm[:HEADER]
    o = HEADER
    out = {"T": int(h[0]), "base": int(h[1]), "rem": int(h[2]), "C": int(h[3]), "B": int(h[4]),
           "S": int(h[5]), "status": int(h[6]), "tile": int(h[7]), "kind": int(h[8]),
           "splits": int(h[9]), "S_cap": int(h[10]), "header_tail": h[11:HEADER].copy()}
    out["lens"] = tm[o:o + B].copy(); o += B
    out["cu_tiles"] = tm[o:o + B + 1].copy(); o += B + 1
    out["cta_begin"] = tm[o:o + C + 1].copy(); o += C + 1
    out["cta_seg"] = tm[o:o + C + 1].copy(); o += C + 1
    out["seg_off"] = tm[o:o + B + 1].copy(); o += B + 1
    o = (o + 3) & ~3
    cap = out["S_cap"]
    out["segs_all"] = tm[o:o + 4 * cap].reshape(cap, 4).copy()
    out["segs"] = out["segs_all"][:out["S"]]
    out["words"] = o + 4 * cap
    return out


def expect_taskmap_equal(gpu: dict, ref: dict, s_cap: int):
    """Bit-exact comparison of every field of the decoded map with the oracle plan."""
    for k in ("T", "C", "B", "S", "tile", "kind", "splits"):
        assert gpu[k] == ref[k], (k, gpu[k], ref[k])
    if ref["kind"] in (0, 2):        # tile budget, or key budget for the token-weighted map
        assert (gpu["base"], gpu["rem"]) == (ref["base"], ref["rem"])
    else:
        assert (gpu["base"], gpu["rem"]) == (-1, -1)
    assert gpu["status"] == 0
    assert gpu["S_cap"] == s_cap
    assert (gpu["header_tail"] == 0).all()
    for k in ("lens", "cu_tiles", "cta_begin", "cta_seg", "seg_off", "segs"):
        np.testing.assert_array_equal(gpu[k], ref[k], err_msg=k)
    assert (gpu["segs_all"][gpu["S"]:] == -1).all()


class DeviceBatch:
    """A workloads.Batch moved to the GPU."""

    def __init__(self, b, device="cuda"):
        self.b = b
        self.q = b.q.to(device)
        if b.kv_dtype == "bf16":
            self.k = b.k_pool.to(device)
            self.v = b.v_pool.to(device)
            self.ks = self.vs = None
        else:
            self.k = b.k_pool.to(device)
            self.v = b.v_pool.to(device)
            self.ks = torch.from_numpy(b.k_scale).to(device)
            self.vs = torch.from_numpy(b.v_scale).to(device)
        self.lens = torch.from_numpy(b.seq_lens).to(device)
        self.indptr = torch.from_numpy(b.page_indptr).to(device)
        self.indices = torch.from_numpy(b.page_indices).to(device)


def num_ctas_for(b, tc=False, allheads=False, mma=False) -> int:
    if b.num_ctas is not None:
        return b.num_ctas
    fn = (hpa.hpa_default_num_ctas_tc if tc else
          hpa.hpa_default_num_ctas_allheads if allheads else
          hpa.hpa_default_num_ctas_mma if mma else hpa.hpa_default_num_ctas)
    return fn(b.Hkv, b.q_len, hpa.KV_BF16 if b.kv_dtype == "bf16" else hpa.KV_E4M3, b.Hq)


def run_gpu(b, num_ctas=None, splits=None, tile=512, db=None, fused=False, weighted=False,
            tc=False, sm_scale=None, allheads=False, mma=False):
    """plan -> attention -> combine on the GPU (fused: one attention launch with the
    combine folded in; tc / mma: the tcgen05 / mma.sync attention kernel forced; by
    default hpa_decode_attn picks by row count).  Returns host numpy results."""
    db = db or DeviceBatch(b)
    if splits is None and num_ctas is None:
        num_ctas = num_ctas_for(b, tc, allheads, mma)
    ws = hpa.Workspace(b.B, b.q_len, b.Hq, b.d, num_ctas=num_ctas, splits=splits,
                       weighted=weighted)
    ws.partial_o.fill_(float("nan"))
    ws.partial_lse.fill_(float("nan"))
    out = torch.empty((b.B, b.q_len, b.Hq, b.d), dtype=torch.bfloat16, device="cuda")
    out_lse = torch.empty((b.B, b.q_len, b.Hq), dtype=torch.float32, device="cuda")
    hpa.decode_step(ws, db.q, db.k, db.v, db.lens, db.indptr, db.indices, out, out_lse,
                    db.ks, db.vs, tile=tile, fused=fused, tc=tc, sm_scale=sm_scale,
                    allheads=allheads, mma=mma)
    torch.cuda.synchronize()
    if fused:
        assert int(ws.arrivals.abs().sum().item()) == 0, "arrival counters not reset"
    tm = decode_taskmap(ws.taskmap.cpu().numpy(), b.B, ws.num_ctas)
    S = tm["S"]
    po = ws.partial_o.view(-1, b.q_len, b.Hq, b.d)[:S].cpu().numpy().astype(np.float64)
    pl = ws.partial_lse.view(-1, b.q_len, b.Hq)[:S].cpu().numpy().astype(np.float64)
    return {"out": out.float().cpu().numpy().astype(np.float64),
            "lse": out_lse.cpu().numpy().astype(np.float64), "po": po, "pl": pl, "tm": tm,
            "num_ctas": ws.num_ctas,
            "capacity": ws.num_ctas if splits is not None else ws.capacity}


def scaled_query_batch(lens, q_len, kv, seed, case):
    """A batch whose query rows lie far outside N(0,1), with the softmax scale that goes
    with them.  "large": every row times 1e5 (elements beyond f16's 65504) and
    sm_scale / 1e5; "tiny": every row times 1e-6 (elements in f16's subnormal range)
    and sm_scale * 1e6, so the scores keep their usual size and any precision lost in
    the query shows in the output; "mixed_rows": rows of one batch times 1e5, 1e-6 or 1
    in turn, default scale; "mixed": the same plus one head whose rows hold a single
    element of 3e5 among N(0,1) values (a ratio of 3e5 inside one row)."""
    import math as _m
    b = W.make_batch(lens, q_len=q_len, kv_dtype=kv, seed=seed)
    q = b.q.float()
    sm = 1.0 / _m.sqrt(b.d)
    if case == "large":
        q *= 1e5
        sm /= 1e5
    elif case == "tiny":
        q *= 1e-6
        sm *= 1e6
    elif case in ("mixed", "mixed_rows"):
        f = torch.ones(q.shape[:3])
        f.view(-1)[0::3] = 1e5
        f.view(-1)[1::3] = 1e-6
        f[:, :, 5] = 1.0
        q *= f[..., None]
        if case == "mixed":
            q[:, :, 5, 7] = 3e5
    else:
        raise ValueError(case)
    b.q = q.to(torch.bfloat16)
    return b, sm


def assert_close(got, ref, kv, what="out"):
    """Element-wise check against the fp64 reference.  The absolute bound covers the
    attention arithmetic; outputs stored as bf16 (everything but the fp32 split
    partials) also carry their own rounding, up to half an ulp of bf16 at the
    reference value (2^-6 for |ref| in [4, 8), more than 1e-2 on its own)."""
    ab, rel = TOL[kv]
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), "%s has non-finite values" % what
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    floor = np.maximum(np.abs(ref), rms)
    d = np.abs(got - ref)
    if not what.startswith("partial"):
        aref = np.abs(ref)
        with np.errstate(divide="ignore"):
            half_ulp = np.where(aref > 0, 2.0 ** (np.floor(np.log2(np.where(aref > 0, aref, 1.0))) - 8), 0.0)
        ab = ab + half_ulp
    bad = (d > ab) | (d > rel * floor)
    if bad.any():
        i = np.unravel_index(np.argmax(d / np.maximum(floor, 1e-30)), d.shape)
        raise AssertionError("%s: %d of %d elements out of tolerance; worst at %s: got %r ref %r"
                             % (what, int(bad.sum()), bad.size, i, got[i], ref[i]))
    return float(d.max()), float((d / np.maximum(floor, 1e-30)).max())


def assert_lse_close(got, ref, what="lse"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isneginf(ref)
    assert (np.isneginf(got) == inf).all(), "%s: -inf pattern differs" % what
    d = np.abs(got[~inf] - ref[~inf])
    lim = LSE_REL * np.maximum(np.abs(ref[~inf]), 1.0)
    assert (d <= lim).all(), "%s: max |d| %g" % (what, d.max() if d.size else 0)
    return float(d.max()) if d.size else 0.0
