"""ORACLE -- test infrastructure only (tests, smoke check, CPU-baseline leg).

Reference tile scheduler for split-KV decode attention, written as plain
sequential loops.  Sources (page title, section):

  [Notes §3.1]  "Hy3 Preview AI Infra 推理优化精读笔记", §3.1 "Attention：动态切分和
                负载均衡", 方案 steps 1-4 and the 1024/5120/2048 example below them.
  [HPC-Ops §二.1] "腾讯混元AI Infra进化：HPC-Ops推理核心算子全面升级", §二.1
                (Task Assign builds a task map before each step; every layer's
                attention kernel takes its work from it).
  [Stack §二.1]  "大模型推理性能优化新范式：Hy3架构下的全栈优化技术拆解", §二.1
                (the per-CTA budget: base = total // ctas, the first
                total % ctas CTAs get one more).

Readings adopted where the pages are silent, ambiguous or at odds:
  1. tiles per request = ceil(L / tile) (the example cannot tell floor from
     ceil; floor would drop keys, and attention must see every key);
  2. the remainder goes to the lowest-indexed CTAs ([Stack §二.1]);
  3. the stream is request-major, tile-minor, requests in batch order;
  4. "greedy" fills CTA 0 up to its budget, then CTA 1, ... along the stream
     (contiguous ranges), not longest-first into the least-loaded bucket;
  5. a partial last tile counts as one whole tile of budget;
  6. when there are more CTAs than tiles, the surplus CTAs get no work.

Token-weighted variant (plan_weighted): the same stream and contiguous
partitions, with budgets counted in keys instead of tiles.

Static split-KV comparator ([Notes §3.1] 问题; the pages do not give its
rule): request r is cut into min(S, n_r) contiguous chunks of near-equal tile
counts (the first n_r % chunks get one more); CTA c = r * S + s owns chunk s of
request r, or nothing when s >= min(S, n_r).
"""
from __future__ import annotations

import numpy as np


def tile_counts(seq_lens, tile):
    """a1: n_r = ceil(L_r / tile)."""
    out = []
    for L in seq_lens:
        L = int(L)
        if L <= 0:
            raise ValueError("sequence length must be positive")
        out.append((L + tile - 1) // tile)
    return out


def stream_offsets(counts):
    """a2: exclusive running sum of tile counts; cu[B] = T."""
    cu = [0]
    for n in counts:
        cu.append(cu[-1] + n)
    return cu


def budgets(T, num_ctas):
    """a3: equal budgets, base = T // C, the first T % C CTAs get +1."""
    base, rem = divmod(T, num_ctas)
    return base, rem, [base + (1 if c < rem else 0) for c in range(num_ctas)]


def plan(seq_lens, tile, num_ctas):
    """a1-a4: the dynamic, load-balanced task map (as plain Python lists)."""
    if tile <= 0 or num_ctas <= 0:
        raise ValueError("tile and num_ctas must be positive")
    counts = tile_counts(seq_lens, tile)
    cu = stream_offsets(counts)
    T = cu[-1]
    base, rem, load = budgets(T, num_ctas)

    # a4: walk the tile stream, filling CTA c until its budget is reached.
    owner = []                 # owner[t] = CTA of stream tile t
    c, filled = 0, 0
    for t in range(T):
        while load[c] == filled:   # move on to the next CTA with budget left
            c, filled = c + 1, 0
        owner.append(c)
        filled += 1

    segs = []                  # (req, tile_lo, tile_hi, cta), request-local tiles
    for r, n in enumerate(counts):
        for i in range(n):
            c = owner[cu[r] + i]
            if segs and segs[-1][0] == r and segs[-1][3] == c:
                segs[-1][2] = i + 1
            else:
                segs.append([r, i, i + 1, c])

    cta_begin = [0]
    for c in range(num_ctas):
        cta_begin.append(cta_begin[-1] + load[c])
    return _assemble(seq_lens, tile, num_ctas, counts, cu, cta_begin, segs, base, rem,
                     kind=0, splits=0)


def plan_weighted(seq_lens, tile, num_ctas):
    """Token-weighted variant: tiles are shared out by the keys they hold.

    A partial last tile weighs its fill, not one whole tile (a reading the
    pages leave open).  With K the total number of keys, P_t the keys before
    stream tile t and w_t the keys in it, tile t goes to the partition whose
    equal share of the key stream holds the tile's middle key:
    floor(C * (2 P_t + w_t) / (2 K)).  Walking the stream, partition c takes
    tiles while their middles fall within its share [c K / C, (c+1) K / C).
    Each partition's key load is within one tile of K / C.
    """
    if tile <= 0 or num_ctas <= 0:
        raise ValueError("tile and num_ctas must be positive")
    counts = tile_counts(seq_lens, tile)
    cu = stream_offsets(counts)
    K = sum(int(L) for L in seq_lens)
    owner, before = [], 0                  # before = keys ahead of the current tile
    for r, L in enumerate(seq_lens):
        for i in range(counts[r]):
            w = min(tile, int(L) - i * tile)
            owner.append((num_ctas * (2 * before + w)) // (2 * K))
            before += w
    segs = []
    for r, n in enumerate(counts):
        for i in range(n):
            c = owner[cu[r] + i]
            if segs and segs[-1][0] == r and segs[-1][3] == c:
                segs[-1][2] = i + 1
            else:
                segs.append([r, i, i + 1, c])
    cta_begin = []
    t = 0
    for c in range(num_ctas):
        while t < len(owner) and owner[t] < c:
            t += 1
        cta_begin.append(t)
    cta_begin.append(cu[-1])
    base = min(K // num_ctas, 2**31 - 1)
    return _assemble(seq_lens, tile, num_ctas, counts, cu, cta_begin, segs, base,
                     K % num_ctas, kind=2, splits=0)


def plan_static(seq_lens, tile, splits):
    """Static split-KV: a fixed number of chunks per request, one CTA per chunk."""
    if tile <= 0 or splits <= 0:
        raise ValueError("tile and splits must be positive")
    counts = tile_counts(seq_lens, tile)
    cu = stream_offsets(counts)
    B = len(counts)
    C = B * splits
    segs, cta_begin = [], []
    for r, n in enumerate(counts):
        k = min(splits, n)
        base, rem = divmod(n, k)
        lo = 0
        for s in range(splits):
            if s < k:
                size = base + (1 if s < rem else 0)
                segs.append([r, lo, lo + size, r * splits + s])
                cta_begin.append(cu[r] + lo)
                lo += size
            else:
                cta_begin.append(cu[r + 1])
    cta_begin.append(cu[-1])
    return _assemble(seq_lens, tile, C, counts, cu, cta_begin, segs, -1, -1, kind=1,
                     splits=splits)


def _assemble(seq_lens, tile, C, counts, cu, cta_begin, segs, base, rem, kind, splits):
    B = len(counts)
    S = len(segs)
    cta_seg = [0] * (C + 1)
    for s in segs:
        cta_seg[s[3] + 1] += 1
    for c in range(C):
        cta_seg[c + 1] += cta_seg[c]
    seg_off = [0] * (B + 1)
    for s in segs:
        seg_off[s[0] + 1] += 1
    for r in range(B):
        seg_off[r + 1] += seg_off[r]
    i32 = lambda x: np.asarray(x, dtype=np.int32)
    return {
        "T": cu[-1], "base": base, "rem": rem, "C": C, "B": B, "S": S, "tile": tile,
        "kind": kind, "splits": splits,
        "lens": i32([int(L) for L in seq_lens]),
        "counts": i32(counts), "cu_tiles": i32(cu), "cta_begin": i32(cta_begin),
        "cta_seg": i32(cta_seg), "seg_off": i32(seg_off),
        "segs": np.asarray(segs, dtype=np.int32).reshape(S, 4),
    }


def cta_loads(p):
    """Tiles owned by each CTA."""
    return np.diff(p["cta_begin"])


def segment_key_ranges(p):
    """[(req, key_lo, key_hi)] of each segment, keys clipped to the request length."""
    out = []
    for r, lo, hi, _ in p["segs"]:
        L = int(p["lens"][r])
        out.append((int(r), int(lo) * p["tile"], min(int(hi) * p["tile"], L)))
    return out
