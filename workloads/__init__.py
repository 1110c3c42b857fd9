"""Seeded synthetic inputs for GQA decode attention over a paged KV cache.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests.  It holds input generation only -- request lengths, query vectors, KV
pages, page tables and the 8-bit encoding of the KV inputs -- and none of the
attention, scheduling or merging arithmetic.

Shapes follow the model the pages describe (Hy3 Preview AI Infra 推理优化精读笔记,
§2 "模型与问题背景": 64 attention heads, 8 KV heads, head dim 128) and the
workloads they quote (same page, §1: average input about 68K tokens, maximum
about 192K; §3.1 "对我们的启发": a mixed batch holding 1K, 4K, 16K, 64K and
128K requests).  No dataset or trace is read: every array is drawn from a
seeded numpy stream, so any page or query block can be regenerated on its own.

Layout of what is produced (host memory, C order):
  q            bf16 [B][q_len][Hq][d]
  k_pool/v_pool bf16 or uint8 (E4M3 codes) [num_pages][Hkv][page_size][d]
  k_scale/v_scale float32 [Hkv] (E4M3 only; value = code * scale)
  seq_lens     int32 [B]   (KV length, counting the q_len new tokens)
  page_indptr  int32 [B+1] (CSR offsets into page_indices)
  page_indices int32 [sum ceil(L/page_size)]
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

HQ, HKV, HEAD_DIM, PAGE_SIZE, TILE = 64, 8, 128, 64, 512
E4M3_MAX = 448.0

# stream ids of the seeded generators (one numpy stream per (seed, id, chunk))
_S_LENS, _S_Q, _S_K, _S_V, _S_PERM = 1, 2, 3, 4, 5
_CHUNK_PAGES = 64


@dataclass
class Batch:
    """One decode batch; host tensors only (the caller moves them)."""
    name: str
    seq_lens: np.ndarray            # int32 [B]
    q: torch.Tensor                 # bf16 [B][q_len][Hq][d]
    k_pool: torch.Tensor            # bf16 or uint8 [P][Hkv][page][d]
    v_pool: torch.Tensor
    page_indptr: np.ndarray         # int32 [B+1]
    page_indices: np.ndarray        # int32 [nnz]
    kv_dtype: str                   # "bf16" | "e4m3"
    q_len: int
    k_scale: np.ndarray | None = None   # float32 [Hkv]
    v_scale: np.ndarray | None = None
    num_ctas: int | None = None     # forced partition count (None: device default)
    tile: int = TILE
    page_size: int = PAGE_SIZE
    Hq: int = HQ
    Hkv: int = HKV
    d: int = HEAD_DIM
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one pass reads: sum L * Hkv * d * 2 (K and V) * element size."""
        es = 2 if self.kv_dtype == "bf16" else 1
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * self.d * 2 * es


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_chunk(seed: int, stream: int, chunk: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    np.random.default_rng([seed, stream, chunk]).standard_normal(out=out, dtype=np.float32)
    return out


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """fp32 -> bf16, round to nearest even (torch's conversion)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def encode_e4m3(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> OCP E4M3 codes (uint8), round to nearest even, saturated at +-448."""
    return x.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


# ----------------------------------------------------------------------------- lengths
def lens_worked_example() -> np.ndarray:
    return np.array([1024, 5120, 2048], dtype=np.int32)


def lens_uniform(B: int = 32, L: int = 8192) -> np.ndarray:
    return np.full(B, L, dtype=np.int32)


def lens_mixed(seed: int = 0, n_random: int = 40) -> np.ndarray:
    """n_random lengths round(exp(U(ln 1K, ln 128K))) plus exactly 1K/4K/16K/64K/128K, shuffled."""
    rng = np.random.default_rng([seed, _S_LENS, 3])
    u = rng.uniform(math.log(1024), math.log(131072), size=n_random)
    L = np.concatenate([np.round(np.exp(u)), [1024, 4096, 16384, 65536, 131072]])
    L = L[rng.permutation(L.shape[0])]
    return np.clip(L, 1024, 131072).astype(np.int32)


def lens_long(L: int = 196608) -> np.ndarray:
    return np.array([L], dtype=np.int32)


def lens_lognormal(seed: int = 0, B: int = 64, mean: float = 68000.0, sigma: float = 0.75,
                   lo: int = 512, hi: int = 196608) -> np.ndarray:
    """B lengths clip(round(exp(mu + sigma z)), lo, hi); mu bisected so the batch mean is ~mean."""
    z = np.random.default_rng([seed, _S_LENS, 5]).standard_normal(B)

    def draw(mu):
        return np.clip(np.round(np.exp(mu + sigma * z)), lo, hi)

    a, b = math.log(lo), math.log(hi)
    for _ in range(200):
        mid = 0.5 * (a + b)
        if draw(mid).mean() < mean:
            a = mid
        else:
            b = mid
    return draw(0.5 * (a + b)).astype(np.int32)


# ----------------------------------------------------------------------------- tensors
def make_q(seed: int, B: int, q_len: int, Hq: int = HQ, d: int = HEAD_DIM) -> torch.Tensor:
    x = _normal_chunk(seed, _S_Q, 0, B * q_len * Hq * d).reshape(B, q_len, Hq, d)
    return to_bf16(x)


def page_table(seed: int, seq_lens: np.ndarray, page_size: int, shuffle: bool):
    npg = (seq_lens.astype(np.int64) + page_size - 1) // page_size
    indptr = np.zeros(seq_lens.shape[0] + 1, dtype=np.int64)
    np.cumsum(npg, out=indptr[1:])
    P = int(indptr[-1])
    if shuffle:
        idx = np.random.default_rng([seed, _S_PERM, 0]).permutation(P)
    else:
        idx = np.arange(P)
    return indptr.astype(np.int32), idx.astype(np.int32), P


def _pool_chunks(P: int):
    return [(c, c * _CHUNK_PAGES, min(P, (c + 1) * _CHUNK_PAGES))
            for c in range((P + _CHUNK_PAGES - 1) // _CHUNK_PAGES)]


def make_pool_bf16(seed: int, stream: int, P: int, Hkv: int, page_size: int, d: int) -> torch.Tensor:
    pool = torch.empty((P, Hkv, page_size, d), dtype=torch.bfloat16)
    per_page = Hkv * page_size * d

    def work(ch):
        c, p0, p1 = ch
        x = _normal_chunk(seed, stream, c, (p1 - p0) * per_page)
        pool[p0:p1].copy_(torch.from_numpy(x).view(p1 - p0, Hkv, page_size, d))

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, _pool_chunks(P)))
    return pool


def make_pool_e4m3(seed: int, stream: int, P: int, Hkv: int, page_size: int, d: int):
    """N(0,1) values encoded as E4M3 with one fp32 scale per KV head: scale = amax / 448.

    Two passes over the same seeded chunks (amax, then encode), so the fp32
    pool is never held whole.
    """
    per_page = Hkv * page_size * d
    chunks = _pool_chunks(P)

    def amax(ch):
        c, p0, p1 = ch
        x = _normal_chunk(seed, stream, c, (p1 - p0) * per_page).reshape(p1 - p0, Hkv, -1)
        return np.abs(x).max(axis=(0, 2))

    with ThreadPoolExecutor(_threads()) as ex:
        am = np.max(np.stack(list(ex.map(amax, chunks))), axis=0)
    scale = (am / E4M3_MAX).astype(np.float32)
    pool = torch.empty((P, Hkv, page_size, d), dtype=torch.uint8)
    inv = torch.from_numpy(scale).view(1, Hkv, 1, 1)

    def enc(ch):
        c, p0, p1 = ch
        x = torch.from_numpy(_normal_chunk(seed, stream, c, (p1 - p0) * per_page))
        x = x.view(p1 - p0, Hkv, page_size, d) / inv
        pool[p0:p1].copy_(encode_e4m3(x))

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(enc, chunks))
    return pool, scale


def make_batch(seq_lens, *, q_len: int = 1, kv_dtype: str = "bf16", seed: int = 0,
               shuffle_pages: bool = True, name: str = "custom", num_ctas: int | None = None,
               Hq: int = HQ, Hkv: int = HKV, d: int = HEAD_DIM, page_size: int = PAGE_SIZE,
               tile: int = TILE) -> Batch:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    indptr, indices, P = page_table(seed, seq_lens, page_size, shuffle_pages)
    q = make_q(seed, seq_lens.shape[0], q_len, Hq, d)
    ks = vs = None
    if kv_dtype == "bf16":
        k = make_pool_bf16(seed, _S_K, P, Hkv, page_size, d)
        v = make_pool_bf16(seed, _S_V, P, Hkv, page_size, d)
    elif kv_dtype == "e4m3":
        k, ks = make_pool_e4m3(seed, _S_K, P, Hkv, page_size, d)
        v, vs = make_pool_e4m3(seed, _S_V, P, Hkv, page_size, d)
    else:
        raise ValueError(kv_dtype)
    return Batch(name=name, seq_lens=seq_lens, q=q, k_pool=k, v_pool=v, page_indptr=indptr,
                 page_indices=indices, kv_dtype=kv_dtype, q_len=q_len, k_scale=ks, v_scale=vs,
                 num_ctas=num_ctas, tile=tile, page_size=page_size, Hq=Hq, Hkv=Hkv, d=d)


# ----------------------------------------------------------------------------- the five workloads
CONFIGS = {
    1: "worked_example_3req_1k_5k_2k",
    2: "uniform_32x8k_paged",
    3: "mixed_45req_1k_128k_paged",
    4: "single_192k_paged",
    5: "mtp2_64req_lognormal68k_e4m3",
}


def config_lens(cfg: int, seed: int = 0) -> np.ndarray:
    return {1: lens_worked_example, 2: lens_uniform, 3: lambda: lens_mixed(seed),
            4: lens_long, 5: lambda: lens_lognormal(seed)}[cfg]()


def make_config(cfg: int, seed: int = 0, max_requests: int | None = None,
                q_len: int | None = None) -> Batch:
    """The five decode workloads (sizes in the docstring of each length recipe).

    max_requests keeps only the first requests of the batch (smaller cases of
    the same workload, e.g. for profiling); q_len overrides the number of new
    query tokens per request (MTP variants)."""
    lens = config_lens(cfg, seed)
    if max_requests is not None:
        lens = lens[:max_requests]
    if cfg == 1:
        return make_batch(lens, q_len=q_len or 1, seed=seed, shuffle_pages=False,
                          name=CONFIGS[1], num_ctas=4)
    if cfg == 5:
        return make_batch(lens, q_len=q_len or 2, kv_dtype="e4m3", seed=seed, name=CONFIGS[5])
    return make_batch(lens, q_len=q_len or 1, seed=seed, name=CONFIGS[cfg])


# ----------------------------------------------------------------------------- KV-store feeder
def rope_cos_sin_table(max_pos: int, d: int = HEAD_DIM, theta: float = 10000.0) -> np.ndarray:
    """fp32 [max_pos][d]: cos(pos * theta^(-2i/d)) in columns i < d/2, sin in columns d/2 + i.

    The angles are formed in float64 and rounded once to fp32 (the table is an
    input of the KV writer, as a serving engine would pass it)."""
    inv = theta ** (-np.arange(0, d // 2, dtype=np.float64) * 2.0 / d)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


@dataclass
class FeederInputs:
    k_new: torch.Tensor        # bf16 [B][q_len][Hkv][d], the projected keys of the new tokens
    v_new: torch.Tensor        # bf16 [B][q_len][Hkv][d]
    norm_w: np.ndarray         # fp32 [d], RMSNorm weight
    cos_sin: np.ndarray        # fp32 [max_pos][d]
    eps: float = 1e-6


def make_feeder_inputs(seed: int, B: int, q_len: int, max_pos: int, Hkv: int = HKV,
                       d: int = HEAD_DIM, theta: float = 10000.0) -> FeederInputs:
    rng = np.random.default_rng([seed, 6, 0])
    k = rng.standard_normal((B, q_len, Hkv, d), dtype=np.float32) * 3.0
    v = rng.standard_normal((B, q_len, Hkv, d), dtype=np.float32)
    w = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    return FeederInputs(k_new=to_bf16(k), v_new=to_bf16(v), norm_w=w,
                        cos_sin=rope_cos_sin_table(max_pos, d, theta))
