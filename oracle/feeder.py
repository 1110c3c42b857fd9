"""ORACLE -- test infrastructure only (tests, smoke check, CPU-baseline leg).

Reference for the fused KV-cache writer that feeds the decode path:
"Hy3 Preview AI Infra 推理优化精读笔记", §4.1 "Rope + Norm + Hadamard + Quant +
Store KV" -- after the QKV projection, rotary position embedding, RMSNorm,
an optional Hadamard transform and quantisation are applied and the result is
written into the KV cache in its low-bit format, in one pass.

Readings where the pages are silent (the same ones the CUDA path takes):
  1. order as the pages list it: RoPE, then RMSNorm, then Hadamard, then
     quantisation; all of them act on K only, V is only quantised and stored;
  2. RoPE rotates halves: for i < d/2, (x_i, x_{i+d/2}) is turned by angle
     theta_{pos,i}; cos/sin come from a table the caller passes
     (cos_sin[pos][i] = cos, cos_sin[pos][d/2 + i] = sin);
  3. RMSNorm over the head dim: x / sqrt(mean(x^2) + eps) * w, w of length d;
  4. Hadamard: the Sylvester Walsh-Hadamard matrix of order d, scaled by
     1/sqrt(d) (orthonormal);
  5. quantisation: E4M3 code = round-to-nearest-even of x / scale[h] on the
     E4M3 grid, saturated at +-448; or bf16 (RNE) for a bf16 cache;
  6. new token j of request r sits at position L_r - q_len + j and goes to
     slot pos % page_size of page page_indices[page_indptr[r] + pos // page_size].
"""
from __future__ import annotations

import math

import numpy as np
import scipy.linalg

E4M3_MAX = 448.0


def e4m3_grid():
    """All finite non-negative E4M3 values, ascending (the encoder's rounding grid)."""
    vals = [0.0]
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                                   # NaN code
            v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
            if v > 0:
                vals.append(v)
    return np.array(sorted(set(vals)))


_GRID = e4m3_grid()


def encode_e4m3_value(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (ties to the even code), saturated at +-448 (fp64 in, fp64 out)."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    idx = np.searchsorted(_GRID, a)                       # _GRID[idx-1] < a <= _GRID[idx]
    idx = np.clip(idx, 1, len(_GRID) - 1)
    lo, hi = _GRID[idx - 1], _GRID[idx]
    pick_hi = (a - lo) > (hi - a)
    tie = (a - lo) == (hi - a)
    # ties: the even code; consecutive grid entries alternate code parity, code(i) = i
    even_hi = (idx % 2) == 0
    pick_hi = np.where(tie, even_hi, pick_hi)
    v = np.where(pick_hi, hi, lo)
    v = np.where(a == 0, 0.0, v)
    return np.copysign(v, x)


def rope_rotate_half(x: np.ndarray, cos_sin_row: np.ndarray) -> np.ndarray:
    d = x.shape[-1]
    h = d // 2
    c, s = cos_sin_row[:h], cos_sin_row[h:]
    out = np.empty_like(x)
    out[:h] = x[:h] * c - x[h:] * s
    out[h:] = x[h:] * c + x[:h] * s
    return out


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    return x / math.sqrt(float(np.mean(x * x)) + eps) * w


def hadamard(d: int) -> np.ndarray:
    return scipy.linalg.hadamard(d).astype(np.float64) / math.sqrt(d)


def store_kv(k_new, v_new, seq_lens, page_indptr, page_indices, cos_sin, norm_w, eps,
             use_hadamard, kv_dtype, k_scale=None, v_scale=None, page_size=64):
    """Returns {(page, head, slot): (k_value, v_value)} in fp64 for every new token.

    k_new, v_new: float64 [B][q_len][Hkv][d] (the bf16 inputs, widened);
    values are the pre-rounding results; `*_value` stored entries are what the
    cache must hold up to the final rounding (bf16 RNE, or E4M3 codes times
    their scale).
    """
    k_new = np.asarray(k_new, np.float64)
    v_new = np.asarray(v_new, np.float64)
    B, q_len, Hkv, d = k_new.shape
    H = hadamard(d) if use_hadamard else None
    out = {}
    for r in range(B):
        L = int(seq_lens[r])
        for j in range(q_len):
            pos = L - q_len + j
            page = int(page_indices[int(page_indptr[r]) + pos // page_size])
            slot = pos % page_size
            for h in range(Hkv):
                k = rope_rotate_half(k_new[r, j, h], np.asarray(cos_sin[pos], np.float64))
                k = rms_norm(k, np.asarray(norm_w, np.float64), eps)
                if H is not None:
                    k = H @ k
                v = v_new[r, j, h].copy()
                if kv_dtype == "e4m3":
                    k = k / float(k_scale[h])
                    v = v / float(v_scale[h])
                out[(page, h, slot)] = (k, v)
    return out
