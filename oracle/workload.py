"""Oracle over a seeded synthetic workload (test infrastructure only).

Builds the oracle's own cache from the raw draws (append in float64, one
rounding to the cache dtype) and decodes from it.  Nothing here reads a value
produced by the CUDA path.
"""
from __future__ import annotations

import numpy as np

from .mla_oracle import (APPEND_RMSNORM, APPEND_ROPE, append_rows, bf16_bits_to_f64,
                         decode_row, softmax_scale, visible_length)

__all__ = ["widen", "append_flags", "sequence_cache", "decode_sequence", "decode_workload",
           "workload_scale"]


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Raw draw (bf16 bits or float32) to float64, exactly."""
    return bf16_bits_to_f64(a) if dtype == "bf16" else np.asarray(a, dtype=np.float64)


def append_flags(w) -> int:
    return (APPEND_RMSNORM if w.rmsnorm else 0) | APPEND_ROPE


def workload_scale(w) -> float:
    return softmax_scale(w.d_h, w.d_r)


def sequence_cache(w, b: int, s0: int = 0, s1: int | None = None, theta=None):
    """Oracle cache rows (C [n, d_c], R [n, d_r], float64) of tokens s0..s1-1 of b
    (`theta`: RoPE frequencies other than the plain ones, e.g. YaRN's)."""
    s1 = int(w.lens[b]) if s1 is None else s1
    c_raw, k_raw = w.raw_rows(b, s0, s1)
    rows = append_rows(widen(c_raw, w.raw_dtype), widen(k_raw, w.raw_dtype),
                       np.arange(s0, s1), np.ones(w.d_c), w.eps, w.rope_base,
                       append_flags(w), w.dtype, theta)
    return rows[:, :w.d_c], rows[:, w.d_c:]


def decode_sequence(w, b: int, cache=None, scale=None):
    """(out [Q,H,d_c], lse [Q,H]) of sequence b, float64 (`scale` overrides the
    workload's softmax scale)."""
    C, R = sequence_cache(w, b) if cache is None else cache
    scale = workload_scale(w) if scale is None else scale
    qn, qr = w.queries_of(b)
    qn, qr = widen(qn, w.raw_dtype), widen(qr, w.raw_dtype)
    out = np.zeros((w.Q, w.H, w.d_c))
    lse = np.zeros((w.Q, w.H))
    for j in range(w.Q):
        n = visible_length(int(w.lens[b]), w.Q, j)
        o, l, _ = decode_row(C[:n], R[:n], qn[j], qr[j], scale)
        out[j], lse[j] = o, l
    return out, lse


def decode_workload(w, seqs=None):
    """Oracle results for the listed sequences (default: all)."""
    seqs = range(w.B) if seqs is None else seqs
    res = {}
    for b in seqs:
        res[int(b)] = decode_sequence(w, int(b))
    return res
