"""Seeded synthetic inputs shared by the fp64 oracle and the CUDA path.

This package draws raw numbers only.  It contains none of the attention
arithmetic (no normalisation, rotation, scores or softmax): the raw latent
rows ``c_kv_raw``, raw RoPE-key rows ``k_R_raw``, absorbed queries ``q_nope``
and ``q_rope``, per-sequence lengths and the page permutation.  Both sides
receive identical bits.  bfloat16 tensors are returned as ``uint16`` bit
patterns, fp32 tensors as ``float32``.

Every tensor of a workload is its own counter-based stream (SplitMix64, see
``gen.c``), so any subset of rows (one sequence, one token) can be drawn on
its own and equals the same rows of the full draw.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libsynth.so")

# Stream ids: one per drawn tensor.
STREAM_C_KV = 1
STREAM_K_R = 2
STREAM_Q_NOPE = 3
STREAM_Q_ROPE = 4
STREAM_LENS = 5
STREAM_PAGES = 6
STREAM_EXTRA = 16  # first id free for test-only draws (weights etc.)


def build(force: bool = False) -> str:
    """Compile gen.c into libsynth.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_stream_key.restype = u64
        lib.synth_stream_key.argtypes = [u64, u64]
        lib.synth_draw_u64.restype = u64
        lib.synth_draw_u64.argtypes = [u64, u64, u64]
        for name in ("synth_normal_f64", "synth_normal_f32", "synth_normal_bf16"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [u64, u64, u64, i64, f64, vp]
        lib.synth_normal_rows_bf16.restype = None
        lib.synth_normal_rows_bf16.argtypes = [u64, u64, vp, i64, i64, f64, vp]
        lib.synth_uniform_int.restype = None
        lib.synth_uniform_int.argtypes = [u64, u64, u64, i64, i64, i64, vp]
        lib.synth_permutation.restype = None
        lib.synth_permutation.argtypes = [u64, u64, i64, vp]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def draw_u64(seed: int, stream: int, i: int) -> int:
    return int(_L().synth_draw_u64(seed, stream, i))


def normal(seed: int, stream: int, n: int, scale: float = 1.0, offset: int = 0,
           dtype: str = "f64") -> np.ndarray:
    """n draws of scale * N(0, 1); dtype 'f64', 'f32' or 'bf16' (uint16 bits)."""
    npdt = {"f64": np.float64, "f32": np.float32, "bf16": np.uint16}[dtype]
    out = np.empty(int(n), dtype=npdt)
    fn = {"f64": _L().synth_normal_f64, "f32": _L().synth_normal_f32,
          "bf16": _L().synth_normal_bf16}[dtype]
    fn(seed, stream, offset, int(n), float(scale), _ptr(out))
    return out


def normal_rows_bf16(seed: int, stream: int, row_index: np.ndarray, width: int,
                     scale: float) -> np.ndarray:
    rows = np.ascontiguousarray(row_index, dtype=np.int64)
    out = np.empty((rows.size, width), dtype=np.uint16)
    _L().synth_normal_rows_bf16(seed, stream, _ptr(rows), rows.size, width, float(scale), _ptr(out))
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.int32)
    _L().synth_uniform_int(seed, stream, offset, int(n), lo, hi, _ptr(out))
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(int(n), dtype=np.int32)
    _L().synth_permutation(seed, stream, int(n), _ptr(out))
    return out


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    """One decode workload: shapes, seeds and the recipe of every raw tensor.

    Sequence b holds ``lens[b]`` cached tokens at positions 0..lens[b]-1; the
    last ``Q`` of them are the query tokens of this decode step.  Raw token
    rows are numbered globally (sequence by sequence), so token s of sequence
    b is raw row ``row_offset[b] + s``.
    """
    name: str
    seed: int
    B: int
    Q: int
    H: int
    d_c: int
    d_r: int
    d_h: int
    dtype: str                 # cache/query dtype: "bf16" or "fp32"
    lens: np.ndarray           # int32 [B]
    paged: bool                # pages placed by a random permutation
    rmsnorm: bool              # c_kv goes through RMSNorm before caching
    rope_base: float = 10000.0
    eps: float = 1e-6
    page_size: int = 64
    std_c: float = 1.0
    std_k: float = 1.0
    std_qn: float = 1.0
    std_qr: float = 1.0
    q_gain: float = 1.0        # extra factor on both query parts
    n_splits: tuple = ()
    row_offset: np.ndarray = field(init=False)
    pages_per_seq: np.ndarray = field(init=False)
    page_offset: np.ndarray = field(init=False)

    def __post_init__(self):
        self.lens = np.asarray(self.lens, dtype=np.int32)
        assert self.lens.shape == (self.B,)
        self.row_offset = np.concatenate([[0], np.cumsum(self.lens, dtype=np.int64)])[:-1]
        self.pages_per_seq = (self.lens.astype(np.int64) + self.page_size - 1) // self.page_size
        self.page_offset = np.concatenate([[0], np.cumsum(self.pages_per_seq)])[:-1]

    # sizes -----------------------------------------------------------------
    @property
    def total_tokens(self) -> int:
        return int(self.lens.sum())

    @property
    def num_pages(self) -> int:
        return int(self.pages_per_seq.sum())

    @property
    def max_pages_per_seq(self) -> int:
        return max(1, int(self.pages_per_seq.max()))

    @property
    def raw_dtype(self) -> str:
        return "bf16" if self.dtype == "bf16" else "f32"

    # page table ------------------------------------------------------------
    def page_table(self) -> np.ndarray:
        """int32 [B, max_pages_per_seq]; unused entries are 0."""
        pt = np.zeros((self.B, self.max_pages_per_seq), dtype=np.int32)
        ids = np.arange(self.num_pages, dtype=np.int32)
        if self.paged:
            ids = permutation(self.seed, STREAM_PAGES, self.num_pages)
        for b in range(self.B):
            n = int(self.pages_per_seq[b])
            o = int(self.page_offset[b])
            pt[b, :n] = ids[o:o + n]
        return pt

    # raw rows --------------------------------------------------------------
    def raw_rows(self, b: int, s0: int = 0, s1: int | None = None):
        """Raw (c_kv, k_R) rows of tokens s0..s1-1 of sequence b."""
        s1 = int(self.lens[b]) if s1 is None else s1
        g0 = int(self.row_offset[b]) + s0
        n = s1 - s0
        c = normal(self.seed, STREAM_C_KV, n * self.d_c, self.std_c, g0 * self.d_c, self.raw_dtype)
        k = normal(self.seed, STREAM_K_R, n * self.d_r, self.std_k, g0 * self.d_r, self.raw_dtype)
        return c.reshape(n, self.d_c), k.reshape(n, self.d_r)

    def all_raw_rows(self):
        """Raw rows of every cached token, in global row order."""
        n = self.total_tokens
        c = normal(self.seed, STREAM_C_KV, n * self.d_c, self.std_c, 0, self.raw_dtype)
        k = normal(self.seed, STREAM_K_R, n * self.d_r, self.std_k, 0, self.raw_dtype)
        return c.reshape(n, self.d_c), k.reshape(n, self.d_r)

    def token_seq_pos(self):
        """(seq_id, position) int32 arrays for every global raw row."""
        seq = np.repeat(np.arange(self.B, dtype=np.int32), self.lens)
        pos = (np.arange(self.total_tokens, dtype=np.int64) - np.repeat(self.row_offset, self.lens)).astype(np.int32)
        return seq, pos

    def queries(self):
        """(q_nope [B,Q,H,d_c], q_rope [B,Q,H,d_r]) in the workload dtype."""
        nq = self.B * self.Q * self.H
        qn = normal(self.seed, STREAM_Q_NOPE, nq * self.d_c, self.std_qn * self.q_gain, 0, self.raw_dtype)
        qr = normal(self.seed, STREAM_Q_ROPE, nq * self.d_r, self.std_qr * self.q_gain, 0, self.raw_dtype)
        return (qn.reshape(self.B, self.Q, self.H, self.d_c),
                qr.reshape(self.B, self.Q, self.H, self.d_r))

    def queries_of(self, b: int):
        nq = self.Q * self.H
        o = b * nq
        qn = normal(self.seed, STREAM_Q_NOPE, nq * self.d_c, self.std_qn * self.q_gain, o * self.d_c, self.raw_dtype)
        qr = normal(self.seed, STREAM_Q_ROPE, nq * self.d_r, self.std_qr * self.q_gain, o * self.d_r, self.raw_dtype)
        return qn.reshape(self.Q, self.H, self.d_c), qr.reshape(self.Q, self.H, self.d_r)


def _std(dim: int) -> float:
    return 1.0 / float(np.sqrt(dim))


def tiny_fp32(seed: int = 1001) -> Workload:
    """B=2, S=64, H=8, d_c=64, d_r=16, d_h=32, fp32, contiguous, no RMSNorm."""
    return Workload("tiny_fp32_B2_S64_H8_dc64", seed, B=2, Q=1, H=8, d_c=64, d_r=16, d_h=32,
                    dtype="fp32", lens=[64, 64], paged=False, rmsnorm=False,
                    std_c=_std(64), std_k=_std(16), std_qn=_std(64), std_qr=_std(16))


def _bf16(name, seed, B, S_or_lens, H, Q=1, paged=False, n_splits=(), q_gain=1.0) -> Workload:
    lens = S_or_lens if isinstance(S_or_lens, np.ndarray) else np.full(B, S_or_lens, np.int32)
    s = _std(576)
    return Workload(name, seed, B=B, Q=Q, H=H, d_c=512, d_r=64, d_h=128, dtype="bf16", lens=lens,
                    paged=paged, rmsnorm=True, std_c=s, std_k=s, std_qn=s, std_qr=s,
                    n_splits=n_splits, q_gain=q_gain)


def small_head(seed: int = 1002) -> Workload:
    """B=32, S=4096, H=16, bf16, contiguous (HBM-bound)."""
    return _bf16("small_head_B32_S4096_H16", seed, 32, 4096, 16)


def full_width(seed: int = 1003) -> Workload:
    """B=64, S=4096, H=128, bf16, contiguous, one query token per sequence."""
    return _bf16("full_width_B64_S4096_H128", seed, 64, 4096, 128)


def ragged_paged(seed: int = 1004, B: int = 128, max_len: int = 32768) -> Workload:
    """B=128, lengths U{1..32768}, 64-token pages by random permutation, H=128, Q=2 causal."""
    lens = uniform_int(seed, STREAM_LENS, B, 1, max_len)
    return _bf16(f"ragged_paged_B{B}_Lmax{max_len}_H128_Q2", seed, B, lens, 128, Q=2, paged=True)


def long_split(seed: int = 1005, S: int = 131072, B: int = 4) -> Workload:
    """B=4, S=131072, H=128, bf16, split-KV into 32..128 chunks."""
    return _bf16(f"long_split_B{B}_S{S}_H128", seed, B, S, 128, n_splits=(32, 64, 128))


def custom_bf16(name: str, seed: int, lens, H: int, Q: int = 1, paged: bool = False,
                q_gain: float = 1.0) -> Workload:
    """Same recipe as the bf16 workloads with arbitrary lengths / heads."""
    lens = np.asarray(lens, dtype=np.int32)
    return _bf16(name, seed, len(lens), lens, H, Q=Q, paged=paged, q_gain=q_gain)


WORKLOADS = {
    "tiny_fp32": tiny_fp32,
    "small_head": small_head,
    "full_width": full_width,
    "ragged_paged": ragged_paged,
    "long_split": long_split,
}


# Prefill (expanded form) draws: the per-head up-projections and the
# queries of T prompt tokens, each its own stream.
STREAM_W_UK = 8
STREAM_W_UV = 9
STREAM_Q_C = 10
STREAM_Q_R = 11


def prefill(T: int = 4096, H: int = 128, seed: int = 1006, paged: bool = False) -> Workload:
    """One sequence of T prompt tokens (bf16, d_c=512, d_r=64, d_h=128):
    raw c_kv ~ N(0,1)/sqrt(576) (RMSNorm'd by the append), raw k_R ~ N(0,1)
    (rotated at positions 0..T-1 by the append)."""
    return Workload(f"prefill_T{T}_H{H}", seed, B=1, Q=1, H=H, d_c=512, d_r=64, d_h=128, dtype="bf16",
                    lens=np.array([T], np.int32), paged=paged, rmsnorm=True, std_c=_std(576), std_k=1.0,
                    std_qn=_std(576), std_qr=_std(576))


def prefill_inputs(w: Workload, heads=None, rows=None) -> dict:
    """bf16 bits of W^UK, W^UV [H, d_h, d_c] ~ N(0,1)/sqrt(d_c) and of the
    queries q_c [T, H, d_h], q_r [T, H, d_r] ~ N(0,1) (`heads` / `rows`:
    draw only those heads of the weights / those query rows)."""
    T, H, dh, dc, dr = int(w.lens[0]), w.H, w.d_h, w.d_c, w.d_r
    heads = np.arange(H) if heads is None else np.asarray(heads)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    wk = np.stack([normal(w.seed, STREAM_W_UK, dh * dc, _std(dc), int(h) * dh * dc, "bf16") for h in heads])
    wv = np.stack([normal(w.seed, STREAM_W_UV, dh * dc, _std(dc), int(h) * dh * dc, "bf16") for h in heads])
    qc_idx = (rows[:, None] * H + heads[None, :]).reshape(-1)
    qc = normal_rows_bf16(w.seed, STREAM_Q_C, qc_idx, dh, 1.0).reshape(len(rows), len(heads), dh)
    qr = normal_rows_bf16(w.seed, STREAM_Q_R, qc_idx, dr, 1.0).reshape(len(rows), len(heads), dr)
    return {"w_uk": wk.reshape(len(heads), dh, dc), "w_uv": wv.reshape(len(heads), dh, dc), "q_c": qc, "q_r": qr}
