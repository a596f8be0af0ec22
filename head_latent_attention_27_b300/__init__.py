"""Python binding of libmla.so: absorbed MLA decode for B300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libmla.so.  PyTorch is used for device memory and streams; the
functions take torch tensors, pass their device pointers and the current
CUDA stream to the C ABI (include/mla.h) and raise RuntimeError when a call
returns a non-OK status.  There is no fallback: importing the package fails
if libmla.so has not been built (python head_latent_attention_27_b300/build.py).
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python head_latent_attention_27_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_TIMEOUT, MLA_ERR_WORKSPACE = range(6)
MLA_BF16, MLA_FP32, MLA_FP8 = 0, 1, 2
FP8_ROW_BYTES = 656   # low-precision row: 512 E4M3 codes, 4 fp32 group scales, 64 bf16 RoPE values
MLA_APPEND_RMSNORM = 1
MLA_APPEND_ROPE = 2
PAGE_SIZE = 64


class mla_cache_t(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("d_c", ctypes.c_int32),
        ("d_r", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
    ]


class mla_rope_t(ctypes.Structure):
    """RoPE parameters; yarn_factor > 1 applies YaRN's frequency interpolation."""
    _fields_ = [
        ("base", ctypes.c_float),
        ("yarn_factor", ctypes.c_float),
        ("yarn_alpha", ctypes.c_float),
        ("yarn_beta", ctypes.c_float),
        ("original_max_position", ctypes.c_int32),
    ]


_vp, _i32, _u32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
_pc = ctypes.POINTER(mla_cache_t)

_SIGS = {
    "mla_cache_append": (_i32, [_pc, _vp, _vp, _i32, _vp, _f32, _f32, _vp, _vp, _i32, _u32, _vp]),
    "mla_cache_append_rope": (_i32, [_pc, _vp, _vp, _i32, _vp, _f32, ctypes.POINTER(mla_rope_t), _vp, _vp, _i32, _u32,
                                     _vp]),
    "mla_yarn_softmax_scale": (_f32, [_f32, _f32, _f32]),
    "mla_decode": (_i32, [_pc, _vp, _i32, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "mla_decode_split_combine": (_i32, [_pc, _vp, _i32, _vp, _vp, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "mla_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "mla_decode_plan": (_i32, [_pc, _vp, _i32, _i32, _i32, _i32, _vp, _sz, _vp]),
    "mla_decode_attend": (_i32, [_pc, _vp, _i32, _vp, _vp, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "mla_decode_combine": (_i32, [_pc, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "mla_decode_read_status": (_i32, [_vp, _sz, _vp, ctypes.POINTER(_i32)]),
    "mla_selftest_bounded_wait": (_i32, [_vp, _sz, _u32, _vp]),
    "mla_decode_noalloc": (_i32, [_pc, _vp, _i32, _vp, _vp, _i32, _i32, _f32, _vp, _vp, _vp]),
    "mla_absorb_query": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "mla_absorb_output": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "mla_prefill_workspace_size": (_sz, [_i32, _i32]),
    "mla_prefill_expanded": (_i32, [_pc, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "mla_prefill_project": (_i32, [_pc, _i32, _i32, _vp, _vp, _i32, _vp, _sz, _vp]),
    "mla_prefill_attend": (_i32, [_pc, _i32, _i32, _vp, _vp, _i32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "mla_status_string": (ctypes.c_char_p, [_i32]),
    "mla_version": (_i32, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def mla_status_string(code: int) -> str:
    return _lib.mla_status_string(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != MLA_OK:
        raise RuntimeError(f"{what}: {mla_status_string(code)}")


def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    if t.dtype == torch.float32:
        return MLA_FP32
    if t.dtype == torch.uint8:
        return MLA_FP8
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t, name, dtype=None, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


@dataclass
class Cache:
    """A paged latent cache: data [num_pages, 64, d_c + d_r] and page_table [B, max_pages]
    (a uint8 `data` [num_pages, 64, 656] is the low-precision cache, MLA_FP8)."""
    data: "object"
    page_table: "object"
    d_c: int
    d_r: int

    def __post_init__(self):
        torch = _torch()
        _need(self.data, "cache.data", ndim=3)
        _need(self.page_table, "cache.page_table", torch.int32, 2)
        width = FP8_ROW_BYTES if self.data.dtype == torch.uint8 else self.d_c + self.d_r
        if self.data.shape[1] != PAGE_SIZE or self.data.shape[2] != width:
            raise ValueError(f"cache.data must be [num_pages, 64, {width}]")

    def c(self) -> mla_cache_t:
        return mla_cache_t(self.data.data_ptr(), self.page_table.data_ptr(), _dtype_code(self.data),
                           self.page_table.shape[0], self.data.shape[0], PAGE_SIZE, self.d_c, self.d_r,
                           self.page_table.shape[1])


def mla_cache_append(cache: Cache, ckv_raw, kr_raw, seq_ids, positions, gamma=None, eps: float = 1e-6,
                     rope_base: float = 10000.0, flags: int = MLA_APPEND_RMSNORM | MLA_APPEND_ROPE,
                     stream=None) -> None:
    """Write T tokens: ckv_raw [T, d_c], kr_raw [T, d_r], seq_ids/positions int32 [T]."""
    torch = _torch()
    _need(ckv_raw, "ckv_raw", ndim=2)
    _need(kr_raw, "kr_raw", ckv_raw.dtype, 2)
    _need(seq_ids, "seq_ids", torch.int32, 1)
    _need(positions, "positions", torch.int32, 1)
    T = ckv_raw.shape[0]
    if kr_raw.shape[0] != T or seq_ids.shape[0] != T or positions.shape[0] != T:
        raise ValueError("row counts differ")
    if ckv_raw.shape[1] != cache.d_c or kr_raw.shape[1] != cache.d_r:
        raise ValueError("row widths do not match the cache")
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, 1)
    cc = cache.c()
    _check(_lib.mla_cache_append(ctypes.byref(cc), _ptr(ckv_raw), _ptr(kr_raw), _dtype_code(ckv_raw), _ptr(gamma),
                                 float(eps), float(rope_base), _ptr(seq_ids), _ptr(positions), T, int(flags),
                                 _stream(stream)), "mla_cache_append")


def mla_cache_append_rope(cache: Cache, ckv_raw, kr_raw, seq_ids, positions, rope: "mla_rope_t", gamma=None,
                          eps: float = 1e-6, flags: int = MLA_APPEND_RMSNORM | MLA_APPEND_ROPE, stream=None) -> None:
    """mla_cache_append with explicit RoPE parameters (YaRN when rope.yarn_factor > 1)."""
    torch = _torch()
    _need(ckv_raw, "ckv_raw", ndim=2)
    _need(kr_raw, "kr_raw", ckv_raw.dtype, 2)
    _need(seq_ids, "seq_ids", torch.int32, 1)
    _need(positions, "positions", torch.int32, 1)
    T = ckv_raw.shape[0]
    if kr_raw.shape[0] != T or seq_ids.shape[0] != T or positions.shape[0] != T:
        raise ValueError("row counts differ")
    if ckv_raw.shape[1] != cache.d_c or kr_raw.shape[1] != cache.d_r:
        raise ValueError("row widths do not match the cache")
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, 1)
    cc = cache.c()
    _check(_lib.mla_cache_append_rope(ctypes.byref(cc), _ptr(ckv_raw), _ptr(kr_raw), _dtype_code(ckv_raw),
                                      _ptr(gamma), float(eps), ctypes.byref(rope), _ptr(seq_ids), _ptr(positions), T,
                                      int(flags), _stream(stream)), "mla_cache_append_rope")


def yarn_rope(base: float = 10000.0, factor: float = 40.0, alpha: float = 1.0, beta: float = 32.0,
              original_max_position: int = 4096) -> "mla_rope_t":
    """RoPE parameters of a YaRN-extended context (defaults: DeepSeek-V2's s=40, alpha=1, beta=32, 4K window)."""
    return mla_rope_t(base, factor, alpha, beta, original_max_position)


def mla_yarn_softmax_scale(softmax_scale: float, yarn_factor: float, coef: float = 0.0707) -> float:
    """softmax_scale * (coef * ln(s) + 1)^2: YaRN's attention temperature on the softmax scale."""
    return float(_lib.mla_yarn_softmax_scale(float(softmax_scale), float(yarn_factor), float(coef)))


def mla_decode_workspace_size(B: int, Q: int, H: int, d_c: int = 512, n_split: int = 0, num_sms: int = 0) -> int:
    n = _lib.mla_decode_workspace_size(B, Q, H, d_c, n_split, num_sms)
    if n == 0:
        raise RuntimeError("mla_decode_workspace_size: invalid arguments")
    return int(n)


def alloc_workspace(B: int, Q: int, H: int, d_c: int = 512, n_split: int = 0, device=None):
    """A uint8 CUDA tensor large enough for a decode of this shape (256-byte aligned)."""
    torch = _torch()
    n = mla_decode_workspace_size(B, Q, H, d_c, n_split)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def _decode_args(cache: Cache, seq_lens, q_nope, q_rope, out, lse):
    torch = _torch()
    _need(seq_lens, "seq_lens", torch.int32, 1)
    qdt = torch.bfloat16 if cache.data.dtype == torch.uint8 else cache.data.dtype   # low-precision cache: bf16 q/out
    _need(q_nope, "q_nope", qdt, 4)
    _need(q_rope, "q_rope", qdt, 4)
    _need(out, "out", qdt, 4)
    B, Q, H, dc = q_nope.shape
    if dc != cache.d_c or tuple(q_rope.shape) != (B, Q, H, cache.d_r) or tuple(out.shape) != (B, Q, H, cache.d_c):
        raise ValueError("q_nope/q_rope/out shapes do not match")
    if seq_lens.shape[0] != B:
        raise ValueError("seq_lens must have B entries")
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
        if tuple(lse.shape) != (B, Q, H):
            raise ValueError("lse must be [B, Q, H]")
    return B, Q, H


def mla_decode(cache: Cache, seq_lens, q_nope, q_rope, out, lse=None, workspace=None,
               softmax_scale: float | None = None, d_h: int = 128, stream=None) -> None:
    """out[b,j,h] = softmax(scale (q_nope.c + q_rope.k_R)) . c over the visible history."""
    B, Q, H = _decode_args(cache, seq_lens, q_nope, q_rope, out, lse)
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d_h + cache.d_r)
    if workspace is None:
        workspace = alloc_workspace(B, Q, H, cache.d_c, 0, out.device)
    cc = cache.c()
    _check(_lib.mla_decode(ctypes.byref(cc), _ptr(seq_lens), B, _ptr(q_nope), _ptr(q_rope), Q, H, float(scale),
                           _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)), "mla_decode")


def mla_decode_split_combine(cache: Cache, seq_lens, q_nope, q_rope, out, n_split: int, lse=None, workspace=None,
                             softmax_scale: float | None = None, d_h: int = 128, stream=None) -> None:
    """mla_decode with every sequence cut into n_split chunks, merged by log-sum-exp."""
    B, Q, H = _decode_args(cache, seq_lens, q_nope, q_rope, out, lse)
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d_h + cache.d_r)
    if workspace is None:
        workspace = alloc_workspace(B, Q, H, cache.d_c, n_split, out.device)
    cc = cache.c()
    _check(_lib.mla_decode_split_combine(ctypes.byref(cc), _ptr(seq_lens), B, _ptr(q_nope), _ptr(q_rope), Q, H,
                                         float(scale), int(n_split), _ptr(out), _ptr(lse), _ptr(workspace),
                                         workspace.numel(), _stream(stream)), "mla_decode_split_combine")


def mla_decode_plan(cache: Cache, seq_lens, Q: int, H: int, workspace, n_split: int = 0, stream=None) -> None:
    torch = _torch()
    _need(seq_lens, "seq_lens", torch.int32, 1)
    cc = cache.c()
    _check(_lib.mla_decode_plan(ctypes.byref(cc), _ptr(seq_lens), seq_lens.shape[0], Q, H, int(n_split),
                                _ptr(workspace), workspace.numel(), _stream(stream)), "mla_decode_plan")


def mla_decode_attend(cache: Cache, seq_lens, q_nope, q_rope, out, workspace, lse=None, n_split: int = 0,
                      softmax_scale: float | None = None, d_h: int = 128, stream=None) -> None:
    B, Q, H = _decode_args(cache, seq_lens, q_nope, q_rope, out, lse)
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d_h + cache.d_r)
    cc = cache.c()
    _check(_lib.mla_decode_attend(ctypes.byref(cc), _ptr(seq_lens), B, _ptr(q_nope), _ptr(q_rope), Q, H,
                                  float(scale), int(n_split), _ptr(out), _ptr(lse), _ptr(workspace),
                                  workspace.numel(), _stream(stream)), "mla_decode_attend")


def mla_decode_combine(cache: Cache, out, workspace, lse=None, n_split: int = 0, stream=None) -> None:
    B, Q, H, _ = out.shape
    cc = cache.c()
    _check(_lib.mla_decode_combine(ctypes.byref(cc), B, Q, H, int(n_split), _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel(), _stream(stream)), "mla_decode_combine")


def mla_decode_noalloc(cache: Cache, seq_lens, q_nope, q_rope, out, lse=None,
                       softmax_scale: float | None = None, d_h: int = 128, stream=None) -> None:
    """mla_decode without a workspace: the library's fixed scratch array is used
    (for callers that cannot allocate device memory; calls must not overlap)."""
    B, Q, H = _decode_args(cache, seq_lens, q_nope, q_rope, out, lse)
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d_h + cache.d_r)
    cc = cache.c()
    _check(_lib.mla_decode_noalloc(ctypes.byref(cc), _ptr(seq_lens), B, _ptr(q_nope), _ptr(q_rope), Q, H,
                                   float(scale), _ptr(out), _ptr(lse), _stream(stream)), "mla_decode_noalloc")


def _absorb_args(w, x, y, d_in: int, d_out: int):
    torch = _torch()
    for t, name in ((w, "weights"), (x, "input"), (y, "output")):
        _need(t, name, torch.bfloat16, 3)
    H, d_h, d_c = w.shape
    n = x.shape[0]
    if tuple(x.shape) != (n, H, (d_h, d_c)[d_in]) or tuple(y.shape) != (n, H, (d_h, d_c)[d_out]):
        raise ValueError("shapes do not match the weights [H, d_h, d_c]")
    return n, H, d_h, d_c


def mla_absorb_query(w_uk, q_c, q_nope, status=None, stream=None) -> None:
    """q_nope[n, h, :] = W^UK[h]^T q_c[n, h, :]  (w_uk [H, d_h, d_c], q_c [n, H, d_h])."""
    n, H, d_h, d_c = _absorb_args(w_uk, q_c, q_nope, 0, 1)
    _check(_lib.mla_absorb_query(_ptr(w_uk), _ptr(q_c), _ptr(q_nope), n, H, d_h, d_c, _ptr(status),
                                 _stream(stream)), "mla_absorb_query")


def mla_absorb_output(w_uv, u, o, status=None, stream=None) -> None:
    """o[n, h, :] = W^UV[h] u[n, h, :]  (w_uv [H, d_h, d_c], u [n, H, d_c])."""
    n, H, d_h, d_c = _absorb_args(w_uv, u, o, 1, 0)
    _check(_lib.mla_absorb_output(_ptr(w_uv), _ptr(u), _ptr(o), n, H, d_h, d_c, _ptr(status), _stream(stream)),
           "mla_absorb_output")


def mla_prefill_workspace_size(T: int, H: int) -> int:
    n = _lib.mla_prefill_workspace_size(int(T), int(H))
    if n == 0:
        raise RuntimeError("mla_prefill_workspace_size: invalid arguments")
    return int(n)


def mla_prefill_expanded(cache: Cache, seq: int, T: int, w_uk, w_uv, q_c, q_r, out, lse=None, workspace=None,
                         softmax_scale: float | None = None, stream=None) -> None:
    """Causal attention of the first T tokens of sequence `seq` in the expanded
    form: K^C = W^UK c and V = W^UV c materialised per head, keys
    [K^C || k^R], queries [q_c || q_r] (w_uk / w_uv [H, 128, 512],
    q_c [T, H, 128], q_r [T, H, 64], out [T, H, 128], lse [T, H])."""
    torch = _torch()
    for t, name in ((w_uk, "w_uk"), (w_uv, "w_uv"), (q_c, "q_c"), (q_r, "q_r"), (out, "out")):
        _need(t, name, torch.bfloat16, 3)
    H = w_uk.shape[0]
    if (tuple(w_uk.shape) != (H, 128, cache.d_c) or tuple(w_uv.shape) != (H, 128, cache.d_c) or
            tuple(q_c.shape) != (T, H, 128) or tuple(q_r.shape) != (T, H, cache.d_r) or
            tuple(out.shape) != (T, H, 128)):
        raise ValueError("prefill shapes do not match")
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
        if tuple(lse.shape) != (T, H):
            raise ValueError("lse must be [T, H]")
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(128 + cache.d_r)
    if workspace is None:
        workspace = torch.empty(mla_prefill_workspace_size(T, H), dtype=torch.uint8, device=out.device)
    cc = cache.c()
    _check(_lib.mla_prefill_expanded(ctypes.byref(cc), int(seq), int(T), _ptr(w_uk), _ptr(w_uv), _ptr(q_c),
                                     _ptr(q_r), H, float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "mla_prefill_expanded")


def mla_prefill_project(cache: Cache, seq: int, T: int, w_uk, w_uv, workspace, stream=None) -> None:
    """First phase of mla_prefill_expanded: K^C and V into the workspace."""
    H = w_uk.shape[0]
    cc = cache.c()
    _check(_lib.mla_prefill_project(ctypes.byref(cc), int(seq), int(T), _ptr(w_uk), _ptr(w_uv), H, _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "mla_prefill_project")


def mla_prefill_attend(cache: Cache, seq: int, T: int, q_c, q_r, out, workspace, lse=None,
                       softmax_scale: float | None = None, stream=None) -> None:
    """Second phase of mla_prefill_expanded: causal attention over the projected K^C, V."""
    H = q_c.shape[1]
    scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(128 + cache.d_r)
    cc = cache.c()
    _check(_lib.mla_prefill_attend(ctypes.byref(cc), int(seq), int(T), _ptr(q_c), _ptr(q_r), H, float(scale),
                                   _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)),
           "mla_prefill_attend")


def mla_decode_read_status(workspace, stream=None) -> int:
    """Synchronise the stream; return and clear the status the kernels recorded."""
    code = ctypes.c_int32(0)
    _lib.mla_decode_read_status(_ptr(workspace), workspace.numel(), _stream(stream), ctypes.byref(code))
    return int(code.value)


def mla_selftest_bounded_wait(workspace, timeout_us: int = 20000, stream=None) -> None:
    _check(_lib.mla_selftest_bounded_wait(_ptr(workspace), workspace.numel(), int(timeout_us), _stream(stream)),
           "mla_selftest_bounded_wait")


def mla_version() -> int:
    return int(_lib.mla_version())
