"""Place a synthetic workload's raw draws in device memory (torch tensors).

Plumbing only: reinterprets the generator's bf16 bit patterns as
torch.bfloat16 and copies arrays to the GPU.  No attention arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch


def to_torch(a: np.ndarray, dtype: str, device="cuda", pin: bool = False) -> torch.Tensor:
    """uint16 bf16 bits -> torch.bfloat16, float32 -> torch.float32."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if pin:
        t = t.pin_memory()
    return t.to(device) if device is not None else t


def empty_pool(w, device="cuda", fill_nan: bool = True) -> torch.Tensor:
    """Cache pool [num_pages, 64, d_c + d_r]; unwritten slots hold NaN."""
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pool = torch.empty((w.num_pages, w.page_size, w.d_c + w.d_r), dtype=dt, device=device)
    if fill_nan:
        pool.fill_(float("nan"))
    return pool


def upload(w, device="cuda", raw: bool = True) -> dict:
    """Device tensors of a workload: page table, lengths, queries, raw rows."""
    d = {
        "page_table": torch.from_numpy(w.page_table()).to(device),
        "seq_lens": torch.from_numpy(w.lens.astype(np.int32)).to(device),
    }
    qn, qr = w.queries()
    d["q_nope"] = to_torch(qn, w.raw_dtype if w.dtype == "bf16" else "f32", device)
    d["q_rope"] = to_torch(qr, w.raw_dtype if w.dtype == "bf16" else "f32", device)
    if raw:
        c, k = w.all_raw_rows()
        seq, pos = w.token_seq_pos()
        d["raw_c"] = to_torch(c, "bf16" if w.raw_dtype == "bf16" else "f32", device)
        d["raw_k"] = to_torch(k, "bf16" if w.raw_dtype == "bf16" else "f32", device)
        d["seq_ids"] = torch.from_numpy(seq).to(device)
        d["positions"] = torch.from_numpy(pos).to(device)
    return d
