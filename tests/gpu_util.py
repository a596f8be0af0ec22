"""Helpers shared by the GPU tests: run the CUDA path on a synthetic
workload and compare its results with the oracle's."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
from synth.device import empty_pool, upload

# Tolerances (stated by the benchmark spec for bf16 inputs with fp32 accumulation, and
# for the fp32 path); LSE tolerances derived from fp32 accumulation.
BF16_MAX_ABS, BF16_REL_L2, BF16_LSE_ABS = 2e-2, 5e-3, 1e-3
FP32_MAX_ABS, FP32_REL_L2, FP32_LSE_ABS = 1e-5, 1e-5, 1e-5


def tolerances(dtype: str):
    return (BF16_MAX_ABS, BF16_REL_L2, BF16_LSE_ABS) if dtype == "bf16" else (FP32_MAX_ABS, FP32_REL_L2, FP32_LSE_ABS)


def mla_pkg():
    import head_latent_attention_27_b300 as m
    return m


def append_flags(mla, w) -> int:
    return (mla.MLA_APPEND_RMSNORM if w.rmsnorm else 0) | mla.MLA_APPEND_ROPE


def build_cache(w, device="cuda", rope=None):
    """Upload the raw rows and append them all through mla_cache_append
    (mla_cache_append_rope when RoPE parameters are given)."""
    mla = mla_pkg()
    d = upload(w, device)
    pool = empty_pool(w, device, fill_nan=True)
    cache = mla.Cache(pool, d["page_table"], w.d_c, w.d_r)
    if rope is None:
        mla.mla_cache_append(cache, d["raw_c"], d["raw_k"], d["seq_ids"], d["positions"], eps=w.eps,
                             rope_base=w.rope_base, flags=append_flags(mla, w))
    else:
        mla.mla_cache_append_rope(cache, d["raw_c"], d["raw_k"], d["seq_ids"], d["positions"], rope, eps=w.eps,
                                  flags=append_flags(mla, w))
    del d["raw_c"], d["raw_k"]
    return cache, d


def run_decode(w, cache, d, n_split=None, phases=False, scale=None):
    """(out float64 [B,Q,H,d_c], lse float64 [B,Q,H]) from the CUDA path."""
    mla = mla_pkg()
    dt = cache.data.dtype
    out = torch.empty((w.B, w.Q, w.H, w.d_c), dtype=dt, device=cache.data.device)
    lse = torch.empty((w.B, w.Q, w.H), dtype=torch.float32, device=cache.data.device)
    scale = 1.0 / math.sqrt(w.d_h + w.d_r) if scale is None else scale
    ws = mla.alloc_workspace(w.B, w.Q, w.H, w.d_c, n_split or 0, cache.data.device)
    if phases:
        ns = n_split or 0
        mla.mla_decode_plan(cache, d["seq_lens"], w.Q, w.H, ws, n_split=ns)
        mla.mla_decode_attend(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, ws, lse=lse, n_split=ns,
                              softmax_scale=scale)
        mla.mla_decode_combine(cache, out, ws, lse=lse, n_split=ns)
    elif n_split:
        mla.mla_decode_split_combine(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, n_split, lse=lse,
                                     workspace=ws, softmax_scale=scale)
    else:
        mla.mla_decode(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, lse=lse, workspace=ws,
                       softmax_scale=scale)
    status = mla.mla_decode_read_status(ws)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def compare(w, out, lse, seqs=None, theta=None, scale=None, ref=None):
    """Element-wise comparison with the oracle on the listed sequences
    (`theta`, `scale`: RoPE frequencies and softmax scale other than the
    workload's plain ones; `ref`: the oracle's (out, lse) of those sequences
    when already computed).

    Returns a dict of max-abs / rel-L2 errors and asserts the tolerances."""
    seqs = list(range(w.B) if seqs is None else seqs)
    if ref is None:
        ref_o, ref_l = [], []
        for b in seqs:
            cache = None if theta is None else O.sequence_cache(w, int(b), theta=theta)
            o, l = O.decode_sequence(w, int(b), cache=cache, scale=scale)
            ref_o.append(o)
            ref_l.append(l)
        ref_o, ref_l = np.stack(ref_o), np.stack(ref_l)
    else:
        ref_o, ref_l = ref
    got_o = np.stack([out[b] for b in seqs])
    got_l = np.stack([lse[b] for b in seqs])
    max_abs_t, rel_t, lse_t = tolerances(w.dtype)
    assert np.all(np.isfinite(got_o)), "non-finite output"
    err = np.abs(got_o - ref_o)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.sqrt(np.sum(ref_o ** 2)))
    rel_l2 = float(np.sqrt(np.sum(err ** 2)) / denom) if denom > 0 else float(np.sqrt(np.sum(err ** 2)))
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(got_l)), "lse -inf pattern differs"
    assert np.all(got_l[~fin] == -np.inf)
    lse_err = float(np.abs(got_l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    res = dict(max_abs=max_abs, rel_l2=rel_l2, lse_abs=lse_err)
    assert max_abs <= max_abs_t and rel_l2 <= rel_t and lse_err <= lse_t, res
    return res
