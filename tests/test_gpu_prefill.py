"""Expanded (prefill) attention through the C ABI against the fp64 oracle's
prefill_expanded: per-head K and V materialised from the cached latent
through W^UK / W^UV, the shared RoPE key concatenated, causal softmax
("02 · DeepSeek-V2 analysis", sections 1.2-1.3 and 6)."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import BF16_MAX_ABS, BF16_REL_L2, build_cache, mla_pkg
from synth.device import to_torch

pytestmark = pytest.mark.gpu


def _run_gpu(w):
    mla = mla_pkg()
    cache, _ = build_cache(w)
    T, H = int(w.lens[0]), w.H
    inp = synth.prefill_inputs(w)
    t = {k: to_torch(v, "bf16") for k, v in inp.items()}
    out = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(mla.mla_prefill_workspace_size(T, H), dtype=torch.uint8, device="cuda")
    mla.mla_prefill_expanded(cache, 0, T, t["w_uk"], t["w_uv"], t["q_c"], t["q_r"], out, lse=lse, workspace=ws)
    status = mla.mla_decode_read_status(ws)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), inp


def _compare(w, inp, out, lse, heads=None, rows=None):
    T, H = int(w.lens[0]), w.H
    heads = np.arange(H) if heads is None else np.asarray(heads)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    C, R = O.sequence_cache(w, 0)
    f = O.bf16_bits_to_f64
    ref_o, ref_l = O.prefill_expanded(C, R, f(inp["q_c"])[rows][:, heads], f(inp["q_r"])[rows][:, heads],
                                      f(inp["w_uk"])[heads], f(inp["w_uv"])[heads], positions=rows)
    got_o = out[rows][:, heads]
    got_l = lse[rows][:, heads]
    assert np.all(np.isfinite(got_o)) and np.all(np.isfinite(got_l))
    err = np.abs(got_o - ref_o)
    rel = float(np.sqrt(np.sum(err ** 2) / np.sum(ref_o ** 2)))
    # lse: the expanded form stores the materialised keys K^C in bf16 (each
    # element within 2^-9 of its value), which moves query t's score with key
    # s by at most scale * 2^-9 * sum_d |q_td K_sd|; the log-sum-exp moves by
    # at most the largest such shift over the visible keys, plus fp32
    # accumulation (1e-4).  The decode path has no such rounding step, hence
    # its tighter 1e-3.
    K = np.einsum("sc,hdc->shd", C, f(inp["w_uk"])[heads])                   # [S, heads, d_h]
    qc = np.abs(f(inp["q_c"])[rows][:, heads])                                # [rows, heads, d_h]
    shift = np.einsum("thd,shd->ths", qc, np.abs(K))                          # [rows, heads, S]
    visible = np.arange(T)[None, :] <= np.asarray(rows)[:, None]
    shift = np.where(visible[:, None, :], shift, 0.0).max(axis=2)
    lse_tol = 2.0 ** -9 * (1.0 / np.sqrt(128 + w.d_r)) * shift + 1e-4
    lse_err = np.abs(got_l - ref_l)
    res = dict(max_abs=float(err.max()), rel_l2=rel, lse_abs=float(lse_err.max()),
               lse_margin=float((lse_err / lse_tol).max()))
    assert res["max_abs"] <= BF16_MAX_ABS and rel <= BF16_REL_L2 and np.all(lse_err <= lse_tol), res
    return res


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 128, 129, 300, 777])
def test_prefill_small_two_heads(T):
    w = synth.prefill(T=T, H=2, seed=1100 + T)
    out, lse, inp = _run_gpu(w)
    _compare(w, inp, out, lse)


def test_prefill_paged_sixteen_heads():
    w = synth.prefill(T=1000, H=16, seed=1201, paged=True)
    out, lse, inp = _run_gpu(w)
    _compare(w, inp, out, lse)


@pytest.mark.parametrize("H", [6, 12])
def test_prefill_head_counts_that_change_the_work_order(H):
    """Work items go head group by head group (8 heads when H allows, else
    4 or 2; the projection needs an even H), and the two softmax warpgroups
    take alternate key tiles, so these head counts change which group owns
    which tile and which item finishes where."""
    w = synth.prefill(T=300, H=H, seed=1250 + H)
    out, lse, inp = _run_gpu(w)
    _compare(w, inp, out, lse)


def test_prefill_full_size_sampled_heads_and_rows():
    """T = 4096, H = 128 (the full-width decode's per-sequence shape); the
    oracle checks 5 heads (first, last, either side of the middle) at query
    rows spanning the first, last and tile-boundary positions."""
    w = synth.prefill(T=4096, H=128)
    out, lse, inp = _run_gpu(w)
    rows = [0, 1, 2, 63, 64, 127, 128, 129, 1000, 2047, 2048, 3071, 4094, 4095]
    _compare(w, inp, out, lse, heads=[0, 1, 63, 64, 127], rows=rows)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_prefill_row_zero_is_its_own_value():
    """Query 0 sees only key 0, so its output is V[0] = W^UV c_0 (rounded to
    bf16 once when materialised, once more on output) and its lse is its
    single scaled score."""
    w = synth.prefill(T=130, H=4, seed=1300)
    out, lse, inp = _run_gpu(w)
    C, _ = O.sequence_cache(w, 0)
    v0 = np.einsum("hdc,c->hd", O.bf16_bits_to_f64(inp["w_uv"]), C[0])
    assert np.abs(out[0] - v0).max() <= 2 * 2.0 ** -8 * np.abs(v0).max()
