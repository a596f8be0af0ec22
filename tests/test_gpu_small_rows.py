"""Parity of the single-SM decode kernel for units of at most 16 query rows
(Q * H <= 16, e.g. 16 heads and one query token) against the oracle.

Every case below is routed to that kernel by the library (bf16 cache,
Q * H <= 16); the larger units of the other GPU tests go to the two-SM
kernel.  Cases cover: padding rows (H < 16), causal rows with Q = 2 (a row
that sees no key), ragged lengths at and around the 32-token stage and
64-token page boundaries, zero-length sequences, random page tables, sharp
softmaxes, forced splits (partial rows merged by the combine), more units
than workers, the three-phase form and the allocation-free entry point.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from gpu_util import build_cache, compare, mla_pkg, run_decode

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 31, 32, 33, 63, 64, 65, 95, 96, 97, 127, 128, 129, 700, 2049]

CASES = [
    # name, lens, H, Q, paged, q_gain
    ("h16_q1_stage_edges", RAGGED, 16, 1, True, 1.0),
    ("h8_q2_causal", [1, 2, 3, 32, 33, 64, 65, 1000], 8, 2, True, 1.0),
    ("h4_q1_padding_rows", [5, 64, 300, 4096], 4, 1, False, 1.0),
    ("h1_q1_one_row", [1, 40, 129, 3000], 1, 1, True, 1.0),
    ("h16_q1_zero_length", [0, 17, 0, 256], 16, 1, True, 1.0),
    ("h16_q1_sharp", [50, 700, 2049, 4096], 16, 1, True, 16.0),
    ("h2_q8_causal", [1, 7, 8, 9, 66, 513], 2, 8, True, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_small_unit_cases(case):
    name, lens, H, Q, paged, q_gain = case
    w = synth.custom_bf16(name, 900 + len(name), lens, H=H, Q=Q, paged=paged, q_gain=q_gain)
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    compare(w, out, lse)


@pytest.mark.parametrize("n_split", [1, 2, 7, 64])
def test_small_unit_forced_splits(n_split):
    w = synth.custom_bf16("h16_split", 931, [1, 33, 640, 1999, 4096], H=16, Q=1, paged=True)
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d, n_split=n_split)
    compare(w, out, lse)


def test_small_unit_more_units_than_workers():
    lens = synth.uniform_int(932, 5, 400, 1, 300)
    w = synth.custom_bf16("h16_many", 932, lens, H=16, Q=1, paged=True)
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    compare(w, out, lse)


def test_small_unit_three_phases_equal_one_call():
    w = synth.custom_bf16("h16_phases", 933, [700, 64, 3001, 1], H=16, Q=1, paged=True)
    cache, d = build_cache(w)
    o1, l1 = run_decode(w, cache, d)
    o3, l3 = run_decode(w, cache, d, phases=True)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)
    compare(w, o1, l1)


def test_small_unit_noalloc_matches_workspace_call():
    mla = mla_pkg()
    w = synth.custom_bf16("h16_noalloc", 934, [129, 4096, 33, 2], H=16, Q=1, paged=True)
    cache, d = build_cache(w)
    o1, l1 = run_decode(w, cache, d)
    out = torch.full((w.B, w.Q, w.H, w.d_c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.Q, w.H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_noalloc(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, lse=lse,
                           softmax_scale=1.0 / np.sqrt(w.d_h + w.d_r))
    torch.cuda.synchronize()
    assert np.array_equal(out.double().cpu().numpy(), o1)
    assert np.array_equal(lse.double().cpu().numpy(), l1)


def test_small_unit_bad_length_is_reported():
    mla = mla_pkg()
    w = synth.custom_bf16("h16_bad_len", 935, [64, 128], H=16, Q=1)
    cache, d = build_cache(w)
    d["seq_lens"][1] = 10 ** 6   # beyond the page table's capacity
    out = torch.empty((2, 1, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 1, 16), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(2, 1, 16)
    mla.mla_decode(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, lse=lse, workspace=ws)
    assert mla.mla_decode_read_status(ws) == mla.MLA_ERR_INVALID_ARG
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))


def test_small_unit_one_plan_serves_several_attention_launches():
    """A caller decoding several layers with the same lengths plans once and
    runs the attention kernel per layer; split units must merge every time."""
    import math
    mla = mla_pkg()
    w = synth.custom_bf16("h16_plan_reuse", 936, [4096, 4096, 700, 64, 3001, 1], H=16, Q=1, paged=True)
    cache, d = build_cache(w)
    scale = 1.0 / math.sqrt(w.d_h + w.d_r)
    ws = mla.alloc_workspace(w.B, w.Q, w.H, w.d_c, 0, "cuda")
    mla.mla_decode_plan(cache, d["seq_lens"], w.Q, w.H, ws)
    outs = []
    for _ in range(3):
        out = torch.full((w.B, w.Q, w.H, w.d_c), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.B, w.Q, w.H), float("nan"), dtype=torch.float32, device="cuda")
        mla.mla_decode_attend(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, ws, lse=lse, softmax_scale=scale)
        mla.mla_decode_combine(cache, out, ws, lse=lse)
        assert mla.mla_decode_read_status(ws) == mla.MLA_OK
        outs.append((out.double().cpu().numpy(), lse.double().cpu().numpy()))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    compare(w, *outs[0])

