"""Absorption GEMMs (q_nope = W^UK_h^T q^C_h, o = W^UV_h u_h) through the C
ABI against the fp64 oracle, element by element.

Bound: the kernel accumulates in fp32 and rounds each output once to bf16,
so |gpu - ref| <= 2^-8 |ref| (one bf16 rounding, half an ulp is 2^-9 of the
value's binade, at most 2^-8 of the value) plus the fp32 accumulation error,
far below 1e-4 of the output's rms for these reductions of 128 / 512 terms.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import mla_pkg
from synth.device import to_torch

pytestmark = pytest.mark.gpu

D_H, D_C = 128, 512


def _draw(seed, shape, scale, stream):
    bits = synth.normal(seed, stream, int(np.prod(shape)), scale, 0, "bf16").reshape(shape)
    return bits, O.bf16_bits_to_f64(bits)


def _check(got: torch.Tensor, ref: np.ndarray):
    g = O.bf16_bits_to_f64(got.view(torch.int16).cpu().numpy().view(np.uint16))
    assert g.shape == ref.shape
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(g - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * rms
    worst = float(np.max(err - bound))
    assert worst <= 0.0, (worst, float(err.max()), rms)
    rel_l2 = float(np.linalg.norm(g - ref) / np.linalg.norm(ref))
    assert rel_l2 <= 3e-3, rel_l2


@pytest.mark.parametrize("n,H", [(1, 16), (64, 16), (100, 16), (64, 128), (257, 4)])
def test_absorb_query_matches_oracle(n, H):
    mla = mla_pkg()
    wb, w = _draw(1100 + n, (H, D_H, D_C), 1 / np.sqrt(D_H), 1)
    qb, q = _draw(1100 + n, (n, H, D_H), 1.0, 2)
    out = torch.full((n, H, D_C), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_query(to_torch(wb, "bf16"), to_torch(qb, "bf16"), out)
    torch.cuda.synchronize()
    _check(out, O.absorb_query(w, q))


@pytest.mark.parametrize("n,H", [(1, 16), (64, 16), (100, 16), (64, 128), (257, 4)])
def test_absorb_output_matches_oracle(n, H):
    mla = mla_pkg()
    wb, w = _draw(1200 + n, (H, D_H, D_C), 1 / np.sqrt(D_C), 3)
    ub, u = _draw(1200 + n, (n, H, D_C), 1.0, 4)
    out = torch.full((n, H, D_H), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_output(to_torch(wb, "bf16"), to_torch(ub, "bf16"), out)
    torch.cuda.synchronize()
    _check(out, O.absorb_output(w, u))


def test_absorb_wider_head_dims_and_status_word():
    # d_h = 256 (two output tiles on the output side, four reduction blocks on
    # the query side); the status word stays MLA_OK
    mla = mla_pkg()
    H, d_h, d_c, n = 8, 256, 384, 70
    wb, w = _draw(1300, (H, d_h, d_c), 1 / np.sqrt(d_h), 5)
    qb, q = _draw(1300, (n, H, d_h), 1.0, 6)
    ub, u = _draw(1300, (n, H, d_c), 1.0, 7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qn = torch.empty((n, H, d_c), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((n, H, d_h), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_query(to_torch(wb, "bf16"), to_torch(qb, "bf16"), qn, status=status)
    mla.mla_absorb_output(to_torch(wb, "bf16"), to_torch(ub, "bf16"), o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _check(qn, O.absorb_query(w, q))
    _check(o, O.absorb_output(w, u))


def test_absorb_empty_batch_is_a_no_op():
    mla = mla_pkg()
    w = torch.zeros((4, D_H, D_C), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((0, 4, D_H), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((0, 4, D_C), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_query(w, x, y)
    torch.cuda.synchronize()
