"""The workspace-free decode entry point (mla_decode_noalloc).

It serves callers that cannot allocate device memory (for example a plugin
that only receives its input and output buffers): it uses a fixed scratch
array inside the library instead of a caller workspace.  These checks call
it through the C ABI, twice in a row, and compare with mla_decode, which
takes a workspace; they also check that a decode too large for the fixed
scratch is refused before anything is launched.  Collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import synth
from gpu_util import BF16_LSE_ABS, BF16_MAX_ABS, BF16_REL_L2, build_cache, compare, mla_pkg, run_decode

pytestmark = pytest.mark.gpu


def _noalloc(mla, w, cache, d, scale):
    out = torch.full((w.B, w.Q, w.H, w.d_c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.Q, w.H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_noalloc(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, lse=lse, softmax_scale=scale)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def test_noalloc_decode_matches_decode_with_workspace_on_two_calls():
    """Two calls in a row on different length mixes (the second one has
    fewer, shorter sequences, so plan arrays or partial rows left in the
    shared array by the first call would show).  Each result must equal
    mla_decode's bit for bit (same plan, same kernels, same device) and the
    oracle's within the bf16 tolerance."""
    mla = mla_pkg()
    workloads = [
        synth.custom_bf16("noalloc_a", 909, [1, 63, 700, 4096, 2049, 130], H=128, Q=2, paged=True),
        synth.custom_bf16("noalloc_b", 910, [5, 3000, 65, 1], H=128, Q=1, paged=True),
    ]
    for w in workloads:
        cache, d = build_cache(w)
        scale = 1.0 / math.sqrt(w.d_h + w.d_r)
        ref_out, ref_lse = run_decode(w, cache, d)
        got_o, got_l = _noalloc(mla, w, cache, d, scale)
        assert np.array_equal(got_o, ref_out)
        assert np.array_equal(got_l, ref_lse)
        res = compare(w, got_o, got_l)
        assert res["max_abs"] <= BF16_MAX_ABS and res["rel_l2"] <= BF16_REL_L2 and res["lse_abs"] <= BF16_LSE_ABS


def test_noalloc_refuses_a_decode_larger_than_its_scratch():
    mla = mla_pkg()
    pool = torch.zeros((4, 64, 576), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((4096, 1), dtype=torch.int32, device="cuda")
    B = 4096                                   # 4096 units need far more than the fixed scratch
    seq = torch.ones(B, dtype=torch.int32, device="cuda")
    q = torch.zeros((1, 1, 128, 512), dtype=torch.bfloat16, device="cuda")
    cc = mla.mla_cache_t(pool.data_ptr(), pt.data_ptr(), mla.MLA_BF16, 4096, 4, 64, 512, 64, 1)
    code = mla._lib.mla_decode_noalloc(ctypes.byref(cc), seq.data_ptr(), B, q.data_ptr(), q.data_ptr(), 1, 128,
                                       0.07, q.data_ptr(), None, None)
    assert code == mla.MLA_ERR_WORKSPACE
