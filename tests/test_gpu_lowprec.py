"""Low-precision latent cache on the GPU (the reading of "02 · DeepSeek-V2
analysis", sections 1.3 and 6.2: E4M3 latent with one fp32 scale per 128
latent values of a token, bf16 RoPE key).

The quantising append must store exactly the oracle's quantisation of the
bf16 row that the bf16 append forms (whose own placement and values are
pinned against the oracle elsewhere): codes, scales and RoPE bits equal,
untouched slots unchanged."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import build_cache, compare, mla_pkg
from oracle import lowprec_cache as LP
from synth.device import upload

pytestmark = pytest.mark.gpu


def _fp8_cache(w):
    mla = mla_pkg()
    d = upload(w, "cuda")
    pool8 = torch.full((w.num_pages, 64, mla.FP8_ROW_BYTES), 0xA5, dtype=torch.uint8, device="cuda")
    cache8 = mla.Cache(pool8, d["page_table"], w.d_c, w.d_r)
    mla.mla_cache_append(cache8, d["raw_c"], d["raw_k"], d["seq_ids"], d["positions"], eps=w.eps,
                         rope_base=w.rope_base, flags=mla.MLA_APPEND_RMSNORM | mla.MLA_APPEND_ROPE)
    torch.cuda.synchronize()
    return cache8, d


def test_quantising_append_stores_the_quantised_bf16_row():
    w = synth.custom_bf16("fp8_append", 1401, [1, 63, 64, 65, 300, 129], H=4, paged=True)
    cache_bf, _ = build_cache(w)
    cache8, _ = _fp8_cache(w)
    bf = cache_bf.data.view(torch.int16).cpu().numpy().view(np.uint16)      # [pages, 64, 576] bf16 bits
    q8 = cache8.data.cpu().numpy()                                          # [pages, 64, 656] bytes
    written = ~np.isnan(O.bf16_bits_to_f64(bf[:, :, 0]))
    assert written.sum() == w.total_tokens
    rows = O.bf16_bits_to_f64(bf[written])                                  # the bf16 rows, exactly
    codes, scales, _ = LP.quantize_cache_rows(rows, 512)
    got = q8[written]
    assert np.array_equal(got[:, :512], codes)                              # E4M3 codes: bit-exact
    got_scales = got[:, 512:528].copy().view(np.float32).astype(np.float64)
    assert np.array_equal(got_scales, scales)                               # fp32 scales: bit-exact
    assert np.array_equal(got[:, 528:].copy().view(np.uint16), bf[written][:, 512:])   # RoPE key: same bf16 bits
    assert np.all(q8[~written] == 0xA5)                                     # untouched slots keep the canary
    # the dequantised latent is within the E4M3 bound of the bf16 row
    deq = LP.dequantize_latent(codes, scales)
    assert np.all(np.abs(deq - rows[:, :512]) <= 2.0 ** -4 * np.abs(rows[:, :512]) + scales.repeat(128, axis=1) * 2.0 ** -10)


# --------------------------------------------------- decode over the rows --

def _oracle_lowp(w, b):
    """Oracle decode of sequence b over the oracle's own low-precision cache:
    its bf16 rows, quantised and dequantised by the oracle."""
    C, R = O.sequence_cache(w, b)
    codes, scales, _ = LP.quantize_cache_rows(np.concatenate([C, R], axis=1), 512)
    return O.decode_sequence(w, b, cache=(LP.dequantize_latent(codes, scales), R))


def _run_lowp(w, n_split=0):
    mla = mla_pkg()
    cache8, d = _fp8_cache(w)
    out = torch.full((w.B, w.Q, w.H, w.d_c), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.Q, w.H), float("nan"), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(w.B, w.Q, w.H, w.d_c, n_split, "cuda")
    scale = 1.0 / np.sqrt(w.d_h + w.d_r)
    if n_split:
        mla.mla_decode_split_combine(cache8, d["seq_lens"], d["q_nope"], d["q_rope"], out, n_split, lse=lse,
                                     workspace=ws, softmax_scale=scale)
    else:
        mla.mla_decode(cache8, d["seq_lens"], d["q_nope"], d["q_rope"], out, lse=lse, workspace=ws,
                       softmax_scale=scale)
    status = mla.mla_decode_read_status(ws)
    assert status == mla.MLA_OK, mla.mla_status_string(status)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


LOWP_CASES = [
    # name, lens, H, Q, q_gain, n_split
    ("lp_h128_ragged", [1, 2, 63, 64, 65, 127, 128, 129, 300, 1000], 128, 1, 1.0, 0),
    ("lp_h128_q2", [1, 2, 64, 65, 500, 3001], 128, 2, 1.0, 0),
    ("lp_h16", [1, 5, 64, 65, 200, 777], 16, 1, 1.0, 0),
    ("lp_sharp", [50, 700, 2049], 128, 1, 16.0, 0),
    ("lp_split", [1, 65, 640, 1999, 4096], 128, 1, 1.0, 32),
]


@pytest.mark.parametrize("case", LOWP_CASES, ids=[c[0] for c in LOWP_CASES])
def test_decode_over_the_low_precision_cache(case):
    name, lens, H, Q, q_gain, n_split = case
    w = synth.custom_bf16(name, 1500 + len(name), lens, H=H, Q=Q, paged=True, q_gain=q_gain)
    out, lse = _run_lowp(w, n_split)
    ref = [_oracle_lowp(w, b) for b in range(w.B)]
    compare(w, out, lse, ref=(np.stack([r[0] for r in ref]), np.stack([r[1] for r in ref])))


def test_decode_over_the_low_precision_cache_full_width():
    """The full-width workload (B=64, S=4096, H=128) over the low-precision
    cache, every sequence against the oracle."""
    w = synth.full_width()
    out, lse = _run_lowp(w)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    ref = [_oracle_lowp(w, b) for b in range(w.B)]
    compare(w, out, lse, ref=(np.stack([r[0] for r in ref]), np.stack([r[1] for r in ref])))
