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
from gpu_util import build_cache, mla_pkg
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
