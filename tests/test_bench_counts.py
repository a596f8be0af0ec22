"""Host-side arithmetic behind every roofline fraction bench.py reports.

`algorithmic_counts` gives the bytes a decode must move and the flops it
must do; each expected value below is written out by hand from the
workload's shape (cache rows of d_c + d_r = 576 bf16 values = 1,152 bytes,
or 656 bytes in the low-precision format; queries of 576 values per row;
outputs of 512 values per row; per visible (query, key) pair 2 * H * (576 +
512) flops, a causal query token j of Q seeing len - Q + j + 1 keys).
`kernel_traffic` must refuse ncu counters whose kernel source has changed.
"""
from __future__ import annotations

import hashlib
import os

import pytest

import bench
import synth


def test_full_width_counts():
    w = synth.full_width()          # B=64, S=4096, H=128, Q=1
    alg, flops, cache = bench.algorithmic_counts(w)
    assert cache == 64 * 4096 * 1152 == 301_989_888
    assert alg == 301_989_888 + 64 * 128 * 576 * 2 + 64 * 128 * 512 * 2 == 319_815_680
    assert flops == 2 * 128 * 1088 * 64 * 4096 == 73_014_444_032


def test_full_width_low_precision_counts():
    w = synth.full_width()
    alg, flops, cache = bench.algorithmic_counts(w, lowp=True)
    assert cache == 64 * 4096 * 656
    assert alg == 64 * 4096 * 656 + 9_437_184 + 8_388_608
    assert flops == 73_014_444_032     # the same contractions


def test_small_head_counts():
    w = synth.small_head()          # B=32, S=4096, H=16
    alg, flops, cache = bench.algorithmic_counts(w)
    assert cache == 32 * 4096 * 1152
    assert alg == 150_994_944 + 32 * 16 * 1152 + 32 * 16 * 1024 == 152_109_056
    assert flops == 2 * 16 * 1088 * 32 * 4096


def test_causal_visible_pairs_with_two_query_tokens():
    # lengths 5 and 1, Q = 2: sequence 0's tokens see 4 and 5 keys, sequence
    # 1's first query token sees none and its second sees 1: 10 pairs
    w = synth.custom_bf16("counts_q2", 7, [5, 1], H=4, Q=2, paged=True)
    alg, flops, cache = bench.algorithmic_counts(w)
    assert cache == 6 * 1152
    assert alg == 6 * 1152 + 2 * 2 * 4 * 1152 + 2 * 2 * 4 * 1024
    assert flops == 2 * 4 * 1088 * 10


def test_kernel_traffic_needs_the_profiled_source(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel body\n")
    digest = hashlib.sha256(b"kernel body\n").hexdigest()
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text(f"kernel_source_sha256: {digest[:16]}\ntraffic_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("k.md", "k.cu") == pytest.approx(12345.0)
    src.write_bytes(b"kernel body, changed\n")
    assert bench.kernel_traffic("k.md", "k.cu") is None
    assert bench.kernel_traffic("missing.md", "k.cu") is None


def test_committed_profiles_match_their_kernels():
    # every committed summary that carries counters names the current
    # source of its kernel (bench.py reports traffic only while they match)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pairs = {
        "decode_tc_full_width.md": "head_latent_attention_27_b300/csrc/decode_tc.cu",
        "decode_tc_lowp_full_width.md": "head_latent_attention_27_b300/csrc/decode_tc.cu",
        "decode_sh_small_head.md": "head_latent_attention_27_b300/csrc/decode_sh.cu",
        "prefill_attn_T4096_H128.md": "head_latent_attention_27_b300/csrc/prefill.cu",
    }
    for prof, src in pairs.items():
        assert os.path.exists(os.path.join(root, "profiles", prof)), prof
        assert bench.kernel_traffic(prof, src) is not None, prof
