"""CUDA path vs the fp64 oracle, element by element, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth
from gpu_util import append_flags, build_cache, compare, mla_pkg, run_decode
from synth.device import empty_pool, to_torch, upload

pytestmark = pytest.mark.gpu


def _ordered(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers ordered like the values (for ulp distance)."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


# ------------------------------------------------------------------ append --

def test_append_places_rows_bit_exactly_and_within_one_ulp():
    w = synth.custom_bf16("append_paged", 501, [1, 63, 64, 65, 130, 257], H=4, paged=True)
    cache, d = build_cache(w)
    pool = cache.data.view(torch.int16).cpu().numpy().view(np.uint16)
    # oracle pool from the same raw draws
    ref = np.full(pool.shape, np.nan)
    seq, pos = w.token_seq_pos()
    c_raw, k_raw = w.all_raw_rows()
    rows = O.append_rows(O.widen(c_raw, "bf16"), O.widen(k_raw, "bf16"), pos, np.ones(w.d_c), w.eps,
                         w.rope_base, O.append_flags(w), "bf16")
    O.cache_write(ref, w.page_table(), seq, pos, rows)
    written_ref = ~np.isnan(ref[:, :, 0])
    got_vals = O.bf16_bits_to_f64(pool)
    written_gpu = ~np.isnan(got_vals[:, :, 0])
    assert np.array_equal(written_ref, written_gpu)            # placement: bit-exact
    assert np.all(np.isnan(got_vals[~written_gpu]))            # untouched slots keep the canary
    ref_bits = O.f64_to_bf16_bits(ref[written_ref])
    ulp = np.abs(_ordered(pool[written_ref]) - _ordered(ref_bits))
    assert ulp.max() <= 1, ulp.max()
    assert np.mean(ulp == 0) > 0.99


def test_append_vector_and_scalar_kernels_write_the_same_rows():
    """The 576-wide bf16 append uses 16-byte accesses when its inputs are
    16-byte aligned and the general kernel otherwise; both must write the
    same bits (same arithmetic and summation order)."""
    mla = mla_pkg()
    w = synth.custom_bf16("append_align", 502, [1, 63, 64, 65, 130, 257], H=4, paged=True)
    d = upload(w, "cuda")
    T = d["raw_c"].shape[0]
    pools = []
    for offset in (0, 1):   # offset 1: the inputs start 2 bytes past a 16-byte boundary
        big_c = torch.zeros(T * w.d_c + 8, dtype=torch.bfloat16, device="cuda")
        big_k = torch.zeros(T * w.d_r + 8, dtype=torch.bfloat16, device="cuda")
        c_in = big_c[offset:offset + T * w.d_c].view(T, w.d_c)
        k_in = big_k[offset:offset + T * w.d_r].view(T, w.d_r)
        c_in.copy_(d["raw_c"])
        k_in.copy_(d["raw_k"])
        pool = empty_pool(w, "cuda", fill_nan=True)
        cache = mla.Cache(pool, d["page_table"], w.d_c, w.d_r)
        mla.mla_cache_append(cache, c_in, k_in, d["seq_ids"], d["positions"], eps=w.eps, rope_base=w.rope_base,
                             flags=append_flags(mla, w))
        torch.cuda.synchronize()
        pools.append(pool.view(torch.int16).cpu().numpy())
    assert np.array_equal(pools[0], pools[1])


@pytest.mark.parametrize("positions", [[0, 4095, 4096, 131071]])
def test_append_rope_at_position_edges(positions):
    mla = mla_pkg()
    pages = 131072 // 64
    perm = synth.permutation(77, 9, pages)
    pool = torch.full((pages, 64, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    pt = torch.from_numpy(perm.reshape(1, pages)).cuda()
    cache = mla.Cache(pool, pt, 512, 64)
    T = len(positions)
    c_raw = synth.normal(5, 1, T * 512, 1 / 24, 0, "bf16").reshape(T, 512)
    k_raw = synth.normal(5, 2, T * 64, 1 / 24, 0, "bf16").reshape(T, 64)
    pos = np.array(positions, dtype=np.int32)
    mla.mla_cache_append(cache, to_torch(c_raw, "bf16"), to_torch(k_raw, "bf16"),
                         torch.zeros(T, dtype=torch.int32, device="cuda"), torch.from_numpy(pos).cuda())
    got = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = O.append_rows(O.widen(c_raw, "bf16"), O.widen(k_raw, "bf16"), pos, np.ones(512), 1e-6, 10000.0, 3, "bf16")
    for i, p in enumerate(positions):
        row = got[perm[p // 64], p % 64]
        ulp = np.abs(_ordered(row) - _ordered(O.f64_to_bf16_bits(ref[i])))
        assert ulp.max() <= 1, (p, ulp.max())
    assert int(np.sum(~np.isnan(O.bf16_bits_to_f64(got[:, :, 0])))) == T
    # position 0: the RoPE key is copied unchanged
    assert np.array_equal(got[perm[0], 0, 512:], k_raw[0])


def test_append_yarn_rope_at_position_edges():
    """YaRN frequencies (s = 40, alpha = 1, beta = 32, 4K window) at the edges
    of the original and the extended window."""
    mla = mla_pkg()
    positions = [0, 4095, 4096, 65535, 131071, 163839]
    pages = 163840 // 64
    perm = synth.permutation(78, 9, pages)
    pool = torch.full((pages, 64, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    pt = torch.from_numpy(perm.reshape(1, pages)).cuda()
    cache = mla.Cache(pool, pt, 512, 64)
    T = len(positions)
    c_raw = synth.normal(6, 1, T * 512, 1 / 24, 0, "bf16").reshape(T, 512)
    k_raw = synth.normal(6, 2, T * 64, 1 / 24, 0, "bf16").reshape(T, 64)
    pos = np.array(positions, dtype=np.int32)
    mla.mla_cache_append_rope(cache, to_torch(c_raw, "bf16"), to_torch(k_raw, "bf16"),
                              torch.zeros(T, dtype=torch.int32, device="cuda"), torch.from_numpy(pos).cuda(),
                              mla.yarn_rope())
    got = pool.view(torch.int16).cpu().numpy().view(np.uint16)
    theta = O.yarn_theta(64, 10000.0, 40.0, 1.0, 32.0, 4096)
    ref = O.append_rows(O.widen(c_raw, "bf16"), O.widen(k_raw, "bf16"), pos, np.ones(512), 1e-6, 10000.0, 3, "bf16",
                        theta)
    for i, p in enumerate(positions):
        row = got[perm[p // 64], p % 64]
        ulp = np.abs(_ordered(row) - _ordered(O.f64_to_bf16_bits(ref[i])))
        assert ulp.max() <= 1, (p, ulp.max())
    # plain RoPE would differ at large positions: the slow pairs really were interpolated
    plain = O.append_rows(O.widen(c_raw, "bf16"), O.widen(k_raw, "bf16"), pos, np.ones(512), 1e-6, 10000.0, 3, "bf16")
    assert not np.array_equal(O.f64_to_bf16_bits(plain[-1]), got[perm[positions[-1] // 64], positions[-1] % 64])


def test_bf16_decode_over_a_yarn_cache_with_the_temperature():
    mla = mla_pkg()
    w = synth.custom_bf16("yarn_decode", 707, [300, 4100, 70, 2048], H=128, Q=1, paged=True, q_gain=4.0)
    cache, d = build_cache(w, rope=mla.yarn_rope())
    scale = mla.mla_yarn_softmax_scale(1.0 / math.sqrt(w.d_h + w.d_r), 40.0)
    out, lse = run_decode(w, cache, d, scale=scale)
    compare(w, out, lse, theta=O.yarn_theta(64, 10000.0, 40.0, 1.0, 32.0, 4096), scale=scale)


# -------------------------------------------------------------- fp32 path --

@pytest.mark.parametrize("n_split", [None, 2, 4, 64])
def test_tiny_fp32_config_within_1e5(n_split):
    w = synth.tiny_fp32()
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d, n_split=n_split)
    compare(w, out, lse)


# -------------------------------------------------------------- bf16 path --

SMALL_CASES = [
    # name, lens, H, Q, paged, q_gain
    ("h128_q1_ragged", [1, 2, 63, 64, 65, 127, 128, 129, 300, 1000], 128, 1, True, 1.0),
    ("h16_q1_ragged", [1, 5, 64, 65, 200, 777], 16, 1, True, 1.0),
    ("h32_q1", [100, 64, 3000], 32, 1, False, 1.0),
    ("h64_q2_one_unit", [1, 2, 64, 65, 66, 400], 64, 2, True, 1.0),
    ("h128_q2_two_units", [1, 2, 3, 64, 65, 66, 500], 128, 2, True, 1.0),
    ("h16_q2", [1, 2, 129, 1025], 16, 2, True, 1.0),
    ("h128_sharp_softmax", [50, 700, 2049], 128, 1, True, 16.0),
    ("h128_q2_sharp", [2, 130, 999], 128, 2, True, 16.0),
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
def test_bf16_small_cases(case):
    name, lens, H, Q, paged, q_gain = case
    w = synth.custom_bf16(name, 600 + len(name), lens, H=H, Q=Q, paged=paged, q_gain=q_gain)
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    compare(w, out, lse)


@pytest.mark.parametrize("n_split", [1, 3, 32, 200])
def test_bf16_split_combine_small(n_split):
    w = synth.custom_bf16("split_small", 701, [1, 65, 640, 1999, 4096], H=128, Q=1, paged=True)
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d, n_split=n_split)
    compare(w, out, lse)


def test_bf16_three_phases_equal_one_call():
    w = synth.custom_bf16("phases", 702, [700, 64, 3001, 1], H=128, Q=2, paged=True)
    cache, d = build_cache(w)
    out1, lse1 = run_decode(w, cache, d)
    out2, lse2 = run_decode(w, cache, d, phases=True)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
    compare(w, out1, lse1)


def test_bf16_one_plan_serves_several_attention_launches():
    """A caller decoding several layers with the same lengths plans once and
    runs the attention kernel per layer; split units must merge every time."""
    mla = mla_pkg()
    w = synth.custom_bf16("plan_reuse", 705, [4096, 4096, 700, 64, 3001], H=128, Q=1, paged=True)
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


def test_bf16_many_short_sequences_more_units_than_workers():
    lens = synth.uniform_int(703, 5, 300, 1, 300)
    w = synth.custom_bf16("many_short", 703, lens, H=128, Q=1, paged=True)
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    compare(w, out, lse, seqs=range(0, 300, 7))


def test_bad_sequence_length_is_reported_not_faulted():
    mla = mla_pkg()
    w = synth.custom_bf16("bad_len", 704, [64, 128], H=128, Q=1)
    cache, d = build_cache(w)
    d["seq_lens"][1] = 10 ** 6          # beyond the page table's capacity
    out = torch.empty((2, 1, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 1, 128), dtype=torch.float32, device="cuda")
    ws = mla.alloc_workspace(2, 1, 128)
    mla.mla_decode(cache, d["seq_lens"], d["q_nope"], d["q_rope"], out, lse=lse, workspace=ws)
    assert mla.mla_decode_read_status(ws) == mla.MLA_ERR_INVALID_ARG
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))


def test_bounded_wait_reports_timeout_and_context_survives():
    mla = mla_pkg()
    ws = mla.alloc_workspace(1, 1, 128)
    ws.zero_()
    mla.mla_selftest_bounded_wait(ws, timeout_us=20000)
    assert mla.mla_decode_read_status(ws) == mla.MLA_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert float(torch.ones(4, device="cuda").sum()) == 4.0


# ------------------------------------------------------- full-size configs --
# The four full-size configurations are compared with the oracle over their
# whole out / lse tensors, except the ragged paged one (about 1.2 TFLOP of
# fp64 work for all 128 sequences), which is compared on a sample that spans
# its shortest and longest sequences and the lengths at page boundaries.

_ORACLE_CACHE = {}


def _oracle_long_sequence(w, b, chunk=4096):
    """Oracle (out, lse) of a one-query-token sequence, computed over chunks of
    its history and merged with the oracle's log-sum-exp combine (which the
    CPU pins prove equal to the whole); the fp64 cache of a 131,072-token
    sequence is built chunk by chunk so that it never sits in memory whole."""
    assert w.Q == 1
    L = int(w.lens[b])
    qn, qr = w.queries_of(b)
    qn, qr = O.widen(qn, w.raw_dtype)[0], O.widen(qr, w.raw_dtype)[0]
    scale = O.workload_scale(w)
    outs, lses = [], []
    for s0 in range(0, L, chunk):
        C, R = O.sequence_cache(w, b, s0, min(L, s0 + chunk))
        o, l, _ = O.decode_row(C, R, qn, qr, scale)
        outs.append(o)
        lses.append(l)
    o, l = O.combine_partials(np.stack(outs), np.stack(lses))
    return o[None], l[None]


def _oracle_for(w, seqs):
    """Oracle (out, lse) of the listed sequences of `w`, computed once per
    workload and reused by the parametrised tests."""
    key = w.name
    have = _ORACLE_CACHE.setdefault(key, {})
    for b in seqs:
        if int(b) not in have:
            if int(w.lens[b]) > 16384 and w.Q == 1:
                have[int(b)] = _oracle_long_sequence(w, int(b))
            else:
                have[int(b)] = O.decode_sequence(w, int(b))
    return have


def _compare_cached(w, out, lse, seqs):
    ref = _oracle_for(w, seqs)
    ref_o = np.stack([ref[int(b)][0] for b in seqs])
    ref_l = np.stack([ref[int(b)][1] for b in seqs])
    return compare(w, out, lse, seqs=seqs, ref=(ref_o, ref_l))


def _ragged_sample(w, k=24):
    """Indices of: the 4 shortest and 4 longest sequences, every sequence whose
    length sits at a page boundary (len % 64 in {0, 1, 63}), then evenly
    spaced ones up to k."""
    lens = np.asarray(w.lens)
    order = np.argsort(lens, kind="stable")
    pick = list(order[:4]) + list(order[-4:])
    pick += [b for b in range(w.B) if int(lens[b]) % 64 in (0, 1, 63)]
    for b in np.linspace(0, w.B - 1, k).astype(int):
        if len(set(pick)) >= k:
            break
        pick.append(int(b))
    return sorted(set(int(b) for b in pick))


def test_full_small_head_config():
    w = synth.small_head()
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    _compare_cached(w, out, lse, range(w.B))


def test_full_width_config():
    w = synth.full_width()
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    _compare_cached(w, out, lse, range(w.B))


def test_full_ragged_paged_q2_config():
    w = synth.ragged_paged()
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d)
    assert np.all(np.isfinite(out))
    seqs = _ragged_sample(w)
    assert len(seqs) >= 16
    _compare_cached(w, out, lse, seqs)


@pytest.mark.parametrize("n_split", [32, 64, 128])
def test_full_long_split_config(n_split):
    w = synth.long_split()
    cache, d = build_cache(w)
    out, lse = run_decode(w, cache, d, n_split=n_split)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    _compare_cached(w, out, lse, range(w.B))
