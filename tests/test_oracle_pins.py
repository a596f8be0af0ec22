"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

None of these retypes the oracle's formula.  They use closed forms, algebraic
identities (the absorbed result equals explicit multi-head attention with K/V
expanded from the latent), invariants of softmax and rotations, brute force
on tiny inputs with a different summation route, and the cache figures the
"DeepSeek-V2 analysis" page prints.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


# ---------------------------------------------------------------- bfloat16 --

def _bf16_by_bits(x32: np.ndarray) -> np.ndarray:
    """Independent RNE float32 -> bfloat16 via integer rounding on the bits."""
    u = x32.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def test_bf16_matches_integer_rounding_on_float32_inputs():
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    assert np.array_equal(O.f64_to_bf16_bits(x32.astype(np.float64)), _bf16_by_bits(x32))


def test_bf16_ties_to_even_and_exact_values():
    one = 1.0
    assert O.round_to_bf16(np.array([one + 2 ** -8]))[0] == 1.0
    assert O.round_to_bf16(np.array([one + 3 * 2 ** -8]))[0] == one + 2 ** -6
    assert O.round_to_bf16(np.array([-(one + 2 ** -8)]))[0] == -1.0
    assert O.round_to_bf16(np.array([one + 2 ** -8 + 2 ** -30]))[0] == one + 2 ** -7
    bits = rng.integers(0, 0x7F80, 5000).astype(np.uint16)   # finite positives
    v = O.bf16_bits_to_f64(bits)
    assert np.array_equal(O.f64_to_bf16_bits(v), bits)


def test_bf16_relative_error_bound():
    x = rng.standard_normal(100000) * 10.0 ** rng.uniform(-6, 6, 100000)
    r = O.round_to_bf16(x)
    assert np.all(np.abs(r - x) <= 2.0 ** -8 * np.abs(x) * (1 + 1e-12))  # unit roundoff, 8 significant bits


# ----------------------------------------------------------------- RMSNorm --

def test_rmsnorm_unit_mean_square_and_scale_invariance():
    x = rng.standard_normal((7, 512))
    y = O.rmsnorm(x, np.ones(512), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(O.rmsnorm(3.7 * x, np.ones(512), 0.0), y, rtol=1e-14, atol=1e-15)
    g = rng.uniform(0.5, 2.0, 512)
    assert np.allclose(O.rmsnorm(x, g, 0.0), y * g, rtol=1e-14)


def test_rmsnorm_eps_enters_inside_the_root():
    x = np.full((1, 4), 2.0)
    eps = 5.0
    # mean square 4 -> divide by sqrt(9) = 3
    assert np.allclose(O.rmsnorm(x, np.ones(4), eps), 2.0 / 3.0)


# -------------------------------------------------------------------- RoPE --

def test_rope_identity_at_position_zero():
    x = rng.standard_normal((5, 64))
    assert np.array_equal(O.rope(x, np.zeros(5), 10000.0), x)


def test_rope_mixes_only_adjacent_pairs_and_preserves_pair_norms():
    d = 64
    for k in (0, 1, 2, 17, 62, 63):
        e = np.zeros(d)
        e[k] = 1.0
        y = O.rope(e, 1234, 10000.0)
        nz = set(np.nonzero(np.abs(y) > 1e-15)[0].tolist())
        assert nz <= {k, k ^ 1}
    x = rng.standard_normal((9, d))
    pos = rng.integers(0, 200000, 9)
    y = O.rope(x, pos, 10000.0)
    n_in = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    n_out = y[:, 0::2] ** 2 + y[:, 1::2] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    d = 64
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for m, n in [(5, 3), (4095, 4096), (131071, 17), (0, 9)]:
        lhs = O.rope(q, m, 10000.0) @ O.rope(k, n, 10000.0)
        rhs = O.rope(q, m - n, 10000.0) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(lhs))


def test_rope_frequencies_are_geometric_from_one():
    d, base = 64, 10000.0
    x = np.zeros(d)
    x[0::2] = 1.0
    y = O.rope(x, 1, base)
    theta = np.arctan2(y[1::2], y[0::2])            # angle of each pair at pos 1
    assert abs(theta[0] - 1.0) < 1e-15
    ratio = theta[1:] / theta[:-1]
    assert np.allclose(ratio, base ** (-2.0 / d), rtol=1e-12)
    # counter-clockwise: the second element of the pair gains +sin
    assert y[1] > 0


# ------------------------------------------------------------------ decode --

def _rand_row(S, H, d_c, d_r, q_gain=1.0):
    C = rng.standard_normal((S, d_c))
    R = rng.standard_normal((S, d_r))
    qn = rng.standard_normal((H, d_c)) * q_gain / math.sqrt(d_c)
    qr = rng.standard_normal((H, d_r)) * q_gain / math.sqrt(d_r)
    return C, R, qn, qr


def test_single_key_returns_that_latent_exactly():
    C, R, qn, qr = _rand_row(1, 4, 32, 8)
    out, lse, a = O.decode_row(C, R, qn, qr, 0.3)
    assert np.array_equal(out, np.broadcast_to(C[0], out.shape))
    assert np.allclose(lse, 0.3 * (qn @ C[0] + qr @ R[0]), rtol=1e-15)


def test_zero_query_gives_mean_of_latents_and_log_length():
    C, R, _, _ = _rand_row(37, 3, 32, 8)
    out, lse, _ = O.decode_row(C, R, np.zeros((3, 32)), np.zeros((3, 8)), 0.2)
    assert np.allclose(out, C.mean(axis=0), rtol=1e-13, atol=1e-14)
    assert np.allclose(lse, math.log(37), rtol=1e-15)


def test_dominant_key_selects_its_latent():
    C, R, qn, qr = _rand_row(50, 2, 16, 8)
    qr[:] = 0
    qn[:] = 0
    R[:] = 0
    R[23] = 1.0
    qr[:, :] = 200.0                                   # score 200*8*scale on key 23 only
    out, _, a = O.decode_row(C, R, qn, qr, 0.5)
    assert np.allclose(out, C[23], atol=1e-12)
    assert np.all(a[:, 23] > 1 - 1e-12)


def test_rows_sum_to_one_and_weights_nonnegative():
    C, R, qn, qr = _rand_row(300, 8, 64, 16, q_gain=16.0)
    _, _, a = O.decode_row(C, R, qn, qr, O.softmax_scale(32, 16))
    assert np.all(a >= 0)
    assert np.allclose(a.sum(axis=1), 1.0, rtol=0, atol=1e-13)


def test_brute_force_tiny_with_separate_summation():
    """Pure-Python loops, exact-rounded sums (math.fsum), no max shift."""
    S, H, d_c, d_r = 5, 2, 4, 2
    C, R, qn, qr = _rand_row(S, H, d_c, d_r, q_gain=2.0)
    scale = 0.37
    out, lse, _ = O.decode_row(C, R, qn, qr, scale)
    for h in range(H):
        e = []
        for s in range(S):
            dot = math.fsum([qn[h, k] * C[s, k] for k in range(d_c)] +
                            [qr[h, k] * R[s, k] for k in range(d_r)])
            e.append(math.exp(scale * dot))
        Z = math.fsum(e)
        assert abs(lse[h] - math.log(Z)) < 1e-13
        for k in range(d_c):
            v = math.fsum([e[s] * C[s, k] for s in range(S)]) / Z
            assert abs(out[h, k] - v) < 1e-13


def test_permuting_the_history_does_not_change_the_result():
    C, R, qn, qr = _rand_row(77, 4, 32, 8, q_gain=8.0)
    p = rng.permutation(77)
    o1, l1, _ = O.decode_row(C, R, qn, qr, 0.25)
    o2, l2, _ = O.decode_row(C[p], R[p], qn, qr, 0.25)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(l1, l2, rtol=1e-14)


def test_two_causal_queries_equal_two_single_query_decodes():
    L, H, d_c, d_r = 40, 3, 16, 8
    C = rng.standard_normal((L, d_c))
    R = rng.standard_normal((L, d_r))
    qn = rng.standard_normal((1, 2, H, d_c))
    qr = rng.standard_normal((1, 2, H, d_r))
    out, lse = O.decode(lambda b: C, lambda b: R, qn, qr, [L], 2, 0.3)
    o0, l0, _ = O.decode_row(C[:L - 1], R[:L - 1], qn[0, 0], qr[0, 0], 0.3)
    o1, l1, _ = O.decode_row(C[:L], R[:L], qn[0, 1], qr[0, 1], 0.3)
    assert np.allclose(out[0, 0], o0, rtol=1e-15) and np.allclose(out[0, 1], o1, rtol=1e-15)
    assert np.allclose(lse[0, 0], l0) and np.allclose(lse[0, 1], l1)


def test_row_with_no_visible_key_is_zero_with_minus_inf_lse():
    C = rng.standard_normal((1, 8))
    R = rng.standard_normal((1, 4))
    qn = rng.standard_normal((1, 2, 2, 8))
    qr = rng.standard_normal((1, 2, 2, 4))
    out, lse = O.decode(lambda b: C, lambda b: R, qn, qr, [1], 2, 0.5)
    assert np.all(out[0, 0] == 0) and np.all(np.isneginf(lse[0, 0]))
    assert np.allclose(out[0, 1], C[0]) and np.all(np.isfinite(lse[0, 1]))


@pytest.mark.parametrize("cuts", [[0, 100, 333, 1000], [0, 1, 2, 1000], [0, 500, 500, 1000]])
def test_split_and_combine_equals_whole(cuts):
    C, R, qn, qr = _rand_row(1000, 4, 32, 8, q_gain=12.0)
    o_all, l_all, _ = O.decode_row(C, R, qn, qr, 0.3)
    parts = [O.decode_row(C[a:b], R[a:b], qn, qr, 0.3)[:2] for a, b in zip(cuts[:-1], cuts[1:])]
    o, l = O.combine_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.allclose(o, o_all, rtol=1e-12, atol=1e-14)
    assert np.allclose(l, l_all, rtol=1e-14)


def test_combine_of_only_empty_parts():
    o, l = O.combine_partials(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))


# ------------------------------------------------------------- absorption --

def _absorption_case(scale_override=None, seed=1001):
    """Tiny fp32 workload; W^UK absorbed into q_nope must equal explicit MHA."""
    w = synth.tiny_fp32(seed)
    d_h = w.d_h
    st = synth.STREAM_EXTRA
    W_UK = synth.normal(w.seed, st + 0, w.H * d_h * w.d_c, 1 / math.sqrt(w.d_c)).reshape(w.H, d_h, w.d_c)
    W_UV = synth.normal(w.seed, st + 1, w.H * d_h * w.d_c, 1 / math.sqrt(w.d_c)).reshape(w.H, d_h, w.d_c)
    qc = synth.normal(w.seed, st + 2, w.B * w.H * d_h, 1 / math.sqrt(d_h)).reshape(w.B, w.H, d_h)
    worst = 0.0
    for b in range(w.B):
        C, R = O.sequence_cache(w, b)
        _, qr = w.queries_of(b)
        qr = O.widen(qr, w.raw_dtype)[0]
        q_nope = O.absorb_query(W_UK, qc[b])                     # W^UK_h^T q^C_h
        scale = O.softmax_scale(d_h, w.d_r) if scale_override is None else scale_override
        u, _, _ = O.decode_row(C, R, q_nope, qr, scale)
        absorbed = O.absorb_output(W_UV, u)                      # W^UV_h u_h
        explicit = O.explicit_mha_row(C, R, qc[b], qr, W_UK, W_UV)
        worst = max(worst, float(np.max(np.abs(absorbed - explicit)) / np.max(np.abs(explicit))))
    return worst


def test_absorbed_equals_explicit_mha():
    assert _absorption_case() <= 1e-12


def test_absorb_functions_against_per_head_products():
    # the batched forms equal the per-head matrix products written out, and a
    # transposed weight (the d_h x d_c block used the wrong way round) or a
    # head mix-up does not pass
    rng = np.random.default_rng(7)
    H, d_h, d_c, n = 3, 4, 6, 5
    W = rng.standard_normal((H, d_h, d_c))
    qc = rng.standard_normal((n, H, d_h))
    u = rng.standard_normal((n, H, d_c))
    q = O.absorb_query(W, qc)
    o = O.absorb_output(W, u)
    for t in range(n):
        for h in range(H):
            assert np.allclose(q[t, h], W[h].T @ qc[t, h], rtol=1e-14, atol=1e-14)
            assert np.allclose(o[t, h], W[h] @ u[t, h], rtol=1e-14, atol=1e-14)
    assert not np.allclose(O.absorb_query(W[::-1], qc), q)
    # q_h^T (W_UK_h c) = (W_UK_h^T q_h)^T c for every latent c: the absorbed
    # query gives the same content score as the expanded key
    c = rng.standard_normal(d_c)
    for h in range(H):
        assert abs(qc[0, h] @ (W[h] @ c) - q[0, h] @ c) < 1e-12


def _prefill_case(seed=1002):
    rng = np.random.default_rng(seed)
    S, T, H, d_h, d_c, d_r = 24, 5, 3, 8, 32, 4
    C, R = rng.standard_normal((S, d_c)), rng.standard_normal((S, d_r))
    W_UK = rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c)
    W_UV = rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c)
    qc, qr = rng.standard_normal((T, H, d_h)), rng.standard_normal((T, H, d_r))
    positions = np.array([0, 3, 10, 22, 23])
    return C, R, qc, qr, W_UK, W_UV, positions


def test_expanded_prefill_equals_absorbed_decode_at_every_position():
    # the prefill (expanded) and decode (absorbed) forms compute one function
    C, R, qc, qr, W_UK, W_UV, pos = _prefill_case()
    o, lse = O.prefill_expanded(C, R, qc, qr, W_UK, W_UV, pos)
    scale = 1 / math.sqrt(qc.shape[2] + R.shape[1])
    for t, p in enumerate(pos):
        u, l, _ = O.decode_row(C[:p + 1], R[:p + 1], O.absorb_query(W_UK, qc[t]), qr[t], scale)
        assert np.allclose(o[t], O.absorb_output(W_UV, u), rtol=1e-12, atol=1e-13)
        assert np.allclose(lse[t], l, rtol=1e-13)
        # and equals the per-head explicit form written as loops
        assert np.allclose(o[t], O.explicit_mha_row(C[:p + 1], R[:p + 1], qc[t], qr[t], W_UK, W_UV),
                           rtol=1e-12, atol=1e-13)


def test_expanded_prefill_is_causal():
    C, R, qc, qr, W_UK, W_UV, pos = _prefill_case()
    o, _ = O.prefill_expanded(C, R, qc, qr, W_UK, W_UV, pos)
    C2, R2 = C.copy(), R.copy()
    C2[11:] += 5.0                                   # keys after position 10 change
    R2[11:] -= 3.0
    o2, _ = O.prefill_expanded(C2, R2, qc, qr, W_UK, W_UV, pos)
    assert np.array_equal(o[:3], o2[:3])             # queries at 0, 3, 10 do not see them
    assert not np.allclose(o[3:], o2[3:])


def test_absorption_check_catches_a_wrong_scale_dimension():
    # A decode scaled by 1/sqrt(d_c + d_r) (the mismatch the page warns about)
    # must not pass the identity.
    assert _absorption_case(scale_override=1 / math.sqrt(64 + 16)) > 1e-6


# ------------------------------------------------------------- accounting --

def _golden():
    with open(os.path.join(GOLDEN, "cache_accounting.json")) as f:
        return {e["id"]: e for e in json.load(f)["entries"]}


def _close(got, e):
    if "abs_tol" in e:
        return abs(got - e["value"]) <= e["abs_tol"]
    tol = e.get("rel_tol", 0)
    return abs(got - e["value"]) <= tol * abs(e["value"])


def test_cache_accounting_matches_printed_figures():
    g = _golden()
    GiB = 2.0 ** 30
    per = O.mla_elements_per_token_layer(512, 64)
    ds67 = O.mha_elements_per_token_layer(8, 128) * 95
    v2 = per * 60
    got = {
        "mla_per_layer": per,
        "mla_60_layers": v2,
        "mla_27_layers": per * 27,
        "mha_same_heads": O.mha_elements_per_token_layer(128, 128),
        "mha_ratio_57": O.mha_elements_per_token_layer(128, 128) / per,
        "ds67b_per_layer": O.mha_elements_per_token_layer(8, 128),
        "ds67b_95_layers": ds67,
        "element_reduction_pct": 100 * (1 - v2 / ds67),
        "six_bit_reduction_pct": 100 * (1 - O.cache_bytes(per, 60, 1, 6) / O.cache_bytes(ds67, 1, 1, 16)),
        "bf16_bytes_per_token_60": O.cache_bytes(per, 60, 1, 16),
        "bf16_kib_per_token_60": O.cache_bytes(per, 60, 1, 16) / 1024,
        "gib_128k": O.cache_bytes(per, 60, 131072, 16) / GiB,
        "gb_decimal_128k": O.cache_bytes(per, 60, 131072, 16) / 1e9,
        "per_head_rope_per_layer": O.mla_elements_per_token_layer(512, 64, per_head_rope_heads=128),
        "per_head_rope_gib": O.cache_bytes(O.mla_elements_per_token_layer(512, 64, 128), 60, 131072, 16) / GiB,
        "no_rope_gib": O.cache_bytes(O.mla_elements_per_token_layer(512, 0), 60, 131072, 16) / GiB,
        "rope_share_pct": 100 * 64 / per,
        "rope128_gib": O.cache_bytes(O.mla_elements_per_token_layer(512, 128), 60, 131072, 16) / GiB,
        "rope32_gib": O.cache_bytes(O.mla_elements_per_token_layer(512, 32), 60, 131072, 16) / GiB,
        # the page scales its rounded 8.44 GiB by 6/16
        "six_bit_packed_gib": round(O.cache_bytes(per, 60, 131072, 16) / GiB, 2) * 6 / 16,
        "eight_bit_container_gib": O.cache_bytes(per, 60, 131072, 8) / GiB,
        "ds67b_gib_128k": O.cache_bytes(ds67, 1, 131072, 16) / GiB,
    }
    assert set(got) == set(g)
    for k, v in got.items():
        assert _close(v, g[k]), (k, v, g[k]["value"], g[k]["cite"])


# ----------------------------------------------------- paged placement --

def test_paged_pool_gather_reproduces_sequence_rows():
    w = synth.custom_bf16("paged_tiny", 77, [1, 63, 64, 65, 130], H=4, Q=1, paged=True)
    pt = w.page_table()
    pool = np.full((w.num_pages, w.page_size, w.d_c + w.d_r), np.nan)
    seq, pos = w.token_seq_pos()
    c_raw, k_raw = w.all_raw_rows()
    rows = O.append_rows(O.widen(c_raw, "bf16"), O.widen(k_raw, "bf16"), pos, np.ones(w.d_c),
                         w.eps, w.rope_base, O.append_flags(w), "bf16")
    O.cache_write(pool, pt, seq, pos, rows)
    # every page slot is written exactly once or is past a sequence end
    assert np.sum(~np.isnan(pool[:, :, 0])) == w.total_tokens
    for b in range(w.B):
        C, R = O.sequence_cache(w, b)
        got = O.cache_gather(pool, pt, b, int(w.lens[b]))
        assert np.array_equal(got, np.concatenate([C, R], axis=1))


def test_page_slot_against_hand_written_placements():
    """Token `pos` of sequence `b` lives in page page_table[b][pos // P] at
    slot pos % P (the cache layout of the C ABI).  The expected (page, slot)
    pairs below are written out by hand for a 2-sequence table with pages of
    4 tokens, so a transposed table index or a swapped // and % fails."""
    pt = np.array([[5, 2, 7], [0, 3, 1]], dtype=np.int32)
    cases = [  # (seq, pos) -> (page, slot)
        ((0, 0), (5, 0)), ((0, 3), (5, 3)), ((0, 4), (2, 0)), ((0, 6), (2, 2)),
        ((0, 9), (7, 1)), ((0, 11), (7, 3)), ((1, 0), (0, 0)), ((1, 5), (3, 1)),
        ((1, 7), (3, 3)), ((1, 8), (1, 0)), ((1, 10), (1, 2)),
    ]
    seq = [c[0][0] for c in cases]
    pos = [c[0][1] for c in cases]
    page, slot = O.page_slot(pt, seq, pos, 4)
    assert [(int(p), int(s)) for p, s in zip(page, slot)] == [c[1] for c in cases]
    # cache_write puts each row at exactly that place and nowhere else
    pool = np.full((8, 4, 3), np.nan)
    rows = np.arange(len(cases) * 3, dtype=np.float64).reshape(len(cases), 3)
    O.cache_write(pool, pt, seq, pos, rows)
    for i, (_, (p, s)) in enumerate(cases):
        assert np.array_equal(pool[p, s], rows[i])
    assert np.sum(~np.isnan(pool[:, :, 0])) == len(cases)
    # cache_gather returns a sequence's rows in position order
    full = np.full((8, 4, 1), np.nan)
    for b in range(2):
        for p in range(12):
            full[pt[b, p // 4], p % 4, 0] = 100 * b + p
    assert np.array_equal(O.cache_gather(full, pt, 1, 11)[:, 0], 100 + np.arange(11))
    assert np.array_equal(O.cache_gather(full, pt, 0, 12)[:, 0], np.arange(12))
