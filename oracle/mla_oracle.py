"""fp64 CPU oracle for absorbed Multi-head Latent Attention decode.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plain reference that the
CUDA path is checked against.  Only the test-suite, the package smoke check
and the benchmark's CPU-baseline leg may import it; the library itself never
does.  It shares no code with the CUDA path.

What it follows (page = "02 · DeepSeek-V2 analysis", PaperTrace):
  * 1.2, eq 9-11 and the absorption paragraph: the cache holds the latent
    c^KV (d_c = 512 per token and layer); with W^UK absorbed into the query,
    every head's content query is a d_c-vector dotted directly with c_s.
  * 1.2, last paragraph: an RMSNorm follows the compressed latent (its extra
    scaling factors are not given; none is applied here).
  * 1.3, eq 14-15 and 18: a separate d_h^R-dim RoPE query per head and ONE
    RoPE key k^R shared by all heads, projected straight from h_t and cached
    already rotated; content and RoPE parts are concatenated and the score is
    divided by sqrt(d_h + d_h^R).
  * 1.3: 512 + 64 = 576 cached elements per token per layer.
  * 6.1: each head aggregates the latents with its own weights,
    u_{t,i} = sum_s a_{t,s,i} c_s in R^{d_c}; W^UV / W^O are applied after.
  * "walking one token through": the new token's 576 elements are appended,
    then scores = content part + RoPE part, scaled, softmax over the history.
RoPE itself (page "DeepSeek-V3 model structure", CSDN, section 2(3)):
position n rotates the dimension pairs (2i, 2i+1).

Readings where the pages are silent (each is also listed in the design
notes): RMSNorm eps = 1e-6 and gamma supplied by the caller; RoPE base
10000 with theta_i = base^(-2i/d_r) and the rotation
(x0 cos - x1 sin, x0 sin + x1 cos); query token j of a step with Q query
tokens sits at position len-Q+j and sees positions <= its own; a row that
sees no key gives out = 0, lse = -inf; lse is the natural log of the sum of
exp(scaled score).

Parity status: every function here is pinned by the CPU tests
(tests/test_oracle_*.py) against closed forms, invariants, the explicit
(un-absorbed) multi-head computation and the printed cache figures.
"""
from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (7 stored + the implicit one) and the
    float32 exponent range.  Returned as float64 holding the rounded value.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    small = finite & (np.abs(x) < 2.0 ** -126)
    normal = finite & ~small
    m, e = np.frexp(x[normal])                      # |m| in [0.5, 1)
    out[normal] = np.ldexp(np.rint(m * 256.0) / 256.0, e)   # np.rint = ties-to-even
    out[small] = np.rint(x[small] * 2.0 ** 133) * 2.0 ** -133
    over = normal & (np.abs(out) > float.fromhex("0x1.FEp127"))
    out[over] = np.copysign(np.inf, x[over])
    return out


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns of round_to_bf16(x)."""
    r = round_to_bf16(x).astype(np.float32)          # exact
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def round_to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------
# Append: RMSNorm on the latent, RoPE on the shared key, paged placement
# ----------------------------------------------------------------------------


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """y_k = x_k / sqrt(mean_k(x^2) + eps) * gamma_k over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def rope_theta(d_r: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d_r) for the pairs i < d_r/2."""
    i = np.arange(d_r // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / d_r)


def yarn_theta(d_r: int, base: float, factor: float, alpha: float, beta: float,
               original_max_position: int) -> np.ndarray:
    """RoPE frequencies after YaRN context extension.

    Page "02 · DeepSeek-V2 analysis", section 3.2: YaRN stretches the window
    from 4K to 128K (factor s = 40, alpha = 1, beta = 32) and, in MLA, acts
    only on the d_r RoPE dims.  The page defers the interpolation rule to
    YaRN itself; this is YaRN's by-parts rule: a pair that turns
    r = L * theta / (2 pi) times over the original window L keeps its
    frequency when r > beta, is divided by s when r < alpha, and in between
    blends the two with weight g = (r - alpha) / (beta - alpha).
    """
    theta = rope_theta(d_r, base)
    if factor == 1.0:
        return theta
    turns = float(original_max_position) * theta / (2.0 * math.pi)
    g = np.clip((turns - alpha) / (beta - alpha), 0.0, 1.0)
    return theta * g + (theta / factor) * (1.0 - g)


def yarn_temperature(factor: float, coef: float) -> float:
    """sqrt(1/t) = coef * ln(s) + 1 (section 3.2: coef 0.0707 in V2, 0.1 in YaRN)."""
    return coef * math.log(factor) + 1.0 if factor > 1.0 else 1.0


def yarn_softmax_scale(scale: float, factor: float, coef: float) -> float:
    """The temperature moved onto the softmax scale: the original scales q and
    k each by sqrt(1/t), i.e. the logits by 1/t = sqrt(1/t)^2 (section 3.2)."""
    m = yarn_temperature(factor, coef)
    return scale * m * m


def rope_angles(pos, d_r: int, base: float, theta=None) -> np.ndarray:
    """phi[..., i] = pos * theta_i for the pair (2i, 2i+1); theta_i = base^(-2i/d_r) unless given."""
    theta = rope_theta(d_r, base) if theta is None else np.asarray(theta, dtype=np.float64)
    return np.asarray(pos, dtype=np.float64)[..., None] * theta


def rope(x: np.ndarray, pos, base: float, theta=None) -> np.ndarray:
    """Rotate each dimension pair (2i, 2i+1) of x by the angle pos*theta_i."""
    x = np.asarray(x, dtype=np.float64)
    d_r = x.shape[-1]
    phi = rope_angles(pos, d_r, base, theta)
    c, s = np.cos(phi), np.sin(phi)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y


APPEND_RMSNORM = 1
APPEND_ROPE = 2


def append_rows(c_raw, k_raw, positions, gamma, eps, base, flags, cache_dtype, theta=None):
    """The 576-element cache rows [c_kv || k_R] of new tokens.

    c_raw [T, d_c] and k_raw [T, d_r] are the raw projections (already widened
    to float64).  The row is computed in float64 and rounded once to the
    cache dtype.  `theta` overrides the RoPE frequencies (YaRN).
    """
    c = np.asarray(c_raw, dtype=np.float64)
    k = np.asarray(k_raw, dtype=np.float64)
    if flags & APPEND_RMSNORM:
        c = rmsnorm(c, gamma, eps)
    if flags & APPEND_ROPE:
        k = rope(k, positions, base, theta)
    return round_to_dtype(np.concatenate([c, k], axis=-1), cache_dtype)


def page_slot(page_table: np.ndarray, seq_ids, positions, page_size: int):
    """Physical (page, slot) of token `positions` of sequence `seq_ids`."""
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    return page_table[seq_ids, positions // page_size].astype(np.int64), positions % page_size


def cache_write(pool: np.ndarray, page_table, seq_ids, positions, rows) -> None:
    """pool[page, slot, :] = row for every new token (pool: [pages, P, 576])."""
    page, slot = page_slot(page_table, seq_ids, positions, pool.shape[1])
    pool[page, slot, :] = rows


def cache_gather(pool: np.ndarray, page_table, b: int, length: int) -> np.ndarray:
    """Rows of tokens 0..length-1 of sequence b, in position order."""
    pos = np.arange(length)
    page, slot = page_slot(page_table, np.full(length, b), pos, pool.shape[1])
    return pool[page, slot, :]


# ----------------------------------------------------------------------------
# Decode: absorbed attention over the latent cache
# ----------------------------------------------------------------------------


def softmax_scale(d_h: int, d_r: int) -> float:
    """1 / sqrt(d_h + d_h^R): the per-head query/key width (eq 18), not d_c."""
    return 1.0 / math.sqrt(d_h + d_r)


def decode_row(C, R, qn, qr, scale: float):
    """One query token of one sequence, all heads.

    C [S, d_c] cached latents, R [S, d_r] cached rotated keys (the S visible
    tokens), qn [H, d_c] absorbed content queries, qr [H, d_r] rotated RoPE
    queries.  Returns (out [H, d_c], lse [H], weights [H, S]).
    """
    C = np.asarray(C, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    qn = np.asarray(qn, dtype=np.float64)
    qr = np.asarray(qr, dtype=np.float64)
    H = qn.shape[0]
    if C.shape[0] == 0:
        return np.zeros((H, C.shape[1])), np.full(H, -np.inf), np.zeros((H, 0))
    x = scale * (qn @ C.T + qr @ R.T)               # [H, S]  content + RoPE part
    m = x.max(axis=1, keepdims=True)
    w = np.exp(x - m)
    Z = w.sum(axis=1, keepdims=True)
    a = w / Z                                        # softmax over the history
    out = a @ C                                      # u = sum_s a_s c_s
    lse = (m + np.log(Z))[:, 0]
    return out, lse, a


def visible_length(length: int, Q: int, j: int) -> int:
    """Tokens seen by query j of Q when the sequence holds `length` tokens."""
    return max(0, int(length) - Q + j + 1)


def decode(C_of, R_of, q_nope, q_rope, lens, Q: int, scale: float):
    """Absorbed MLA decode for a batch.

    C_of(b) / R_of(b) return the cached latents / keys of sequence b in
    position order (at least lens[b] rows).  q_nope [B,Q,H,d_c],
    q_rope [B,Q,H,d_r].  Returns out [B,Q,H,d_c] and lse [B,Q,H] (float64).
    """
    B, Qq, H, d_c = q_nope.shape
    assert Qq == Q
    out = np.zeros((B, Q, H, d_c))
    lse = np.zeros((B, Q, H))
    for b in range(B):
        C = np.asarray(C_of(b), dtype=np.float64)
        R = np.asarray(R_of(b), dtype=np.float64)
        for j in range(Q):
            n = visible_length(lens[b], Q, j)
            o, l, _ = decode_row(C[:n], R[:n], q_nope[b, j], q_rope[b, j], scale)
            out[b, j], lse[b, j] = o, l
    return out, lse


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge softmax-normalised partial results of disjoint key ranges.

    o_parts [n, ..., d_c], lse_parts [n, ...]:  lse = ln sum_j exp(lse_j),
    out = sum_j exp(lse_j - lse) o_j.  Empty ranges carry lse = -inf.
    """
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lse_parts - m_safe)                   # exp(-inf) = 0
    Z = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, Z, 1.0)), -np.inf)
    scale = np.where(finite, 1.0 / np.where(finite, Z, 1.0), 0.0)
    out = np.einsum("n...,n...d->...d", w * scale, np.asarray(o_parts, dtype=np.float64))
    return out, lse


# ----------------------------------------------------------------------------
# The un-absorbed (expanded) multi-head form, for the absorption identity
# ----------------------------------------------------------------------------


def explicit_mha_row(C, R, qc, qr, W_UK, W_UV):
    """Per-head MHA with K and V expanded from the latent (eq 10-11, 14-18).

    C [S, d_c], R [S, d_r] (shared rotated key), qc [H, d_h] content queries,
    qr [H, d_r], W_UK / W_UV [H, d_h, d_c].  k_{s,h} = [W_UK_h c_s || R_s],
    v_{s,h} = W_UV_h c_s, score divided by the square root of the key width.
    Returns o [H, d_h].
    """
    H = qc.shape[0]
    outs = []
    for h in range(H):
        K = np.concatenate([C @ W_UK[h].T, R], axis=1)           # [S, d_h + d_r]
        V = C @ W_UV[h].T                                        # [S, d_h]
        q = np.concatenate([qc[h], qr[h]])
        x = (K @ q) / math.sqrt(K.shape[1])
        w = np.exp(x - x.max())
        outs.append((w / w.sum()) @ V)
    return np.stack(outs)


def prefill_expanded(C, R, qc, qr, W_UK, W_UV, positions, scale=None):
    """Expanded (prefill) form of the same attention (section 1.2 eq 10-11,
    1.3 eq 14-18; section 6: prefill materialises K and V, decode absorbs).

    Per head h the keys k_{s,h} = [W_UK_h c_s || R_s] and values
    v_{s,h} = W_UV_h c_s of the whole sequence are materialised; query t
    (content qc[t, h], RoPE part qr[t, h], at position positions[t]) attends
    causally to the keys at positions 0..positions[t], scores divided by
    sqrt(d_h + d_r) unless `scale` is given.
    C [S, d_c], R [S, d_r], qc [T, H, d_h], qr [T, H, d_r], W_UK / W_UV
    [H, d_h, d_c].  Returns o [T, H, d_h] and lse [T, H] (natural log of the
    sum of exp(scaled score); -inf for a query that sees no key).
    """
    C = np.asarray(C, dtype=np.float64)
    R = np.asarray(R, dtype=np.float64)
    qc = np.asarray(qc, dtype=np.float64)
    qr = np.asarray(qr, dtype=np.float64)
    T, H, d_h = qc.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d_h + R.shape[1])
    K_c = np.einsum("sc,hdc->hsd", C, W_UK)                    # [H, S, d_h]
    V = np.einsum("sc,hdc->hsd", C, W_UV)                      # [H, S, d_h]
    x = (np.einsum("thd,hsd->ths", qc, K_c) + np.einsum("thr,sr->ths", qr, R)) * scale
    visible = np.arange(C.shape[0])[None, :] <= np.asarray(positions)[:, None]      # [T, S]
    x = np.where(visible[:, None, :], x, -np.inf)
    m = np.max(x, axis=2, keepdims=True)
    any_key = np.isfinite(m)
    w = np.exp(x - np.where(any_key, m, 0.0))
    z = w.sum(axis=2, keepdims=True)
    o = np.einsum("ths,hsd->thd", w / np.where(any_key, z, 1.0), V)
    lse = np.where(any_key[..., 0], (m + np.log(np.where(any_key, z, 1.0)))[..., 0], -np.inf)
    return o, lse


def absorb_query(W_UK, q_c):
    """W^UK absorbed into the query (section 1.2, the absorption paragraph):
    q_nope[..., h, :] = W^UK_h^T q^C_h, so that q_h^T k_{s,h} = q_nope_h^T c_s.

    W_UK [H, d_h, d_c] (k^C_{s,h} = W_UK[h] @ c_s), q_c [..., H, d_h].
    Returns [..., H, d_c] (float64).
    """
    return np.einsum("hdc,...hd->...hc", np.asarray(W_UK, dtype=np.float64), np.asarray(q_c, dtype=np.float64))


def absorb_output(W_UV, u):
    """W^UV applied after the latent aggregation (section 6.1): each head
    first aggregates the latents, u_h = sum_s a_{s,h} c_s, then
    o_h = W^UV_h u_h.

    W_UV [H, d_h, d_c] (v_{s,h} = W_UV[h] @ c_s), u [..., H, d_c].
    Returns [..., H, d_h] (float64).
    """
    return np.einsum("hdc,...hc->...hd", np.asarray(W_UV, dtype=np.float64), np.asarray(u, dtype=np.float64))


# ----------------------------------------------------------------------------
# Cache accounting (section 1.1, 1.3 and 6.2 of the DeepSeek-V2 analysis page)
# ----------------------------------------------------------------------------


def mla_elements_per_token_layer(d_c: int, d_r: int, per_head_rope_heads: int = 0) -> int:
    """c^KV plus the shared RoPE key (or one RoPE key per head if asked)."""
    return d_c + d_r * (per_head_rope_heads if per_head_rope_heads else 1)


def mha_elements_per_token_layer(kv_heads: int, d_h: int) -> int:
    """Standard MHA/GQA: K and V per KV head, 2 n_h d_h."""
    return 2 * kv_heads * d_h


def cache_bytes(elements_per_token_layer: int, layers: int, tokens: int, bits: int) -> float:
    return elements_per_token_layer * layers * tokens * bits / 8.0
