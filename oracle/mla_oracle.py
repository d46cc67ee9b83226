"""CPU oracle for absorbed Multi-Head Latent Attention (MLA) decode.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline may import this module.  It shares no code with the CUDA library and
must never be called by the product path.

Plain, slow and fp64 throughout: every input is converted to float64 and every
intermediate stays float64, except where the method itself stores a value in the
cache's element type (the appended latent row is rounded to bf16 for bf16
caches).  numpy's matmul is the only library primitive used as a step.

Notation (column vectors, as in "Grouped-query and latent attention", section
"Multi-head latent attention"):

* ``c = W_DKV h`` is the latent (d_c numbers) that the cache keeps per token.
* ``k_R = RoPE(W_KR h, pos)`` is ONE rotary key per token shared by every head
  ("MLA storage", section "Storing a positional key separately").
* per head i, ``W_UK^(i), W_UV^(i)`` are the rows i*d_h .. (i+1)*d_h-1 of
  ``W_UK, W_UV`` (shape (n_h*d_h) x d_c); arrays here are shaped [n_h, d_h, d_c].
* a cache row is ``[c ; k_R]``, d_c + d_r elements ("DeepSeek MLA: 4 Attention
  Methods Compared", section "Decoupled RoPE": 512 + 64 = 576 values).
* score ``s_ij = [q_C,i ; q_R,i] . [k_C,ij ; k_R,j] / sqrt(d_h + d_r)``
  ("Grouped-query and latent attention", section "Why a separate rotary key").

Readings of points the pages leave open (each also listed in the design notes):

* RoPE pairs dimensions (2k, 2k+1) with angle pos * base^(-2k/d_r); the pages
  refer to a chapter on rotary embeddings that is not among them.
* The query of a sequence with n cached rows (new token included) sits at
  position n-1 and attends over all n rows, itself included.
* No normalisation is applied to latents or rotary parts.
* An empty sequence (n < 1) has no defined output; the oracle raises.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "f64", "round_to_bf16", "rope_inverse_frequencies", "rope", "append_rows",
    "expand_heads", "full_keys", "decode_explicit", "decode_absorbed",
    "project_query", "project_out", "project_output", "merge_output_weights",
    "project_output_merged", "softmax_scale", "cache_elements_per_token", "cache_bytes",
    "E4M3_MAX", "FP8_GROUP", "round_to_e4m3", "e4m3_value", "quantize_row_fp8", "dequantize_row_fp8",
]


def f64(x) -> np.ndarray:
    """A float64 numpy copy of a numpy array or a CPU torch tensor (any float dtype)."""
    if hasattr(x, "detach"):                      # torch tensor: bf16/fp32 widen exactly
        import torch  # local import: the oracle's arithmetic needs only numpy
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.array(x, dtype=np.float64, copy=True)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps the float32 exponent and the top 7 fraction bits.  Starting from
    float64 (52 fraction bits) that means dropping the low 45 bits with
    round-to-nearest-even.  Valid for finite values inside bf16's normal range.
    """
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    u = a.view(np.uint64)
    drop = np.uint64(45)
    lsb = (u >> drop) & np.uint64(1)
    half_minus_one = np.uint64((1 << 44) - 1)
    r = (u + half_minus_one + lsb) & ~np.uint64((1 << 45) - 1)
    return r.view(np.float64).reshape(a.shape)


def softmax_scale(d_h: int, d_r: int) -> float:
    """1/sqrt(d_h + d_r): "Grouped-query and latent attention", section
    "Why a separate rotary key" (scores scaled by 1/sqrt(128 + 64))."""
    return 1.0 / math.sqrt(d_h + d_r)


def rope_inverse_frequencies(d_r: int, base: float) -> np.ndarray:
    """theta_k = base^(-2k/d_r), k = 0 .. d_r/2 - 1 (reading: standard RoPE)."""
    if d_r % 2:
        raise ValueError("rotary width must be even")
    k = np.arange(d_r // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * k / d_r)


def rope(x, pos, base: float) -> np.ndarray:
    """Rotate each pair (x_2k, x_2k+1) of the last axis by the angle pos*theta_k.

    ``pos`` broadcasts against ``x[..., 0]``.  RoPE rotates by a position
    dependent angle ("DeepSeek MLA: 4 Attention Methods Compared", section "Why
    RoPE complicates MLA"); the pairing is this build's reading.
    """
    x = np.asarray(x, dtype=np.float64)
    theta = rope_inverse_frequencies(x.shape[-1], base)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    cs, sn = np.cos(ang), np.sin(ang)
    even, odd = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (x.shape[-1],)))
    out[..., 0::2] = even * cs - odd * sn
    out[..., 1::2] = even * sn + odd * cs
    return out


def append_rows(h, w_dkv, w_kr, positions, base: float, cache_bf16: bool) -> np.ndarray:
    """Latent cache rows [n, d_c + d_r] for tokens ``h`` [n, hidden] at ``positions`` [n].

    c = W_DKV h ("Grouped-query and latent attention", section "Multi-head
    latent attention"), k_R = RoPE(W_KR h, pos) (same page, "Why a separate
    rotary key"), stored side by side as one row ("MLA storage", section
    "Storing a positional key separately": [1, 2, 3, r0, r1]).  The row is then
    held in the cache's element type.
    """
    h = f64(h)
    c = h @ f64(w_dkv).T
    k_r = rope(h @ f64(w_kr).T, np.asarray(positions), base)
    row = np.concatenate([c, k_r], axis=-1)
    return round_to_bf16(row) if cache_bf16 else row


def expand_heads(c, w_uk, w_uv):
    """Explicit per-head content keys and values from latents.

    k_C,ij = W_UK^(i) c_j and v_C,ij = W_UV^(i) c_j ("MLA storage", section
    "Forming head-specific K and V from a small vector"; "Grouped-query and
    latent attention", section "Multi-head latent attention").
    Returns (k_c, v), each [n_rows, n_h, d_h].
    """
    c = f64(c)
    w_uk, w_uv = f64(w_uk), f64(w_uv)
    n_h = w_uk.shape[0]
    k_c = np.stack([c @ w_uk[i].T for i in range(n_h)], axis=1)
    v = np.stack([c @ w_uv[i].T for i in range(n_h)], axis=1)
    return k_c, v


def full_keys(rows, w_uk, d_c: int) -> np.ndarray:
    """Full per-head keys [k_C,ij ; k_R,j], [n_rows, n_h, d_h + d_r].

    Concatenated, not added; the rotary part is the same for every head ("MLA
    storage", section "Two paths for forming keys and values").
    """
    rows = f64(rows)
    c, k_r = rows[:, :d_c], rows[:, d_c:]
    k_c, _ = expand_heads(c, w_uk, np.zeros_like(f64(w_uk)))
    n_h = k_c.shape[1]
    return np.concatenate([k_c, np.broadcast_to(k_r[:, None, :], (k_r.shape[0], n_h, k_r.shape[1]))],
                          axis=-1)


def _check_rows(rows):
    if rows.shape[0] < 1:
        raise ValueError("a sequence needs at least one cached row")


def decode_explicit(q_c, q_r, w_uk, w_uv, rows, base: float, scale=None) -> dict:
    """Decode one query against one sequence WITHOUT absorption.

    Materialises every head's full keys and values from the cached latents,
    then applies softmax attention for the new token ("The Journey to
    Multi-Head Latent Attention", section "The KV cache": the attention row is
    Softmax(Q_last K^T) and the context is that row times V).

    q_c [n_h, d_h]; q_r [n_h, d_r] not yet rotated; rows [n, d_c + d_r].
    Returns o [n_h, d_h], o_lat [n_h, d_c] (= sum_j a_ij c_j), lse [n_h]
    (natural log of sum_j exp(s_ij)) and the attention weights a [n_h, n].
    """
    rows = f64(rows)
    _check_rows(rows)
    q_c, q_r = f64(q_c), f64(q_r)
    n_h, d_h, d_c = f64(w_uk).shape
    d_r = q_r.shape[-1]
    if scale is None:
        scale = softmax_scale(d_h, d_r)
    n = rows.shape[0]
    p = n - 1                                        # the new token's own position
    w_uk, w_uv = f64(w_uk), f64(w_uv)
    q_rot = rope(q_r, p, base)
    o = np.zeros((n_h, d_h))
    o_lat = np.zeros((n_h, d_c))
    lse = np.zeros(n_h)
    a_all = np.zeros((n_h, n))
    for i in range(n_h):                             # one head's K and V at a time (memory)
        keys = full_keys(rows, w_uk[i:i + 1], d_c)[:, 0, :]                   # [n, d_h + d_r]
        values = expand_heads(rows[:, :d_c], w_uk[i:i + 1], w_uv[i:i + 1])[1][:, 0, :]  # [n, d_h]
        q = np.concatenate([q_c[i], q_rot[i]])
        s = keys @ q * scale
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        a = e / l
        o[i] = a @ values
        o_lat[i] = a @ rows[:, :d_c]
        lse[i] = m + math.log(l)
        a_all[i] = a
    return {"o": o, "o_lat": o_lat, "lse": lse, "a": a_all}


def decode_absorbed(q_c, q_r, w_uk, w_uv, rows, base: float, scale=None) -> dict:
    """Decode one query with both absorptions, written independently of
    ``decode_explicit``.

    Key side: q'_i = W_UK^(i)T q_C,i and q_C,i . (W_UK^(i) c_j) = q'_i . c_j.
    Value side: sum_j a_ij W_UV^(i) c_j = W_UV^(i) (sum_j a_ij c_j)
    ("Grouped-query and latent attention", section "The absorption trick").
    """
    rows = f64(rows)
    _check_rows(rows)
    q_c, q_r, w_uk, w_uv = f64(q_c), f64(q_r), f64(w_uk), f64(w_uv)
    n_h, d_h, d_c = w_uk.shape
    d_r = q_r.shape[-1]
    if scale is None:
        scale = softmax_scale(d_h, d_r)
    n = rows.shape[0]
    c, k_r = rows[:, :d_c], rows[:, d_c:]
    q_fold = np.einsum("hdc,hd->hc", w_uk, q_c)      # [n_h, d_c]
    q_rot = rope(q_r, n - 1, base)                    # [n_h, d_r]
    s = (c @ q_fold.T + k_r @ q_rot.T) * scale        # [n, n_h]
    m = s.max(axis=0)
    e = np.exp(s - m)
    l = e.sum(axis=0)
    a = e / l                                         # [n, n_h]
    o_lat = a.T @ c                                   # [n_h, d_c]
    o = np.einsum("hdc,hc->hd", w_uv, o_lat)
    return {"o": o, "o_lat": o_lat, "lse": m + np.log(l), "a": a.T}


def project_query(x, w_uq, w_qr, n_h: int, w_dq=None):
    """Per-head query parts from a token's input: c_q = W_DQ h (c_q = h when no
    W_DQ is given), q_C = W_UQ c_q, q_R = W_QR c_q before rotation
    ("Grouped-query and latent attention", sections "Multi-head latent
    attention" and "Why a separate rotary key").  x [..., in]; returns
    (q_c [..., n_h, d_h], q_r [..., n_h, d_r])."""
    x = f64(x)
    c_q = x if w_dq is None else x @ f64(w_dq).T
    q_c = c_q @ f64(w_uq).T
    q_r = c_q @ f64(w_qr).T
    return (q_c.reshape(*q_c.shape[:-1], n_h, -1), q_r.reshape(*q_r.shape[:-1], n_h, -1))


def project_out(o_lat, w_uv) -> np.ndarray:
    """o_i = W_UV^(i) o_lat_i for every head: [..., n_h, d_c] -> [..., n_h, d_h]."""
    return np.einsum("hdc,...hc->...hd", f64(w_uv), f64(o_lat))


def project_output(o, w_o) -> np.ndarray:
    """The layer output u = W_O [o_1 ; ... ; o_n_h]: the heads' outputs side by side, then
    the output matrix.  o [..., n_h, d_h], W_O [hidden, n_h*d_h] -> u [..., hidden]."""
    o = f64(o)
    return o.reshape(*o.shape[:-2], -1) @ f64(w_o).T


def merge_output_weights(w_o, w_uv) -> np.ndarray:
    """W_UV merged into W_O ("Grouped-query and latent attention", section "The absorption
    trick"): W_OV^(i) = W_O^(i) W_UV^(i), W_O^(i) being the d_h columns of head i.
    W_O [hidden, n_h*d_h], W_UV [n_h, d_h, d_c] -> [n_h, hidden, d_c]."""
    w_o, w_uv = f64(w_o), f64(w_uv)
    n_h, d_h, _ = w_uv.shape
    return np.stack([w_o[:, i * d_h:(i + 1) * d_h] @ w_uv[i] for i in range(n_h)])


def project_output_merged(o_lat, w_ov) -> np.ndarray:
    """u = sum_i W_OV^(i) o_lat_i: o_lat [..., n_h, d_c], W_OV [n_h, hidden, d_c]."""
    return np.einsum("hmc,...hc->...m", f64(w_ov), f64(o_lat))


def cache_elements_per_token(kind: str, *, n_h: int = 0, d_h: int = 0, n_g: int = 0,
                             d_c: int = 0, d_r: int = 0) -> int:
    """Cached values per token per layer for each attention design
    ("Grouped-query and latent attention", section "Multi-head latent
    attention": MHA 2 n_h d_h, GQA 2 n_g d_h, MQA 2 d_h, MLA d_c + d_R)."""
    if kind == "mha":
        return 2 * n_h * d_h
    if kind == "gqa":
        return 2 * n_g * d_h
    if kind == "mqa":
        return 2 * d_h
    if kind == "mla":
        return d_c + d_r
    raise ValueError(kind)


def cache_bytes(elements_per_token: int, tokens: int, layers: int, bytes_per_value: int) -> int:
    """Whole-cache bytes for one request ("DeepSeek MLA: 4 Attention Methods
    Compared", section "DeepSeek KV-cache memory comparison")."""
    return elements_per_token * tokens * layers * bytes_per_value


# ---------------------------------------------------------------- fp8 latent cache
# The pages name quantization among the things a cache layout may add ("DeepSeek MLA: 4
# Attention Methods Compared", section "Memory savings do not automatically equal
# latency savings") without fixing a format.  Reading taken here (the plainest one that
# keeps the method's arithmetic): the latent part c of a row is stored as FP8 E4M3 codes
# in groups of 128 columns, each group with one scale, a power of two stored as fp32 (the
# smallest 2^k with largest magnitude / 2^k <= 448, as in microscaling formats), so that
# code * scale is exact in bf16 as well; the rotary part k_R stays bf16, since it is small
# and carries the position.  A value is code * scale.

E4M3_MAX = 448.0
FP8_GROUP = 128


def round_to_e4m3(x) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value, ties to even.

    E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits, no infinities.  Normal
    values 2^e (1 + f/8) for e in [-6, 8] (the largest finite, 2^8 * 1.75 = 448);
    subnormals k 2^-9 for k = 1..7.  In the binade [2^e, 2^(e+1)) the spacing is 2^(e-3)
    (below 2^-6 it stays 2^-9), so a value rounds to step * round_half_even(|x| / step).
    Magnitudes above 448 saturate to 448.
    """
    a = np.asarray(x, dtype=np.float64)
    m = np.abs(a)
    _, p = np.frexp(np.where(m > 0, m, 1.0))        # m = f 2^p with f in [0.5, 1): binade e = p - 1
    e = np.clip(p - 1, -6, 8)
    step = np.ldexp(1.0, e - 3)
    v = np.minimum(np.round(m / step) * step, E4M3_MAX)   # np.round: half to even
    return np.copysign(v, a)


def e4m3_value(codes) -> np.ndarray:
    """The value of FP8 E4M3 codes (uint8): sign s, exponent field E, fraction F give
    (-1)^s 2^(E-7) (1 + F/8) for E > 0 and (-1)^s F 2^-9 for E = 0; codes 0x7F and 0xFF
    (E = 15, F = 7) are NaN."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s, e, f = b >> 7, (b >> 3) & 15, b & 7
    v = np.where(e > 0, np.ldexp(1.0 + f / 8.0, e - 7), np.ldexp(f.astype(np.float64), -9))
    v = np.where((e == 15) & (f == 7), np.nan, v)
    return np.where(s == 1, -v, v)


def quantize_row_fp8(row, d_c: int, group: int = FP8_GROUP):
    """A cache row [..., d_c + d_r] -> (values [..., d_c] on the E4M3 grid, scales
    [..., d_c / group], rotary part [..., d_r] in bf16); value * scale is the stored latent.

    The decisions are taken in fp32, the precision of the kernel that writes the cache:
    q = fp32(amax) / 448 (an fp32 division), scale = 2^k with k the smallest integer such
    that q <= 2^k (exact: from q's binary exponent), then c / scale (exact: a power of two)
    rounded to E4M3.  A group of zeros gets scale 1.
    """
    r = f64(row)
    c32 = r[..., :d_c].astype(np.float32)
    g = c32.reshape(c32.shape[:-1] + (d_c // group, group))
    amax = np.max(np.abs(g), axis=-1)
    q = (amax / np.float32(E4M3_MAX)).astype(np.float32).astype(np.float64)
    m, e = np.frexp(np.where(q > 0, q, 1.0))          # q = m 2^e, m in [0.5, 1)
    k = np.where(m == 0.5, e - 1, e)                   # q == 2^(e-1) exactly: that power itself
    scale = np.where(q > 0, np.ldexp(1.0, k), 1.0)
    y = g.astype(np.float64) / scale[..., None]
    vals = round_to_e4m3(y).reshape(c32.shape)
    return vals, scale, round_to_bf16(r[..., d_c:])


def dequantize_row_fp8(values, scales, k_r, group: int = FP8_GROUP) -> np.ndarray:
    """Rows [..., d_c + d_r] from quantize_row_fp8's parts: [values * scale ; k_R]."""
    v = f64(values)
    s = np.repeat(f64(scales), group, axis=-1)
    return np.concatenate([v * s, f64(k_r)], axis=-1)
