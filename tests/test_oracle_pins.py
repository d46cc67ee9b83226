"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each ``pin_*`` function raises AssertionError on a mismatch.  The tests run
them against the oracle as written, then plant plausible mistakes in the oracle
(on the CPU, by monkeypatching) and check that some pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.mla_oracle as mo

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _worked_example_weights():
    g = _load("mla_storage_worked_example.json")
    # column convention: W_UK^(i) = U_iK^T, stacked as [n_h, d_h, d_c]
    w_uk = np.stack([np.array(g["U_K"][h], float).T for h in ("1", "2")])
    w_uv = np.stack([np.array(g["U_V"][h], float).T for h in ("1", "2")])
    return g, w_uk, w_uv


# --------------------------------------------------------------------------- pins

def pin_worked_example_heads():
    """c = [1,2,3] gives head-1 k = [1,2], v = [4,2] and head-2 k = [2,3], v = [1,5]."""
    g, w_uk, w_uv = _worked_example_weights()
    k, v = mo.expand_heads(np.array([g["c"]], float), w_uk, w_uv)
    for i, h in enumerate(("1", "2")):
        assert np.array_equal(k[0, i], g["expected_k"][h]), (h, k[0, i])
        assert np.array_equal(v[0, i], g["expected_v"][h]), (h, v[0, i])


def pin_full_key_concat():
    """Full key = [content key ; shared rotary key]: [1,2,r0,r1] and [2,3,r0,r1]."""
    g, w_uk, _ = _worked_example_weights()
    r0, r1 = 0.25, -0.5
    row = np.array([g["c"] + [r0, r1]], float)
    assert row.shape[1] == g["cache_row_components"]
    keys = mo.full_keys(row, w_uk, g["latent_dim"])
    assert keys.shape == (1, 2, g["head_dim"] + g["rope_dim"])
    assert np.array_equal(keys[0, 0], [1, 2, r0, r1])
    assert np.array_equal(keys[0, 1], [2, 3, r0, r1])


def pin_single_row_decode():
    """One cached row at position 0: softmax weight 1, so o = v_0, o_lat = c_0 and
    lse = the only score.  Head 1 of the worked example with q_C = [1,1],
    q_R = [2,1], k_R = [0.5,-1]: score (3 + 0) / sqrt(2 + 2) = 1.5."""
    g, w_uk, w_uv = _worked_example_weights()
    rows = np.array([g["c"] + [0.5, -1.0]], float)
    q_c = np.array([[1.0, 1.0], [0.0, 0.0]])
    q_r = np.array([[2.0, 1.0], [0.0, 0.0]])
    for dec in (mo.decode_explicit, mo.decode_absorbed):
        r = dec(q_c, q_r, w_uk, w_uv, rows, 10000.0)
        assert abs(r["lse"][0] - 1.5) < 1e-14, r["lse"]
        assert np.allclose(r["o"][0], [4, 2], atol=1e-14)
        assert np.allclose(r["o_lat"][0], g["c"], atol=1e-14)
        assert abs(r["lse"][1] - 0.0) < 1e-14        # head 2 has a zero query: score 0


def pin_two_rows_content():
    """Content-only scores with the worked example's head 1: rows c0=[1,2,3],
    c1=[2,0,1] give keys [1,2], [2,0] and values [4,2], [3,0]; with q_C=[1,0]
    the scores are [1,2]/2, so a0 = 1/(1+e^0.5)."""
    _, w_uk, w_uv = _worked_example_weights()
    rows = np.array([[1, 2, 3, 0, 0], [2, 0, 1, 0, 0]], float)
    q_c = np.array([[1.0, 0.0], [0.0, 0.0]])
    q_r = np.zeros((2, 2))
    a0 = 1.0 / (1.0 + math.exp(0.5))
    a1 = 1.0 - a0
    for dec in (mo.decode_explicit, mo.decode_absorbed):
        r = dec(q_c, q_r, w_uk, w_uv, rows, 10000.0)
        assert np.allclose(r["o"][0], a0 * np.array([4, 2]) + a1 * np.array([3, 0]), atol=1e-14)
        assert np.allclose(r["o_lat"][0], a0 * rows[0, :3] + a1 * rows[1, :3], atol=1e-14)
        assert abs(r["lse"][0] - math.log(math.exp(0.5) + math.exp(1.0))) < 1e-14
        assert np.allclose(r["o_lat"][1], rows[:, :3].mean(0), atol=1e-14)  # zero query: uniform


def pin_rotary_query_position():
    """Two rows, rotary term only (d_r = 2, so theta_0 = 1 whatever the base).
    Row 0 holds k_R = [1,0] (position 0), row 1 holds [cos 1, sin 1] (position 1).
    The query sits at position 1, so q_R = [0,1] rotates to [-sin 1, cos 1]:
    scores are -sin(1)/2 and 0 (scale 1/sqrt(2+2))."""
    _, w_uk, w_uv = _worked_example_weights()
    rows = np.array([[0, 0, 0, 1.0, 0.0], [0, 0, 0, math.cos(1.0), math.sin(1.0)]])
    q_c = np.zeros((2, 2))
    q_r = np.array([[0.0, 1.0], [1.0, 0.0]])
    s0 = -math.sin(1.0) / 2.0
    # head 2: q_R = [1,0] rotates to [cos 1, sin 1]: scores cos(1)/2 and 1/2
    t0, t1 = math.cos(1.0) / 2.0, 0.5
    for dec in (mo.decode_explicit, mo.decode_absorbed):
        r = dec(q_c, q_r, w_uk, w_uv, rows, 10000.0)
        assert abs(r["lse"][0] - math.log(math.exp(s0) + 1.0)) < 1e-14, r["lse"]
        assert abs(r["lse"][1] - math.log(math.exp(t0) + math.exp(t1))) < 1e-14, r["lse"]
        assert abs(r["a"][0][0] - 1.0 / (1.0 + math.exp(-s0))) < 1e-14


def pin_identical_rows():
    """n identical rows: uniform weights, o = W_UV c, lse = s + log n."""
    rng = np.random.default_rng(5)
    n_h, d_h, d_c, d_r, n = 3, 4, 6, 2, 7
    w_uk, w_uv = rng.normal(size=(n_h, d_h, d_c)), rng.normal(size=(n_h, d_h, d_c))
    c = rng.normal(size=d_c)
    rows = np.tile(np.concatenate([c, [0.0, 0.0]]), (n, 1))
    q_c, q_r = rng.normal(size=(n_h, d_h)), np.zeros((n_h, d_r))
    for dec in (mo.decode_explicit, mo.decode_absorbed):
        r = dec(q_c, q_r, w_uk, w_uv, rows, 10000.0)
        for i in range(n_h):
            s = float(q_c[i] @ (w_uk[i] @ c)) / math.sqrt(d_h + d_r)
            assert abs(r["lse"][i] - (s + math.log(n))) < 1e-12
            assert np.allclose(r["o"][i], w_uv[i] @ c, atol=1e-12)
            assert np.allclose(r["a"][i], 1.0 / n, atol=1e-15)


def pin_dominant_row():
    """A row whose score exceeds the others by ~1000 takes all the weight."""
    _, w_uk, w_uv = _worked_example_weights()
    rows = np.array([[1, 2, 3, 0, 0], [2000, 0, 0, 0, 0], [0, 1, 1, 0, 0]], float)
    q_c = np.array([[1.0, 0.0], [0.0, 0.0]])
    for dec in (mo.decode_explicit, mo.decode_absorbed):
        r = dec(q_c, np.zeros((2, 2)), w_uk, w_uv, rows, 10000.0)
        assert np.allclose(r["o"][0], [2000, 0], rtol=0, atol=1e-9)
        assert np.allclose(r["a"][0], [0, 1, 0], atol=1e-12)


def pin_absorption_invariant():
    """Explicit (K/V materialised) and absorbed decodes agree to fp64 rounding
    ("Grouped-query and latent attention", section "The absorption trick")."""
    rng = np.random.default_rng(11)
    for (n_h, d_h, d_c, d_r, n) in [(2, 2, 3, 2, 1), (3, 5, 7, 4, 9), (4, 16, 32, 8, 33), (2, 3, 2, 6, 5)]:
        w_uk, w_uv = rng.normal(size=(n_h, d_h, d_c)), rng.normal(size=(n_h, d_h, d_c))
        rows = rng.normal(size=(n, d_c + d_r))
        q_c, q_r = rng.normal(size=(n_h, d_h)), rng.normal(size=(n_h, d_r))
        e = mo.decode_explicit(q_c, q_r, w_uk, w_uv, rows, 500.0)
        a = mo.decode_absorbed(q_c, q_r, w_uk, w_uv, rows, 500.0)
        for key in ("o", "o_lat", "lse", "a"):
            assert np.max(np.abs(e[key] - a[key])) <= 1e-10, (key, n_h, d_h, d_c, d_r, n)


def pin_rope_closed_forms():
    """RoPE: identity at position 0; a 2-D pair turns by pos radians (theta_0 = 1);
    the second pair of a width-4 key turns by pos * base^(-1/2); norms are
    kept; dot products depend only on the position difference."""
    x = np.array([0.3, -1.2, 2.0, 0.7])
    assert np.array_equal(mo.rope(x, 0, 10000.0), x)
    assert np.allclose(mo.rope([1.0, 0.0], 1, 10000.0), [math.cos(1), math.sin(1)], atol=1e-15)
    assert np.allclose(mo.rope([0.0, 1.0], 1, 10000.0), [-math.sin(1), math.cos(1)], atol=1e-15)
    assert np.allclose(mo.rope([0, 0, 1.0, 0], 100, 10000.0), [0, 0, math.cos(1), math.sin(1)], atol=1e-13)
    assert np.allclose(mo.rope([0, 0, 1.0, 0], 3, 16.0), [0, 0, math.cos(0.75), math.sin(0.75)], atol=1e-15)
    rng = np.random.default_rng(3)
    q, k = rng.normal(size=8), rng.normal(size=8)
    for m, n, d in [(5, 2, 17), (131071, 7, 1000)]:
        assert abs(np.linalg.norm(mo.rope(q, m, 10000.0)) - np.linalg.norm(q)) < 1e-12
        lhs = mo.rope(q, m, 10000.0) @ mo.rope(k, n, 10000.0)
        rhs = mo.rope(q, m + d, 10000.0) @ mo.rope(k, n + d, 10000.0)
        assert abs(lhs - rhs) < 1e-9


def pin_append_closed_form():
    """With W_DKV = [I | 0] and W_KR = [0 | I] the row is [h_c ; h_r turned by pos]."""
    d_c, d_r = 3, 2
    w_dkv = np.hstack([np.eye(d_c), np.zeros((d_c, d_r))])
    w_kr = np.hstack([np.zeros((d_r, d_c)), np.eye(d_r)])
    h = np.array([[1.0, 2.0, 3.0, 1.0, 0.0], [4.0, 5.0, 6.0, 0.0, 2.0]])
    rows = mo.append_rows(h, w_dkv, w_kr, [0, 2], 10000.0, cache_bf16=False)
    assert np.allclose(rows[0], [1, 2, 3, 1, 0], atol=1e-15)
    assert np.allclose(rows[1], [4, 5, 6, -2 * math.sin(2), 2 * math.cos(2)], atol=1e-15)


def pin_query_and_out_projections():
    """q_C = W_UQ h, q_R = W_QR h reshaped per head; o_i = W_UV^(i) o_lat_i
    (the worked example's value projection applied to c = [1,2,3])."""
    g, _, w_uv = _worked_example_weights()
    o = mo.project_out(np.array([g["c"], g["c"]], float), w_uv)
    assert np.array_equal(o, [g["expected_v"]["1"], g["expected_v"]["2"]])
    w_uq = np.arange(12, dtype=float).reshape(4, 3)        # 2 heads x d_h 2, input 3
    w_qr = -np.eye(4, 3)
    q_c, q_r = mo.project_query(np.array([1.0, 0.0, 2.0]), w_uq, w_qr, 2)
    assert np.array_equal(q_c, [[4, 13], [22, 31]])
    assert np.array_equal(q_r, [[-1, 0], [-2, 0]])


def pin_query_latent_projection():
    """With a query down-projection the query parts come from c_q = W_DQ h ("Grouped-query
    and latent attention", section "Multi-head latent attention"): here W_DQ picks h_0 and
    h_2, so c_q = [1, 3]; W_UQ (2 heads of width 1) and W_QR (2 heads of width 2) are
    integer matrices with hand-computed products."""
    h = np.array([1.0, 7.0, 3.0, -5.0])
    w_dq = np.array([[1.0, 0.0, 0.0, 0.0], [0.0, 0.0, 1.0, 0.0]])
    w_uq = np.array([[1.0, 0.0], [0.0, 2.0]])
    w_qr = np.array([[1.0, 1.0], [0.0, 1.0], [2.0, 0.0], [0.0, 0.0]])
    q_c, q_r = mo.project_query(h, w_uq, w_qr, 2, w_dq=w_dq)
    assert np.array_equal(q_c, [[1.0], [6.0]])
    assert np.array_equal(q_r, [[4.0, 3.0], [2.0, 0.0]])
    # a batch of tokens is projected row by row
    q_c2, q_r2 = mo.project_query(np.stack([h, 2 * h]), w_uq, w_qr, 2, w_dq=w_dq)
    assert np.array_equal(q_c2[1], 2 * q_c) and np.array_equal(q_r2[1], 2 * q_r)


def pin_output_projection_and_merge():
    """u = W_O [o_1; o_2] with the worked example's value projections; W_UV merged into W_O
    gives the same u straight from the latents (hand-computed integers), and the merged
    and two-step forms agree on random shapes."""
    g, _, w_uv = _worked_example_weights()                # 2 heads, d_h 2, d_c 3
    c = np.array(g["c"], float)                           # [1, 2, 3]
    w_o = np.array([[1.0, 0.0, 0.0, 1.0], [0.0, 2.0, 1.0, 0.0]])   # hidden 2, n_h*d_h 4
    o = mo.project_out(np.array([c, c]), w_uv)            # [[4, 2], [1, 5]]
    u = mo.project_output(o, w_o)
    assert np.array_equal(u, [4 + 5, 2 * 2 + 1])
    w_ov = mo.merge_output_weights(w_o, w_uv)
    assert w_ov.shape == (2, 2, 3)
    assert np.array_equal(mo.project_output_merged(np.array([c, c]), w_ov), u)
    rng = np.random.default_rng(5)
    w_o = rng.normal(size=(6, 3 * 4))
    w_uv = rng.normal(size=(3, 4, 5))
    o_lat = rng.normal(size=(2, 3, 5))
    two_step = mo.project_output(mo.project_out(o_lat, w_uv), w_o)
    merged = mo.project_output_merged(o_lat, mo.merge_output_weights(w_o, w_uv))
    assert np.allclose(two_step, merged, rtol=0, atol=1e-12)


def pin_bf16_rounding():
    """The cache's bf16 rounding equals torch's round-to-nearest-even conversion."""
    rng = np.random.default_rng(0)
    x32 = np.concatenate([rng.normal(scale=s, size=4000) for s in (1e-3, 0.02, 1.0, 300.0)]).astype(np.float32)
    # exact ties: a bf16 value plus half an ulp, both parities of the kept last bit
    base = torch.tensor(rng.normal(size=256).astype(np.float32)).to(torch.bfloat16).float().numpy()
    ulp_half = np.abs(base) * 2.0 ** -8
    ties = (base + np.sign(base) * ulp_half * (1 - 2.0 ** -24)).astype(np.float32)
    x32 = np.concatenate([x32, base, ties, (base + ulp_half).astype(np.float32)])
    want = torch.tensor(x32).to(torch.bfloat16).double().numpy()
    got = mo.round_to_bf16(x32.astype(np.float64))
    assert np.array_equal(got, want)


def pin_cache_tables():
    g = _load("mla_storage_worked_example.json")["growth"]
    e_mla = mo.cache_elements_per_token("mla", d_c=g["mla"]["latent"], d_r=g["mla"]["rope"])
    e_mha = mo.cache_elements_per_token("mha", n_h=g["mha"]["kv_heads"], d_h=g["mha"]["head_dim"])
    e_gqa = mo.cache_elements_per_token("gqa", n_g=g["gqa"]["kv_heads"], d_h=g["gqa"]["head_dim"])
    for e, k in ((e_mla, "mla"), (e_mha, "mha"), (e_gqa, "gqa")):
        assert e == g[k]["per_token"]
        assert e * g["tokens_before"] == g[k]["before"] and e * g["tokens_after"] == g[k]["after"]
    t = _load("cache_size_tables.json")
    c = t["config"]
    el = {k: mo.cache_elements_per_token(k, n_h=c["n_h"], d_h=c["d_h"], n_g=c["n_g"], d_c=c["d_c"], d_r=c["d_r"])
          for k in ("mha", "gqa", "mqa", "mla")}
    assert el == t["elements"]
    for k, pct in t["relative_to_mha_percent"].items():
        assert round(100.0 * el[k] / el["mha"], 2 if k == "mla" else 3) == pct
    for k, gib in t["gib"].items():
        b = mo.cache_bytes(el[k], t["tokens"], t["layers"], t["bytes_per_value"])
        assert round(b / 2 ** 30, 3) == gib
    assert round(el["mha"] / el["mla"], 1) == t["mla_vs_mha_ratio"]
    v3 = t["v3"]
    assert mo.cache_elements_per_token("mla", d_c=v3["d_c"], d_r=v3["d_r"]) == v3["mla"]
    assert v3["n_h"] * (v3["key_dim"] + v3["value_dim"]) == v3["mha_same_head_sizes"]
    v2 = t["v2"]
    ratio = (mo.cache_elements_per_token("mha", n_h=v2["n_h"], d_h=v2["d_h"])
             / mo.cache_elements_per_token("mla", d_c=v2["d_c"], d_r=v2["d_r"]))
    assert round(ratio) == v2["claimed_ratio"]


def pin_scale():
    assert mo.softmax_scale(128, 64) == 1.0 / math.sqrt(192)
    assert mo.softmax_scale(16, 8) == 1.0 / math.sqrt(24)


ALL_PINS = [pin_worked_example_heads, pin_full_key_concat, pin_single_row_decode,
            pin_two_rows_content, pin_rotary_query_position, pin_identical_rows,
            pin_dominant_row, pin_absorption_invariant, pin_rope_closed_forms,
            pin_append_closed_form, pin_query_and_out_projections, pin_query_latent_projection,
            pin_output_projection_and_merge, pin_bf16_rounding,
            pin_cache_tables, pin_scale]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ------------------------------------------------------------ planted mistakes

def _any_pin_fails(pins):
    for p in pins:
        try:
            p()
        except AssertionError:
            return True
    return False


DECODE_PINS = [pin_single_row_decode, pin_two_rows_content, pin_rotary_query_position,
               pin_identical_rows, pin_absorption_invariant, pin_append_closed_form,
               pin_rope_closed_forms]


def test_planted_rotation_sign_is_caught(monkeypatch):
    real = mo.rope
    monkeypatch.setattr(mo, "rope", lambda x, pos, base: real(x, -np.asarray(pos), base))
    assert _any_pin_fails(DECODE_PINS)


def test_planted_query_position_off_by_one_is_caught(monkeypatch):
    real = mo.rope
    # only the decode's query rotation is affected by this shift (rows are fixtures)
    monkeypatch.setattr(mo, "rope", lambda x, pos, base: real(x, np.asarray(pos) + 1, base))
    assert _any_pin_fails([pin_rotary_query_position])


def test_planted_dropped_rotary_term_is_caught(monkeypatch):
    monkeypatch.setattr(mo, "rope", lambda x, pos, base: np.zeros_like(np.asarray(x, float)))
    assert _any_pin_fails([pin_rotary_query_position])


def test_planted_wrong_scale_is_caught(monkeypatch):
    monkeypatch.setattr(mo, "softmax_scale", lambda d_h, d_r: 1.0 / math.sqrt(d_h))
    assert _any_pin_fails([pin_single_row_decode, pin_two_rows_content, pin_rotary_query_position])


def test_planted_transposed_up_projection_is_caught(monkeypatch):
    def swapped(c, w_uk, w_uv):      # uses W_UV where W_UK belongs and vice versa
        return real(c, w_uv, w_uk)
    real = mo.expand_heads
    monkeypatch.setattr(mo, "expand_heads", swapped)
    assert _any_pin_fails([pin_worked_example_heads, pin_two_rows_content])


def test_planted_pairing_convention_change_is_caught(monkeypatch):
    def half_split(x, pos, base):    # (k, k + d/2) pairing instead of (2k, 2k+1)
        x = np.asarray(x, float)
        d = x.shape[-1]
        perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
        inv = np.argsort(perm)
        return real(x[..., inv], pos, base)[..., perm]
    real = mo.rope
    monkeypatch.setattr(mo, "rope", half_split)
    assert _any_pin_fails([pin_rope_closed_forms])


def test_planted_bf16_truncation_is_caught(monkeypatch):
    def truncate(x):
        a = np.ascontiguousarray(np.asarray(x, np.float64))
        return (a.view(np.uint64) & ~np.uint64((1 << 45) - 1)).view(np.float64)
    monkeypatch.setattr(mo, "round_to_bf16", truncate)
    assert _any_pin_fails([pin_bf16_rounding])


# -------------------------------------------------- brute force and negative case

def test_brute_force_tiny_shapes():
    """A third evaluation with scalar loops in 40-digit arithmetic, on tiny shapes."""
    import mpmath
    mpmath.mp.dps = 40
    rng = np.random.default_rng(21)
    n_h, d_h, d_c, d_r = 2, 2, 3, 2
    base = 10000.0
    for n in (1, 2, 5):
        w_uk, w_uv = rng.normal(size=(n_h, d_h, d_c)), rng.normal(size=(n_h, d_h, d_c))
        rows = rng.normal(size=(n, d_c + d_r))
        q_c, q_r = rng.normal(size=(n_h, d_h)), rng.normal(size=(n_h, d_r))
        want = mo.decode_explicit(q_c, q_r, w_uk, w_uv, rows, base)
        p = n - 1
        for i in range(n_h):
            # query rotary part at position p: one pair, angle p * base^0 = p
            cs, sn = mpmath.cos(p), mpmath.sin(p)
            qr0 = q_r[i][0] * cs - q_r[i][1] * sn
            qr1 = q_r[i][0] * sn + q_r[i][1] * cs
            scores = []
            for j in range(n):
                dot = mpmath.mpf(0)
                for d in range(d_h):
                    kc = mpmath.fsum(mpmath.mpf(w_uk[i][d][c]) * rows[j][c] for c in range(d_c))
                    dot += q_c[i][d] * kc
                dot += qr0 * rows[j][d_c] + qr1 * rows[j][d_c + 1]
                scores.append(dot / mpmath.sqrt(d_h + d_r))
            z = mpmath.fsum(mpmath.exp(s) for s in scores)
            assert abs(float(mpmath.log(z)) - want["lse"][i]) < 1e-12
            for d in range(d_h):
                od = mpmath.fsum(mpmath.exp(scores[j]) / z *
                                 mpmath.fsum(mpmath.mpf(w_uv[i][d][c]) * rows[j][c] for c in range(d_c))
                                 for j in range(n))
                assert abs(float(od) - want["o"][i][d]) < 1e-12


def test_rotary_on_expanded_keys_blocks_the_fold():
    """If RoPE rotated the expanded content key, the folded query would depend on
    the key's position ("Grouped-query and latent attention", section "Why a
    separate rotary key"): W_UK^T R(n)^T R(m) q differs across n."""
    rng = np.random.default_rng(8)
    d_h, d_c, m = 4, 6, 9
    w_uk = rng.normal(size=(d_h, d_c))
    q = rng.normal(size=d_h)
    q_m = mo.rope(q, m, 100.0)
    folded = []
    for n in (0, 1, 5):
        # rotation by -n applied to the rotated query gives R(n)^T R(m) q
        folded.append(w_uk.T @ mo.rope(q_m, -n, 100.0))
    assert np.max(np.abs(folded[0] - folded[1])) > 1e-3
    assert np.max(np.abs(folded[1] - folded[2])) > 1e-3
    # with the decoupled design the content fold ignores position entirely
    c = rng.normal(size=d_c)
    assert abs((w_uk.T @ q) @ c - q @ (w_uk @ c)) < 1e-12


def test_empty_sequence_rejected():
    with pytest.raises(ValueError):
        mo.decode_explicit(np.zeros((1, 2)), np.zeros((1, 2)), np.zeros((1, 2, 3)),
                           np.zeros((1, 2, 3)), np.zeros((0, 5)), 10000.0)


# ---------------------------------------------------------------- fp8 latent cache
def test_pin_e4m3_rounding_matches_library_conversion():
    """round_to_e4m3 against torch's float -> float8_e4m3fn conversion (round to nearest
    even) on every representable value, every midpoint between neighbours (the ties) and
    dense grids across the normal and subnormal ranges."""
    torch = pytest.importorskip("torch")
    vals = mo.e4m3_value(np.arange(256, dtype=np.uint8))
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (fin[:-1] + fin[1:]) / 2
    grid = np.concatenate([fin, mids, np.linspace(-460, 460, 40001), np.geomspace(1e-6, 460, 4001),
                           -np.geomspace(1e-6, 460, 4001)]).astype(np.float32)
    ref = torch.from_numpy(grid).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mo.round_to_e4m3(grid.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_pin_e4m3_decoding_matches_library_view():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mo.e4m3_value(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    np.testing.assert_array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    # closed forms: the largest finite value, the smallest normal and subnormal, signed zero
    assert mo.e4m3_value(np.uint8(0x7E)) == 448.0
    assert mo.e4m3_value(np.uint8(0x08)) == 2.0 ** -6
    assert mo.e4m3_value(np.uint8(0x01)) == 2.0 ** -9
    assert mo.e4m3_value(np.uint8(0x80)) == 0.0


def test_pin_fp8_row_quantization():
    """Each 128-column group: the scale is a power of two and the group's largest magnitude
    lands in (224, 448], every value is on the E4M3 grid and within half a grid step of
    c / scale, the rotary part is bf16, and a group of zeros keeps scale 1."""
    rng = np.random.default_rng(7)
    d_c, d_r = 512, 64
    row = rng.normal(0.0, 0.02, (3, d_c + d_r))
    row[2, 128:256] = 0.0
    vals, scales, k_r = mo.quantize_row_fp8(row, d_c)
    assert vals.shape == (3, d_c) and scales.shape == (3, 4) and k_r.shape == (3, d_r)
    g = vals.reshape(3, 4, 128)
    for r in range(3):
        for q in range(4):
            if r == 2 and q == 1:
                assert scales[r, q] == 1.0 and not g[r, q].any()
                continue
            sc = scales[r, q]
            assert sc == 2.0 ** np.round(np.log2(sc))
            # before rounding the group's largest |c| / scale lies in (224, 448]; on the grid
            # it can round down onto 224
            amax = np.max(np.abs(row[r, 128 * q:128 * q + 128].astype(np.float32).astype(np.float64)))
            assert mo.E4M3_MAX / 2 < amax / sc <= mo.E4M3_MAX
            assert mo.E4M3_MAX / 2 <= np.max(np.abs(g[r, q])) <= mo.E4M3_MAX
    np.testing.assert_array_equal(mo.round_to_e4m3(vals), vals)
    y = row[:, :d_c].astype(np.float32).astype(np.float64) / np.repeat(scales, 128, axis=1)
    _, p = np.frexp(np.where(np.abs(y) > 0, np.abs(y), 1.0))
    half_step = np.ldexp(1.0, np.clip(p - 1, -6, 8) - 4)
    assert np.all(np.abs(vals - y) <= half_step * (1 + 1e-6))
    np.testing.assert_array_equal(k_r, mo.round_to_bf16(row[:, d_c:]))
    deq = mo.dequantize_row_fp8(vals, scales, k_r)
    assert deq.shape == row.shape
    assert np.max(np.abs(deq[:, :d_c] - row[:, :d_c])) <= 0.0625 * np.max(np.abs(row[:, :d_c]))


def test_pin_fp8_scale_boundaries():
    """Closed forms of the group scale (the smallest power of two 2^k with amax / 2^k <= 448):
    amax 448 -> 1, 448 (1 + 2^-20) -> 2, 896 -> 2, 224 -> 1/2, 2^-20 -> 2^-28; a sign flip
    changes nothing but the signs; the largest magnitude itself lands on a grid value."""
    d_c, d_r = 256, 8
    cases = [(448.0, 1.0), (448.0 * (1 + 2.0 ** -20), 2.0), (896.0, 2.0), (224.0, 0.5), (2.0 ** -20, 2.0 ** -28)]
    for amax, want in cases:
        row = np.zeros((1, d_c + d_r))
        row[0, 5] = amax
        row[0, 130] = -amax                      # second group, negative maximum
        row[0, 7] = amax / 3.0
        vals, scales, _ = mo.quantize_row_fp8(row, d_c)
        assert scales.tolist() == [[want, want]], (amax, scales)
        assert vals[0, 5] == -vals[0, 130]
        assert mo.E4M3_MAX / 2 <= abs(vals[0, 5]) <= mo.E4M3_MAX
        back = mo.dequantize_row_fp8(vals, scales, np.zeros((1, d_r)))
        # one grid step of E4M3 near amax / scale is 2^(e - 3) with amax / scale in [2^e, 2^(e+1))
        step = 2.0 ** (np.floor(np.log2(amax / want)) - 3) * want
        assert abs(back[0, 7] - amax / 3.0) <= step / 2 * (1 + 1e-9)
