"""Whole-step oracle on the synthetic workloads (CPU only)."""
import numpy as np
import torch

import mla_inputs
from oracle import oracle_step, oracle_sequence
import oracle.mla_oracle as mo


def test_inputs_are_deterministic_and_shaped():
    wl = mla_inputs.WORKLOADS["small_bf16"]
    w1, h1, q1 = mla_inputs.make_all(wl)
    w2, h2, q2 = mla_inputs.make_all(wl)
    assert torch.equal(w1["w_uk"], w2["w_uk"]) and torch.equal(h1, h2) and torch.equal(q1[0], q2[0])
    assert w1["w_dkv"].shape == (512, 2048) and w1["w_uk"].shape == (16, 128, 512)
    assert h1.shape == (8, 8, 2048) and q1[1].shape == (8, 16, 64)
    assert w1["w_dkv"].dtype == torch.bfloat16
    r = mla_inputs.make_prefill_rows(wl, 3, 10)
    assert torch.equal(r, mla_inputs.make_prefill_rows(wl, 3, 10)) and r.shape == (10, 576)
    # one sequence's rows do not depend on how many rows were asked for
    assert torch.equal(mla_inputs.make_prefill_rows(wl, 3, 20)[:10], r)


def test_ragged_lengths_in_range():
    wl = mla_inputs.WORKLOADS["v3_ragged_b16"]
    lens = mla_inputs.context_lengths(wl)
    assert len(lens) == 16 and all(1024 <= n <= 131072 for n in lens)
    assert lens == mla_inputs.context_lengths(wl)


def test_tiny_f32_step_explicit_equals_absorbed():
    wl = mla_inputs.WORKLOADS["tiny_f32"]
    e = oracle_step(wl, [0])[0]
    a = oracle_step(wl, [0], form="absorbed")[0]
    assert e["rows_new"].shape == (129, 40)
    for k in ("o", "o_lat", "lse"):
        assert np.max(np.abs(e[k] - a[k])) < 1e-10
    # fp32 cache: rows are not rounded; row 0 is at position 0 so k_R is unrotated
    w, h, _ = mla_inputs.make_all(wl)
    row0 = mo.f64(h[0, 0]) @ mo.f64(torch.cat([w["w_dkv"], w["w_kr"]])).T
    assert np.allclose(e["rows_new"][0], row0, atol=1e-12)


def test_small_bf16_sequence_head_subset():
    wl = mla_inputs.WORKLOADS["small_bf16"]
    w, h, q = mla_inputs.make_all(wl)
    full = oracle_sequence(wl, w, h, q, 2, 1024, heads=None, form="absorbed")
    sub = oracle_sequence(wl, w, h, q, 2, 1024, heads=[3, 11], form="explicit")
    assert np.max(np.abs(full["o_lat"][[3, 11]] - sub["o_lat"])) < 1e-10
    assert np.max(np.abs(full["o"][[3, 11]] - sub["o"])) < 1e-10
    # appended rows are bf16 values
    assert np.array_equal(mo.round_to_bf16(full["rows_new"]), full["rows_new"])
