"""GPU path (through the C ABI) against the CPU oracle, element by element.

Small workloads are compared in full; the DeepSeek-V3-shaped workloads run at
their full sizes in the bench's launch configuration and are compared on
sampled sequences and heads, which the oracle computes one by one.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mla_inputs
from head_latent_attention_25_b300 import runner, _lib as L
from oracle import oracle_sequence
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _run(wl, ctx_lens=None, num_splits=0):
    st = runner.from_workload(wl, ctx_lens=ctx_lens, num_splits=num_splits)
    st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    return st


def _compare(st, wl, b, heads=None, ctx_len=None, what=""):
    weights, h, queries = mla_inputs.make_all(wl)
    n = st.ctx_lens[b] if ctx_len is None else ctx_len
    ref = oracle_sequence(wl, weights, h, queries, b, n, heads=heads)
    idx = slice(None) if heads is None else list(heads)
    tag = f"{wl.name} seq {b}{what}"
    assert_parity(st.new_rows(b), ref["rows_new"], wl.dtype, tag + " appended rows")
    assert_parity(st.o_lat[b][idx], ref["o_lat"], wl.dtype, tag + " o_lat")
    assert_parity(st.lse[b][idx], ref["lse"], wl.dtype, tag + " lse")
    assert_parity(st.out[b][idx], ref["o"], wl.dtype, tag + " o")
    return ref


def test_tiny_f32_end_to_end():
    """The whole cache is built by appending h_0..h_128; the query comes from h_128."""
    wl = mla_inputs.WORKLOADS["tiny_f32"]
    st = _run(wl)
    _compare(st, wl, 0)


def test_small_bf16_all_sequences():
    wl = mla_inputs.WORKLOADS["small_bf16"]
    st = _run(wl)
    for b in range(wl.batch):
        _compare(st, wl, b)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 64])
def test_small_bf16_split_count_invariance(num_splits):
    wl = mla_inputs.WORKLOADS["small_bf16"]
    auto = _run(wl)
    st = _run(wl, num_splits=num_splits)
    a, b = auto.o_lat.double(), st.o_lat.double()
    # o_lat is stored in bf16: allow two units in the last place of the largest value
    assert float((a - b).abs().max()) <= 2.0 ** -7 * float(a.abs().max())
    # lse: P is rounded to bf16 against a running maximum that depends on the split
    assert float((auto.lse - st.lse).abs().max()) <= 1e-4 * float(auto.lse.abs().max()) + 1e-4
    for b in range(wl.batch):
        _compare(st, wl, b, what=f" splits={num_splits}")


@pytest.mark.parametrize("num_splits", [0, 3, 64])
def test_repeated_runs_are_bitwise_identical(num_splits):
    """No atomics take part in the accumulation, so a fixed schedule gives the same bits;
    a difference would point to a race between pipeline stages."""
    wl = mla_inputs.WORKLOADS["small_bf16"]
    st = _run(wl, num_splits=num_splits)
    first_o, first_l = st.o_lat.clone(), st.lse.clone()
    for _ in range(5):
        st.step()
        torch.cuda.synchronize()
        assert torch.equal(st.o_lat, first_o) and torch.equal(st.lse, first_l)
    assert int(st.dev_status.item()) == 0


def test_peaked_scores_exercise_rescaling():
    """Cache ~N(0,1), queries ~N(0,16): scores spread over several units, so the
    running maximum moves across tiles and splits.  The appended tokens keep
    h ~ N(0,1): with much larger h a one-ulp bf16 rounding difference of an
    appended row (fp32 on the GPU, fp64 in the oracle; both correct roundings)
    would be amplified by the peaked softmax beyond the output tolerance."""
    wl = dataclasses.replace(mla_inputs.WORKLOADS["small_bf16"], name="small_bf16_peaked",
                             cache_std=1.0, query_std=4.0)
    st = _run(wl, num_splits=5)
    for b in (0, 7):
        _compare(st, wl, b)


def test_v3_b64_full_size_sampled():
    wl = mla_inputs.WORKLOADS["v3_b64_l4096"]
    st = _run(wl)
    _compare(st, wl, 0)
    for b in (37, 63):
        _compare(st, wl, b, heads=[0, 1, 64, 127])


def test_v3_ragged_full_size_sampled():
    wl = mla_inputs.WORKLOADS["v3_ragged_b16"]
    lens = mla_inputs.context_lengths(wl)
    st = _run(wl)
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    for b in sorted({longest, shortest, 7}):
        _compare(st, wl, b, heads=[0, 5, 77, 127])


@pytest.mark.parametrize("batch,ctx", [(1, 32768), (256, 512), (32, 8192)])
def test_sweep_points_sampled(batch, ctx):
    wl = mla_inputs.sweep_workloads([batch], [ctx])[0]
    st = _run(wl)
    for b in sorted({0, batch - 1}):
        _compare(st, wl, b, heads=[3, 100])


def test_short_and_ragged_tails():
    """Single-row sequences and lengths just around multiples of 32 and 64."""
    base = mla_inputs.WORKLOADS["small_bf16"]
    lens = [0, 1, 30, 31, 32, 62, 63, 64, 126, 127, 0, 255]
    wl = dataclasses.replace(base, name="small_bf16_tails", batch=len(lens), n_new=1)
    for ns in (0, 3):
        st = _run(wl, ctx_lens=lens, num_splits=ns)
        for b in range(len(lens)):
            _compare(st, wl, b, what=f" splits={ns}")


def test_empty_sequence_flags_status_and_zeros_output():
    wl = dataclasses.replace(mla_inputs.WORKLOADS["small_bf16"], name="small_bf16_empty", batch=3,
                             n_new=1)
    st = runner.from_workload(wl, ctx_lens=[10, 10, 10])
    st.append()
    st.seq_len[1] = 0
    st.o_lat.fill_(7.0)
    st.decode()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & L.MLA_DEV_BAD_LENGTH
    assert float(st.o_lat[1].abs().max()) == 0.0
    assert torch.isinf(st.lse[1]).all() and (st.lse[1] < 0).all()
    st.project_out()
    torch.cuda.synchronize()
    # the other sequences are unaffected
    st.seq_len[1] = 11
    _compare(st, wl, 0)


def test_append_out_of_capacity_is_flagged_and_skipped():
    wl = dataclasses.replace(mla_inputs.WORKLOADS["small_bf16"], name="small_bf16_cap", batch=2, n_new=4)
    st = runner.from_workload(wl, ctx_lens=[16, 16])
    before = st.cache.clone()
    st.pos0[1] = 17                      # cap is 16 + 4 = 20 rows and 17 + 4 > 20
    st.append()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & L.MLA_DEV_BAD_POSITION
    o1 = int(st.row_off[1])
    assert torch.equal(st.cache[o1:o1 + 20], before[o1:o1 + 20])
    o0 = int(st.row_off[0])
    assert not torch.equal(st.cache[o0 + 16:o0 + 20], before[o0 + 16:o0 + 20])


def test_host_errors():
    wl = mla_inputs.WORKLOADS["small_bf16"]
    st = runner.from_workload(wl, load_inputs=False)
    with pytest.raises(L.MlaError) as e:
        L.mla_decode_absorbed(st.dims, st.dt, st.batch, st.q_c, st.q_r, st.q_c, st.cache, st.total_rows,
                              st.row_off, st.seq_len, st.max_seq_len, 0, st.workspace, 64, st.o_lat,
                              st.lse, st.dev_status)
    assert e.value.status == L.MLA_ERR_WORKSPACE
    big = L.make_dims(4, 16, 1024, 64, 64)
    with pytest.raises(L.MlaError) as e:
        L.mla_decode_absorbed(big, st.dt, st.batch, st.q_c, st.q_r, st.q_c, st.cache, st.total_rows,
                              st.row_off, st.seq_len, st.max_seq_len, 0, st.workspace, st.ws_bytes,
                              st.o_lat, st.lse, st.dev_status)
    assert e.value.status == L.MLA_ERR_UNSUPPORTED
