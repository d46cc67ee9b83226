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
from oracle import mla_oracle as mo
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


@pytest.mark.parametrize("num_splits", [1, 2, 3, 7, 8, 64])
def test_small_bf16_split_count_invariance(num_splits):
    """8 workers for the 8 sequences take one whole sequence each (no cut, no merge);
    every other count cuts sequences across workers and merges their pieces."""
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


@pytest.mark.parametrize("num_splits", [0, 3, 8, 64])
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


# Eight heads spread over the 128 of the V3 shapes: both ends of the MMA's M tile, both
# TMEM lane quarters' edges and the middle.
SAMPLED_HEADS = [0, 1, 31, 32, 63, 64, 100, 127]


def test_v3_b64_full_size_sampled():
    wl = mla_inputs.WORKLOADS["v3_b64_l4096"]
    st = _run(wl)
    _compare(st, wl, 0)
    for b in (1, 37, 63):
        _compare(st, wl, b, heads=SAMPLED_HEADS)


def test_v3_ragged_full_size_sampled():
    wl = mla_inputs.WORKLOADS["v3_ragged_b16"]
    lens = mla_inputs.context_lengths(wl)
    st = _run(wl)
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    for b in sorted({longest, shortest, 7}):
        _compare(st, wl, b, heads=SAMPLED_HEADS)


def test_v3_peaked_long_context():
    """The ragged V3 workload (16 sequences up to 131072 rows, 128 heads) with a cache
    ~N(0,1) and queries ~N(0,4): per head the scores spread over tens of log2 units, so
    the running maximum moves late in long sequences and the partial scores the two CTAs
    of a pair exchange have wide spreads within a tile.  The query spread is as large as
    the bf16 rounding of the folded query (needed by the tensor cores) allows inside the
    tolerance; the exchanged partials then lose less than that rounding does."""
    wl = dataclasses.replace(mla_inputs.WORKLOADS["v3_ragged_b16"], name="v3_ragged_b16_peaked",
                             cache_std=1.0, query_std=4.0)
    lens = mla_inputs.context_lengths(wl)
    st = _run(wl)
    longest = int(np.argmax(lens))
    assert lens[longest] >= 32768
    for b in sorted({longest, 0}):
        _compare(st, wl, b, heads=SAMPLED_HEADS + [15, 90, 111])


@pytest.mark.parametrize("batch,ctx", [(b, c) for b in mla_inputs.SWEEP_BATCHES
                                       for c in mla_inputs.SWEEP_CONTEXTS])
def test_sweep_points_sampled(batch, ctx):
    """Every point of the batch x context sweep, in the bench's launch configuration."""
    wl = mla_inputs.sweep_workloads([batch], [ctx])[0]
    st = _run(wl)
    for b in sorted({0, batch // 2, batch - 1}):
        _compare(st, wl, b, heads=SAMPLED_HEADS)
    del st
    torch.cuda.empty_cache()


def test_v3_query_from_h_full_size_sampled():
    """The query computed on the GPU from the new token's h: c_q = W_DQ h (query latent
    1536, split-K tensor-core GEMM), q_C = W_UQ c_q and q_R = W_QR c_q (one tensor-core
    launch), then the decode; q_C, q_R and the outputs are compared with the oracle."""
    wl = mla_inputs.WORKLOADS["v3_b64_l4096_from_h"]
    st = _run(wl)
    for b in (0, 41):
        ref = _compare(st, wl, b, heads=SAMPLED_HEADS)
        assert_parity(st.q_c[b][SAMPLED_HEADS], ref["q_c"], wl.dtype, f"seq {b} q_C")
        assert_parity(st.q_r[b][SAMPLED_HEADS], ref["q_r"], wl.dtype, f"seq {b} q_R (before rotation)")


@pytest.mark.parametrize("dtype,d_q", [("bf16", 96), ("f32", 24)])
def test_query_latent_cuda_core_shapes(dtype, d_q):
    """Query latent widths outside the tensor-core GEMM run on CUDA cores."""
    base = mla_inputs.WORKLOADS["tiny_f32" if dtype == "f32" else "small_bf16"]
    wl = dataclasses.replace(base, name=f"query_latent_{dtype}", batch=3, prefill=40, n_new=2,
                             query_from_h=True, d_q=d_q)
    st = _run(wl)
    weights, h, queries = mla_inputs.make_all(wl)
    for b in range(wl.batch):
        ref = _compare(st, wl, b)
        assert_parity(st.q_c[b], ref["q_c"], wl.dtype, f"seq {b} q_C")


@pytest.mark.parametrize("name,batch,prefill,n_q", [("small_bf16", 4, 300, 4), ("v3_b64_l4096", 8, 1000, 4),
                                                   ("tiny_f32", 2, 50, 3)])
def test_multi_query_causal_decode(name, batch, prefill, n_q):
    """n_q new tokens appended per sequence and all n_q of them decoded at once: query j
    attends over the rows up to its own position (causal), on the same kernels."""
    base = mla_inputs.WORKLOADS[name]
    wl = dataclasses.replace(base, name=f"{name}_multi{n_q}", batch=batch, prefill=prefill, n_new=n_q,
                             n_q=n_q, query_from_h=False)
    st = _run(wl)
    heads = None if wl.n_heads <= 16 else SAMPLED_HEADS
    idx = slice(None) if heads is None else heads
    weights, h, queries = mla_inputs.make_all(wl)
    for b in sorted({0, batch - 1}):
        ref = oracle_sequence(wl, weights, h, queries, b, st.ctx_lens[b], heads=heads)
        for j in range(n_q):
            tag = f"{wl.name} seq {b} query {j}"
            assert_parity(st.o_lat[b, j][idx], ref["o_lat"][j], wl.dtype, tag + " o_lat")
            assert_parity(st.lse[b, j][idx], ref["lse"][j], wl.dtype, tag + " lse")
            assert_parity(st.out[b, j][idx], ref["o"][j], wl.dtype, tag + " o")


def test_multi_query_shorter_than_its_queries_is_flagged():
    wl = dataclasses.replace(mla_inputs.WORKLOADS["small_bf16"], name="small_bf16_multi_short", batch=2,
                             prefill=20, n_new=3, n_q=3)
    st = runner.from_workload(wl)
    st.append()
    st.seq_len[1] = 2                       # query 0 of sequence 1 would sit at position -1
    st.o_lat.fill_(7.0)
    st.decode()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & L.MLA_DEV_BAD_LENGTH
    assert float(st.o_lat[1, 0].abs().max()) == 0.0 and torch.isinf(st.lse[1, 0]).all()
    assert float(st.o_lat[1, 1].abs().max()) > 0.0          # position 0: one row


@pytest.mark.parametrize("name,seqs", [("small_bf16", (0, 5)), ("v3_b64_l4096", (0, 63))])
def test_output_projection_two_step_and_merged(name, seqs):
    """The layer output u = W_O [o_1; ...; o_n_h] after the step, by the two-step path
    (W_UV per head, then W_O) and by the merged weights W_OV^(i) = W_O^(i) W_UV^(i) applied
    to the latent output; the merged weights themselves are compared too."""
    wl = dataclasses.replace(mla_inputs.WORKLOADS[name], name=f"{name}_out", w_o=True)
    st = _run(wl)
    st.project_output()
    u_two = st.u.clone()
    st.merge_output_weights()
    u_m = torch.empty_like(st.u)
    st.project_output_merged(u=u_m)
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    weights, h, queries = mla_inputs.make_all(wl)
    w_ov_ref = mo.merge_output_weights(weights["w_o"], weights["w_uv"])      # [n_h, hidden, d_c]
    for i in (0, wl.n_heads - 1):
        assert_parity(st.w_ov[i].transpose(0, 1), w_ov_ref[i], wl.dtype, f"W_OV head {i}")
    for b in seqs:
        ref = oracle_sequence(wl, weights, h, queries, b, st.ctx_lens[b])
        u_ref = mo.project_output(ref["o"], weights["w_o"])
        assert_parity(u_two[b], u_ref, wl.dtype, f"seq {b} u (two-step)")
        assert_parity(u_m[b], u_ref, wl.dtype, f"seq {b} u (merged)")


LAYOUTS = [("split", 64), ("paged", 64), ("paged", 128), ("paged_split", 256)]


@pytest.mark.parametrize("layout,block_size", LAYOUTS)
@pytest.mark.parametrize("lens,num_splits", [(None, 0), ([1, 30, 63, 64, 65, 127, 200, 1000], 3),
                                             ([1, 30, 63, 64, 65, 127, 200, 1000], 0)])
def test_cache_layouts(layout, block_size, lens, num_splits):
    """The cache append and the decode through an mla_cache_layout: latents and rotary keys
    in separate buffers and/or a paged pool whose blocks a seeded shuffle scatters; ranges
    cut sequences (a paged cache flattens them in whole 64-row tiles)."""
    wl = mla_inputs.WORKLOADS["small_bf16"]
    if lens is not None:
        wl = dataclasses.replace(wl, name="small_bf16_layout_tails", batch=len(lens), n_new=1)
    st = runner.from_workload(wl, ctx_lens=lens, num_splits=num_splits, layout=layout, block_size=block_size)
    st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    for b in range(wl.batch):
        _compare(st, wl, b, what=f" {layout}/{block_size} splits={num_splits}")
    if layout == "split":
        # the same schedule as the packed cache: the same bits
        ref = runner.from_workload(wl, ctx_lens=lens, num_splits=num_splits)
        ref.step()
        torch.cuda.synchronize()
        assert torch.equal(ref.o_lat, st.o_lat) and torch.equal(ref.out, st.out)


@pytest.mark.parametrize("layout", ["paged", "paged_split"])
def test_v3_b64_paged_sampled(layout):
    """The bench's V3 batch-64 decode with a paged cache of 64-row blocks."""
    wl = mla_inputs.WORKLOADS["v3_b64_l4096"]
    st = runner.from_workload(wl, layout=layout, block_size=64)
    st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    for b in (0, 40):
        _compare(st, wl, b, heads=SAMPLED_HEADS, what=f" {layout}")


def test_cuda_core_bf16_odd_shapes():
    """bf16 shapes outside the tensor-core kernels (latent 256, rotary 32, 8 heads of
    width 64): the append, fold, attention and W_UV all run on CUDA cores."""
    wl = dataclasses.replace(mla_inputs.WORKLOADS["small_bf16"], name="small_bf16_odd", batch=4,
                             n_heads=8, d_h=64, d_c=256, d_r=32, hidden=512, prefill=300, n_new=3)
    for ns in (0, 5):
        st = _run(wl, num_splits=ns)
        for b in range(wl.batch):
            _compare(st, wl, b, what=f" splits={ns}")


def test_latent_shape_cache_smaller_than_a_tile():
    """bf16 with the 512 + 64 latent shape but a cache buffer of fewer than 32 rows: the
    attention runs on CUDA cores (the tensor-core kernel needs one 32-row box)."""
    wl = dataclasses.replace(mla_inputs.WORKLOADS["small_bf16"], name="small_bf16_tiny_cache", batch=2,
                             prefill=7, n_new=2)
    st = _run(wl)
    assert st.total_rows < 32
    for b in range(wl.batch):
        _compare(st, wl, b)


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


def test_empty_sequence_with_whole_sequence_workers():
    """Eight workers for eight sequences of equal length, one of them emptied: each worker
    takes a sequence whole, the empty one is flagged and its outputs are zero."""
    wl = mla_inputs.WORKLOADS["small_bf16"]
    st = runner.from_workload(wl, num_splits=8)
    st.append()
    st.seq_len[3] = 0
    st.o_lat.fill_(7.0)
    st.decode()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & L.MLA_DEV_BAD_LENGTH
    assert float(st.o_lat[3].abs().max()) == 0.0 and torch.isinf(st.lse[3]).all()
    st.project_out()
    torch.cuda.synchronize()
    for b in (0, 7):
        _compare(st, wl, b)


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


@pytest.mark.parametrize("num_splits", [5, 6, 12])
def test_worker_ranges_starting_on_sequence_boundaries(num_splits):
    """Lengths 100, 100, 100, 300 cut into equal ranges: with 6 (or 12) workers every range
    boundary falls exactly on a sequence start or inside the long sequence, with 5 none
    does; each worker's start record (first sequence, its span and first row) must still
    lead to the right rows."""
    base = mla_inputs.WORKLOADS["small_bf16"]
    lens = [99, 99, 99, 299]
    wl = dataclasses.replace(base, name="small_bf16_boundaries", batch=len(lens), n_new=1)
    st = _run(wl, ctx_lens=lens, num_splits=num_splits)
    for b in range(len(lens)):
        _compare(st, wl, b, what=f" splits={num_splits}")
