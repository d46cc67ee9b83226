"""The allocation-free decode entry point, for callers that cannot call cudaMalloc.

It must give the results of the regular entry point (which takes a caller-allocated
workspace), on two calls in a row, since every call reuses the same built-in scratch.
This file is named to be collected last, so that a run stopping at the first failure
has already run every other test.
"""
import pytest
import torch

import mla_inputs
from head_latent_attention_25_b300 import runner, _lib as L
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _noalloc(st, o_lat, lse, num_splits):
    L.mla_decode_absorbed_noalloc(st.dims, st.dt, st.batch, st.q_c, st.q_r, st.w["w_uk"], st.cache,
                                  st.total_rows, st.row_off, st.seq_len, st.max_seq_len, num_splits,
                                  o_lat, lse, st.dev_status)


@pytest.mark.parametrize("name,num_splits", [("small_bf16", 0), ("small_bf16", 3), ("tiny_f32", 0)])
def test_noalloc_matches_workspace_decode_on_two_calls(name, num_splits):
    wl = mla_inputs.WORKLOADS[name]
    st = runner.from_workload(wl, num_splits=num_splits)
    st.step()                                  # regular path: append, decode with workspace, W_UV
    torch.cuda.synchronize()
    ref_o, ref_l = st.o_lat.clone(), st.lse.clone()
    for call in range(2):
        o = torch.full_like(st.o_lat, 7.0)
        l = torch.full_like(st.lse, 7.0)
        _noalloc(st, o, l, num_splits)
        torch.cuda.synchronize()
        assert int(st.dev_status.item()) == 0
        assert_parity(o, ref_o, wl.dtype, f"{name} call {call} o_lat")
        assert_parity(l, ref_l, wl.dtype, f"{name} call {call} lse")


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # 1024 sequences of up to 131072 rows need far more than 32 MiB of split partials;
    # the refusal happens before any pointer is used
    d = L.make_dims(128, 128, 512, 64, 7168)
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert L.mla_decode_workspace_size(d, L.MLA_BF16, 1024, 131072, 0) > (32 << 20)
    with pytest.raises(L.MlaError) as e:
        L.mla_decode_absorbed_noalloc(d, L.MLA_BF16, 1024, dummy, dummy, dummy, dummy, 1 << 20, dummy,
                                      dummy, 131072, 0, dummy, None, status)
    assert e.value.status == L.MLA_ERR_WORKSPACE
