"""The kernels' bounded waits run out, report it and leave the GPU usable.

Every wait inside the pipelined tensor-core kernels (on an mbarrier, a peer CTA or a
copy) is bounded in time.  Here the bound is lowered to 1 ns through
mla_set_wait_limit_ns, so the first wait that is not already complete gives up: the
kernel raises MLA_DEV_TIMEOUT, lets its own copies and MMAs finish, frees its tensor
memory and returns.  Nothing faults or hangs: the next call at the default bound runs
normally and matches the oracle.
"""
import pytest
import torch

import mla_inputs
from head_latent_attention_25_b300 import runner, _lib as L
from oracle import oracle_sequence
from parity import assert_parity

pytestmark = pytest.mark.gpu


def _timed_out(st, run, tries=3):
    """Run ``run`` under a 1 ns wait bound until one launch reports a time-out."""
    old = L.mla_set_wait_limit_ns(1)
    try:
        for _ in range(tries):
            st.dev_status.zero_()
            run()
            torch.cuda.synchronize()
            if int(st.dev_status.item()) & L.MLA_DEV_TIMEOUT:
                return True
    finally:
        L.mla_set_wait_limit_ns(0)
    return False


def _check_against_oracle(st, wl):
    st.dev_status.zero_()
    st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    weights, h, queries = mla_inputs.make_all(wl)
    for b in range(wl.batch):
        ref = oracle_sequence(wl, weights, h, queries, b, st.ctx_lens[b])
        assert_parity(st.o_lat[b], ref["o_lat"], wl.dtype, f"seq {b} o_lat after a time-out")
        assert_parity(st.out[b], ref["o"], wl.dtype, f"seq {b} o after a time-out")


def test_set_wait_limit_returns_previous_and_zero_restores_default():
    default = L.mla_set_wait_limit_ns(123)
    assert L.mla_set_wait_limit_ns(0) == 123
    assert L.mla_set_wait_limit_ns(0) == default == 2_000_000_000


@pytest.mark.parametrize("kernel", ["attention", "gemm"])
def test_wait_runs_out_and_context_stays_usable(kernel):
    wl = mla_inputs.WORKLOADS["small_bf16"]
    st = runner.from_workload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    if kernel == "attention":
        # the fold and schedule run at the default bound; only the attention kernel
        # (split_tc_kernel: a 2-CTA cluster with DSMEM exchange) runs at 1 ns
        st.decode_prepare()
        torch.cuda.synchronize()
        assert _timed_out(st, st.decode_attend)
    else:
        assert _timed_out(st, st.project_out)           # gemm_tc_kernel (W_UV)
    _check_against_oracle(st, wl)
