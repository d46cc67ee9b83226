"""The decode step captured once into a CUDA graph and replayed.

Every call of the path is asynchronous and allocation-free, so the whole step
(append -> fold -> split -> merge -> W_UV) can be recorded into one graph.  The
replay must reproduce the eager step bit for bit (the kernels are deterministic
for a fixed schedule), and must follow a change of the device-side inputs made
between replays.
"""
import pytest
import torch

import mla_inputs
from head_latent_attention_25_b300 import runner

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["small_bf16", "v3_b64_l4096"])
def test_graph_replay_matches_eager(name):
    wl = mla_inputs.WORKLOADS[name]
    st = runner.from_workload(wl)
    st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    eager = (st.o_lat.clone(), st.lse.clone(), st.out.clone())

    g = st.capture()
    for t in (st.o_lat, st.lse, st.out):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    assert torch.equal(st.o_lat, eager[0])
    assert torch.equal(st.lse, eager[1])
    assert torch.equal(st.out, eager[2])


def test_graph_follows_new_queries():
    """New query values written into the bound buffers between replays are used."""
    wl = mla_inputs.WORKLOADS["small_bf16"]
    st = runner.from_workload(wl)
    g = st.capture()
    g.replay()
    torch.cuda.synchronize()
    first = st.out.clone()
    gen = torch.Generator(device="cpu").manual_seed(123)
    st.q_c.copy_(torch.randn(st.q_c.shape, generator=gen).to(st.q_c.dtype))
    g.replay()
    torch.cuda.synchronize()
    replayed = st.out.clone()
    st.step()                                   # the same inputs, eagerly
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    assert not torch.equal(replayed, first)
    assert torch.equal(replayed, st.out)


@pytest.mark.parametrize("name", ["small_bf16", "tiny_f32"])
def test_two_stream_step_matches_one_stream(name):
    """step() runs the cache append on a second stream beside the query fold
    (mla_decode_prepare), then the attention (mla_decode_attend); the results equal
    those of the whole path on one stream, appended rows included."""
    wl = mla_inputs.WORKLOADS[name]
    a = runner.from_workload(wl)
    b = runner.from_workload(wl)
    a.step()
    b.step_serial()
    torch.cuda.synchronize()
    assert int(a.dev_status.item()) == 0 and int(b.dev_status.item()) == 0
    assert torch.equal(a.cache, b.cache)
    for x, y in ((a.o_lat, b.o_lat), (a.lse, b.lse), (a.out, b.out)):
        assert torch.equal(x, y)


def test_prepare_reads_no_cache_row():
    """mla_decode_prepare may run before the new rows are in the cache: prepare, then
    append, then attend (one stream) gives the same results as the whole step."""
    wl = mla_inputs.WORKLOADS["small_bf16"]
    a = runner.from_workload(wl)
    b = runner.from_workload(wl)
    a.decode_prepare()
    a.append()
    a.decode_attend()
    a.project_out()
    b.step_serial()
    torch.cuda.synchronize()
    assert int(a.dev_status.item()) == 0 and int(b.dev_status.item()) == 0
    for x, y in ((a.cache, b.cache), (a.o_lat, b.o_lat), (a.lse, b.lse), (a.out, b.out)):
        assert torch.equal(x, y)
