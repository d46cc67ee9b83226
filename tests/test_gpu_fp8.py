"""fp8 latent cache: append (tensor-core GEMM + fp8 finalize) and decode (tensor cores for
DeepSeek-V3 shapes, with the codes turned into bf16 tiles in shared memory; CUDA cores for a
cache of fewer than 32 rows).

The appended rows are compared with the oracle's quantization of the oracle's own row
(scales, codes within one grid step where the fp32 row and the fp64 row round differently,
rotary part in bf16).  The decode is compared with the oracle's absorbed decode over the
rows the device actually stored (read back and decoded by the oracle), so that its parity
does not depend on the quantization's ties.
"""
import numpy as np
import pytest
import torch

from oracle import mla_oracle as mo
from parity import assert_parity

pytestmark = pytest.mark.gpu

N_H, D_H, D_C, D_R, HIDDEN, BASE = 16, 128, 512, 64, 2048, 10000.0


def _L():
    import head_latent_attention_25_b300 as pkg
    return pkg


def _encode_rows(vals, scales, k_r):
    """Host bytes of fp8 rows from the oracle's parts (vals are exact E4M3 values)."""
    n = vals.shape[0]
    codes = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    sc = scales.astype(np.float32).view(np.uint8).reshape(n, -1)
    kr = torch.from_numpy(k_r.astype(np.float32)).to(torch.bfloat16).view(torch.uint8).numpy().reshape(n, -1)
    return np.concatenate([codes, sc, kr], axis=1)


def _decode_rows(raw):
    """(values, scales, rotary) of device fp8 rows read back as uint8 [n, row_bytes]."""
    raw = np.ascontiguousarray(raw)
    vals = mo.e4m3_value(raw[:, :D_C])
    scales = raw[:, D_C:D_C + 4 * (D_C // 128)].copy().view(np.float32).astype(np.float64)
    kr = torch.from_numpy(raw[:, D_C + 4 * (D_C // 128):].copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return vals, scales, kr


def _setup(prefill, n_new, seed, n_h=N_H, extra_rows=7):
    L = _L()
    g = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    w_dkv = (torch.randn(D_C, HIDDEN, generator=g) * 0.02).to(bf)
    w_kr = (torch.randn(D_R, HIDDEN, generator=g) * 0.02).to(bf)
    w_uk = (torch.randn(n_h, D_H, D_C, generator=g) * 0.02).to(bf)
    batch = len(prefill)
    h = torch.randn(batch * n_new, HIDDEN, generator=g).to(bf)
    q_c = torch.randn(batch, n_h, D_H, generator=g).to(bf)
    q_r = torch.randn(batch, n_h, D_R, generator=g).to(bf)
    cap = [p + n_new for p in prefill]
    row_off = np.concatenate([[0], np.cumsum(cap)[:-1]]).astype(np.int64)
    rows_total = int(sum(cap)) + extra_rows               # a few rows past the last sequence
    rb = L.fp8_row_bytes(D_C, D_R)
    # prefilled rows: random latents quantized by the oracle, encoded on the host
    pre = np.random.default_rng(seed).normal(0.0, 0.02, (rows_total, D_C + D_R))
    vals, scales, kr = mo.quantize_row_fp8(pre, D_C)
    host = _encode_rows(vals, scales, kr)
    assert host.shape == (rows_total, rb)
    dims = L.make_dims(n_h, D_H, D_C, D_R, HIDDEN, BASE)
    dev = dict(
        w_dkv=w_dkv.cuda(), w_kr=w_kr.cuda(), w_uk=w_uk.cuda(), h=h.cuda(), q_c=q_c.cuda(), q_r=q_r.cuda(),
        cache=torch.from_numpy(host).cuda(), row_off=torch.from_numpy(row_off).cuda(),
        cap=torch.tensor(cap, dtype=torch.int32).cuda(), pos0=torch.tensor(prefill, dtype=torch.int32).cuda(),
        seq_len=torch.tensor(cap, dtype=torch.int32).cuda(), status=torch.zeros(1, dtype=torch.int32).cuda())
    return L, dims, dev, dict(w_dkv=w_dkv, w_kr=w_kr, w_uk=w_uk, h=h, q_c=q_c, q_r=q_r), row_off, cap, host


def _append(L, dims, dev, n_new, rows_total):
    batch = dev["pos0"].numel()
    ws_bytes = L.mla_append_workspace_size(dims, L.MLA_BF16, batch, n_new)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    L.mla_cache_append_fp8(dims, batch, n_new, dev["h"], dev["w_dkv"], dev["w_kr"], dev["row_off"], dev["cap"],
                           dev["pos0"], dev["cache"], rows_total, ws, ws_bytes, dev["status"])


@pytest.mark.parametrize("prefill,n_new", [([300, 129, 64], 2), ([1000], 1), ([5, 63, 64, 65, 200], 3)])
def test_fp8_append_rows(prefill, n_new):
    L, dims, dev, hostw, row_off, cap, host = _setup(prefill, n_new, seed=11 + n_new)
    rows_total = host.shape[0]
    _append(L, dims, dev, n_new, rows_total)
    torch.cuda.synchronize()
    assert int(dev["status"].item()) == 0
    got = dev["cache"].cpu().numpy()
    for b, p in enumerate(prefill):
        toks = hostw["h"][b * n_new:(b + 1) * n_new]
        pos = np.arange(p, p + n_new)
        ref_row = mo.append_rows(toks, hostw["w_dkv"], hostw["w_kr"], pos, BASE, cache_bf16=False)
        rv, rs, rk = mo.quantize_row_fp8(ref_row, D_C)
        new = got[row_off[b] + p:row_off[b] + p + n_new]
        gv, gs, gk = _decode_rows(new)
        np.testing.assert_allclose(gs, rs, rtol=1e-5, err_msg="scales")
        # codes: equal, or one grid step apart where the fp32 row and the fp64 row round apart
        y = np.abs(rv)
        _, e = np.frexp(np.where(y > 0, y, 1.0))
        step = np.ldexp(1.0, np.clip(e - 1, -6, 8) - 3)
        diff = np.abs(gv - rv)
        assert np.all(diff <= step * (1 + 1e-9)), "codes more than one step apart"
        assert np.mean(diff > 0) < 0.02, f"{np.mean(diff > 0):.3f} of the codes differ"
        assert_parity(gk, rk, "bf16", "rotary part")
    # rows outside the appended positions keep their bytes
    mask = np.ones(rows_total, dtype=bool)
    for b, p in enumerate(prefill):
        mask[row_off[b] + p:row_off[b] + p + n_new] = False
    np.testing.assert_array_equal(got[mask], host[mask])


def _decode_and_compare(prefill, n_new, num_splits, n_h, seed, heads=None, extra_rows=7):
    L, dims, dev, hostw, row_off, cap, host = _setup(prefill, n_new, seed, n_h=n_h, extra_rows=extra_rows)
    rows_total = host.shape[0]
    _append(L, dims, dev, n_new, rows_total)
    batch = len(prefill)
    max_len = max(cap)
    ws_bytes = L.mla_decode_workspace_size(dims, L.MLA_BF16, batch, max_len, num_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o_lat = torch.full((batch, n_h, D_C), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((batch, n_h), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_decode_absorbed_fp8(dims, batch, dev["q_c"], dev["q_r"], dev["w_uk"], dev["cache"], rows_total,
                              dev["row_off"], dev["seq_len"], max_len, num_splits, ws, ws_bytes, o_lat, lse,
                              dev["status"])
    torch.cuda.synchronize()
    assert int(dev["status"].item()) == 0
    got = dev["cache"].cpu().numpy()
    hs = list(range(n_h)) if heads is None else heads
    w_uv = np.zeros((len(hs), D_H, D_C))
    for b in range(batch):
        vals, scales, kr = _decode_rows(got[row_off[b]:row_off[b] + cap[b]])
        rows = mo.dequantize_row_fp8(vals, scales, kr)
        ref = mo.decode_absorbed(hostw["q_c"][b][hs], hostw["q_r"][b][hs], hostw["w_uk"][hs], w_uv, rows, BASE)
        assert_parity(o_lat[b][hs].cpu(), ref["o_lat"], "bf16", f"o_lat b={b}")
        assert_parity(lse[b][hs].cpu(), ref["lse"], "bf16", f"lse b={b}")


@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_fp8_decode_matches_oracle_on_device_rows(num_splits):
    """16 heads, ragged lengths with partial last tiles: the tensor-core kernel."""
    _decode_and_compare([300, 129, 64, 1], 2, num_splits, N_H, seed=5)


def test_fp8_decode_v3_heads_sampled():
    """128 heads (DeepSeek-V3), several tiles per sequence, sampled heads against the oracle."""
    _decode_and_compare([1500, 700, 4100], 1, 0, 128, seed=9, heads=[0, 1, 63, 64, 127])


def test_fp8_decode_tiny_cache_cuda_cores():
    """A cache of fewer than 32 rows runs on the CUDA-core kernel."""
    _decode_and_compare([10, 3], 2, 0, N_H, seed=2, extra_rows=0)


def test_fp8_append_bad_position_is_flagged_and_skipped():
    L, dims, dev, hostw, row_off, cap, host = _setup([10, 20], 2, seed=3)
    # sequence 0: new rows at 9, 10 against a capacity of 10 (refused); sequence 1: rows 18, 19 of 22
    dev["pos0"] = torch.tensor([9, 18], dtype=torch.int32, device="cuda")
    dev["cap"] = torch.tensor([10, 22], dtype=torch.int32, device="cuda")
    _append(L, dims, dev, 2, host.shape[0])
    torch.cuda.synchronize()
    assert int(dev["status"].item()) & L.MLA_DEV_BAD_POSITION
    got = dev["cache"].cpu().numpy()
    np.testing.assert_array_equal(got[row_off[0]:row_off[0] + 12], host[row_off[0]:row_off[0] + 12])


def test_fp8_refuses_unsupported_shapes():
    L = _L()
    dims = L.make_dims(N_H, D_H, 192, D_R, HIDDEN, BASE)          # d_c not a multiple of 128
    dummy = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    i64 = torch.zeros(1, dtype=torch.int64, device="cuda")
    i32 = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(L.MlaError) as e:
        L.mla_decode_absorbed_fp8(dims, 1, dummy, dummy, dummy, dummy, 16, i64, i32, 1, 0, dummy, dummy.numel(),
                                  dummy, None, st)
    assert e.value.status == L.MLA_ERR_UNSUPPORTED
