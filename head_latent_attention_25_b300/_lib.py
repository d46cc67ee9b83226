"""ctypes binding of ``libmla.so`` (argument marshalling only).

Every function here has the name and argument order of the C entry point in
``include/mla.h``.  Tensor arguments may be torch tensors (their ``data_ptr()`` is
passed) or integer addresses.  Nothing is computed here: every step runs in the
CUDA library, and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA = range(5)
MLA_F32, MLA_BF16 = 0, 1
MLA_DEV_BAD_LENGTH, MLA_DEV_BAD_POSITION, MLA_DEV_TIMEOUT, MLA_DEV_SMEM_ALIGN = 0x1, 0x2, 0x4, 0x8

EXPORTED = ("mla_cache_append", "mla_project_query", "mla_decode_workspace_size",
            "mla_decode_absorbed", "mla_project_out", "mla_status_string", "mla_launch_count",
            "mla_profile_events", "mla_append_workspace_size", "mla_decode_absorbed_noalloc",
            "mla_decode_prepare", "mla_decode_attend", "mla_set_wait_limit_ns",
            "mla_project_query_latent", "mla_query_latent_workspace_size",
            "mla_decode_absorbed_multi", "mla_decode_multi_workspace_size", "mla_project_output",
            "mla_merge_output_weights", "mla_project_output_merged", "mla_output_workspace_size",
            "mla_cache_append_ex", "mla_decode_absorbed_ex", "mla_copy_from_host",
            "mla_decode_prepare_beside", "mla_cache_append_fp8", "mla_decode_absorbed_fp8")


class MlaDims(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("d_h", ctypes.c_int32), ("d_c", ctypes.c_int32),
                ("d_r", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("softmax_scale", ctypes.c_float)]


class MlaCacheLayout(ctypes.Structure):
    """mla_cache_layout: where the latent rows live (packed or split, contiguous or paged)."""
    _fields_ = [("kv", ctypes.c_void_p), ("pe", ctypes.c_void_p), ("kv_stride", ctypes.c_int64),
                ("pe_stride", ctypes.c_int64), ("rows", ctypes.c_int64), ("block_table", ctypes.c_void_p),
                ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32)]


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


_lib = None


def load():
    """The loaded library; raises if ``libmla.so`` is missing (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run `python -m head_latent_attention_25_b300.build`)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(MlaDims)
    lib.mla_cache_append.argtypes = [D, I32, I32, I32, P, P, P, P, P, P, P, I64, P, SZ, P, P]
    lib.mla_append_workspace_size.argtypes = [D, I32, I32, I32]
    lib.mla_append_workspace_size.restype = SZ
    lib.mla_cache_append.restype = I32
    lib.mla_project_query.argtypes = [D, I32, I32, I32, P, P, P, P, P, P, P]
    lib.mla_project_query.restype = I32
    lib.mla_project_query_latent.argtypes = [D, I32, I32, I32, P, P, P, SZ, P, P, P]
    lib.mla_project_query_latent.restype = I32
    lib.mla_query_latent_workspace_size.argtypes = [D, I32, I32, I32]
    lib.mla_query_latent_workspace_size.restype = SZ
    lib.mla_decode_workspace_size.argtypes = [D, I32, I32, I32, I32]
    lib.mla_decode_workspace_size.restype = SZ
    lib.mla_decode_absorbed.argtypes = [D, I32, I32, P, P, P, P, I64, P, P, I32, I32, P, SZ, P, P, P, P]
    lib.mla_decode_absorbed.restype = I32
    lib.mla_decode_absorbed_multi.argtypes = [D, I32, I32, I32, P, P, P, P, I64, P, P, I32, I32, P, SZ, P, P, P,
                                              P]
    lib.mla_decode_absorbed_multi.restype = I32
    lib.mla_decode_multi_workspace_size.argtypes = [D, I32, I32, I32, I32, I32]
    lib.mla_decode_multi_workspace_size.restype = SZ
    CL = ctypes.POINTER(MlaCacheLayout)
    lib.mla_cache_append_ex.argtypes = [D, I32, I32, I32, P, P, P, CL, P, P, P, P, SZ, P, P]
    lib.mla_cache_append_ex.restype = I32
    lib.mla_decode_absorbed_ex.argtypes = [D, I32, I32, P, P, P, CL, P, P, I32, I32, P, SZ, P, P, P, P]
    lib.mla_decode_absorbed_ex.restype = I32
    lib.mla_project_output.argtypes = [D, I32, I32, P, P, P, SZ, P, P, P]
    lib.mla_project_output.restype = I32
    lib.mla_project_output_merged.argtypes = [D, I32, I32, P, P, P, SZ, P, P, P]
    lib.mla_project_output_merged.restype = I32
    lib.mla_merge_output_weights.argtypes = [D, I32, P, P, P, P, P]
    lib.mla_merge_output_weights.restype = I32
    lib.mla_output_workspace_size.argtypes = [D, I32, I32, I32]
    lib.mla_output_workspace_size.restype = SZ
    for name in ("mla_decode_prepare", "mla_decode_attend", "mla_decode_prepare_beside"):
        getattr(lib, name).argtypes = lib.mla_decode_absorbed.argtypes
        getattr(lib, name).restype = I32
    lib.mla_project_out.argtypes = [D, I32, I32, P, P, P, P, P]
    lib.mla_decode_absorbed_noalloc.argtypes = [D, I32, I32, P, P, P, P, I64, P, P, I32, I32, P, P, P, P]
    lib.mla_decode_absorbed_noalloc.restype = I32
    lib.mla_project_out.restype = I32
    lib.mla_status_string.argtypes = [I32]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_launch_count.argtypes = []
    lib.mla_launch_count.restype = ctypes.c_uint64
    lib.mla_profile_events.argtypes = [P, P]
    lib.mla_profile_events.restype = I32
    lib.mla_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.mla_set_wait_limit_ns.restype = ctypes.c_uint64
    lib.mla_cache_append_fp8.argtypes = [D, I32, I32, P, P, P, P, P, P, P, I64, P, SZ, P, P]
    lib.mla_cache_append_fp8.restype = I32
    lib.mla_decode_absorbed_fp8.argtypes = [D, I32, P, P, P, P, I64, P, P, I32, I32, P, SZ, P, P, P, P]
    lib.mla_decode_absorbed_fp8.restype = I32
    lib.mla_copy_from_host.argtypes = [P, P, ctypes.c_size_t, P]
    lib.mla_copy_from_host.restype = I32
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().mla_status_string(int(status)).decode()


def _p(x):
    """Device address of a tensor (or None / int passthrough)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != MLA_OK:
        raise MlaError(fn, status)


def make_dims(n_heads, d_h, d_c, d_r, hidden, rope_base=10000.0, softmax_scale=0.0) -> MlaDims:
    return MlaDims(n_heads, d_h, d_c, d_r, hidden, rope_base, softmax_scale)


def mla_append_workspace_size(dims, dtype, batch, n_new) -> int:
    return int(load().mla_append_workspace_size(ctypes.byref(dims), dtype, batch, n_new))


def mla_cache_append(dims, dtype, batch, n_new, h, w_dkv, w_kr, row_off, cap, pos0, cache,
                     cache_rows, workspace, workspace_bytes, dev_status, stream=None):
    _check("mla_cache_append", load().mla_cache_append(
        ctypes.byref(dims), dtype, batch, n_new, _p(h), _p(w_dkv), _p(w_kr), _p(row_off), _p(cap),
        _p(pos0), _p(cache), cache_rows, _p(workspace), workspace_bytes, _p(dev_status),
        _stream(stream)))


def fp8_row_bytes(d_c: int, d_r: int) -> int:
    """MLA_FP8_ROW_BYTES: E4M3 latent codes, one fp32 scale per 128 columns, bf16 rotary part."""
    return d_c + 4 * (d_c // 128) + 2 * d_r


def mla_cache_append_fp8(dims, batch, n_new, h, w_dkv, w_kr, row_off, cap, pos0, cache, cache_rows,
                         workspace, workspace_bytes, dev_status, stream=None):
    """mla_cache_append into the fp8 row layout (bf16 h and weights)."""
    _check("mla_cache_append_fp8", load().mla_cache_append_fp8(
        ctypes.byref(dims), batch, n_new, _p(h), _p(w_dkv), _p(w_kr), _p(row_off), _p(cap), _p(pos0),
        _p(cache), cache_rows, _p(workspace), workspace_bytes, _p(dev_status), _stream(stream)))


def mla_decode_absorbed_fp8(dims, batch, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len, max_seq_len,
                            num_splits, workspace, workspace_bytes, o_lat, lse, dev_status, stream=None):
    """mla_decode_absorbed over an fp8 cache (bf16 queries, weights and o_lat)."""
    _check("mla_decode_absorbed_fp8", load().mla_decode_absorbed_fp8(
        ctypes.byref(dims), batch, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows, _p(row_off),
        _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes, _p(o_lat), _p(lse),
        _p(dev_status), _stream(stream)))


def mla_project_query(dims, dtype, batch, d_in, x, w_uq, w_qr, q_c, q_r, dev_status, stream=None):
    _check("mla_project_query", load().mla_project_query(
        ctypes.byref(dims), dtype, batch, d_in, _p(x), _p(w_uq), _p(w_qr), _p(q_c), _p(q_r),
        _p(dev_status), _stream(stream)))


def mla_query_latent_workspace_size(dims, dtype, batch, d_q) -> int:
    return int(load().mla_query_latent_workspace_size(ctypes.byref(dims), dtype, batch, d_q))


def mla_project_query_latent(dims, dtype, batch, d_q, h, w_dq, workspace, workspace_bytes, c_q,
                             dev_status, stream=None):
    _check("mla_project_query_latent", load().mla_project_query_latent(
        ctypes.byref(dims), dtype, batch, d_q, _p(h), _p(w_dq), _p(workspace), workspace_bytes, _p(c_q),
        _p(dev_status), _stream(stream)))


def mla_decode_workspace_size(dims, dtype, batch, max_seq_len, num_splits=0) -> int:
    return int(load().mla_decode_workspace_size(ctypes.byref(dims), dtype, batch, max_seq_len,
                                                num_splits))


def mla_decode_absorbed(dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len,
                        max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                        stream=None):
    _check("mla_decode_absorbed", load().mla_decode_absorbed(
        ctypes.byref(dims), dtype, batch, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows,
        _p(row_off), _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes,
        _p(o_lat), _p(lse), _p(dev_status), _stream(stream)))


def mla_decode_multi_workspace_size(dims, dtype, batch, n_q, max_seq_len, num_splits=0) -> int:
    return int(load().mla_decode_multi_workspace_size(ctypes.byref(dims), dtype, batch, n_q, max_seq_len,
                                                      num_splits))


def mla_decode_absorbed_multi(dims, dtype, batch, n_q, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len,
                              max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                              stream=None):
    """n_q causal queries per sequence (query j at position seq_len[b] - n_q + j)."""
    _check("mla_decode_absorbed_multi", load().mla_decode_absorbed_multi(
        ctypes.byref(dims), dtype, batch, n_q, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows,
        _p(row_off), _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes,
        _p(o_lat), _p(lse), _p(dev_status), _stream(stream)))


def mla_decode_prepare(dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len,
                       max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                       stream=None):
    """First half of mla_decode_absorbed: query fold, q_R rotation, schedule (no cache reads)."""
    _check("mla_decode_prepare", load().mla_decode_prepare(
        ctypes.byref(dims), dtype, batch, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows,
        _p(row_off), _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes,
        _p(o_lat), _p(lse), _p(dev_status), _stream(stream)))


def mla_decode_prepare_beside(dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len,
                              max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                              stream=None):
    """mla_decode_prepare that may run beside the kernel before it on the stream."""
    _check("mla_decode_prepare_beside", load().mla_decode_prepare_beside(
        ctypes.byref(dims), dtype, batch, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows,
        _p(row_off), _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes,
        _p(o_lat), _p(lse), _p(dev_status), _stream(stream)))


def mla_decode_attend(dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off, seq_len,
                      max_seq_len, num_splits, workspace, workspace_bytes, o_lat, lse, dev_status,
                      stream=None):
    """Second half of mla_decode_absorbed: split-K attention over the cache and the merge."""
    _check("mla_decode_attend", load().mla_decode_attend(
        ctypes.byref(dims), dtype, batch, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows,
        _p(row_off), _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes,
        _p(o_lat), _p(lse), _p(dev_status), _stream(stream)))


def mla_decode_absorbed_noalloc(dims, dtype, batch, q_c, q_r, w_uk, cache, cache_rows, row_off,
                                seq_len, max_seq_len, num_splits, o_lat, lse, dev_status, stream=None):
    """mla_decode_absorbed without a workspace: uses the library's built-in 32 MiB scratch."""
    _check("mla_decode_absorbed_noalloc", load().mla_decode_absorbed_noalloc(
        ctypes.byref(dims), dtype, batch, _p(q_c), _p(q_r), _p(w_uk), _p(cache), cache_rows,
        _p(row_off), _p(seq_len), max_seq_len, num_splits, _p(o_lat), _p(lse), _p(dev_status),
        _stream(stream)))


def mla_project_out(dims, dtype, batch, o_lat, w_uv, out, dev_status, stream=None):
    _check("mla_project_out", load().mla_project_out(
        ctypes.byref(dims), dtype, batch, _p(o_lat), _p(w_uv), _p(out), _p(dev_status),
        _stream(stream)))


def mla_launch_count() -> int:
    return int(load().mla_launch_count())


def mla_profile_events(start, stop):
    """``start``/``stop``: torch.cuda.Event (timing enabled), raw handles, or None."""
    def h(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    _check("mla_profile_events", load().mla_profile_events(h(start), h(stop)))


def mla_copy_from_host(dst, src, nbytes: int, stream=None):
    """dst: device buffer (tensor or pointer); src: page-locked host buffer (pinned tensor or
    pointer); a kernel reads src over the bus (see include/mla.h)."""
    _check("mla_copy_from_host", load().mla_copy_from_host(_p(dst), _p(src), int(nbytes), _stream(stream)))


def mla_set_wait_limit_ns(ns: int) -> int:
    """Limit of the kernels' bounded waits for later launches (0 = default 2 s); returns the old one."""
    return int(load().mla_set_wait_limit_ns(int(ns)))


def mla_output_workspace_size(dims, dtype, batch, merged) -> int:
    return int(load().mla_output_workspace_size(ctypes.byref(dims), dtype, batch, 1 if merged else 0))


def mla_project_output(dims, dtype, batch, o, w_o, workspace, workspace_bytes, u, dev_status, stream=None):
    """u = W_O [o_1; ...; o_n_h]."""
    _check("mla_project_output", load().mla_project_output(
        ctypes.byref(dims), dtype, batch, _p(o), _p(w_o), _p(workspace), workspace_bytes, _p(u),
        _p(dev_status), _stream(stream)))


def mla_merge_output_weights(dims, dtype, w_o, w_uv, w_ov, dev_status, stream=None):
    """W_OV^(i) = W_O^(i) W_UV^(i), stored [n_h, d_c, hidden]."""
    _check("mla_merge_output_weights", load().mla_merge_output_weights(
        ctypes.byref(dims), dtype, _p(w_o), _p(w_uv), _p(w_ov), _p(dev_status), _stream(stream)))


def mla_project_output_merged(dims, dtype, batch, o_lat, w_ov, workspace, workspace_bytes, u, dev_status,
                              stream=None):
    """u = sum_i W_OV^(i) o_lat_i."""
    _check("mla_project_output_merged", load().mla_project_output_merged(
        ctypes.byref(dims), dtype, batch, _p(o_lat), _p(w_ov), _p(workspace), workspace_bytes, _p(u),
        _p(dev_status), _stream(stream)))


def make_cache_layout(kv, pe=None, kv_stride=None, pe_stride=None, rows=None, block_table=None,
                      block_size=0, max_blocks=0) -> MlaCacheLayout:
    """An mla_cache_layout from tensors (strides and rows default to the tensors' own)."""
    return MlaCacheLayout(_p(kv), _p(pe), kv_stride if kv_stride is not None else kv.shape[-1],
                          (pe_stride if pe_stride is not None else pe.shape[-1]) if pe is not None else 0,
                          rows if rows is not None else kv.shape[0], _p(block_table), block_size, max_blocks)


def mla_cache_append_ex(dims, dtype, batch, n_new, h, w_dkv, w_kr, layout, row_off, cap, pos0, workspace,
                        workspace_bytes, dev_status, stream=None):
    """mla_cache_append into the cache described by ``layout`` (an MlaCacheLayout)."""
    _check("mla_cache_append_ex", load().mla_cache_append_ex(
        ctypes.byref(dims), dtype, batch, n_new, _p(h), _p(w_dkv), _p(w_kr), ctypes.byref(layout), _p(row_off),
        _p(cap), _p(pos0), _p(workspace), workspace_bytes, _p(dev_status), _stream(stream)))


def mla_decode_absorbed_ex(dims, dtype, batch, q_c, q_r, w_uk, layout, row_off, seq_len, max_seq_len,
                           num_splits, workspace, workspace_bytes, o_lat, lse, dev_status, stream=None):
    """mla_decode_absorbed over the cache described by ``layout`` (an MlaCacheLayout)."""
    _check("mla_decode_absorbed_ex", load().mla_decode_absorbed_ex(
        ctypes.byref(dims), dtype, batch, _p(q_c), _p(q_r), _p(w_uk), ctypes.byref(layout), _p(row_off),
        _p(seq_len), max_seq_len, num_splits, _p(workspace), workspace_bytes, _p(o_lat), _p(lse), _p(dev_status),
        _stream(stream)))
