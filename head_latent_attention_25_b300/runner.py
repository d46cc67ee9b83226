"""One decode step of one MLA layer over resident device buffers.

``DecodeStep`` owns the device memory of a batch of sequences (latent cache,
index arrays, workspace, outputs; torch allocates it) and enqueues the path
through the C ABI: cache append -> [query projection] -> absorbed decode ->
W_UV projection.  It computes nothing itself.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import _lib as L


class DecodeStep:
    """Device buffers and C-ABI calls of one decode step for ``batch`` sequences.

    ``ctx_lens[b]`` rows are already in the cache before the step; ``n_new``
    tokens are appended at positions ctx_lens[b] .. ctx_lens[b]+n_new-1, and the
    query (position ctx_lens[b]+n_new-1) attends over ctx_lens[b]+n_new rows.
    """

    def __init__(self, *, n_heads: int, d_h: int, d_c: int, d_r: int, hidden: int,
                 dtype: str, ctx_lens: Sequence[int], n_new: int, rope_base: float = 10000.0,
                 softmax_scale: float = 0.0, query_from_h: bool = False, d_q: Optional[int] = None,
                 n_q: int = 1, num_splits: int = 0, extra_rows: int = 0, layout: str = "packed",
                 block_size: int = 64, device: str = "cuda"):
        L.load()
        self.dims = L.make_dims(n_heads, d_h, d_c, d_r, hidden, rope_base, softmax_scale)
        self.dt = L.MLA_BF16 if dtype == "bf16" else L.MLA_F32
        self.tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.batch = B = len(ctx_lens)
        self.n_new = n_new
        # n_q > 1: that many causal queries per sequence (the last n_q positions)
        self.n_q = n_q
        if n_q > 1 and query_from_h:
            raise ValueError("several queries per sequence come with given q_C, q_R")
        if n_q > 1 and layout != "packed":
            raise ValueError("several queries per sequence run on the packed contiguous cache")
        Q = (n_q,) if n_q > 1 else ()
        self.ctx_lens = [int(x) for x in ctx_lens]
        self.query_from_h = query_from_h
        # with a query latent (d_q), c_q = W_DQ h first; without one the query parts come
        # from h itself
        self.d_q = d_q if query_from_h else None
        self.d_q_in = self.d_q if self.d_q else hidden
        self.row_elems = d_c + d_r
        self.device = device
        caps = [c + n_new + extra_rows for c in self.ctx_lens]
        offs, o = [], 0
        for c in caps:
            offs.append(o)
            o += c
        self.total_rows = o
        self.row_off = torch.tensor(offs, dtype=torch.int64, device=device)
        self.cap = torch.tensor(caps, dtype=torch.int32, device=device)
        self.pos0 = torch.tensor(self.ctx_lens, dtype=torch.int32, device=device)
        self.seq_len = torch.tensor([c + n_new for c in self.ctx_lens], dtype=torch.int32, device=device)
        self.max_seq_len = max(c + n_new for c in self.ctx_lens)
        # cache layout: "packed" rows [c ; k_R] in one contiguous buffer (the entry points
        # without a layout), or through an mla_cache_layout: "split" (latents and rotary keys
        # in two buffers), "paged" (blocks of block_size rows, scattered through a pool by a
        # block table), "paged_split" (both)
        self.layout = layout
        self.paged = layout.startswith("paged")
        self.split = layout.endswith("split")
        if self.paged:
            nblk = [(c + block_size - 1) // block_size for c in caps]
            self.max_blocks = max(nblk)
            pool = sum(nblk) + 1                            # one block never used
            perm = torch.randperm(pool, generator=torch.Generator("cpu").manual_seed(12345))
            table = torch.full((B, self.max_blocks), pool - 1, dtype=torch.int32)
            k = 0
            for b, n in enumerate(nblk):
                table[b, :n] = perm[k:k + n].to(torch.int32)
                k += n
            self.block_table = table.to(device)
            self.block_size = block_size
            self.phys_rows = pool * block_size
        else:
            self.block_table = None
            self.phys_rows = self.total_rows
        if self.split:
            self.kv = torch.zeros(self.phys_rows, d_c, dtype=self.tdt, device=device)
            self.pe = torch.zeros(self.phys_rows, d_r, dtype=self.tdt, device=device)
            self.cache = self.kv
        else:
            self.cache = torch.zeros(self.phys_rows, self.row_elems, dtype=self.tdt, device=device)
            self.pe = None
        self.cache_layout = None
        if layout != "packed":
            self.cache_layout = L.make_cache_layout(self.cache, self.pe, rows=self.phys_rows,
                                                    block_table=self.block_table,
                                                    block_size=block_size if self.paged else 0,
                                                    max_blocks=self.max_blocks if self.paged else 0)
        # the step's inputs h, q_c, q_r are views of one contiguous buffer (each part starts
        # on a 256-byte boundary), so a caller can move them with one copy
        def _round(n):
            return (n + 127) // 128 * 128
        n_h, n_c, n_r = B * n_new * hidden, B * n_q * n_heads * d_h, B * n_q * n_heads * d_r
        o_c = _round(n_h)
        o_r = o_c + _round(n_c)
        self.inputs = torch.zeros(o_r + _round(n_r), dtype=self.tdt, device=device)
        self.h = self.inputs[:n_h].view(B, n_new, hidden)
        self.q_c = self.inputs[o_c:o_c + n_c].view(B, *Q, n_heads, d_h)
        self.q_r = self.inputs[o_r:o_r + n_r].view(B, *Q, n_heads, d_r)
        self.x_q = torch.zeros(B, hidden, dtype=self.tdt, device=device) if query_from_h else None
        self.c_q = torch.zeros(B, self.d_q, dtype=self.tdt, device=device) if self.d_q else None
        self.q_ws_bytes = (L.mla_query_latent_workspace_size(self.dims, self.dt, B, self.d_q)
                           if self.d_q else 0)
        self.q_workspace = torch.empty(max(self.q_ws_bytes, 256), dtype=torch.uint8, device=device)
        self.o_lat = torch.zeros(B, *Q, n_heads, d_c, dtype=self.tdt, device=device)
        self.lse = torch.zeros(B, *Q, n_heads, dtype=torch.float32, device=device)
        self.out = torch.zeros(B, *Q, n_heads, d_h, dtype=self.tdt, device=device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)
        self.num_splits = num_splits
        self.ws_bytes = (L.mla_decode_workspace_size(self.dims, self.dt, B, self.max_seq_len, num_splits)
                         if n_q == 1 else
                         L.mla_decode_multi_workspace_size(self.dims, self.dt, B, n_q, self.max_seq_len,
                                                           num_splits))
        if self.ws_bytes == 0:
            raise L.MlaError("mla_decode_workspace_size", L.MLA_ERR_UNSUPPORTED)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.app_ws_bytes = L.mla_append_workspace_size(self.dims, self.dt, B, n_new)
        self.app_workspace = torch.empty(max(self.app_ws_bytes, 256), dtype=torch.uint8, device=device)
        self.w = {}
        self.side = torch.cuda.Stream(device=device)     # the cache append runs here, see step()

    # ------------------------------------------------------------------ inputs
    def set_weights(self, weights: dict):
        for k, v in weights.items():
            self.w[k] = v.to(self.device, self.tdt).contiguous()
        if "w_o" in self.w:
            # the layer output after the step: u = W_O [o_1; ...; o_n_h], two-step or merged
            B = self.batch * self.n_q
            self.u = torch.zeros(B, self.dims.hidden, dtype=self.tdt, device=self.device)
            self.out_ws_bytes = max(L.mla_output_workspace_size(self.dims, self.dt, B, False),
                                    L.mla_output_workspace_size(self.dims, self.dt, B, True))
            self.out_workspace = torch.empty(max(self.out_ws_bytes, 256), dtype=torch.uint8, device=self.device)
            self.w_ov = None

    def physical_rows(self, b: int, positions) -> torch.Tensor:
        """Cache rows of the given positions of sequence b (the layout's addressing)."""
        pos = torch.as_tensor(positions, dtype=torch.int64)
        if not self.paged:
            return pos + int(self.row_off[b].item())
        table = self.block_table[b].to("cpu", torch.int64)
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def read_rows(self, b: int, positions) -> torch.Tensor:
        """Logical rows [c ; k_R] of sequence b at the given positions."""
        idx = self.physical_rows(b, positions).to(self.device)
        if self.split:
            return torch.cat([self.kv[idx], self.pe[idx]], dim=1)
        return self.cache[idx]

    def set_prefill(self, b: int, rows: torch.Tensor):
        n = rows.shape[0]
        rows = rows.to(self.device, self.tdt)
        if self.layout == "packed":
            o = int(self.row_off[b].item())
            self.cache[o:o + n].copy_(rows)
            return
        idx = self.physical_rows(b, range(n)).to(self.device)
        if self.split:
            self.kv[idx] = rows[:, :self.dims.d_c]
            self.pe[idx] = rows[:, self.dims.d_c:]
        else:
            self.cache[idx] = rows

    def set_tokens(self, h: torch.Tensor):
        self.h.copy_(h)
        if self.query_from_h:
            self.x_q.copy_(h[:, -1, :])

    def set_queries(self, q_c: torch.Tensor, q_r: torch.Tensor):
        self.q_c.copy_(q_c)
        self.q_r.copy_(q_r)

    # ------------------------------------------------------------------ path
    def append(self, stream=None):
        if self.cache_layout is not None:
            L.mla_cache_append_ex(self.dims, self.dt, self.batch, self.n_new, self.h, self.w["w_dkv"],
                                  self.w["w_kr"], self.cache_layout, self.row_off, self.cap, self.pos0,
                                  self.app_workspace, self.app_ws_bytes, self.dev_status, stream)
            return
        L.mla_cache_append(self.dims, self.dt, self.batch, self.n_new, self.h, self.w["w_dkv"],
                           self.w["w_kr"], self.row_off, self.cap, self.pos0, self.cache,
                           self.total_rows, self.app_workspace, self.app_ws_bytes, self.dev_status,
                           stream)

    def project_query(self, stream=None):
        if self.d_q:
            L.mla_project_query_latent(self.dims, self.dt, self.batch, self.d_q, self.x_q, self.w["w_dq"],
                                       self.q_workspace, self.q_ws_bytes, self.c_q, self.dev_status, stream)
        L.mla_project_query(self.dims, self.dt, self.batch, self.d_q_in, self.c_q if self.d_q else self.x_q,
                            self.w["w_uq"], self.w["w_qr"], self.q_c, self.q_r, self.dev_status, stream)

    def decode(self, stream=None, num_splits=None, o_lat=None, lse=None):
        ns = self.num_splits if num_splits is None else num_splits
        ws = self.workspace
        if self.n_q > 1:
            if ns != self.num_splits:
                nb = L.mla_decode_multi_workspace_size(self.dims, self.dt, self.batch, self.n_q,
                                                       self.max_seq_len, ns)
                ws = torch.empty(nb, dtype=torch.uint8, device=self.device)
            L.mla_decode_absorbed_multi(self.dims, self.dt, self.batch, self.n_q, self.q_c, self.q_r,
                                        self.w["w_uk"], self.cache, self.total_rows, self.row_off,
                                        self.seq_len, self.max_seq_len, ns, ws, ws.numel(),
                                        self.o_lat if o_lat is None else o_lat,
                                        self.lse if lse is None else lse, self.dev_status, stream)
            return
        if ns != self.num_splits:
            nb = L.mla_decode_workspace_size(self.dims, self.dt, self.batch, self.max_seq_len, ns)
            ws = torch.empty(nb, dtype=torch.uint8, device=self.device)
        if self.cache_layout is not None:
            L.mla_decode_absorbed_ex(self.dims, self.dt, self.batch, self.q_c, self.q_r, self.w["w_uk"],
                                     self.cache_layout, self.row_off, self.seq_len, self.max_seq_len, ns, ws,
                                     ws.numel(), self.o_lat if o_lat is None else o_lat,
                                     self.lse if lse is None else lse, self.dev_status, stream)
            return
        L.mla_decode_absorbed(self.dims, self.dt, self.batch, self.q_c, self.q_r, self.w["w_uk"],
                              self.cache, self.total_rows, self.row_off, self.seq_len,
                              self.max_seq_len, ns, ws,
                              ws.numel(), self.o_lat if o_lat is None else o_lat,
                              self.lse if lse is None else lse, self.dev_status, stream)

    def _decode_args(self):
        return (self.dims, self.dt, self.batch, self.q_c, self.q_r, self.w["w_uk"], self.cache,
                self.total_rows, self.row_off, self.seq_len, self.max_seq_len, self.num_splits,
                self.workspace, self.workspace.numel(), self.o_lat, self.lse, self.dev_status)

    def decode_prepare(self, stream=None, beside=False):
        """Query fold, q_R rotation and schedule into the workspace; reads no cache row.

        beside: the kernels may run beside the kernel enqueued before them on the stream
        (the cache append, which writes nothing they read)."""
        (L.mla_decode_prepare_beside if beside else L.mla_decode_prepare)(*self._decode_args(), stream)

    def decode_attend(self, stream=None):
        """Attention over the cache and merge, from what decode_prepare left in the workspace."""
        L.mla_decode_attend(*self._decode_args(), stream)

    def project_out(self, stream=None):
        L.mla_project_out(self.dims, self.dt, self.batch * self.n_q, self.o_lat, self.w["w_uv"], self.out,
                          self.dev_status, stream)

    def project_output(self, stream=None):
        """u = W_O [o_1; ...; o_n_h] from the step's per-head outputs."""
        L.mla_project_output(self.dims, self.dt, self.batch * self.n_q, self.out, self.w["w_o"],
                             self.out_workspace, self.out_ws_bytes, self.u, self.dev_status, stream)

    def merge_output_weights(self, stream=None):
        """W_OV^(i) = W_O^(i) W_UV^(i) ([n_h, d_c, hidden]), once."""
        d = self.dims
        self.w_ov = torch.empty(d.n_heads, d.d_c, d.hidden, dtype=self.tdt, device=self.device)
        L.mla_merge_output_weights(d, self.dt, self.w["w_o"], self.w["w_uv"], self.w_ov, self.dev_status, stream)

    def project_output_merged(self, u=None, stream=None):
        """u = sum_i W_OV^(i) o_lat_i straight from the latent output."""
        L.mla_project_output_merged(self.dims, self.dt, self.batch * self.n_q, self.o_lat, self.w_ov,
                                    self.out_workspace, self.out_ws_bytes, self.u if u is None else u,
                                    self.dev_status, stream)

    def step(self, stream=None):
        """The whole path: append, [query projection], decode, up-projection.

        The cache append and the query-side half of the decode are independent (the fold
        reads no cache row).  With the query given, both go on one stream and the fold runs
        beside the append (mla_decode_prepare_beside: no fork and join, every launch chained
        to the one before it).  With the query projected from h, the append runs on a second
        stream beside the query projection and the fold; the attention waits for both.
        Under stream capture the second form becomes two branches of the graph.
        """
        if self.n_q > 1 or self.cache_layout is not None:   # the decode is one call
            self.step_serial(stream)
            return
        if not self.query_from_h:
            self.append(stream)
            self.decode_prepare(stream, beside=True)
            self.decode_attend(stream)
            self.project_out(stream)
            return
        main = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.current_stream(self.device)
        self.side.wait_stream(main)             # this step's inputs, and earlier reads of the cache
        self.append(self.side)
        if self.query_from_h:
            self.project_query(main)
        self.decode_prepare(main)
        main.wait_stream(self.side)
        self.decode_attend(main)
        self.project_out(main)

    def step_serial(self, stream=None):
        """The same path as step(), every call on one stream."""
        self.append(stream)
        if self.query_from_h:
            self.project_query(stream)
        self.decode(stream)
        self.project_out(stream)

    def capture(self, stream: Optional[torch.cuda.Stream] = None) -> torch.cuda.CUDAGraph:
        """Record ``step`` once into a CUDA graph; ``graph.replay()`` re-runs the whole path.

        Every call of the path is asynchronous, allocation-free and synchronisation-free,
        so it can be captured; the buffers (and the workspace) are the ones bound here,
        and the device-side index arrays may change between replays.
        """
        g = torch.cuda.CUDAGraph()
        s = stream if stream is not None else torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step(s)                       # warm-up outside capture (lazy loads, attributes)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            self.step(s)
        return g

    def new_rows(self, b: int) -> torch.Tensor:
        return self.read_rows(b, range(self.ctx_lens[b], self.ctx_lens[b] + self.n_new))


def from_workload(wl, ctx_lens=None, num_splits: int = 0, device: str = "cuda", load_inputs: bool = True,
                  layout: str = "packed", block_size: int = 64):
    """A ``DecodeStep`` for a synthetic workload, inputs uploaded from the seeded generators."""
    import mla_inputs
    if ctx_lens is None:
        ctx_lens = mla_inputs.context_lengths(wl)
    st = DecodeStep(n_heads=wl.n_heads, d_h=wl.d_h, d_c=wl.d_c, d_r=wl.d_r, hidden=wl.hidden,
                    dtype=wl.dtype, ctx_lens=ctx_lens, n_new=wl.n_new, rope_base=wl.rope_base,
                    query_from_h=wl.query_from_h, d_q=wl.d_q, n_q=wl.n_q, num_splits=num_splits,
                    layout=layout, block_size=block_size, device=device)
    if load_inputs:
        weights, h, queries = mla_inputs.make_all(wl)
        st.set_weights(weights)
        st.set_tokens(h)
        if queries is not None:
            st.set_queries(*queries)
        for b, n in enumerate(ctx_lens):
            if n:
                st.set_prefill(b, mla_inputs.make_prefill_rows(wl, b, n))
    return st
