"""Seeded synthetic inputs for absorbed MLA decode.

This module only draws random numbers and names workload shapes.  It holds none
of the method's arithmetic (no projection, rotation, softmax or rounding rule of
the method): both the CPU oracle and the CUDA path consume exactly the tensors
produced here.

Recipe (every draw uses ``torch.Generator('cpu')``):

* One master generator seeded with the workload seed draws, in this order:
  the ragged context lengths (only for ragged workloads), ``W_DKV``, ``W_KR``,
  ``W_UK``, ``W_UV``, ``W_DQ`` (only when the query is projected from ``h`` through
  a query latent), ``W_UQ``/``W_QR`` (only when the query is projected from ``h``),
  then ``h`` for the appended tokens, then ``q_C`` and ``q_R`` (only when the query
  is drawn directly), then ``W_O`` (only for workloads that include the output
  projection).
* The pre-filled latent rows of sequence ``b`` come from a generator of their
  own, seeded ``seed * 1_000_003 + 1 + b``, so any one sequence can be rebuilt
  without drawing the others.
* Normal draws are fp32; for bf16 workloads they are rounded to bf16 by torch's
  round-to-nearest-even conversion before either side sees them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

__all__ = ["Workload", "WORKLOADS", "sweep_workloads", "context_lengths",
           "make_weights", "make_tokens", "make_queries", "make_prefill_rows",
           "torch_dtype"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and value distributions of one synthetic decode workload.

    ``prefill`` rows per sequence are drawn directly into the latent cache;
    ``n_new`` tokens per sequence are then appended by the cache-append step,
    and one query per sequence attends over ``prefill + n_new`` rows.
    """
    name: str
    dtype: str                      # "f32" or "bf16": storage type of weights, cache, activations
    batch: int
    n_heads: int
    d_h: int
    d_c: int
    d_r: int
    hidden: int
    prefill: Optional[int]          # rows per sequence before the step; None = ragged
    n_new: int
    seed: int
    weight_std: Optional[float]     # None -> 1/sqrt(fan_in)
    cache_std: float = 0.02
    act_std: float = 1.0            # std of h (and of q_C, q_R unless query_std is set)
    query_std: Optional[float] = None
    query_from_h: bool = False      # q_C = W_UQ h, q_R = W_QR h (no query down-projection given)
    ragged: Optional[tuple] = None  # (low, high) inclusive bounds for ragged context lengths
    d_q: Optional[int] = None       # query latent width (c_q = W_DQ h) when the query comes from h
    rope_base: float = 10000.0
    n_q: int = 1                    # causal queries per sequence (the last n_q new tokens)
    w_o: bool = False               # also draw the output matrix W_O [hidden, n_h*d_h] (drawn last)

    @property
    def row_elems(self) -> int:
        return self.d_c + self.d_r


WORKLOADS = {
    # tiny fp32 decode: the whole cache is built by appending h_0..h_L (positions 0..L, L=128)
    "tiny_f32": Workload("tiny_f32", "f32", batch=1, n_heads=4, d_h=16, d_c=32, d_r=8,
                         hidden=64, prefill=0, n_new=129, seed=0, weight_std=None,
                         query_from_h=True),
    # small bf16 decode: 8 sequences with 1024 cached rows, 8 tokens appended at 1024..1031
    "small_bf16": Workload("small_bf16", "bf16", batch=8, n_heads=16, d_h=128, d_c=512, d_r=64,
                           hidden=2048, prefill=1024, n_new=8, seed=1, weight_std=0.02),
    # DeepSeek-V3-shaped decode: 64 sequences with 4096 cached rows, one new token each
    "v3_b64_l4096": Workload("v3_b64_l4096", "bf16", batch=64, n_heads=128, d_h=128, d_c=512,
                             d_r=64, hidden=7168, prefill=4096, n_new=1, seed=2,
                             weight_std=0.02, d_q=1536),
    # the same decode with the query computed from the new token's h: c_q = W_DQ h (query
    # latent 1536), q_C = W_UQ c_q, q_R = W_QR c_q
    "v3_b64_l4096_from_h": Workload("v3_b64_l4096_from_h", "bf16", batch=64, n_heads=128, d_h=128,
                                    d_c=512, d_r=64, hidden=7168, prefill=4096, n_new=1, seed=2,
                                    weight_std=0.02, d_q=1536, query_from_h=True),
    # long-context ragged decode: 16 sequences, context lengths uniform in [1024, 131072]
    "v3_ragged_b16": Workload("v3_ragged_b16", "bf16", batch=16, n_heads=128, d_h=128, d_c=512,
                              d_r=64, hidden=7168, prefill=None, n_new=1, seed=3,
                              weight_std=0.02, ragged=(1024, 131072), d_q=1536),
}

SWEEP_BATCHES = (1, 32, 128, 256)
SWEEP_CONTEXTS = (512, 8192, 32768)


def sweep_workloads(batches: Sequence[int] = SWEEP_BATCHES,
                    contexts: Sequence[int] = SWEEP_CONTEXTS):
    """The high-concurrency sweep: V3 shapes, batch x context grid, seed 4."""
    out = []
    for b in batches:
        for L in contexts:
            out.append(Workload(f"v3_sweep_b{b}_l{L}", "bf16", batch=b, n_heads=128, d_h=128,
                                d_c=512, d_r=64, hidden=7168, prefill=L, n_new=1, seed=4,
                                weight_std=0.02, d_q=1536))
    return out


def torch_dtype(wl: Workload) -> torch.dtype:
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def _normal(gen: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _master(wl: Workload) -> torch.Generator:
    return torch.Generator("cpu").manual_seed(wl.seed)


def context_lengths(wl: Workload) -> list:
    """Rows per sequence present before the step (ragged ones drawn first from the seed)."""
    if wl.ragged is None:
        return [wl.prefill] * wl.batch
    g = _master(wl)
    lo, hi = wl.ragged
    return torch.randint(lo, hi + 1, (wl.batch,), generator=g).tolist()


def _std(wl: Workload, fan_in: int) -> float:
    return wl.weight_std if wl.weight_std is not None else 1.0 / math.sqrt(fan_in)


def _draw_all(wl: Workload):
    g = _master(wl)
    if wl.ragged is not None:                 # keep the draw order: lengths come first
        lo, hi = wl.ragged
        torch.randint(lo, hi + 1, (wl.batch,), generator=g)
    dt = torch_dtype(wl)
    w = {}
    w["w_dkv"] = _normal(g, (wl.d_c, wl.hidden), _std(wl, wl.hidden), dt)
    w["w_kr"] = _normal(g, (wl.d_r, wl.hidden), _std(wl, wl.hidden), dt)
    w["w_uk"] = _normal(g, (wl.n_heads, wl.d_h, wl.d_c), _std(wl, wl.d_c), dt)
    w["w_uv"] = _normal(g, (wl.n_heads, wl.d_h, wl.d_c), _std(wl, wl.d_c), dt)
    if wl.query_from_h:
        d_in = wl.hidden
        if wl.d_q:
            w["w_dq"] = _normal(g, (wl.d_q, wl.hidden), _std(wl, wl.hidden), dt)
            d_in = wl.d_q
        w["w_uq"] = _normal(g, (wl.n_heads * wl.d_h, d_in), _std(wl, d_in), dt)
        w["w_qr"] = _normal(g, (wl.n_heads * wl.d_r, d_in), _std(wl, d_in), dt)
    h = _normal(g, (wl.batch, wl.n_new, wl.hidden), wl.act_std, dt)
    q = None
    if not wl.query_from_h:
        q_std = wl.act_std if wl.query_std is None else wl.query_std
        lead = (wl.batch,) if wl.n_q == 1 else (wl.batch, wl.n_q)
        q_c = _normal(g, lead + (wl.n_heads, wl.d_h), q_std, dt)
        q_r = _normal(g, lead + (wl.n_heads, wl.d_r), q_std, dt)
        q = (q_c, q_r)
    if wl.w_o:
        w["w_o"] = _normal(g, (wl.hidden, wl.n_heads * wl.d_h), _std(wl, wl.n_heads * wl.d_h), dt)
    return w, h, q


def make_weights(wl: Workload) -> dict:
    """W_DKV [d_c,hidden], W_KR [d_r,hidden], W_UK/W_UV [n_h,d_h,d_c] (+ W_DQ, W_UQ, W_QR)."""
    return _draw_all(wl)[0]


def make_tokens(wl: Workload) -> torch.Tensor:
    """Hidden states of the appended tokens, [B, n_new, hidden]."""
    return _draw_all(wl)[1]


def make_queries(wl: Workload):
    """(q_C [B,n_h,d_h], q_R [B,n_h,d_r]) drawn directly ([B,n_q,...] for several queries
    per sequence); None when projected from h."""
    return _draw_all(wl)[2]


def make_all(wl: Workload):
    """(weights, h, queries) from one pass over the master generator."""
    return _draw_all(wl)


def make_prefill_rows(wl: Workload, b: int, n_rows: int) -> torch.Tensor:
    """Latent rows [n_rows, d_c + d_r] already in the cache for sequence ``b``."""
    g = torch.Generator("cpu").manual_seed(wl.seed * 1_000_003 + 1 + b)
    return _normal(g, (n_rows, wl.row_elems), wl.cache_std, torch_dtype(wl))
