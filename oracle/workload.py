"""Whole-step oracle over a synthetic workload (test infrastructure only).

One step of the path for sequence b: append the step's new tokens to the latent
cache, decode the last new token's query over every cached row (absorbed on the
GPU, explicit here), then project the latent output up per head.  Built only
from ``mla_oracle`` functions and the shared seeded input generators.
"""
from __future__ import annotations

import numpy as np

import mla_inputs
from . import mla_oracle as mo

__all__ = ["oracle_sequence", "oracle_step"]


def oracle_sequence(wl, weights, h, queries, b: int, ctx_len: int, heads=None,
                    form: str = "explicit") -> dict:
    """Oracle outputs of one sequence ``b`` with ``ctx_len`` pre-filled rows.

    ``heads`` restricts the decode to a subset of head indices (outputs are
    then given for those heads only, in that order).  ``form`` picks the
    explicit (K/V materialising) or the absorbed oracle.
    Returns appended rows [n_new, d_c+d_r], o_lat [H, d_c], lse [H], o [H, d_h].
    """
    bf16 = wl.dtype == "bf16"
    prefill = mla_inputs.make_prefill_rows(wl, b, ctx_len)
    pos = np.arange(ctx_len, ctx_len + wl.n_new)
    new_rows = mo.append_rows(h[b], weights["w_dkv"], weights["w_kr"], pos, wl.rope_base, bf16)
    rows = np.concatenate([mo.f64(prefill), new_rows], axis=0)
    if wl.query_from_h:
        q_c, q_r = mo.project_query(h[b, -1], weights["w_uq"], weights["w_qr"], wl.n_heads,
                                    w_dq=weights.get("w_dq"))
    else:
        q_c, q_r = mo.f64(queries[0][b]), mo.f64(queries[1][b])
    w_uk, w_uv = mo.f64(weights["w_uk"]), mo.f64(weights["w_uv"])
    dec = mo.decode_explicit if form == "explicit" else mo.decode_absorbed
    if wl.n_q > 1:
        # several causal queries: query j sits at position n - n_q + j of the n rows and
        # attends over rows 0 .. that position
        n = rows.shape[0]
        outs = []
        for j in range(wl.n_q):
            qc, qr, wk, wv = q_c[j], q_r[j], w_uk, w_uv
            if heads is not None:
                idx = np.asarray(heads)
                qc, qr, wk, wv = qc[idx], qr[idx], wk[idx], wv[idx]
            outs.append(dec(qc, qr, wk, wv, rows[:n - wl.n_q + j + 1], wl.rope_base))
        return {"rows_new": new_rows, "o_lat": np.stack([r["o_lat"] for r in outs]),
                "lse": np.stack([r["lse"] for r in outs]), "o": np.stack([r["o"] for r in outs]),
                "q_c": q_c, "q_r": q_r}
    if heads is not None:
        idx = np.asarray(heads)
        q_c, q_r, w_uk, w_uv = q_c[idx], q_r[idx], w_uk[idx], w_uv[idx]
    r = dec(q_c, q_r, w_uk, w_uv, rows, wl.rope_base)
    return {"rows_new": new_rows, "o_lat": r["o_lat"], "lse": r["lse"], "o": r["o"],
            "q_c": q_c, "q_r": q_r}


def oracle_step(wl, seqs, heads=None, form: str = "explicit") -> dict:
    """Oracle outputs for the listed sequences of workload ``wl``: {b: outputs}."""
    weights, h, queries = mla_inputs.make_all(wl)
    lens = mla_inputs.context_lengths(wl)
    return {b: oracle_sequence(wl, weights, h, queries, b, lens[b], heads, form) for b in seqs}
