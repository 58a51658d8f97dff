"""The compute-friendly MLA path in fp64 -- TEST INFRASTRUCTURE ONLY.

vllm/v1/attention/backends/mla/common.py, module docstring:

* "Compute Friendly Approach": expand the latent cache per head,
  ``k_nope = kv_c @ W_UK`` and ``v = kv_c @ W_UV``, then run ordinary MHA with
  QK head dim P+R (query ``[q_nope | q_pe]``, key ``[k_nope | k_pe]`` with
  k_pe shared by all heads) and V head dim V.
* "Data-Movement Friendly Approach": absorb W_UK into the query,
  ``ql_nope = einsum("snp,lnp->snl", q_nope, W_UK)`` (the page writes the
  subscripts garbled as "snh,lnh" and the operand as ``q``), run MQA over the
  latent rows, then up-project with ``einsum("snl,lnv->snv", o, W_UV)``.

The two must agree when both use the same softmax scale; the kernels pass
``self.scale`` = 1/sqrt(P+R) explicitly, which is the reading taken here.
This module implements the first path and the two einsums of the second; the
MQA itself is the C oracle (``oracle.decode``), so the identity pins it.
"""
from __future__ import annotations

import numpy as np


def absorb_query(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """ql_nope[t, n, l] = sum_p q_nope[t, n, p] * W_UK[l, n, p]."""
    return np.einsum("snp,lnp->snl", q_nope, w_uk)


def up_project(o_latent: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """o[t, n, v] = sum_l o_latent[t, n, l] * W_UV[l, n, v]."""
    return np.einsum("snl,lnv->snv", o_latent, w_uv)


def expanded_mha(q_nope, q_pe, kv_c, k_pe, w_uk, w_uv, scale, visible):
    """MHA of the expanded keys/values.

    q_nope [T, N, P], q_pe [T, N, R], kv_c [S, Lkv], k_pe [S, R] (keys in
    position order), W_UK [Lkv, N, P], W_UV [Lkv, N, V]; ``visible[t]`` is the
    number of leading keys query token t may see.  Returns (o [T, N, V],
    lse [T, N]) with a natural-log LSE.
    """
    T, N, _ = q_nope.shape
    k_nope = np.einsum("sl,lnp->snp", kv_c, w_uk)          # [S, N, P]
    v = np.einsum("sl,lnv->snv", kv_c, w_uv)               # [S, N, V]
    out = np.zeros((T, N, w_uv.shape[2]))
    lse = np.full((T, N), -np.inf)
    for t in range(T):
        L = int(visible[t])
        if L <= 0:
            continue
        for n in range(N):
            q = np.concatenate([q_nope[t, n], q_pe[t, n]])                 # [P+R]
            k = np.concatenate([k_nope[:L, n], k_pe[:L]], axis=1)          # [L, P+R]
            s = scale * (k @ q)
            m = s.max()
            p = np.exp(s - m)
            out[t, n] = (p[:, None] * v[:L, n]).sum(0) / p.sum()
            lse[t, n] = m + np.log(p.sum())
    return out, lse
