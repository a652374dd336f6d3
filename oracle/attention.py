"""Causal GQA softmax attention over a logical KV sequence (test infrastructure only).

The "Paged KV cache" design page states that a page boundary is neither a mask
nor a frontier boundary, that the valid frontier is exact to one token, and
that bytes past the frontier are outside the consumer's valid domain
(granularity table; decode page growth and truncate paragraph).  The logical
attention is the textbook one; this module writes it out in float64 on the
dequantized K/V that ``store.PoolImage.gather`` returns.

Notation: q [T, Hq, D]; K, V [F, Hkv, D]; G = Hq / Hkv; query head i reads
KV head h(i) = i // G (contiguous grouping, the plainest reading: the pages
give no grouping rule).  Scores s_j = scale * <q_i, K_j>; out = softmax(s) V;
lse = ln sum_j exp(s_j) (natural log).

* decode / verify: the T query tokens are the last T positions of a sequence
  of valid length F, so query t sees keys j <= F - T + t.
* chunked prefill / replay: query i of a chunk that starts after ``prefix``
  committed tokens sits at position prefix + i and sees keys j <= prefix + i.
* an empty key set gives out = 0 and lse = -inf (reading taken here).

Pinned by: torch's scaled_dot_product_attention (a library routine) in
float64 on the BF16 profile with an identity table; an explicit-loop brute
force on tiny shapes; closed forms (all-zero keys give lse = ln n and
out = mean V).
"""

from __future__ import annotations

import numpy as np


def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_keys: int, scale: float):
    """One query vector against keys [0, n_keys): returns (out [D], lse)."""
    D = q.shape[-1]
    if n_keys <= 0:
        return np.zeros(D), -np.inf
    s = scale * (K[:n_keys] @ q)
    m = np.max(s)
    e = np.exp(s - m)
    z = np.sum(e)
    return (e @ V[:n_keys]) / z, m + np.log(z)


def decode(q: np.ndarray, K: np.ndarray, V: np.ndarray, F: int, scale: float):
    """Decode / multi-query verify for one sequence.

    q float64 [T, Hq, D]; K, V float64 [>=F, Hkv, D]; F = valid length that
    already includes the T new tokens.  Returns out [T, Hq, D], lse [T, Hq].
    """
    T, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((T, Hq, D))
    lse = np.zeros((T, Hq))
    for t in range(T):
        n = F - T + t + 1
        for i in range(Hq):
            h = i // G
            out[t, i], lse[t, i] = _attend(q[t, i], K[:, h], V[:, h], n, scale)
    return out, lse


def prefill(q: np.ndarray, K: np.ndarray, V: np.ndarray, prefix: int, chunk: int, scale: float):
    """Chunked prefill / replay for one sequence.

    q float64 [Tc, Hq, D] (rows >= chunk are not computed and returned as 0 /
    -inf); K, V float64 [>= prefix + chunk, Hkv, D].
    """
    Tc, Hq, D = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((Tc, Hq, D))
    lse = np.full((Tc, Hq), -np.inf)
    for i_q in range(chunk):
        n = prefix + i_q + 1
        for i in range(Hq):
            h = i // G
            out[i_q, i], lse[i_q, i] = _attend(q[i_q, i], K[:, h], V[:, h], n, scale)
    return out, lse
